/*
 * dflash.h — C ABI of the GB300 (sm_103a) DFlash 2 block drafter.
 *
 * The drafter (page "cortiq-engine 0.8.71 — src/dflash.rs", module
 * documentation) is a few Qwen3-shaped layers beside a target model:
 *
 *   context  t = norm(FC . [target layer outputs of a row])
 *            K_l = rot(norm(Wk_l . t)),  V_l = Wv_l . t     kept per position
 *   block    rows [anchor, MASK, ..., MASK] at positions a, a+1, ...
 *            x = norm(h); q,k,v = W . x; attention over K_l, V_l before a and
 *            the block's own rows (not causal); h += O . y; the MLP likewise
 *   tokens   logits = head . norm(h); row j >= 1 drafts the token at a + j
 *
 * The DFlash 2 row convolution is bypassed (x and the sub-layer outputs pass
 * unchanged): the workloads this library serves fix no convolution geometry.
 *
 * Conventions for every call:
 *  - Return 0 (DFLASH_OK) on success, a negative DFLASH_E* code otherwise;
 *    dflash_last_error() gives a human-readable reason.  No C++ exception
 *    crosses the ABI and there is no CPU fallback: every step of the path
 *    runs in this library's CUDA kernels.
 *  - After DFLASH_ECUDA the model is poisoned: every later call on it (and
 *    on its sequences) returns DFLASH_ECUDA until dflash_free().
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Work is
 *    queued on it.  Calls on one model (and its sequences) must not overlap:
 *    the model's scratch buffers are shared by its calls.
 *  - Matrices are row-major [out][in] float32, as the page's tensors are.
 *  - Weights and context K/V live in device memory the library allocates and
 *    owns; inputs and outputs are owned by the caller.
 */
#ifndef DFLASH_H
#define DFLASH_H

#include <stdint.h>

#if defined(__GNUC__)
#define DFLASH_API __attribute__((visibility("default")))
#else
#define DFLASH_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* status codes */
#define DFLASH_OK 0
#define DFLASH_EINVAL (-1)    /* a null pointer, a bad size or shape */
#define DFLASH_EGEOM (-2)     /* a geometry the page or the kernels reject */
#define DFLASH_ECAPACITY (-3) /* context rows beyond the sequence's capacity */
#define DFLASH_ERANGE (-4)    /* block_len or a position outside its range */
#define DFLASH_ECUDA (-5)     /* a CUDA call failed; the model is poisoned */
#define DFLASH_ENOMEM (-6)    /* a device or host allocation failed */

/* number formats (dflash_geometry.quant) */
#define DFLASH_QUANT_F32 0   /* every matrix, activation and the head in f32 */
#define DFLASH_QUANT_Q4G32 1 /* draft-layer matrices, fc, Wk/Wv: 4-bit, groups of
                                32 along K with f16 scales; head: int8 per row
                                with an f32 row scale; every matrix input row:
                                int8 per row with an f32 scale; the rest f32 */

typedef struct dflash_model dflash_model; /* weights, geometry, scratch */
typedef struct dflash_seq dflash_seq;     /* one sequence's context K/V */

/*
 * What a DFlash 2 checkpoint fixes (page "cortiq-engine 0.8.71 —
 * src/dflash.rs", `Geometry` and `Geometry::of`).
 * Rules (DFLASH_EGEOM otherwise): layers >= 1; block >= 2; n_taps >= 1;
 * kv_heads >= 1; heads % kv_heads == 0 (the page's rules); and the kernels'
 * limits: head_dim 64 or 128; hidden and intermediate multiples of 64;
 * 0 <= mask_token < vocab; window >= 0 and every windows[l] >= 0;
 * eps > 0; rope_theta > 0; quant one of DFLASH_QUANT_*.
 * Windows (page "cortiq-engine 0.8.71 — src/dflash.rs", `Geometry`:
 * `window`, `windows`; `Drafter::block`, `settle_rows`): block row i of a
 * layer with window w > 0 sees the context positions >= anchor_pos + i + 1
 * - w (and every row of the block); once a layer holds more than 2 w
 * context rows, all but its last w are dropped for good (a later block of
 * that layer reads from the first row still held).
 * Row convolution (page "cortiq-engine 0.8.71 — src/dflash.rs", module
 * documentation, `conv_in` / `conv`, `Drafter::block`): with conv_kernel =
 * kn > 0, each layer wraps attention and the MLP alike: with x the normed
 * rows, d = proj . x (f32; per row 2 kn G values, G = hidden / conv_group,
 * order [stage][offset][group]); the sub-layer reads stage 0 of x and its
 * output passes stage 1 (with the same d) before the residual add, where
 * stage s of rows z is y[i] = sum_{o < min(kn, i + 1)} (base[s][o] +
 * d[i][s][o][group]) * z[i - o] over a block's rows i.  conv_kernel = 0: the
 * sub-layers unwrapped (the same as kn = 1, base 1, proj 0).
 * Candidate selector (page "cortiq-engine 0.8.71 — src/dflash.rs", `select`,
 * `top_k`): with selector_rank > 0 the draft tokens are chosen row by row:
 * row j's selector_top largest logits (the lower index first among equals)
 * scored logit + (P[prev] * (S . hn_j)) . C[candidate] in f32 (products
 * rounded, summed in order), the first best taken; prev is the anchor for
 * row 1 and the previous row's choice after it (hn: the rows after the last
 * norm, f32).
 * windows / no_rope point to `layers` entries each, or are NULL (windows:
 * `window` for every layer; no_rope: every layer rotary).  dflash_init
 * copies them; dflash_geometry_of returns pointers to the model's copies
 * (valid until dflash_free).
 */
typedef struct {
    int32_t hidden;       /* H */
    int32_t intermediate; /* I, the SwiGLU width */
    int32_t layers;       /* L */
    int32_t heads;        /* query heads */
    int32_t kv_heads;     /* key/value heads; query head h reads kv head h / (heads / kv_heads) */
    int32_t head_dim;     /* hd */
    int32_t vocab;        /* V, rows of the target's embedding and head */
    int32_t block;        /* rows of a block: the anchor and block - 1 drafts */
    int32_t n_taps;       /* target layers a context row joins; a row is n_taps * H wide */
    int32_t mask_token;   /* token whose embedding fills rows 1.. of a block */
    int32_t window;       /* positions a block row sees back; 0 = all */
    int32_t quant;        /* DFLASH_QUANT_F32 or DFLASH_QUANT_Q4G32 */
    float eps;            /* RMSNorm epsilon */
    double rope_theta;    /* RoPE base: inv_freq[i] = theta^(-2i/hd) */
    const int32_t* windows; /* per layer, where the layers differ (0 = all); NULL: `window` everywhere */
    const int32_t* no_rope; /* per layer, nonzero: no rotary position on its queries and keys; NULL: none */
    int32_t conv_kernel;    /* rows of the row convolution around each sub-layer; 0 = none */
    int32_t conv_group;     /* columns sharing a dynamic kernel value (conv_kernel > 0: a multiple of 4
                               dividing hidden) */
    int32_t selector_rank;  /* the candidate selector's rank; 0 = none (draft tokens: each row's argmax) */
    int32_t selector_top;   /* candidates it re-scores a row (selector_rank > 0: 1 .. 32, <= vocab) */
} dflash_geometry;

/*
 * The drafter's weights (page "cortiq-engine 0.8.71 — src/dflash.rs",
 * `Drafter::new`: the sidecar's tensor names and shapes), float32 row-major.
 * Per-layer fields point to arrays of `layers` pointers.
 *   fc [H][n_taps*H]   hidden_norm [H]   norm [H]
 *   embed [V][H] (the target's embedding)   head [V][H] (the target's head)
 *   in_norm, post_norm [H];  q_norm, k_norm [hd]
 *   q [heads*hd][H];  k, v [kv_heads*hd][H];  o [H][heads*hd]
 *   gate, up [I][H];  down [H][I]
 * The pointers are host pointers, or device pointers when dflash_init's
 * weights_on_device is 1.  They are read during dflash_init only; the library
 * keeps its own (quantised and packed) copies.
 */
typedef struct {
    const float* fc;
    const float* hidden_norm;
    const float* norm;
    const float* embed;
    const float* head;
    const float* const* in_norm;
    const float* const* post_norm;
    const float* const* q_norm;
    const float* const* k_norm;
    const float* const* q;
    const float* const* k;
    const float* const* v;
    const float* const* o;
    const float* const* gate;
    const float* const* up;
    const float* const* down;
    /* the row convolutions (conv_kernel > 0; NULL otherwise): per layer, for
     * attention and for the MLP, base [2][conv_kernel][H] and the kernel
     * projection [2 * conv_kernel * (H / conv_group)][H] */
    const float* const* attn_conv_base;
    const float* const* attn_conv_proj;
    const float* const* mlp_conv_base;
    const float* const* mlp_conv_proj;
    /* the candidate selector (selector_rank > 0; NULL otherwise): S
     * [selector_rank][H] f32, and the predecessor (P) and successor (C)
     * codebooks [V][selector_rank] as IEEE half bit patterns */
    const float* selector_projection;
    const uint16_t* predecessor_codebook;
    const uint16_t* successor_codebook;
} dflash_weights;

/*
 * Build a model on the current CUDA device: check the geometry, upload the
 * weights and, for DFLASH_QUANT_Q4G32, quantise and pack them on the device
 * (the page's sidecar arrives quantised; this library quantises float32
 * weights itself by the format above).  Blocks until the weights are ready
 * (page "cortiq-engine 0.8.75 — src/gpu_wgpu/dflash_dev.rs", `Dev::new`: the
 * weights are resident before the first block).
 * Errors: EINVAL (null), EGEOM, ENOMEM, ECUDA.  On error *out is NULL and
 * dflash_last_error(NULL) gives the reason.
 */
DFLASH_API int dflash_init(const dflash_geometry* geom, const dflash_weights* weights, int weights_on_device, void* stream,
                dflash_model** out);

/* Free a model and its device memory (sequences must be freed first). NULL is a no-op. */
DFLASH_API void dflash_free(dflash_model* model);

/* The reason of the last failed call on `model` (NULL: the last failed
 * dflash_init of this thread).  Never NULL; "" when nothing failed. */
DFLASH_API const char* dflash_last_error(const dflash_model* model);

/* Copy the geometry a model was built with into *out. */
DFLASH_API int dflash_geometry_of(const dflash_model* model, dflash_geometry* out);

/*
 * A sequence: device K/V storage for up to `max_ctx_rows` context positions
 * in every layer, laid out per layer [kv_heads][max_ctx_rows][head_dim] for
 * keys and the same for values (page "cortiq-engine 0.8.71 —
 * src/dflash.rs", `Ctx`: per layer, per KV head, a row of head_dim per
 * position).  Each f32 value is held as the f16 pair the attention's
 * tensor-core products take, hi = f16(x) and lo = f16(x - hi) (hi + lo = x to
 * about 2^-22 relative), in two planes of the 4 bytes an f32 would take.
 * The context starts empty at position 0.
 * Errors: EINVAL (null, max_ctx_rows < 1), ENOMEM, ECUDA.
 */
DFLASH_API int dflash_seq_new(dflash_model* model, int64_t max_ctx_rows, dflash_seq** out);

/* Free a sequence. NULL is a no-op. */
DFLASH_API void dflash_seq_free(dflash_seq* seq);

/* The positions the context covers: [*first, *next), queued rows included
 * (`Drafter::span`). */
DFLASH_API int dflash_seq_span(const dflash_seq* seq, int64_t* first, int64_t* next);

/*
 * Add the target's rows of positions pos, pos+1, ... to the context
 * (page "cortiq-engine 0.8.71 — src/dflash.rs", `Drafter::push_context`,
 * `queue_context` and `settle_rows`):
 *   t = rms(FC . Q(taps_r), hidden_norm); for every layer
 *   K_l[p] = rot_p(rms_head(Wk_l . Q(t), k_norm_l)),  V_l[p] = Wv_l . Q(t)
 * where Q is the int8 row quantiser in DFLASH_QUANT_Q4G32 and the identity in
 * DFLASH_QUANT_F32.  `taps` is [n_rows][n_taps*hidden] f32, the tapped
 * layers' outputs joined in tap order; a host pointer, or a device pointer
 * when taps_on_device is 1.  Positions: with first <= pos <= next the rows
 * replace position pos and everything after it; pos < first or pos > next
 * starts the context over at pos (next counts queued rows, see
 * dflash_ctx_queue).  The rows are settled at once, after the queued rows
 * still held (`push_context`: queue, then settle).  n_rows == 0 applies the
 * position rule and settles the queue.  Host taps: the call returns once
 * the rows are copied (the caller may reuse its buffer; the work itself may
 * still run, and a device wait that expires in it is reported by the next
 * call that reads the device back: a block with host buffers); device taps:
 * the work is queued on `stream`.
 * Errors: EINVAL (null taps with n_rows > 0, n_rows < 0, pos < 0),
 * ECAPACITY (the context would exceed max_ctx_rows), ECUDA.
 */
DFLASH_API int dflash_ctx_append(dflash_model* model, dflash_seq* seq, int64_t pos, const float* taps, int64_t n_rows,
                      int taps_on_device, void* stream);

/*
 * `dflash_ctx_append` put off (page "cortiq-engine 0.8.71 — src/dflash.rs",
 * `queue_context`, `settle`): the position rule as for an append, then the
 * rows wait, copied into the sequence's device queue, until a block reads
 * the context (dflash_block settles every queued row of its sequences first)
 * or dflash_settle / dflash_ctx_append settle them.  At most 512 rows wait
 * (with every layer windowed: the widest window + 256, if more); past that
 * the oldest are settled now, a multiple of 64 of them.  A truncation cuts
 * queued rows first.  Errors as dflash_ctx_append.
 */
DFLASH_API int dflash_ctx_queue(dflash_model* model, dflash_seq* seq, int64_t pos, const float* taps,
                                int64_t n_rows, int taps_on_device, void* stream);

/* Settle every queued row of `seq` (`settle`).  Errors: EINVAL, ECUDA. */
DFLASH_API int dflash_settle(dflash_model* model, dflash_seq* seq, void* stream);

/* Forget the context from position `pos` on (`Drafter::truncate`). */
DFLASH_API int dflash_truncate(dflash_seq* seq, int64_t pos);

/* Empty the context and move its start back to position 0 (`Drafter::reset`). */
DFLASH_API int dflash_reset(dflash_seq* seq);

/*
 * One block per sequence (page "cortiq-engine 0.8.71 — src/dflash.rs",
 * `Drafter::block` and `block_dev`; page "cortiq-engine 0.8.75 —
 * src/gpu_wgpu/dflash_dev.rs", `Dev::block`): for sequence s the rows
 * [anchor_tok[s], mask, ..., mask] (block_len rows) at positions
 * anchor_pos[s], anchor_pos[s]+1, ... run through every draft layer,
 * attending to context positions [first, min(anchor_pos[s], next)) and to
 * the block's own rows (not causal); then
 *   logits[s][j-1] = head . Q(rms(h_j, norm))  for j = 1 .. block_len-1
 *   draft_tok[s][j-1] = argmax of that row, the lowest index among equals
 *                       (`top_k` with k = 1), decided on the f32 logits.
 * Layout: logits [n_seqs][block_len-1][vocab] f32, draft_tok
 * [n_seqs][block_len-1] u32; either may be NULL (not written).  anchor_tok
 * [n_seqs] and the outputs are host pointers, or device pointers when
 * io_on_device is 1; anchor_pos [n_seqs] is always a host pointer (the
 * positions decide which context rows are read).  Host outputs: the call
 * returns after one device-to-host copy of the results (one round trip);
 * device outputs: the work is queued on `stream`.
 * Errors: EINVAL (null seqs/anchor_tok/anchor_pos, n_seqs < 1, a sequence of
 * another model, anchor_pos < 0), ERANGE (block_len < 2 or > block), ECUDA.
 */
DFLASH_API int dflash_block(dflash_model* model, dflash_seq* const* seqs, int32_t n_seqs, const uint32_t* anchor_tok,
                 const int64_t* anchor_pos, int32_t block_len, float* logits, uint32_t* draft_tok, int io_on_device,
                 void* stream);

/* ---------------------------------------------------------------------------
 * Tracing (the device-side counterpart of the page's stage timers:
 * page "cortiq-engine 0.8.71 — src/dflash.rs", `stage` / `stage_report`, and
 * page "cortiq-engine 0.8.75 — src/gpu_wgpu/dflash_dev.rs", the timestamp
 * queries of `Dev::block`).  While a profile is open, every kernel launch of
 * the library is bracketed by a pair of CUDA events on the launch's stream and
 * tagged with the kernel's name and its algorithmic bytes.
 * ------------------------------------------------------------------------- */

/* Open a profile (clears the previous one).  Errors: EINVAL. */
DFLASH_API int dflash_profile_start(dflash_model* model);

/* Close the profile: waits for the recorded events, then sums device time,
 * launches and algorithmic bytes per kernel name.  Errors: EINVAL, ECUDA. */
DFLASH_API int dflash_profile_stop(dflash_model* model);

/* Entry `index` (0-based) of the closed profile: the kernel's name (a static
 * string), its launches, total device milliseconds between its event pairs
 * and total algorithmic bytes.  Returns ERANGE past the last entry. */
DFLASH_API int dflash_profile_entry(const dflash_model* model, int32_t index, const char** name, int64_t* launches,
                                    double* total_ms, double* total_bytes);

/* Kernels of this library launched on behalf of `model` since dflash_init
 * (-1 for NULL). */
DFLASH_API int64_t dflash_launch_count(const dflash_model* model);

/*
 * Test hook (the pages have no counterpart): switch one of the model's
 * kernel choices, for comparing the alternatives against the oracle.
 *   "tc"         1 (default): matmuls and the head of more than 16 rows on
 *                the tcgen05 kernels; 0: the warp-MMA kernel and the
 *                streaming head.
 *   "dense"      1 (default): the tcgen05 kernels read dense f16 copies of
 *                the weights (built on the first call that needs them);
 *                0: they dequantise the packed weights in shared memory.
 *   "attn_tc_min_keys"  the block attention runs on the tcgen05 kernel
 *                when each of its CTAs streams at least this many keys
 *                (default 256; 0: always where the geometry allows), on
 *                the warp-MMA kernel otherwise.
 *   "head_bound" the dense head trusts its tensor-memory f32 sums while a
 *                row pair's squared code norms multiply to at most this
 *                (default and maximum 2^48); 0 recomputes every element as
 *                an integer dot product.
 * Takes effect for calls after it (captured kernel sequences are dropped).
 * Errors: EINVAL (NULL, unknown name, negative head_bound).
 */
DFLASH_API int dflash_debug_option(dflash_model* model, const char* name, int64_t value);

/* ---------------------------------------------------------------------------
 * Test hooks: views of the library's internal state, for parity checks.
 * All pointers are host pointers; each call synchronises `stream`.
 * ------------------------------------------------------------------------- */

/* Matrix ids for the hooks below: DFLASH_MAT_FC, DFLASH_MAT_HEAD, and for
 * layer l: DFLASH_MAT_LAYER(l, DFLASH_Q) ... DFLASH_MAT_LAYER(l, DFLASH_DOWN). */
#define DFLASH_MAT_FC 0
#define DFLASH_MAT_HEAD 1
#define DFLASH_Q 0
#define DFLASH_K 1
#define DFLASH_V 2
#define DFLASH_O 3
#define DFLASH_GATE 4
#define DFLASH_UP 5
#define DFLASH_DOWN 6
#define DFLASH_MAT_LAYER(l, which) (2 + 7 * (l) + (which))

/*
 * The 4-bit codes and f16 scales the library holds for a matrix, unpacked
 * from its device layout: codes [rows][cols] int8 in [-8, 7] and scales
 * [rows][cols/32] as f16 bit patterns (the quantiser of
 * DFLASH_QUANT_Q4G32).  DFLASH_MAT_HEAD is not a 4-bit matrix: use
 * dflash_debug_head_codes.  Errors: EINVAL (f32 model, bad id), ECUDA.
 */
DFLASH_API int dflash_debug_q4_codes(dflash_model* model, int32_t matrix_id, int8_t* codes, uint16_t* scales, void* stream);

/* The head's int8 codes [vocab][hidden] and f32 row scales [vocab]. */
DFLASH_API int dflash_debug_head_codes(dflash_model* model, int8_t* codes, float* scales, void* stream);

/*
 * The exact integer group sums of the 4-bit matvec kernel for given int8
 * activation codes: out[r][n][g] = sum_{k in group g} x[r][k] * q[n][k],
 * x [rows][cols] int8 (|x| <= 127), out [rows][rows_of_matrix][cols/32]
 * int32, computed by the same tensor-core inner loop the matmuls run.
 * Errors: EINVAL (f32 model, bad id, rows < 1 or > 16), ECUDA.
 */
DFLASH_API int dflash_debug_q4_groupsums(dflash_model* model, int32_t matrix_id, const int8_t* x, int32_t rows, int32_t* out,
                              void* stream);

/*
 * One 4-bit matmul of the library on given int8 activation codes, through
 * the same dispatch the path uses (the streaming kernel for rows <= 16, the
 * tcgen05 tensor-core kernel beyond, where its alignment rules hold):
 * y[r][n] = xs[r] * sum_g s[n][g] * sum_{k in g} q[n][k] x[r][k]
 * (page "cortiq-engine 0.8.75 -- src/gpu_wgpu/dflash_dev.rs", `Dev::q4`,
 * with one activation scale per row).  x [rows][cols] int8 (|x| <= 127), xs
 * [rows] f32, y [rows][rows_of_matrix] f32, all host memory; the call
 * synchronises the stream.  Errors: EINVAL (f32 model, bad id, rows < 1,
 * code -128), ECUDA.
 */
DFLASH_API int dflash_debug_q4_matmul(dflash_model* model, int32_t matrix_id, const int8_t* x, const float* xs,
                                      int32_t rows, float* y, void* stream);

/*
 * Failure detection without a GPU fault: one warp waits, with the bounded
 * wait (a %globaltimer limit) that every kernel of the library uses for its
 * data, on an mbarrier that nothing ever arrives on.  The wait gives up after
 * limit_ns, the kernel raises the model's error flag and returns, and the call
 * reports it exactly as a call whose kernel's data never arrived: ECUDA, and
 * the model is poisoned (every later call on it returns ECUDA); the CUDA
 * context stays usable.  The pages have no counterpart.
 * Errors: EINVAL (limit_ns outside [1 us, 10 s]), ECUDA.
 */
DFLASH_API int dflash_debug_wait_expiry(dflash_model* model, int64_t limit_ns, void* stream);

/*
 * The stored keys and values of context positions [pos, pos + n) of one
 * layer: k and v [n][kv_heads][head_dim] f32 (either may be NULL), each the
 * stored pair's hi + lo.  Errors: EINVAL, ERANGE (positions not held), ECUDA.
 */
DFLASH_API int dflash_debug_read_kv(dflash_model* model, const dflash_seq* seq, int32_t layer, int64_t pos, int64_t n, float* k,
                         float* v, void* stream);

/*
 * Quantisation-site trace, for parity tests that hold the quantised path to
 * f32-level tolerances: an f32 computation and an f64 one quantise the same
 * value to different int8 codes whenever it lies within rounding of a
 * half-step boundary, and one different code moves every later value by a
 * whole quantisation step.  With the trace on, every quantisation site of
 * dflash_ctx_append and dflash_block (the taps; t; per layer the inputs of
 * the fused Wq/Wk/Wv, of Wo, of the fused gate/up and of down; the final
 * normed draft rows), in execution order, records its pre-quantisation f32
 * values [rows][cols], its own int8 codes and its f32 row scales; a decision
 * queued with dflash_debug_trace_force replaces the next site's codes and
 * scales (the site's own are still recorded).  Tracing synchronises the
 * stream at every site.  enable = 1 clears the record and the queue.
 */
DFLASH_API int dflash_debug_trace(dflash_model* model, int32_t enable);
DFLASH_API int dflash_debug_trace_force(dflash_model* model, int32_t rows, int32_t cols, const int8_t* codes,
                                        const float* scales);
/* Site `index` of the record: dims, and (when non-NULL) values, codes and
 * scales copied out.  ERANGE past the last site. */
DFLASH_API int dflash_debug_trace_site(const dflash_model* model, int32_t index, int32_t* rows, int32_t* cols,
                                       float* values, int8_t* codes, float* scales);

/*
 * The block's attention alone (row b4 of the path; page "cortiq-engine 0.8.71
 * — src/dflash.rs", `Drafter::block`: scores of every (head, row) over the
 * context before the anchor and the block's own rows, not causal, softmax,
 * values).  qkv: device [n_seqs*block_len][(heads + 2*kv_heads)*head_dim] f32,
 * each row its q heads, then k heads, then v heads, q and k already normed and
 * rotated, the pointer 16-byte aligned (EINVAL otherwise: the kernel reads
 * it as float4); sequence s reads its layer-`layer` context positions
 * [first, min(anchor_pos[s], next)) and rows s*block_len .. of qkv.  y: device
 * [n_seqs*block_len][heads*head_dim] f32.  anchor_pos is a host array.  Uses
 * the model's scratch (allocated on first need).  Work is queued on `stream`.
 * Errors: EINVAL (null, bad layer or sizes), ERANGE (block_len), ECUDA.
 */
DFLASH_API int dflash_debug_attention(dflash_model* model, dflash_seq* const* seqs, int32_t n_seqs, int32_t layer,
                                      const int64_t* anchor_pos, int32_t block_len, const float* qkv, float* y,
                                      void* stream);

/*
 * dflash_debug_attention without allocating anything (the pages have no
 * counterpart).  It exists for callers that cannot allocate device memory
 * when they run the attention: a host framework that owns every device byte
 * through its own pool allocator (a cudaMalloc behind its back can fail or
 * take memory the pool has promised elsewhere), or a latency-critical loop
 * that must never block in the allocator or synchronise the device, as
 * cudaMalloc and cudaFree can.
 * Same arguments, layouts and result as dflash_debug_attention.  Its scratch
 * is a fixed 16 MiB device array inside this library, held by every GPU that
 * loads the library until the process exits; the call makes no cudaMalloc /
 * cudaFree and calls no allocating library routine.  The array's head takes
 * the context views, which the call passes by value to a small kernel (no
 * host buffer outlives the call); the rest holds, for a long context whose
 * keys split over more CTAs than clusters place, the splits' partial rows
 * (written before they are read: nothing needs to start at zero); when those
 * rows do not fit, the call runs the cluster merge (distributed shared
 * memory), which needs no partials in global memory.  The first call on a
 * device looks up that array's device address (cudaGetSymbolAddress, with
 * the device current) and keeps it.  Every call shares the one array and
 * overwrites what the previous call left there, so calls whose work overlaps
 * on the GPU (other streams, other threads) race: order them on one stream.
 * Errors: as dflash_debug_attention, and ERANGE when the context views do not
 * fit the array (more than 256 sequences) -- nothing is launched then.
 */
DFLASH_API int dflash_attention_noalloc(dflash_model* model, dflash_seq* const* seqs, int32_t n_seqs, int32_t layer,
                                        const int64_t* anchor_pos, int32_t block_len, const float* qkv, float* y,
                                        void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DFLASH_H */
