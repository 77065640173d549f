// Host-side launchers of the library's kernels.  Each returns a cudaError_t
// value as int (0 = queued fine).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "common.cuh"

namespace dflash {

// ---- init-time quantisers / packers (k_quant.cu)
// 4-bit matrices in layout L (common.cuh); tile0: first 16-row tile of the
// sub-matrix inside the fused matrix.
int q4_quantize_pack(const float* w_dev, int N, int K, uint8_t* packed, Q4Layout L, int tile0, __half* scale_scratch,
                     cudaStream_t st);
int q4_unpack(const uint8_t* packed, Q4Layout L, int tile0, int N, int K, int8_t* codes, uint16_t* scales,
              cudaStream_t st);
int i8_rows_quantize_pack(const float* w_dev, int N, int K, int Npad, int ksteps, int8_t* packed, float* row_scale,
                          cudaStream_t st);
int i8_unpack(const int8_t* packed, int N, int K, int ksteps, int8_t* codes, cudaStream_t st);

// ---- launching: every kernel of the library goes out with the programmatic
// stream-serialisation attribute (programmatic dependent launch), so that it
// may start -- and stream its weights -- while the previous kernel on the
// stream finishes; each kernel waits (pdl_wait) before it touches what its
// predecessors write.  Without a predecessor kernel the attribute is inert.
template <typename... KArgs, typename... Args>
cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Raises a kernel's dynamic shared-memory limit to `bytes` where `*limit` (the
// call site's record of what it set) is below it.  One lock guards every such
// record and call, so host threads may run the library's entry points at once.
std::mutex& attr_mutex();
template <typename Kernel>
cudaError_t raise_smem_limit(Kernel kernel, size_t bytes, size_t* limit) {
    std::lock_guard<std::mutex> lock(attr_mutex());
    if (bytes <= *limit) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess) *limit = bytes;
    return e;
}

// Row maps: output row i reads source row  (i / per) * stride + skip + i % per.
struct RowMap {
    int per, stride, skip;
};

// ---- matmuls (k_gemm.cu, k_stream.cu)
// Activation operand of the quantised matmuls: int8 codes [rows][ld]
// (ld >= K, a multiple of 16), one f32 scale a row.
struct QAct {
    const int8_t* codes;
    const float* scale;
    int ld;
};

// y[t][n] (+)= xs[t] * sum_g s[n][g] * sum_{k in g} q[n][k] x[t][k] for n < N,
// t < T, any T (16 rows per CTA).  accumulate: add into y (atomically);
// otherwise y is overwritten.
int q4_gemm(const uint8_t* packed, Q4Layout L, int tile0, int N, QAct x, int T, float* y, int ldy, bool accumulate,
            int num_sms, cudaStream_t st);
// The int32 group sums of the same inner loop (T <= 16): out[t][n][g].
int q4_groupsums(const uint8_t* packed, Q4Layout L, int tile0, int N, QAct x, int T, int32_t* out, cudaStream_t st);

// The same product for many rows on the tcgen05 tensor cores (k_tc.cu):
// 128-row x 256-output tiles, the 4-bit weights dequantised in shared memory
// to exact hi + lo f16 pairs, f32 accumulation in tensor memory.  Needs
// tile0 % 4 == 0, N % 64 == 0, x.ld % 16 == 0, 16-byte aligned codes, y and
// ldy (q4_tc_supported); err_flag is raised when a bounded wait expires.
// x16: the same codes as f16 [T][K] (codes_to_f16), which the kernel's TMA
// reads; x.scale the rows' scales.
bool q4_tc_supported(Q4Layout L, int tile0, int N, int K, QAct x);
int q4_tc(const uint8_t* packed, Q4Layout L, int tile0, int N, QAct x, const __half* x16, int T, float* y, int ldy,
          bool accumulate, int num_sms, int* err_flag, cudaStream_t st);
// The head for many rows on the same kernel (exact int32 row sums, drained
// from tensor memory every 512 columns): logits (may be nullptr) and the
// argmax keys as head_stream.
bool head_tc_supported(int ksteps, QAct x);
int head_tc(const int8_t* packed, const float* row_scale, int V, int ksteps, QAct x, const __half* x16, int T,
            float* logits, int ldl, unsigned long long* keys, int* err_flag, cudaStream_t st);
// Dense f16 weight copies for the many-row path (k_tc.cu): hi = f16(s q),
// lo = f16(s q - hi) [N][K] from a 4-bit matrix's codes and f16 scales.
int dequant_hilo(const int8_t* codes, const uint16_t* scales, int N, int K, __half* hi, __half* lo, cudaStream_t st);
// The 4-bit matmul and the head on those copies (k_tc_pair.cu): every operand
// tile by TMA, no conversion in the kernel; 256-row x 256-output units on
// pairs of SMs (tcgen05.mma cta_group::2), a persistent grid of at most one
// pair per two SMs with two accumulators in tensor memory, so the epilogue of
// one unit overlaps the MMAs of the next.  y as q4_tc (cleared first where K
// is split over units and accumulate is off).
int q4_tc_dense(const __half* hi, const __half* lo, int N, int K, QAct x, const __half* x16, int T, float* y, int ldy,
                bool accumulate, int* err_flag, cudaStream_t st);
// The head takes the squared code norms of its vocabulary rows (w_norm2 [V],
// largest w_norm2_max) and of the activation rows (x_norm2 [T]): an element
// whose norm product passes `bound` (2^48: a partial sum could leave the
// exact f32 integers) is recomputed as an integer dot product; logits (may
// be nullptr) and the argmax keys as head_stream.
int head_tc_dense(const __half* w16, const int* w_norm2, const float* row_scale, int V, int K, QAct x,
                  const __half* x16, const int* x_norm2, int T, float* logits, int ldl, unsigned long long* keys,
                  unsigned long long bound, unsigned long long w_norm2_max, int* err_flag, cudaStream_t st);
// int8 activation codes [T][ld] -> f16 [T][K] (exact), for the tcgen05 kernels'
// TMA; with norm2 non-null also each row's squared code norm (K < 2^17).
int codes_to_f16(const int8_t* x, int ld, int T, int K, __half* out, int* norm2, int num_sms, cudaStream_t st);

// The streaming form for up to 16 rows: every CTA streams a contiguous slice
// of the matrix (tile0 and N multiples of 64 rows) through a bulk-copy ring
// and ADDS its partial sums into y (which must hold zeros or the residual).
int q4_stream(const uint8_t* packed, Q4Layout L, int tile0, int N, QAct x, int T, float* y, int ldy, int num_sms,
              int* err_flag, cudaStream_t st);
size_t q4_stream_smem_bytes(Q4Layout L, int N, int num_sms);

// The head: logits[t][n] = xs[t] * sw[n] * sum_k q[n][k] x[t][k] (exact int32
// sums on f16 tensor cores), and keys[t] = max over n of argmax_key(logit, n)
// (keys zeroed before).  logits may be nullptr.  Any T (16 rows per pass).
int head_stream(const int8_t* packed, const float* row_scale, int V, int ksteps, QAct x, int T, float* logits,
                int ldl, unsigned long long* keys, int num_sms, int* err_flag, cudaStream_t st);

// y[t][n] (+)= sum_k W[n][k] x[t][k]; W f32 [N][K] (K % 4 == 0).
int linear_f32(const float* W, int N, int K, const float* x, int ldx, int T, float* y, int ldy, bool accumulate,
               cudaStream_t st);
// keys[t] = max over n < V of argmax_key(logits[t][n], n).
int argmax_rows(const float* logits, int ldl, int V, int T, unsigned long long* keys, cudaStream_t st);
// tokens[t] = index encoded in keys[t].
int keys_to_tokens(const unsigned long long* keys, int T, uint32_t* tokens, cudaStream_t st);
// The candidate selector: per row the k (<= 32, <= V) largest logits as
// argmax keys, largest first (out [T][k]); then per sequence, its `rows` rows
// in order, the choices (chosen) and each row's own top token (plain) from
// the candidates, hp [n_seqs*rows][rank] (the rows' projection) and the f16
// codebooks [V][rank].
// (two launches: the rows' parts, then their merge; scratch holds
// T * topk_parts(V, k) * k keys)
int topk_parts(int V, int k);
int topk_rows(const float* logits, int ldl, int V, int T, int k, unsigned long long* scratch, unsigned long long* out,
              cudaStream_t st);
int select_tokens(const unsigned long long* cand, int k, const float* hp, int rank, const __half* book_p,
                  const __half* book_c, int V, const uint32_t* anchors, int n_seqs, int rows, uint32_t* chosen,
                  uint32_t* plain, cudaStream_t st);

// ---- layer pieces (k_layer.cu)
// x = rms(src, w) (w == nullptr: no norm, x = src); then either f32 out
// (out_f32 != nullptr) or int8 codes + an f32 scale per row.
// zero_buf / zero_n: a buffer the kernel clears on the side (nullptr: none).
// out16 (nullptr: none): the codes also as exact f16 values [rows][n] (the
// tcgen05 matmuls' activation operand).
// div (nullptr: none): the source row is a sum of parts, and each div_seg
// columns of source row r are first divided by div[r][segment] (the
// attention's accumulate mode: y = yacc / lacc per head).
int rms_rows(const float* src, int ld_src, RowMap map, int rows, int n, const float* w, float eps, float* out_f32,
             int ld_out, int8_t* out_codes, float* out_scale, int ld_codes, cudaStream_t st,
             float* zero_buf = nullptr, int64_t zero_n = 0, const float* div = nullptr, int div_seg = 0,
             __half* out16 = nullptr);
// h[r] = embed[tok(r)]: row r of sequence s = r / block_len is the anchor
// (anchor_tok[s]) for r % block_len == 0, the mask token otherwise.  Side
// duty (rope != nullptr): the block rows' rotation table rope[r][i] =
// (cos, sin) of f32(pos0[s] + r % block_len) * inv_freq[i], i < hd / 2.
int embed_rows(const float* embed, int H, int vocab, const uint32_t* anchor_tok, int mask_token, int n_seqs,
               int block_len, float* h, cudaStream_t st, const int64_t* pos0 = nullptr,
               const float* inv_freq = nullptr, int hd = 0, float2* rope = nullptr);
// Context rows: kv [n][L * 2 * nkv * hd] (per layer k then v) -> the
// sequence's store: K rows normed (k_norm_l) and rotated at position
// pos0 + r, V rows as they are; stored at index idx0 + r as (hi, lo) f16
// pairs (plane hi [nkv][cap][hd], then plane lo), where pos_dev = {pos0,
// idx0} lives in device memory (set per call).
// rotary_dev: per layer, 0 where the layer's keys carry no rotary position
// (nullptr: every layer rotary).
int kv_append(const float* kv, int n, int L, int nkv, int hd, const float* const* k_norm_dev, const float* inv_freq,
              float eps, const int64_t* pos_dev, __half* const* kstore_dev, __half* const* vstore_dev, int64_t cap,
              cudaStream_t st, const int* rotary_dev = nullptr);
// a = silu(g) * u for gu [rows][2I] (gate then up); f32 out or int8 codes.
// The same with the grid in clusters of cluster_x CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                           int cluster_x, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)cluster_x;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

int silu_mul(const float* gu, int ld_gu, int rows, int I, float* out_f32, int ld_out, int8_t* out_codes,
             float* out_scale, int ld_codes, cudaStream_t st, __half* out16 = nullptr);
// One stage of the row convolution over `rows` block rows (block_len rows a
// sequence) of n columns: y[r] = sum_{o < min(kn, r % block_len + 1)}
// (base[stage][o] + d[r][(stage kn + o) (n / gs) + group]) * x[r - o], base
// [2][kn][n], d [rows][ldd] (2 kn n / gs used); then h_add[r] += y, y as f32
// (out_f32) and / or as int8 codes + scale (out_codes), each where non-null.
// gs % 4 == 0, n % gs == 0, n <= 32768; zero_buf / zero_n cleared on the side.
int conv_rows(const float* x, int ldx, const float* d, int ldd, const float* base, int stage, int kn, int gs, int n,
              int rows, int block_len, float* h_add, int ldh, float* out_f32, int ld_out, int8_t* out_codes,
              float* out_scale, int ld_codes, cudaStream_t st, float* zero_buf = nullptr, int64_t zero_n = 0);

// Attention of a block over its sequence's context and its own rows.
struct AttnSeq {
    // The layer's key and value stores, each value as its (hi, lo) f16 pair
    // (hi = f16(x), lo = f16(x - hi)): plane hi [nkv][cap][hd], then plane lo
    // [nkv][cap][hd].
    const __half* kc;
    const __half* vc;
    int64_t cap;
    int64_t lo;  // first context index read (position - first)
    int n;       // context rows read
    // context rows (of the n) block row 0 does not see, row i: cut + i
    // (a layer's window; kNoCut: every row sees all n)
    int cut;
    // the tcgen05 attention's tensor maps of the two stores (keys, then
    // values: kv_tensor_maps), in device memory; nullptr where not built
    const void* maps;
};
constexpr int kNoCut = -(1 << 30);
// qkv [n_seqs*block_len][ld] (q, k, v of the block); with q_norm != nullptr
// the kernel applies the per-head RMSNorm (q_norm / k_norm) and the rotation
// (table `rope` of embed_rows) to q and to the block's k as it loads them,
// otherwise q and k arrive normed and rotated; rope == nullptr with the
// norms: normed, not rotated (a layer without the rotary position).  Each
// view's `cut` masks the leading context rows a windowed layer's block row
// does not see.  y [n_seqs*block_len][nq*hd].  `part` / part_floats: scratch of
// attn_scratch_floats() floats: none when the key splits merge in
// distributed shared memory (clusters), the splits' partial rows when long
// contexts split the keys over more CTAs than the clusters place and merge
// through global memory (nothing in it needs to start at zero).
// max_ctx: the largest context any sequence of the call may hold (its
// capacity); the launch depends on it, each CTA's key range on the actual n.
// windowed: some view has a cut (kNoCut everywhere otherwise: the kernel
// without the window mask runs).
// kv_ready: no kernel that may still run when this one starts (the chain of
// programmatic dependent launches before it) writes the context stores, so
// their copies may go out before the kernel's dependency wait.
int attention(const float* qkv, int ld, int n_seqs, int block_len, const AttnSeq* seqs_dev, int max_ctx, int nq,
              int nkv, int hd, float scale, float* part, int64_t part_floats, float* y, int num_sms, cudaStream_t st,
              const float* q_norm = nullptr, const float* k_norm = nullptr, const float2* rope = nullptr,
              float eps = 0.f, bool kv_ready = false, bool windowed = false);
int64_t attn_scratch_floats(int n_seqs, int block_len, int max_ctx, int nq, int nkv, int hd, int num_sms);
// Kernels one attention call with part_floats of scratch launches (2 when
// the key splits merge through global memory: the split kernel, then the
// merge; with less scratch than attn_scratch_floats() the call falls back to
// the cluster merge).
int attn_kernels(int n_seqs, int block_len, int max_ctx, int nq, int nkv, int hd, int num_sms, int64_t part_floats);

// Accumulate mode of the attention, for layers whose queries and keys the
// kernel RMS-norms (q_norm, k_norm): every score s of the layer then obeys
// s * log2(e) * scale <= ref_log2 (the bound the gains give), so each CTA's
// partial rows, rescaled by 2^(m - ref_log2), add into yacc [rows][nq * hd]
// (unnormalised output) and lacc [rows][nq] (softmax sums) with atomics, in
// any order: the merge of the key splits needs neither clusters nor a second
// kernel.  Both must hold zeros before the launch; y = yacc / lacc per head
// (rms_rows' divisor) finishes it.  attn_acc_plan: the key splits a unit
// takes in this mode (0: not worth it -- as many units as SMs, or a single
// key step -- use attention()).
int attn_acc_plan(int n_seqs, int block_len, int max_ctx, int nq, int nkv, int hd, int num_sms);
int attention_acc(const float* qkv, int ld, int n_seqs, int block_len, const AttnSeq* seqs_dev, int nsplit, int nq,
                  int nkv, int hd, float scale, float* yacc, float* lacc, float ref_log2, cudaStream_t st,
                  const float* q_norm, const float* k_norm, const float2* rope, float eps, bool kv_ready,
                  bool windowed);

// The same accumulate mode on the tcgen05 tensor cores (k_attn_tc.cu): one
// CTA takes all query rows of a (sequence, kv head) unit (rep * block_len <=
// 128) against its share of the keys, 64 keys a step.  attn_tc_plan: the key
// splits a unit takes (1 when the units fill the SMs).  err: raised when a
// bounded wait expires.
bool attention_tc_supported(int nq, int nkv, int hd, int block_len);
// The two tensor maps (CUtensorMap, 128 bytes each: keys, then values) of a
// layer's stores [2 planes][nkv][cap][hd] f16 that the tcgen05 attention
// reads 64-row x 64-column boxes of, in the 128-byte swizzle.  out: host
// memory of 256 bytes, 64-byte aligned.  false when the driver lacks the
// encoder or rejects the shape.
bool kv_tensor_maps(const __half* k, const __half* v, int nkv, int64_t cap, int hd, void* out);
int attn_tc_plan(int n_seqs, int block_len, int max_ctx, int nkv, int num_sms);
int attention_tc(const float* qkv, int ld, int n_seqs, int block_len, const AttnSeq* seqs_dev, int nsplit, int nq,
                 int nkv, int hd, float scale, float* yacc, float* lacc, float ref_log2, cudaStream_t st,
                 const float* q_norm, const float* k_norm, const float2* rope, float eps, bool kv_ready, bool windowed,
                 int* err);

// Up to kViewsMax context views passed by value (a kernel parameter of
// about 10 KB), for a caller that must not keep a host buffer alive past its
// call: attn_views_store writes them to dst (device memory) in stream order
// -- it waits for the kernels before it, and an attention kernel after it
// reads the views after its own dependency wait (kv_ready false).
constexpr int kViewsMax = 256;
struct AttnViews {
    int n;
    AttnSeq v[kViewsMax];
};
int attn_views_store(const AttnViews& views, AttnSeq* dst, cudaStream_t st);

// Failure detection without a fault: one warp's bounded wait on an mbarrier
// that nothing arrives on runs out after limit_ns and raises *err_flag.
int wait_expiry(int* err_flag, uint64_t limit_ns, cudaStream_t st);

}  // namespace dflash
