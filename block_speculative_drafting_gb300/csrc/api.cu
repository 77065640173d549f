// The C ABI of include/dflash.h: model and sequence state, weight upload and
// packing, and the order of kernels of a context append and of a block.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/dflash.h"
#include "common.cuh"
#include "kernels.cuh"

using namespace dflash;

namespace {

thread_local std::string g_init_error;

// Context rows projected per pass of an append (bounds the scratch buffers).
constexpr int64_t kAppendRows = 8192;
// Keys a CTA of the tcgen05 attention streams at least for it to be chosen
// over the warp-MMA kernel (measured on GB300: the tcgen05 kernel wins from
// about four 64-key steps a CTA; at context 2048 a split holds under two)
constexpr int64_t kTcAttnMinKeys = 256;

struct DevBuf {
    void* p = nullptr;
    size_t bytes = 0;
};

struct Layer {
    float *in_norm = nullptr, *post_norm = nullptr, *q_norm = nullptr, *k_norm = nullptr;
    uint8_t *qkv_p = nullptr, *o_p = nullptr, *gu_p = nullptr, *down_p = nullptr;  // 4-bit packed
    float *qkv_f = nullptr, *o_f = nullptr, *gu_f = nullptr, *down_f = nullptr;    // f32
    // the row convolutions around attention (a) and the MLP (m): base
    // [2][kn][H], kernel projection [2 kn G][H] (f32)
    float *a_base = nullptr, *a_proj = nullptr, *m_base = nullptr, *m_proj = nullptr;
};

struct MatView {
    const uint8_t* packed;
    const float* f32;
    int tile0, N, K;
    Q4Layout L;
};

Q4Layout make_layout(int rows, int K) {
    Q4Layout L;
    L.ngroups = rows / 64;
    L.ksteps = K / kQ4KStep;
    L.kb = q4_kblock_steps(L.ksteps);
    return L;
}

}  // namespace

struct dflash_model {
    dflash_geometry g{};
    int device = 0, num_sms = kSMs;
    bool poisoned = false;
    std::string err;
    std::vector<void*> owned;  // device allocations freed with the model
    int live_seqs = 0;

    float *embed = nullptr, *hidden_norm = nullptr, *norm = nullptr, *inv_freq = nullptr;
    uint8_t *fc_p = nullptr, *kvctx_p = nullptr;
    float *fc_f = nullptr, *kvctx_f = nullptr, *head_f = nullptr;
    int8_t* head_p = nullptr;
    float* head_scale = nullptr;
    std::vector<Layer> layers;
    const float** k_norm_dev = nullptr;  // [L] device pointers to k_norm

    int qd = 0, kd = 0, qkv_w = 0, tap_w = 0, kvctx_w = 0;
    // layouts of the packed 4-bit matrices (the same for every layer)
    Q4Layout L_fc{}, L_kvctx{}, L_qkv{}, L_o{}, L_gu{}, L_down{};
    int* err_dev = nullptr;   // raised by a kernel whose bounded wait expired
    // per layer: the window (positions a block row sees back, 0 = all) and
    // whether queries and keys carry the rotary position; rot_dev: the
    // latter on the device (kv_append)
    std::vector<int32_t> win, norope;
    // per layer: the attention's accumulate-mode reference (log2 domain): a
    // bound on every score the layer's normed queries and keys can make, or
    // NaN when the gains are too large for the mode's f32 range
    std::vector<float> attn_ref;
    int* rot_dev = nullptr;
    // the candidate selector: S [rank][H] f32, codebooks P, C [V][rank] f16
    float* sel = nullptr;
    __half *book_p = nullptr, *book_c = nullptr;
    DevBuf hn, hp, cand, plain;  // its scratch: normed rows, their projection, candidates, own top tokens
    // options (dflash_debug_option): matmuls of more than 16 rows on the
    // tcgen05 kernels (off: the mma.sync kernel), from dense f16 weight copies
    // (off: dequantised in the kernel)
    bool use_tc = true;
    bool use_dense = true;
    int64_t tc_attn_min_keys = kTcAttnMinKeys;  // keys a CTA of the tcgen05 attention streams at least
    // dense f16 copies of the matrices for the many-row path, built on first need:
    // the 4-bit matrices as (hi, lo) planes [N][K], the head's codes [vocab][hidden]
    struct DenseMat {
        const uint8_t* packed;
        int N, K;
        __half *hi, *lo;
    };
    std::vector<DenseMat> dense;
    __half* head16 = nullptr;
    int* head_norm2 = nullptr;  // squared code norm of each vocabulary row (the dense head's guard)
    unsigned long long head_norm2_max = 0;
    // the dense head trusts its f32 sums while |x|^2 |w|^2 <= this (2^48:
    // every partial sum within 2^24); option "head_bound" lowers it (0
    // recomputes every element as an integer dot product)
    unsigned long long head_bound = 1ull << 48;
    bool dense_ready = false;
    // set while run_enqueue captures a graph of the library's own: the
    // context stores are then final for every kernel of a block
    bool own_capture = false;
    int* err_host = nullptr;  // pinned copy, read after a synchronising call

    // launch accounting and the optional per-launch event profile
    int64_t launches = 0;  // kernels of this library launched since init
    bool profiling = false;
    struct ProfRec {
        const char* name;
        cudaEvent_t e0, e1;
        double bytes;
        int kernels;
    };
    std::vector<ProfRec> prof_open;
    std::vector<cudaEvent_t> ev_pool;
    // recorded after a call's last copy from caller host memory: the call
    // waits for it (the caller may reuse its buffer), not for the work after
    cudaEvent_t copy_ev = nullptr;
    struct ProfSum {
        const char* name;
        int64_t launches = 0;
        double ms = 0, bytes = 0;
    };
    std::vector<ProfSum> prof_sum;

    // quantisation-site trace (test hook): every site's pre-quantisation
    // values, codes and scales in execution order, and queued decisions that
    // replace a site's own codes and scales
    struct Site {
        int rows = 0, cols = 0;
        std::vector<float> values, scales;
        std::vector<int8_t> codes;
    };
    bool tracing = false;
    std::vector<Site> trace;
    std::vector<Site> forced;
    size_t forced_next = 0;
    DevBuf trace_buf;

    // scratch, grown on demand (a call that needs more memory than any call
    // before it allocates; calls of the same sizes allocate nothing)
    DevBuf h, xq, xs, qkv, y, gu, logits, keys, toks, part, anchors, pos0, aseqs, rope;
    DevBuf a_taps, a_codes, a_scale, a_t, a_kv, a_pos;
    DevBuf x16;  // activation codes as f16 for the tcgen05 kernels (matmuls of more than 16 rows)
    DevBuf cx, cd, co;  // the row convolution: normed rows, their dynamic kernels, a sub-layer's output
    bool grown = false;  // a scratch buffer moved since the graphs were captured

    // CUDA graphs of the kernel sequences of a block and of a short append,
    // captured once per shape (and buffer set) on cap_stream, replayed on
    // the caller's stream
    struct GraphEntry {
        std::vector<int64_t> key;
        cudaGraphExec_t exec;
        int64_t kernels;
    };
    std::vector<GraphEntry> graphs;
    cudaStream_t cap_stream = nullptr;
    bool use_graphs = true;
};

struct dflash_seq {
    dflash_model* m = nullptr;
    int64_t cap = 0, first = 0, len = 0;
    // per layer, each value as its (hi, lo) f16 pair: plane hi [nkv][cap][hd]
    // then plane lo [nkv][cap][hd] (the 4 bytes of an f32 a value)
    std::vector<__half*> k, v;
    __half** k_dev = nullptr;  // device arrays of the per-layer pointers
    __half** v_dev = nullptr;
    // per layer, the tensor maps of its key and value stores for the tcgen05
    // attention (device memory, 2 x 128 bytes a layer; null when the driver
    // could not encode them: that attention is then not used)
    void* maps_dev = nullptr;
    // per layer: context rows no block row of the layer can see any more
    // (its window), dropped for good; the layer reads from first + dropped
    std::vector<int64_t> dropped;
    // queued tap rows (positions first + len ..): rows [pend_off, pend_off +
    // pending) of a device buffer of pend_cap rows
    float* pend = nullptr;
    int64_t pend_cap = 0, pend_off = 0, pending = 0;
};

namespace {

int set_err(dflash_model* m, int code, const std::string& msg) {
    if (m)
        m->err = msg;
    else
        g_init_error = msg;
    return code;
}

int cuda_fail(dflash_model* m, int e, const char* what) {
    std::string msg = std::string(what) + ": " + cudaGetErrorString((cudaError_t)e);
    if (m) m->poisoned = true;
    return set_err(m, (e == cudaErrorMemoryAllocation) ? DFLASH_ENOMEM : DFLASH_ECUDA, msg);
}

#define CK(m, expr)                                                      \
    do {                                                                 \
        int e__ = (int)(expr);                                           \
        if (e__ != 0) return cuda_fail((m), e__, #expr);                 \
    } while (0)

cudaEvent_t pool_event(dflash_model* m) {
    if (!m->ev_pool.empty()) {
        cudaEvent_t e = m->ev_pool.back();
        m->ev_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
}

// Launch `expr` (a launcher returning a cudaError_t as int) that starts
// `nk` kernels moving `bytes` algorithmic bytes; with profiling on, bracket
// it with a pair of events on `st`.
#define KL(m, name, nk, bytes, st, expr)                                       \
    do {                                                                       \
        cudaEvent_t e0__ = nullptr;                                            \
        if ((m)->profiling) {                                                  \
            e0__ = pool_event(m);                                              \
            cudaEventRecord(e0__, (st));                                       \
        }                                                                      \
        int e__ = (int)(expr);                                                 \
        if (e__ != 0) return cuda_fail((m), e__, #expr);                       \
        (m)->launches += (nk);                                                 \
        if ((m)->profiling) {                                                  \
            cudaEvent_t e1__ = pool_event(m);                                  \
            cudaEventRecord(e1__, (st));                                       \
            (m)->prof_open.push_back({(name), e0__, e1__, (double)(bytes), (nk)}); \
        }                                                                      \
    } while (0)

template <class T>
int dalloc(dflash_model* m, T** p, size_t count) {
    void* q = nullptr;
    cudaError_t e = cudaMalloc(&q, std::max<size_t>(count * sizeof(T), 16));
    if (e != cudaSuccess) return (int)e;
    m->owned.push_back(q);
    *p = static_cast<T*>(q);
    return 0;
}

int ensure(DevBuf& b, size_t bytes, bool* grown = nullptr) {
    if (b.bytes >= bytes) return 0;
    if (grown) *grown = true;
    if (b.p) cudaFree(b.p);
    b.p = nullptr;
    b.bytes = 0;
    cudaError_t e = cudaMalloc(&b.p, std::max<size_t>(bytes, 256));
    if (e != cudaSuccess) return (int)e;
    b.bytes = std::max<size_t>(bytes, 256);
    return 0;
}

void free_buf(DevBuf& b) {
    if (b.p) cudaFree(b.p);
    b.p = nullptr;
    b.bytes = 0;
}

void clear_graphs(dflash_model* m) {
    for (auto& e : m->graphs) cudaGraphExecDestroy(e.exec);
    m->graphs.clear();
}

// A model's scratch buffer of at least `bytes`; growing it drops the
// captured graphs (they hold the old address).
int ensure_m(dflash_model* m, DevBuf& b, size_t bytes) {
    bool grown = false;
    int e = ensure(b, bytes, &grown);
    if (grown) clear_graphs(m);
    return e;
}

template <class T>
T* P(const DevBuf& b) {
    return static_cast<T*>(b.p);
}

// The context view of layer `l` of sequence `q` for a block anchored at
// `anchor`: positions [lo, hi) with hi = min(anchor, first + len) and lo the
// first held position (first + the rows the layer dropped), raised under a
// window w > 0 to anchor + 1 - w, the first position block row 0 sees; row i
// sees from anchor + i + 1 - w on (page "cortiq-engine 0.8.71 —
// src/dflash.rs", `Drafter::block`).
AttnSeq layer_view(const dflash_model* m, const dflash_seq* q, int l, int64_t anchor) {
    const int64_t w = m->win[l];
    const int64_t base = q->first + q->dropped[l];
    const int64_t hi = std::max(std::min(anchor, q->first + q->len), base);
    const int64_t lo = w > 0 ? std::min(std::max(anchor + 1 - w, base), hi) : base;
    AttnSeq a{};
    a.kc = q->k[l];
    a.vc = q->v[l];
    a.cap = q->cap;
    a.lo = lo - q->first;
    a.n = (int)(hi - lo);
    a.cut = w > 0 ? (int)std::max<int64_t>(anchor + 1 - w - lo, kNoCut) : kNoCut;
    a.maps = q->maps_dev ? static_cast<const unsigned char*>(q->maps_dev) + (size_t)l * 256 : nullptr;
    return a;
}

std::string geometry_problem(const dflash_geometry& g) {
    char buf[256];
    if (g.layers < 1) return "layers < 1";
    if (g.block < 2) return "block < 2";
    if (g.n_taps < 1) return "n_taps < 1";
    if (g.kv_heads < 1 || g.heads < 1 || g.heads % g.kv_heads) return "heads must be a multiple of kv_heads >= 1";
    if (g.head_dim != 64 && g.head_dim != 128) return "head_dim must be 64 or 128";
    if (g.hidden < 64 || g.hidden % 64) return "hidden must be a positive multiple of 64";
    if (g.intermediate < 64 || g.intermediate % 64) return "intermediate must be a positive multiple of 64";
    if (g.vocab < 1) return "vocab < 1";
    if (g.mask_token < 0 || g.mask_token >= g.vocab) return "mask_token outside [0, vocab)";
    if (g.window < 0) return "window < 0";
    if (g.conv_kernel < 0 || g.conv_kernel > 64) return "conv_kernel outside [0, 64]";
    if (g.selector_rank < 0 || g.selector_rank > 4096) return "selector_rank outside [0, 4096]";
    if (g.selector_rank > 0 && (g.selector_top < 1 || g.selector_top > 32 || g.selector_top > g.vocab))
        return "selector_top outside [1, min(32, vocab)]";
    if (g.conv_kernel > 0 && (g.conv_group < 4 || g.conv_group % 4 || g.hidden % g.conv_group))
        return "conv_group must be a multiple of 4 dividing hidden";
    if (g.windows)
        for (int l = 0; l < g.layers; ++l)
            if (g.windows[l] < 0) return "windows[" + std::to_string(l) + "] < 0";
    if (!(g.eps > 0.f)) return "eps must be > 0";
    if (!(g.rope_theta > 0.0)) return "rope_theta must be > 0";
    if (g.quant != DFLASH_QUANT_F32 && g.quant != DFLASH_QUANT_Q4G32) return "unknown quant";
    if ((int64_t)g.vocab * g.hidden > ((int64_t)1 << 40)) {
        snprintf(buf, sizeof buf, "vocab * hidden too large");
        return buf;
    }
    return "";
}

// A weight tensor as a device pointer: `src` itself when the caller's
// weights are on the device, else copied into `stage`.
int to_device(dflash_model* m, const float* src, size_t count, bool on_device, float* stage, const float** out) {
    if (on_device) {
        *out = src;
        return 0;
    }
    cudaError_t e = cudaMemcpy(stage, src, count * sizeof(float), cudaMemcpyHostToDevice);
    *out = stage;
    return (int)e;
}

int copy_f32(dflash_model* m, float* dst, const float* src, size_t count, bool on_device) {
    return (int)cudaMemcpy(dst, src, count * sizeof(float), on_device ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice);
}

MatView mat_view(const dflash_model* m, int id) {
    const dflash_geometry& g = m->g;
    MatView v{nullptr, nullptr, 0, 0, 0, Q4Layout{}};
    if (id == DFLASH_MAT_FC) return MatView{m->fc_p, m->fc_f, 0, g.hidden, m->tap_w, m->L_fc};
    if (id == DFLASH_MAT_HEAD) return MatView{nullptr, m->head_f, 0, g.vocab, g.hidden, Q4Layout{}};
    int rel = id - 2;
    if (rel < 0 || rel >= 7 * g.layers) return v;
    const Layer& L = m->layers[rel / 7];
    const size_t H = g.hidden, I = g.intermediate;
    switch (rel % 7) {
        case DFLASH_Q: return MatView{L.qkv_p, L.qkv_f, 0, m->qd, g.hidden, m->L_qkv};
        case DFLASH_K: return MatView{L.qkv_p, L.qkv_f ? L.qkv_f + (size_t)m->qd * H : nullptr, m->qd / 16, m->kd, g.hidden, m->L_qkv};
        case DFLASH_V: return MatView{L.qkv_p, L.qkv_f ? L.qkv_f + (size_t)(m->qd + m->kd) * H : nullptr, (m->qd + m->kd) / 16, m->kd, g.hidden, m->L_qkv};
        case DFLASH_O: return MatView{L.o_p, L.o_f, 0, g.hidden, m->qd, m->L_o};
        case DFLASH_GATE: return MatView{L.gu_p, L.gu_f, 0, g.intermediate, g.hidden, m->L_gu};
        case DFLASH_UP: return MatView{L.gu_p, L.gu_f ? L.gu_f + I * H : nullptr, g.intermediate / 16, g.intermediate, g.hidden, m->L_gu};
        case DFLASH_DOWN: return MatView{L.down_p, L.down_f, 0, g.hidden, g.intermediate, m->L_down};
    }
    return v;
}

// A kernel gave up a bounded wait (its data never arrived): the results of
// the call are incomplete and the model is not trusted any more.
int device_wait_expired(dflash_model* m) {
    m->poisoned = true;
    return set_err(m, DFLASH_ECUDA, "a kernel's bounded wait for its data expired; results are incomplete");
}

int check_model(dflash_model* m) {
    if (!m) return DFLASH_EINVAL;
    if (m->poisoned) return set_err(m, DFLASH_ECUDA, "model poisoned by an earlier CUDA error");
    cudaError_t e = cudaSetDevice(m->device);
    if (e != cudaSuccess) return cuda_fail(m, (int)e, "cudaSetDevice");
    return 0;
}

int build_model(dflash_model* m, const dflash_weights* w, bool on_dev, cudaStream_t st) {
    const dflash_geometry& g = m->g;
    const int H = g.hidden, I = g.intermediate, L = g.layers, hd = g.head_dim;
    m->qd = g.heads * hd;
    m->kd = g.kv_heads * hd;
    m->qkv_w = m->qd + 2 * m->kd;
    m->tap_w = g.n_taps * H;
    m->kvctx_w = L * 2 * m->kd;
    m->L_fc = make_layout(H, m->tap_w);
    m->L_kvctx = make_layout(m->kvctx_w, H);
    m->L_qkv = make_layout(m->qkv_w, H);
    m->L_o = make_layout(H, m->qd);
    m->L_gu = make_layout(2 * I, H);
    m->L_down = make_layout(H, I);
    CK(m, dalloc(m, &m->err_dev, 1));
    CK(m, cudaMemset(m->err_dev, 0, sizeof(int)));
    CK(m, cudaEventCreateWithFlags(&m->copy_ev, cudaEventDisableTiming));
    {
        std::vector<int> rot(g.layers);
        for (int l = 0; l < g.layers; ++l) rot[l] = m->norope[l] ? 0 : 1;
        CK(m, dalloc(m, &m->rot_dev, (size_t)g.layers));
        CK(m, cudaMemcpy(m->rot_dev, rot.data(), rot.size() * sizeof(int), cudaMemcpyHostToDevice));
    }
    CK(m, cudaMallocHost(&m->err_host, sizeof(int)));
    *m->err_host = 0;
    const bool quant = g.quant == DFLASH_QUANT_Q4G32;

    // staging buffer for host weights: the largest tensor
    size_t biggest = std::max({(size_t)H * m->tap_w, (size_t)g.vocab * H, (size_t)I * H, (size_t)m->qd * H});
    float* stage = nullptr;
    if (!on_dev) CK(m, dalloc(m, &stage, biggest));
    __half* sc_scratch = nullptr;
    if (quant) {
        size_t most = std::max({(size_t)H * (m->tap_w / 32), (size_t)I * (H / 32), (size_t)H * (I / 32),
                                (size_t)(m->qd + 16) * (H / 32), (size_t)H * (m->qd / 32)});
        CK(m, dalloc(m, &sc_scratch, most + 64));
    }

    // small f32 vectors
    CK(m, dalloc(m, &m->hidden_norm, H));
    CK(m, copy_f32(m, m->hidden_norm, w->hidden_norm, H, on_dev));
    CK(m, dalloc(m, &m->norm, H));
    CK(m, copy_f32(m, m->norm, w->norm, H, on_dev));
    CK(m, dalloc(m, &m->embed, (size_t)g.vocab * H));
    CK(m, copy_f32(m, m->embed, w->embed, (size_t)g.vocab * H, on_dev));
    std::vector<float> invf(hd / 2);
    for (int i = 0; i < hd / 2; ++i) invf[i] = (float)std::pow(g.rope_theta, -(2.0 * i) / (double)hd);
    CK(m, dalloc(m, &m->inv_freq, hd / 2));
    CK(m, cudaMemcpy(m->inv_freq, invf.data(), invf.size() * sizeof(float), cudaMemcpyHostToDevice));

    const float* d = nullptr;
    auto pack = [&](const float* src, int N, int K, uint8_t* dst, int tile0, Q4Layout Lo) -> int {
        int e = to_device(m, src, (size_t)N * K, on_dev, stage, &d);
        if (e) return e;
        e = q4_quantize_pack(d, N, K, dst, Lo, tile0, sc_scratch, st);
        if (e) return e;
        return (int)cudaStreamSynchronize(st);  // the stage is reused by the next tensor
    };
    auto q4_bytes = [](Q4Layout Lo) { return (size_t)Lo.ngroups * Lo.ksteps * 4 * kQ4Chunk; };

    // fc and the all-layer Wk||Wv of the context projection
    if (quant) {
        CK(m, dalloc(m, &m->fc_p, q4_bytes(m->L_fc)));
        CK(m, pack(w->fc, H, m->tap_w, m->fc_p, 0, m->L_fc));
        CK(m, dalloc(m, &m->kvctx_p, q4_bytes(m->L_kvctx)));
        for (int l = 0; l < L; ++l) {
            CK(m, pack(w->k[l], m->kd, H, m->kvctx_p, (l * 2 * m->kd) / 16, m->L_kvctx));
            CK(m, pack(w->v[l], m->kd, H, m->kvctx_p, (l * 2 * m->kd + m->kd) / 16, m->L_kvctx));
        }
    } else {
        CK(m, dalloc(m, &m->fc_f, (size_t)H * m->tap_w));
        CK(m, copy_f32(m, m->fc_f, w->fc, (size_t)H * m->tap_w, on_dev));
        CK(m, dalloc(m, &m->kvctx_f, (size_t)m->kvctx_w * H));
        for (int l = 0; l < L; ++l) {
            CK(m, copy_f32(m, m->kvctx_f + (size_t)l * 2 * m->kd * H, w->k[l], (size_t)m->kd * H, on_dev));
            CK(m, copy_f32(m, m->kvctx_f + (size_t)(l * 2 + 1) * m->kd * H, w->v[l], (size_t)m->kd * H, on_dev));
        }
    }
    // head
    if (quant) {
        const int vpad = (g.vocab + 63) / 64 * 64;
        CK(m, dalloc(m, &m->head_p, (size_t)vpad * H));
        CK(m, dalloc(m, &m->head_scale, vpad));
        CK(m, to_device(m, w->head, (size_t)g.vocab * H, on_dev, stage, &d));
        CK(m, i8_rows_quantize_pack(d, g.vocab, H, vpad, H / kI8KStep, m->head_p, m->head_scale, st));
        CK(m, cudaStreamSynchronize(st));
    } else {
        CK(m, dalloc(m, &m->head_f, (size_t)g.vocab * H));
        CK(m, copy_f32(m, m->head_f, w->head, (size_t)g.vocab * H, on_dev));
    }
    if (g.selector_rank > 0) {
        const size_t rk = (size_t)g.selector_rank, nb = (size_t)g.vocab * rk;
        CK(m, dalloc(m, &m->sel, rk * H));
        CK(m, copy_f32(m, m->sel, w->selector_projection, rk * H, on_dev));
        const cudaMemcpyKind kind = on_dev ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice;
        CK(m, dalloc(m, &m->book_p, nb));
        CK(m, cudaMemcpy(m->book_p, w->predecessor_codebook, nb * sizeof(__half), kind));
        CK(m, dalloc(m, &m->book_c, nb));
        CK(m, cudaMemcpy(m->book_c, w->successor_codebook, nb * sizeof(__half), kind));
    }
    // layers
    m->layers.resize(L);
    std::vector<const float*> knorm_ptrs(L);
    for (int l = 0; l < L; ++l) {
        Layer& Ly = m->layers[l];
        CK(m, dalloc(m, &Ly.in_norm, H));
        CK(m, copy_f32(m, Ly.in_norm, w->in_norm[l], H, on_dev));
        CK(m, dalloc(m, &Ly.post_norm, H));
        CK(m, copy_f32(m, Ly.post_norm, w->post_norm[l], H, on_dev));
        CK(m, dalloc(m, &Ly.q_norm, hd));
        CK(m, copy_f32(m, Ly.q_norm, w->q_norm[l], hd, on_dev));
        CK(m, dalloc(m, &Ly.k_norm, hd));
        CK(m, copy_f32(m, Ly.k_norm, w->k_norm[l], hd, on_dev));
        knorm_ptrs[l] = Ly.k_norm;
        if (g.conv_kernel > 0) {
            const size_t nb = (size_t)2 * g.conv_kernel * H, np = nb / g.conv_group * H;
            CK(m, dalloc(m, &Ly.a_base, nb));
            CK(m, copy_f32(m, Ly.a_base, w->attn_conv_base[l], nb, on_dev));
            CK(m, dalloc(m, &Ly.a_proj, np));
            CK(m, copy_f32(m, Ly.a_proj, w->attn_conv_proj[l], np, on_dev));
            CK(m, dalloc(m, &Ly.m_base, nb));
            CK(m, copy_f32(m, Ly.m_base, w->mlp_conv_base[l], nb, on_dev));
            CK(m, dalloc(m, &Ly.m_proj, np));
            CK(m, copy_f32(m, Ly.m_proj, w->mlp_conv_proj[l], np, on_dev));
        }
        if (quant) {
            CK(m, dalloc(m, &Ly.qkv_p, q4_bytes(m->L_qkv)));
            CK(m, pack(w->q[l], m->qd, H, Ly.qkv_p, 0, m->L_qkv));
            CK(m, pack(w->k[l], m->kd, H, Ly.qkv_p, m->qd / 16, m->L_qkv));
            CK(m, pack(w->v[l], m->kd, H, Ly.qkv_p, (m->qd + m->kd) / 16, m->L_qkv));
            CK(m, dalloc(m, &Ly.o_p, q4_bytes(m->L_o)));
            CK(m, pack(w->o[l], H, m->qd, Ly.o_p, 0, m->L_o));
            CK(m, dalloc(m, &Ly.gu_p, q4_bytes(m->L_gu)));
            CK(m, pack(w->gate[l], I, H, Ly.gu_p, 0, m->L_gu));
            CK(m, pack(w->up[l], I, H, Ly.gu_p, I / 16, m->L_gu));
            CK(m, dalloc(m, &Ly.down_p, q4_bytes(m->L_down)));
            CK(m, pack(w->down[l], H, I, Ly.down_p, 0, m->L_down));
        } else {
            CK(m, dalloc(m, &Ly.qkv_f, (size_t)m->qkv_w * H));
            CK(m, copy_f32(m, Ly.qkv_f, w->q[l], (size_t)m->qd * H, on_dev));
            CK(m, copy_f32(m, Ly.qkv_f + (size_t)m->qd * H, w->k[l], (size_t)m->kd * H, on_dev));
            CK(m, copy_f32(m, Ly.qkv_f + (size_t)(m->qd + m->kd) * H, w->v[l], (size_t)m->kd * H, on_dev));
            CK(m, dalloc(m, &Ly.o_f, (size_t)H * m->qd));
            CK(m, copy_f32(m, Ly.o_f, w->o[l], (size_t)H * m->qd, on_dev));
            CK(m, dalloc(m, &Ly.gu_f, (size_t)2 * I * H));
            CK(m, copy_f32(m, Ly.gu_f, w->gate[l], (size_t)I * H, on_dev));
            CK(m, copy_f32(m, Ly.gu_f + (size_t)I * H, w->up[l], (size_t)I * H, on_dev));
            CK(m, dalloc(m, &Ly.down_f, (size_t)H * I));
            CK(m, copy_f32(m, Ly.down_f, w->down[l], (size_t)H * I, on_dev));
        }
    }
    // The attention's accumulate-mode reference per layer.  After the per-head
    // RMSNorm a query has |q| <= sqrt(hd) * max|q_norm| (the normed row's
    // squares sum to hd * ms / (ms + eps) < hd), likewise a key, so a score in
    // the kernel's log2 domain obeys |s| <= sqrt(hd) * max|gq| * max|gk| *
    // log2(e) (the 1/sqrt(hd) scale taken in).  Rescaled partial sums then
    // stay within [2^(-2 ref), 1]: usable while 2 ref + 2 < 126.
    m->attn_ref.assign(L, NAN);
    for (int l = 0; l < L; ++l) {
        std::vector<float> gq(hd), gk(hd);
        CK(m, cudaMemcpy(gq.data(), m->layers[l].q_norm, hd * sizeof(float), cudaMemcpyDeviceToHost));
        CK(m, cudaMemcpy(gk.data(), m->layers[l].k_norm, hd * sizeof(float), cudaMemcpyDeviceToHost));
        double aq = 0, ak = 0;
        for (int i = 0; i < hd; ++i) {
            aq = std::max(aq, (double)std::fabs(gq[i]));
            ak = std::max(ak, (double)std::fabs(gk[i]));
        }
        const double ref = std::sqrt((double)hd) * aq * ak * 1.4426950408889634 * (1.0 + 1e-3) + 0.5;
        if (std::isfinite(ref) && 2 * ref + 2 < 126) m->attn_ref[l] = (float)ref;
    }
    CK(m, dalloc(m, &m->k_norm_dev, L));
    CK(m, cudaMemcpy(m->k_norm_dev, knorm_ptrs.data(), L * sizeof(float*), cudaMemcpyHostToDevice));
    CK(m, cudaStreamSynchronize(st));
    // the staging buffers are not needed after init
    auto drop = [&](void* p) {
        if (!p) return;
        cudaFree(p);
        m->owned.erase(std::remove(m->owned.begin(), m->owned.end(), p), m->owned.end());
    };
    drop(stage);
    drop(sc_scratch);
    return DFLASH_OK;
}

bool weights_complete(const dflash_weights* w, int L, bool conv, bool sel) {
    if (!w->fc || !w->hidden_norm || !w->norm || !w->embed || !w->head) return false;
    const float* const* per[] = {w->in_norm, w->post_norm, w->q_norm, w->k_norm, w->q, w->k,
                                 w->v,       w->o,         w->gate,   w->up,     w->down};
    for (auto a : per) {
        if (!a) return false;
        for (int l = 0; l < L; ++l)
            if (!a[l]) return false;
    }
    if (sel && (!w->selector_projection || !w->predecessor_codebook || !w->successor_codebook)) return false;
    if (conv) {
        const float* const* cv[] = {w->attn_conv_base, w->attn_conv_proj, w->mlp_conv_base, w->mlp_conv_proj};
        for (auto a : cv) {
            if (!a) return false;
            for (int l = 0; l < L; ++l)
                if (!a[l]) return false;
        }
    }
    return true;
}

// Apply one matrix (4-bit or f32) to activations: quantised formats take the
// int8 codes in m->xq / m->xs, the f32 format the f32 rows `xf`.
#define APPLY(expr)                 \
    do {                            \
        int rc__ = (expr);          \
        if (rc__) return rc__;      \
    } while (0)

double q4_bytes_of(int N, int K, int T, bool accumulate) {
    // 4-bit weights (0.5 B a weight, 2 B per 32) + int8 activations + f32 outputs
    return (double)N * K * 0.5 + (double)N * (K / 32) * 2 + (double)T * (K + 4) + (double)T * N * 4 * (accumulate ? 2 : 1);
}
double f32_bytes_of(int N, int K, int T, bool accumulate) {
    return (double)N * K * 4 + (double)T * K * 4 + (double)T * N * 4 * (accumulate ? 2 : 1);
}

// The dense f16 copies of every 4-bit matrix and of the head, for the
// tensor-core kernels of the many-row path (about 5.6 GB at the Qwen3-8B
// shapes), built once on the first call that needs them -- never inside a
// graph capture (callers run it before any).
int ensure_dense(dflash_model* m, cudaStream_t st) {
    if (m->dense_ready || !m->use_tc || !m->use_dense || m->g.quant != DFLASH_QUANT_Q4G32) return 0;
    const dflash_geometry& g = m->g;
    const int H = g.hidden, I = g.intermediate;
    struct Src {
        const uint8_t* p;
        Q4Layout L;
        int N, K;
    };
    std::vector<Src> srcs = {{m->fc_p, m->L_fc, H, m->tap_w}, {m->kvctx_p, m->L_kvctx, m->kvctx_w, H}};
    for (const Layer& Ly : m->layers) {
        srcs.push_back({Ly.qkv_p, m->L_qkv, m->qkv_w, H});
        srcs.push_back({Ly.o_p, m->L_o, H, m->qd});
        srcs.push_back({Ly.gu_p, m->L_gu, 2 * I, H});
        srcs.push_back({Ly.down_p, m->L_down, H, I});
    }
    size_t most = (size_t)g.vocab * H;
    for (const Src& q : srcs) most = std::max(most, (size_t)q.N * q.K);
    int8_t* codes = nullptr;
    uint16_t* scales = nullptr;
    CK(m, cudaMalloc(&codes, most));
    cudaError_t e = cudaMalloc(&scales, most / 32 * sizeof(uint16_t));
    int rc = 0;
    if (e != cudaSuccess) rc = (int)e;
    std::vector<dflash_model::DenseMat> made;
    for (const Src& q : srcs) {
        if (rc) break;
        dflash_model::DenseMat d{q.p, q.N, q.K, nullptr, nullptr};
        rc = dalloc(m, &d.hi, (size_t)q.N * q.K);
        if (!rc) rc = dalloc(m, &d.lo, (size_t)q.N * q.K);
        if (!rc) rc = q4_unpack(q.p, q.L, 0, q.N, q.K, codes, scales, st);
        if (!rc) rc = dequant_hilo(codes, scales, q.N, q.K, d.hi, d.lo, st);
        if (!rc) made.push_back(d);
        if (!rc) rc = (int)cudaStreamSynchronize(st);  // the temporaries are reused
    }
    __half* h16 = nullptr;
    int* hn2 = nullptr;
    if (!rc) rc = dalloc(m, &h16, (size_t)g.vocab * H);
    if (!rc) rc = dalloc(m, &hn2, (size_t)g.vocab);
    if (!rc) rc = i8_unpack(m->head_p, g.vocab, H, H / kI8KStep, codes, st);
    if (!rc) rc = codes_to_f16(codes, H, g.vocab, H, h16, hn2, m->num_sms, st);
    std::vector<int> hn2_host(g.vocab);
    if (!rc) rc = (int)cudaMemcpyAsync(hn2_host.data(), hn2, (size_t)g.vocab * sizeof(int), cudaMemcpyDeviceToHost, st);
    if (!rc) rc = (int)cudaStreamSynchronize(st);
    unsigned long long hn2_max = 0;
    for (int v : hn2_host) hn2_max = std::max(hn2_max, (unsigned long long)(uint32_t)v);
    cudaFree(codes);
    cudaFree(scales);
    CK(m, (cudaError_t)rc);
    m->dense = made;
    m->head16 = h16;
    m->head_norm2 = hn2;
    m->head_norm2_max = hn2_max;
    m->dense_ready = true;
    return 0;
}

// The dense copy of a packed 4-bit matrix's rows [row0, row0 + N), or null.
bool dense_of(const dflash_model* m, const uint8_t* packed, int row0, int N, int K, const __half** hi,
              const __half** lo) {
    if (!m->dense_ready || !m->use_dense) return false;
    for (const auto& d : m->dense)
        if (d.packed == packed && d.K == K && row0 + N <= d.N) {
            *hi = d.hi + (size_t)row0 * K;
            *lo = d.lo + (size_t)row0 * K;
            return true;
        }
    return false;
}

// A 4-bit matmul on int8 codes: the streaming kernel for up to 16 rows (it
// ADDS into y, which an earlier kernel cleared or which holds the residual),
// the general one beyond.
int q4_mm(dflash_model* m, const uint8_t* packed, Q4Layout L, int tile0, int N, int K, QAct x, int T, float* y,
          int ldy, bool accumulate, cudaStream_t st, bool x16_ready = false) {
    if (T <= 16) {
        KL(m, "q4_stream", 1, q4_bytes_of(N, K, T, true), st,
           q4_stream(packed, L, tile0, N, x, T, y, ldy, m->num_sms, m->err_dev, st));
    } else if (m->use_tc && q4_tc_supported(L, tile0, N, K, x) && ldy % 4 == 0 &&
               (reinterpret_cast<uintptr_t>(y) & 15) == 0 && m->x16.bytes >= (size_t)T * K * sizeof(__half)) {
        __half* x16 = P<__half>(m->x16);
        // (x16_ready: the kernel that quantised x wrote these f16 codes already)
        if (!x16_ready)
            KL(m, "act_f16", 1, (double)T * K * 3, st,
               codes_to_f16(x.codes, x.ld, T, K, x16, nullptr, m->num_sms, st));
        const __half *hi = nullptr, *lo = nullptr;
        if (dense_of(m, packed, tile0 * 16, N, K, &hi, &lo)) {
            // dense weight bytes: 4 a weight
            KL(m, "q4_tc", 1, (double)N * K * 4 + (double)T * K * 2 + (double)T * N * 4 * (accumulate ? 2 : 1), st,
               q4_tc_dense(hi, lo, N, K, x, x16, T, y, ldy, accumulate, m->err_dev, st));
        } else {
            KL(m, "q4_tc", 1, q4_bytes_of(N, K, T, accumulate), st,
               q4_tc(packed, L, tile0, N, x, x16, T, y, ldy, accumulate, m->num_sms, m->err_dev, st));
        }
    } else {
        KL(m, "q4_gemm", 1, q4_bytes_of(N, K, T, accumulate), st,
           q4_gemm(packed, L, tile0, N, x, T, y, ldy, accumulate, m->num_sms, st));
    }
    return 0;
}

// The head over D rows: the streaming kernel (one pass over the head per 16
// rows) for a single block, the tcgen05 kernel for many rows.
int run_head(dflash_model* m, QAct xh, int D, float* logit_out, unsigned long long* keys, double hb, cudaStream_t st) {
    const dflash_geometry& g = m->g;
    const int H = g.hidden;
    if (D > 16 && m->use_tc && head_tc_supported(H / kI8KStep, xh) &&
        m->x16.bytes >= (size_t)D * H * sizeof(__half)) {
        __half* x16 = P<__half>(m->x16);
        // the rows' squared code norms sit after their f16 codes
        int* xn2 = reinterpret_cast<int*>(x16 + (size_t)D * H);
        if (m->dense_ready && m->use_dense && m->head16 && m->x16.bytes >= (size_t)D * (H * sizeof(__half) + sizeof(int))) {
            KL(m, "act_f16", 1, (double)D * H * 3 + (double)D * 4, st,
               codes_to_f16(xh.codes, xh.ld, D, H, x16, xn2, m->num_sms, st));
            KL(m, "head_tc", 1, hb + (double)g.vocab * H + (double)g.vocab * 4, st,
               head_tc_dense(m->head16, m->head_norm2, m->head_scale, g.vocab, H, xh, x16, xn2, D, logit_out, g.vocab,
                             keys, m->head_bound, m->head_norm2_max, m->err_dev, st));
        } else {
            KL(m, "act_f16", 1, (double)D * H * 3, st,
               codes_to_f16(xh.codes, xh.ld, D, H, x16, nullptr, m->num_sms, st));
            KL(m, "head_tc", 1, hb, st,
               head_tc(m->head_p, m->head_scale, g.vocab, H / kI8KStep, xh, x16, D, logit_out, g.vocab, keys,
                       m->err_dev, st));
        }
    } else {
        KL(m, "head_stream", 1, hb, st,
           head_stream(m->head_p, m->head_scale, g.vocab, H / kI8KStep, xh, D, logit_out, g.vocab, keys, m->num_sms,
                       m->err_dev, st));
    }
    return DFLASH_OK;
}

// The candidate selector after the head: the rows after the last norm (f32),
// their projection S . hn, each row's top candidates from its logits, then
// the choices row by row per sequence (into tok_out).
int run_selector(dflash_model* m, cudaStream_t st, const float* h, RowMap drafts, int D, int n_seqs, int B,
                 const float* logits, const uint32_t* anchors, uint32_t* tok_out) {
    const dflash_geometry& g = m->g;
    const int H = g.hidden, rank = g.selector_rank, top = g.selector_top;
    float* hn = P<float>(m->hn);
    float* hp = P<float>(m->hp);
    unsigned long long* cand = P<unsigned long long>(m->cand);
    KL(m, "rms_f32", 1, (double)D * H * 8, st,
       rms_rows(h, H, drafts, D, H, m->norm, g.eps, hn, H, nullptr, nullptr, 0, st));
    KL(m, "linear_f32", 1, f32_bytes_of(rank, H, D, false), st, linear_f32(m->sel, rank, H, hn, H, D, hp, rank, false, st));
    unsigned long long* parts = cand + (size_t)D * top;  // the first phase's keys, after the candidates
    KL(m, "topk_rows", 2, (double)D * g.vocab * 4, st, topk_rows(logits, g.vocab, g.vocab, D, top, parts, cand, st));
    KL(m, "select", 1, (double)D * top * rank * 4, st,
       select_tokens(cand, top, hp, rank, m->book_p, m->book_c, g.vocab, anchors, n_seqs, B - 1, tok_out,
                     P<uint32_t>(m->plain), st));
    return DFLASH_OK;
}

// Apply one matrix to the block's rows.  Quantised format: the int8 codes in
// m->xq / m->xs.  Up to 16 rows take the streaming kernel, which ADDS into y:
// a fresh output must have been cleared by an earlier kernel (the zeroing
// side duty of the row kernel before it).  f32 format: the f32 rows `xf`.
int apply(dflash_model* m, const uint8_t* packed, const float* f32w, Q4Layout L, int tile0, int N, int K,
          const float* xf, int ldxf, int T, float* y, int ldy, bool accumulate, int ldq, cudaStream_t st,
          bool x16_ready = false) {
    if (m->g.quant == DFLASH_QUANT_Q4G32) {
        QAct x{P<int8_t>(m->xq), P<float>(m->xs), ldq};
        return q4_mm(m, packed, L, tile0, N, K, x, T, y, ldy, accumulate, st, x16_ready);
    }
    KL(m, "linear_f32", 1, f32_bytes_of(N, K, T, accumulate), st,
       linear_f32(f32w, N, K, xf, ldxf, T, y, ldy, accumulate, st));
    return 0;
}

// A quantisation site just written: `rows` rows of int8 codes (as f16, row
// stride ld) and f32 scales on the device.  With tracing on, record the
// site's pre-quantisation values (`values_fn` writes them, f32 [rows][cols],
// into the device pointer it is given), its codes and scales; and if a
// forced decision is queued, replace the codes and scales with it.
template <class F>
int trace_site(dflash_model* m, cudaStream_t st, int rows, int cols, int8_t* codes, int ld, float* scales,
               F values_fn) {
    if (!m->tracing) return 0;
    CK(m, ensure_m(m, m->trace_buf, (size_t)rows * cols * sizeof(float)));
    CK(m, values_fn(P<float>(m->trace_buf)));
    dflash_model::Site site;
    site.rows = rows;
    site.cols = cols;
    site.values.resize((size_t)rows * cols);
    site.scales.resize(rows);
    std::vector<int8_t> hc((size_t)rows * ld);
    CK(m, cudaMemcpyAsync(site.values.data(), m->trace_buf.p, site.values.size() * sizeof(float),
                          cudaMemcpyDeviceToHost, st));
    CK(m, cudaMemcpyAsync(hc.data(), codes, hc.size(), cudaMemcpyDeviceToHost, st));
    CK(m, cudaMemcpyAsync(site.scales.data(), scales, rows * sizeof(float), cudaMemcpyDeviceToHost, st));
    CK(m, cudaStreamSynchronize(st));
    site.codes.resize((size_t)rows * cols);
    for (int r = 0; r < rows; ++r)
        for (int c = 0; c < cols; ++c) site.codes[(size_t)r * cols + c] = hc[(size_t)r * ld + c];
    m->trace.push_back(std::move(site));
    if (m->forced_next < m->forced.size()) {
        const dflash_model::Site& f = m->forced[m->forced_next++];
        if (f.rows != rows || f.cols != cols)
            return set_err(m, DFLASH_EINVAL, "forced site " + std::to_string(m->forced_next - 1) + " is " +
                                                 std::to_string(f.rows) + "x" + std::to_string(f.cols) + ", the site is " +
                                                 std::to_string(rows) + "x" + std::to_string(cols));
        for (int r = 0; r < rows; ++r)
            for (int c = 0; c < cols; ++c) hc[(size_t)r * ld + c] = f.codes[(size_t)r * cols + c];
        CK(m, cudaMemcpyAsync(codes, hc.data(), hc.size(), cudaMemcpyHostToDevice, st));
        CK(m, cudaMemcpyAsync(scales, f.scales.data(), rows * sizeof(float), cudaMemcpyHostToDevice, st));
        CK(m, cudaStreamSynchronize(st));
    }
    return 0;
}

#define TRACE(expr)                \
    do {                           \
        int rc__ = (expr);         \
        if (rc__) return rc__;     \
    } while (0)

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Run `enqueue(stream)` (a fixed kernel sequence) on `st`: replayed from a
// graph captured once per key, or directly when graphs are off (profiling,
// tracing, or a stream capture of the caller's own in progress).
template <class F>
int run_enqueue(dflash_model* m, const std::vector<int64_t>& key, cudaStream_t st, F enqueue) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (!m->use_graphs || m->profiling || m->tracing || cudaStreamIsCapturing(st, &cs) != cudaSuccess ||
        cs != cudaStreamCaptureStatusNone)
        return enqueue(st);
    for (auto& e : m->graphs)
        if (e.key == key) {
            CK(m, cudaGraphLaunch(e.exec, st));
            m->launches += e.kernels;
            return DFLASH_OK;
        }
    if (!m->cap_stream) CK(m, cudaStreamCreateWithFlags(&m->cap_stream, cudaStreamNonBlocking));
    const int64_t before = m->launches;
    CK(m, cudaStreamBeginCapture(m->cap_stream, cudaStreamCaptureModeThreadLocal));
    // a graph of its own runs after all earlier work on the stream, whatever
    // its kernels' programmatic dependencies inside it
    m->own_capture = true;
    int rc = enqueue(m->cap_stream);
    m->own_capture = false;
    cudaGraph_t graph = nullptr;
    cudaError_t e2 = cudaStreamEndCapture(m->cap_stream, &graph);
    const int64_t kernels = m->launches - before;
    m->launches = before;
    if (rc != DFLASH_OK) {
        if (graph) cudaGraphDestroy(graph);
        return rc;
    }
    CK(m, e2);
    cudaGraphExec_t exec = nullptr;
    cudaError_t e3 = cudaGraphInstantiate(&exec, graph, 0);
    cudaGraphDestroy(graph);
    CK(m, e3);
    if (m->graphs.size() >= 16) {
        cudaGraphExecDestroy(m->graphs.front().exec);
        m->graphs.erase(m->graphs.begin());
    }
    m->graphs.push_back(dflash_model::GraphEntry{key, exec, kernels});
    CK(m, cudaGraphLaunch(exec, st));
    m->launches += kernels;
    return DFLASH_OK;
}

// Project `n` context rows (device taps) at positions pos0.. into the store.
// {pos0, idx0} of the rows are in m->a_pos (device).
int append_rows(dflash_model* m, dflash_seq* s, const float* taps_dev, int64_t n, cudaStream_t st) {
    const dflash_geometry& g = m->g;
    const int H = g.hidden;
    const bool quant = g.quant == DFLASH_QUANT_Q4G32;
    const int rows = (int)n;
    RowMap ident{1, 1, 0};
    float* t = P<float>(m->a_t);
    float* kv = P<float>(m->a_kv);
    if (quant) {
        // taps -> int8 rows (t cleared on the side); t = FC . Q(taps);
        // x = Q(rms(t, hidden_norm)) (kv cleared on the side); kv = [Wk;Wv]_all . x
        int8_t* codes = P<int8_t>(m->a_codes);
        float* sc = P<float>(m->a_scale);
        // (the side duties clear the streaming matvecs' outputs; the many-row
        // matmuls clear their own when they split K)
        const bool stream = rows <= 16;
        // (more rows: the f16 codes of the tcgen05 matmuls written beside the int8 ones)
        __half* a16 = (!stream && !m->tracing && m->use_tc) ? P<__half>(m->x16) : nullptr;
        KL(m, "rms_quant", 1, (double)rows * m->tap_w * 5, st,
           rms_rows(taps_dev, m->tap_w, ident, rows, m->tap_w, nullptr, g.eps, nullptr, 0, codes, sc, m->tap_w, st,
                    stream ? t : nullptr, stream ? (int64_t)rows * H : 0, nullptr, 0, a16));
        TRACE(trace_site(m, st, rows, m->tap_w, codes, m->tap_w, sc, [&](float* v) {
            return rms_rows(taps_dev, m->tap_w, ident, rows, m->tap_w, nullptr, g.eps, v, m->tap_w, nullptr, nullptr, 0, st);
        }));
        QAct xt{codes, sc, m->tap_w};
        APPLY(q4_mm(m, m->fc_p, m->L_fc, 0, H, m->tap_w, xt, rows, t, H, false, st, a16 != nullptr));
        KL(m, "rms_quant", 1, (double)rows * H * 5, st,
           rms_rows(t, H, ident, rows, H, m->hidden_norm, g.eps, nullptr, 0, codes, sc, H, st, stream ? kv : nullptr,
                    stream ? (int64_t)rows * m->kvctx_w : 0, nullptr, 0, a16));
        TRACE(trace_site(m, st, rows, H, codes, H, sc, [&](float* v) {
            return rms_rows(t, H, ident, rows, H, m->hidden_norm, g.eps, v, H, nullptr, nullptr, 0, st);
        }));
        QAct xh{codes, sc, H};
        APPLY(q4_mm(m, m->kvctx_p, m->L_kvctx, 0, m->kvctx_w, H, xh, rows, kv, m->kvctx_w, false, st, a16 != nullptr));
    } else {
        KL(m, "linear_f32", 1, f32_bytes_of(H, m->tap_w, rows, false), st,
           linear_f32(m->fc_f, H, m->tap_w, taps_dev, m->tap_w, rows, t, H, false, st));
        float* tn = P<float>(m->a_codes);  // reuse as f32 rows
        KL(m, "rms_f32", 1, (double)rows * H * 8, st,
           rms_rows(t, H, ident, rows, H, m->hidden_norm, g.eps, tn, H, nullptr, nullptr, 0, st));
        KL(m, "linear_f32", 1, f32_bytes_of(m->kvctx_w, H, rows, false), st,
           linear_f32(m->kvctx_f, m->kvctx_w, H, tn, H, rows, kv, m->kvctx_w, false, st));
    }
    KL(m, "kv_append", 1, (double)rows * m->kvctx_w * 8, st,
       kv_append(kv, rows, g.layers, g.kv_heads, g.head_dim, m->k_norm_dev, m->inv_freq, g.eps, P<int64_t>(m->a_pos),
                 s->k_dev, s->v_dev, s->cap, st, m->rot_dev));
    return DFLASH_OK;
}

int ensure_append_scratch(dflash_model* m, int64_t rows) {
    const bool quant = m->g.quant == DFLASH_QUANT_Q4G32;
    const size_t r = (size_t)rows;
    CK(m, ensure_m(m, m->a_taps, r * m->tap_w * sizeof(float)));
    CK(m, ensure_m(m, m->a_codes, quant ? r * m->tap_w : r * m->g.hidden * sizeof(float)));
    CK(m, ensure_m(m, m->a_scale, r * sizeof(float)));
    CK(m, ensure_m(m, m->a_t, r * m->g.hidden * sizeof(float)));
    CK(m, ensure_m(m, m->a_kv, r * m->kvctx_w * sizeof(float)));
    CK(m, ensure_m(m, m->a_pos, 2 * sizeof(int64_t)));
    if (quant && rows > 16)
        CK(m, ensure_m(m, m->x16, r * std::max(m->tap_w, m->g.hidden) * sizeof(__half)));
    return 0;
}

}  // namespace

// ============================================================================
extern "C" {

int dflash_init(const dflash_geometry* geom, const dflash_weights* weights, int weights_on_device, void* stream,
                dflash_model** out) {
    g_init_error.clear();
    if (!out) return set_err(nullptr, DFLASH_EINVAL, "out is NULL");
    *out = nullptr;
    if (!geom || !weights) return set_err(nullptr, DFLASH_EINVAL, "geometry or weights is NULL");
    std::string why = geometry_problem(*geom);
    if (!why.empty()) return set_err(nullptr, DFLASH_EGEOM, "unsupported geometry: " + why);
    if (!weights_complete(weights, geom->layers, geom->conv_kernel > 0, geom->selector_rank > 0))
        return set_err(nullptr, DFLASH_EINVAL, "a weight pointer is NULL");
    dflash_model* m = new (std::nothrow) dflash_model();
    if (!m) return set_err(nullptr, DFLASH_ENOMEM, "host allocation failed");
    m->g = *geom;
    // the per-layer lists as the model's own copies (what geometry_of returns)
    m->win.assign(geom->layers, geom->window);
    m->norope.assign(geom->layers, 0);
    for (int l = 0; l < geom->layers; ++l) {
        if (geom->windows) m->win[l] = geom->windows[l];
        if (geom->no_rope) m->norope[l] = geom->no_rope[l] != 0;
    }
    m->g.windows = geom->windows ? m->win.data() : nullptr;
    m->g.no_rope = geom->no_rope ? m->norope.data() : nullptr;
    cudaStream_t st = (cudaStream_t)stream;
    int rc = DFLASH_OK;
    cudaError_t e = cudaGetDevice(&m->device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&m->num_sms, cudaDevAttrMultiProcessorCount, m->device);
    if (e != cudaSuccess) {
        rc = cuda_fail(m, (int)e, "cudaGetDevice");
    } else {
        rc = build_model(m, weights, weights_on_device != 0, st);
    }
    if (rc != DFLASH_OK) {
        g_init_error = m->err;
        dflash_free(m);
        return rc;
    }
    *out = m;
    return DFLASH_OK;
}

void dflash_free(dflash_model* m) {
    if (!m) return;
    cudaSetDevice(m->device);
    for (auto& r : m->prof_open) {
        cudaEventDestroy(r.e0);
        cudaEventDestroy(r.e1);
    }
    for (cudaEvent_t e : m->ev_pool) cudaEventDestroy(e);
    if (m->copy_ev) cudaEventDestroy(m->copy_ev);
    if (m->err_host) cudaFreeHost(m->err_host);
    clear_graphs(m);
    if (m->cap_stream) cudaStreamDestroy(m->cap_stream);
    for (void* p : m->owned) cudaFree(p);
    for (DevBuf* b : {&m->h, &m->xq, &m->xs, &m->qkv, &m->y, &m->gu, &m->logits, &m->keys, &m->toks, &m->part,
                      &m->anchors, &m->pos0, &m->aseqs, &m->rope, &m->a_taps, &m->a_codes, &m->a_scale, &m->a_t,
                      &m->a_kv, &m->a_pos, &m->x16, &m->trace_buf, &m->cx, &m->cd, &m->co, &m->hn, &m->hp,
                      &m->cand, &m->plain})
        free_buf(*b);
    delete m;
}

const char* dflash_last_error(const dflash_model* m) { return m ? m->err.c_str() : g_init_error.c_str(); }

namespace {

// the context queue's limits (page "cortiq-engine 0.8.71 — src/dflash.rs",
// `queue_context`: PENDING_ROWS, CONTEXT_CHUNK, BLOCK_SLACK)
constexpr int64_t kPendingRows = 512, kContextChunk = 64, kBlockSlack = 256;

// Forget the positions from pos on, queued rows first (`truncate`).
void seq_truncate(dflash_seq* s, int64_t pos) {
    const int64_t held = s->first + s->len;
    s->pending = std::min(s->pending, std::max<int64_t>(pos - held, 0));
    if (s->pending == 0) s->pend_off = 0;
    const int64_t keep = std::min(std::max<int64_t>(pos - s->first, 0), s->len);
    s->len = keep;
    for (auto& d : s->dropped) d = std::min(d, keep);
}

// The position rule of an append or a queue of n rows at pos: a held position
// replaces it and what follows, a gap (or a position before the first) starts
// the context over; ECAPACITY (nothing changed) when the rows would not fit.
int seq_place(dflash_model* m, dflash_seq* s, int64_t pos, int64_t n) {
    const int64_t held = s->first + s->len, next = held + s->pending;
    const bool restart = pos > next || pos < s->first;
    const int64_t keep = restart ? 0 : std::min(pos - s->first, s->len);
    const int64_t pend = restart ? 0 : std::min(s->pending, std::max<int64_t>(pos - held, 0));
    if (keep + pend + n > s->cap)
        return set_err(m, DFLASH_ECAPACITY, "context of " + std::to_string(keep + pend + n) +
                                                " rows exceeds capacity " + std::to_string(s->cap));
    if (restart) {
        seq_truncate(s, 0);
        s->first = pos;
    } else {
        seq_truncate(s, pos);
    }
    return DFLASH_OK;
}

// n tap rows (host or device) onto the end of the queue.
int queue_rows(dflash_model* m, dflash_seq* s, const float* taps, int64_t n, bool on_device, cudaStream_t st) {
    if (n <= 0) return DFLASH_OK;
    const int64_t tw = m->tap_w;
    if (s->pend_off + s->pending + n > s->pend_cap) {
        // a larger buffer, the queued rows at its start
        const int64_t cap = std::max<int64_t>({2 * s->pend_cap, s->pending + n, kContextChunk});
        float* q = nullptr;
        CK(m, cudaMalloc(&q, (size_t)cap * tw * sizeof(float)));
        if (s->pending > 0)
            CK(m, cudaMemcpyAsync(q, s->pend + s->pend_off * tw, (size_t)s->pending * tw * sizeof(float),
                                  cudaMemcpyDeviceToDevice, st));
        if (s->pend) {
            CK(m, cudaStreamSynchronize(st));
            cudaFree(s->pend);
        }
        s->pend = q;
        s->pend_cap = cap;
        s->pend_off = 0;
    }
    CK(m, cudaMemcpyAsync(s->pend + (s->pend_off + s->pending) * tw, taps, (size_t)n * tw * sizeof(float),
                          on_device ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice, st));
    if (!on_device) CK(m, cudaEventRecord(m->copy_ev, st));
    s->pending += n;
    return DFLASH_OK;
}

// Make n rows of taps (host or device) context at position first + len
// (`settle_rows`): the projection passes, then the window drop.
int settle_rows(dflash_model* m, dflash_seq* s, const float* taps, int64_t n_rows, bool taps_on_device,
                cudaStream_t st) {
    if (n_rows <= 0) return DFLASH_OK;
    const int64_t first = s->first, len = s->len;
    const int64_t chunk = std::min<int64_t>(n_rows, kAppendRows);
    int rc = ensure_append_scratch(m, chunk);
    if (!rc && chunk > 16) rc = ensure_dense(m, st);
    if (rc) return rc;
    for (int64_t r0 = 0; r0 < n_rows; r0 += chunk) {
        const int64_t n = std::min(chunk, n_rows - r0);
        const float* src = taps + r0 * m->tap_w;
        if (!taps_on_device) {
            CK(m, cudaMemcpyAsync(m->a_taps.p, src, (size_t)n * m->tap_w * sizeof(float), cudaMemcpyHostToDevice, st));
            CK(m, cudaEventRecord(m->copy_ev, st));
            src = P<float>(m->a_taps);
        }
        const int64_t pos2[2] = {first + len + r0, len + r0};
        CK(m, cudaMemcpyAsync(m->a_pos.p, pos2, sizeof(pos2), cudaMemcpyHostToDevice, st));
        const std::vector<int64_t> key = {1, (int64_t)(intptr_t)s, (int64_t)(intptr_t)s->k_dev, n,
                                          (int64_t)(intptr_t)src};
        rc = run_enqueue(m, key, st, [&](cudaStream_t q) { return append_rows(m, s, src, n, q); });
        if (rc) return rc;
        if (!taps_on_device && r0 + chunk < n_rows) CK(m, cudaStreamSynchronize(st));  // staging reused
    }
    s->len = len + n_rows;
    // no row of a layer sees further back than its window: once a layer holds
    // more than twice its window, all but the last window of rows are dropped
    // (page "cortiq-engine 0.8.71 — src/dflash.rs", `settle_rows`)
    for (int l = 0; l < m->g.layers; ++l) {
        const int64_t w = m->win[l], held = s->len - s->dropped[l];
        if (w > 0 && held > 2 * w) s->dropped[l] += held - w;
    }
    return DFLASH_OK;
}

// Every queued row made context (`settle`).
int settle_pending(dflash_model* m, dflash_seq* s, cudaStream_t st) {
    if (s->pending == 0) return DFLASH_OK;
    const int64_t n = s->pending;
    int rc = settle_rows(m, s, s->pend + s->pend_off * m->tap_w, n, true, st);
    if (rc) return rc;
    s->pending = 0;
    s->pend_off = 0;
    return DFLASH_OK;
}

}  // namespace

int dflash_geometry_of(const dflash_model* m, dflash_geometry* out) {
    if (!m || !out) return DFLASH_EINVAL;
    *out = m->g;
    return DFLASH_OK;
}

int dflash_seq_new(dflash_model* m, int64_t max_ctx_rows, dflash_seq** out) {
    if (!m || !out) return DFLASH_EINVAL;
    *out = nullptr;
    int rc = check_model(m);
    if (rc) return rc;
    if (max_ctx_rows < 1) return set_err(m, DFLASH_EINVAL, "max_ctx_rows < 1");
    dflash_seq* s = new (std::nothrow) dflash_seq();
    if (!s) return set_err(m, DFLASH_ENOMEM, "host allocation failed");
    s->m = m;
    s->cap = max_ctx_rows;
    const int L = m->g.layers;
    const size_t per = (size_t)m->g.kv_heads * (size_t)max_ctx_rows * m->g.head_dim;
    s->k.assign(L, nullptr);
    s->dropped.assign(L, 0);
    s->v.assign(L, nullptr);
    cudaError_t e = cudaSuccess;
    for (int l = 0; l < L && e == cudaSuccess; ++l) {
        e = cudaMalloc(&s->k[l], 2 * per * sizeof(__half));
        if (e == cudaSuccess) e = cudaMalloc(&s->v[l], 2 * per * sizeof(__half));
    }
    if (e == cudaSuccess) e = cudaMalloc(&s->k_dev, L * sizeof(__half*));
    if (e == cudaSuccess) e = cudaMalloc(&s->v_dev, L * sizeof(__half*));
    if (e == cudaSuccess) e = cudaMemcpy(s->k_dev, s->k.data(), L * sizeof(__half*), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(s->v_dev, s->v.data(), L * sizeof(__half*), cudaMemcpyHostToDevice);
    // every stored value finite from the start: the tcgen05 attention's
    // tensor copies read whole 128-row boxes, rows past the context included
    // (their weights are exactly zero, and 0 times a finite value is 0)
    for (int l = 0; l < L && e == cudaSuccess; ++l) {
        e = cudaMemset(s->k[l], 0, 2 * per * sizeof(__half));
        if (e == cudaSuccess) e = cudaMemset(s->v[l], 0, 2 * per * sizeof(__half));
    }
    if (e == cudaSuccess) {
        alignas(64) unsigned char maps[256];
        std::vector<unsigned char> all((size_t)L * 256);
        bool built = true;
        for (int l = 0; l < L && built; ++l) {
            built = kv_tensor_maps(s->k[l], s->v[l], m->g.kv_heads, max_ctx_rows, m->g.head_dim, maps);
            if (built) std::memcpy(all.data() + (size_t)l * 256, maps, 256);
        }
        if (built) {
            e = cudaMalloc(&s->maps_dev, all.size());
            if (e == cudaSuccess) e = cudaMemcpy(s->maps_dev, all.data(), all.size(), cudaMemcpyHostToDevice);
        }
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        dflash_seq_free(s);
        return set_err(m, e == cudaErrorMemoryAllocation ? DFLASH_ENOMEM : DFLASH_ECUDA,
                       std::string("sequence allocation: ") + cudaGetErrorString(e));
    }
    m->live_seqs++;
    *out = s;
    return DFLASH_OK;
}

void dflash_seq_free(dflash_seq* s) {
    if (!s) return;
    if (s->m) cudaSetDevice(s->m->device);
    for (__half* p : s->k) if (p) cudaFree(p);
    for (__half* p : s->v) if (p) cudaFree(p);
    if (s->k_dev) cudaFree(s->k_dev);
    if (s->v_dev) cudaFree(s->v_dev);
    if (s->maps_dev) cudaFree(s->maps_dev);
    if (s->pend) cudaFree(s->pend);
    if (s->m && s->m->live_seqs > 0) s->m->live_seqs--;
    delete s;
}

int dflash_seq_span(const dflash_seq* s, int64_t* first, int64_t* next) {
    if (!s || !first || !next) return DFLASH_EINVAL;
    *first = s->first;
    *next = s->first + s->len + s->pending;
    return DFLASH_OK;
}

int dflash_truncate(dflash_seq* s, int64_t pos) {
    if (!s) return DFLASH_EINVAL;
    seq_truncate(s, pos);
    return DFLASH_OK;
}

int dflash_reset(dflash_seq* s) {
    if (!s) return DFLASH_EINVAL;
    seq_truncate(s, 0);
    s->first = 0;
    return DFLASH_OK;
}

int dflash_ctx_append(dflash_model* m, dflash_seq* s, int64_t pos, const float* taps, int64_t n_rows,
                      int taps_on_device, void* stream) {
    int rc = check_model(m);
    if (rc) return rc;
    if (!s || s->m != m) return set_err(m, DFLASH_EINVAL, "sequence is NULL or belongs to another model");
    if (n_rows < 0 || pos < 0) return set_err(m, DFLASH_EINVAL, "n_rows < 0 or pos < 0");
    if (n_rows > 0 && !taps) return set_err(m, DFLASH_EINVAL, "taps is NULL");
    cudaStream_t st = (cudaStream_t)stream;
    rc = seq_place(m, s, pos, n_rows);
    if (rc) return rc;
    if (s->pending > 0) {
        // queued rows still held go first, in the same settle
        rc = queue_rows(m, s, taps, n_rows, taps_on_device != 0, st);
        if (!rc) rc = settle_pending(m, s, st);
    } else {
        rc = settle_rows(m, s, taps, n_rows, taps_on_device != 0, st);
    }
    if (rc) return rc;
    // host taps: back once they are copied; a wait that expires in this
    // work is reported by the next call that reads the device (a block with
    // host buffers)
    if (!taps_on_device && n_rows > 0) CK(m, cudaEventSynchronize(m->copy_ev));
    return DFLASH_OK;
}

int dflash_ctx_queue(dflash_model* m, dflash_seq* s, int64_t pos, const float* taps, int64_t n_rows,
                     int taps_on_device, void* stream) {
    int rc = check_model(m);
    if (rc) return rc;
    if (!s || s->m != m) return set_err(m, DFLASH_EINVAL, "sequence is NULL or belongs to another model");
    if (n_rows < 0 || pos < 0) return set_err(m, DFLASH_EINVAL, "n_rows < 0 or pos < 0");
    if (n_rows > 0 && !taps) return set_err(m, DFLASH_EINVAL, "taps is NULL");
    cudaStream_t st = (cudaStream_t)stream;
    rc = seq_place(m, s, pos, n_rows);
    if (!rc) rc = queue_rows(m, s, taps, n_rows, taps_on_device != 0, st);
    if (rc) return rc;
    if (!taps_on_device && n_rows > 0) CK(m, cudaEventSynchronize(m->copy_ev));  // the caller's rows are copied
    // past the queue's limit the oldest rows go through, a multiple of the granule
    int64_t limit = kPendingRows;
    bool all_windowed = true;
    int64_t widest = 0;
    for (int l = 0; l < m->g.layers; ++l) {
        all_windowed = all_windowed && m->win[l] > 0;
        widest = std::max<int64_t>(widest, m->win[l]);
    }
    if (all_windowed) limit = std::max<int64_t>(kPendingRows, widest + kBlockSlack);
    if (s->pending > limit) {
        const int64_t over = std::min((s->pending - limit + kContextChunk - 1) / kContextChunk * kContextChunk, s->pending);
        rc = settle_rows(m, s, s->pend + s->pend_off * m->tap_w, over, true, st);
        if (rc) return rc;
        s->pend_off += over;
        s->pending -= over;
        if (s->pending == 0) s->pend_off = 0;
    }
    return DFLASH_OK;
}

int dflash_settle(dflash_model* m, dflash_seq* s, void* stream) {
    int rc = check_model(m);
    if (rc) return rc;
    if (!s || s->m != m) return set_err(m, DFLASH_EINVAL, "sequence is NULL or belongs to another model");
    return settle_pending(m, s, (cudaStream_t)stream);
}

int dflash_block(dflash_model* m, dflash_seq* const* seqs, int32_t n_seqs, const uint32_t* anchor_tok,
                 const int64_t* anchor_pos, int32_t block_len, float* logits, uint32_t* draft_tok, int io_on_device,
                 void* stream) {
    int rc = check_model(m);
    if (rc) return rc;
    const dflash_geometry& g = m->g;
    if (!seqs || !anchor_tok || !anchor_pos || n_seqs < 1)
        return set_err(m, DFLASH_EINVAL, "seqs / anchor_tok / anchor_pos NULL or n_seqs < 1");
    if (block_len < 2 || block_len > g.block)
        return set_err(m, DFLASH_ERANGE, "block_len " + std::to_string(block_len) + " outside [2, block]");
    for (int s = 0; s < n_seqs; ++s) {
        if (!seqs[s] || seqs[s]->m != m) return set_err(m, DFLASH_EINVAL, "a sequence is NULL or of another model");
        if (anchor_pos[s] < 0) return set_err(m, DFLASH_EINVAL, "anchor_pos < 0");
        if (!io_on_device && anchor_tok[s] >= (uint32_t)g.vocab)
            return set_err(m, DFLASH_EINVAL, "anchor token outside the vocabulary");
    }
    cudaStream_t st = (cudaStream_t)stream;
    // the queued rows become context before the block reads it
    for (int s = 0; s < n_seqs; ++s) {
        rc = settle_pending(m, seqs[s], st);
        if (rc) return rc;
    }
    const bool quant = g.quant == DFLASH_QUANT_Q4G32;
    const int H = g.hidden, I = g.intermediate, hd = g.head_dim, B = block_len;
    const int R = n_seqs * B, D = n_seqs * (B - 1);
    const int maxK = std::max({H, I, m->qd});

    std::vector<int64_t> p0(anchor_pos, anchor_pos + n_seqs);
    int max_ctx = 0;  // the launch is planned for the largest capacity, so that it stays as contexts grow
    for (int s = 0; s < n_seqs; ++s) max_ctx = (int)std::max<int64_t>(max_ctx, seqs[s]->cap);
    // every layer's context views: [layer][sequence], and each layer's attention bytes
    std::vector<AttnSeq> as_all((size_t)g.layers * n_seqs);
    std::vector<double> attn_bytes_l(g.layers, (double)R * m->qkv_w * 4 + (double)R * m->qd * 4);
    for (int l = 0; l < g.layers; ++l)
        for (int s = 0; s < n_seqs; ++s) {
            as_all[(size_t)l * n_seqs + s] = layer_view(m, seqs[s], l, anchor_pos[s]);
            attn_bytes_l[l] += (double)as_all[(size_t)l * n_seqs + s].n * m->kd * 8;
        }
    const int64_t part_floats = attn_scratch_floats(n_seqs, B, max_ctx, g.heads, g.kv_heads, hd, m->num_sms);
    // layers whose attention accumulates its key splits' rescaled partial
    // rows (few units: a single sequence's 8 kv heads spread over every SM)
    // (on the tcgen05 kernel when its single query tile holds a unit's rows:
    // then every unit count, a batch filling the SMs included)
    bool tc_attn = quant && m->use_tc && attention_tc_supported(g.heads, g.kv_heads, hd, B);
    for (int s = 0; s < n_seqs; ++s) tc_attn = tc_attn && seqs[s]->maps_dev != nullptr;
    int tc_split = tc_attn ? attn_tc_plan(n_seqs, B, max_ctx, g.kv_heads, m->num_sms) : 0;
    // the tcgen05 kernel where each CTA has a few key steps to stream (its
    // fixed cost -- queries, tensor memory, the pipeline's ramp -- then
    // amortises: long contexts, batches); the warp-MMA kernel for short splits
    if (tc_attn && tc_split > 1 && (int64_t)(max_ctx + B) / tc_split < m->tc_attn_min_keys) tc_attn = false;
    const int acc_split = !quant    ? 0
                          : tc_attn ? tc_split
                                    : attn_acc_plan(n_seqs, B, max_ctx, g.heads, g.kv_heads, hd, m->num_sms);
    std::vector<char> acc_l(g.layers, 0);
    bool any_acc = false;
    for (int l = 0; l < g.layers; ++l) {
        acc_l[l] = acc_split > 0 && !std::isnan(m->attn_ref[l]);
        any_acc = any_acc || acc_l[l];
    }
    // qkv, then (accumulate mode) the attention's unnormalised output and its
    // softmax sums: one buffer, cleared together before each layer's qkv
    const int64_t qkv_zero = (int64_t)R * m->qkv_w + (any_acc ? (int64_t)R * (m->qd + g.heads) : 0);
    CK(m, ensure_m(m, m->h, (size_t)R * H * sizeof(float)));
    CK(m, ensure_m(m, m->xq, (size_t)R * (quant ? maxK : maxK * sizeof(float))));
    CK(m, ensure_m(m, m->xs, (size_t)R * sizeof(float)));
    CK(m, ensure_m(m, m->qkv, (size_t)qkv_zero * sizeof(float)));
    CK(m, ensure_m(m, m->y, (size_t)R * m->qd * sizeof(float)));
    CK(m, ensure_m(m, m->gu, (size_t)R * 2 * I * sizeof(float)));
    CK(m, ensure_m(m, m->part, (size_t)part_floats * sizeof(float)));
    CK(m, ensure_m(m, m->keys, (size_t)D * sizeof(unsigned long long)));
    CK(m, ensure_m(m, m->toks, (size_t)D * sizeof(uint32_t)));
    CK(m, ensure_m(m, m->anchors, (size_t)n_seqs * sizeof(uint32_t)));
    CK(m, ensure_m(m, m->pos0, (size_t)n_seqs * sizeof(int64_t)));
    CK(m, ensure_m(m, m->rope, (size_t)R * (hd / 2) * sizeof(float2)));
    CK(m, ensure_m(m, m->aseqs, (size_t)g.layers * n_seqs * sizeof(AttnSeq)));
    if (g.selector_rank > 0) {
        CK(m, ensure_m(m, m->hn, (size_t)D * H * sizeof(float)));
        CK(m, ensure_m(m, m->hp, (size_t)D * g.selector_rank * sizeof(float)));
        CK(m, ensure_m(m, m->cand, (size_t)D * g.selector_top * (1 + topk_parts(g.vocab, g.selector_top)) *
                                       sizeof(unsigned long long)));
        CK(m, ensure_m(m, m->plain, (size_t)D * sizeof(uint32_t)));
    }
    if (g.conv_kernel > 0) {
        CK(m, ensure_m(m, m->cx, (size_t)R * H * sizeof(float)));
        CK(m, ensure_m(m, m->cd, (size_t)R * 2 * g.conv_kernel * (H / g.conv_group) * sizeof(float)));
        CK(m, ensure_m(m, m->co, (size_t)R * H * sizeof(float)));
    }
    if (quant && R > 16) {
        // f16 codes of the widest matmul input, then the head rows' code norms
        CK(m, ensure_m(m, m->x16, (size_t)R * (maxK * sizeof(__half) + sizeof(int))));
        rc = ensure_dense(m, st);
        if (rc) return rc;
    }
    float* logit_out = io_on_device ? logits : nullptr;
    if (!io_on_device && logits) {
        CK(m, ensure_m(m, m->logits, (size_t)D * g.vocab * sizeof(float)));
        logit_out = P<float>(m->logits);
    }
    if ((!quant || g.selector_rank > 0) && !logit_out) {  // the f32 head's argmax and the selector read the logits
        CK(m, ensure_m(m, m->logits, (size_t)D * g.vocab * sizeof(float)));
        logit_out = P<float>(m->logits);
    }
    // per-call vectors (pageable sources: the driver copies them before returning)
    const uint32_t* anchors_dev = anchor_tok;
    if (!io_on_device) {
        CK(m, cudaMemcpyAsync(m->anchors.p, anchor_tok, n_seqs * sizeof(uint32_t), cudaMemcpyHostToDevice, st));
        anchors_dev = P<uint32_t>(m->anchors);
    }
    CK(m, cudaMemcpyAsync(m->pos0.p, p0.data(), n_seqs * sizeof(int64_t), cudaMemcpyHostToDevice, st));
    // every layer's context views in one upload
    CK(m, cudaMemcpyAsync(m->aseqs.p, as_all.data(), as_all.size() * sizeof(AttnSeq), cudaMemcpyHostToDevice, st));

    auto enqueue = [&](cudaStream_t st) -> int {
    float* h = P<float>(m->h);
    float* qkv = P<float>(m->qkv);
    float* y = P<float>(m->y);
    const float scale = 1.0f / sqrtf((float)hd);
    float* yacc = qkv + (size_t)R * m->qkv_w;  // accumulate mode (any_acc)
    float* lacc = yacc + (size_t)R * m->qd;
    // the many-row matmuls' f16 activation codes, written by the kernels that
    // quantise (not while tracing: a forced decision replaces the int8 codes
    // after them, and the matmul converts those itself)
    __half* o16 = (quant && R > 16 && !m->tracing && m->use_tc) ? P<__half>(m->x16) : nullptr;
    const bool x16r = o16 != nullptr;
    // what the in_norm quantisation clears on the side: the streaming matvec
    // (up to 16 rows) adds into qkv, so qkv and the attention's accumulators;
    // the many-row matmuls clear their own output when they split K, so only
    // the accumulators
    float* qz = R <= 16 ? qkv : yacc;
    const int64_t qz_n = R <= 16 ? qkv_zero : (any_acc ? (int64_t)R * (m->qd + g.heads) : 0);
    // the block's attention of layer l into y (or, accumulate mode, into
    // yacc / lacc, which the clearing before the layer's qkv zeroed)
    auto run_attention = [&](int l) -> int {
        const Layer& Ly = m->layers[l];
        const AttnSeq* aseq_dev = P<AttnSeq>(m->aseqs) + (size_t)l * n_seqs;
        const float2* rl = m->norope[l] ? nullptr : P<float2>(m->rope);
        if (acc_l[l] && tc_attn) {
            KL(m, "attention", 1, attn_bytes_l[l] + (double)R * g.heads * (hd + 1) * 4, st,
               attention_tc(qkv, m->qkv_w, n_seqs, B, aseq_dev, acc_split, g.heads, g.kv_heads, hd, scale, yacc, lacc,
                            m->attn_ref[l], st, Ly.q_norm, Ly.k_norm, rl, g.eps, m->own_capture, m->win[l] > 0,
                            m->err_dev));
        } else if (acc_l[l]) {
            KL(m, "attention", 1, attn_bytes_l[l] + (double)R * g.heads * (hd + 1) * 4, st,
               attention_acc(qkv, m->qkv_w, n_seqs, B, aseq_dev, acc_split, g.heads, g.kv_heads, hd, scale, yacc, lacc,
                             m->attn_ref[l], st, Ly.q_norm, Ly.k_norm, rl, g.eps, m->own_capture, m->win[l] > 0));
        } else {
            KL(m, "attention", attn_kernels(n_seqs, B, max_ctx, g.heads, g.kv_heads, hd, m->num_sms, part_floats),
               attn_bytes_l[l], st,
               attention(qkv, m->qkv_w, n_seqs, B, aseq_dev, max_ctx, g.heads, g.kv_heads, hd, scale,
                         P<float>(m->part), part_floats, y, m->num_sms, st, Ly.q_norm, Ly.k_norm, rl, g.eps,
                         m->own_capture, m->win[l] > 0));
        }
        return DFLASH_OK;
    };
    float* gu = P<float>(m->gu);
    float* xf = P<float>(m->xq);  // the f32 path's normed rows
    int8_t* xq = P<int8_t>(m->xq);
    float* xs = P<float>(m->xs);
    RowMap ident{1, 1, 0};

    // the embedding also writes the block rows' rotation table (cos, sin per
    // position and frequency) that the attention applies as it loads q and k
    float2* rope = P<float2>(m->rope);
    KL(m, "embed_rows", 1, (double)R * H * 8, st,
       embed_rows(m->embed, H, g.vocab, anchors_dev, g.mask_token, n_seqs, B, h, st, P<int64_t>(m->pos0),
                  m->inv_freq, hd, rope));
    RowMap drafts{B - 1, B, 1};
    unsigned long long* keys = P<unsigned long long>(m->keys);
    uint32_t* tok_out = (io_on_device && draft_tok) ? draft_tok : P<uint32_t>(m->toks);
    // with a row convolution: x = conv_in(rms(h, norm)) before each
    // sub-layer, h += conv_out(its output) after it (a separate sequence of
    // launches; the sub-layers' own kernels are the same)
    for (int l = 0; l < g.layers && g.conv_kernel > 0; ++l) {
        const Layer& Ly = m->layers[l];
        const int kn = g.conv_kernel, gs = g.conv_group, nd = 2 * kn * (H / gs);
        float* cx = P<float>(m->cx);
        float* cd = P<float>(m->cd);
        float* co = P<float>(m->co);
        // cx = rms(h, w); cd = proj . cx; then stage 0 of cx: the codes of the
        // next matmul (quantised) or its f32 rows; `zero` cleared on the side
        // of the norm's launch, `zero2` of stage 0's
        auto conv_in = [&](const float* w, const float* base, const float* proj, float* zero, int64_t zero_n,
                           float* zero2, int64_t zero2_n) -> int {
            KL(m, "rms_f32", 1, (double)R * H * 8, st,
               rms_rows(h, H, ident, R, H, w, g.eps, cx, H, nullptr, nullptr, 0, st, zero, zero_n));
            KL(m, "linear_f32", 1, f32_bytes_of(nd, H, R, false), st,
               linear_f32(proj, nd, H, cx, H, R, cd, nd, false, st));
            if (quant) {
                KL(m, "conv_rows", 1, (double)R * H * 4 * (kn + 1), st,
                   conv_rows(cx, H, cd, nd, base, 0, kn, gs, H, R, B, nullptr, 0, nullptr, 0, xq, xs, maxK, st, zero2,
                             zero2_n));
                TRACE(trace_site(m, st, R, H, xq, maxK, xs, [&](float* v) {
                    return conv_rows(cx, H, cd, nd, base, 0, kn, gs, H, R, B, nullptr, 0, v, H, nullptr, nullptr, 0,
                                     st);
                }));
            } else {
                KL(m, "conv_rows", 1, (double)R * H * 4 * (kn + 1), st,
                   conv_rows(cx, H, cd, nd, base, 0, kn, gs, H, R, B, nullptr, 0, xf, maxK, nullptr, nullptr, 0, st, zero2,
                             zero2_n));
            }
            return DFLASH_OK;
        };
        // h += stage 1 of the sub-layer's output co
        auto conv_out = [&](const float* base) -> int {
            KL(m, "conv_rows", 1, (double)R * H * 4 * (kn + 2), st,
               conv_rows(co, H, cd, nd, base, 1, kn, gs, H, R, B, h, H, nullptr, 0, nullptr, nullptr, 0, st));
            return DFLASH_OK;
        };
        APPLY(conv_in(Ly.in_norm, Ly.a_base, Ly.a_proj, quant ? qkv : nullptr, quant ? qkv_zero : 0, nullptr, 0));
        if (quant)
            APPLY(apply(m, Ly.qkv_p, nullptr, m->L_qkv, 0, m->qkv_w, H, nullptr, 0, R, qkv, m->qkv_w, false, maxK, st));
        else
            APPLY(apply(m, nullptr, Ly.qkv_f, Q4Layout{}, 0, m->qkv_w, H, xf, maxK, R, qkv, m->qkv_w, false, 0, st));
        APPLY(run_attention(l));
        // co = O y (the streaming matvec adds: co cleared by the quantisation of y)
        if (quant) {
            const float* ysrc = acc_l[l] ? yacc : y;
            const float* ydiv = acc_l[l] ? lacc : nullptr;
            KL(m, "rms_quant", 1, (double)R * m->qd * 5, st,
               rms_rows(ysrc, m->qd, ident, R, m->qd, nullptr, g.eps, nullptr, 0, xq, xs, maxK, st, co, (int64_t)R * H,
                        ydiv, hd));
            TRACE(trace_site(m, st, R, m->qd, xq, maxK, xs, [&](float* v) {
                return rms_rows(ysrc, m->qd, ident, R, m->qd, nullptr, g.eps, v, m->qd, nullptr, nullptr, 0, st,
                                nullptr, 0, ydiv, hd);
            }));
            APPLY(apply(m, Ly.o_p, nullptr, m->L_o, 0, H, m->qd, nullptr, 0, R, co, H, false, maxK, st));
        } else {
            APPLY(apply(m, nullptr, Ly.o_f, Q4Layout{}, 0, H, m->qd, y, m->qd, R, co, H, false, 0, st));
        }
        APPLY(conv_out(Ly.a_base));
        // the MLP the same way (gu cleared by the norm's launch, co by stage 0's)
        APPLY(conv_in(Ly.post_norm, Ly.m_base, Ly.m_proj, quant ? gu : nullptr, quant ? (int64_t)R * 2 * I : 0,
                      quant ? co : nullptr, quant ? (int64_t)R * H : 0));
        if (quant) {
            APPLY(apply(m, Ly.gu_p, nullptr, m->L_gu, 0, 2 * I, H, nullptr, 0, R, gu, 2 * I, false, maxK, st));
            KL(m, "silu_quant", 1, (double)R * I * 9, st, silu_mul(gu, 2 * I, R, I, nullptr, 0, xq, xs, maxK, st));
            TRACE(trace_site(m, st, R, I, xq, maxK, xs, [&](float* v) {
                return silu_mul(gu, 2 * I, R, I, v, I, nullptr, nullptr, 0, st);
            }));
            APPLY(apply(m, Ly.down_p, nullptr, m->L_down, 0, H, I, nullptr, 0, R, co, H, false, maxK, st));
        } else {
            APPLY(apply(m, nullptr, Ly.gu_f, Q4Layout{}, 0, 2 * I, H, xf, maxK, R, gu, 2 * I, false, 0, st));
            KL(m, "silu_f32", 1, (double)R * I * 12, st, silu_mul(gu, 2 * I, R, I, xf, maxK, nullptr, nullptr, 0, st));
            APPLY(apply(m, nullptr, Ly.down_f, Q4Layout{}, 0, H, I, xf, maxK, R, co, H, false, 0, st));
        }
        APPLY(conv_out(Ly.m_base));
    }
    for (int l = 0; l < g.layers && g.conv_kernel == 0; ++l) {
        const Layer& Ly = m->layers[l];
        // attention half: x = rms(h, in_norm); q, k, v; norms and rotation; attention; h += O y
        if (quant) {
            KL(m, "rms_quant", 1, (double)R * H * 5, st,
               rms_rows(h, H, ident, R, H, Ly.in_norm, g.eps, nullptr, 0, xq, xs, maxK, st, qz, qz_n, nullptr, 0,
                        o16));
            TRACE(trace_site(m, st, R, H, xq, maxK, xs, [&](float* v) {
                return rms_rows(h, H, ident, R, H, Ly.in_norm, g.eps, v, H, nullptr, nullptr, 0, st);
            }));
            APPLY(apply(m, Ly.qkv_p, nullptr, m->L_qkv, 0, m->qkv_w, H, nullptr, 0, R, qkv, m->qkv_w, false, maxK, st,
                        x16r));
        } else {
            KL(m, "rms_f32", 1, (double)R * H * 8, st, rms_rows(h, H, ident, R, H, Ly.in_norm, g.eps, xf, maxK, nullptr, nullptr, 0, st));
            APPLY(apply(m, nullptr, Ly.qkv_f, Q4Layout{}, 0, m->qkv_w, H, xf, maxK, R, qkv, m->qkv_w, false, 0, st));
        }
        // q/k norms and rotation run inside the attention, as it loads them
        APPLY(run_attention(l));
        if (quant) {
            // y (accumulate mode: yacc / lacc per head) -> int8 rows
            const float* ysrc = acc_l[l] ? yacc : y;
            const float* ydiv = acc_l[l] ? lacc : nullptr;
            KL(m, "rms_quant", 1, (double)R * m->qd * 5, st,
               rms_rows(ysrc, m->qd, ident, R, m->qd, nullptr, g.eps, nullptr, 0, xq, xs, maxK, st, nullptr, 0, ydiv,
                        hd, o16));
            TRACE(trace_site(m, st, R, m->qd, xq, maxK, xs, [&](float* v) {
                return rms_rows(ysrc, m->qd, ident, R, m->qd, nullptr, g.eps, v, m->qd, nullptr, nullptr, 0, st,
                                nullptr, 0, ydiv, hd);
            }));
            APPLY(apply(m, Ly.o_p, nullptr, m->L_o, 0, H, m->qd, nullptr, 0, R, h, H, true, maxK, st, x16r));
        } else {
            APPLY(apply(m, nullptr, Ly.o_f, Q4Layout{}, 0, H, m->qd, y, m->qd, R, h, H, true, 0, st));
        }
        // MLP half: x = rms(h, post_norm); h += down (silu(gate x) * up x)
        if (quant) {
            KL(m, "rms_quant", 1, (double)R * H * 5, st,
               rms_rows(h, H, ident, R, H, Ly.post_norm, g.eps, nullptr, 0, xq, xs, maxK, st, R <= 16 ? gu : nullptr,
                        R <= 16 ? (int64_t)R * 2 * I : 0, nullptr, 0, o16));
            TRACE(trace_site(m, st, R, H, xq, maxK, xs, [&](float* v) {
                return rms_rows(h, H, ident, R, H, Ly.post_norm, g.eps, v, H, nullptr, nullptr, 0, st);
            }));
            APPLY(apply(m, Ly.gu_p, nullptr, m->L_gu, 0, 2 * I, H, nullptr, 0, R, gu, 2 * I, false, maxK, st, x16r));
            KL(m, "silu_quant", 1, (double)R * I * 9, st, silu_mul(gu, 2 * I, R, I, nullptr, 0, xq, xs, maxK, st, o16));
            TRACE(trace_site(m, st, R, I, xq, maxK, xs, [&](float* v) {
                return silu_mul(gu, 2 * I, R, I, v, I, nullptr, nullptr, 0, st);
            }));
            APPLY(apply(m, Ly.down_p, nullptr, m->L_down, 0, H, I, nullptr, 0, R, h, H, true, maxK, st, x16r));
        } else {
            KL(m, "rms_f32", 1, (double)R * H * 8, st, rms_rows(h, H, ident, R, H, Ly.post_norm, g.eps, xf, maxK, nullptr, nullptr, 0, st));
            APPLY(apply(m, nullptr, Ly.gu_f, Q4Layout{}, 0, 2 * I, H, xf, maxK, R, gu, 2 * I, false, 0, st));
            KL(m, "silu_f32", 1, (double)R * I * 12, st, silu_mul(gu, 2 * I, R, I, xf, maxK, nullptr, nullptr, 0, st));
            APPLY(apply(m, nullptr, Ly.down_f, Q4Layout{}, 0, H, I, xf, maxK, R, h, H, true, 0, st));
        }
    }
    // head over the rows after each anchor: row i of the output is row
    // (i / (B-1)) * B + 1 + i % (B-1) of h
    if (quant) {
        KL(m, "rms_quant", 1, (double)D * H * 5, st,
           rms_rows(h, H, drafts, D, H, m->norm, g.eps, nullptr, 0, xq, xs, maxK, st, reinterpret_cast<float*>(keys),
                    (int64_t)D * 2));
        TRACE(trace_site(m, st, D, H, xq, maxK, xs, [&](float* v) {
            return rms_rows(h, H, drafts, D, H, m->norm, g.eps, v, H, nullptr, nullptr, 0, st);
        }));
        QAct xh{xq, xs, maxK};
        const double hb = (double)g.vocab * H + (double)g.vocab * 4 + (double)D * H + (logit_out ? (double)D * g.vocab * 4 : 0.0);
        APPLY(run_head(m, xh, D, logit_out, keys, hb, st));
    } else {
        KL(m, "rms_f32", 1, (double)D * H * 8, st, rms_rows(h, H, drafts, D, H, m->norm, g.eps, xf, maxK, nullptr, nullptr, 0, st,
                                                         reinterpret_cast<float*>(keys), (int64_t)D * 2));
        KL(m, "linear_f32", 1, f32_bytes_of(g.vocab, H, D, false), st,
           linear_f32(m->head_f, g.vocab, H, xf, maxK, D, logit_out, g.vocab, false, st));
        KL(m, "argmax_rows", 1, (double)D * g.vocab * 4, st, argmax_rows(logit_out, g.vocab, g.vocab, D, keys, st));
    }
    if (g.selector_rank > 0)
        APPLY(run_selector(m, st, h, drafts, D, n_seqs, B, logit_out, anchors_dev, tok_out));
    else
        KL(m, "keys_to_tokens", 1, (double)D * 12, st, keys_to_tokens(keys, D, tok_out, st));
    return DFLASH_OK;
    };
    uint32_t* tok_out = (io_on_device && draft_tok) ? draft_tok : P<uint32_t>(m->toks);
    const std::vector<int64_t> key = {2, n_seqs, B, max_ctx, (int64_t)(intptr_t)logit_out, (int64_t)(intptr_t)tok_out,
                                      (int64_t)(intptr_t)anchors_dev};
    rc = run_enqueue(m, key, st, enqueue);
    if (rc) return rc;
    if (!io_on_device) {
        if (logits)
            CK(m, cudaMemcpyAsync(logits, logit_out, (size_t)D * g.vocab * sizeof(float), cudaMemcpyDeviceToHost, st));
        if (draft_tok)
            CK(m, cudaMemcpyAsync(draft_tok, tok_out, (size_t)D * sizeof(uint32_t), cudaMemcpyDeviceToHost, st));
        CK(m, cudaMemcpyAsync(m->err_host, m->err_dev, sizeof(int), cudaMemcpyDeviceToHost, st));
        CK(m, cudaStreamSynchronize(st));
        if (*m->err_host) return device_wait_expired(m);
    }
    return DFLASH_OK;
}

// ------------------------------------------------------------------ attention alone
namespace {

// Checks of an attention call and the per-sequence context views of one layer.
int attention_views(dflash_model* m, dflash_seq* const* seqs, int32_t n_seqs, int32_t layer,
                    const int64_t* anchor_pos, int32_t block_len, const float* qkv, const float* y,
                    std::vector<AttnSeq>& views, int* max_ctx) {
    const dflash_geometry& g = m->g;
    if (!seqs || !anchor_pos || !qkv || !y || n_seqs < 1 || layer < 0 || layer >= g.layers)
        return set_err(m, DFLASH_EINVAL, "attention: null pointer, n_seqs < 1 or bad layer");
    if (block_len < 2 || block_len > g.block) return set_err(m, DFLASH_ERANGE, "attention: block_len outside [2, block]");
    if (reinterpret_cast<uintptr_t>(qkv) % 16 != 0)
        return set_err(m, DFLASH_EINVAL, "attention: qkv must be 16-byte aligned");
    views.assign(n_seqs, AttnSeq{});
    *max_ctx = 0;
    for (int s = 0; s < n_seqs; ++s) {
        const dflash_seq* q = seqs[s];
        if (!q || q->m != m) return set_err(m, DFLASH_EINVAL, "attention: a sequence is NULL or of another model");
        if (anchor_pos[s] < 0) return set_err(m, DFLASH_EINVAL, "attention: anchor_pos < 0");
        views[s] = layer_view(m, q, layer, anchor_pos[s]);
        *max_ctx = std::max(*max_ctx, views[s].n);
    }
    return DFLASH_OK;
}

}  // namespace

int dflash_debug_attention(dflash_model* m, dflash_seq* const* seqs, int32_t n_seqs, int32_t layer,
                           const int64_t* anchor_pos, int32_t block_len, const float* qkv, float* y, void* stream) {
    int rc = check_model(m);
    if (rc) return rc;
    std::vector<AttnSeq> views;
    int max_ctx = 0;
    rc = attention_views(m, seqs, n_seqs, layer, anchor_pos, block_len, qkv, y, views, &max_ctx);
    if (rc) return rc;
    const dflash_geometry& g = m->g;
    cudaStream_t st = (cudaStream_t)stream;
    const int64_t part_floats =
        attn_scratch_floats(n_seqs, block_len, max_ctx, g.heads, g.kv_heads, g.head_dim, m->num_sms);
    CK(m, ensure_m(m, m->part, (size_t)part_floats * sizeof(float)));
    CK(m, ensure_m(m, m->aseqs, (size_t)n_seqs * sizeof(AttnSeq)));
    CK(m, cudaMemcpyAsync(m->aseqs.p, views.data(), views.size() * sizeof(AttnSeq), cudaMemcpyHostToDevice, st));
    KL(m, "attention", attn_kernels(n_seqs, block_len, max_ctx, g.heads, g.kv_heads, g.head_dim, m->num_sms, part_floats), 0.0, st,
       attention(qkv, m->qkv_w, n_seqs, block_len, P<AttnSeq>(m->aseqs), max_ctx, g.heads, g.kv_heads, g.head_dim,
                 1.0f / sqrtf((float)g.head_dim), P<float>(m->part), part_floats, y, m->num_sms, st, nullptr, nullptr,
                 nullptr, 0.f, false, m->win[layer] > 0));
    return DFLASH_OK;
}

// ------------------------------------------------------------------ site trace
int dflash_debug_trace(dflash_model* m, int32_t enable) {
    if (!m) return DFLASH_EINVAL;
    m->tracing = enable != 0;
    m->trace.clear();
    m->forced.clear();
    m->forced_next = 0;
    return DFLASH_OK;
}

int dflash_debug_trace_force(dflash_model* m, int32_t rows, int32_t cols, const int8_t* codes, const float* scales) {
    if (!m || rows < 1 || cols < 1 || !codes || !scales) return DFLASH_EINVAL;
    dflash_model::Site f;
    f.rows = rows;
    f.cols = cols;
    f.codes.assign(codes, codes + (size_t)rows * cols);
    f.scales.assign(scales, scales + rows);
    m->forced.push_back(std::move(f));
    return DFLASH_OK;
}

int dflash_debug_trace_site(const dflash_model* m, int32_t i, int32_t* rows, int32_t* cols, float* values,
                            int8_t* codes, float* scales) {
    if (!m) return DFLASH_EINVAL;
    if (i < 0 || i >= (int32_t)m->trace.size()) return DFLASH_ERANGE;
    const auto& t = m->trace[i];
    if (rows) *rows = t.rows;
    if (cols) *cols = t.cols;
    if (values) std::memcpy(values, t.values.data(), t.values.size() * sizeof(float));
    if (codes) std::memcpy(codes, t.codes.data(), t.codes.size());
    if (scales) std::memcpy(scales, t.scales.data(), t.scales.size() * sizeof(float));
    return DFLASH_OK;
}

// ------------------------------------------------------------------ tracing
int dflash_profile_start(dflash_model* m) {
    if (!m) return DFLASH_EINVAL;
    for (auto& r : m->prof_open) {
        m->ev_pool.push_back(r.e0);
        m->ev_pool.push_back(r.e1);
    }
    m->prof_open.clear();
    m->prof_sum.clear();
    m->profiling = true;
    return DFLASH_OK;
}

int dflash_profile_stop(dflash_model* m) {
    if (!m) return DFLASH_EINVAL;
    m->profiling = false;
    int rc = DFLASH_OK;
    for (auto& r : m->prof_open) {
        float ms = 0.f;
        cudaError_t e = cudaEventSynchronize(r.e1);
        if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, r.e0, r.e1);
        if (e != cudaSuccess && rc == DFLASH_OK) rc = cuda_fail(m, (int)e, "profile events");
        auto it = std::find_if(m->prof_sum.begin(), m->prof_sum.end(),
                               [&](const dflash_model::ProfSum& p) { return std::strcmp(p.name, r.name) == 0; });
        if (it == m->prof_sum.end()) {
            m->prof_sum.push_back(dflash_model::ProfSum{r.name});
            it = m->prof_sum.end() - 1;
        }
        it->launches += r.kernels;
        it->ms += ms;
        it->bytes += r.bytes;
        m->ev_pool.push_back(r.e0);
        m->ev_pool.push_back(r.e1);
    }
    m->prof_open.clear();
    return rc;
}

int dflash_profile_entry(const dflash_model* m, int32_t i, const char** name, int64_t* launches, double* total_ms,
                         double* total_bytes) {
    if (!m) return DFLASH_EINVAL;
    if (i < 0 || i >= (int32_t)m->prof_sum.size()) return DFLASH_ERANGE;
    const auto& p = m->prof_sum[i];
    if (name) *name = p.name;
    if (launches) *launches = p.launches;
    if (total_ms) *total_ms = p.ms;
    if (total_bytes) *total_bytes = p.bytes;
    return DFLASH_OK;
}

int64_t dflash_launch_count(const dflash_model* m) { return m ? m->launches : -1; }

int dflash_debug_option(dflash_model* m, const char* name, int64_t value) {
    if (!m || !name) return DFLASH_EINVAL;
    const std::string opt(name);
    if (opt == "tc") {
        m->use_tc = value != 0;
    } else if (opt == "dense") {
        m->use_dense = value != 0;

    } else if (opt == "attn_tc_min_keys") {
        if (value < 0) return set_err(m, DFLASH_EINVAL, "attn_tc_min_keys < 0");
        m->tc_attn_min_keys = value;
    } else if (opt == "head_bound") {
        if (value < 0) return set_err(m, DFLASH_EINVAL, "head_bound < 0");
        m->head_bound = std::min<unsigned long long>((unsigned long long)value, 1ull << 48);
    } else {
        return set_err(m, DFLASH_EINVAL, "unknown option " + opt);
    }
    clear_graphs(m);  // the captured kernel sequences may change
    return DFLASH_OK;
}

// ------------------------------------------------------------------ test hooks
int dflash_debug_q4_codes(dflash_model* m, int32_t id, int8_t* codes, uint16_t* scales, void* stream) {
    int rc = check_model(m);
    if (rc) return rc;
    if (m->g.quant != DFLASH_QUANT_Q4G32 || id == DFLASH_MAT_HEAD || !codes || !scales)
        return set_err(m, DFLASH_EINVAL, "not a 4-bit matrix, or NULL output");
    MatView v = mat_view(m, id);
    if (!v.packed) return set_err(m, DFLASH_EINVAL, "bad matrix id");
    cudaStream_t st = (cudaStream_t)stream;
    int8_t* dc = nullptr;
    uint16_t* ds = nullptr;
    CK(m, cudaMalloc(&dc, (size_t)v.N * v.K));
    CK(m, cudaMalloc(&ds, (size_t)v.N * (v.K / 32) * 2));
    int e = q4_unpack(v.packed, v.L, v.tile0, v.N, v.K, dc, ds, st);
    if (!e) e = (int)cudaMemcpyAsync(codes, dc, (size_t)v.N * v.K, cudaMemcpyDeviceToHost, st);
    if (!e) e = (int)cudaMemcpyAsync(scales, ds, (size_t)v.N * (v.K / 32) * 2, cudaMemcpyDeviceToHost, st);
    if (!e) e = (int)cudaStreamSynchronize(st);
    cudaFree(dc);
    cudaFree(ds);
    CK(m, e);
    return DFLASH_OK;
}

int dflash_debug_head_codes(dflash_model* m, int8_t* codes, float* scales, void* stream) {
    int rc = check_model(m);
    if (rc) return rc;
    if (m->g.quant != DFLASH_QUANT_Q4G32 || !codes || !scales) return set_err(m, DFLASH_EINVAL, "f32 model or NULL");
    cudaStream_t st = (cudaStream_t)stream;
    const int V = m->g.vocab, H = m->g.hidden;
    int8_t* dc = nullptr;
    CK(m, cudaMalloc(&dc, (size_t)V * H));
    int e = i8_unpack(m->head_p, V, H, H / kI8KStep, dc, st);
    if (!e) e = (int)cudaMemcpyAsync(codes, dc, (size_t)V * H, cudaMemcpyDeviceToHost, st);
    if (!e) e = (int)cudaMemcpyAsync(scales, m->head_scale, (size_t)V * sizeof(float), cudaMemcpyDeviceToHost, st);
    if (!e) e = (int)cudaStreamSynchronize(st);
    cudaFree(dc);
    CK(m, e);
    return DFLASH_OK;
}

int dflash_debug_q4_groupsums(dflash_model* m, int32_t id, const int8_t* x, int32_t rows, int32_t* out, void* stream) {
    int rc = check_model(m);
    if (rc) return rc;
    if (m->g.quant != DFLASH_QUANT_Q4G32 || id == DFLASH_MAT_HEAD || !x || !out || rows < 1 || rows > 16)
        return set_err(m, DFLASH_EINVAL, "bad arguments");
    MatView v = mat_view(m, id);
    if (!v.packed) return set_err(m, DFLASH_EINVAL, "bad matrix id");
    cudaStream_t st = (cudaStream_t)stream;
    const int ldk = v.L.ksteps * kQ4KStep;
    std::vector<int8_t> hx((size_t)rows * ldk, 0);
    for (int r = 0; r < rows; ++r)
        for (int k = 0; k < v.K; ++k) {
            int xv = x[(size_t)r * v.K + k];
            if (xv < -127) return set_err(m, DFLASH_EINVAL, "activation code -128");
            hx[(size_t)r * ldk + k] = (int8_t)xv;
        }
    std::vector<float> ones(rows, 1.f);
    int8_t* dx = nullptr;
    float* dsc = nullptr;
    int32_t* dout = nullptr;
    const size_t outn = (size_t)rows * v.N * (v.K / 32);
    CK(m, cudaMalloc(&dx, hx.size()));
    CK(m, cudaMalloc(&dsc, rows * sizeof(float)));
    CK(m, cudaMalloc(&dout, outn * sizeof(int32_t)));
    int e = (int)cudaMemcpyAsync(dx, hx.data(), hx.size(), cudaMemcpyHostToDevice, st);
    if (!e) e = (int)cudaMemcpyAsync(dsc, ones.data(), rows * sizeof(float), cudaMemcpyHostToDevice, st);
    QAct qa{dx, dsc, ldk};
    if (!e) e = q4_groupsums(v.packed, v.L, v.tile0, v.N, qa, rows, dout, st);
    if (!e) e = (int)cudaMemcpyAsync(out, dout, outn * sizeof(int32_t), cudaMemcpyDeviceToHost, st);
    if (!e) e = (int)cudaStreamSynchronize(st);
    cudaFree(dx);
    cudaFree(dsc);
    cudaFree(dout);
    CK(m, e);
    return DFLASH_OK;
}

int dflash_debug_q4_matmul(dflash_model* m, int32_t id, const int8_t* x, const float* xs, int32_t rows, float* y,
                           void* stream) {
    int rc = check_model(m);
    if (rc) return rc;
    if (m->g.quant != DFLASH_QUANT_Q4G32 || id == DFLASH_MAT_HEAD || !x || !xs || !y || rows < 1)
        return set_err(m, DFLASH_EINVAL, "bad arguments");
    MatView v = mat_view(m, id);
    if (!v.packed) return set_err(m, DFLASH_EINVAL, "bad matrix id");
    cudaStream_t st = (cudaStream_t)stream;
    const int ldk = v.L.ksteps * kQ4KStep;
    std::vector<int8_t> hx((size_t)rows * ldk, 0);
    for (int r = 0; r < rows; ++r)
        for (int k = 0; k < v.K; ++k) {
            int xv = x[(size_t)r * v.K + k];
            if (xv < -127) return set_err(m, DFLASH_EINVAL, "activation code -128");
            hx[(size_t)r * ldk + k] = (int8_t)xv;
        }
    int8_t* dx = nullptr;
    float* dsc = nullptr;
    float* dy = nullptr;
    const size_t outn = (size_t)rows * v.N;
    CK(m, cudaMalloc(&dx, hx.size()));
    CK(m, cudaMalloc(&dsc, rows * sizeof(float)));
    CK(m, cudaMalloc(&dy, outn * sizeof(float)));
    int e = (int)cudaMemcpyAsync(dx, hx.data(), hx.size(), cudaMemcpyHostToDevice, st);
    if (!e) e = (int)cudaMemcpyAsync(dsc, xs, rows * sizeof(float), cudaMemcpyHostToDevice, st);
    // the streaming kernel adds into y: start from zeros on every path
    if (!e) e = (int)cudaMemsetAsync(dy, 0, outn * sizeof(float), st);
    if (!e && rows > 16) e = ensure_m(m, m->x16, (size_t)rows * ldk * sizeof(__half));
    if (!e && rows > 16) {
        const int drc = ensure_dense(m, st);
        if (drc) {
            cudaFree(dx);
            cudaFree(dsc);
            cudaFree(dy);
            return drc;
        }
    }
    QAct qa{dx, dsc, ldk};
    int lib_rc = DFLASH_OK;
    if (!e) lib_rc = q4_mm(m, v.packed, v.L, v.tile0, v.N, v.K, qa, rows, dy, v.N, false, st);
    if (!e && lib_rc == DFLASH_OK) e = (int)cudaMemcpyAsync(y, dy, outn * sizeof(float), cudaMemcpyDeviceToHost, st);
    if (!e && lib_rc == DFLASH_OK)
        e = (int)cudaMemcpyAsync(m->err_host, m->err_dev, sizeof(int), cudaMemcpyDeviceToHost, st);
    if (!e) e = (int)cudaStreamSynchronize(st);
    cudaFree(dx);
    cudaFree(dsc);
    cudaFree(dy);
    if (lib_rc != DFLASH_OK) return lib_rc;
    CK(m, (cudaError_t)e);
    if (*m->err_host) return device_wait_expired(m);
    return DFLASH_OK;
}

int dflash_debug_wait_expiry(dflash_model* m, int64_t limit_ns, void* stream) {
    int rc = check_model(m);
    if (rc) return rc;
    if (limit_ns < 1000 || limit_ns > 10000000000ll)
        return set_err(m, DFLASH_EINVAL, "limit_ns outside [1 us, 10 s]");
    cudaStream_t st = (cudaStream_t)stream;
    KL(m, "wait_expiry", 1, 0.0, st, wait_expiry(m->err_dev, (uint64_t)limit_ns, st));
    CK(m, cudaMemcpyAsync(m->err_host, m->err_dev, sizeof(int), cudaMemcpyDeviceToHost, st));
    CK(m, cudaStreamSynchronize(st));
    if (*m->err_host) return device_wait_expired(m);
    return DFLASH_OK;
}

int dflash_debug_read_kv(dflash_model* m, const dflash_seq* s, int32_t layer, int64_t pos, int64_t n, float* k,
                         float* v, void* stream) {
    int rc = check_model(m);
    if (rc) return rc;
    if (!s || s->m != m || layer < 0 || layer >= m->g.layers || n < 0)
        return set_err(m, DFLASH_EINVAL, "bad arguments");
    if (pos < s->first || pos + n > s->first + s->len) return set_err(m, DFLASH_ERANGE, "positions not held");
    cudaStream_t st = (cudaStream_t)stream;
    const int hd = m->g.head_dim, kv = m->g.kv_heads;
    const int64_t idx = pos - s->first;
    const size_t plane = (size_t)kv * s->cap * hd;
    // each stored value is the pair (hi, lo): the value read back is hi + lo,
    // summed in f32 (exact: the two halves' bits fit one f32 significand)
    std::vector<__half> hh((size_t)n * kv * hd), hl((size_t)n * kv * hd);
    for (int which = 0; which < 2; ++which) {
        float* dst = which ? v : k;
        const __half* src = which ? s->v[layer] : s->k[layer];
        if (!dst || n == 0) continue;
        for (int part = 0; part < 2; ++part) {
            __half* h = part ? hl.data() : hh.data();
            for (int gq = 0; gq < kv; ++gq)
                CK(m, cudaMemcpy2DAsync(h + (size_t)gq * hd, (size_t)kv * hd * sizeof(__half),
                                        src + part * plane + ((size_t)gq * s->cap + idx) * hd,
                                        (size_t)hd * sizeof(__half), (size_t)hd * sizeof(__half), (size_t)n,
                                        cudaMemcpyDeviceToHost, st));
        }
        CK(m, cudaStreamSynchronize(st));
        for (size_t i = 0; i < hh.size(); ++i) dst[i] = __half2float(hh[i]) + __half2float(hl[i]);
    }
    CK(m, cudaStreamSynchronize(st));
    return DFLASH_OK;
}

}  // extern "C"

// ============================================================================
// The block's attention without any allocation.
//
// Some callers cannot allocate device memory at the moment they need the
// attention: processes in which a host framework owns every device byte
// through its own pool allocator (a cudaMalloc behind its back can fail, or
// take memory the pool has already promised elsewhere), and latency-critical
// loops that must never block in the allocator or synchronise the device, as
// cudaMalloc and cudaFree can.  For them, dflash_attention_noalloc runs the
// same attention kernels as dflash_debug_attention, but its scratch (the
// per-sequence context views and the split partials) lives in the fixed
// array below, which is part of this library's device image: every GPU that
// loads the library holds these 16 MiB until the process exits.
// ============================================================================
namespace {

constexpr int64_t kNoAllocFloats = int64_t(4) << 20;  // 16 MiB of f32 scratch
constexpr int64_t kNoAllocViewFloats = 4096;           // the first 16 KiB hold the context views
constexpr int kNoAllocMaxSeqs = kViewsMax;             // 256 views * 40 B fit in those 16 KiB
constexpr int kNoAllocMaxDevices = 64;
static_assert(kNoAllocMaxSeqs * sizeof(AttnSeq) <= kNoAllocViewFloats * sizeof(float), "view area");

std::mutex g_noalloc_mutex;
float* g_noalloc_base[kNoAllocMaxDevices] = {};

}  // namespace

static __device__ __align__(256) float g_noalloc_scratch[kNoAllocFloats];

namespace {

// The device address of the fixed array on `device` (which must be current):
// looked up once per device, then reused.  In host code the array's name is
// only a host-side stand-in, so kernels must be given this address.
int noalloc_base(int device, float** out) {
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (device < 0 || device >= kNoAllocMaxDevices) return (int)cudaErrorInvalidDevice;
    if (!g_noalloc_base[device]) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return (int)e;
        g_noalloc_base[device] = static_cast<float*>(p);
    }
    *out = g_noalloc_base[device];
    return 0;
}

}  // namespace

int dflash_attention_noalloc(dflash_model* m, dflash_seq* const* seqs, int32_t n_seqs, int32_t layer,
                             const int64_t* anchor_pos, int32_t block_len, const float* qkv, float* y, void* stream) {
    int rc = check_model(m);
    if (rc) return rc;
    std::vector<AttnSeq> views;
    int max_ctx = 0;
    rc = attention_views(m, seqs, n_seqs, layer, anchor_pos, block_len, qkv, y, views, &max_ctx);
    if (rc) return rc;
    if (n_seqs > kNoAllocMaxSeqs)
        return set_err(m, DFLASH_ERANGE, "attention without allocation: " + std::to_string(n_seqs) +
                                             " sequences, at most " + std::to_string(kNoAllocMaxSeqs));
    const dflash_geometry& g = m->g;
    // the fixed array's room for the key splits' partial rows: a call whose
    // rows do not fit runs the cluster merge, which needs none (on 152 SMs the
    // split plan needs at most ~3.8 Mi floats, so it always fits there)
    const int64_t part_floats = kNoAllocFloats - kNoAllocViewFloats;
    float* base = nullptr;
    CK(m, noalloc_base(m->device, &base));
    cudaStream_t st = (cudaStream_t)stream;
    AttnSeq* views_dev = reinterpret_cast<AttnSeq*>(base);
    // The array's head takes the context views, passed by value to a small
    // kernel (no host buffer has to outlive the call); the attention reads
    // them after its dependency wait.  The rest holds the key splits' partial
    // rows when a long context splits the keys over more CTAs than clusters
    // place (each launch writes them before the merge reads them, so nothing
    // in it needs to start at zero); otherwise the splits merge in
    // distributed shared memory and the rest is not read.
    AttnViews byval;
    byval.n = n_seqs;
    std::copy(views.begin(), views.end(), byval.v);
    KL(m, "attn_views", 1, (double)n_seqs * sizeof(AttnSeq), st, attn_views_store(byval, views_dev, st));
    KL(m, "attention_noalloc",
       attn_kernels(n_seqs, block_len, max_ctx, g.heads, g.kv_heads, g.head_dim, m->num_sms, part_floats), 0.0, st,
       attention(qkv, m->qkv_w, n_seqs, block_len, views_dev, max_ctx, g.heads, g.kv_heads, g.head_dim,
                 1.0f / sqrtf((float)g.head_dim), base + kNoAllocViewFloats, part_floats, y, m->num_sms, st, nullptr,
                 nullptr, nullptr, 0.f, false, m->win[layer] > 0));
    return DFLASH_OK;
}
