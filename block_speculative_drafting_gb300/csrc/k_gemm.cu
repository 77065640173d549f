// Matmuls of the drafter.
//
// q4_gemm: the 4-bit g32 x int8 matvec over up to 16 rows at a time (page
// "cortiq-engine 0.8.75 — src/gpu_wgpu/dflash_dev.rs", `Dev::q4`: the
// block's rows against a four-bit matrix, int8 activations), here on the
// tensor cores: weight rows are the MMA's M (16 per warp tile), the block's
// rows its N (2 x 8), one 32-column quantisation group two m16n8k16 steps.
// Codes enter the MMA as exact f16 integers (weights -8..7, activations
// -127..127), so each group's sum -- at most 32 * 8 * 127 in magnitude -- is
// an exact integer in the f32 fragment; that integer is the format's int32
// group sum, and it is scaled by the group's f16 scale into the f32
// accumulator: y = xs * sum_g s_g * acc_g.
//
// head_i8: the int8-per-row head (page "cortiq-engine 0.8.71 —
// src/dflash.rs", `block_dev`: the logits of the draft rows over the whole
// head) on s8 MMAs with exact int32 accumulation, fused with the draft
// token's argmax (lowest index among equal values, as `top_k` keeps the first
// of equals).
#include <algorithm>

#include "common.cuh"
#include "kernels.cuh"

namespace dflash {

constexpr int kGemmWarps = 8;
constexpr int kXPadHalves = 32;  // row pad of the staged activations: conflict-free 16-byte fragment loads
constexpr int kMaxKstepsPerCta = 64;

template <bool kGroupSums>
__global__ void __launch_bounds__(256) q4_gemm16_kernel(const uint8_t* __restrict__ wp, Q4Layout L, int tile0,
                                                        int ntiles, int N, QAct x, int T, float* __restrict__ y,
                                                        int ldy, int ksteps_per_split, int accumulate,
                                                        int32_t* __restrict__ gsum) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __half* xsm = reinterpret_cast<__half*>(smem_raw);
    const int ksteps = L.ksteps;
    const int ks0 = blockIdx.y * ksteps_per_split;
    const int ks1 = min(ks0 + ksteps_per_split, ksteps);
    const int nks = ks1 - ks0;
    const int ld = nks * kQ4KStep + kXPadHalves;
    const int tok0 = blockIdx.z * 16;
    pdl_trigger();
    pdl_wait();
    // stage the 16 rows' codes of this k range as exact f16 (rows past T are zero)
    const int vecs = nks * (kQ4KStep / 8);
    for (int i = threadIdx.x; i < 16 * vecs; i += blockDim.x) {
        const int r = i / vecs, c = i - r * vecs;
        uint2 v = make_uint2(0u, 0u);
        if (tok0 + r < T)
            v = *reinterpret_cast<const uint2*>(x.codes + (int64_t)(tok0 + r) * x.ld + ks0 * kQ4KStep + c * 8);
        uint4 h;
        i8x4_to_half2x2(v.x, h.x, h.y);
        i8x4_to_half2x2(v.y, h.z, h.w);
        *reinterpret_cast<uint4*>(xsm + r * ld + c * 8) = h;
    }
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile = blockIdx.x * kGemmWarps + warp;
    if (tile >= ntiles) return;  // no block-wide barrier below
    const int gq = lane >> 2, tq = lane & 3;
    const __half* xr0 = xsm + gq * ld + 8 * tq;        // B fragment rows: block rows gq (n half 0)
    const __half* xr1 = xsm + (gq + 8) * ld + 8 * tq;  // and gq + 8 (n half 1)
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    const float zero[4] = {0.f, 0.f, 0.f, 0.f};

#pragma unroll 4
    for (int j = 0; j < nks; ++j) {
        const uint8_t* chunk = wp + q4_chunk_offset(L, tile0 + tile, ks0 + j);
        const uint4 wv = ldg_stream_v4(chunk + lane * 16);
        const uint2 sv = ldg_stream_v2(chunk + 512 + gq * 8);
        const uint32_t wds[4] = {wv.x, wv.y, wv.z, wv.w};
        const uint32_t svs[2] = {sv.x, sv.y};
#pragma unroll
        for (int gi = 0; gi < 2; ++gi) {
            uint32_t a0[4], a1[4];
            unpack_q4_word(wds[gi * 2 + 0], a0);
            unpack_q4_word(wds[gi * 2 + 1], a1);
            const int kc = j * kQ4KStep + gi * 32;
            const uint4 b0 = *reinterpret_cast<const uint4*>(xr0 + kc);
            const uint4 b1 = *reinterpret_cast<const uint4*>(xr1 + kc);
            float d0[4], d1[4];
            mma_f16_16816(d0, a0, b0.x, b0.y, zero);
            mma_f16_16816(d0, a1, b0.z, b0.w, d0);
            mma_f16_16816(d1, a0, b1.x, b1.y, zero);
            mma_f16_16816(d1, a1, b1.z, b1.w, d1);
            if constexpr (kGroupSums) {
                const int G = ksteps * 2, g = (ks0 + j) * 2 + gi;
                const int n0 = tile * 16 + gq, n1 = n0 + 8;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float* d = h ? d1 : d0;
                    const int t0 = tok0 + h * 8 + 2 * tq, t1 = t0 + 1;
                    if (n0 < N && t0 < T) gsum[((int64_t)t0 * N + n0) * G + g] = (int32_t)d[0];
                    if (n0 < N && t1 < T) gsum[((int64_t)t1 * N + n0) * G + g] = (int32_t)d[1];
                    if (n1 < N && t0 < T) gsum[((int64_t)t0 * N + n1) * G + g] = (int32_t)d[2];
                    if (n1 < N && t1 < T) gsum[((int64_t)t1 * N + n1) * G + g] = (int32_t)d[3];
                }
            } else {
                uint32_t sbits = svs[gi];
                const float2 sc = __half22float2(*reinterpret_cast<const __half2*>(&sbits));  // rows gq, gq+8
                acc[0][0] = fmaf(sc.x, d0[0], acc[0][0]);
                acc[0][1] = fmaf(sc.x, d0[1], acc[0][1]);
                acc[0][2] = fmaf(sc.y, d0[2], acc[0][2]);
                acc[0][3] = fmaf(sc.y, d0[3], acc[0][3]);
                acc[1][0] = fmaf(sc.x, d1[0], acc[1][0]);
                acc[1][1] = fmaf(sc.x, d1[1], acc[1][1]);
                acc[1][2] = fmaf(sc.y, d1[2], acc[1][2]);
                acc[1][3] = fmaf(sc.y, d1[3], acc[1][3]);
            }
        }
    }
    if constexpr (!kGroupSums) {
        const int n0 = tile * 16 + gq, n1 = n0 + 8;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int t0 = tok0 + h * 8 + 2 * tq, t1 = t0 + 1;
            const float s0 = t0 < T ? x.scale[t0] : 0.f, s1 = t1 < T ? x.scale[t1] : 0.f;
            const float v[4] = {acc[h][0] * s0, acc[h][1] * s1, acc[h][2] * s0, acc[h][3] * s1};
            const int tt[4] = {t0, t1, t0, t1};
            const int nn[4] = {n0, n0, n1, n1};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (tt[e] < T && nn[e] < N) {
                    float* p = y + (int64_t)tt[e] * ldy + nn[e];
                    if (accumulate)
                        atomicAdd(p, v[e]);
                    else
                        *p = v[e];
                }
            }
        }
    }
}

static size_t q4_smem_bytes(int kps) { return (size_t)16 * (kps * kQ4KStep + kXPadHalves) * sizeof(__half); }

static void q4_set_smem_limits() {
    static size_t limit0 = 0, limit1 = 0;
    const size_t bytes = q4_smem_bytes(kMaxKstepsPerCta);
    raise_smem_limit(q4_gemm16_kernel<false>, bytes, &limit0);
    raise_smem_limit(q4_gemm16_kernel<true>, bytes, &limit1);
}

int q4_gemm(const uint8_t* packed, Q4Layout L, int tile0, int N, QAct x, int T, float* y, int ldy, bool accumulate,
            int num_sms, cudaStream_t st) {
    if (T <= 0 || N <= 0) return 0;
    q4_set_smem_limits();
    const int ksteps = L.ksteps;
    const int ntiles = (N + 15) / 16;
    const int nblk = (ntiles + kGemmWarps - 1) / kGemmWarps;
    const int tchunks = (T + 15) / 16;
    // split K so that the grid covers the SMs about twice, no CTA holding more than 64 k-steps
    int ksplit = (2 * num_sms + nblk * tchunks - 1) / (nblk * tchunks);
    ksplit = std::max(1, std::min(ksplit, std::max(1, ksteps / 4)));
    ksplit = std::max(ksplit, (ksteps + kMaxKstepsPerCta - 1) / kMaxKstepsPerCta);
    const int kps = (ksteps + ksplit - 1) / ksplit;
    ksplit = (ksteps + kps - 1) / kps;
    int acc_mode = accumulate ? 1 : 0;
    if (ksplit > 1 && !accumulate) {
        cudaError_t e = cudaMemset2DAsync(y, (size_t)ldy * sizeof(float), 0, (size_t)N * sizeof(float), T, st);
        if (e != cudaSuccess) return (int)e;
        acc_mode = 1;
    }
    dim3 grid(nblk, ksplit, tchunks);
    return (int)launch(q4_gemm16_kernel<false>, grid, dim3(256), q4_smem_bytes(kps), st, packed, L, tile0, ntiles, N,
                       x, T, y, ldy, kps, acc_mode, (int32_t*)nullptr);
}

int q4_groupsums(const uint8_t* packed, Q4Layout L, int tile0, int N, QAct x, int T, int32_t* out, cudaStream_t st) {
    q4_set_smem_limits();
    const int ksteps = L.ksteps;
    const int ntiles = (N + 15) / 16;
    const int nblk = (ntiles + kGemmWarps - 1) / kGemmWarps;
    const int ksplit = (ksteps + kMaxKstepsPerCta - 1) / kMaxKstepsPerCta;
    const int kps = (ksteps + ksplit - 1) / ksplit;
    dim3 grid(nblk, (ksteps + kps - 1) / kps, (T + 15) / 16);
    return (int)launch(q4_gemm16_kernel<true>, grid, dim3(256), q4_smem_bytes(kps), st, packed, L, tile0, ntiles, N,
                       x, T, (float*)nullptr, 0, kps, 0, out);
}

// ------------------------------------------------------------------ f32 path
constexpr int kLinTok = 8;

// A CTA an output n and up to kLinTok rows: its eight warps take eighths of
// K (float4 a lane), and the CTA adds the warps' sums.
__global__ void __launch_bounds__(256) linear_f32_kernel(const float* __restrict__ W, int N, int K,
                                                         const float* __restrict__ x, int ldx, int T,
                                                         float* __restrict__ y, int ldy, int accumulate) {
    __shared__ float part[8][kLinTok];
    const int n = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_trigger();
    pdl_wait();
    const int t0 = blockIdx.y * kLinTok;
    float acc[kLinTok];
#pragma unroll
    for (int i = 0; i < kLinTok; ++i) acc[i] = 0.f;
    const float* wr = W + (int64_t)n * K;
    const int k4 = K / 4, per = (k4 + 7) / 8, lo = warp * per, hi = min(k4, lo + per);
    for (int c = lo + lane; c < hi; c += 32) {
        const float4 w = reinterpret_cast<const float4*>(wr)[c];
#pragma unroll
        for (int i = 0; i < kLinTok; ++i) {
            if (t0 + i < T) {
                const float4 v = reinterpret_cast<const float4*>(x + (int64_t)(t0 + i) * ldx)[c];
                acc[i] = fmaf(w.x, v.x, fmaf(w.y, v.y, fmaf(w.z, v.z, fmaf(w.w, v.w, acc[i]))));
            }
        }
    }
#pragma unroll
    for (int i = 0; i < kLinTok; ++i) {
        const float s = warp_sum(acc[i]);
        if (lane == 0) part[warp][i] = s;
    }
    __syncthreads();
    if (threadIdx.x < kLinTok && t0 + (int)threadIdx.x < T) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) s += part[w][threadIdx.x];
        float* p = y + (int64_t)(t0 + threadIdx.x) * ldy + n;
        *p = accumulate ? *p + s : s;
    }
}

int linear_f32(const float* W, int N, int K, const float* x, int ldx, int T, float* y, int ldy, bool accumulate,
               cudaStream_t st) {
    if (T <= 0 || N <= 0) return 0;
    if (K % 4 || ldx % 4 || (reinterpret_cast<uintptr_t>(W) & 15) || (reinterpret_cast<uintptr_t>(x) & 15))
        return (int)cudaErrorInvalidValue;
    dim3 grid(N, (T + kLinTok - 1) / kLinTok);
    return (int)launch(linear_f32_kernel, grid, dim3(256), 0, st, W, N, K, x, ldx, T, y, ldy, accumulate ? 1 : 0);
}

__global__ void argmax_rows_kernel(const float* __restrict__ logits, int ldl, int V,
                                   unsigned long long* __restrict__ keys) {
    __shared__ unsigned long long red[32];
    const int t = blockIdx.x;
    pdl_trigger();
    pdl_wait();
    unsigned long long b = 0ull;
    for (int n = threadIdx.x; n < V; n += blockDim.x) b = max(b, argmax_key(logits[(int64_t)t * ldl + n], (uint32_t)n));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) b = max(b, __shfl_xor_sync(0xffffffffu, b, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = b;
    __syncthreads();
    if (threadIdx.x < 32) {
        b = threadIdx.x < blockDim.x / 32 ? red[threadIdx.x] : 0ull;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) b = max(b, __shfl_xor_sync(0xffffffffu, b, o));
        if (threadIdx.x == 0) keys[t] = b;
    }
}

int argmax_rows(const float* logits, int ldl, int V, int T, unsigned long long* keys, cudaStream_t st) {
    if (T <= 0) return 0;
    return (int)launch(argmax_rows_kernel, dim3(T), dim3(256), 0, st, logits, ldl, V, keys);
}

__global__ void keys_to_tokens_kernel(const unsigned long long* __restrict__ keys, int T, uint32_t* __restrict__ tok) {
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    pdl_trigger();
    pdl_wait();
    if (t < T) tok[t] = 0xFFFFFFFFu - (uint32_t)(keys[t] & 0xFFFFFFFFull);
}

int keys_to_tokens(const unsigned long long* keys, int T, uint32_t* tokens, cudaStream_t st) {
    if (T <= 0) return 0;
    return (int)launch(keys_to_tokens_kernel, dim3((T + 255) / 256), dim3(256), 0, st, keys, T, tokens);
}

// ------------------------------------------------------------------ candidate selector
// Per row, its K largest logits as argmax keys, largest first (the lower
// index first among equal values: page "cortiq-engine 0.8.71 — src/dflash.rs",
// `top_k`).  A CTA a row: each thread keeps the K best of its strided share
// (a compare-exchange pass a candidate), which holds every row-wide top-K
// element of that share; then k rounds of a CTA-wide maximum over the
// threads' lists, each round taking out its winner.
template <int K>
struct TopShape {
    static constexpr int kThreads = K >= 32 ? 128 : 256;  // the lists in 32 KB of shared memory at most
};
// Phase 1 (logits != nullptr): CTA (t, part) over the part-th of row t's
// columns, its k best into out[(t * parts + part) * k ..].  Phase 2 (logits
// == nullptr): CTA t over the parts * k keys of phase 1 (`keys`), the row's
// k best into out[t * k ..].  Either keeps the exact top k: a key among the
// row's best k is among its part's best k.
template <int K>
__global__ void __launch_bounds__(TopShape<K>::kThreads) topk_rows_kernel(const float* __restrict__ logits, int ldl,
                                                                           int V, int k, int parts,
                                                                           const unsigned long long* __restrict__ keys,
                                                                           unsigned long long* __restrict__ out) {
    constexpr int kTopThreads = TopShape<K>::kThreads;
    __shared__ unsigned long long cand[kTopThreads * K];
    __shared__ unsigned long long red[kTopThreads / 32];
    const int t = blockIdx.x, tid = threadIdx.x;
    pdl_trigger();
    pdl_wait();
    unsigned long long mine[K];
#pragma unroll
    for (int i = 0; i < K; ++i) mine[i] = 0ull;  // no real key is 0 (its index part is below 2^32 - 1 - V)
    const float* row = logits ? logits + (int64_t)t * ldl : nullptr;
    const int chunk = logits ? (V + parts - 1) / parts : parts * k;
    const int c0 = logits ? blockIdx.y * chunk : 0, c1 = logits ? min(V, c0 + chunk) : parts * k;
    for (int n = c0 + tid; n < c1; n += kTopThreads) {
        unsigned long long x = logits ? argmax_key(row[n], (uint32_t)n) : keys[(int64_t)t * parts * k + n];
        if (x <= mine[K - 1]) continue;
#pragma unroll
        for (int i = 0; i < K; ++i) {
            const unsigned long long hi = max(x, mine[i]), lo = min(x, mine[i]);
            mine[i] = hi;
            x = lo;
        }
    }
#pragma unroll
    for (int i = 0; i < K; ++i) cand[tid * K + i] = mine[i];
    __syncthreads();
    for (int r = 0; r < k; ++r) {
        unsigned long long b = 0ull;
#pragma unroll
        for (int i = 0; i < K; ++i) b = max(b, cand[tid * K + i]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) b = max(b, __shfl_xor_sync(0xffffffffu, b, o));
        if ((tid & 31) == 0) red[tid >> 5] = b;
        __syncthreads();
        b = 0ull;
#pragma unroll
        for (int w = 0; w < kTopThreads / 32; ++w) b = max(b, red[w]);
        if (tid == 0) out[((int64_t)t * gridDim.y + blockIdx.y) * k + r] = b;
#pragma unroll
        for (int i = 0; i < K; ++i)
            if (cand[tid * K + i] == b) cand[tid * K + i] = 0ull;  // keys are unique: its one owner
        __syncthreads();
    }
}

template <int K>
static int topk_two_phase(const float* logits, int ldl, int V, int T, int k, int parts, unsigned long long* scratch,
                          unsigned long long* out, cudaStream_t st) {
    constexpr int nt = TopShape<K>::kThreads;
    cudaError_t e = launch(topk_rows_kernel<K>, dim3(T, parts), dim3(nt), 0, st, logits, ldl, V, k, parts,
                           (const unsigned long long*)nullptr, scratch);
    if (e != cudaSuccess) return (int)e;
    return (int)launch(topk_rows_kernel<K>, dim3(T, 1), dim3(nt), 0, st, (const float*)nullptr, 0, V, k, parts,
                       (const unsigned long long*)scratch, out);
}

int topk_parts(int V, int k) { return std::max(1, std::min(32, V / (8 * k))); }

int topk_rows(const float* logits, int ldl, int V, int T, int k, unsigned long long* scratch, unsigned long long* out,
              cudaStream_t st) {
    if (T <= 0) return 0;
    if (k < 1 || k > 32 || k > V) return (int)cudaErrorInvalidValue;
    const int parts = topk_parts(V, k);
    if (k <= 8) return topk_two_phase<8>(logits, ldl, V, T, k, parts, scratch, out, st);
    if (k <= 16) return topk_two_phase<16>(logits, ldl, V, T, k, parts, scratch, out, st);
    return topk_two_phase<32>(logits, ldl, V, T, k, parts, scratch, out, st);
}

// The selector's choices, a warp a sequence (its rows one after another):
// row j's candidates (lane c: the c-th) scored unary + sum_i (P[prev][i] *
// hp[j][i]) * C[tok][i] in f32 as the page sums (products rounded, added in
// order i), the best taken (the first candidate among equals) and fed to the
// next row; the anchor is the first row's prev.
// (An anchor outside [0, V), possible only for anchors already on the device,
// has a predecessor row of zeros.)
__global__ void select_kernel(const unsigned long long* __restrict__ cand, int k, const float* __restrict__ hp,
                              int rank, const __half* __restrict__ book_p, const __half* __restrict__ book_c, int V,
                              const uint32_t* __restrict__ anchors, int n_seqs, int rows, uint32_t* __restrict__ chosen,
                              uint32_t* __restrict__ plain) {
    const int s = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    pdl_trigger();
    pdl_wait();
    if (s >= n_seqs) return;
    uint32_t prev = anchors[s];
    for (int j = 0; j < rows; ++j) {
        const int r = s * rows + j;
        float best = -INFINITY;
        uint32_t best_t = 0;
        for (int c0 = 0; c0 < k; c0 += 32) {
            const int c = c0 + lane;
            float sc = -INFINITY;
            uint32_t tok = 0;
            if (c < k) {
                const unsigned long long key = cand[(int64_t)r * k + c];
                tok = 0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull);
                const float unary = float_of_order_key((uint32_t)(key >> 32));
                const __half* pp = book_p + (int64_t)prev * rank;
                const __half* cc = book_c + (int64_t)tok * rank;
                const float* hh = hp + (int64_t)r * rank;
                float acc = 0.f;
                if (prev < (uint32_t)V)
                    for (int i = 0; i < rank; ++i)
                        acc = __fadd_rn(acc, __fmul_rn(__fmul_rn(__half2float(pp[i]), hh[i]), __half2float(cc[i])));
                sc = __fadd_rn(unary, acc);
            }
            // the best of these 32 (the lowest candidate among equals), then against the earlier ones
            float v = sc;
            int vc = c < k ? c : 0x7FFFFFFF;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, v, o);
                const int oc = __shfl_xor_sync(0xffffffffu, vc, o);
                if (ov > v || (ov == v && oc < vc)) {
                    v = ov;
                    vc = oc;
                }
            }
            const uint32_t vt = __shfl_sync(0xffffffffu, tok, vc & 31);
            if (c0 == 0) {
                // the first candidate stands unless one scores strictly higher
                best_t = __shfl_sync(0xffffffffu, tok, 0);
                if (v > -INFINITY) {
                    best = v;
                    best_t = vt;
                }
            } else if (v > best) {
                best = v;
                best_t = vt;
            }
            if (c0 == 0 && lane == 0) plain[r] = tok;
        }
        prev = best_t;
        if (lane == 0) chosen[r] = prev;
    }
}

int select_tokens(const unsigned long long* cand, int k, const float* hp, int rank, const __half* book_p,
                  const __half* book_c, int V, const uint32_t* anchors, int n_seqs, int rows, uint32_t* chosen,
                  uint32_t* plain, cudaStream_t st) {
    if (n_seqs <= 0 || rows <= 0) return 0;
    if (k < 1 || k > 32 || rank < 1) return (int)cudaErrorInvalidValue;
    const int warps = 4;
    return (int)launch(select_kernel, dim3((n_seqs + warps - 1) / warps), dim3(32 * warps), 0, st, cand, k, hp, rank,
                       book_p, book_c, V, anchors, n_seqs, rows, chosen, plain);
}

}  // namespace dflash
