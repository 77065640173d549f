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
__global__ void __launch_bounds__(256) q4_gemm16_kernel(const uint8_t* __restrict__ wp, int ntiles, int ksteps, int N,
                                                        QAct x, int T, float* __restrict__ y, int ldy,
                                                        int ksteps_per_split, int accumulate,
                                                        int32_t* __restrict__ gsum) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __half* xsm = reinterpret_cast<__half*>(smem_raw);
    const int ks0 = blockIdx.y * ksteps_per_split;
    const int ks1 = min(ks0 + ksteps_per_split, ksteps);
    const int nks = ks1 - ks0;
    const int ld = nks * kQ4KStep + kXPadHalves;
    const int tok0 = blockIdx.z * 16;
    // stage the 16 rows' codes of this k range (rows past T are zero)
    const int vecs = nks * (kQ4KStep / 8);
    for (int i = threadIdx.x; i < 16 * vecs; i += blockDim.x) {
        const int r = i / vecs, c = i - r * vecs;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (tok0 + r < T)
            v = *reinterpret_cast<const uint4*>(x.codes + (int64_t)(tok0 + r) * x.ld + ks0 * kQ4KStep + c * 8);
        *reinterpret_cast<uint4*>(xsm + r * ld + c * 8) = v;
    }
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile = blockIdx.x * kGemmWarps + warp;
    if (tile >= ntiles) return;  // no block-wide barrier below
    const int gq = lane >> 2, tq = lane & 3;
    const uint8_t* wt = wp + ((int64_t)tile * ksteps + ks0) * kQ4Chunk;
    const __half* xr0 = xsm + gq * ld + 8 * tq;        // B fragment rows: block rows gq (n half 0)
    const __half* xr1 = xsm + (gq + 8) * ld + 8 * tq;  // and gq + 8 (n half 1)
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    const float zero[4] = {0.f, 0.f, 0.f, 0.f};

#pragma unroll 4
    for (int j = 0; j < nks; ++j) {
        const uint8_t* chunk = wt + (int64_t)j * kQ4Chunk;
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
    static bool done = false;
    if (done) return;
    const int bytes = (int)q4_smem_bytes(kMaxKstepsPerCta);
    cudaFuncSetAttribute(q4_gemm16_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    cudaFuncSetAttribute(q4_gemm16_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    done = true;
}

int q4_gemm(const uint8_t* packed, int tile0, int N, int ksteps, QAct x, int T, float* y, int ldy, bool accumulate,
            int num_sms, cudaStream_t st) {
    if (T <= 0 || N <= 0) return 0;
    q4_set_smem_limits();
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
    q4_gemm16_kernel<false><<<grid, 256, q4_smem_bytes(kps), st>>>(packed + (int64_t)tile0 * ksteps * kQ4Chunk,
                                                                     ntiles, ksteps, N, x, T, y, ldy, kps, acc_mode,
                                                                     nullptr);
    return (int)cudaGetLastError();
}

int q4_groupsums(const uint8_t* packed, int tile0, int N, int ksteps, QAct x, int T, int32_t* out, cudaStream_t st) {
    q4_set_smem_limits();
    const int ntiles = (N + 15) / 16;
    const int nblk = (ntiles + kGemmWarps - 1) / kGemmWarps;
    const int ksplit = (ksteps + kMaxKstepsPerCta - 1) / kMaxKstepsPerCta;
    const int kps = (ksteps + ksplit - 1) / ksplit;
    dim3 grid(nblk, (ksteps + kps - 1) / kps, (T + 15) / 16);
    q4_gemm16_kernel<true><<<grid, 256, q4_smem_bytes(kps), st>>>(packed + (int64_t)tile0 * ksteps * kQ4Chunk, ntiles,
                                                                    ksteps, N, x, T, nullptr, 0, kps, 0, out);
    return (int)cudaGetLastError();
}

// ------------------------------------------------------------------ head
constexpr int kHeadXPad = 32;  // bytes: conflict-free 8-byte fragment loads

__global__ void __launch_bounds__(256) head_i8_kernel(const int8_t* __restrict__ wp, const float* __restrict__ sw,
                                                      int ntiles, int ksteps, int V, QAct x, int T,
                                                      float* __restrict__ logits, int ldl,
                                                      unsigned long long* __restrict__ keys) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    int8_t* xsm = reinterpret_cast<int8_t*>(smem_raw);
    const int K = ksteps * kI8KStep;
    const int ldb = K + kHeadXPad;
    const int tok0 = blockIdx.y * 16;
    for (int i = threadIdx.x; i < 16 * (K / 2); i += blockDim.x) {
        const int r = i / (K / 2), c = (i - r * (K / 2)) * 2;
        char2 v = make_char2(0, 0);
        if (tok0 + r < T) {
            const __half2 h = *reinterpret_cast<const __half2*>(x.codes + (int64_t)(tok0 + r) * x.ld + c);
            v = make_char2((signed char)__half2int_rn(h.x), (signed char)__half2int_rn(h.y));
        }
        *reinterpret_cast<char2*>(xsm + r * ldb + c) = v;
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gq = lane >> 2, tq = lane & 3;
    const int8_t* xr0 = xsm + gq * ldb + 8 * tq;
    const int8_t* xr1 = xsm + (gq + 8) * ldb + 8 * tq;
    float xs_tok[4];
    int tk[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        tk[e] = tok0 + (e >> 1) * 8 + 2 * tq + (e & 1);
        xs_tok[e] = tk[e] < T ? x.scale[tk[e]] : 0.f;
    }
    unsigned long long best[4] = {0ull, 0ull, 0ull, 0ull};
    for (int tile = blockIdx.x * kGemmWarps + warp; tile < ntiles; tile += gridDim.x * kGemmWarps) {
        const int8_t* wt = wp + (int64_t)tile * ksteps * kI8Chunk + lane * 16;
        int d0[4] = {0, 0, 0, 0}, d1[4] = {0, 0, 0, 0};
#pragma unroll 8
        for (int j = 0; j < ksteps; ++j) {
            const uint4 a = ldg_stream_v4(wt + (int64_t)j * kI8Chunk);
            const uint2 b0 = *reinterpret_cast<const uint2*>(xr0 + j * kI8KStep);
            const uint2 b1 = *reinterpret_cast<const uint2*>(xr1 + j * kI8KStep);
            mma_s8_16832(d0, a, b0.x, b0.y);
            mma_s8_16832(d1, a, b1.x, b1.y);
        }
        const int n0 = tile * 16 + gq, n1 = n0 + 8;
        const float sw0 = n0 < V ? sw[n0] : 0.f, sw1 = n1 < V ? sw[n1] : 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int* d = (e >> 1) ? d1 : d0;
            const int c = e & 1;
            const float l0 = xs_tok[e] * sw0 * (float)d[c];      // row n0
            const float l1 = xs_tok[e] * sw1 * (float)d[2 + c];  // row n1
            if (tk[e] < T) {
                if (n0 < V) {
                    if (logits) logits[(int64_t)tk[e] * ldl + n0] = l0;
                    best[e] = max(best[e], argmax_key(l0, (uint32_t)n0));
                }
                if (n1 < V) {
                    if (logits) logits[(int64_t)tk[e] * ldl + n1] = l1;
                    best[e] = max(best[e], argmax_key(l1, (uint32_t)n1));
                }
            }
        }
    }
    if (keys) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            unsigned long long b = best[e];
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) b = max(b, __shfl_xor_sync(0xffffffffu, b, o));
            if (gq == 0 && tk[e] < T && b) atomicMax(keys + tk[e], b);
        }
    }
}

int head_i8(const int8_t* packed, const float* row_scale, int V, int ksteps, QAct x, int T, float* logits, int ldl,
            unsigned long long* keys, int num_sms, cudaStream_t st) {
    if (T <= 0) return 0;
    const size_t smem = (size_t)16 * (ksteps * kI8KStep + kHeadXPad);
    static size_t limit_set = 0;
    if (smem > limit_set) {
        cudaFuncSetAttribute(head_i8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        limit_set = smem;
    }
    const int ntiles = (V + 15) / 16;
    const int nblk = std::min((ntiles + kGemmWarps - 1) / kGemmWarps, 2 * num_sms);
    dim3 grid(nblk, (T + 15) / 16);
    head_i8_kernel<<<grid, 256, smem, st>>>(packed, row_scale, ntiles, ksteps, V, x, T, logits, ldl, keys);
    return (int)cudaGetLastError();
}

// ------------------------------------------------------------------ f32 path
constexpr int kLinTok = 8;

__global__ void __launch_bounds__(256) linear_f32_kernel(const float* __restrict__ W, int N, int K,
                                                         const float* __restrict__ x, int ldx, int T,
                                                         float* __restrict__ y, int ldy, int accumulate) {
    const int n = (int)((blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (n >= N) return;
    const int t0 = blockIdx.y * kLinTok;
    float acc[kLinTok];
#pragma unroll
    for (int i = 0; i < kLinTok; ++i) acc[i] = 0.f;
    const float* wr = W + (int64_t)n * K;
    for (int k = lane * 4; k < K; k += 128) {
        const float4 w = *reinterpret_cast<const float4*>(wr + k);
#pragma unroll
        for (int i = 0; i < kLinTok; ++i) {
            if (t0 + i < T) {
                const float4 v = *reinterpret_cast<const float4*>(x + (int64_t)(t0 + i) * ldx + k);
                acc[i] = fmaf(w.x, v.x, fmaf(w.y, v.y, fmaf(w.z, v.z, fmaf(w.w, v.w, acc[i]))));
            }
        }
    }
#pragma unroll
    for (int i = 0; i < kLinTok; ++i) {
        const float s = warp_sum(acc[i]);
        if (lane == 0 && t0 + i < T) {
            float* p = y + (int64_t)(t0 + i) * ldy + n;
            *p = accumulate ? *p + s : s;
        }
    }
}

int linear_f32(const float* W, int N, int K, const float* x, int ldx, int T, float* y, int ldy, bool accumulate,
               cudaStream_t st) {
    if (T <= 0 || N <= 0) return 0;
    dim3 grid((N * 32 + 255) / 256, (T + kLinTok - 1) / kLinTok);
    linear_f32_kernel<<<grid, 256, 0, st>>>(W, N, K, x, ldx, T, y, ldy, accumulate ? 1 : 0);
    return (int)cudaGetLastError();
}

__global__ void argmax_rows_kernel(const float* __restrict__ logits, int ldl, int V,
                                   unsigned long long* __restrict__ keys) {
    __shared__ unsigned long long red[32];
    const int t = blockIdx.x;
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
    argmax_rows_kernel<<<T, 256, 0, st>>>(logits, ldl, V, keys);
    return (int)cudaGetLastError();
}

__global__ void keys_to_tokens_kernel(const unsigned long long* __restrict__ keys, int T, uint32_t* __restrict__ tok) {
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t < T) tok[t] = 0xFFFFFFFFu - (uint32_t)(keys[t] & 0xFFFFFFFFull);
}

int keys_to_tokens(const unsigned long long* keys, int T, uint32_t* tokens, cudaStream_t st) {
    if (T <= 0) return 0;
    keys_to_tokens_kernel<<<(T + 255) / 256, 256, 0, st>>>(keys, T, tokens);
    return (int)cudaGetLastError();
}

}  // namespace dflash
