// Row-wise pieces of a draft layer and the attention.
//
// Page "cortiq-engine 0.8.71 — src/dflash.rs": `rms` (RMSNorm of a row),
// `Drafter::rotate` (half-split RoPE at the row's position, angle
// f32(position) * inv_freq in f32), `Drafter::mlp` (silu(gate x) * up x),
// `Drafter::settle_rows` (context keys normed then rotated, values as they
// come), `Drafter::block` (attention of the block's rows over the context
// before the anchor and the block's own rows, not causal, softmax by
// max-subtract / exp / divide).  Page "cortiq-engine 0.8.75 —
// src/gpu_wgpu/dflash_dev.rs": the same steps as the kernels `dflash_rms`,
// `dflash_qk`, `dflash_attn`, `dflash_silu`.
#include <cooperative_groups.h>

#include <algorithm>
#include <array>

#include "common.cuh"
#include "kernels.cuh"
#include "attn.cuh"

namespace dflash {

namespace cg = cooperative_groups;

constexpr int kRowThreads = 1024;

// Block-wide sum / max over kRowThreads threads.
template <bool kMax>
DF_DEV float row_reduce(float v, float* red) {
    v = kMax ? warp_max(v) : warp_sum(v);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    if (threadIdx.x < 32) {
        float u = red[threadIdx.x];
        u = kMax ? warp_max(u) : warp_sum(u);
        if (threadIdx.x == 0) red[32] = u;
    }
    __syncthreads();
    float r = red[32];
    __syncthreads();
    return r;
}

// The same over NT threads (NT / 32 warps).
template <bool kMax, int NT>
DF_DEV float row_reduce_nt(float v, float* red) {
    v = kMax ? warp_max(v) : warp_sum(v);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    if (threadIdx.x < 32) {
        float u = threadIdx.x < NT / 32 ? red[threadIdx.x] : 0.f;  // 0: the identity of both (the max is of |x|)
        u = kMax ? warp_max(u) : warp_sum(u);
        if (threadIdx.x == 0) red[32] = u;
    }
    __syncthreads();
    float r = red[32];
    __syncthreads();
    return r;
}

// A word of four int8 codes, and (out16 != nullptr) the same codes as exact
// f16 values at out16 + 4 c (the tcgen05 matmuls' activation operand).
DF_DEV void put_codes4(uint32_t* q4, __half* out16, int c, uint32_t w) {
    q4[c] = w;
    if (out16 != nullptr) {
        uint32_t lo, hi;
        i8x4_to_half2x2(w, lo, hi);
        *reinterpret_cast<uint2*>(out16 + 4 * c) = make_uint2(lo, hi);
    }
}

// Zero `n` floats at `p`, spread over the grid (a side duty that clears the
// buffer a later kernel accumulates into).
DF_DEV void zero_side(float* p, int64_t n) {
    if (!p) return;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) p[i] = 0.f;
}

__global__ void __launch_bounds__(kRowThreads) rms_rows_kernel(const float* __restrict__ src, int ld_src, RowMap map,
                                                               int n, const float* __restrict__ w, float eps,
                                                               float* __restrict__ out_f32, int ld_out,
                                                               int8_t* __restrict__ out_codes,
                                                               float* __restrict__ out_scale, int ld_codes,
                                                               float* zero_buf, int64_t zero_n,
                                                               const float* __restrict__ div, int div_seg,
                                                               __half* __restrict__ out16) {
    __shared__ float red[33];
    pdl_trigger();
    pdl_wait();
    zero_side(zero_buf, zero_n);
    const int i = blockIdx.x;
    const int srow = (i / map.per) * map.stride + map.skip + (i % map.per);
    const float* x = src + (int64_t)srow * ld_src;
    // with div: each div_seg-column segment of the source divided by its divisor first
    const float* dv = div ? div + (int64_t)srow * (n / div_seg) : nullptr;
    auto src_at = [&](int c) { return dv ? x[c] / dv[c / div_seg] : x[c]; };
    float s = 1.f;
    if (w) {
        float ss = 0.f;
        for (int c = threadIdx.x; c < n; c += kRowThreads) ss = fmaf(src_at(c), src_at(c), ss);
        ss = row_reduce<false>(ss, red);
        s = 1.0f / sqrtf(ss / (float)n + eps);
    }
    if (out_f32) {
        for (int c = threadIdx.x; c < n; c += kRowThreads)
            out_f32[(int64_t)i * ld_out + c] = w ? src_at(c) * s * w[c] : src_at(c);
        return;
    }
    float amax = 0.f;
    for (int c = threadIdx.x; c < n; c += kRowThreads) amax = fmaxf(amax, fabsf(w ? src_at(c) * s * w[c] : src_at(c)));
    amax = row_reduce<true>(amax, red);
    const float sx = __fdiv_rn(amax, 127.0f);
    int8_t* q = out_codes + (int64_t)i * ld_codes;
    for (int c = threadIdx.x; c < n; c += kRowThreads) {
        const float v = w ? src_at(c) * s * w[c] : src_at(c);
        q[c] = sx > 0.f ? code_of(v, sx) : (int8_t)0;
        if (out16 != nullptr) out16[(int64_t)i * n + c] = __int2half_rn(q[c]);
    }
    if (threadIdx.x == 0) out_scale[i] = sx;
}

// The same in one read: the row sits in registers (NV float4 per thread) from
// the load to the codes.  Rows must be 16-byte aligned, n % 4 == 0 and
// n <= 4 * NV * kRowThreads.
template <int NV, int NT = kRowThreads>
__global__ void __launch_bounds__(NT, NT == kRowThreads || NV > 12 ? 1 : 2) rms_rows_reg_kernel(const float* __restrict__ src, int ld_src, RowMap map,
                                                                   int n, const float* __restrict__ w, float eps,
                                                                   float* __restrict__ out_f32, int ld_out,
                                                                   int8_t* __restrict__ out_codes,
                                                                   float* __restrict__ out_scale, int ld_codes,
                                                                   float* zero_buf, int64_t zero_n, int rows,
                                                                   const float* __restrict__ div, int div_seg,
                                                                   __half* __restrict__ out16) {
    __shared__ float red[33];
    pdl_trigger();
    pdl_wait();
    if ((int)blockIdx.x >= rows) {
        // the CTAs past the rows clear the side buffer, float4 at a time
        const int64_t stride = (int64_t)(gridDim.x - rows) * blockDim.x;
        const int64_t first = (int64_t)(blockIdx.x - rows) * blockDim.x + threadIdx.x;
        float4* p4 = reinterpret_cast<float4*>(zero_buf);
        for (int64_t k = first; k < zero_n / 4; k += stride) p4[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (first < zero_n % 4) zero_buf[zero_n / 4 * 4 + first] = 0.f;
        return;
    }
    const int i = blockIdx.x;
    const int srow = (i / map.per) * map.stride + map.skip + (i % map.per);
    const float4* x4 = reinterpret_cast<const float4*>(src + (int64_t)srow * ld_src);
    const int n4 = n / 4;
    float4 v[NV];
    float ss = 0.f;
#pragma unroll
    for (int u = 0; u < NV; ++u) {
        const int c = threadIdx.x + u * NT;
        v[u] = c < n4 ? x4[c] : make_float4(0.f, 0.f, 0.f, 0.f);
        if (div != nullptr && c < n4) {
            // a sum of parts: the float4's segment divided by its divisor (div_seg % 4 == 0)
            const float d = div[(int64_t)srow * (n / div_seg) + (4 * c) / div_seg];
            v[u] = make_float4(v[u].x / d, v[u].y / d, v[u].z / d, v[u].w / d);
        }
        ss = fmaf(v[u].x, v[u].x, ss);
        ss = fmaf(v[u].y, v[u].y, ss);
        ss = fmaf(v[u].z, v[u].z, ss);
        ss = fmaf(v[u].w, v[u].w, ss);
    }
    if (w) {
        ss = row_reduce_nt<false, NT>(ss, red);
        const float s = 1.f / sqrtf(ss / (float)n + eps);
        const float4* w4 = reinterpret_cast<const float4*>(w);
#pragma unroll
        for (int u = 0; u < NV; ++u) {
            const int c = threadIdx.x + u * NT;
            if (c < n4) {
                const float4 g = w4[c];
                v[u] = make_float4(v[u].x * s * g.x, v[u].y * s * g.y, v[u].z * s * g.z, v[u].w * s * g.w);
            }
        }
    }
    if (out_f32) {
        float4* o4 = reinterpret_cast<float4*>(out_f32 + (int64_t)i * ld_out);
#pragma unroll
        for (int u = 0; u < NV; ++u) {
            const int c = threadIdx.x + u * NT;
            if (c < n4) o4[c] = v[u];
        }
        return;
    }
    float amax = 0.f;
#pragma unroll
    for (int u = 0; u < NV; ++u) amax = fmaxf(amax, amax4(v[u]));  // lanes past n hold zeros
    amax = row_reduce_nt<true, NT>(amax, red);
    const float sx = __fdiv_rn(amax, 127.0f);
    uint32_t* q4 = reinterpret_cast<uint32_t*>(out_codes + (int64_t)i * ld_codes);
#pragma unroll
    for (int u = 0; u < NV; ++u) {
        const int c = threadIdx.x + u * NT;
        if (c < n4) put_codes4(q4, out16 ? out16 + (int64_t)i * n : nullptr, c, codes4(v[u], sx));
    }
    if (threadIdx.x == 0) out_scale[i] = sx;
}

// Rows from which a row kernel takes the many-rows configuration.
constexpr int kManyRows = 128;

// Many rows (a batch, a prefill) quantised: a CTA of kManyThreads threads a
// row, NV float4 of the row a thread, held in registers.  Unlike the kernels
// above, every load (the row's and the norm weights') is issued before the
// first use, and each block-wide reduction takes one barrier: every thread
// folds the warps' partials itself, in the same order, into the same value.
constexpr int kManyThreads = 512;

template <bool kMax>
DF_DEV float block_fold(float v, float* part) {
    v = kMax ? warp_max(v) : warp_sum(v);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = v;
    __syncthreads();
    float r = part[0];
#pragma unroll
    for (int k = 1; k < kManyThreads / 32; ++k) r = kMax ? fmaxf(r, part[k]) : r + part[k];
    return r;
}

template <int NV, bool kW, int kMinBlocks>
__global__ void __launch_bounds__(kManyThreads, kMinBlocks)
    rms_rows_many_kernel(const float* __restrict__ src, int ld_src, RowMap map, int n, const float* __restrict__ w,
                         float eps, int8_t* __restrict__ out_codes, float* __restrict__ out_scale, int ld_codes,
                         float* zero_buf, int64_t zero_n, int rows, const float* __restrict__ div, int div_seg,
                         __half* __restrict__ out16) {
    __shared__ float part[2][kManyThreads / 32];  // one array a reduction: no barrier between them
    const int n4 = n / 4;
    pdl_trigger();
    pdl_wait();
    if ((int)blockIdx.x >= rows) {
        // the CTAs past the rows clear the side buffer, float4 at a time
        const int64_t stride = (int64_t)(gridDim.x - rows) * blockDim.x;
        const int64_t first = (int64_t)(blockIdx.x - rows) * blockDim.x + threadIdx.x;
        float4* p4 = reinterpret_cast<float4*>(zero_buf);
        for (int64_t k = first; k < zero_n / 4; k += stride) p4[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (first < zero_n % 4) zero_buf[zero_n / 4 * 4 + first] = 0.f;
        return;
    }
    const int i = blockIdx.x;
    const int srow = (i / map.per) * map.stride + map.skip + (i % map.per);
    const float4* x4 = reinterpret_cast<const float4*>(src + (int64_t)srow * ld_src);
    float4 v[NV], g[kW ? NV : 1];
#pragma unroll
    for (int u = 0; u < NV; ++u) {
        const int c = threadIdx.x + u * kManyThreads;
        v[u] = c < n4 ? x4[c] : make_float4(0.f, 0.f, 0.f, 0.f);
        if (kW) g[u] = c < n4 ? reinterpret_cast<const float4*>(w)[c] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (div != nullptr) {
#pragma unroll
        for (int u = 0; u < NV; ++u) {
            const int c = threadIdx.x + u * kManyThreads;
            if (c < n4) {
                // a sum of parts: the float4's segment divided by its divisor (div_seg % 4 == 0)
                const float d = div[(int64_t)srow * (n / div_seg) + (4 * c) / div_seg];
                v[u] = make_float4(v[u].x / d, v[u].y / d, v[u].z / d, v[u].w / d);
            }
        }
    }
    if (kW) {
        float ss = 0.f;
#pragma unroll
        for (int u = 0; u < NV; ++u) {
            ss = fmaf(v[u].x, v[u].x, ss);
            ss = fmaf(v[u].y, v[u].y, ss);
            ss = fmaf(v[u].z, v[u].z, ss);
            ss = fmaf(v[u].w, v[u].w, ss);
        }
        ss = block_fold<false>(ss, part[0]);
        const float s = 1.f / sqrtf(ss / (float)n + eps);
#pragma unroll
        for (int u = 0; u < NV; ++u)
            v[u] = make_float4(v[u].x * s * g[u].x, v[u].y * s * g[u].y, v[u].z * s * g[u].z, v[u].w * s * g[u].w);
    }
    float amax = 0.f;
#pragma unroll
    for (int u = 0; u < NV; ++u) amax = fmaxf(amax, amax4(v[u]));  // lanes past n hold zeros
    amax = block_fold<true>(amax, part[1]);
    const float sx = __fdiv_rn(amax, 127.0f);
    uint32_t* q4 = reinterpret_cast<uint32_t*>(out_codes + (int64_t)i * ld_codes);
#pragma unroll
    for (int u = 0; u < NV; ++u) {
        const int c = threadIdx.x + u * kManyThreads;
        if (c < n4) put_codes4(q4, out16 ? out16 + (int64_t)i * n : nullptr, c, codes4(v[u], sx));
    }
    if (threadIdx.x == 0) out_scale[i] = sx;
}

static bool rows_fit_reg(int n, const void* src, int ld_src, const void* out_f32, int ld_out, const void* codes,
                         int ld_codes, int max_n) {
    auto al = [](const void* p, int a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; };
    return n % 4 == 0 && n <= max_n && ld_src % 4 == 0 && al(src, 16) && (!out_f32 || (ld_out % 4 == 0 && al(out_f32, 16))) &&
           (!codes || (ld_codes % 4 == 0 && al(codes, 4)));
}

int rms_rows(const float* src, int ld_src, RowMap map, int rows, int n, const float* w, float eps, float* out_f32,
             int ld_out, int8_t* out_codes, float* out_scale, int ld_codes, cudaStream_t st, float* zero_buf,
             int64_t zero_n, const float* div, int div_seg, __half* out16) {
    if (rows <= 0) return 0;
    if (div && (div_seg <= 0 || div_seg % 4 || n % div_seg)) return (int)cudaErrorInvalidValue;
    if (out16 && (!out_codes || out_f32 || n % 4 || (reinterpret_cast<uintptr_t>(out16) & 7)))
        return (int)cudaErrorInvalidValue;
    const bool wal = !w || (reinterpret_cast<uintptr_t>(w) % 16) == 0;
    const bool zal = !zero_buf || (reinterpret_cast<uintptr_t>(zero_buf) % 16) == 0;
    if (wal && zal && rows_fit_reg(n, src, ld_src, out_f32, ld_out, out_codes, ld_codes, 8 * 4 * kRowThreads)) {
        const int nv = (n + 4 * kRowThreads - 1) / (4 * kRowThreads);
        // extra CTAs clear the side buffer (about four float4 stores a thread, at most 128 CTAs)
        const int extra =
            zero_buf && zero_n > 0 ? (int)std::min<int64_t>(128, zero_n / 4 / (kRowThreads * 4) + 1) : 0;
        auto go = [&](auto kern) {
            return (int)launch(kern, dim3(rows + extra), dim3(kRowThreads), 0, st, src, ld_src, map, n, w, eps, out_f32,
                               ld_out, out_codes, out_scale, ld_codes, zero_buf, zero_n, rows, div, div_seg, out16);
        };
        const int nv512 = (n + 4 * 512 - 1) / (4 * 512);
        auto go512 = [&](auto kern) {
            const int extra512 = zero_buf && zero_n > 0 ? (int)std::min<int64_t>(256, zero_n / 4 / (512 * 4) + 1) : 0;
            return (int)launch(kern, dim3(rows + extra512), dim3(512), 0, st, src, ld_src, map, n, w, eps, out_f32, ld_out,
                               out_codes, out_scale, ld_codes, zero_buf, zero_n, rows, div, div_seg, out16);
        };
        // many rows (a batch, a prefill) quantised: 512 threads a row, so that
        // more rows share an SM and the launch runs in fewer waves
        if (rows >= kManyRows && out_codes && !out_f32 && nv512 <= 12) {
            auto many = [&](auto kern) {
                // (few clearing CTAs, each with more to clear: a launch of 512 rows
                // and its side duty stay one wave at four CTAs an SM)
                const int extra512 =
                    zero_buf && zero_n > 0 ? (int)std::min<int64_t>(96, zero_n / 4 / (512 * 4) + 1) : 0;
                return (int)launch(kern, dim3(rows + extra512), dim3(kManyThreads), 0, st, src, ld_src, map, n, w, eps,
                                   out_codes, out_scale, ld_codes, zero_buf, zero_n, rows, div, div_seg, out16);
            };
            if (nv512 <= 2) return w ? many(rms_rows_many_kernel<2, true, 4>) : many(rms_rows_many_kernel<2, false, 4>);
            if (nv512 <= 4) return w ? many(rms_rows_many_kernel<4, true, 2>) : many(rms_rows_many_kernel<4, false, 2>);
            if (!w) return many(rms_rows_many_kernel<12, false, 2>);
        }
        if (rows >= kManyRows && nv512 <= 2) return go512(rms_rows_reg_kernel<2, 512>);
        if (nv <= 1) return go(rms_rows_reg_kernel<1>);
        if (nv <= 2) return go(rms_rows_reg_kernel<2>);
        if (nv <= 4) return go(rms_rows_reg_kernel<4>);
        // wider rows (the taps): 512 threads a row, so that two rows share an SM
        if (nv512 <= 12) return go512(rms_rows_reg_kernel<12, 512>);
        return go512(rms_rows_reg_kernel<16, 512>);
    }
    return (int)launch(rms_rows_kernel, dim3(rows), dim3(kRowThreads), 0, st, src, ld_src, map, n, w, eps, out_f32,
                       ld_out, out_codes, out_scale, ld_codes, zero_buf, zero_n, div, div_seg, out16);
}

// ------------------------------------------------------------------ row convolution
// One stage of the DFlash 2 row convolution (page "cortiq-engine 0.8.71 —
// src/dflash.rs", `conv`), a CTA per row r of the block rows: with i = r %
// block_len the row's index in its sequence's block,
//   y[r] = sum_{o < min(kn, i + 1)} (base[stage][o] + d[r][(stage kn + o) G + group]) * x[r - o]
// (G = n / gs groups of gs columns; every float4 of a thread in one group).
// Then, as asked: h[r] += y (stage 1: the sub-layer output into the residual),
// y as f32, and / or y as int8 codes with one f32 scale (stage 0: a matmul
// input).  CTAs past the rows clear the side buffer.
template <int NV>
__global__ void __launch_bounds__(kRowThreads) conv_rows_kernel(
    const float* __restrict__ x, int ldx, const float* __restrict__ d, int ldd, const float* __restrict__ base,
    int stage, int kn, int gs, int n, int block_len, float* __restrict__ h_add, int ldh, float* __restrict__ out_f32,
    int ld_out, int8_t* __restrict__ out_codes, float* __restrict__ out_scale, int ld_codes, float* zero_buf,
    int64_t zero_n, int rows) {
    __shared__ float red[33];
    pdl_trigger();
    pdl_wait();
    if ((int)blockIdx.x >= rows) {
        const int64_t stride = (int64_t)(gridDim.x - rows) * blockDim.x;
        const int64_t first = (int64_t)(blockIdx.x - rows) * blockDim.x + threadIdx.x;
        float4* p4 = reinterpret_cast<float4*>(zero_buf);
        for (int64_t k = first; k < zero_n / 4; k += stride) p4[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (first < zero_n % 4) zero_buf[zero_n / 4 * 4 + first] = 0.f;
        return;
    }
    const int r = blockIdx.x, i = r % block_len, groups = n / gs, n4 = n / 4;
    const int taps = min(kn, i + 1);
    float4 y[NV];
#pragma unroll
    for (int u = 0; u < NV; ++u) y[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int o = 0; o < taps; ++o) {
        const float4* x4 = reinterpret_cast<const float4*>(x + (int64_t)(r - o) * ldx);
        const float4* b4 = reinterpret_cast<const float4*>(base + (int64_t)(stage * kn + o) * n);
        const float* dyn = d + (int64_t)r * ldd + (int64_t)(stage * kn + o) * groups;
#pragma unroll
        for (int u = 0; u < NV; ++u) {
            const int c = threadIdx.x + u * kRowThreads;
            if (c < n4) {
                const float4 xv = x4[c], bv = b4[c];
                const float k = dyn[(4 * c) / gs];
                y[u].x = fmaf(bv.x + k, xv.x, y[u].x);
                y[u].y = fmaf(bv.y + k, xv.y, y[u].y);
                y[u].z = fmaf(bv.z + k, xv.z, y[u].z);
                y[u].w = fmaf(bv.w + k, xv.w, y[u].w);
            }
        }
    }
#pragma unroll
    for (int u = 0; u < NV; ++u) {
        const int c = threadIdx.x + u * kRowThreads;
        if (c < n4) {
            if (h_add) {
                float4* h4 = reinterpret_cast<float4*>(h_add + (int64_t)r * ldh) + c;
                const float4 hv = *h4;
                *h4 = make_float4(hv.x + y[u].x, hv.y + y[u].y, hv.z + y[u].z, hv.w + y[u].w);
            }
            if (out_f32) reinterpret_cast<float4*>(out_f32 + (int64_t)r * ld_out)[c] = y[u];
        }
    }
    if (!out_codes) return;
    float amax = 0.f;
#pragma unroll
    for (int u = 0; u < NV; ++u) amax = fmaxf(amax, amax4(y[u]));  // lanes past n hold zeros
    amax = row_reduce<true>(amax, red);
    const float sx = __fdiv_rn(amax, 127.0f);
    uint32_t* q4 = reinterpret_cast<uint32_t*>(out_codes + (int64_t)r * ld_codes);
#pragma unroll
    for (int u = 0; u < NV; ++u) {
        const int c = threadIdx.x + u * kRowThreads;
        if (c < n4) q4[c] = codes4(y[u], sx);
    }
    if (threadIdx.x == 0) out_scale[r] = sx;
}

int conv_rows(const float* x, int ldx, const float* d, int ldd, const float* base, int stage, int kn, int gs, int n,
              int rows, int block_len, float* h_add, int ldh, float* out_f32, int ld_out, int8_t* out_codes,
              float* out_scale, int ld_codes, cudaStream_t st, float* zero_buf, int64_t zero_n) {
    if (rows <= 0) return 0;
    auto al = [](const void* p, int a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; };
    if (kn < 1 || gs < 4 || gs % 4 || n % gs || block_len < 1 || rows % block_len || stage < 0 || stage > 1 ||
        n > 8 * 4 * kRowThreads || ldx % 4 || !al(x, 16) || !al(base, 16) || (h_add && (ldh % 4 || !al(h_add, 16))) ||
        (out_f32 && (ld_out % 4 || !al(out_f32, 16))) || (out_codes && (ld_codes % 4 || !al(out_codes, 4))) ||
        (zero_buf && !al(zero_buf, 16)))
        return (int)cudaErrorInvalidValue;
    const int nv = (n + 4 * kRowThreads - 1) / (4 * kRowThreads);
    const int extra = zero_buf && zero_n > 0 ? (int)std::min<int64_t>(128, zero_n / 4 / (kRowThreads * 4) + 1) : 0;
    auto go = [&](auto kern) {
        return (int)launch(kern, dim3(rows + extra), dim3(kRowThreads), 0, st, x, ldx, d, ldd, base, stage, kn, gs, n,
                           block_len, h_add, ldh, out_f32, ld_out, out_codes, out_scale, ld_codes, zero_buf, zero_n,
                           rows);
    };
    if (nv <= 1) return go(conv_rows_kernel<1>);
    if (nv <= 2) return go(conv_rows_kernel<2>);
    if (nv <= 4) return go(conv_rows_kernel<4>);
    return go(conv_rows_kernel<8>);
}

// A token outside [0, vocab) (only possible for anchors already on the
// device, which the host cannot check) embeds as a row of zeros.
__global__ void embed_rows_kernel(const float* __restrict__ embed, int H, int vocab,
                                  const uint32_t* __restrict__ anchor_tok, int mask_token, int block_len,
                                  float* __restrict__ h, const int64_t* __restrict__ pos0,
                                  const float* __restrict__ inv_freq, int half_hd, float2* __restrict__ rope) {
    const int r = blockIdx.x;
    pdl_trigger();
    pdl_wait();
    if (rope != nullptr) {
        // the same angle and sincosf as the context keys' rotation
        const float p = (float)(pos0[r / block_len] + r % block_len);
        for (int i = threadIdx.x; i < half_hd; i += blockDim.x) {
            float sn, cs;
            sincosf(__fmul_rn(p, inv_freq[i]), &sn, &cs);
            rope[(int64_t)r * half_hd + i] = make_float2(cs, sn);
        }
    }
    const uint32_t tok = (r % block_len == 0) ? anchor_tok[r / block_len] : (uint32_t)mask_token;
    float4* d = reinterpret_cast<float4*>(h + (int64_t)r * H);
    if (tok >= (uint32_t)vocab) {
        for (int c = threadIdx.x; c < H / 4; c += blockDim.x) d[c] = make_float4(0.f, 0.f, 0.f, 0.f);
        return;
    }
    const float4* s = reinterpret_cast<const float4*>(embed + (int64_t)tok * H);
    for (int c = threadIdx.x; c < H / 4; c += blockDim.x) d[c] = s[c];
}

int embed_rows(const float* embed, int H, int vocab, const uint32_t* anchor_tok, int mask_token, int n_seqs,
               int block_len, float* h, cudaStream_t st, const int64_t* pos0, const float* inv_freq, int hd,
               float2* rope) {
    return (int)launch(embed_rows_kernel, dim3(n_seqs * block_len), dim3(256), 0, st, embed, H, vocab, anchor_tok,
                       mask_token, block_len, h, pos0, inv_freq, hd / 2, rope);
}

// RMSNorm of one head (hd = 32 * E elements, lane holds lane + 32 j) and its
// half-split rotation at `pos` (pairs (i, i + hd/2) sit in one lane).
template <int E>
DF_DEV void norm_rope_head(float (&v)[E], const float* __restrict__ gain, const float* __restrict__ inv_freq,
                           float eps, int64_t pos, bool rotary) {
    constexpr int HD = 32 * E;
    const int lane = threadIdx.x & 31;
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < E; ++j) ss = fmaf(v[j], v[j], ss);
    ss = warp_sum(ss);
    const float s = 1.0f / sqrtf(ss / (float)HD + eps);
#pragma unroll
    for (int j = 0; j < E; ++j) v[j] = v[j] * s * gain[lane + 32 * j];
    if (!rotary) return;
    const float p = (float)pos;
#pragma unroll
    for (int j = 0; j < E / 2; ++j) {
        const float ang = __fmul_rn(p, inv_freq[lane + 32 * j]);
        float sn, cs;
        sincosf(ang, &sn, &cs);
        const float lo = v[j], hi = v[j + E / 2];
        v[j] = lo * cs - hi * sn;
        v[j + E / 2] = hi * cs + lo * sn;
    }
}

template <int E>
__global__ void kv_append_kernel(const float* __restrict__ kv, int n, int L, int nkv,
                                 const float* const* __restrict__ k_norm, const float* __restrict__ inv_freq,
                                 float eps, const int64_t* __restrict__ pos, __half* const* __restrict__ kstore,
                                 __half* const* __restrict__ vstore, int64_t cap, const int* __restrict__ rotary) {
    constexpr int HD = 32 * E;
    const int64_t wid = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
    pdl_trigger();
    pdl_wait();
    const int64_t pos0 = pos[0], idx0 = pos[1];
    if (wid >= (int64_t)n * L * nkv) return;
    const int lane = threadIdx.x & 31;
    const int g = (int)(wid % nkv), l = (int)((wid / nkv) % L);
    const int64_t r = wid / ((int64_t)nkv * L);
    const float* src = kv + r * ((int64_t)L * 2 * nkv * HD) + (int64_t)l * 2 * nkv * HD;
    float kvv[E], vv[E];
#pragma unroll
    for (int j = 0; j < E; ++j) {
        kvv[j] = src[g * HD + lane + 32 * j];
        vv[j] = src[(nkv + g) * HD + lane + 32 * j];
    }
    norm_rope_head<E>(kvv, k_norm[l], inv_freq, eps, pos0 + r, rotary == nullptr || rotary[l] != 0);
    // the store keeps each value as its (hi, lo) f16 pair: plane hi then plane lo
    const int64_t plane = (int64_t)nkv * cap * HD;
    __half* kd = kstore[l] + ((int64_t)g * cap + idx0 + r) * HD;
    __half* vd = vstore[l] + ((int64_t)g * cap + idx0 + r) * HD;
#pragma unroll
    for (int j = 0; j < E; ++j) {
        __half h, lo;
        split_f16(kvv[j], h, lo);
        kd[lane + 32 * j] = h;
        kd[plane + lane + 32 * j] = lo;
        split_f16(vv[j], h, lo);
        vd[lane + 32 * j] = h;
        vd[plane + lane + 32 * j] = lo;
    }
}

int kv_append(const float* kv, int n, int L, int nkv, int hd, const float* const* k_norm_dev, const float* inv_freq,
              float eps, const int64_t* pos_dev, __half* const* kstore_dev, __half* const* vstore_dev, int64_t cap,
              cudaStream_t st, const int* rotary_dev) {
    if (n <= 0) return 0;
    const int64_t warps = (int64_t)n * L * nkv;
    const unsigned blocks = (unsigned)((warps * 32 + 255) / 256);
    if (hd == 128)
        return (int)launch(kv_append_kernel<4>, dim3(blocks), dim3(256), 0, st, kv, n, L, nkv, k_norm_dev, inv_freq,
                           eps, pos_dev, kstore_dev, vstore_dev, cap, rotary_dev);
    return (int)launch(kv_append_kernel<2>, dim3(blocks), dim3(256), 0, st, kv, n, L, nkv, k_norm_dev, inv_freq, eps,
                       pos_dev, kstore_dev, vstore_dev, cap, rotary_dev);
}


__global__ void __launch_bounds__(kRowThreads) silu_mul_kernel(const float* __restrict__ gu, int ld_gu, int I,
                                                               float* __restrict__ out_f32, int ld_out,
                                                               int8_t* __restrict__ out_codes,
                                                               float* __restrict__ out_scale, int ld_codes,
                                                               __half* __restrict__ out16) {
    __shared__ float red[33];
    pdl_trigger();
    pdl_wait();
    const int r = blockIdx.x;
    const float* g = gu + (int64_t)r * ld_gu;
    const float* u = g + I;
    if (out_f32) {
        for (int c = threadIdx.x; c < I; c += kRowThreads) out_f32[(int64_t)r * ld_out + c] = silu_f(g[c]) * u[c];
        return;
    }
    float amax = 0.f;
    for (int c = threadIdx.x; c < I; c += kRowThreads) amax = fmaxf(amax, fabsf(silu_f(g[c]) * u[c]));
    amax = row_reduce<true>(amax, red);
    const float sx = __fdiv_rn(amax, 127.0f);
    int8_t* q = out_codes + (int64_t)r * ld_codes;
    for (int c = threadIdx.x; c < I; c += kRowThreads) {
        const float a = silu_f(g[c]) * u[c];
        q[c] = sx > 0.f ? code_of(a, sx) : (int8_t)0;
        if (out16 != nullptr) out16[(int64_t)r * I + c] = __int2half_rn(q[c]);
    }
    if (threadIdx.x == 0) out_scale[r] = sx;
}

// The same in one read, the products kept in registers (NV float4 per thread).
template <int NV>
__global__ void __launch_bounds__(kRowThreads) silu_mul_reg_kernel(const float* __restrict__ gu, int ld_gu, int I,
                                                                   float* __restrict__ out_f32, int ld_out,
                                                                   int8_t* __restrict__ out_codes,
                                                                   float* __restrict__ out_scale, int ld_codes,
                                                                   __half* __restrict__ out16) {
    __shared__ float red[33];
    pdl_trigger();
    pdl_wait();
    const int r = blockIdx.x;
    const float4* g4 = reinterpret_cast<const float4*>(gu + (int64_t)r * ld_gu);
    const float4* u4 = reinterpret_cast<const float4*>(gu + (int64_t)r * ld_gu + I);
    const int n4 = I / 4;
    float4 gv[NV], uv[NV];
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int c = threadIdx.x + k * kRowThreads;
        gv[k] = c < n4 ? g4[c] : make_float4(0.f, 0.f, 0.f, 0.f);
        uv[k] = c < n4 ? u4[c] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float4 a[NV];
    float amax = 0.f;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        a[k] = make_float4(silu_f(gv[k].x) * uv[k].x, silu_f(gv[k].y) * uv[k].y, silu_f(gv[k].z) * uv[k].z,
                           silu_f(gv[k].w) * uv[k].w);
        amax = fmaxf(amax, amax4(a[k]));  // lanes past I: silu(0) * 0 = 0
    }
    if (out_f32) {
        float4* o4 = reinterpret_cast<float4*>(out_f32 + (int64_t)r * ld_out);
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int c = threadIdx.x + k * kRowThreads;
            if (c < n4) o4[c] = a[k];
        }
        return;
    }
    amax = row_reduce<true>(amax, red);
    const float sx = __fdiv_rn(amax, 127.0f);
    uint32_t* q4 = reinterpret_cast<uint32_t*>(out_codes + (int64_t)r * ld_codes);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int c = threadIdx.x + k * kRowThreads;
        if (c < n4) put_codes4(q4, out16 ? out16 + (int64_t)r * I : nullptr, c, codes4(a[k], sx));
    }
    if (threadIdx.x == 0) out_scale[r] = sx;
}

// Many rows (a batch, a prefill): kManyThreads threads a row, NV float4 of
// the gate and of the up half a thread, every load issued before the first
// use and the products kept in registers (two rows an SM).  Same arithmetic
// as silu_mul_reg_kernel.
template <int NV>
__global__ void __launch_bounds__(kManyThreads, 2)
    silu_mul_many_kernel(const float* __restrict__ gu, int ld_gu, int I, int8_t* __restrict__ out_codes,
                         float* __restrict__ out_scale, int ld_codes, __half* __restrict__ out16) {
    __shared__ float part[kManyThreads / 32];
    pdl_trigger();
    pdl_wait();
    const int r = blockIdx.x;
    const float4* g4 = reinterpret_cast<const float4*>(gu + (int64_t)r * ld_gu);
    const float4* u4 = reinterpret_cast<const float4*>(gu + (int64_t)r * ld_gu + I);
    const int n4 = I / 4;
    float4 gv[NV], uv[NV];
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int c = threadIdx.x + k * kManyThreads;
        gv[k] = c < n4 ? g4[c] : make_float4(0.f, 0.f, 0.f, 0.f);
        uv[k] = c < n4 ? u4[c] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float amax = 0.f;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        gv[k] = make_float4(silu_f(gv[k].x) * uv[k].x, silu_f(gv[k].y) * uv[k].y, silu_f(gv[k].z) * uv[k].z,
                            silu_f(gv[k].w) * uv[k].w);
        amax = fmaxf(amax, amax4(gv[k]));  // lanes past I: silu(0) * 0 = 0
    }
    amax = block_fold<true>(amax, part);
    const float sx = __fdiv_rn(amax, 127.0f);
    uint32_t* q4 = reinterpret_cast<uint32_t*>(out_codes + (int64_t)r * ld_codes);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int c = threadIdx.x + k * kManyThreads;
        if (c < n4) put_codes4(q4, out16 ? out16 + (int64_t)r * I : nullptr, c, codes4(gv[k], sx));
    }
    if (threadIdx.x == 0) out_scale[r] = sx;
}

// The same with a row split over the kSiluSplit CTAs of a cluster (one float4
// of the row per thread): each CTA reduces its share's max|a|, the cluster
// takes the row's max through distributed shared memory.
constexpr int kSiluSplit = 4;
__global__ void __launch_bounds__(kRowThreads) silu_mul_cluster_kernel(const float* __restrict__ gu, int ld_gu, int I,
                                                                       float* __restrict__ out_f32, int ld_out,
                                                                       int8_t* __restrict__ out_codes,
                                                                       float* __restrict__ out_scale, int ld_codes,
                                                                       __half* __restrict__ out16) {
    __shared__ float red[33];
    cg::cluster_group cluster = cg::this_cluster();
    pdl_trigger();
    pdl_wait();
    const int r = blockIdx.y, part = (int)cluster.block_rank();
    const int share4 = I / 4 / kSiluSplit;  // float4 of the row per CTA
    const int c = part * share4 + threadIdx.x;
    const bool in = threadIdx.x < share4;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    if (in) {
        const float4 gv = reinterpret_cast<const float4*>(gu + (int64_t)r * ld_gu)[c];
        const float4 uv = reinterpret_cast<const float4*>(gu + (int64_t)r * ld_gu + I)[c];
        a = make_float4(silu_f(gv.x) * uv.x, silu_f(gv.y) * uv.y, silu_f(gv.z) * uv.z, silu_f(gv.w) * uv.w);
    }
    if (out_f32) {
        if (in) reinterpret_cast<float4*>(out_f32 + (int64_t)r * ld_out)[c] = a;
        return;  // no cluster-wide step on this path: every CTA leaves here
    }
    const float local = row_reduce<true>(amax4(a), red);  // red[32] holds this CTA's max
    cluster.sync();
    float amax = local;
#pragma unroll
    for (int k = 0; k < kSiluSplit; ++k) amax = fmaxf(amax, cluster.map_shared_rank(red, k)[32]);
    cluster.sync();  // no CTA leaves while another may still read its max
    const float sx = __fdiv_rn(amax, 127.0f);
    if (in)
        put_codes4(reinterpret_cast<uint32_t*>(out_codes + (int64_t)r * ld_codes), out16 ? out16 + (int64_t)r * I : nullptr,
                   c, codes4(a, sx));
    if (part == 0 && threadIdx.x == 0) out_scale[r] = sx;
}

int silu_mul(const float* gu, int ld_gu, int rows, int I, float* out_f32, int ld_out, int8_t* out_codes,
             float* out_scale, int ld_codes, cudaStream_t st, __half* out16) {
    if (rows <= 0) return 0;
    if (out16 && (!out_codes || out_f32 || I % 4 || (reinterpret_cast<uintptr_t>(out16) & 7)))
        return (int)cudaErrorInvalidValue;
    // few rows: a row over a cluster of kSiluSplit CTAs; many rows: a CTA a row
    const bool cluster_ok = rows < kManyRows && I % (4 * kSiluSplit) == 0 && I / 4 / kSiluSplit <= kRowThreads &&
                            rows_fit_reg(I, gu, ld_gu, out_f32, ld_out, out_codes, ld_codes, 4 * kSiluSplit * kRowThreads) &&
                            (reinterpret_cast<uintptr_t>(gu + I) % 16) == 0;
    if (cluster_ok)
        return (int)launch_cluster(silu_mul_cluster_kernel, dim3(kSiluSplit, rows), dim3(kRowThreads), 0, st,
                                   kSiluSplit, gu, ld_gu, I, out_f32, ld_out, out_codes, out_scale, ld_codes, out16);
    if (rows >= kManyRows && out_codes && !out_f32 &&
        rows_fit_reg(I, gu, ld_gu, nullptr, 0, out_codes, ld_codes, 8 * 4 * kManyThreads) &&
        (reinterpret_cast<uintptr_t>(gu + I) % 16) == 0) {
        const int nv = (I / 4 + kManyThreads - 1) / kManyThreads;
        auto go = [&](auto kern) {
            return (int)launch(kern, dim3(rows), dim3(kManyThreads), 0, st, gu, ld_gu, I, out_codes, out_scale, ld_codes,
                               out16);
        };
        if (nv <= 2) return go(silu_mul_many_kernel<2>);
        if (nv <= 4) return go(silu_mul_many_kernel<4>);
        if (nv <= 6) return go(silu_mul_many_kernel<6>);
        return go(silu_mul_many_kernel<8>);
    }
    if (rows_fit_reg(I, gu, ld_gu, out_f32, ld_out, out_codes, ld_codes, 4 * 4 * kRowThreads) &&
        (reinterpret_cast<uintptr_t>(gu + I) % 16) == 0) {
        const int nv = (I + 4 * kRowThreads - 1) / (4 * kRowThreads);
        auto go = [&](auto kern) {
            return (int)launch(kern, dim3(rows), dim3(kRowThreads), 0, st, gu, ld_gu, I, out_f32, ld_out, out_codes,
                               out_scale, ld_codes, out16);
        };
        if (nv <= 1) return go(silu_mul_reg_kernel<1>);
        if (nv <= 2) return go(silu_mul_reg_kernel<2>);
        return go(silu_mul_reg_kernel<4>);
    }
    return (int)launch(silu_mul_kernel, dim3(rows), dim3(kRowThreads), 0, st, gu, ld_gu, I, out_f32, ld_out,
                       out_codes, out_scale, ld_codes, out16);
}

// ------------------------------------------------------------------ attention
// The key range of one (sequence, kv head, query tile) is split over the CTAs
// of a thread-block cluster; each CTA runs an online softmax over its keys
// and the cluster merges the CTAs' partial results through distributed
// shared memory, so that nothing but y is written to global memory.
constexpr int kAttnQW = 4;                     // query warps of a CTA, 16 query vectors each
constexpr int kAttnKH = 2;                     // key lanes: warps that share a query warp's rows
constexpr int kAttnQ = 16 * kAttnQW;           // query vectors of a CTA
constexpr int kAttnK = 32;                     // keys of a tile; each key lane takes one tile per step
constexpr int kAttnStep = kAttnKH * kAttnK;    // keys per step of the CTA
constexpr int kAttnWarps = kAttnQW * kAttnKH;
constexpr int kAttnMaxCluster = 32 / kAttnKH < 16 ? 32 / kAttnKH : 16;  // CTAs of a cluster (non-portable above 8)


DF_DEV void ldsm_x4(uint32_t (&r)[4], const __half* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_addr(p)));
}
DF_DEV void ldsm_x4_t(uint32_t (&r)[4], const __half* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_addr(p)));
}

template <int HD, int ST>
struct AttnSmem {
    static constexpr int LD = HD + 8;  // halves: 16-byte row pad, conflict-free ldmatrix
    static constexpr int PART = HD + 4;  // floats of a partial row: m, l, -, -, acc[HD]
    __half qh[kAttnQ][LD], ql[kAttnQ][LD];
    // [stage][key lane][key][dim]; after the key loop this area holds the
    // partial rows [key lane][query][PART] that the cluster merges
    __half kh[ST][kAttnKH][kAttnK][LD], kl[ST][kAttnKH][kAttnK][LD];
    __half vh[ST][kAttnKH][kAttnK][LD], vl[ST][kAttnKH][kAttnK][LD];
    DF_DEV float* part() { return reinterpret_cast<float*>(&kh[0][0][0][0]); }
};
static_assert(kAttnQW <= 4, "the partial rows must fit the key/value area");

// CTA (split sp of the cluster, kv head x query tile, sequence).  The query
// tile is up to kAttnQ (q head of the group, block row) pairs, 16 per query
// warp; the CTA's keys (context rows [lo, lo + n) then the block's rows, its
// share of them) go by in steps of kAttnKH tiles of 32 keys, tile k of a step
// to the warps of key lane k.  Scores and values go through f16 tensor-core MMAs as
// hi/lo splits (q.k = qh.kh + qh.kl + ql.kh, likewise p.v), which keeps
// f32-level accuracy; the softmax is online in f32 (running max in the log2
// domain, running sum, unnormalised output).  At the end every query row has
// kAttnKH x nsplit partial results in the cluster's shared memory; CTA sp merges
// rows sp, sp + nsplit, ... and writes them to y.
// ST key-step stages in shared memory: 2 (double-buffered copies, the next
// step in flight while the current one is multiplied; one CTA an SM) or 1 (two
// CTAs an SM at 128 registers a thread, each one's copies overlapping the
// other's products).
template <int HD, int ST, bool WIN>
__global__ void __launch_bounds__(kAttnWarps * 32, ST == 1 ? 2 : 1) attn_cluster_kernel(const float* __restrict__ qkv, int ld,
                                                                       int block_len, const AttnSeq* __restrict__ seqs,
                                                                       int nq, int nkv, int qtiles, int nsplit,
                                                                       float scale_log2, float* __restrict__ y,
                                                                       const float* __restrict__ q_norm,
                                                                       const float* __restrict__ k_norm,
                                                                       const float2* __restrict__ rope, float eps,
                                                                       float* __restrict__ gpart, int kv_ready,
                                                                       float* __restrict__ lacc, float ref_log2) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    AttnSmem<HD, ST>& sm = *reinterpret_cast<AttnSmem<HD, ST>*>(smem_raw);
    constexpr int PART = AttnSmem<HD, ST>::PART;
    constexpr int NT = HD / 8;   // n8 tiles of the output
    constexpr int KS = HD / 16;  // k16 steps of the scores
    constexpr int kThreads = kAttnWarps * 32;
    cg::cluster_group cluster = cg::this_cluster();
    // the key split: the CTA's rank in its cluster, or, when the splits merge
    // through global memory (gpart) or add into accumulators (lacc), its x
    // index in a launch without clusters
    const int sp = (gpart || lacc) ? (int)blockIdx.x : (int)cluster.block_rank();
    const int g = blockIdx.y / qtiles, qt = blockIdx.y % qtiles, s = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gq = lane >> 2, tq = lane & 3;
    const int qw = warp % kAttnQW, half = warp / kAttnQW;  // query warp, key lane
    pdl_trigger();
    // the context views: read ahead of the dependency wait when the caller
    // vouches that the views and the stores were final before the launch
    // sequence (kv_ready), after it otherwise (the kernel just before this one
    // may have written them)
    if (!kv_ready) pdl_wait();
    const AttnSeq sq = seqs[s];
    const int rep = nq / nkv, mq = rep * block_len;
    const int total = sq.n + block_len;
    // this sequence's keys, the block's rows first (keys 0 .. block_len - 1)
    // then its context rows, in nsplit equal shares (the last step of a share
    // may be partial); the softmax sees the keys as a set, so their order
    // only moves the f32 rounding
    const int kps = (total + nsplit - 1) / nsplit;
    const int j0 = sp * kps, j1 = min(total, j0 + kps);
    const int64_t row0 = (int64_t)s * block_len;

    // The query tile is read as float4 (all of a thread's loads in flight at
    // once), normed, rotated and split into (hi, lo) f16 halves.  Context keys
    // and values arrive as stored -- their (hi, lo) f16 pairs -- and go to
    // shared memory by 16-byte cp.async copies, with no registers held; the
    // block's own rows (f32, normed and rotated here) are split on the way.
    // Two CTAs share an SM (128 registers a thread), so one's loads overlap
    // the other's products.
    constexpr int D4 = HD / 4;
    constexpr int NQ4 = kAttnQ * D4 / kThreads, NK4 = kAttnStep * D4 / kThreads;
    constexpr int C8 = HD / 8, NC8 = kAttnStep * C8 / kThreads;  // 16-byte chunks of a key step, per thread
    static_assert(NQ4 * kThreads == kAttnQ * D4 && NK4 * kThreads == kAttnStep * D4, "tile split");
    static_assert(NC8 * kThreads == kAttnStep * C8, "chunk split");
    const int64_t plane = (int64_t)nkv * sq.cap * HD;
    // context rows of step jt: cp.async from the store (zeros past the split)
    auto issue_ctx = [&](int jt, int st) {
#pragma unroll
        for (int u = 0; u < NC8; ++u) {
            const int i = tid + u * kThreads, kr = i / C8, c = (i % C8) * 8, j = jt + kr;
            const int hf = kr / kAttnK, k = kr % kAttnK;
            if (j >= block_len && j < j1) {
                const int64_t off = ((int64_t)g * sq.cap + sq.lo + (j - block_len)) * HD + c;
                cp_async16(&sm.kh[st][hf][k][c], sq.kc + off);
                cp_async16(&sm.kl[st][hf][k][c], sq.kc + plane + off);
                cp_async16(&sm.vh[st][hf][k][c], sq.vc + off);
                cp_async16(&sm.vl[st][hf][k][c], sq.vc + plane + off);
            } else if (j >= j1) {
                const uint4 z = make_uint4(0u, 0u, 0u, 0u);
                *reinterpret_cast<uint4*>(&sm.kh[st][hf][k][c]) = z;
                *reinterpret_cast<uint4*>(&sm.kl[st][hf][k][c]) = z;
                *reinterpret_cast<uint4*>(&sm.vh[st][hf][k][c]) = z;
                *reinterpret_cast<uint4*>(&sm.vl[st][hf][k][c]) = z;
            }
        }
        cp_async_commit();
    };
    // block rows of step jt (keys j < min(block_len, j1)): f32 from qkv; keys
    // normed and rotated; split into shared memory.  Two float4 of a thread
    // at a time, all their loads issued before any is used.
    auto store_block_rows = [&](int jt, int st) {
        const int d4 = tid % D4;
        float4 gk = make_float4(1.f, 1.f, 1.f, 1.f);
        if (k_norm != nullptr) gk = *reinterpret_cast<const float4*>(k_norm + 4 * d4);
        const int lim = min(block_len, j1);
        // one CTA an SM: two float4 a thread per round, every load of the
        // round issued before any is used; two CTAs an SM (registers short):
        // one
        constexpr int CH = ST == 2 ? 2 : 1;
#pragma unroll 1
        for (int u0 = 0; u0 < NK4; u0 += CH) {
            if (jt + (u0 * kThreads) / D4 >= lim) break;  // no block row in this round or later (CTA-uniform)
            float4 kk[CH], vv[CH], t01[CH], t23[CH];
            bool mine[CH];
#pragma unroll
            for (int e = 0; e < CH; ++e) {
                const int i = tid + (u0 + e) * kThreads, kr = i / D4, d = (i % D4) * 4, j = jt + kr;
                mine[e] = j < lim;  // uniform over the lanes of a row
                kk[e] = make_float4(0.f, 0.f, 0.f, 0.f);
                vv[e] = kk[e];
                if (mine[e]) {
                    const int64_t off = (row0 + j) * ld + d;
                    kk[e] = *reinterpret_cast<const float4*>(qkv + off + (int64_t)(nq + g) * HD);
                    vv[e] = *reinterpret_cast<const float4*>(qkv + off + (int64_t)(nq + nkv + g) * HD);
                }
                t01[e] = t23[e] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (k_norm != nullptr && rope != nullptr)
                    rope_pairs<HD>(rope, row0 + min(j, block_len - 1), d4, t01[e], t23[e]);
            }
#pragma unroll
            for (int e = 0; e < CH; ++e) {
                const int i = tid + (u0 + e) * kThreads, kr = i / D4, d = (i % D4) * 4;
                const int hf = kr / kAttnK, k = kr % kAttnK;
                if (k_norm != nullptr) norm_rope4<HD>(kk[e], mine[e], gk, t01[e], t23[e], d4, eps, rope != nullptr);
                if (mine[e]) {
                    split_store4(kk[e], &sm.kh[st][hf][k][d], &sm.kl[st][hf][k][d]);
                    split_store4(vv[e], &sm.vh[st][hf][k][d], &sm.vl[st][hf][k][d]);
                }
            }
        }
    };
    // The context copies of the first steps go out before the wait when the
    // caller vouches that no kernel of the dependency chain writes the store
    // (kv_ready); otherwise just after it.
    auto issue_first = [&]() {
        if (j0 < j1) issue_ctx(j0, 0);
        if (ST == 2 && j0 + kAttnStep < j1) issue_ctx(j0 + kAttnStep, 1);
    };
    if (kv_ready) issue_first();
    pdl_wait();
    if (!kv_ready) issue_first();
    {
        // the query tile (and, one CTA an SM, its rotation pairs), then the
        // block rows of this split's first step: their loads all in flight
        // before the first is used
        constexpr int NR = ST == 2 ? NQ4 : 1;  // two CTAs an SM: the pairs are loaded as used
        float4 qv[NQ4], qt01[NR], qt23[NR];
        const int d4 = tid % D4;
#pragma unroll
        for (int u = 0; u < NQ4; ++u) {
            const int i = tid + u * kThreads, qr = i / D4, d = (i % D4) * 4, ii = qt * kAttnQ + qr;
            qv[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (ii < mq) {
                const int head = g * rep + ii / block_len, r = ii % block_len;
                qv[u] = *reinterpret_cast<const float4*>(qkv + (row0 + r) * ld + (int64_t)head * HD + d);
            }
            if constexpr (ST == 2)
                if (q_norm != nullptr && rope != nullptr) rope_pairs<HD>(rope, row0 + ii % block_len, d4, qt01[u], qt23[u]);
        }
        if (j0 < j1 && j0 < block_len) store_block_rows(j0, 0);
        if (q_norm != nullptr) {
            const float4 gq = *reinterpret_cast<const float4*>(q_norm + 4 * d4);
#pragma unroll
            for (int u = 0; u < NQ4; ++u) {
                const int ii = qt * kAttnQ + (tid + u * kThreads) / D4;
                if constexpr (ST == 2) {
                    norm_rope4<HD>(qv[u], ii < mq, gq, qt01[u], qt23[u], d4, eps, rope != nullptr);
                } else {
                    float4 t01 = make_float4(0.f, 0.f, 0.f, 0.f), t23 = t01;
                    if (rope != nullptr) rope_pairs<HD>(rope, row0 + ii % block_len, d4, t01, t23);
                    norm_rope4<HD>(qv[u], ii < mq, gq, t01, t23, d4, eps, rope != nullptr);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < NQ4; ++u) {
            const int i = tid + u * kThreads, qr = i / D4, d = (i % D4) * 4;
            split_store4(qv[u], &sm.qh[qr][d], &sm.ql[qr][d]);
        }
    }

    float o[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    const int qbase = qw * 16;
    // the leading context rows each of this lane's two query rows does not
    // see (block row i of a windowed layer: sq.cut + i; WIN: some view of
    // the launch has a window)
    int cutr[2] = {kNoCut, kNoCut};
    if constexpr (WIN) {
#pragma unroll
        for (int h = 0; h < 2; ++h) cutr[h] = sq.cut + (qt * kAttnQ + qbase + gq + 8 * h) % block_len;
    }
    // ldmatrix row addresses: A (queries x dims) and B (keys x dims) operands
    const int lrow = (lane & 7) + ((lane >> 3) & 1) * 8, lcol = (lane >> 4) * 8;

    int it = 0;
    for (int jt = j0; jt < j1; jt += kAttnStep, ++it) {
        const int st = ST == 1 ? 0 : (it & 1);
        if (it > 0) __syncthreads();  // the stage refilled below is no longer read
        if (ST == 1) {
            if (it > 0) issue_ctx(jt, 0);
        } else if (it > 0 && jt + kAttnStep < j1) {
            issue_ctx(jt + kAttnStep, st ^ 1);  // the next step's copies, in flight during this one
        }
        if (it > 0 && jt < block_len) store_block_rows(jt, st);  // the first step's went with the queries
        if (ST == 2 && jt + kAttnStep < j1)
            cp_async_wait_one();  // this step's copies done; the next step's may still fly
        else
            cp_async_wait_all();
        __syncthreads();
        const int kt = jt + half * kAttnK;  // first key of this warp's tile
        if (kt >= j1) continue;              // warp-uniform: nothing of this lane in the last step
        // scores: 16 queries x 32 keys per warp
        float sc[4][4];
#pragma unroll
        for (int n = 0; n < 4; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
#pragma unroll
        for (int k = 0; k < KS; ++k) {
            uint32_t ah[4], al[4];
            ldsm_x4(ah, &sm.qh[qbase + lrow][k * 16 + lcol]);
            ldsm_x4(al, &sm.ql[qbase + lrow][k * 16 + lcol]);
#pragma unroll
            for (int nb = 0; nb < 2; ++nb) {  // keys 16 nb .. 16 nb + 15
                uint32_t bh[4], bl[4];
                // matrices: (keys +0..7, dims +0..7), (keys +0..7, dims +8..15), (keys +8..15, ...), ...
                const int brow = nb * 16 + (lane & 7) + (lane >> 4) * 8, bcol = k * 16 + ((lane >> 3) & 1) * 8;
                ldsm_x4(bh, &sm.kh[st][half][brow][bcol]);
                ldsm_x4(bl, &sm.kl[st][half][brow][bcol]);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float* c = sc[nb * 2 + h];
                    float cc[4] = {c[0], c[1], c[2], c[3]};
                    mma_f16_16816(cc, ah, bh[h * 2], bh[h * 2 + 1], cc);
                    mma_f16_16816(cc, ah, bl[h * 2], bl[h * 2 + 1], cc);
                    mma_f16_16816(cc, al, bh[h * 2], bh[h * 2 + 1], cc);
                    c[0] = cc[0];
                    c[1] = cc[1];
                    c[2] = cc[2];
                    c[3] = cc[3];
                }
            }
        }
        // online softmax over the tile; rows gq and gq + 8 of the warp's 16
        float tmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int n = 0; n < 4; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int key = kt + n * 8 + 2 * tq + (e & 1);
                // past the split, or a context row before the query row's window
                const bool seen = key < j1 && (!WIN || key < block_len || key - block_len >= cutr[e >> 1]);
                const float v = seen ? sc[n][e] * scale_log2 : -INFINITY;
                sc[n][e] = v;
                tmax[e >> 1] = fmaxf(tmax[e >> 1], v);
            }
        float corr[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            tmax[h] = fmaxf(tmax[h], __shfl_xor_sync(0xffffffffu, tmax[h], 1));
            tmax[h] = fmaxf(tmax[h], __shfl_xor_sync(0xffffffffu, tmax[h], 2));
            const float m_new = fmaxf(m_run[h], tmax[h]);
            corr[h] = (m_run[h] == -INFINITY) ? 0.f : exp2f(m_run[h] - m_new);
            m_run[h] = m_new;
        }
        float psum[2] = {0.f, 0.f};
        uint32_t ph[2][4], pl[2][4];  // A fragments of P for the two k16 steps (keys 0..15, 16..31)
#pragma unroll
        for (int n = 0; n < 4; ++n) {
            float p[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                p[e] = (sc[n][e] == -INFINITY) ? 0.f : exp2f(sc[n][e] - m_run[e >> 1]);
                psum[e >> 1] += p[e];
            }
            __half h0, l0, h1, l1, h2, l2, h3, l3;
            split_f16(p[0], h0, l0);
            split_f16(p[1], h1, l1);
            split_f16(p[2], h2, l2);
            split_f16(p[3], h3, l3);
            const int kstep = n >> 1, hcol = n & 1;  // keys 8n..8n+7 -> k16 step n/2, column half n%2
            ph[kstep][hcol * 2 + 0] = pack_half2(h0, h1);  // row gq
            ph[kstep][hcol * 2 + 1] = pack_half2(h2, h3);  // row gq + 8
            pl[kstep][hcol * 2 + 0] = pack_half2(l0, l1);
            pl[kstep][hcol * 2 + 1] = pack_half2(l2, l3);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            psum[h] += __shfl_xor_sync(0xffffffffu, psum[h], 1);
            psum[h] += __shfl_xor_sync(0xffffffffu, psum[h], 2);
            l_run[h] = l_run[h] * corr[h] + psum[h];
        }
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            o[j][0] *= corr[0];
            o[j][1] *= corr[0];
            o[j][2] *= corr[1];
            o[j][3] *= corr[1];
        }
        // o += p . v over the tile's 32 keys
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
            // A fragment order: {row gq keys 2t.., row gq+8 keys 2t.., row gq keys 8+2t.., row gq+8 keys 8+2t..}
            const uint32_t ahp[4] = {ph[ks][0], ph[ks][1], ph[ks][2], ph[ks][3]};
            const uint32_t alp[4] = {pl[ks][0], pl[ks][1], pl[ks][2], pl[ks][3]};
#pragma unroll
            for (int jb = 0; jb < NT / 2; ++jb) {  // dims 16 jb .. 16 jb + 15
                uint32_t bh[4], bl[4];
                // .trans matrices: (keys +0..7, dims +0..7), (keys +8..15, dims +0..7), (keys +0..7, dims +8..15), ...
                const int vrow = ks * 16 + (lane & 7) + ((lane >> 3) & 1) * 8, vcol = jb * 16 + (lane >> 4) * 8;
                ldsm_x4_t(bh, &sm.vh[st][half][vrow][vcol]);
                ldsm_x4_t(bl, &sm.vl[st][half][vrow][vcol]);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float* c = o[jb * 2 + h];
                    float cc[4] = {c[0], c[1], c[2], c[3]};
                    mma_f16_16816(cc, ahp, bh[h * 2], bh[h * 2 + 1], cc);
                    mma_f16_16816(cc, ahp, bl[h * 2], bl[h * 2 + 1], cc);
                    mma_f16_16816(cc, alp, bh[h * 2], bh[h * 2 + 1], cc);
                    c[0] = cc[0];
                    c[1] = cc[1];
                    c[2] = cc[2];
                    c[3] = cc[3];
                }
            }
        }
    }
    if (gpart) {
        // this split's partial rows (running max in the log2 domain, sum,
        // unnormalised output) to global memory, for attn_merge_kernel:
        // [unit][split][key lane][query row][PART]
        const int unit = blockIdx.z * gridDim.y + blockIdx.y;
        float* gp = gpart + ((int64_t)(unit * nsplit + sp) * kAttnKH + half) * kAttnQ * PART;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float* out = gp + (int64_t)(qbase + gq + 8 * h) * PART;
            if (tq == 0) {
                out[0] = m_run[h];
                out[1] = l_run[h];
            }
#pragma unroll
            for (int j = 0; j < NT; ++j)
                *reinterpret_cast<float2*>(out + 4 + j * 8 + 2 * tq) = make_float2(o[j][2 * h], o[j][2 * h + 1]);
        }
        return;
    }
    __syncthreads();  // every warp is done with the key/value tiles: their area takes the partial rows
    float* part = sm.part();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        float* out = part + (half * kAttnQ + qbase + gq + 8 * h) * PART;
        if (tq == 0) {
            out[0] = m_run[h];
            out[1] = l_run[h];
        }
#pragma unroll
        for (int j = 0; j < NT; ++j) *reinterpret_cast<float2*>(out + 4 + j * 8 + 2 * tq) = make_float2(o[j][2 * h], o[j][2 * h + 1]);
    }
    if (lacc) {
        // Accumulate: the two key lanes' partial rows of each query row are
        // rescaled to the fixed reference 2^ref_log2 (at least every score of
        // the layer: its queries and keys are RMS-normed, so |q.k| is bounded
        // by the norms' gains) and added into y (the unnormalised output)
        // and lacc (the softmax sum); a later kernel divides.  Exactly the
        // merge of the splits, in any order, with no second kernel.
        constexpr int VEC = HD / 32;
        __syncthreads();  // every warp's partial rows are written
        for (int qr = warp; qr < kAttnQ; qr += kAttnWarps) {
            const int ii = qt * kAttnQ + qr;
            if (ii >= mq) break;  // rows grow with qr (warp-uniform)
            const float* p0 = part + qr * PART;
            const float* p1 = part + (kAttnQ + qr) * PART;
            const float m0 = p0[0], m1 = p1[0];
            const float f0 = (m0 == -INFINITY) ? 0.f : exp2f(m0 - ref_log2);
            const float f1 = (m1 == -INFINITY) ? 0.f : exp2f(m1 - ref_log2);
            const int head = g * rep + ii / block_len, r = ii % block_len;
            float* dst = y + (row0 + r) * ((int64_t)nq * HD) + (int64_t)head * HD + VEC * lane;
            if constexpr (VEC == 4) {
                const float4 a = *reinterpret_cast<const float4*>(p0 + 4 + 4 * lane);
                const float4 b = *reinterpret_cast<const float4*>(p1 + 4 + 4 * lane);
                red_add_v4(dst, fmaf(a.x, f0, b.x * f1), fmaf(a.y, f0, b.y * f1), fmaf(a.z, f0, b.z * f1),
                           fmaf(a.w, f0, b.w * f1));
            } else {
                const float2 a = *reinterpret_cast<const float2*>(p0 + 4 + 2 * lane);
                const float2 b = *reinterpret_cast<const float2*>(p1 + 4 + 2 * lane);
                atomicAdd(dst, fmaf(a.x, f0, b.x * f1));
                atomicAdd(dst + 1, fmaf(a.y, f0, b.y * f1));
            }
            if (lane == 0) atomicAdd(lacc + (row0 + r) * nq + head, fmaf(p0[1], f0, p1[1] * f1));
        }
        return;
    }
    cluster.sync();  // every CTA's partial rows are written

    // merge: one warp per query row; lane k < kAttnKH nsplit reads partial
    // k's running max and sum (CTA k / kAttnKH, key lane k % kAttnKH), then
    // every lane sums its VEC dims over the partials
    constexpr int VEC = HD / 32;
    const int nparts = kAttnKH * nsplit;
    for (int qr = sp + warp * nsplit; qr < kAttnQ; qr += kAttnWarps * nsplit) {
        const int ii = qt * kAttnQ + qr;
        if (ii >= mq) break;  // rows grow with qr: none further (warp-uniform)
        float mk = -INFINITY, lk = 0.f;
        if (lane < nparts) {
            const float* src =
                cluster.map_shared_rank(part, lane / kAttnKH) + ((lane % kAttnKH) * kAttnQ + qr) * PART;
            mk = src[0];
            lk = src[1];
        }
        const float M = warp_max(mk);
        const float wk = (mk == -INFINITY) ? 0.f : exp2f(mk - M);
        const float L = warp_sum(lk * wk);
        float acc[VEC];
#pragma unroll
        for (int j = 0; j < VEC; ++j) acc[j] = 0.f;
#pragma unroll 8
        for (int k = 0; k < nparts; ++k) {
            const float w = __shfl_sync(0xffffffffu, wk, k);
            const float* src =
                cluster.map_shared_rank(part, k / kAttnKH) + ((k % kAttnKH) * kAttnQ + qr) * PART + 4 + VEC * lane;
            if constexpr (VEC == 4) {
                const float4 a = *reinterpret_cast<const float4*>(src);
                acc[0] = fmaf(a.x, w, acc[0]);
                acc[1] = fmaf(a.y, w, acc[1]);
                acc[2] = fmaf(a.z, w, acc[2]);
                acc[3] = fmaf(a.w, w, acc[3]);
            } else {
                const float2 a = *reinterpret_cast<const float2*>(src);
                acc[0] = fmaf(a.x, w, acc[0]);
                acc[1] = fmaf(a.y, w, acc[1]);
            }
        }
        const int head = g * rep + ii / block_len, r = ii % block_len;
        float* dst = y + (row0 + r) * ((int64_t)nq * HD) + (int64_t)head * HD + VEC * lane;
#pragma unroll
        for (int j = 0; j < VEC; ++j) dst[j] = acc[j] / L;
    }
    cluster.sync();  // no CTA leaves while another may still read its partial rows
}

// The global-memory merge of the key splits (long contexts): CTA (x, unit)
// merges query rows 2 x and 2 x + 1 of the unit's tile from their
// kAttnKH * nsplit partial rows, as the cluster merge does; four warps share
// a row, each taking every fourth partial row (four times the loads in flight
// of one warp a row), and meet in shared memory.
constexpr int kMergeWays = 4;
template <int HD>
__global__ void __launch_bounds__(256) attn_merge_kernel(const float* __restrict__ gpart, int nsplit, int qtiles,
                                                         int nkv, int nq, int block_len, float* __restrict__ y) {
    constexpr int PART = HD + 4, VEC = HD / 32;
    __shared__ float red[8][HD + 4];  // per warp: its share's sum and unnormalised output
    pdl_trigger();
    pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, way = warp % kMergeWays;
    const int unit = blockIdx.y, qr = blockIdx.x * (8 / kMergeWays) + warp / kMergeWays;
    const int qt = unit % qtiles, g = (unit / qtiles) % nkv, s = unit / (qtiles * nkv);
    const int rep = nq / nkv, mq = rep * block_len;
    const int ii = qt * kAttnQ + qr;
    const bool live = qr < kAttnQ && ii < mq;  // warp-uniform
    const int nparts = kAttnKH * nsplit;
    const float* base = gpart + (int64_t)unit * nparts * kAttnQ * PART + (int64_t)min(qr, kAttnQ - 1) * PART;
    float L = 0.f, acc[VEC];
#pragma unroll
    for (int j = 0; j < VEC; ++j) acc[j] = 0.f;
    if (live) {
        float M = -INFINITY;
        for (int p = lane; p < nparts; p += 32) M = fmaxf(M, base[(int64_t)p * kAttnQ * PART]);
        M = warp_max(M);
#pragma unroll 4
        for (int p = way; p < nparts; p += kMergeWays) {
            const float* src = base + (int64_t)p * kAttnQ * PART;
            const float2 ml = *reinterpret_cast<const float2*>(src);
            float a[VEC];
            if constexpr (VEC == 4) {
                const float4 v = *reinterpret_cast<const float4*>(src + 4 + 4 * lane);
                a[0] = v.x;
                a[1] = v.y;
                a[2] = v.z;
                a[3] = v.w;
            } else {
                const float2 v = *reinterpret_cast<const float2*>(src + 4 + 2 * lane);
                a[0] = v.x;
                a[1] = v.y;
            }
            const float w = (ml.x == -INFINITY) ? 0.f : exp2f(ml.x - M);
            L = fmaf(ml.y, w, L);
#pragma unroll
            for (int j = 0; j < VEC; ++j) acc[j] = fmaf(a[j], w, acc[j]);
        }
    }
    if (lane == 0) red[warp][0] = L;
#pragma unroll
    for (int j = 0; j < VEC; ++j) red[warp][4 + VEC * lane + j] = acc[j];
    __syncthreads();
    if (!live || way != 0) return;
    float Lt = 0.f;
#pragma unroll
    for (int w = 0; w < kMergeWays; ++w) Lt += red[warp + w][0];
    const int head = g * rep + ii / block_len, r = ii % block_len;
    float* dst = y + ((int64_t)s * block_len + r) * ((int64_t)nq * HD) + (int64_t)head * HD + VEC * lane;
#pragma unroll
    for (int j = 0; j < VEC; ++j) {
        float t = 0.f;
#pragma unroll
        for (int w = 0; w < kMergeWays; ++w) t += red[warp + w][4 + VEC * lane + j];
        dst[j] = t / Lt;
    }
}

// Cluster size (the key splits).  max_active[c]: clusters of c CTAs the
// device holds at once.  With few (sequence, kv head, query tile) units the
// largest cluster whose units all run in one wave, capped by the key steps
// of the longest context `max_ctx` (callers pass the sequences' capacity, so
// that the launch does not change as contexts grow); with many units, enough
// splits to cover the SMs.
// Global-memory merge (*gmerge): when the clusters leave a quarter of the SMs
// idle, the keys are split over plain CTAs instead (every SM busy, each with
// at least kAttnMinSteps key steps).  (Splitting the units of a batch that
// outnumber the SMs, to even out the waves, measured slower: the merge
// kernels cost more than the waves gain.)
constexpr int kAttnMinSteps = 2;  // key steps a CTA gets at least when the splits merge through global memory

static void attn_plan(int n_seqs, int block_len, int max_ctx, int nq, int nkv, int num_sms, const int* max_active,
                      int* qtiles, int* nsplit, bool* gmerge, bool allow_gmerge) {
    const int mq = (nq / nkv) * block_len;
    *qtiles = (mq + kAttnQ - 1) / kAttnQ;
    const int total = max_ctx + block_len;
    const int max_split = std::max(1, (total + kAttnStep - 1) / kAttnStep);
    const int units = nkv * *qtiles * n_seqs;
    const int slots = std::max(max_active[1], num_sms);  // CTAs the device holds at once
    const int want = std::min(max_split, std::max(1, (slots + units - 1) / units));
    int best = 1;
    for (int c = 1; c <= std::min(want, kAttnMaxCluster); ++c)
        if (max_active[c] >= std::min(units, max_active[1])) best = c;
    *nsplit = best;
    *gmerge = false;
    if (!allow_gmerge) return;
    if (units * best * 4 < num_sms * 3) {
        const int gsplit = std::min(max_split, std::max(1, (slots + units - 1) / units));
        if (gsplit > best && total >= kAttnMinSteps * kAttnStep * gsplit) {
            *nsplit = gsplit;
            *gmerge = true;
        }
    }
}

template <int HD, int ST>
static const int* attn_cluster_table(cudaStream_t st);

// The whole launch plan: stages (2: one CTA an SM with double-buffered key
// steps, for few units; 1: two CTAs an SM, when the units alone fill the
// SMs), query tiles, key splits, and whether they merge through global memory.
struct AttnPlan {
    int stages, qtiles, nsplit;
    bool gmerge;
};
template <int HD>
static AttnPlan attn_plan_hd(int n_seqs, int block_len, int max_ctx, int nq, int nkv, int num_sms, bool allow_gmerge) {
    AttnPlan p;
    const int mq = (nq / nkv) * block_len;
    const int units = nkv * ((mq + kAttnQ - 1) / kAttnQ) * n_seqs;
    p.stages = units >= num_sms ? 1 : 2;
    const int* table = p.stages == 1 ? attn_cluster_table<HD, 1>(0) : attn_cluster_table<HD, 2>(0);
    attn_plan(n_seqs, block_len, max_ctx, nq, nkv, num_sms, table, &p.qtiles, &p.nsplit, &p.gmerge, allow_gmerge);
    return p;
}
static AttnPlan attn_plan_any(int n_seqs, int block_len, int max_ctx, int nq, int nkv, int hd, int num_sms,
                              bool allow_gmerge) {
    return hd == 128 ? attn_plan_hd<128>(n_seqs, block_len, max_ctx, nq, nkv, num_sms, allow_gmerge)
                     : attn_plan_hd<64>(n_seqs, block_len, max_ctx, nq, nkv, num_sms, allow_gmerge);
}

int64_t attn_scratch_floats(int n_seqs, int block_len, int max_ctx, int nq, int nkv, int hd, int num_sms) {
    const AttnPlan p = attn_plan_any(n_seqs, block_len, max_ctx, nq, nkv, hd, num_sms, true);
    if (!p.gmerge) return 0;
    return (int64_t)nkv * p.qtiles * n_seqs * p.nsplit * kAttnKH * kAttnQ * (hd + 4);
}

int attn_kernels(int n_seqs, int block_len, int max_ctx, int nq, int nkv, int hd, int num_sms, int64_t part_floats) {
    const int64_t need = attn_scratch_floats(n_seqs, block_len, max_ctx, nq, nkv, hd, num_sms);
    return (need > 0 && part_floats >= need) ? 2 : 1;
}

// How many clusters of c = 1..16 CTAs of attn_cluster_kernel<HD, ST> the
// device holds at once (0 where it cannot place one), found once per process.
template <int HD, int ST>
static void attn_cluster_fill(int* table, cudaStream_t st);

template <int HD, int ST>
static const int* attn_cluster_table(cudaStream_t st) {
    // built once, thread-safely (a function-local static's initialiser runs
    // exactly once even when several host threads make their first call together)
    static const std::array<int, kAttnMaxCluster + 1> table = [st] {
        std::array<int, kAttnMaxCluster + 1> t{};
        attn_cluster_fill<HD, ST>(t.data(), st);
        return t;
    }();
    return table.data();
}

template <int HD, int ST>
static void attn_cluster_fill(int* table, cudaStream_t st) {
    for (auto kern : {attn_cluster_kernel<HD, ST, false>, attn_cluster_kernel<HD, ST, true>}) {
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(AttnSmem<HD, ST>));
        cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    }
    for (int c = 1; c <= kAttnMaxCluster; ++c) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(c, 1, 1);
        cfg.blockDim = dim3(kAttnWarps * 32);
        cfg.dynamicSmemBytes = sizeof(AttnSmem<HD, ST>);
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = c;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        // (the windowed variant takes the same resources within its launch bounds)
        if (cudaOccupancyMaxActiveClusters(&n, attn_cluster_kernel<HD, ST, false>, &cfg) != cudaSuccess) {
            cudaGetLastError();
            n = 0;
        }
        table[c] = n;
    }
    if (table[1] < 1) table[1] = 1;
}

template <int HD, int ST, bool WIN>
static int attention_launch(const AttnPlan& p, const float* qkv, int ld, int n_seqs, int block_len,
                            const AttnSeq* seqs_dev, int nq, int nkv, float scale_log2, float* part, float* y,
                            cudaStream_t st, const float* q_norm, const float* k_norm, const float2* rope, float eps,
                            int kv_ready) {
    dim3 grid(p.nsplit, nkv * p.qtiles, n_seqs);
    if (p.gmerge) {
        cudaError_t e = launch(attn_cluster_kernel<HD, ST, WIN>, grid, dim3(kAttnWarps * 32), sizeof(AttnSmem<HD, ST>),
                               st, qkv, ld, block_len, seqs_dev, nq, nkv, p.qtiles, p.nsplit, scale_log2, y, q_norm,
                               k_norm, rope, eps, part, kv_ready, (float*)nullptr, 0.f);
        if (e != cudaSuccess) return (int)e;
        return (int)launch(attn_merge_kernel<HD>, dim3(kAttnQ / (8 / kMergeWays), nkv * p.qtiles * n_seqs), dim3(256), 0, st,
                           (const float*)part, p.nsplit, p.qtiles, nkv, nq, block_len, y);
    }
    return (int)launch_cluster(attn_cluster_kernel<HD, ST, WIN>, grid, dim3(kAttnWarps * 32),
                               sizeof(AttnSmem<HD, ST>), st, p.nsplit, qkv, ld, block_len, seqs_dev, nq, nkv, p.qtiles,
                               p.nsplit, scale_log2, y, q_norm, k_norm, rope, eps, (float*)nullptr, kv_ready,
                               (float*)nullptr, 0.f);
}

template <int HD, int ST>
static int attention_run(const AttnPlan& p, const float* qkv, int ld, int n_seqs, int block_len,
                         const AttnSeq* seqs_dev, int nq, int nkv, float scale_log2, float* part, float* y,
                         cudaStream_t st, const float* q_norm, const float* k_norm, const float2* rope, float eps,
                         int kv_ready, bool windowed) {
    if (windowed)
        return attention_launch<HD, ST, true>(p, qkv, ld, n_seqs, block_len, seqs_dev, nq, nkv, scale_log2, part, y,
                                              st, q_norm, k_norm, rope, eps, kv_ready);
    return attention_launch<HD, ST, false>(p, qkv, ld, n_seqs, block_len, seqs_dev, nq, nkv, scale_log2, part, y, st,
                                           q_norm, k_norm, rope, eps, kv_ready);
}

template <int HD>
static int attention_hd(const float* qkv, int ld, int n_seqs, int block_len, const AttnSeq* seqs_dev, int max_ctx,
                        int nq, int nkv, float scale, float* part, int64_t part_floats, float* y, int num_sms,
                        cudaStream_t st, const float* q_norm, const float* k_norm, const float2* rope, float eps,
                        int kv_ready, bool windowed) {
    AttnPlan p = attn_plan_hd<HD>(n_seqs, block_len, max_ctx, nq, nkv, num_sms, true);
    const int64_t need = (int64_t)nkv * p.qtiles * n_seqs * p.nsplit * kAttnKH * kAttnQ * (HD + 4);
    if (p.gmerge && (part == nullptr || part_floats < need))  // no room for the partial rows: clusters
        p = attn_plan_hd<HD>(n_seqs, block_len, max_ctx, nq, nkv, num_sms, false);
    const float scale_log2 = scale * 1.4426950408889634f;
    if (p.stages == 1)
        return attention_run<HD, 1>(p, qkv, ld, n_seqs, block_len, seqs_dev, nq, nkv, scale_log2, part, y, st, q_norm,
                                    k_norm, rope, eps, kv_ready, windowed);
    return attention_run<HD, 2>(p, qkv, ld, n_seqs, block_len, seqs_dev, nq, nkv, scale_log2, part, y, st, q_norm,
                                k_norm, rope, eps, kv_ready, windowed);
}

int attention(const float* qkv, int ld, int n_seqs, int block_len, const AttnSeq* seqs_dev, int max_ctx, int nq,
              int nkv, int hd, float scale, float* part, int64_t part_floats, float* y, int num_sms, cudaStream_t st,
              const float* q_norm, const float* k_norm, const float2* rope, float eps, bool kv_ready, bool windowed) {
    if ((q_norm == nullptr) != (k_norm == nullptr)) return (int)cudaErrorInvalidValue;
    if (hd == 128)
        return attention_hd<128>(qkv, ld, n_seqs, block_len, seqs_dev, max_ctx, nq, nkv, scale, part, part_floats, y,
                                 num_sms, st, q_norm, k_norm, rope, eps, kv_ready ? 1 : 0, windowed);
    return attention_hd<64>(qkv, ld, n_seqs, block_len, seqs_dev, max_ctx, nq, nkv, scale, part, part_floats, y,
                            num_sms, st, q_norm, k_norm, rope, eps, kv_ready ? 1 : 0, windowed);
}

// ------------------------------------------------------------------ accumulate mode
// Few units (fewer than the SMs): the keys of each unit split over
// floor(SMs / units) plain CTAs (one wave, every SM busy for a single
// sequence), each adding its rescaled partial rows into y and lacc.
template <int HD>
static int attn_acc_splits(int n_seqs, int block_len, int max_ctx, int nq, int nkv, int num_sms) {
    const int mq = (nq / nkv) * block_len;
    const int units = nkv * ((mq + kAttnQ - 1) / kAttnQ) * n_seqs;
    if (units >= num_sms) return 0;
    const int* table = attn_cluster_table<HD, 2>(0);
    const int slots = std::max(table[1], num_sms);
    const int max_split = std::max(1, (max_ctx + block_len + kAttnStep - 1) / kAttnStep);
    const int nsplit = std::min(max_split, slots / units);
    return nsplit > 1 ? nsplit : 0;
}

int attn_acc_plan(int n_seqs, int block_len, int max_ctx, int nq, int nkv, int hd, int num_sms) {
    return hd == 128 ? attn_acc_splits<128>(n_seqs, block_len, max_ctx, nq, nkv, num_sms)
                     : attn_acc_splits<64>(n_seqs, block_len, max_ctx, nq, nkv, num_sms);
}

template <int HD, bool WIN>
static int attention_acc_hd(const float* qkv, int ld, int n_seqs, int block_len, const AttnSeq* seqs_dev, int nsplit,
                            int nq, int nkv, float scale, float* yacc, float* lacc, float ref_log2, cudaStream_t st,
                            const float* q_norm, const float* k_norm, const float2* rope, float eps, int kv_ready) {
    const int mq = (nq / nkv) * block_len, qtiles = (mq + kAttnQ - 1) / kAttnQ;
    attn_cluster_table<HD, 2>(0);  // the kernels' shared-memory attributes
    const float scale_log2 = scale * 1.4426950408889634f;
    return (int)launch(attn_cluster_kernel<HD, 2, WIN>, dim3(nsplit, nkv * qtiles, n_seqs), dim3(kAttnWarps * 32),
                       sizeof(AttnSmem<HD, 2>), st, qkv, ld, block_len, seqs_dev, nq, nkv, qtiles, nsplit, scale_log2,
                       yacc, q_norm, k_norm, rope, eps, (float*)nullptr, kv_ready, lacc, ref_log2);
}

int attention_acc(const float* qkv, int ld, int n_seqs, int block_len, const AttnSeq* seqs_dev, int nsplit, int nq,
                  int nkv, int hd, float scale, float* yacc, float* lacc, float ref_log2, cudaStream_t st,
                  const float* q_norm, const float* k_norm, const float2* rope, float eps, bool kv_ready,
                  bool windowed) {
    if (!q_norm || !k_norm || !yacc || !lacc || nsplit < 1 || (reinterpret_cast<uintptr_t>(yacc) & 15))
        return (int)cudaErrorInvalidValue;
    const int kr = kv_ready ? 1 : 0;
    if (hd == 128)
        return windowed ? attention_acc_hd<128, true>(qkv, ld, n_seqs, block_len, seqs_dev, nsplit, nq, nkv, scale,
                                                      yacc, lacc, ref_log2, st, q_norm, k_norm, rope, eps, kr)
                        : attention_acc_hd<128, false>(qkv, ld, n_seqs, block_len, seqs_dev, nsplit, nq, nkv, scale,
                                                       yacc, lacc, ref_log2, st, q_norm, k_norm, rope, eps, kr);
    return windowed ? attention_acc_hd<64, true>(qkv, ld, n_seqs, block_len, seqs_dev, nsplit, nq, nkv, scale, yacc,
                                                 lacc, ref_log2, st, q_norm, k_norm, rope, eps, kr)
                    : attention_acc_hd<64, false>(qkv, ld, n_seqs, block_len, seqs_dev, nsplit, nq, nkv, scale, yacc,
                                                  lacc, ref_log2, st, q_norm, k_norm, rope, eps, kr);
}

// ------------------------------------------------------------------ views by value
__global__ void __launch_bounds__(256) attn_views_store_kernel(const __grid_constant__ AttnViews views,
                                                                AttnSeq* __restrict__ dst) {
    pdl_wait();  // a kernel before this one may still read the views it replaces
    for (int i = threadIdx.x; i < views.n; i += blockDim.x) dst[i] = views.v[i];
}

int attn_views_store(const AttnViews& views, AttnSeq* dst, cudaStream_t st) {
    if (views.n < 0 || views.n > kViewsMax || dst == nullptr) return (int)cudaErrorInvalidValue;
    return (int)launch(attn_views_store_kernel, dim3(1), dim3(256), 0, st, views, dst);
}

// ------------------------------------------------------------------ wait expiry
// One warp waits, with the bounded wait every kernel of the library uses, on an
// mbarrier that nothing arrives on: the wait gives up after limit_ns, and the
// kernel raises *err exactly as a kernel whose data never arrived does.
__global__ void wait_expiry_kernel(int* __restrict__ err, unsigned long long limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    bool ok = true;
    if (threadIdx.x == 0) ok = mbar_wait(&bar, 0, limit_ns);
    if (!__all_sync(0xffffffffu, ok) && threadIdx.x == 0) atomicExch(err, 1);
}

int wait_expiry(int* err_flag, uint64_t limit_ns, cudaStream_t st) {
    return (int)launch(wait_expiry_kernel, dim3(1), dim3(32), 0, st, err_flag, (unsigned long long)limit_ns);
}

}  // namespace dflash
