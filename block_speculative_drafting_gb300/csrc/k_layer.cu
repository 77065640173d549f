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
#include <algorithm>

#include "common.cuh"
#include "kernels.cuh"

namespace dflash {

// Block-wide sum / max over 256 threads (deterministic tree order).
template <bool kMax>
DF_DEV float block_reduce_256(float v, float* red) {
    v = kMax ? warp_max(v) : warp_sum(v);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    if (threadIdx.x < 32) {
        float u = threadIdx.x < 8 ? red[threadIdx.x] : (kMax ? 0.f : 0.f);
        u = kMax ? warp_max(u) : warp_sum(u);
        if (threadIdx.x == 0) red[8] = u;
    }
    __syncthreads();
    float r = red[8];
    __syncthreads();
    return r;
}

// int8 code of v under scale sx (sx > 0), as an exact f16 integer
DF_DEV __half code_of(float v, float sx) {
    float q = rintf(__fdiv_rn(v, sx));
    q = fminf(fmaxf(q, -127.f), 127.f);
    return __float2half_rn(q);
}

__global__ void __launch_bounds__(256) rms_rows_kernel(const float* __restrict__ src, int ld_src, RowMap map, int n,
                                                       const float* __restrict__ w, float eps,
                                                       float* __restrict__ out_f32, int ld_out,
                                                       __half* __restrict__ out_codes, float* __restrict__ out_scale,
                                                       int ld_codes) {
    __shared__ float red[16];
    const int i = blockIdx.x;
    const int srow = (i / map.per) * map.stride + map.skip + (i % map.per);
    const float* x = src + (int64_t)srow * ld_src;
    float s = 1.f;
    if (w) {
        float ss = 0.f;
        for (int c = threadIdx.x; c < n; c += 256) ss = fmaf(x[c], x[c], ss);
        ss = block_reduce_256<false>(ss, red);
        s = 1.0f / sqrtf(ss / (float)n + eps);
    }
    if (out_f32) {
        for (int c = threadIdx.x; c < n; c += 256) out_f32[(int64_t)i * ld_out + c] = w ? x[c] * s * w[c] : x[c];
        return;
    }
    float amax = 0.f;
    for (int c = threadIdx.x; c < n; c += 256) amax = fmaxf(amax, fabsf(w ? x[c] * s * w[c] : x[c]));
    amax = block_reduce_256<true>(amax, red);
    const float sx = __fdiv_rn(amax, 127.0f);
    __half* q = out_codes + (int64_t)i * ld_codes;
    for (int c = threadIdx.x; c < n; c += 256) {
        const float v = w ? x[c] * s * w[c] : x[c];
        q[c] = sx > 0.f ? code_of(v, sx) : __float2half_rn(0.f);
    }
    if (threadIdx.x == 0) out_scale[i] = sx;
}

int rms_rows(const float* src, int ld_src, RowMap map, int rows, int n, const float* w, float eps, float* out_f32,
             int ld_out, __half* out_codes, float* out_scale, int ld_codes, cudaStream_t st) {
    if (rows <= 0) return 0;
    rms_rows_kernel<<<rows, 256, 0, st>>>(src, ld_src, map, n, w, eps, out_f32, ld_out, out_codes, out_scale,
                                          ld_codes);
    return (int)cudaGetLastError();
}

// A token outside [0, vocab) (only possible for anchors already on the
// device, which the host cannot check) embeds as a row of zeros.
__global__ void embed_rows_kernel(const float* __restrict__ embed, int H, int vocab,
                                  const uint32_t* __restrict__ anchor_tok, int mask_token, int block_len,
                                  float* __restrict__ h) {
    const int r = blockIdx.x;
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
               int block_len, float* h, cudaStream_t st) {
    embed_rows_kernel<<<n_seqs * block_len, 256, 0, st>>>(embed, H, vocab, anchor_tok, mask_token, block_len, h);
    return (int)cudaGetLastError();
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
__global__ void qk_norm_rope_kernel(float* __restrict__ qkv, int ld, int rows, int block_len,
                                    const int64_t* __restrict__ pos0, int nq, int nkv,
                                    const float* __restrict__ q_norm, const float* __restrict__ k_norm,
                                    const float* __restrict__ inv_freq, float eps) {
    constexpr int HD = 32 * E;
    const int wid = (int)((blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5);
    const int heads = nq + nkv;
    if (wid >= rows * heads) return;
    const int r = wid / heads, hh = wid % heads, lane = threadIdx.x & 31;
    float* p = qkv + (int64_t)r * ld + hh * HD;  // q heads then k heads are contiguous
    float v[E];
#pragma unroll
    for (int j = 0; j < E; ++j) v[j] = p[lane + 32 * j];
    const int64_t pos = pos0[r / block_len] + r % block_len;
    norm_rope_head<E>(v, hh < nq ? q_norm : k_norm, inv_freq, eps, pos, true);
#pragma unroll
    for (int j = 0; j < E; ++j) p[lane + 32 * j] = v[j];
}

int qk_norm_rope(float* qkv, int ld, int rows, int block_len, const int64_t* pos0_dev, int nq, int nkv, int hd,
                 const float* q_norm, const float* k_norm, const float* inv_freq, float eps, cudaStream_t st) {
    const int64_t warps = (int64_t)rows * (nq + nkv);
    const unsigned blocks = (unsigned)((warps * 32 + 255) / 256);
    if (hd == 128)
        qk_norm_rope_kernel<4><<<blocks, 256, 0, st>>>(qkv, ld, rows, block_len, pos0_dev, nq, nkv, q_norm, k_norm,
                                                       inv_freq, eps);
    else
        qk_norm_rope_kernel<2><<<blocks, 256, 0, st>>>(qkv, ld, rows, block_len, pos0_dev, nq, nkv, q_norm, k_norm,
                                                       inv_freq, eps);
    return (int)cudaGetLastError();
}

template <int E>
__global__ void kv_append_kernel(const float* __restrict__ kv, int n, int L, int nkv,
                                 const float* const* __restrict__ k_norm, const float* __restrict__ inv_freq,
                                 float eps, int64_t pos0, int64_t idx0, float* const* __restrict__ kstore,
                                 float* const* __restrict__ vstore, int64_t cap) {
    constexpr int HD = 32 * E;
    const int64_t wid = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
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
    norm_rope_head<E>(kvv, k_norm[l], inv_freq, eps, pos0 + r, true);
    float* kd = kstore[l] + ((int64_t)g * cap + idx0 + r) * HD;
    float* vd = vstore[l] + ((int64_t)g * cap + idx0 + r) * HD;
#pragma unroll
    for (int j = 0; j < E; ++j) {
        kd[lane + 32 * j] = kvv[j];
        vd[lane + 32 * j] = vv[j];
    }
}

int kv_append(const float* kv, int n, int L, int nkv, int hd, const float* const* k_norm_dev, const float* inv_freq,
              float eps, int64_t pos0, int64_t idx0, float* const* kstore_dev, float* const* vstore_dev, int64_t cap,
              cudaStream_t st) {
    if (n <= 0) return 0;
    const int64_t warps = (int64_t)n * L * nkv;
    const unsigned blocks = (unsigned)((warps * 32 + 255) / 256);
    if (hd == 128)
        kv_append_kernel<4><<<blocks, 256, 0, st>>>(kv, n, L, nkv, k_norm_dev, inv_freq, eps, pos0, idx0, kstore_dev,
                                                    vstore_dev, cap);
    else
        kv_append_kernel<2><<<blocks, 256, 0, st>>>(kv, n, L, nkv, k_norm_dev, inv_freq, eps, pos0, idx0, kstore_dev,
                                                    vstore_dev, cap);
    return (int)cudaGetLastError();
}

DF_DEV float silu_f(float a) { return a / (1.0f + expf(-a)); }

__global__ void __launch_bounds__(256) silu_mul_kernel(const float* __restrict__ gu, int ld_gu, int I,
                                                       float* __restrict__ out_f32, int ld_out,
                                                       __half* __restrict__ out_codes, float* __restrict__ out_scale,
                                                       int ld_codes) {
    __shared__ float red[16];
    const int r = blockIdx.x;
    const float* g = gu + (int64_t)r * ld_gu;
    const float* u = g + I;
    if (out_f32) {
        for (int c = threadIdx.x; c < I; c += 256) out_f32[(int64_t)r * ld_out + c] = silu_f(g[c]) * u[c];
        return;
    }
    float amax = 0.f;
    for (int c = threadIdx.x; c < I; c += 256) amax = fmaxf(amax, fabsf(silu_f(g[c]) * u[c]));
    amax = block_reduce_256<true>(amax, red);
    const float sx = __fdiv_rn(amax, 127.0f);
    __half* q = out_codes + (int64_t)r * ld_codes;
    for (int c = threadIdx.x; c < I; c += 256) {
        const float a = silu_f(g[c]) * u[c];
        q[c] = sx > 0.f ? code_of(a, sx) : __float2half_rn(0.f);
    }
    if (threadIdx.x == 0) out_scale[r] = sx;
}

int silu_mul(const float* gu, int ld_gu, int rows, int I, float* out_f32, int ld_out, __half* out_codes,
             float* out_scale, int ld_codes, cudaStream_t st) {
    if (rows <= 0) return 0;
    silu_mul_kernel<<<rows, 256, 0, st>>>(gu, ld_gu, I, out_f32, ld_out, out_codes, out_scale, ld_codes);
    return (int)cudaGetLastError();
}

// ------------------------------------------------------------------ attention
// One CTA per (key split, kv head x query tile, sequence).  The query tile is
// up to 64 (q head of the group, block row) pairs; keys are the context rows
// [lo, lo + n) then the block's rows; a split keeps an online softmax (running
// max in the log2 domain, running sum, unnormalised output) and writes it to
// `part`; attn_combine merges the splits.
constexpr int kAttnQ = 64;
constexpr int kAttnK = 32;

template <int HD>
struct AttnSmem {
    float q[kAttnQ][HD + 4];
    float k[kAttnK][HD + 4];
    float v[kAttnK][HD];
    float p[kAttnQ][kAttnK + 1];
};

template <int HD>
__global__ void __launch_bounds__(256) attn_split_kernel(const float* __restrict__ qkv, int ld, int block_len,
                                                         const AttnSeq* __restrict__ seqs, int nq, int nkv, int qtiles,
                                                         int nsplit, int keys_per_split, float scale_log2,
                                                         float* __restrict__ part) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    AttnSmem<HD>& sm = *reinterpret_cast<AttnSmem<HD>*>(smem_raw);
    constexpr int DV = HD / 16;  // float4 groups of the output a thread keeps
    const int sp = blockIdx.x, g = blockIdx.y / qtiles, qt = blockIdx.y % qtiles, s = blockIdx.z;
    const AttnSeq sq = seqs[s];
    const int rep = nq / nkv, mq = rep * block_len;
    const int total = sq.n + block_len;
    const int j0 = sp * keys_per_split, j1 = min(total, j0 + keys_per_split);
    const int tid = threadIdx.x, qrow = tid >> 2, sub = tid & 3;
    const int64_t row0 = (int64_t)s * block_len;

    // queries of this tile: query ii = qt*64 + qrow is head g*rep + ii / block_len at row ii % block_len
    for (int i = tid; i < kAttnQ * (HD / 4); i += 256) {
        const int qr = i / (HD / 4), c4 = i % (HD / 4), ii = qt * kAttnQ + qr;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (ii < mq) {
            const int head = g * rep + ii / block_len, r = ii % block_len;
            v = *reinterpret_cast<const float4*>(qkv + (row0 + r) * ld + (int64_t)head * HD + c4 * 4);
        }
        *reinterpret_cast<float4*>(&sm.q[qr][c4 * 4]) = v;
    }
    float m_run = -INFINITY, l_run = 0.f;
    float4 acc[DV];
#pragma unroll
    for (int d = 0; d < DV; ++d) acc[d] = make_float4(0.f, 0.f, 0.f, 0.f);

    for (int jt = j0; jt < j1; jt += kAttnK) {
        __syncthreads();  // previous tile's k/v/p no longer read
        for (int i = tid; i < kAttnK * (HD / 4); i += 256) {
            const int kr = i / (HD / 4), c4 = i % (HD / 4), j = jt + kr;
            float4 kk = make_float4(0.f, 0.f, 0.f, 0.f), vv = kk;
            if (j < j1) {
                if (j < sq.n) {
                    const int64_t off = ((int64_t)g * sq.cap + sq.lo + j) * HD + c4 * 4;
                    kk = *reinterpret_cast<const float4*>(sq.kc + off);
                    vv = *reinterpret_cast<const float4*>(sq.vc + off);
                } else {
                    const int64_t off = (row0 + (j - sq.n)) * ld + c4 * 4;
                    kk = *reinterpret_cast<const float4*>(qkv + off + (int64_t)(nq + g) * HD);
                    vv = *reinterpret_cast<const float4*>(qkv + off + (int64_t)(nq + nkv + g) * HD);
                }
            }
            *reinterpret_cast<float4*>(&sm.k[kr][c4 * 4]) = kk;
            *reinterpret_cast<float4*>(&sm.v[kr][c4 * 4]) = vv;
        }
        __syncthreads();
        // scores of keys sub + 4m
        float sc[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) sc[m] = 0.f;
#pragma unroll 4
        for (int d = 0; d < HD; d += 4) {
            const float4 qv = *reinterpret_cast<const float4*>(&sm.q[qrow][d]);
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const float4 kv4 = *reinterpret_cast<const float4*>(&sm.k[sub + 4 * m][d]);
                sc[m] = fmaf(qv.x, kv4.x, fmaf(qv.y, kv4.y, fmaf(qv.z, kv4.z, fmaf(qv.w, kv4.w, sc[m]))));
            }
        }
        float tmax = -INFINITY;
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            sc[m] = (jt + sub + 4 * m < j1) ? sc[m] * scale_log2 : -INFINITY;
            tmax = fmaxf(tmax, sc[m]);
        }
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
        const float m_new = fmaxf(m_run, tmax);
        const float corr = (m_run == -INFINITY) ? 0.f : exp2f(m_run - m_new);
        float psum = 0.f;
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const float p = (sc[m] == -INFINITY) ? 0.f : exp2f(sc[m] - m_new);
            sm.p[qrow][sub + 4 * m] = p;
            psum += p;
        }
        psum += __shfl_xor_sync(0xffffffffu, psum, 1);
        psum += __shfl_xor_sync(0xffffffffu, psum, 2);
        l_run = l_run * corr + psum;
        m_run = m_new;
#pragma unroll
        for (int d = 0; d < DV; ++d) {
            acc[d].x *= corr;
            acc[d].y *= corr;
            acc[d].z *= corr;
            acc[d].w *= corr;
        }
        __syncwarp();
        // the 4 threads of a query row wrote its 32 probabilities; they are in one warp
#pragma unroll 4
        for (int kk = 0; kk < kAttnK; ++kk) {
            const float p = sm.p[qrow][kk];
#pragma unroll
            for (int d = 0; d < DV; ++d) {
                const float4 vv = *reinterpret_cast<const float4*>(&sm.v[kk][4 * (sub + 4 * d)]);
                acc[d].x = fmaf(p, vv.x, acc[d].x);
                acc[d].y = fmaf(p, vv.y, acc[d].y);
                acc[d].z = fmaf(p, vv.z, acc[d].z);
                acc[d].w = fmaf(p, vv.w, acc[d].w);
            }
        }
    }
    // partial: [s][g][qt][sp][qrow] -> {m, l, -, -, acc[HD]} (16-byte aligned)
    const int64_t e = ((((int64_t)s * nkv + g) * qtiles + qt) * nsplit + sp) * kAttnQ + qrow;
    float* out = part + e * (HD + 4);
    if (sub == 0) {
        out[0] = m_run;
        out[1] = l_run;
    }
#pragma unroll
    for (int d = 0; d < DV; ++d) *reinterpret_cast<float4*>(out + 4 + 4 * (sub + 4 * d)) = acc[d];
}

// One warp per (sequence, block row, q head): merge the splits, divide by the sum.
template <int HD>
__global__ void attn_combine_kernel(const float* __restrict__ part, int n_seqs, int block_len, int nq, int nkv,
                                    int qtiles, int nsplit, float* __restrict__ y) {
    const int64_t wid = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
    if (wid >= (int64_t)n_seqs * block_len * nq) return;
    const int lane = threadIdx.x & 31;
    const int h = (int)(wid % nq), r = (int)((wid / nq) % block_len), s = (int)(wid / ((int64_t)nq * block_len));
    const int rep = nq / nkv, g = h / rep, ii = (h % rep) * block_len + r;
    const int qt = ii / kAttnQ, qrow = ii % kAttnQ;
    const int64_t base = (((int64_t)s * nkv + g) * qtiles + qt) * nsplit;
    float M = -INFINITY;
    for (int sp = 0; sp < nsplit; ++sp) M = fmaxf(M, part[((base + sp) * kAttnQ + qrow) * (HD + 4)]);
    constexpr int E = HD / 32;
    float o[E];
#pragma unroll
    for (int j = 0; j < E; ++j) o[j] = 0.f;
    float L = 0.f;
    for (int sp = 0; sp < nsplit; ++sp) {
        const float* pp = part + ((base + sp) * kAttnQ + qrow) * (HD + 4);
        const float m = pp[0];
        if (m == -INFINITY) continue;
        const float w = exp2f(m - M);
        L = fmaf(pp[1], w, L);
#pragma unroll
        for (int j = 0; j < E; ++j) o[j] = fmaf(pp[4 + lane + 32 * j], w, o[j]);
    }
    float* dst = y + ((int64_t)s * block_len + r) * ((int64_t)nq * HD) + (int64_t)h * HD;
#pragma unroll
    for (int j = 0; j < E; ++j) dst[lane + 32 * j] = o[j] / L;
}

static void attn_plan(int n_seqs, int block_len, int max_ctx, int nq, int nkv, int num_sms, int* qtiles, int* nsplit,
                      int* kps) {
    const int mq = (nq / nkv) * block_len;
    *qtiles = (mq + kAttnQ - 1) / kAttnQ;
    const int total = max_ctx + block_len;
    const int max_split = (total + kAttnK - 1) / kAttnK;
    const int units = nkv * *qtiles * n_seqs;
    int ns = std::max(1, std::min(max_split, (2 * num_sms + units - 1) / units));
    int k = (total + ns - 1) / ns;
    k = (k + kAttnK - 1) / kAttnK * kAttnK;
    *kps = k;
    *nsplit = (total + k - 1) / k;
}

int64_t attn_scratch_floats(int n_seqs, int block_len, int max_ctx, int nq, int nkv, int hd, int num_sms) {
    int qt, ns, kps;
    attn_plan(n_seqs, block_len, max_ctx, nq, nkv, num_sms, &qt, &ns, &kps);
    return (int64_t)n_seqs * nkv * qt * ns * kAttnQ * (hd + 4);
}

template <int HD>
static int attention_hd(const float* qkv, int ld, int n_seqs, int block_len, const AttnSeq* seqs_dev, int max_ctx,
                        int nq, int nkv, float scale, float* part, int64_t part_floats, float* y, int num_sms,
                        cudaStream_t st) {
    int qtiles, nsplit, kps;
    attn_plan(n_seqs, block_len, max_ctx, nq, nkv, num_sms, &qtiles, &nsplit, &kps);
    if ((int64_t)n_seqs * nkv * qtiles * nsplit * kAttnQ * (HD + 4) > part_floats) return (int)cudaErrorInvalidValue;
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(attn_split_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sizeof(AttnSmem<HD>));
        attr = true;
    }
    const float scale_log2 = scale * 1.4426950408889634f;
    dim3 grid(nsplit, nkv * qtiles, n_seqs);
    attn_split_kernel<HD><<<grid, 256, sizeof(AttnSmem<HD>), st>>>(qkv, ld, block_len, seqs_dev, nq, nkv, qtiles,
                                                                   nsplit, kps, scale_log2, part);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return (int)e;
    const int64_t warps = (int64_t)n_seqs * block_len * nq;
    attn_combine_kernel<HD><<<(unsigned)((warps * 32 + 255) / 256), 256, 0, st>>>(part, n_seqs, block_len, nq, nkv,
                                                                                  qtiles, nsplit, y);
    return (int)cudaGetLastError();
}

int attention(const float* qkv, int ld, int n_seqs, int block_len, const AttnSeq* seqs_dev, int max_ctx, int nq,
              int nkv, int hd, float scale, float* part, int64_t part_floats, float* y, int num_sms, cudaStream_t st) {
    if (hd == 128)
        return attention_hd<128>(qkv, ld, n_seqs, block_len, seqs_dev, max_ctx, nq, nkv, scale, part, part_floats, y,
                                 num_sms, st);
    return attention_hd<64>(qkv, ld, n_seqs, block_len, seqs_dev, max_ctx, nq, nkv, scale, part, part_floats, y,
                            num_sms, st);
}

}  // namespace dflash
