// Weight quantisers and packers (run once at dflash_init) and their inverses
// for the test hooks.
//
// 4-bit g32: per row n and group g of 32 columns, s = f16(max|w| / 7) (the
// division in f32), q = clamp(rint(w / f32(s)), -8, 7), q = 0 where s is 0.
// int8 rows (the head): s = max|w| / 127 in f32, q = clamp(rint(w / s), -127,
// 127), q = 0 for a zero row.  IEEE division and round-half-to-even
// throughout, so the codes are those of a plain scalar quantiser.
#include "common.cuh"
#include "kernels.cuh"

namespace dflash {

// scales[n][g] (f16) of a [N][K] f32 matrix, rows >= N and groups >= K/32 give 0
__global__ void q4_scales_kernel(const float* __restrict__ w, int N, int K, int Npad, int Gpad,
                                 __half* __restrict__ scales) {
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)Npad * Gpad) return;
    int n = (int)(i / Gpad), g = (int)(i % Gpad);
    float amax = 0.f;
    if (n < N && g * 32 < K) {
        const float4* p = reinterpret_cast<const float4*>(w + (int64_t)n * K + g * 32);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float4 v = p[j];
            amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
        }
    }
    scales[i] = __float2half_rn(__fdiv_rn(amax, 7.0f));
}

DF_DEV uint32_t q4_nibble(const float* __restrict__ w, int N, int K, int n, int c, float sf) {
    if (n >= N || c >= K || !(sf > 0.f)) return 8u;  // code 0
    float q = rintf(__fdiv_rn(w[(int64_t)n * K + c], sf));
    q = fminf(fmaxf(q, -8.f), 7.f);
    return (uint32_t)((int)q + 8);
}

// One thread per (tile, kstep, lane): the lane's 16 bytes, and (tq == 0) its
// 8 scale bytes, at the chunk of tile tile0 + tile in layout L.
__global__ void q4_pack_kernel(const float* __restrict__ w, int N, int K, const __half* __restrict__ scales,
                               int Gpad, int ntiles, Q4Layout L, int tile0, uint8_t* __restrict__ out) {
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int ksteps = L.ksteps;
    if (i >= (int64_t)ntiles * ksteps * 32) return;
    int lane = (int)(i % 32);
    int64_t chunk = i / 32;
    int ks = (int)(chunk % ksteps), tile = (int)(chunk / ksteps);
    int gq = lane >> 2, tq = lane & 3;
    int r0 = tile * 16 + gq, r1 = r0 + 8;
    uint32_t words[4];
#pragma unroll
    for (int gi = 0; gi < 2; ++gi) {
        int grp = ks * 2 + gi;
        float s0 = __half2float(scales[(int64_t)r0 * Gpad + grp]);
        float s1 = __half2float(scales[(int64_t)r1 * Gpad + grp]);
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            int c = grp * 32 + 8 * tq + 4 * s;
            uint32_t wd = 0;
            wd |= q4_nibble(w, N, K, r0, c + 0, s0) << 0;
            wd |= q4_nibble(w, N, K, r0, c + 1, s0) << 16;
            wd |= q4_nibble(w, N, K, r1, c + 0, s1) << 4;
            wd |= q4_nibble(w, N, K, r1, c + 1, s1) << 20;
            wd |= q4_nibble(w, N, K, r0, c + 2, s0) << 8;
            wd |= q4_nibble(w, N, K, r0, c + 3, s0) << 24;
            wd |= q4_nibble(w, N, K, r1, c + 2, s1) << 12;
            wd |= q4_nibble(w, N, K, r1, c + 3, s1) << 28;
            words[gi * 2 + s] = wd;
        }
    }
    uint8_t* base = out + q4_chunk_offset(L, tile0 + tile, ks);
    *reinterpret_cast<uint4*>(base + lane * 16) = make_uint4(words[0], words[1], words[2], words[3]);
    if (tq == 0) {
        __half sc[4] = {scales[(int64_t)r0 * Gpad + 2 * ks], scales[(int64_t)r1 * Gpad + 2 * ks],
                        scales[(int64_t)r0 * Gpad + 2 * ks + 1], scales[(int64_t)r1 * Gpad + 2 * ks + 1]};
        *reinterpret_cast<uint2*>(base + 512 + gq * 8) = *reinterpret_cast<uint2*>(sc);
    }
}

int q4_quantize_pack(const float* w_dev, int N, int K, uint8_t* packed, Q4Layout L, int tile0, __half* scratch,
                     cudaStream_t st) {
    int Npad = (N + 15) / 16 * 16, Gpad = L.ksteps * 2;
    int64_t ns = (int64_t)Npad * Gpad;
    q4_scales_kernel<<<(unsigned)((ns + 255) / 256), 256, 0, st>>>(w_dev, N, K, Npad, Gpad, scratch);
    int ntiles = Npad / 16;
    int64_t nt = (int64_t)ntiles * L.ksteps * 32;
    q4_pack_kernel<<<(unsigned)((nt + 255) / 256), 256, 0, st>>>(w_dev, N, K, scratch, Gpad, ntiles, L, tile0, packed);
    return (int)cudaGetLastError();
}

// Inverse of the packing: codes [N][K] and scale bits [N][K/32] of rows
// [tile0*16, tile0*16 + N).
__global__ void q4_unpack_kernel(const uint8_t* __restrict__ packed, Q4Layout L, int tile0, int N, int K,
                                 int8_t* __restrict__ codes, uint16_t* __restrict__ scales) {
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)N * K) return;
    int n = (int)(i / K), c = (int)(i % K);
    int tile = tile0 + n / 16, rr = n % 16, gq = rr % 8, up = rr / 8;
    int ks = c / 64, gi = (c % 64) / 32, wc = c % 32, tq = wc / 8, s = (wc % 8) / 4, cc = wc % 4;
    const uint8_t* base = packed + q4_chunk_offset(L, tile, ks);
    uint32_t word = reinterpret_cast<const uint32_t*>(base + (4 * gq + tq) * 16)[gi * 2 + s];
    // bit position of (row half `up`, column offset cc) inside the word
    int pos = (cc & 1 ? 16 : 0) + (cc & 2 ? 8 : 0) + (up ? 4 : 0);
    codes[i] = (int8_t)((int)((word >> pos) & 0xF) - 8);
    if (wc == 0) {
        const __half* sc = reinterpret_cast<const __half*>(base + 512 + gq * 8);
        scales[(int64_t)n * (K / 32) + c / 32] = __half_as_ushort(sc[gi * 2 + up]);
    }
}

int q4_unpack(const uint8_t* packed, Q4Layout L, int tile0, int N, int K, int8_t* codes, uint16_t* scales,
              cudaStream_t st) {
    int64_t n = (int64_t)N * K;
    q4_unpack_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(packed, L, tile0, N, K, codes, scales);
    return (int)cudaGetLastError();
}

// --------------------------------------------------------------- int8 rows
// One CTA per row (rows >= N: zero codes and scale).
__global__ void i8_rows_pack_kernel(const float* __restrict__ w, int N, int K, int ksteps, int8_t* __restrict__ packed,
                                    float* __restrict__ row_scale) {
    __shared__ float red[32];
    int n = blockIdx.x;
    float amax = 0.f;
    if (n < N)
        for (int c = threadIdx.x; c < K; c += blockDim.x) amax = fmaxf(amax, fabsf(w[(int64_t)n * K + c]));
    amax = warp_max(amax);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    if (threadIdx.x < 32) {
        float v = threadIdx.x < blockDim.x / 32 ? red[threadIdx.x] : 0.f;
        v = warp_max(v);
        if (threadIdx.x == 0) red[0] = v;
    }
    __syncthreads();
    float s = __fdiv_rn(red[0], 127.0f);
    if (threadIdx.x == 0) row_scale[n] = s;
    for (int c = threadIdx.x; c < ksteps * kI8KStep; c += blockDim.x) {
        int q = 0;
        if (n < N && c < K && s > 0.f) {
            float v = rintf(__fdiv_rn(w[(int64_t)n * K + c], s));
            q = (int)fminf(fmaxf(v, -127.f), 127.f);
        }
        packed[i8_byte_offset(n, c, ksteps)] = (int8_t)q;
    }
}

int i8_rows_quantize_pack(const float* w_dev, int N, int K, int Npad, int ksteps, int8_t* packed, float* row_scale,
                          cudaStream_t st) {
    i8_rows_pack_kernel<<<Npad, 256, 0, st>>>(w_dev, N, K, ksteps, packed, row_scale);
    return (int)cudaGetLastError();
}

__global__ void i8_unpack_kernel(const int8_t* __restrict__ packed, int N, int K, int ksteps, int8_t* __restrict__ codes) {
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)N * K) return;
    int n = (int)(i / K), c = (int)(i % K);
    codes[i] = packed[i8_byte_offset(n, c, ksteps)];
}

int i8_unpack(const int8_t* packed, int N, int K, int ksteps, int8_t* codes, cudaStream_t st) {
    int64_t n = (int64_t)N * K;
    i8_unpack_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(packed, N, K, ksteps, codes);
    return (int)cudaGetLastError();
}

}  // namespace dflash
