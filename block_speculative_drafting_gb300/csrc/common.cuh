// Shared device helpers of the DFlash 2 block drafter library (sm_103a).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define DF_DEV __device__ __forceinline__

namespace dflash {

constexpr int kSMs = 152;  // GB300: 2 dies x 76 SMs (grids are sized from the device's count at run time)

// ---------------------------------------------------------------------------
// 4-bit g32 packed layout ("q4 tile").
// A matrix [N][K] (N padded to a multiple of 16, K to a multiple of 64) is cut
// into 16-row tiles and 64-column k-steps (two 32-column quantisation
// groups).  Chunk (tile, kstep) is 576 bytes, tile-major:
//   bytes [0, 512): lane-major, 16 bytes per lane l = 4*gq + tq (gq = l / 4,
//     tq = l % 4): four u32 words w[gi*2 + s] for group gi in {0,1} of the
//     k-step and half s in {0,1} of the group.  Word (gi, s) holds eight
//     offset nibbles (code + 8) of rows gq and gq + 8 at the group's columns
//     8*tq + 4*s + {0,1,2,3}:
//        bits  0- 3: row gq,   col +0   bits 16-19: row gq,   col +1
//        bits  4- 7: row gq+8, col +0   bits 20-23: row gq+8, col +1
//        bits  8-11: row gq,   col +2   bits 24-27: row gq,   col +3
//        bits 12-15: row gq+8, col +2   bits 28-31: row gq+8, col +3
//     so that four LOP3s turn a word into the m16n8k16 A fragment
//     {a0a1, a2a3, a4a5, a6a7} of a 16x16 f16 tile whose k slot 2*tq + {0,1}
//     is column 8*tq + 4*s + {0,1} and slot 2*tq + 8 + {0,1} is column
//     8*tq + 4*s + {2,3} (a permutation of the group's columns that the B
//     fragment follows as well, so the dot products are unchanged).
//   bytes [512, 576): f16 scales, 8 bytes per gq: s[gq][g0], s[gq+8][g0],
//     s[gq][g1], s[gq+8][g1] (g0, g1 the k-step's two groups).
// ---------------------------------------------------------------------------
constexpr int kQ4Chunk = 576;
constexpr int kQ4KStep = 64;

// int8 head layout ("i8 tile"): rows padded to 16; per (tile, 32-column
// k-step) 512 bytes, lane-major 16 bytes per lane l = 4*gq + tq:
//   [row gq cols 8tq..8tq+3][row gq+8 cols 8tq..+3][row gq cols 8tq+4..+7][row gq+8 cols 8tq+4..+7]
// = the m16n8k32 s8 A fragment {a0,a1,a2,a3} with k slot 4tq+{0..3} <-> column
// 8tq+{0..3} and slot 16+4tq+{0..3} <-> column 8tq+4+{0..3}.
constexpr int kI8Chunk = 512;
constexpr int kI8KStep = 32;

DF_DEV uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
    // (a & b) | c
    uint32_t d;
    asm volatile("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Eight offset nibbles -> four half2 of exact integers (code = nibble - 8).
DF_DEV void unpack_q4_word(uint32_t w, uint32_t (&a)[4]) {
    const uint32_t kLo = 0x000F000Fu, kHi = 0x00F000F0u, kMagic = 0x64006400u;  // 0x6400 = 1024.0h
    const uint32_t kSub = 0x64086408u;                                        // 1032.0h: 1024 + 8
    const uint32_t kMul = 0x2C002C00u;                                        // 1/16
    const uint32_t kAdd = 0xD480D480u;                                        // -72.0h: -(64 + 8)
    uint32_t h0 = lop3_and_or(w, kLo, kMagic);
    uint32_t h1 = lop3_and_or(w, kHi, kMagic);
    uint32_t w8 = w >> 8;
    uint32_t h2 = lop3_and_or(w8, kLo, kMagic);
    uint32_t h3 = lop3_and_or(w8, kHi, kMagic);
    __half2 r0 = __hsub2(*reinterpret_cast<__half2*>(&h0), *reinterpret_cast<const __half2*>(&kSub));
    __half2 r1 = __hfma2(*reinterpret_cast<__half2*>(&h1), *reinterpret_cast<const __half2*>(&kMul),
                         *reinterpret_cast<const __half2*>(&kAdd));
    __half2 r2 = __hsub2(*reinterpret_cast<__half2*>(&h2), *reinterpret_cast<const __half2*>(&kSub));
    __half2 r3 = __hfma2(*reinterpret_cast<__half2*>(&h3), *reinterpret_cast<const __half2*>(&kMul),
                         *reinterpret_cast<const __half2*>(&kAdd));
    a[0] = *reinterpret_cast<uint32_t*>(&r0);
    a[1] = *reinterpret_cast<uint32_t*>(&r1);
    a[2] = *reinterpret_cast<uint32_t*>(&r2);
    a[3] = *reinterpret_cast<uint32_t*>(&r3);
}

// D = A(16x16 f16) * B(16x8 f16) + C, f32 accumulate (warp-level tensor-core MMA).
DF_DEV void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1, const float (&c)[4]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]),
          "f"(c[3]));
}

// D = A(16x32 s8) * B(32x8 s8) + C, s32 accumulate.
DF_DEV void mma_s8_16832(int (&d)[4], const uint4& a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
        : "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b0), "r"(b1));
}

// Streaming 16-byte load that skips L1 (weights are read once per launch).
DF_DEV uint4 ldg_stream_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
DF_DEV uint2 ldg_stream_v2(const void* p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

DF_DEV float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
DF_DEV float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Float -> u32 key whose unsigned order is the float order (no NaNs expected).
DF_DEV uint32_t float_order_key(float f) {
    uint32_t b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
// (value, index) -> u64 key: larger value wins, then the lower index.
DF_DEV unsigned long long argmax_key(float f, uint32_t idx) {
    return ((unsigned long long)float_order_key(f) << 32) | (unsigned long long)(0xFFFFFFFFu - idx);
}

}  // namespace dflash
