// Shared device helpers of the DFlash 2 block drafter library (sm_103a).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define DF_DEV __device__ __forceinline__

namespace dflash {

constexpr int kSMs = 152;  // GB300: 2 dies x 76 SMs (grids are sized from the device's count at run time)

// ---------------------------------------------------------------------------
// Order of the 576-byte chunks of a 4-bit matrix in memory.  Four 16-row tiles
// form a 64-row group; a (group, k-step) "super-chunk" is the group's four
// chunks of that k-step, 2304 contiguous bytes.  K is cut into K-blocks of KB
// k-steps (KB the largest divisor of the k-step count not above 32, i.e. at
// most 2048 columns), and super-chunks are stored [K-block][group][k-step in
// block]: a contiguous slice of the matrix needs the activations of one
// K-block only, and one group's k-steps inside a K-block are contiguous.
// ---------------------------------------------------------------------------
struct Q4Layout {
    int ngroups;  // 64-row groups of the whole (fused) matrix
    int ksteps;   // 64-column k-steps
    int kb;       // k-steps per K-block
};

__host__ __device__ __forceinline__ int q4_kblock_steps(int ksteps) {
    int best = 1;
    for (int d = 1; d <= 32 && d <= ksteps; ++d)
        if (ksteps % d == 0) best = d;
    return best;
}

// byte offset of the chunk of tile `tile` (16-row tile of the whole matrix)
// and k-step `ks`
__host__ __device__ __forceinline__ int64_t q4_chunk_offset(const Q4Layout& L, int tile, int ks) {
    const int g = tile >> 2, r = tile & 3;
    const int kblk = ks / L.kb, ksl = ks - kblk * L.kb;
    const int64_t sc = ((int64_t)kblk * L.ngroups + g) * L.kb + ksl;
    return sc * (4 * 576) + r * 576;
}

// The share of a streaming CTA: the CTAs of the grid are dealt out to the
// K-blocks in order (as evenly as they go), and the CTAs of one K-block split
// its span of super-chunks (groups g0 .. g0 + ng, every k-step of the block)
// into equal contiguous parts.
struct StreamGeom {
    int64_t lo, hi;  // super-chunks of this CTA inside its K-block's span
    int64_t base;    // global super-chunk index of the span's start
    int kblk;
};

__device__ __forceinline__ StreamGeom stream_geom(const Q4Layout& L, int g0, int ng) {
    const int nkb = L.ksteps / L.kb;
    const int G = gridDim.x, c = blockIdx.x;
    const int kblk = (int)((int64_t)c * nkb / G);
    const int first = (int)(((int64_t)kblk * G + nkb - 1) / nkb);
    const int nxt = (int)(((int64_t)(kblk + 1) * G + nkb - 1) / nkb);
    const int cnt = nxt - first, lc = c - first;
    const int64_t span = (int64_t)ng * L.kb;
    StreamGeom s;
    s.lo = span * lc / cnt;
    s.hi = span * (lc + 1) / cnt;
    s.base = ((int64_t)kblk * L.ngroups + g0) * L.kb;
    s.kblk = kblk;
    return s;
}

// ---------------------------------------------------------------------------
// Within a chunk ("q4 tile").
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

// int8 head layout: rows padded to 64; per (64-row group, 64-column k-step)
// a 4096-byte super-chunk of four 1024-byte tile chunks, group-major
// ([group][k-step][tile]).  In a tile chunk lane l = 4*gq + tq holds 32 bytes:
// for group-half gi in {0,1} and half s in {0,1} of it, 4 bytes of row gq then
// 4 bytes of row gq + 8, at columns 32*gi + 8*tq + 4*s + {0,1,2,3} -- the
// m16n8k16 A fragment order of the 4-bit layout, as bytes.
constexpr int kI8Chunk = 1024;
constexpr int kI8Super = 4 * kI8Chunk;
constexpr int kI8KStep = 64;

// byte offset of the head code at row n, column c (K = ksteps * 64)
__host__ __device__ __forceinline__ int64_t i8_byte_offset(int n, int c, int ksteps) {
    const int g = n >> 6, r = (n >> 4) & 3, rr = n & 15, gq = rr & 7, up = rr >> 3;
    const int ks = c >> 6, w = c & 63, gi = w >> 5, wc = w & 31, tq = wc >> 3, s = (wc >> 2) & 1, cc = wc & 3;
    return (((int64_t)g * ksteps + ks) * 4 + r) * kI8Chunk + (4 * gq + tq) * 32 + (gi * 2 + s) * 8 + up * 4 + cc;
}

// Four int8 (a u32) -> two half2 of exact integers: bytes (0,1) and (2,3).
DF_DEV void i8x4_to_half2x2(uint32_t v, uint32_t& lo, uint32_t& hi) {
    const uint32_t u = v ^ 0x80808080u;  // offset binary: b + 128
    uint32_t a, b;
    asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(a) : "r"(u), "r"(0x64646464u));
    asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(b) : "r"(u), "r"(0x64646464u));
    const uint32_t k1152 = 0x64806480u;  // 1152.0h = 1024 + 128
    __half2 ra = __hsub2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<const __half2*>(&k1152));
    __half2 rb = __hsub2(*reinterpret_cast<__half2*>(&b), *reinterpret_cast<const __half2*>(&k1152));
    lo = *reinterpret_cast<uint32_t*>(&ra);
    hi = *reinterpret_cast<uint32_t*>(&rb);
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch: a kernel launched with the programmatic
// stream-serialisation attribute may start while its predecessor runs; it
// reads or writes nothing the predecessor touches before pdl_wait().
DF_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
DF_DEV void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------------------
// mbarrier and bulk-copy (TMA, non-tensor) helpers.
DF_DEV uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
DF_DEV void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
DF_DEV void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}
DF_DEV void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
DF_DEV bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
DF_DEV uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}
// Bounded wait: gives up once `limit_ns` nanoseconds have passed, returning false.
DF_DEV bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (;;) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > limit_ns) return false;
    }
}
DF_DEV void bulk_g2s(void* dst_smem, const void* src_gmem, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst_smem)),
        "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}
DF_DEV void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
DF_DEV void red_add_v4(float* gaddr, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(gaddr), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

// Add a warp's partial sums of one 64-row group -- the m16n8k16 C fragments
// acc[r][h][e] of its four 16-row tiles r and two 8-token halves h (lane
// 4 gq + tq holds rows gq / gq + 8 of tokens h*8 + 2tq + {0,1}) -- each times
// its token's activation scale xs[h][e & 1], into y[t][row0 + ...] for
// tokens t < T.  The fragments of one (tile, half) go through a 512-byte
// per-warp shared scratch, so that each lane adds four consecutive rows of
// one token with a single 16-byte vector reduction (y and ldy 16-byte
// aligned): a quarter of the reductions of one add per value.
DF_DEV void dump_group_v4(const float (&acc)[4][2][4], const float (&xs)[2][2], float* y, int ldy, int row0, int T,
                          float* scratch, int lane) {
    const int gq = lane >> 2, tq = lane & 3;
    const int t = lane >> 2, q = lane & 3;  // the reading view: token t of the half, rows 4q .. 4q + 3
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            scratch[(2 * tq) * 16 + gq] = acc[r][h][0] * xs[h][0];
            scratch[(2 * tq + 1) * 16 + gq] = acc[r][h][1] * xs[h][1];
            scratch[(2 * tq) * 16 + gq + 8] = acc[r][h][2] * xs[h][0];
            scratch[(2 * tq + 1) * 16 + gq + 8] = acc[r][h][3] * xs[h][1];
            __syncwarp();
            const float4 v = *reinterpret_cast<const float4*>(scratch + t * 16 + 4 * q);
            const int tok = h * 8 + t;
            if (tok < T) red_add_v4(y + (int64_t)tok * ldy + row0 + r * 16 + 4 * q, v.x, v.y, v.z, v.w);
            __syncwarp();
        }
}

DF_DEV uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
    // (a & b) | c
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Eight offset nibbles -> four half2 of exact integers (code = nibble - 8):
// a nibble n ORed into the mantissa of 1024.0h reads 1024 + n (low nibbles)
// or 1024 + 16 n (high nibbles), and one subtraction (or multiply-add) per
// half2 removes the offset.  The mask-and-insert is one explicit LOP3 each
// (measured: fewer integer instructions than the compiler's own lowering).
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
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]),
          "f"(c[3]));
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

// int8 code of v under scale sx (sx > 0): round half to even of the IEEE
// quotient, clamped to [-127, 127]
DF_DEV int8_t code_of(float v, float sx) {
    float q = rintf(__fdiv_rn(v, sx));
    q = fminf(fmaxf(q, -127.f), 127.f);
    return (int8_t)(int)q;
}
DF_DEV float amax4(float4 v) { return fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))); }
// four codes in one word (all zero when sx is 0: a row of zeros)
DF_DEV uint32_t codes4(float4 v, float sx) {
    if (!(sx > 0.f)) return 0u;
    const uint32_t a = (uint8_t)code_of(v.x, sx), b = (uint8_t)code_of(v.y, sx);
    const uint32_t c = (uint8_t)code_of(v.z, sx), d = (uint8_t)code_of(v.w, sx);
    return a | (b << 8) | (c << 16) | (d << 24);
}
// silu(a) = a / (1 + exp(-a))
DF_DEV float silu_f(float a) { return a / (1.0f + expf(-a)); }

// Float -> u32 key whose unsigned order is the float order (no NaNs expected).
DF_DEV uint32_t float_order_key(float f) {
    uint32_t b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
// The inverse of float_order_key.
DF_DEV float float_of_order_key(uint32_t k) { return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k); }
// (value, index) -> u64 key: larger value wins, then the lower index.
DF_DEV unsigned long long argmax_key(float f, uint32_t idx) {
    return ((unsigned long long)float_order_key(f) << 32) | (unsigned long long)(0xFFFFFFFFu - idx);
}

}  // namespace dflash
