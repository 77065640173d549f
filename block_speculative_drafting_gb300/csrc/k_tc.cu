// Dense contractions of many rows on the fifth-generation tensor cores
// (tcgen05) with the weights converted in the kernel: the 4-bit g32 matrices
// of page "cortiq-engine 0.8.75 — src/gpu_wgpu/dflash_dev.rs" (`Dev::q4`:
// four-bit codes with one scale per 32 columns against int8 activations) and
// the int8 head (`Dev::q8`, the head of page "cortiq-engine 0.8.71 —
// src/dflash.rs", `block_dev`) applied to a batch of rows.  The library runs
// the products from dense f16 weight copies (k_tc_pair.cu); these kernels
// are the form without the copies (the model option "dense" at 0), and this
// file also holds the host side the tensor-core kernels share: tensor maps,
// the f16 activation codes, the dense copies' conversion.
//
// 4-bit (q4_tc2_kernel): y[t][n] = xs[t] * sum_k (s[n][k/32] q[n][k]) x[t][k],
// the quantised matvec with the group scale folded into the weight.  s (f16)
// times q (-8..7) needs up to 14 significant bits, so the weight goes to the
// tensor core as the exact sum of two f16 values, hi = f16(s q) and
// lo = f16(s q - hi) (an fma; the remainder is representable), and every k
// slice runs two MMAs (x . hi + x . lo).  The int8 codes of x are exact in
// f16, so every product is exact.
// Head (tc_head_kernel): logits[t][n] = xs[t] * sw[n] * sum_k q[n][k] x[t][k],
// one MMA a k slice on exact f16 integers, and the draft token's argmax
// (lowest index among equal values) folded into the epilogue.
//
// Accumulation.  The tensor core's f32 accumulation truncates, which over
// long K shrinks sums measurably; so the head's tensor memory only ever holds
// a chunk of kTcChunk k-blocks (512 columns), in two alternating
// accumulators, and the converter warps drain each finished chunk into exact
// int32 registers (a chunk's integer sum is below 512 * 127 * 127 < 2^24, so
// the f32 chunk value is the exact integer).  The 4-bit kernel splits K over
// CTAs in slices of at most 2048 columns instead.
//
// The head's CTA computes a 128-row x 128-output tile, D[t][n], in tensor
// memory (128 lanes x 128 f32 columns per accumulator).  Roles:
//   warp 8 (one lane): TMA -- the f16 activation tile of each 64-column
//     k-block (cp.async.bulk.tensor over a tensor map of the activation
//     codes as f16, 128-byte swizzle: it lands in the layout the MMA reads)
//     into the activation ring, and the packed codes of the k-block's two
//     64-row groups (cp.async.bulk) into the raw ring;
//   warps 0-7: convert a raw stage into a converted stage (the codes as f16)
//     in the K-major 128-byte-swizzled layout the MMA descriptors name; drain
//     finished chunks; run the epilogue (warp w reads tensor-memory lanes
//     32 (w % 4) .., columns 64 (w / 4) ..);
//   warp 9: allocates the tensor memory; one lane issues the MMAs
//     (tcgen05.mma kind::f16, M 128, N 128, K 16) and commits every converted
//     stage and every finished chunk.
// Every wait is bounded (1 s of %globaltimer): on expiry the kernel raises the
// error flag, the roles stop, copies and MMAs in flight are waited for
// (bounded), and the tensor memory is freed.
#include <cuda.h>

#include <algorithm>
#include <cstring>

#include "common.cuh"
#include "kernels.cuh"
#include "tc.cuh"

namespace dflash {

constexpr int kTcM = 128;    // rows of a tile: MMA M, tensor-memory lanes
constexpr int kTcN = 128;    // outputs of a tile: MMA N, tensor-memory columns of one accumulator
constexpr int kTcKB = 64;    // columns of a k-block: one 128-byte swizzle row of f16
constexpr int kTcChunk = 8;  // k-blocks accumulated in tensor memory before a drain
constexpr int kTcCvt = 3;    // converted stages
constexpr int kTcCvtWarps = 8;
constexpr int kTcThreads = (kTcCvtWarps + 2) * 32;
constexpr int kTcTmaWarp = kTcCvtWarps, kTcMmaWarp = kTcCvtWarps + 1;
constexpr int kTcCols = 64;  // accumulator columns a converter thread drains
constexpr uint64_t kTcWait = 1000000000ull;  // ns a wait may take before the kernel gives up
static_assert(kTcChunk >= 3, "a chunk is drained at the third k-block of the next one");
static_assert(kTcCvtWarps * 32 * kTcCols == kTcM * kTcN, "drain split");

constexpr int kTcMaxRaw = 12;  // raw stages at most (the control block's barrier arrays)
constexpr int kTcAct = 4;      // activation stages
constexpr int kTcA = kTcM * kTcKB * 2;  // f16 activation tile (swizzled by the TMA)
// Raw stages are compact (packed weights), so the ring is deep: enough bytes
// in flight to cover the load latency at the tensor cores' pace; converted
// stages (f16) are double-buffered.
struct TcShape {
    static constexpr int kRawBytes = 2 * kI8Super;  // two 64-row groups of one k-block
    static constexpr int kB = kTcN * kTcKB * 2;     // f16 weight tile, swizzled
    static constexpr int kCvtBytes = kB;
    static constexpr int kRaw = 8;                  // raw stages
    static constexpr size_t kSmem = 1024 /*alignment slack*/ + 1024 /*control*/ + (size_t)kTcAct * kTcA +
                                    (size_t)kTcCvt * kCvtBytes + (size_t)kRaw * kRawBytes;
    static_assert(kCvtBytes % 1024 == 0 && kRawBytes % 128 == 0, "stage alignment");
    static_assert(kRaw <= kTcMaxRaw && kSmem <= 227 * 1024, "shared memory");
};

// Instruction descriptor of tcgen05.mma kind::f16: D f32 (bits 4-5 = 1), A and
// B f16 (bits 7-9, 10-12 = 0), both K-major (bits 15, 16 = 0), N >> 3 at bits
// 17-22, M >> 4 at bits 24-28.
constexpr uint32_t kTcIdesc = (1u << 4) | ((uint32_t)(kTcN >> 3) << 17) | ((uint32_t)(kTcM >> 4) << 24);

// byte offset of the 16-byte chunk c (columns 8c .. 8c+7) of row r in such a tile
DF_DEV uint32_t tc_swz(int r, int c) { return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4)); }

DF_DEV void tc_mma(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(kTcIdesc), "r"(accumulate)
        : "memory");
}
DF_DEV void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}




// hi / lo of s * q for four half2 of codes q
DF_DEV void split_scaled(const uint32_t (&q)[4], uint32_t s2, uint4& hi, uint4& lo) {
    const __half2 s = *reinterpret_cast<const __half2*>(&s2);
    uint32_t h[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __half2 qi = *reinterpret_cast<const __half2*>(&q[i]);
        const __half2 hh = __hmul2(qi, s);
        const __half2 ll = __hfma2(qi, s, __hneg2(hh));
        h[i] = *reinterpret_cast<const uint32_t*>(&hh);
        l[i] = *reinterpret_cast<const uint32_t*>(&ll);
    }
    hi = make_uint4(h[0], h[1], h[2], h[3]);
    lo = make_uint4(l[0], l[1], l[2], l[3]);
}

struct TcCtl {
    uint64_t raw_full[kTcMaxRaw], raw_empty[kTcMaxRaw], act_full[kTcAct], act_empty[kTcAct], cvt_full[kTcCvt],
        cvt_empty[kTcCvt], dfull[2], dempty[2], fin;
    uint32_t tmem;
    int abort;
};
static_assert(sizeof(TcCtl) <= 1024, "control block");

struct TcArgs {
    const uint8_t* w;          // 4-bit: packed matrix; head: int8 super-chunks
    Q4Layout L;                // 4-bit layout (head: ksteps only)
    int g0;                    // first 64-row group of the sub-matrix (4-bit)
    int N;                     // outputs (4-bit: multiple of 64; head: vocab)
    const float* xscale;       // [T]
    int T;
    float* y;                  // [T][ldy] (head: logits, may be null)
    int ldy;
    int accumulate;            // 4-bit: add into y
    int kb_per_split;          // k-blocks per CTA along grid z
    const float* wscale;       // head: row scales [>= N]
    unsigned long long* keys;  // head: argmax keys [T]
    int* err;
    // dense head: the exactness guard -- squared code norms of the rows [T]
    // and of the vocabulary rows [N], the f16 codes of both, the row length K
    // and the largest norm product the f32 sums are trusted under
    const int* xn2;
    const int* wn2;
    const __half* xf;
    const __half* wf;
    int K;
    unsigned long long bound;
    unsigned long long wn2_max;  // the largest of wn2: rows under the bound against it skip the check
    int y_tma;                   // dense kernels: y is written through the output tensor map
};

__global__ void __launch_bounds__(kTcThreads, 1) tc_head_kernel(const __grid_constant__ CUtensorMap xmap, TcArgs a) {
    using S = TcShape;
    extern __shared__ __align__(1024) unsigned char sm_raw[];
    // 1024-aligned base (the swizzled tiles need it)
    unsigned char* sm = sm_raw + ((1024 - (smem_addr(sm_raw) & 1023)) & 1023);
    TcCtl& ctl = *reinterpret_cast<TcCtl*>(sm);
    unsigned char* act = sm + 1024;
    unsigned char* cvt = act + kTcAct * kTcA;
    unsigned char* raw = cvt + kTcCvt * S::kCvtBytes;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // the row tiles of one output tile run together (x = row tile): the
    // weights are the large operand
    const int m0 = blockIdx.x * kTcM, nt = blockIdx.y;
    const int ksteps = a.L.ksteps;
    const int kb_lo = blockIdx.z * a.kb_per_split, kb_hi = min(ksteps, kb_lo + a.kb_per_split);
    const int nkb = kb_hi - kb_lo;
    const int nchunks = (nkb + kTcChunk - 1) / kTcChunk;
    const int ngroups_n = (a.N + 63) / 64;  // 64-row groups of the outputs

    constexpr int kTcRaw = S::kRaw;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kTcRaw; ++i) {
            mbar_init(&ctl.raw_full[i], 1);
            mbar_init(&ctl.raw_empty[i], kTcCvtWarps);
        }
        for (int i = 0; i < kTcAct; ++i) {
            mbar_init(&ctl.act_full[i], 1);
            mbar_init(&ctl.act_empty[i], 1);
        }
        for (int i = 0; i < kTcCvt; ++i) {
            mbar_init(&ctl.cvt_full[i], kTcCvtWarps);
            mbar_init(&ctl.cvt_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&ctl.dfull[i], 1);
            mbar_init(&ctl.dempty[i], kTcCvtWarps);
        }
        mbar_init(&ctl.fin, 1);
        ctl.abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kTcMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&ctl.tmem)),
                     "r"(2 * kTcN)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl.tmem;
    pdl_trigger();
    pdl_wait();

    auto give_up = [&]() {
        atomicExch(a.err, 1);
        *reinterpret_cast<volatile int*>(&ctl.abort) = 1;
    };
    auto aborted = [&]() { return *reinterpret_cast<volatile int*>(&ctl.abort) != 0; };

    if (warp == kTcTmaWarp) {
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(&xmap) : "memory");
            int issued = 0;
            int ng = 0;  // valid 64-row groups of this tile
            for (int gg = 0; gg < kTcN / 64; ++gg) ng += (nt * (kTcN / 64) + gg < ngroups_n) ? 1 : 0;
            const int wbytes = kI8Super;
            for (int i = 0; i < nkb; ++i) {
                const int r = i % kTcRaw, sa = i % kTcAct;
                bool ok = true;
                if (i >= kTcRaw) ok = mbar_wait(&ctl.raw_empty[r], ((i / kTcRaw) - 1) & 1, kTcWait);
                if (ok && i >= kTcAct) ok = mbar_wait(&ctl.act_empty[sa], ((i / kTcAct) - 1) & 1, kTcWait);
                if (!ok) give_up();
                if (!ok || aborted()) break;
                fence_proxy_async_smem();
                const int kb = kb_lo + i;
                mbar_arrive_expect_tx(&ctl.act_full[sa], (uint32_t)kTcA);
                tma_load_2d(act + sa * kTcA, &xmap, kb * kTcKB, m0, &ctl.act_full[sa]);
                unsigned char* dst = raw + r * S::kRawBytes;
                mbar_arrive_expect_tx(&ctl.raw_full[r], (uint32_t)(ng * wbytes));
                for (int gg = 0; gg < ng; ++gg) {
                    const int grp = nt * (kTcN / 64) + gg;
                    const uint8_t* src = a.w + ((int64_t)grp * ksteps + kb) * kI8Super;
                    bulk_g2s(dst + gg * wbytes, src, (uint32_t)wbytes, &ctl.raw_full[r]);
                }
                issued = i + 1;
            }
            // copies still in flight land before the CTA can leave
            for (int i = max(0, issued - kTcRaw); i < issued; ++i)
                mbar_wait(&ctl.raw_full[i % kTcRaw], (i / kTcRaw) & 1, kTcWait);
            for (int i = max(0, issued - kTcAct); i < issued; ++i)
                mbar_wait(&ctl.act_full[i % kTcAct], (i / kTcAct) & 1, kTcWait);
        }
    } else if (warp == kTcMmaWarp) {
        if (lane == 0) {
            for (int i = 0; i < nkb; ++i) {
                const int st = i % kTcCvt, ch = i / kTcChunk, buf = ch & 1;
                const bool first = i % kTcChunk == 0;
                bool ok = true;
                const int sx = i % kTcAct;
                if (first && ch >= 2) ok = mbar_wait(&ctl.dempty[buf], ((ch >> 1) - 1) & 1, kTcWait);
                if (ok) ok = mbar_wait(&ctl.act_full[sx], (i / kTcAct) & 1, kTcWait);
                if (ok) ok = mbar_wait(&ctl.cvt_full[st], (i / kTcCvt) & 1, kTcWait);
                if (!ok) give_up();
                if (!ok || aborted()) break;
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(buf * kTcN);
                const uint32_t sa = smem_addr(act + sx * kTcA);
                const uint32_t sb = smem_addr(cvt + st * S::kCvtBytes);
#pragma unroll
                for (int j = 0; j < kTcKB / 16; ++j) {
                    tc_mma(d, tc_desc_sw128(sa + 32 * j), tc_desc_sw128(sb + 32 * j), (first && j == 0) ? 0u : 1u);
                }
                tc_commit(&ctl.cvt_empty[st]);
                tc_commit(&ctl.act_empty[sx]);
                if (i % kTcChunk == kTcChunk - 1 || i == nkb - 1) tc_commit(&ctl.dfull[buf]);
            }
            // arrives once every MMA issued so far has completed (the memory is freed after it)
            tc_commit(&ctl.fin);
            mbar_wait(&ctl.fin, 0, kTcWait);
        }
    } else {
        // ---------------------------------------------------------------- converters
        const int sub = warp & 3, half = warp >> 2;  // tensor-memory lane quadrant, 64-column half
        const uint32_t lane_base = (uint32_t)(32 * sub) << 16;
        int32_t iacc[kTcCols];
#pragma unroll
        for (int j = 0; j < kTcCols; ++j) iacc[j] = 0;
        bool ok = true;
        int drained = 0;
        // add finished chunk `ch` (tensor-memory accumulator ch & 1) into the registers
        auto drain = [&](int ch) {
            const int buf = ch & 1;
            const bool w = mbar_wait(&ctl.dfull[buf], (ch >> 1) & 1, kTcWait);
            if (!w) give_up();
            if (__any_sync(0xffffffffu, !w || aborted())) {
                ok = false;
                return;
            }
            tc_fence_after();
            const uint32_t base = tmem + lane_base + (uint32_t)(buf * kTcN + half * kTcCols);
#pragma unroll
            for (int c = 0; c < kTcCols; c += 16) {
                uint32_t r[16];
                tc_ld16(base + (uint32_t)c, r);
                tc_wait_ld();
#pragma unroll
                for (int q = 0; q < 16; ++q) iacc[c + q] += (int32_t)__uint_as_float(r[q]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl.dempty[buf]);
        };

        for (int i = 0; i < nkb && ok; ++i) {
            const int r = i % kTcRaw, c = i % kTcCvt;
            bool w = mbar_wait(&ctl.raw_full[r], (i / kTcRaw) & 1, kTcWait);
            if (w && i >= kTcCvt) w = mbar_wait(&ctl.cvt_empty[c], ((i / kTcCvt) - 1) & 1, kTcWait);
            if (!w) give_up();
            // warp-uniform: every lane leaves together
            if (__any_sync(0xffffffffu, !w || aborted())) {
                ok = false;
                break;
            }
            const unsigned char* rs = raw + r * S::kRawBytes;
            unsigned char* cs = cvt + c * S::kCvtBytes;
            // weights: 8 chunks of 16 rows x 64 columns, chunk w to warp w, one
            // lane slot a lane.  Lane L converts slot 4 gq + tq with, in
            // quarter-warp q = L / 8, gq = 2q (L % 8 < 4) or 2q ^ 5: the eight
            // 16-byte stores of a quarter then fall on eight distinct swizzled
            // positions (their rows differ in bit 2).
            {
                const int gg = warp >> 2, rr = warp & 3;
                const int qw = lane >> 3, jw = lane & 7;
                const int gq = (jw < 4) ? 2 * qw : ((2 * qw) ^ 5), tq = jw & 3;
                const int slot = 4 * gq + tq;
                const int nl0 = gg * 64 + rr * 16 + gq, nl1 = nl0 + 8;
                unsigned char* bt = cs;
                const bool valid = nt * (kTcN / 64) + gg < ngroups_n;
                uint4 w[2] = {make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u)};
                if (valid) {
                    const unsigned char* ch = rs + gg * kI8Super + rr * kI8Chunk + slot * 32;
                    w[0] = *reinterpret_cast<const uint4*>(ch);
                    w[1] = *reinterpret_cast<const uint4*>(ch + 16);
                }
#pragma unroll
                for (int gi = 0; gi < 2; ++gi) {
                    // words (s, up) of group half gi: four codes of row gq + 8 up at
                    // columns 32 gi + 8 tq + 4 s + 0..3
                    uint4 r0, r1;  // rows gq, gq + 8
                    i8x4_to_half2x2(w[gi].x, r0.x, r0.y);
                    i8x4_to_half2x2(w[gi].z, r0.z, r0.w);
                    i8x4_to_half2x2(w[gi].y, r1.x, r1.y);
                    i8x4_to_half2x2(w[gi].w, r1.z, r1.w);
                    *reinterpret_cast<uint4*>(bt + tc_swz(nl0, 4 * gi + tq)) = r0;
                    *reinterpret_cast<uint4*>(bt + tc_swz(nl1, 4 * gi + tq)) = r1;
                }
            }
            // the converted tiles are read by the tensor cores (async proxy)
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&ctl.raw_empty[r]);
                mbar_arrive(&ctl.cvt_full[c]);
            }
            // chunk ch - 1 is finished by now or soon (its last MMAs went out
            // before k-block i - 2 was converted): drain it while the tensor
            // cores run chunk ch
            if (i % kTcChunk == 2 && i >= kTcChunk) {
                drain(i / kTcChunk - 1);
                ++drained;
            }
        }
        while (ok && drained < nchunks) drain(drained++);

        // ---------------------------------------------------------------- epilogue
        if (ok) {
            const int t = m0 + 32 * sub + lane;
            const int n0 = nt * kTcN + half * kTcCols;
            unsigned long long best = 0ull;
            if (t < a.T) {
                const float xs = a.xscale[t];
                const bool vec = a.y != nullptr && (a.ldy & 3) == 0;
#pragma unroll
                for (int q = 0; q < kTcCols / 4; ++q) {
                    const int n = n0 + 4 * q;
                    if (n >= a.N) break;
                    float l[4];
                    if (n + 4 <= a.N) {
                        // the head's row scales are padded to whole 64-row groups
                        const float4 sw = *reinterpret_cast<const float4*>(a.wscale + n);
                        l[0] = xs * sw.x * (float)iacc[4 * q];
                        l[1] = xs * sw.y * (float)iacc[4 * q + 1];
                        l[2] = xs * sw.z * (float)iacc[4 * q + 2];
                        l[3] = xs * sw.w * (float)iacc[4 * q + 3];
                        if (vec)
                            *reinterpret_cast<float4*>(a.y + (int64_t)t * a.ldy + n) = make_float4(l[0], l[1], l[2], l[3]);
                        else if (a.y)
                            for (int e = 0; e < 4; ++e) a.y[(int64_t)t * a.ldy + n + e] = l[e];
#pragma unroll
                        for (int e = 0; e < 4; ++e) best = max(best, argmax_key(l[e], (uint32_t)(n + e)));
                    } else {
                        for (int e = 0; e < 4 && n + e < a.N; ++e) {
                            const float le = xs * a.wscale[n + e] * (float)iacc[4 * q + e];
                            if (a.y) a.y[(int64_t)t * a.ldy + n + e] = le;
                            best = max(best, argmax_key(le, (uint32_t)(n + e)));
                        }
                    }
                }
                if (best) atomicMax(a.keys + t, best);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kTcMmaWarp) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(2 * kTcN) : "memory");
    }
}

// ---------------------------------------------------------------- 4-bit, 256 rows a CTA
// The 4-bit matmuls of many rows: a CTA runs two 128-row tiles (256 rows)
// against each converted 128-row weight tile, so that every dequantised
// weight feeds 2 x 128 rows of MMAs (the converters' work per multiply-add
// is half that of one tile a CTA), and K is split over CTAs in slices of at
// most kT2MaxKb k-blocks (2048 columns): tensor memory accumulates no more
// than that (its truncating f32 accumulation stays at the f32 level), and the
// slices' partial sums meet in y through round-to-nearest vector reductions.
// Measured against the quantised definition (relative rms error): K = 20480
// in ten slices 1.4e-6, K = 4096 4.3e-7 (the chunk-draining kernel before
// it: 1.6e-7, at 1.2 - 1.4x the time; 1024-column slices: 4.4e-7 at K =
// 20480, at 1.15x the time of these).
// Roles as tc_head_kernel: one TMA lane (the 256-row f16 activation box and
// the packed weights), eight converter warps (which also run the epilogue),
// one MMA lane.
constexpr int kT2Tiles = 2;               // 128-row tiles a CTA
constexpr int kT2MaxKb = 32;              // k-blocks a CTA at most
constexpr int kT2Act = 3, kT2Cvt = 2, kT2Raw = 8;
constexpr int kT2A = kT2Tiles * kTcA;     // one 256-row f16 activation box, 128-byte swizzle
constexpr int kT2B = 2 * kTcN * kTcKB * 2;  // hi and lo weight tiles
constexpr int kT2Raw_ = 2 * 4 * kQ4Chunk;   // two 64-row groups of packed weights
constexpr size_t kT2Smem = 1024 + 1024 + (size_t)kT2Act * kT2A + (size_t)kT2Cvt * kT2B + (size_t)kT2Raw * kT2Raw_;
static_assert(kT2Smem <= 227 * 1024, "shared memory");

struct T2Ctl {
    uint64_t raw_full[kT2Raw], raw_empty[kT2Raw], act_full[kT2Act], act_empty[kT2Act], cvt_full[kT2Cvt],
        cvt_empty[kT2Cvt], acc_full;
    uint32_t tmem;
    int abort;
};
static_assert(sizeof(T2Ctl) <= 1024, "control block");

// hi / lo f16 tiles of one 16-row chunk's lane slot (both 32-column groups),
// the lane-slot permutation of tc_head_kernel (conflict-free stores)
DF_DEV void t2_convert_q4(const unsigned char* rs, unsigned char* bt, int warp, int lane, bool valid) {
    unsigned char* blo = bt + kTcN * kTcKB * 2;
    const int gg = warp >> 2, rr = warp & 3;
    const int qw = lane >> 3, jw = lane & 7;
    const int gq = (jw < 4) ? 2 * qw : ((2 * qw) ^ 5), tq = jw & 3;
    const int slot = 4 * gq + tq;
    const int nl0 = gg * 64 + rr * 16 + gq, nl1 = nl0 + 8;
    if (valid) {
        const unsigned char* ch = rs + gg * 4 * kQ4Chunk + rr * kQ4Chunk;
        const uint4 wv = *reinterpret_cast<const uint4*>(ch + slot * 16);
        const uint2 sv = *reinterpret_cast<const uint2*>(ch + 512 + gq * 8);
        const uint32_t wd[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
        for (int gi = 0; gi < 2; ++gi) {
            uint32_t a0[4], a1[4];
            unpack_q4_word(wd[gi * 2 + 0], a0);  // columns 8 tq + 0..3
            unpack_q4_word(wd[gi * 2 + 1], a1);  // columns 8 tq + 4..7
            const uint32_t sw = gi ? sv.y : sv.x;  // (s[gq][g], s[gq+8][g])
            const uint32_t s0 = __byte_perm(sw, 0, 0x1010), s1 = __byte_perm(sw, 0, 0x3232);
            const uint32_t q0[4] = {a0[0], a0[2], a1[0], a1[2]};  // row gq
            const uint32_t q1[4] = {a0[1], a0[3], a1[1], a1[3]};  // row gq + 8
            uint4 hi, lo;
            split_scaled(q0, s0, hi, lo);
            *reinterpret_cast<uint4*>(bt + tc_swz(nl0, 4 * gi + tq)) = hi;
            *reinterpret_cast<uint4*>(blo + tc_swz(nl0, 4 * gi + tq)) = lo;
            split_scaled(q1, s1, hi, lo);
            *reinterpret_cast<uint4*>(bt + tc_swz(nl1, 4 * gi + tq)) = hi;
            *reinterpret_cast<uint4*>(blo + tc_swz(nl1, 4 * gi + tq)) = lo;
        }
    } else {
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int gi = 0; gi < 2; ++gi) {
            *reinterpret_cast<uint4*>(bt + tc_swz(nl0, 4 * gi + tq)) = z;
            *reinterpret_cast<uint4*>(blo + tc_swz(nl0, 4 * gi + tq)) = z;
            *reinterpret_cast<uint4*>(bt + tc_swz(nl1, 4 * gi + tq)) = z;
            *reinterpret_cast<uint4*>(blo + tc_swz(nl1, 4 * gi + tq)) = z;
        }
    }
}

__global__ void __launch_bounds__(kTcThreads, 1) q4_tc2_kernel(const __grid_constant__ CUtensorMap xmap, TcArgs a) {
    extern __shared__ __align__(1024) unsigned char sm_raw[];
    unsigned char* sm = sm_raw + ((1024 - (smem_addr(sm_raw) & 1023)) & 1023);
    T2Ctl& ctl = *reinterpret_cast<T2Ctl*>(sm);
    unsigned char* act = sm + 1024;
    unsigned char* cvt = act + kT2Act * kT2A;
    unsigned char* raw = cvt + kT2Cvt * kT2B;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nt = blockIdx.x, m0 = blockIdx.y * (kT2Tiles * kTcM);
    const int tiles = min(kT2Tiles, (a.T - m0 + kTcM - 1) / kTcM);  // row tiles holding rows
    const int kb_lo = blockIdx.z * a.kb_per_split, kb_hi = min(a.L.ksteps, kb_lo + a.kb_per_split);
    const int nkb = kb_hi - kb_lo;
    const int ngroups_n = a.N / 64;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kT2Raw; ++i) {
            mbar_init(&ctl.raw_full[i], 1);
            mbar_init(&ctl.raw_empty[i], kTcCvtWarps);
        }
        for (int i = 0; i < kT2Act; ++i) {
            mbar_init(&ctl.act_full[i], 1);
            mbar_init(&ctl.act_empty[i], 1);
        }
        for (int i = 0; i < kT2Cvt; ++i) {
            mbar_init(&ctl.cvt_full[i], kTcCvtWarps);
            mbar_init(&ctl.cvt_empty[i], 1);
        }
        mbar_init(&ctl.acc_full, 1);
        ctl.abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kTcMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&ctl.tmem)),
                     "r"(kT2Tiles * kTcN)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl.tmem;
    pdl_trigger();
    pdl_wait();

    auto give_up = [&]() {
        atomicExch(a.err, 1);
        *reinterpret_cast<volatile int*>(&ctl.abort) = 1;
    };
    auto aborted = [&]() { return *reinterpret_cast<volatile int*>(&ctl.abort) != 0; };

    if (warp == kTcTmaWarp) {
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(&xmap) : "memory");
            int issued = 0, ng = 0;
            for (int gg = 0; gg < kTcN / 64; ++gg) ng += (nt * (kTcN / 64) + gg < ngroups_n) ? 1 : 0;
            for (int i = 0; i < nkb; ++i) {
                const int r = i % kT2Raw, sa = i % kT2Act;
                bool ok = true;
                if (i >= kT2Raw) ok = mbar_wait(&ctl.raw_empty[r], ((i / kT2Raw) - 1) & 1, kTcWait);
                if (ok && i >= kT2Act) ok = mbar_wait(&ctl.act_empty[sa], ((i / kT2Act) - 1) & 1, kTcWait);
                if (!ok) give_up();
                if (!ok || aborted()) break;
                fence_proxy_async_smem();
                const int kb = kb_lo + i;
                // the whole 256-row box: rows past T read as zeros and count toward the bytes
                mbar_arrive_expect_tx(&ctl.act_full[sa], (uint32_t)kT2A);
                tma_load_2d(act + sa * kT2A, &xmap, kb * kTcKB, m0, &ctl.act_full[sa]);
                unsigned char* dst = raw + r * kT2Raw_;
                mbar_arrive_expect_tx(&ctl.raw_full[r], (uint32_t)(ng * 4 * kQ4Chunk));
                for (int gg = 0; gg < ng; ++gg)
                    bulk_g2s(dst + gg * 4 * kQ4Chunk, a.w + q4_chunk_offset(a.L, 4 * (a.g0 + nt * (kTcN / 64) + gg), kb),
                             4 * kQ4Chunk, &ctl.raw_full[r]);
                issued = i + 1;
            }
            for (int i = max(0, issued - kT2Raw); i < issued; ++i)
                mbar_wait(&ctl.raw_full[i % kT2Raw], (i / kT2Raw) & 1, kTcWait);
            for (int i = max(0, issued - kT2Act); i < issued; ++i)
                mbar_wait(&ctl.act_full[i % kT2Act], (i / kT2Act) & 1, kTcWait);
        }
    } else if (warp == kTcMmaWarp) {
        if (lane == 0) {
            for (int i = 0; i < nkb; ++i) {
                const int sx = i % kT2Act, sc = i % kT2Cvt;
                bool ok = mbar_wait(&ctl.act_full[sx], (i / kT2Act) & 1, kTcWait);
                if (ok) ok = mbar_wait(&ctl.cvt_full[sc], (i / kT2Cvt) & 1, kTcWait);
                if (!ok) give_up();
                if (!ok || aborted()) break;
                tc_fence_after();
                const uint32_t sa = smem_addr(act + sx * kT2A);
                const uint32_t sb = smem_addr(cvt + sc * kT2B);
#pragma unroll
                for (int j = 0; j < kTcKB / 16; ++j) {
                    const uint64_t bh = tc_desc_sw128(sb + 32 * j), bl = tc_desc_sw128(sb + kTcN * kTcKB * 2 + 32 * j);
                    for (int t = 0; t < tiles; ++t) {
                        const uint64_t ad = tc_desc_sw128(sa + t * kTcA + 32 * j);
                        const uint32_t d = tmem + (uint32_t)(t * kTcN);
                        tc_mma(d, ad, bh, (i > 0 || j > 0) ? 1u : 0u);
                        tc_mma(d, ad, bl, 1u);
                    }
                }
                tc_commit(&ctl.cvt_empty[sc]);
                tc_commit(&ctl.act_empty[sx]);
            }
            // arrives once every MMA issued so far has completed
            tc_commit(&ctl.acc_full);
        }
    } else {
        // ---------------------------------------------------------------- converters
        for (int i = 0; i < nkb; ++i) {
            const int r = i % kT2Raw, c = i % kT2Cvt;
            bool w = mbar_wait(&ctl.raw_full[r], (i / kT2Raw) & 1, kTcWait);
            if (w && i >= kT2Cvt) w = mbar_wait(&ctl.cvt_empty[c], ((i / kT2Cvt) - 1) & 1, kTcWait);
            if (!w) give_up();
            if (__any_sync(0xffffffffu, !w || aborted())) break;
            t2_convert_q4(raw + r * kT2Raw_, cvt + c * kT2B, warp, lane, nt * (kTcN / 64) + (warp >> 2) < ngroups_n);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&ctl.raw_empty[r]);
                mbar_arrive(&ctl.cvt_full[c]);
            }
        }
        // ---------------------------------------------------------------- epilogue
        const bool ok = mbar_wait(&ctl.acc_full, 0, kTcWait);
        if (!ok) give_up();
        tc_fence_after();
        if (__all_sync(0xffffffffu, ok && !aborted()) && nkb > 0) {
            const int sub = warp & 3, half = warp >> 2;
            const bool red = a.accumulate != 0 || gridDim.z > 1;
            for (int t = 0; t < tiles; ++t) {
                const int row = m0 + t * kTcM + 32 * sub + lane;
                const int n0 = nt * kTcN + half * 64;
                const float xs = row < a.T ? a.xscale[row] : 0.f;
#pragma unroll 1
                for (int cc = 0; cc < 64; cc += 16) {
                    uint32_t v[16];
                    tc_ld16(tmem + ((uint32_t)(32 * sub) << 16) + (uint32_t)(t * kTcN + half * 64 + cc), v);
                    tc_wait_ld();
                    if (row < a.T && n0 + cc < a.N) {
                        float* dst = a.y + (int64_t)row * a.ldy + n0 + cc;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float f0 = __uint_as_float(v[4 * q]) * xs, f1 = __uint_as_float(v[4 * q + 1]) * xs,
                                        f2 = __uint_as_float(v[4 * q + 2]) * xs, f3 = __uint_as_float(v[4 * q + 3]) * xs;
                            if (red)
                                red_add_v4(dst + 4 * q, f0, f1, f2, f3);
                            else
                                *reinterpret_cast<float4*>(dst + 4 * q) = make_float4(f0, f1, f2, f3);
                        }
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kTcMmaWarp) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kT2Tiles * kTcN)
                     : "memory");
    }
}

// ---------------------------------------------------------------- dense weight copies
// For the many-row path the library can hold a second copy of each matrix as
// dense f16: the 4-bit matrices as the exact pair hi = f16(s q), lo =
// f16(s q - hi) (two planes [N][K]), the head as its int8 codes in f16
// ([V][K]).  With those the tensor-core kernels take every operand tile by
// TMA and convert nothing (HBM is plentiful; conversion was their limit).
__global__ void dequant_hilo_kernel(const int8_t* __restrict__ codes, const uint16_t* __restrict__ scales, int N,
                                    int K, __half* __restrict__ hi, __half* __restrict__ lo) {
    const int64_t n = (int64_t)N * K;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / K;
        const int c = (int)(i - r * K);
        const float sf = __half2float(__ushort_as_half(scales[r * (K / 32) + c / 32]));
        const float p = sf * (float)codes[i];  // exact: 11 x 4 significant bits
        const __half h = __float2half_rn(p);
        hi[i] = h;
        lo[i] = __float2half_rn(p - __half2float(h));  // exact remainder
    }
}

int dequant_hilo(const int8_t* codes, const uint16_t* scales, int N, int K, __half* hi, __half* lo, cudaStream_t st) {
    if (N <= 0 || K <= 0 || K % 32) return (int)cudaErrorInvalidValue;
    dequant_hilo_kernel<<<1024, 256, 0, st>>>(codes, scales, N, K, hi, lo);
    return (int)cudaGetLastError();
}

// ---------------------------------------------------------------- host side
// (shared with the tcgen05 attention's tensor maps)

std::mutex& attr_mutex() {
    static std::mutex m;
    return m;
}

EncodeTiledFn encode_fn() {
    // looked up once (a thread-safe static initialisation)
    static const EncodeTiledFn fn = []() -> EncodeTiledFn {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeTiledFn>(p);
        cudaGetLastError();
        return nullptr;
    }();
    return fn;
}

// the tensor map of the activation codes as f16 [T][K] (rows of K halves):
// 64 x 128 boxes in the 128-byte swizzle, rows past T read as zeros
bool act_map(CUtensorMap* map, const __half* codes, int K, int T, int box_rows) {
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)T};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kTcKB, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return encode_fn()(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half*>(codes), dims, strides, box, estr,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// int8 codes [T][ld] -> f16 [T][K] (exact integers), 16 codes a thread
__global__ void codes_to_f16_kernel(const int8_t* __restrict__ x, int ld, int T, int K, __half* __restrict__ out) {
    pdl_trigger();
    pdl_wait();
    const int per_row = K / 16;
    const int64_t n = (int64_t)T * per_row;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int r = (int)(i / per_row), c = (int)(i - (int64_t)r * per_row);
        const uint4 v = *reinterpret_cast<const uint4*>(x + (int64_t)r * ld + c * 16);
        uint4 h0, h1;
        i8x4_to_half2x2(v.x, h0.x, h0.y);
        i8x4_to_half2x2(v.y, h0.z, h0.w);
        i8x4_to_half2x2(v.z, h1.x, h1.y);
        i8x4_to_half2x2(v.w, h1.z, h1.w);
        uint4* o = reinterpret_cast<uint4*>(out + (int64_t)r * K + c * 16);
        o[0] = h0;
        o[1] = h1;
    }
}

// ... and the squared norm of each row's codes (exact in int32 for K < 2^17),
// a block per row
__global__ void __launch_bounds__(256) codes_to_f16_norm_kernel(const int8_t* __restrict__ x, int ld, int T, int K,
                                                                __half* __restrict__ out, int* __restrict__ norm2) {
    pdl_trigger();
    pdl_wait();
    __shared__ int part[8];
    for (int r = blockIdx.x; r < T; r += gridDim.x) {
        int s = 0;
        for (int c = threadIdx.x; c < K / 16; c += blockDim.x) {
            const uint4 v = *reinterpret_cast<const uint4*>(x + (int64_t)r * ld + c * 16);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) s = __dp4a((int)w[j], (int)w[j], s);
            uint4 h0, h1;
            i8x4_to_half2x2(v.x, h0.x, h0.y);
            i8x4_to_half2x2(v.y, h0.z, h0.w);
            i8x4_to_half2x2(v.z, h1.x, h1.y);
            i8x4_to_half2x2(v.w, h1.z, h1.w);
            uint4* o = reinterpret_cast<uint4*>(out + (int64_t)r * K + c * 16);
            o[0] = h0;
            o[1] = h1;
        }
#pragma unroll
        for (int d = 16; d; d >>= 1) s += __shfl_xor_sync(0xffffffffu, s, d);
        if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = s;
        __syncthreads();
        if (threadIdx.x == 0) {
            int t = 0;
            for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += part[w];
            norm2[r] = t;
        }
        __syncthreads();
    }
}

int codes_to_f16(const int8_t* x, int ld, int T, int K, __half* out, int* norm2, int num_sms, cudaStream_t st) {
    if (T <= 0) return 0;
    if (K % 16 || ld % 16 || (reinterpret_cast<uintptr_t>(x) & 15) || (reinterpret_cast<uintptr_t>(out) & 15))
        return (int)cudaErrorInvalidValue;
    if (norm2) {
        if (K >= (1 << 17)) return (int)cudaErrorInvalidValue;
        const int blocks = std::min(T, num_sms * 8);
        return (int)launch(codes_to_f16_norm_kernel, dim3(blocks), dim3(256), 0, st, x, ld, T, K, out, norm2);
    }
    const int64_t n = (int64_t)T * (K / 16);
    const int blocks = (int)std::min<int64_t>((n + 255) / 256, (int64_t)num_sms * 8);
    return (int)launch(codes_to_f16_kernel, dim3(blocks), dim3(256), 0, st, x, ld, T, K, out);
}

static cudaError_t tc_set_smem() {
    static size_t limit = 0;
    return raise_smem_limit(tc_head_kernel, TcShape::kSmem, &limit);
}

bool q4_tc_supported(Q4Layout L, int tile0, int N, int K, QAct x) {
    return encode_fn() != nullptr && tile0 % 4 == 0 && N % 64 == 0 && N > 0 && K == L.ksteps * kQ4KStep &&
           x.ld % 16 == 0 && (reinterpret_cast<uintptr_t>(x.codes) & 15) == 0;
}

int q4_tc(const uint8_t* packed, Q4Layout L, int tile0, int N, QAct x, const __half* x16, int T, float* y, int ldy,
          bool accumulate, int num_sms, int* err_flag, cudaStream_t st) {
    if (T <= 0 || N <= 0) return 0;
    const int K = L.ksteps * kQ4KStep;
    if (!q4_tc_supported(L, tile0, N, K, x) || ldy % 4 || (reinterpret_cast<uintptr_t>(y) & 15) ||
        (reinterpret_cast<uintptr_t>(x16) & 15))
        return (int)cudaErrorInvalidValue;
    CUtensorMap map;
    if (!act_map(&map, x16, K, T, kT2Tiles * kTcM)) return (int)cudaErrorInvalidValue;
    static size_t limit = 0;
    cudaError_t e = raise_smem_limit(q4_tc2_kernel, kT2Smem, &limit);
    if (e != cudaSuccess) return (int)e;
    const int mt = (T + kT2Tiles * kTcM - 1) / (kT2Tiles * kTcM), ntl = (N + kTcN - 1) / kTcN;
    // K slices of at most kT2MaxKb k-blocks (the accumulation bound); more
    // slices while the tiles alone leave more than a third of the SMs idle
    int splits = (L.ksteps + kT2MaxKb - 1) / kT2MaxKb;
    while (mt * ntl * splits * 3 < num_sms * 2 && splits * 2 <= L.ksteps) splits *= 2;
    const int kps = (L.ksteps + splits - 1) / splits;
    splits = (L.ksteps + kps - 1) / kps;
    if (splits > 1 && !accumulate) {
        cudaError_t e = cudaMemset2DAsync(y, (size_t)ldy * sizeof(float), 0, (size_t)N * sizeof(float), T, st);
        if (e != cudaSuccess) return (int)e;
    }
    TcArgs args{packed, L, tile0 / 4, N, x.scale, T, y, ldy, accumulate ? 1 : 0, kps, nullptr, nullptr, err_flag};
    return (int)launch(q4_tc2_kernel, dim3(ntl, mt, splits), dim3(kTcThreads), kT2Smem, st, map, args);
}

bool head_tc_supported(int ksteps, QAct x) {
    return encode_fn() != nullptr && ksteps > 0 && x.ld % 16 == 0 && (reinterpret_cast<uintptr_t>(x.codes) & 15) == 0;
}

int head_tc(const int8_t* packed, const float* row_scale, int V, int ksteps, QAct x, const __half* x16, int T,
            float* logits, int ldl, unsigned long long* keys, int* err_flag, cudaStream_t st) {
    if (T <= 0 || V <= 0) return 0;
    if (!head_tc_supported(ksteps, x) || (reinterpret_cast<uintptr_t>(x16) & 15)) return (int)cudaErrorInvalidValue;
    CUtensorMap map;
    if (!act_map(&map, x16, ksteps * kI8KStep, T, kTcM)) return (int)cudaErrorInvalidValue;
    cudaError_t e = tc_set_smem();
    if (e != cudaSuccess) return (int)e;
    const int mt = (T + kTcM - 1) / kTcM, ntl = (V + kTcN - 1) / kTcN;
    Q4Layout L{0, ksteps, 1};
    TcArgs args{reinterpret_cast<const uint8_t*>(packed), L, 0, V, x.scale, T, logits, ldl, 0, ksteps, row_scale,
                keys, err_flag};
    return (int)launch(tc_head_kernel, dim3(mt, ntl, 1), dim3(kTcThreads), TcShape::kSmem, st, map, args);
}

// a dense f16 weight copy [N][K] as a TMA tensor map: 64 x 128 boxes, 128-byte swizzle
bool dense_map(CUtensorMap* map, const __half* w, int K, int N, int box_rows) {
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)N};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kTcKB, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return encode_fn()(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half*>(w), dims, strides, box, estr,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// an f32 output [T][ldy] as a TMA tensor map of its first N columns
bool out_map(CUtensorMap* map, float* y, int ldy, int N, int T) {
    if (!y || ldy % 4 || (reinterpret_cast<uintptr_t>(y) & 15)) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)T};
    const cuuint64_t strides[1] = {(cuuint64_t)ldy * 4};
    const cuuint32_t box[2] = {32, 32};
    const cuuint32_t estr[2] = {1, 1};
    return encode_fn()(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, y, dims, strides, box, estr,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace dflash
