// Streaming matvecs of the block's rows (up to 16) against the 4-bit draft
// matrices and the int8 head: the weight stream is the HBM-bound part of the
// drafter (page "cortiq-engine 0.8.75 — src/gpu_wgpu/dflash_dev.rs", module
// documentation: 2.3 GB of weights streamed per block; `Dev::q4`, `Dev::q8`).
//
// One CTA per SM.  Weights move through shared-memory rings with bulk copies
// (TMA, completion on mbarriers), and the first copies go out before the
// previous kernel on the stream has finished (programmatic dependent launch),
// since weights do not depend on it.  The block's int8 activation codes are
// staged in shared memory once the previous kernel is done, and the products
// run as f16 tensor-core MMAs on exact integer operands; a 64-row group's four
// 16-row tiles share each B fragment.  Every mbarrier wait is bounded: on
// expiry the kernel raises *err_flag and finishes without the remaining work.
#include <algorithm>

#include "common.cuh"
#include "kernels.cuh"

namespace dflash {

constexpr int kConsumers = 8;
constexpr int kStreamThreads = (kConsumers + 1) * 32;
constexpr uint64_t kWaitLimit = 1000000000ull;  // ns an mbarrier wait may take before the kernel gives up

// ------------------------------------------------------------------ 4-bit
// Each warp streams its own contiguous share of the CTA's span through a
// private ring of two-super-chunk slots (its lane 0 issues the bulk copies and
// refills a slot as soon as the warp has read it), accumulates consecutive
// k-steps of a 64-row group in registers, and adds a group's 16 x 64 partial
// sums, times the rows' activation scales, straight into y when it moves to
// the next group.  Warps never wait on one another after the activation codes
// are staged.
constexpr int kQ4Warps = 16;
constexpr int kQ4Threads = kQ4Warps * 32;
constexpr int kQ4SC = 4 * kQ4Chunk;  // super-chunk: 4 tiles x one k-step
constexpr int kQ4SlotSC = 2;         // super-chunks per ring slot (one bulk copy)
constexpr int kQ4WarpSlots = 2;      // ring slots per warp
constexpr int kQ4ActPad = 32;        // halves of row pad: conflict-free 16-byte B-fragment loads
constexpr int kQ4BarBytes = 1024;    // the warps' mbarriers, ahead of the ring
constexpr int kQ4DumpBytes = 512;    // a warp's scratch for the vector reductions of a group
// The offsets the unpacking leaves in the weights are taken out by the MMA's
// C input: per 32-column group g of the K-block and 8-row half h of the
// block's rows, lane quad tq reads {-1032 X[t0], -1032 X[t1], -72 X[t0],
// -72 X[t1]} (t0 = 8 h + 2 tq, t1 = t0 + 1; X[t] the group's sum of row t's
// activation codes) -- the m16n8k16 C fragment of weight rows gq (offset
// 1032) and gq + 8 (offset 72).
constexpr int kQ4OffBytes = (32 * kQ4KStep / 32) * 2 * 4 * 16;  // 64 groups x 2 halves x 4 quads x 16 B

// Eight offset nibbles (code + 8) -> four half2 of the m16n8k16 A fragment
// with the offsets left in: the low nibbles (rows gq) ORed into the mantissa
// of 1024.0h read 1024 + nibble = 1032 + code, the high nibbles (rows gq + 8)
// ORed into that of 64.0h (unit 1/16) read 64 + nibble = 72 + code.  One LOP3
// per half2.
DF_DEV void unpack_q4_word_biased(uint32_t w, uint32_t (&a)[4]) {
    const uint32_t kLo = 0x000F000Fu, kHi = 0x00F000F0u;
    const uint32_t kM1024 = 0x64006400u, kM64 = 0x54005400u;
    a[0] = lop3_and_or(w, kLo, kM1024);
    a[1] = lop3_and_or(w, kHi, kM64);
    const uint32_t w8 = w >> 8;
    a[2] = lop3_and_or(w8, kLo, kM1024);
    a[3] = lop3_and_or(w8, kHi, kM64);
}

// B fragments of one k-step (two 32-column groups, block rows gq and gq + 8)
// from int8 codes in shared memory: 8 codes per (group, row half) -> 4 half2.
DF_DEV void load_b_frags_i8(const int8_t* a_lo, const int8_t* a_hi, uint32_t (&bf)[2][2][4]) {
#pragma unroll
    for (int gi = 0; gi < 2; ++gi) {
        const uint2 v0 = *reinterpret_cast<const uint2*>(a_lo + gi * 32);
        const uint2 v1 = *reinterpret_cast<const uint2*>(a_hi + gi * 32);
        i8x4_to_half2x2(v0.x, bf[gi][0][0], bf[gi][0][1]);
        i8x4_to_half2x2(v0.y, bf[gi][0][2], bf[gi][0][3]);
        i8x4_to_half2x2(v1.x, bf[gi][1][0], bf[gi][1][1]);
        i8x4_to_half2x2(v1.y, bf[gi][1][2], bf[gi][1][3]);
    }
}

__global__ void __launch_bounds__(kQ4Threads, 1)
    q4_stream_kernel(const uint8_t* __restrict__ wp, Q4Layout L, int g0, int ng, QAct x, int T,
                     float* __restrict__ y, int ldy, int* __restrict__ err) {
    extern __shared__ __align__(128) unsigned char sm[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint64_t* full = reinterpret_cast<uint64_t*>(sm) + warp * kQ4WarpSlots;
    unsigned char* ring = sm + kQ4BarBytes + warp * (kQ4WarpSlots * kQ4SlotSC * kQ4SC);
    __half* act = reinterpret_cast<__half*>(sm + kQ4BarBytes + kQ4Warps * (kQ4WarpSlots * kQ4SlotSC * kQ4SC));
    const int kbc = L.kb * kQ4KStep;  // columns of a K-block
    const int ldact = kbc + kQ4ActPad;
    float* dscr = reinterpret_cast<float*>(sm + kQ4BarBytes + kQ4Warps * (kQ4WarpSlots * kQ4SlotSC * kQ4SC) +
                                           (size_t)16 * ldact * sizeof(__half)) +
                  warp * (kQ4DumpBytes / 4);
    float4* offs = reinterpret_cast<float4*>(sm + kQ4BarBytes + kQ4Warps * (kQ4WarpSlots * kQ4SlotSC * kQ4SC) +
                                             (size_t)16 * ldact * sizeof(__half) + (size_t)kQ4Warps * kQ4DumpBytes);

    const StreamGeom sg = stream_geom(L, g0, ng);
    const int64_t span = sg.hi - sg.lo;
    const int64_t wlo = sg.lo + span * warp / kQ4Warps;
    const int n = (int)(sg.lo + span * (warp + 1) / kQ4Warps - wlo);  // this warp's super-chunks
    const int nslots = (n + kQ4SlotSC - 1) / kQ4SlotSC;
    const uint8_t* src = wp + (sg.base + wlo) * kQ4SC;

    pdl_trigger();
    // the first slots go out before the previous kernel has finished: weights do not depend on it
    int issued = 0;
    auto issue = [&](int j) {
        const int slot = j % kQ4WarpSlots;
        const uint32_t bytes = (uint32_t)min(kQ4SlotSC, n - j * kQ4SlotSC) * kQ4SC;
        mbar_arrive_expect_tx(&full[slot], bytes);
        bulk_g2s(ring + slot * (kQ4SlotSC * kQ4SC), src + (int64_t)j * (kQ4SlotSC * kQ4SC), bytes, &full[slot]);
    };
    if (lane == 0) {
        for (int i = 0; i < kQ4WarpSlots; ++i) mbar_init(&full[i], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        for (; issued < min(kQ4WarpSlots, nslots); ++issued) issue(issued);
    }

    pdl_wait();
    {
        // the K-block's codes of the 16 rows as exact f16 (rows past T are
        // zero), eight loads of a thread in flight at once
        const int vec = kbc / 8, total = 16 * vec;
        // X[t][g]: the sums of each row's codes over each 32-column group,
        // gathered first as integers in the offset area
        int* xsum = reinterpret_cast<int*>(offs) + (kQ4OffBytes / 4) / 2;  // [16][64], the area's upper half
        constexpr int kBatch = 8;
        for (int base = threadIdx.x; base < total; base += kBatch * kQ4Threads) {
            uint2 v[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int i = base + u * kQ4Threads, r = i / vec, c = i - r * vec;
                v[u] = make_uint2(0u, 0u);
                if (i < total && r < T)
                    v[u] = *reinterpret_cast<const uint2*>(x.codes + (int64_t)r * x.ld + sg.kblk * kbc + c * 8);
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int i = base + u * kQ4Threads, r = i / vec, c = i - r * vec;
                // four consecutive vectors (threads) make a group: vec and the
                // thread count are multiples of 4, so a quad never straddles rows
                int gs = __dp4a((int)v[u].x, 0x01010101, __dp4a((int)v[u].y, 0x01010101, 0));
                gs += __shfl_xor_sync(0xffffffffu, gs, 1);
                gs += __shfl_xor_sync(0xffffffffu, gs, 2);
                if (i < total) {
                    uint4 h;
                    i8x4_to_half2x2(v[u].x, h.x, h.y);
                    i8x4_to_half2x2(v[u].y, h.z, h.w);
                    *reinterpret_cast<uint4*>(act + r * ldact + c * 8) = h;
                    if ((c & 3) == 0) xsum[r * 64 + (c >> 2)] = gs;
                }
            }
        }
        __syncthreads();
        // the C-fragment table from the sums: entry j = (g, h, tq), at most
        // (kbc / 32) * 8 <= 512 entries, one a thread; the table overwrites
        // the sums, so every thread reads before any writes
        const int j = threadIdx.x;
        const bool has = j < (kbc / 32) * 8;
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
        if (has) {
            const int g = j >> 3, h = (j >> 2) & 1, tq = j & 3, t0 = 8 * h + 2 * tq;
            const float x0 = (float)xsum[t0 * 64 + g], x1 = (float)xsum[(t0 + 1) * 64 + g];
            o = make_float4(-1032.f * x0, -1032.f * x1, -72.f * x0, -72.f * x1);
        }
        __syncthreads();
        if (has) offs[j] = o;
        __syncthreads();
    }
    const int gq = lane >> 2, tq = lane & 3;
    const __half* a_lo = act + gq * ldact + 8 * tq;
    const __half* a_hi = act + (gq + 8) * ldact + 8 * tq;
    // activation scales of this lane's four output rows (tokens h * 8 + 2 tq + e)
    float xs[2][2];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int t = h * 8 + 2 * tq + e;
            xs[h][e] = t < T ? x.scale[t] : 0.f;
        }
    const float zero[4] = {0.f, 0.f, 0.f, 0.f};
    __align__(8) float acc[4][2][4];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[r][h][e] = 0.f;

    // a group's partial sums into y (rows >= T are not written)
    auto dump = [&](int grp) { dump_group_v4(acc, xs, y, ldy, grp * 64, T, dscr, lane); };

    // one super-chunk at scp: k-step ks of group grp
    auto sc_step = [&](const unsigned char* scp, int ks) {
        uint4 bq[2][2];  // [group][row half]: 8 halves = the two k16 B fragments
#pragma unroll
        for (int gi = 0; gi < 2; ++gi) {
            bq[gi][0] = *reinterpret_cast<const uint4*>(a_lo + ks * kQ4KStep + gi * 32);
            bq[gi][1] = *reinterpret_cast<const uint4*>(a_hi + ks * kQ4KStep + gi * 32);
        }
        const float4* ok = offs + (2 * ks) * 8 + tq;  // entries (group 2 ks + gi, half h) at ok[gi * 8 + h * 4]
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const uint4 wv = *reinterpret_cast<const uint4*>(scp + r * kQ4Chunk + lane * 16);
            const uint2 sv = *reinterpret_cast<const uint2*>(scp + r * kQ4Chunk + 512 + gq * 8);
            const uint32_t wds[4] = {wv.x, wv.y, wv.z, wv.w};
            const uint32_t svs[2] = {sv.x, sv.y};
#pragma unroll
            for (int gi = 0; gi < 2; ++gi) {
                uint32_t a0[4], a1[4];
                unpack_q4_word_biased(wds[gi * 2 + 0], a0);
                unpack_q4_word_biased(wds[gi * 2 + 1], a1);
                // the offsets' C fragments (re-read per tile: registers are short)
                const float4 o0 = ok[gi * 8], o1 = ok[gi * 8 + 4];
                const float c0[4] = {o0.x, o0.y, o0.z, o0.w}, c1[4] = {o1.x, o1.y, o1.z, o1.w};
                float d0[4], d1[4];
                // group sums are exact integers below 2^23 at every step
                mma_f16_16816(d0, a0, bq[gi][0].x, bq[gi][0].y, c0);
                mma_f16_16816(d0, a1, bq[gi][0].z, bq[gi][0].w, d0);
                mma_f16_16816(d1, a0, bq[gi][1].x, bq[gi][1].y, c1);
                mma_f16_16816(d1, a1, bq[gi][1].z, bq[gi][1].w, d1);
                // the group's f16 scales of rows gq and gq + 8, each as an f32
                // pair, for packed f32x2 fused multiply-adds (same rounding as
                // two fmaf)
                uint32_t sbits = svs[gi];
                const __half2 sh = *reinterpret_cast<const __half2*>(&sbits);
                const float2 s0 = __half22float2(__low2half2(sh)), s1 = __half22float2(__high2half2(sh));
                float2* a00 = reinterpret_cast<float2*>(&acc[r][0][0]);
                float2* a01 = reinterpret_cast<float2*>(&acc[r][0][2]);
                float2* a10 = reinterpret_cast<float2*>(&acc[r][1][0]);
                float2* a11 = reinterpret_cast<float2*>(&acc[r][1][2]);
                *a00 = __ffma2_rn(s0, make_float2(d0[0], d0[1]), *a00);
                *a01 = __ffma2_rn(s1, make_float2(d0[2], d0[3]), *a01);
                *a10 = __ffma2_rn(s0, make_float2(d1[0], d1[1]), *a10);
                *a11 = __ffma2_rn(s1, make_float2(d1[2], d1[3]), *a11);
            }
        }
    };

    const int kb = L.kb;
    int ks = (int)(wlo % kb), grp = (int)(wlo / kb), cur = grp;
    int j = 0;
    bool ok = true;
    for (; j < nslots; ++j) {
        const int slot = j % kQ4WarpSlots;
        // ok is warp-uniform after the vote, so the warp leaves the loop whole
        ok = __all_sync(0xffffffffu, mbar_wait(&full[slot], (j / kQ4WarpSlots) & 1, kWaitLimit));
        if (!ok) break;
        const unsigned char* sb = ring + slot * (kQ4SlotSC * kQ4SC);
#pragma unroll
        for (int u = 0; u < kQ4SlotSC; ++u) {
            if (u > 0 && j * kQ4SlotSC + u >= n) break;  // the warp's last slot may be short (uniform)
            if (grp != cur) {
                dump(cur);
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int e = 0; e < 4; ++e) acc[r][h][e] = 0.f;
                cur = grp;
            }
            sc_step(sb + u * kQ4SC, ks);
            if (++ks == kb) {
                ks = 0;
                ++grp;
            }
        }
        // every lane has read the slot: refill it with the slot kQ4WarpSlots ahead
        __syncwarp();
        if (lane == 0 && issued < nslots) {
            fence_proxy_async_smem();
            issue(issued++);
        }
    }
    if (ok) {
        if (n > 0) dump(cur);
    } else {
        // a wait gave up: record it, and let no copy still land in this CTA's memory after it exits
        if (lane == 0) {
            atomicExch(err, 1);
            for (int k = j; k < issued; ++k)
                mbar_wait(&full[k % kQ4WarpSlots], (k / kQ4WarpSlots) & 1, kWaitLimit);
        }
    }
}

static size_t q4_stream_bytes(Q4Layout L) {
    return (size_t)kQ4BarBytes + (size_t)kQ4Warps * kQ4WarpSlots * kQ4SlotSC * kQ4SC +
           (size_t)16 * (L.kb * kQ4KStep + kQ4ActPad) * sizeof(__half) + (size_t)kQ4Warps * kQ4DumpBytes +
           (size_t)kQ4OffBytes;
}

size_t q4_stream_smem_bytes(Q4Layout L, int, int) { return q4_stream_bytes(L); }

int q4_stream(const uint8_t* packed, Q4Layout L, int tile0, int N, QAct x, int T, float* y, int ldy, int num_sms,
              int* err_flag, cudaStream_t st) {
    if (T <= 0 || N <= 0) return 0;
    if (T > 16 || N % 64 || tile0 % 4 || L.ksteps / L.kb > num_sms || ldy % 4 || (reinterpret_cast<uintptr_t>(y) & 15))
        return (int)cudaErrorInvalidValue;
    const size_t smem = q4_stream_bytes(L);
    if (smem > 227 * 1024) return (int)cudaErrorInvalidValue;
    static size_t limit = 0;
    const cudaError_t e = raise_smem_limit(q4_stream_kernel, smem, &limit);
    if (e != cudaSuccess) return (int)e;
    return (int)launch(q4_stream_kernel, dim3(num_sms), dim3(kQ4Threads), smem, st, packed, L, tile0 / 4, N / 64, x, T,
                       y, ldy, err_flag);
}

// ------------------------------------------------------------------ head
constexpr int kActPad = 32;     // bytes of row pad of the head's staged int8 codes
constexpr int kHeadSlotSC = 8;  // super-chunks (k-steps of one group) per slot
constexpr int kHeadSlots = 4;  // 4 x 32 KB of weights in flight per SM

__global__ void __launch_bounds__(kStreamThreads, 1)
    head_stream_kernel(const int8_t* __restrict__ wp, const float* __restrict__ sw, int ngroups, int ksteps, int V,
                       QAct x, int T, float* __restrict__ logits, int ldl, unsigned long long* __restrict__ keys,
                       int* __restrict__ err) {
    extern __shared__ __align__(128) unsigned char sm[];
    uint64_t* full = reinterpret_cast<uint64_t*>(sm);
    uint64_t* empty = full + kHeadSlots;
    unsigned char* ring = sm + 128;
    int32_t* part = reinterpret_cast<int32_t*>(ring + kHeadSlots * kHeadSlotSC * kI8Super);  // [8 warps][1024]
    int8_t* act = reinterpret_cast<int8_t*>(part + kConsumers * 1024);
    const int K = ksteps * kI8KStep;
    const int ldact = K + kActPad;
    const int tok0 = blockIdx.y * 16;
    const int G = gridDim.x, c = blockIdx.x;
    const int glo = (int)((int64_t)ngroups * c / G), ghi = (int)((int64_t)ngroups * (c + 1) / G);
    const int spg = (ksteps + kHeadSlotSC - 1) / kHeadSlotSC;  // slots per group
    const int nslots = (ghi - glo) * spg;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    pdl_trigger();
    if (threadIdx.x == 0) {
        for (int i = 0; i < kHeadSlots; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kConsumers);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (warp == kConsumers) {
        if (lane == 0) {
            int issued = 0;
            for (int i = 0; i < nslots; ++i) {
                const int slot = i % kHeadSlots;
                if (i >= kHeadSlots && !mbar_wait(&empty[slot], ((i / kHeadSlots) - 1) & 1, kWaitLimit)) {
                    atomicExch(err, 1);
                    break;
                }
                const int grp = glo + i / spg, k0 = (i % spg) * kHeadSlotSC;
                const int n = min(kHeadSlotSC, ksteps - k0);
                const uint32_t bytes = (uint32_t)n * kI8Super;
                mbar_arrive_expect_tx(&full[slot], bytes);
                bulk_g2s(ring + slot * kHeadSlotSC * kI8Super, wp + ((int64_t)grp * ksteps + k0) * kI8Super, bytes,
                         &full[slot]);
                issued = i + 1;
            }
            for (int i = max(0, issued - kHeadSlots); i < issued; ++i)
                mbar_wait(&full[i % kHeadSlots], (i / kHeadSlots) & 1, kWaitLimit);
        }
        return;
    }

    pdl_wait();
    {
        // eight loads of a thread in flight at once
        const int vec = K / 16, total = 16 * vec;
        constexpr int kBatch = 8, kN = kConsumers * 32;
        for (int base = threadIdx.x; base < total; base += kBatch * kN) {
            uint4 v[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int i = base + u * kN, r = i / vec, cc = i - r * vec;
                v[u] = make_uint4(0u, 0u, 0u, 0u);
                if (i < total && tok0 + r < T)
                    v[u] = *reinterpret_cast<const uint4*>(x.codes + (int64_t)(tok0 + r) * x.ld + cc * 16);
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int i = base + u * kN, r = i / vec, cc = i - r * vec;
                if (i < total) *reinterpret_cast<uint4*>(act + r * ldact + cc * 16) = v[u];
            }
        }
        asm volatile("bar.sync 1, %0;" ::"r"(kConsumers * 32) : "memory");
    }
    const int gq = lane >> 2, tq = lane & 3;
    const int8_t* a_lo = act + gq * ldact + 8 * tq;
    const int8_t* a_hi = act + (gq + 8) * ldact + 8 * tq;
    const float zero[4] = {0.f, 0.f, 0.f, 0.f};
    // the epilogue's view: thread i owns row offset i % 64 and tokens i / 64 + 4j
    const int et = threadIdx.x >> 6, en = threadIdx.x & 63;
    unsigned long long best[4] = {0ull, 0ull, 0ull, 0ull};
    float xs_e[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) xs_e[j] = (tok0 + et + 4 * j < T) ? x.scale[tok0 + et + 4 * j] : 0.f;

    float facc[4][2][4];
    int32_t iacc[4][2][4];
    int since = 0;  // k-steps in facc since the last move to iacc (each k-step adds at most 64*127*127)
    int i = 0;
    bool ok = true;  // false once a wait gave up: the loops still run, every barrier is still met
    for (int grp = glo; grp < ghi; ++grp) {
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    facc[r][h][e] = 0.f;
                    iacc[r][h][e] = 0;
                }
        since = 0;
        for (int k = 0; k < spg; ++k, ++i) {
            const int slot = i % kHeadSlots;
            if (ok && !mbar_wait(&full[slot], (i / kHeadSlots) & 1, kWaitLimit)) {
                atomicExch(err, 1);
                ok = false;
            }
            ok = __all_sync(0xffffffffu, ok);
            const int ks = k * kHeadSlotSC + warp;
            if (ok && ks < ksteps) {
                uint32_t bf[2][2][4];
                load_b_frags_i8(a_lo + ks * kI8KStep, a_hi + ks * kI8KStep, bf);
                const unsigned char* scp = ring + (slot * kHeadSlotSC + warp) * kI8Super;
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const uint4 w0 = *reinterpret_cast<const uint4*>(scp + r * kI8Chunk + lane * 32);
                    const uint4 w1 = *reinterpret_cast<const uint4*>(scp + r * kI8Chunk + lane * 32 + 16);
                    const uint32_t wd[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                    for (int gi = 0; gi < 2; ++gi) {
                        // words (gi, s): [row gq 4 codes][row gq+8 4 codes]
                        uint32_t a_s[2][4];
#pragma unroll
                        for (int s = 0; s < 2; ++s) {
                            i8x4_to_half2x2(wd[(gi * 2 + s) * 2 + 0], a_s[s][0], a_s[s][2]);
                            i8x4_to_half2x2(wd[(gi * 2 + s) * 2 + 1], a_s[s][1], a_s[s][3]);
                        }
                        mma_f16_16816(facc[r][0], a_s[0], bf[gi][0][0], bf[gi][0][1], facc[r][0]);
                        mma_f16_16816(facc[r][0], a_s[1], bf[gi][0][2], bf[gi][0][3], facc[r][0]);
                        mma_f16_16816(facc[r][1], a_s[0], bf[gi][1][0], bf[gi][1][1], facc[r][1]);
                        mma_f16_16816(facc[r][1], a_s[1], bf[gi][1][2], bf[gi][1][3], facc[r][1]);
                    }
                }
                if (++since == 16) {  // 16 * 64 * 127 * 127 < 2^24: still exact; move to int32
#pragma unroll
                    for (int r = 0; r < 4; ++r)
#pragma unroll
                        for (int h = 0; h < 2; ++h)
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                iacc[r][h][e] += (int32_t)facc[r][h][e];
                                facc[r][h][e] = 0.f;
                            }
                    since = 0;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
        }
        // this warp's partial sums of the group -> shared, then reduce over the warps
        int32_t* pw = part + warp * 1024;
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int t0 = h * 8 + 2 * tq, n0 = r * 16 + gq;
                pw[t0 * 64 + n0] = iacc[r][h][0] + (int32_t)facc[r][h][0];
                pw[(t0 + 1) * 64 + n0] = iacc[r][h][1] + (int32_t)facc[r][h][1];
                pw[t0 * 64 + n0 + 8] = iacc[r][h][2] + (int32_t)facc[r][h][2];
                pw[(t0 + 1) * 64 + n0 + 8] = iacc[r][h][3] + (int32_t)facc[r][h][3];
            }
        asm volatile("bar.sync 1, %0;" ::"r"(kConsumers * 32) : "memory");
        const int n = grp * 64 + en;
        const float swn = n < V ? sw[n] : 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int t = et + 4 * j;
            int32_t tot = 0;
#pragma unroll
            for (int w = 0; w < kConsumers; ++w) tot += part[w * 1024 + t * 64 + en];
            const int tg = tok0 + t;
            if (ok && tg < T && n < V) {
                const float l = xs_e[j] * swn * (float)tot;
                if (logits) logits[(int64_t)tg * ldl + n] = l;
                best[j] = max(best[j], argmax_key(l, (uint32_t)n));
            }
        }
        asm volatile("bar.sync 1, %0;" ::"r"(kConsumers * 32) : "memory");
    }
    // per token: the best key of this CTA -> one atomicMax
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        unsigned long long b = best[j];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) b = max(b, __shfl_xor_sync(0xffffffffu, b, o));
        best[j] = b;
    }
    // threads et = warp / 2: two warps per token group; combine through shared memory
    unsigned long long* red = reinterpret_cast<unsigned long long*>(part);
    if (lane == 0)
#pragma unroll
        for (int j = 0; j < 4; ++j) red[warp * 4 + j] = best[j];
    asm volatile("bar.sync 1, %0;" ::"r"(kConsumers * 32) : "memory");
    if (threadIdx.x < 16) {
        const int t = threadIdx.x, e = t & 3, j = t >> 2;  // token t = e + 4 j
        const unsigned long long b = max(red[(2 * e) * 4 + j], red[(2 * e + 1) * 4 + j]);
        if (tok0 + t < T && b) atomicMax(keys + tok0 + t, b);
    }
}

int head_stream(const int8_t* packed, const float* row_scale, int V, int ksteps, QAct x, int T, float* logits,
                int ldl, unsigned long long* keys, int num_sms, int* err_flag, cudaStream_t st) {
    if (T <= 0) return 0;
    const int ngroups = (V + 63) / 64;
    const size_t smem = 128 + (size_t)kHeadSlots * kHeadSlotSC * kI8Super + (size_t)kConsumers * 1024 * 4 +
                        (size_t)16 * (ksteps * kI8KStep + kActPad);
    static size_t limit = 0;
    const cudaError_t e = raise_smem_limit(head_stream_kernel, smem, &limit);
    if (e != cudaSuccess) return (int)e;
    dim3 grid(std::min(num_sms, ngroups), (T + 15) / 16);
    return (int)launch(head_stream_kernel, grid, dim3(kStreamThreads), smem, st, packed, row_scale, ngroups, ksteps, V,
                       x, T, logits, ldl, keys, err_flag);
}

}  // namespace dflash
