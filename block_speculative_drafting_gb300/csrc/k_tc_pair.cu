// Dense contractions of many rows on pairs of SMs (tcgen05.mma cta_group::2):
// the 4-bit g32 matrices from their exact hi + lo f16 copies and the int8
// head from its f16 copy, against the rows' int8 codes as f16 -- the same
// products as the kernels of k_tc.cu ("cortiq-engine 0.8.75 --
// src/gpu_wgpu/dflash_dev.rs", `Dev::q4` / `Dev::q8`, applied to many rows:
// the prefill of context rows and the blocks of many sequences at once).
//
// Layout of the work.  A unit is 256 rows x 256 outputs x a slice of K.  The
// two CTAs of a cluster run it together: CTA r holds rows 128 r .. of the
// activation tile and weight rows (outputs) 128 r .. of each plane in its own
// shared memory, and the pair's leader (rank 0) issues M 256 x N 256 x K 16
// MMAs that read both CTAs' halves -- each SM's tensor core reads a weight
// tile half from its own shared memory and shares it with the other, so a
// multiply-add takes a third less operand traffic per SM than a one-SM tile
// of the same size.  D (f32) lands in tensor memory, 128 lanes x 256 columns
// in each CTA.
//
// Persistence.  The grid is one pair per two SMs (at most); pair p takes
// units p, p + P, p + 2P, ... (row tiles fastest, so the pairs that run at
// the same time share weight tiles).  Tensor memory holds two accumulators:
// while the epilogue warps drain unit j's, the MMAs of unit j + 1 fill the
// other, and the TMA ring keeps loading across unit boundaries -- the
// epilogue and the pipeline fill of a one-unit CTA no longer show.
//
// Roles (per CTA):
//   warp 8, one lane: TMA -- this CTA's activation rows and weight halves of
//     each k-block into a ring of stages; completion is counted on the
//     leader's barrier (the cta_group::2 form of the copy).  Weight tiles go
//     out before the wait on the previous kernel (they are written only when
//     the model is built), and later ones are prefetched into L2 ahead.
//   warp 9: allocates the pair's tensor memory (both CTAs, collectively);
//     on the leader one lane issues the MMAs and commits each consumed stage
//     and each finished accumulator to both CTAs' barriers.
//   warps 0-7: the epilogue.  Warp w reads lanes 32 (w % 4) .. (its 32 rows)
//     and columns 128 (w / 4) .. of the accumulator, 32 columns at a time,
//     scales them (the 4-bit matrices: the row scale; the head: row and
//     vocabulary scales, the argmax, the exactness guard), and writes each
//     32 x 32 block through a 4 KB shared-memory box in the 128-byte
//     swizzle with one TMA store or reduce-add.  It then hands the
//     accumulator back to the leader (a remote arrive for the other CTA).
// Every wait is bounded (1 s of %globaltimer); on expiry the kernel raises
// the error flag and the roles stop.  Both CTAs meet at a cluster barrier
// before either frees its tensor memory or leaves, so no CTA's barriers or
// tensor memory go away while the other may still use them.
#include <cuda.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.cuh"
#include "tc.cuh"

namespace dflash {

constexpr int kPM = 128;                  // rows of a CTA: its half of the pair's M = 256
constexpr int kPN = 256;                  // outputs of a unit: MMA N (each CTA holds 128 weight rows)
constexpr int kPKB = 64;                  // k-block: one 128-byte swizzle row of f16
constexpr int kPA = kPM * kPKB * 2;       // 16 KB: a CTA's activation tile of a k-block
constexpr int kPB = (kPN / 2) * kPKB * 2; // 16 KB: a CTA's half of one weight plane
constexpr int kPEpiWarps = 8;
constexpr int kPThreads = (kPEpiWarps + 2) * 32;
constexpr int kPTmaWarp = kPEpiWarps, kPMmaWarp = kPEpiWarps + 1;
constexpr int kPBox = 32 * 32 * 4;        // a warp's staging box: 32 rows x 32 f32 columns
constexpr int kPMaxKb = 32;               // k-blocks of a 4-bit unit at most (the f32 accumulation)
constexpr int kPTmemCols = 2 * kPN;       // two accumulators
constexpr uint64_t kPWait = 1000000000ull;
// kind::f16 instruction descriptor: D f32, A and B f16, both K-major, N 256, M 256
constexpr uint32_t kPIdesc = (1u << 4) | ((uint32_t)(kPN >> 3) << 17) | ((uint32_t)(256 >> 4) << 24);

template <bool kHead>
struct PShape {
    static constexpr int kPlanes = kHead ? 1 : 2;
    static constexpr int kStage = kPA + kPlanes * kPB;  // 48 KB (hi + lo) or 32 KB (head)
    static constexpr int kStages = kHead ? 6 : 4;
    static constexpr int kAhead = kHead ? 8 : 4;  // k-blocks of weights prefetched into L2 ahead of the ring
    static constexpr size_t kSmem = 1024 /*alignment*/ + 1024 /*control*/ + (size_t)kStages * kStage +
                                    (size_t)kPEpiWarps * kPBox;
    static_assert(kSmem <= 227 * 1024, "shared memory");
};
constexpr int kPMaxStages = 6;

struct PCtl {
    uint64_t full[kPMaxStages], empty[kPMaxStages], acc_full[2], acc_empty[2];
    uint32_t tmem;
    int abort;
};
static_assert(sizeof(PCtl) <= 1024, "control block");

struct PairArgs {
    int T, N, K;
    int mt, ntl, splits, kps;  // units: 256-row tiles x output tiles x K slices; k-blocks of a unit
    int slices_inner;          // unit order: row tile, K slice, output tile (else row tile, output tile, K slice)
    const float* xscale;       // [T]
    int reduce;                // add into y (accumulate, or K split over units)
    int y_tma;                 // y through the output map; else plain stores (a head with odd rows)
    float* y;                  // (head: logits, may be null)
    int ldy;
    const float* wscale;       // head: vocabulary row scales [N]
    unsigned long long* keys;  // head: argmax keys [T]
    const int* xn2;            // head guard: squared code norms of the rows [T] and of the vocabulary rows [N],
    const int* wn2;            //   the f16 codes of both, and the largest norm product f32 sums are exact under
    const __half* xf;
    const __half* wf;
    unsigned long long bound;
    unsigned long long wn2_max;
    int* err;
};

DF_DEV uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// the address of the same shared-memory word in CTA `rank` of the cluster
DF_DEV uint32_t peer_addr(const void* p, uint32_t rank) {
    uint32_t d;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(smem_addr(p)), "r"(rank));
    return d;
}
DF_DEV void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
// global -> this CTA's shared memory, completion counted on a barrier of
// either CTA of the pair (a shared::cluster address)
DF_DEV void tma_load_2d_pair(void* dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, {%2, "
        "%3}], [%4];" ::"r"(smem_addr(dst)),
        "l"(map), "r"(x), "r"(y), "r"(bar)
        : "memory");
}
DF_DEV void pair_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
        "l"(a), "l"(b), "r"(kPIdesc), "r"(accumulate)
        : "memory");
}
// arrives on the barrier at this offset in both CTAs once the MMAs issued so far complete
DF_DEV void pair_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_addr(bar)),
        "h"((uint16_t)3)
        : "memory");
}
DF_DEV void mbar_arrive_remote(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar) : "memory");
}
// bounded wait with cluster-scope acquire (arrivals from the other CTA)
DF_DEV bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
    auto poll = [&]() {
        uint32_t ok;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
            " selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(ok)
            : "r"(smem_addr(bar)), "r"(parity)
            : "memory");
        return ok != 0;
    };
    if (poll()) return true;
    const uint64_t t0 = global_ns();
    for (;;) {
        for (int i = 0; i < 64; ++i)
            if (poll()) return true;
        if (global_ns() - t0 > limit_ns) return false;
    }
}

// The exact integer dot product of two rows of f16 codes (|code| <= 127: every
// product is exact in f32), for the head elements the norm guard rejects.
__device__ __noinline__ int exact_dot_codes(const __half* __restrict__ x, const __half* __restrict__ w, int K) {
    int s = 0;
    for (int k = 0; k < K; k += 8) {
        const uint4 a = *reinterpret_cast<const uint4*>(x + k), b = *reinterpret_cast<const uint4*>(w + k);
        const __half2* ah = reinterpret_cast<const __half2*>(&a);
        const __half2* bh = reinterpret_cast<const __half2*>(&b);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 fa = __half22float2(ah[j]), fb = __half22float2(bh[j]);
            s += (int)(fa.x * fb.x) + (int)(fa.y * fb.y);
        }
    }
    return s;
}

// The sequence of k-blocks a pair runs: its units in order, each unit's k-blocks.
struct PairWalk {
    int u, i, mi, ni, kb0, nkb;
    // row tiles fastest; then, with few row tiles, the K slices of an output
    // tile (their partial sums meet in y while its lines are still in L2) and
    // the output tiles, or, with many, the output tiles and the K slices (the
    // pairs at work share the activations of one K slice)
    DF_DEV void decode(const PairArgs& a) {
        mi = u % a.mt;
        const int r = u / a.mt;
        const int si = a.slices_inner ? r % a.splits : r / a.ntl;
        ni = a.slices_inner ? r / a.splits : r % a.ntl;
        kb0 = si * a.kps;
        nkb = min(a.K / kPKB, kb0 + a.kps) - kb0;
    }
    DF_DEV void start(int pair, const PairArgs& a) {
        u = pair;
        i = 0;
        decode(a);
    }
    DF_DEV bool valid(int units) const { return u < units; }
    DF_DEV void next(int npairs, const PairArgs& a) {
        if (++i == nkb) {
            u += npairs;
            i = 0;
            decode(a);
        }
    }
};

// kHead: the head's codes (one plane) against the rows, the logits and the
// argmax in the epilogue, the whole K in tensor memory.  Its products are
// integers, so a sum is exact in f32 while every partial sum stays within
// 2^24 in magnitude; by Cauchy-Schwarz each is at most |x| |w| (code norms),
// so an element whose norm product passes the bound is recomputed as an
// integer dot product instead.
template <bool kHead>
__global__ void __launch_bounds__(kPThreads, 1)
    pair_tc_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap hmap,
                   const __grid_constant__ CUtensorMap lmap, const __grid_constant__ CUtensorMap ymap, PairArgs a) {
    using S = PShape<kHead>;
    extern __shared__ __align__(1024) unsigned char sm_raw[];
    unsigned char* sm = sm_raw + ((1024 - (smem_addr(sm_raw) & 1023)) & 1023);
    PCtl& ctl = *reinterpret_cast<PCtl*>(sm);
    unsigned char* ring = sm + 1024;
    unsigned char* stg = ring + S::kStages * S::kStage;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();  // 0: the pair's leader
    const int pair = (int)(blockIdx.x >> 1), npairs = (int)(gridDim.x >> 1);
    const int units = a.mt * a.ntl * a.splits;

    if (threadIdx.x == 0) {
        for (int i = 0; i < S::kStages; ++i) {
            mbar_init(&ctl.full[i], 1);
            mbar_init(&ctl.empty[i], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&ctl.acc_full[b], 1);
            mbar_init(&ctl.acc_empty[b], 2 * kPEpiWarps);  // every epilogue warp of both CTAs
        }
        ctl.abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kPMmaWarp) {
        // the pair's tensor memory: one warp of each CTA, collectively
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&ctl.tmem)),
                     "r"(kPTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    cluster_sync_all();  // both CTAs' barriers initialised and their tensor memory allocated
    tc_fence_after();
    const uint32_t tmem = ctl.tmem;
    pdl_trigger();

    auto give_up = [&]() {
        atomicExch(a.err, 1);
        *reinterpret_cast<volatile int*>(&ctl.abort) = 1;
    };
    auto aborted = [&]() { return *reinterpret_cast<volatile int*>(&ctl.abort) != 0; };

    if (warp == kPTmaWarp) {
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(&xmap) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(&hmap) : "memory");
            if (!kHead) asm volatile("prefetch.tensormap [%0];" ::"l"(&lmap) : "memory");
            // whole boxes: rows past T or past N read as zeros and count toward the bytes
            auto load_w = [&](const PairWalk& w, int s) {
                unsigned char* dst = ring + s * S::kStage + kPA;
                const uint32_t bar = peer_addr(&ctl.full[s], 0);
                const int x = (w.kb0 + w.i) * kPKB, y = w.ni * kPN + (int)rank * (kPN / 2);
                tma_load_2d_pair(dst, &hmap, x, y, bar);
                if (!kHead) tma_load_2d_pair(dst + kPB, &lmap, x, y, bar);
            };
            auto load_x = [&](const PairWalk& w, int s) {
                tma_load_2d_pair(ring + s * S::kStage, &xmap, (w.kb0 + w.i) * kPKB, w.mi * 256 + (int)rank * kPM,
                                 peer_addr(&ctl.full[s], 0));
            };
            auto prefetch_w = [&](const PairWalk& w) {
                const int x = (w.kb0 + w.i) * kPKB, y = w.ni * kPN + (int)rank * (kPN / 2);
                tma_prefetch_2d(&hmap, x, y);
                if (!kHead) tma_prefetch_2d(&lmap, x, y);
            };
            // the leader's barrier counts both CTAs' bytes of a stage
            auto arm = [&](int s) {
                if (rank == 0) mbar_arrive_expect_tx(&ctl.full[s], (uint32_t)(2 * S::kStage));
            };
            PairWalk cur, pf;
            cur.start(pair, a);
            // the first stages' weights, and an L2 prefetch of the next ones,
            // before the wait on the kernel before (which writes the activations)
            PairWalk w = cur;
            int pre = 0;
            for (; pre < S::kStages && w.valid(units); ++pre, w.next(npairs, a)) {
                arm(pre);
                load_w(w, pre);
            }
            pf = w;
            for (int q = 0; q < S::kAhead && pf.valid(units); ++q, pf.next(npairs, a)) prefetch_w(pf);
            pdl_wait();
            for (int q = 0; q < pre; ++q, cur.next(npairs, a)) load_x(cur, q);
            int g = pre;
            for (; cur.valid(units); ++g, cur.next(npairs, a)) {
                const int s = g % S::kStages;
                if (!mbar_wait(&ctl.empty[s], ((g / S::kStages) - 1) & 1, kPWait)) {
                    give_up();
                    break;
                }
                if (aborted()) break;
                if (pf.valid(units)) {
                    prefetch_w(pf);
                    pf.next(npairs, a);
                }
                arm(s);
                load_x(cur, s);
                load_w(cur, s);
            }
            // until the MMAs have taken the last stages (their commits reach this CTA)
            for (int q = max(0, g - S::kStages); q < g; ++q)
                if (!mbar_wait(&ctl.empty[q % S::kStages], (q / S::kStages) & 1, kPWait)) break;
        }
    } else if (warp == kPMmaWarp) {
        if (rank == 0 && lane == 0) {
            int g = 0;
            bool stop = false;
            for (int u = pair, j = 0; u < units && !stop; u += npairs, ++j) {
                PairWalk w;
                w.u = u;
                w.i = 0;
                w.decode(a);
                const int b = j & 1;
                // the epilogues of both CTAs have drained this accumulator (unit j - 2)
                if (j >= 2 && !mbar_wait_cluster(&ctl.acc_empty[b], ((j >> 1) - 1) & 1, kPWait)) {
                    give_up();
                    break;
                }
                if (aborted()) break;
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(b * kPN);
                for (int i = 0; i < w.nkb; ++i, ++g) {
                    const int s = g % S::kStages;
                    const bool ok = mbar_wait(&ctl.full[s], (g / S::kStages) & 1, kPWait);
                    if (!ok) give_up();
                    if (!ok || aborted()) {
                        stop = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_addr(ring + s * S::kStage), sb = sa + kPA;
#pragma unroll
                    for (int k = 0; k < kPKB / 16; ++k) {
                        const uint64_t ad = tc_desc_sw128(sa + 32 * k);
                        pair_mma(d, ad, tc_desc_sw128(sb + 32 * k), (i > 0 || k > 0) ? 1u : 0u);
                        if (!kHead) pair_mma(d, ad, tc_desc_sw128(sb + kPB + 32 * k), 1u);
                    }
                    pair_commit(&ctl.empty[s]);
                }
                if (!stop) pair_commit(&ctl.acc_full[b]);
            }
        }
    } else {
        // ---------------------------------------------------------------- epilogue
        pdl_wait();  // (the row scales and the outputs belong to the kernels before)
        const int sub = warp & 3, half = warp >> 2;
        unsigned char* box = stg + warp * kPBox;
        bool pending = false;  // lane 0 has a store reading `box`
        for (int u = pair, j = 0; u < units; u += npairs, ++j) {
            PairWalk w;
            w.u = u;
            w.i = 0;
            w.decode(a);
            const int b = j & 1;
            const bool ok = mbar_wait(&ctl.acc_full[b], (j >> 1) & 1, kPWait);
            if (!ok) give_up();
            if (!__all_sync(0xffffffffu, ok && !aborted())) break;
            tc_fence_after();
            const int r0 = w.mi * 256 + (int)rank * kPM + 32 * sub, row = r0 + lane;
            if (r0 < a.T) {  // (uniform in the warp)
                const float xs = row < a.T ? a.xscale[row] : 0.f;
                const unsigned long long xn = kHead && row < a.T ? (uint32_t)a.xn2[row] : 0ull;
                const bool guard = kHead && xn * a.wn2_max > a.bound;
                const bool any_guard = __any_sync(0xffffffffu, guard);
                unsigned long long best = 0ull;
#pragma unroll 1
                for (int cc = 0; cc < kPN / 2; cc += 32) {
                    const int n0 = w.ni * kPN + half * (kPN / 2) + cc;
                    if (n0 >= a.N) break;  // (uniform)
                    // per-column factors, one column a lane, shuffled to the rows
                    const int nl = n0 + lane;
                    const float ws_l = kHead && nl < a.N ? a.wscale[nl] : 0.f;
                    const int wn_l = kHead && any_guard && nl < a.N ? a.wn2[nl] : 0;
                    uint32_t v[32];
                    const uint32_t ta =
                        tmem + ((uint32_t)(32 * sub) << 16) + (uint32_t)(b * kPN + half * (kPN / 2) + cc);
                    tc_ld16(ta, *reinterpret_cast<uint32_t(*)[16]>(v));
                    tc_ld16(ta + 16, *reinterpret_cast<uint32_t(*)[16]>(v + 16));
                    tc_wait_ld();
                    float f[32];
#pragma unroll
                    for (int q = 0; q < 32; ++q) {
                        float acc = __uint_as_float(v[q]);
                        if (kHead) {
                            // logits = xs * sw[n] * (integer row sum), as the streaming head
                            const int n = n0 + q;
                            const float ws = __shfl_sync(0xffffffffu, ws_l, q);
                            if (any_guard) {
                                const int wn = __shfl_sync(0xffffffffu, wn_l, q);
                                if (guard && n < a.N && xn * (uint32_t)wn > a.bound)
                                    acc = (float)exact_dot_codes(a.xf + (int64_t)row * a.K, a.wf + (int64_t)n * a.K,
                                                                 a.K);
                            }
                            f[q] = n < a.N ? xs * ws * acc : 0.f;
                            if (n < a.N && row < a.T) best = max(best, argmax_key(f[q], (uint32_t)n));
                        } else {
                            f[q] = acc * xs;
                        }
                    }
                    if (!a.y) continue;  // (the head's argmax alone)
                    if (!a.y_tma) {
                        // (logit rows that are not 16-byte multiples: plain stores)
                        if (row < a.T)
                            for (int q = 0; q < 32; ++q)
                                if (n0 + q < a.N) a.y[(int64_t)row * a.ldy + n0 + q] = f[q];
                        continue;
                    }
                    if (pending) {
                        if (lane == 0) bulk_wait_read<0>();
                        __syncwarp();
                    }
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        *reinterpret_cast<float4*>(box + lane * 128 + ((c ^ (lane & 7)) << 4)) =
                            make_float4(f[4 * c], f[4 * c + 1], f[4 * c + 2], f[4 * c + 3]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        if (a.reduce)
                            tma_reduce_add_2d(&ymap, box, n0, r0);
                        else
                            tma_store_2d(&ymap, box, n0, r0);
                        bulk_commit();
                    }
                    pending = true;
                }
                if (kHead && row < a.T && best) atomicMax(a.keys + row, best);
            }
            // this warp is done reading the accumulator: back to the leader's MMAs
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(peer_addr(&ctl.acc_empty[b], 0));
        }
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }
    // no CTA of the pair frees its tensor memory or leaves while the other
    // may still signal its barriers or its MMAs may still run
    tc_fence_before();
    cluster_sync_all();
    if (warp == kPMmaWarp) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kPTmemCols) : "memory");
    }
}

// ---------------------------------------------------------------- host side
template <bool kHead>
static cudaError_t pair_setup(int* max_pairs) {
    static bool done[2] = {false, false};
    static int pairs[2] = {0, 0};
    std::lock_guard<std::mutex> lock(attr_mutex());
    if (!done[kHead]) {
        cudaError_t e = cudaFuncSetAttribute(pair_tc_kernel<kHead>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)PShape<kHead>::kSmem);
        if (e != cudaSuccess) return e;
        // how many pairs the GPU holds at once (SMs that cannot pair up stay out)
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2, 1, 1);
        cfg.blockDim = dim3(kPThreads);
        cfg.dynamicSmemBytes = PShape<kHead>::kSmem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, pair_tc_kernel<kHead>, &cfg);
        if (e != cudaSuccess) return e;
        if (n < 1) return cudaErrorInvalidConfiguration;
        pairs[kHead] = n;
        done[kHead] = true;
    }
    *max_pairs = pairs[kHead];
    return cudaSuccess;
}

int q4_tc_dense(const __half* hi, const __half* lo, int N, int K, QAct x, const __half* x16, int T, float* y, int ldy,
               bool accumulate, int* err_flag, cudaStream_t st) {
    if (T <= 0 || N <= 0) return 0;
    if (encode_fn() == nullptr || K % kPKB || N % 64 || ldy % 4 || (reinterpret_cast<uintptr_t>(y) & 15) ||
        (reinterpret_cast<uintptr_t>(x16) & 15) || (reinterpret_cast<uintptr_t>(hi) & 15) ||
        (reinterpret_cast<uintptr_t>(lo) & 15))
        return (int)cudaErrorInvalidValue;
    CUtensorMap xm, hm, lm, ym;
    if (!act_map(&xm, x16, K, T, kPM) || !dense_map(&hm, hi, K, N, kPN / 2) || !dense_map(&lm, lo, K, N, kPN / 2) ||
        !out_map(&ym, y, ldy, N, T))
        return (int)cudaErrorInvalidValue;
    int max_pairs = 0;
    cudaError_t e = pair_setup<false>(&max_pairs);
    if (e != cudaSuccess) return (int)e;
    const int ksteps = K / kPKB, mt = (T + 255) / 256, ntl = (N + kPN - 1) / kPN;
    // K slices of at most kPMaxKb k-blocks: of those, the count whose rounds
    // of units over the pairs, times a unit's k-blocks (plus three for its
    // accumulator hand-over and the reduction of its partial tile into y:
    // measured on the batched step, a charge of one chose five slices for the
    // gate/up matrix where three run faster, and none many more), is least
    const int s_min = (ksteps + kPMaxKb - 1) / kPMaxKb;
    int splits = s_min, kps = (ksteps + s_min - 1) / s_min;
    int64_t best = INT64_MAX;
    for (int sp = s_min; sp <= std::min(ksteps, 8 * s_min); ++sp) {
        const int k = (ksteps + sp - 1) / sp, real = (ksteps + k - 1) / k;
        const int64_t rounds = ((int64_t)mt * ntl * real + max_pairs - 1) / max_pairs;
        const int64_t cost = rounds * (k + 3);
        if (cost < best) {
            best = cost;
            splits = real;
            kps = k;
        }
    }
    if (splits > 1 && !accumulate) {
        e = cudaMemset2DAsync(y, (size_t)ldy * sizeof(float), 0, (size_t)N * sizeof(float), T, st);
        if (e != cudaSuccess) return (int)e;
    }
    PairArgs args{};
    args.T = T;
    args.N = N;
    args.K = K;
    args.mt = mt;
    args.ntl = ntl;
    args.splits = splits;
    args.kps = kps;
    args.xscale = x.scale;
    args.reduce = (accumulate || splits > 1) ? 1 : 0;
    args.slices_inner = mt < 8 ? 1 : 0;
    args.y_tma = 1;
    args.y = y;
    args.ldy = ldy;
    args.err = err_flag;
    const int units = mt * ntl * splits;
    const int pairs = std::min(max_pairs, units);
    return (int)launch_cluster(pair_tc_kernel<false>, dim3(2 * pairs), dim3(kPThreads), PShape<false>::kSmem, st, 2, xm,
                               hm, lm, ym, args);
}

int head_tc_dense(const __half* w16, const int* w_norm2, const float* row_scale, int V, int K, QAct x,
                 const __half* x16, const int* x_norm2, int T, float* logits, int ldl, unsigned long long* keys,
                 unsigned long long bound, unsigned long long w_norm2_max, int* err_flag, cudaStream_t st) {
    if (T <= 0 || V <= 0) return 0;
    if (encode_fn() == nullptr || K % kPKB || (reinterpret_cast<uintptr_t>(x16) & 15) ||
        (reinterpret_cast<uintptr_t>(w16) & 15) || !w_norm2 || !x_norm2)
        return (int)cudaErrorInvalidValue;
    CUtensorMap xm, wm, ym;
    if (!act_map(&xm, x16, K, T, kPM) || !dense_map(&wm, w16, K, V, kPN / 2)) return (int)cudaErrorInvalidValue;
    // the logits through the output map where their rows allow one, else plain stores
    const bool y_tma = out_map(&ym, logits, ldl, V, T);
    if (!y_tma) memset(&ym, 0, sizeof(ym));
    int max_pairs = 0;
    cudaError_t e = pair_setup<true>(&max_pairs);
    if (e != cudaSuccess) return (int)e;
    PairArgs args{};
    args.T = T;
    args.N = V;
    args.K = K;
    args.mt = (T + 255) / 256;
    args.ntl = (V + kPN - 1) / kPN;
    args.splits = 1;
    args.kps = K / kPKB;
    args.xscale = x.scale;
    args.y_tma = y_tma ? 1 : 0;
    args.y = logits;
    args.ldy = ldl;
    args.wscale = row_scale;
    args.keys = keys;
    args.xn2 = x_norm2;
    args.wn2 = w_norm2;
    args.xf = x16;
    args.wf = w16;
    args.bound = bound;
    args.wn2_max = w_norm2_max;
    args.err = err_flag;
    const int units = args.mt * args.ntl;
    const int pairs = std::min(max_pairs, units);
    return (int)launch_cluster(pair_tc_kernel<true>, dim3(2 * pairs), dim3(kPThreads), PShape<true>::kSmem, st, 2, xm,
                               wm, wm, ym, args);
}

}  // namespace dflash
