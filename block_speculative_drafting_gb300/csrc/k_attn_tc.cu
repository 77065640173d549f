// The block's attention on the fifth-generation tensor cores (tcgen05):
// page "cortiq-engine 0.8.71 — src/dflash.rs", `Drafter::block` (scores of
// the block's queries against [context keys ‖ block keys], softmax, the
// weighted sum of the values), with the key splits of one (sequence, kv
// head) unit merged as the accumulate mode of the warp-MMA kernel does.
//
// One CTA takes the unit's query rows (the rep q heads of the kv head times
// the block rows, at most 128: the MMA's M, zero-padded) against its share of
// the unit's keys, in steps of 128 keys:
//   S = Q K^T    (tcgen05.mma kind::f16, M 128, N 128: three products a k16
//                 slice, qh.kh + qh.kl + ql.kh, f32 in tensor memory),
//   P = 2^(S * scale * log2(e) - m)   (two threads a query row, f32, online:
//                 m moves only when a row's maximum passes it by more than
//                 kAtLazy, so P stays within 2^kAtLazy, and the output rows in
//                 tensor memory are then rescaled in place),
//   O += P V     (M 128, N = head_dim, K 128: ph.vh + ph.vl + pl.vh).
// Every operand reaches the tensor cores as the f16 (hi, lo) pair of an f32
// value (the context store keeps its keys and values in that form already);
// the products hi*hi + hi*lo + lo*hi keep f32-level accuracy.  Q and P sit in
// tensor memory (the A operands); K is a K-major tile in the 128-byte swizzle
// and V is read as stored ([key][dim]), the B operand in its MN-major form.
// Steps of 128 keys, not 64: a scores MMA of N 64 runs at two thirds of the
// pipe's rate (measured, chained M 128 x K 16 MMAs: 24.9 ns at N 64, 33.0 ns
// at N 128), so the larger step takes a quarter less MMA time a key.
//
// Roles: warps 0-7 prepare the queries (RMSNorm, rotation, split; staged 64
// rows at a time on their way to tensor memory) and run the softmax and the
// epilogue, threads t and t + 128 owning query row t (tensor-memory lane t),
// each one half of a step's keys; warp 8 allocates the tensor memory and one
// of its lanes issues the MMAs; warps 9-12 move the keys and values into a
// ring of three slots (tensor copies of the store; the block's own rows
// normed, rotated and split from qkv by threads).  S holds one step: the MMAs
// of the next step's scores wait until the softmax has read this step's.
// Every wait is bounded (1 s of %globaltimer): on expiry the CTA raises the
// error flag, the roles stop, work in flight is waited for and the tensor
// memory is freed.
#include <cuda.h>

#include <algorithm>

#include "attn.cuh"
#include "common.cuh"
#include "kernels.cuh"
#include "tc.cuh"

namespace dflash {

constexpr int kAtM = 128;        // MMA M: a unit's query rows, zero-padded
constexpr int kAtKeys = 128;     // keys a step: the scores' N, the values' K
constexpr int kAtSoftWarps = 8;  // two threads a query row: warps w and w + 4 share tensor-memory lanes
constexpr int kAtSoft = kAtSoftWarps * 32;
constexpr int kAtMmaWarp = kAtSoftWarps;
constexpr int kAtLoadWarp0 = kAtSoftWarps + 1;
constexpr int kAtLoadWarps = 4;                    // the block step: two write the keys, two the values
constexpr int kAtLoaders = kAtLoadWarps / 2 * 32;  // threads of one loader group
constexpr int kAtThreads = (kAtSoftWarps + 1 + kAtLoadWarps) * 32;  // 416
constexpr int kAtSlots = 3;      // ring slots, each one step's keys or values (hi and lo planes)
constexpr int kAtQRows = 64;     // query rows staged at a time on their way to tensor memory
constexpr float kAtLazy = 8.f;   // log2 units a row's maximum may pass its reference before a rescale
constexpr uint64_t kAtWait = 1000000000ull;

template <int HD>
struct AtShape {
    static constexpr int KB = HD / 64;                // 64-column (128-byte) blocks of a row
    static constexpr int kPlane = kAtKeys * HD * 2;   // a K or V plane of a step: KB blocks of 128 rows x 128 B
    static constexpr int kItem = 2 * kPlane;          // a ring slot: the step's hi and lo planes
    static constexpr int kQStage = kAtQRows * HD * 2;  // a staged plane of Q: KB blocks of 64 rows x 128 B
    static constexpr size_t kSmem =
        1024 /*alignment*/ + 2048 /*control*/ + 2 * (size_t)kQStage + (size_t)kAtSlots * kItem;
    // tensor memory: S (the step's 128 scores a row), O, then the A operands
    // of the two products -- Q (hi, lo) and P (hi, lo), two f16 a column
    static constexpr int kCols = 512;
    static constexpr int kColS = 0, kColO = kAtKeys, kColQ = 256, kColQl = kColQ + HD / 2, kColP = 384,
                         kColPl = kColP + kAtKeys / 2;
    static_assert(kColO + HD <= kColQ && kColQl + HD / 2 <= kColP && kColPl + kAtKeys / 2 <= kCols, "tensor memory");
    static_assert(kSmem <= 227 * 1024, "shared memory");
};

struct AtCtl {
    // per ring slot: its tile landed / its MMAs done; the scores landed /
    // read out by the softmax; Q in tensor memory; P written / its MMAs
    // done; every MMA done
    uint64_t full[kAtSlots], empty[kAtSlots], s_full, s_free, q_ready, p_full, p_empty, fin;
    uint32_t tmem;
    int abort;
    float xch[2][kAtM];  // the two halves of each row's step maximum (then of its softmax sum)
};
constexpr int kAtCtl = 2048;  // the control block's bytes (a multiple of 1024: the tiles after it stay aligned)
static_assert(sizeof(AtCtl) <= kAtCtl, "control block");

// tcgen05.mma kind::f16 instruction descriptor: D f32, A and B f16, A K-major,
// B K-major (b_mn false) or MN-major, N and M.
__host__ __device__ constexpr uint32_t at_idesc(int M, int N, bool b_mn) {
    return (1u << 4) | ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// Shared-memory matrix descriptor in the 128-byte swizzle: 8-row atoms of
// 128-byte rows (1024 bytes, SBO between atoms along the rows), `lbo` between
// 64-element blocks along the contiguous dimension (used by the MN-major form).
DF_DEV uint64_t at_desc(uint32_t saddr, uint32_t lbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// byte offset of the 16-byte chunk c of row r in a 128-byte-swizzled block
DF_DEV uint32_t at_swz(int r, int c) { return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4)); }

// tcgen05.mma kind::f16 with the A operand in tensor memory (lane = row, two
// f16 a column) and B in shared memory by its descriptor
DF_DEV void at_mma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}
DF_DEV void at_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}
DF_DEV void at_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
DF_DEV void at_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
DF_DEV void at_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
DF_DEV void at_st16(uint32_t taddr, const float (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15]))
        : "memory");
}
DF_DEV void at_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
DF_DEV void at_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// Named barrier 1 of the softmax warps that also ORs a predicate over them:
// every participant leaves with the same answer, so loops that end on it end
// together (no warp is left waiting at a later barrier).
DF_DEV bool at_bar_or(bool v) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n bar.red.or.pred p, 1, %2, q;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(kAtSoft)
        : "memory");
    return r != 0;
}
// a 4-D tensor copy (box at coordinates x, y, z, w) completing on `bar`
DF_DEV void at_tma_4d(void* dst, const CUtensorMap* map, int x, int y, int z, int w, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, "
        "%5}], [%6];" ::"r"(smem_addr(dst)),
        "l"(map), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_addr(bar))
        : "memory");
}
// 2^x by the special-function unit (ex2.approx: relative error about 2^-22,
// the level of f32 rounding; results below 2^-126 flush to zero)
DF_DEV float at_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// CTA (split sp, kv head g, sequence s).  yacc / lacc as the accumulate mode
// of attn_cluster_kernel: each query row's output, rescaled to 2^ref_log2,
// is added into yacc and its softmax sum into lacc.
template <int HD, bool WIN>
__global__ void __launch_bounds__(kAtThreads, 1)
    attn_tc_kernel(const float* __restrict__ qkv, int ld, int block_len, const AttnSeq* __restrict__ seqs, int nq,
                   int nkv, int nsplit, float scale_log2, float* __restrict__ yacc, float* __restrict__ lacc,
                   float ref_log2, const float* __restrict__ q_norm, const float* __restrict__ k_norm,
                   const float2* __restrict__ rope, float eps, int kv_ready, int* __restrict__ err) {
    using S = AtShape<HD>;
    constexpr int D4 = HD / 4;       // lanes of a row (float4 each)
    constexpr int RPW = 32 / D4;     // rows a warp handles at once
    extern __shared__ __align__(1024) unsigned char sm_raw[];
    unsigned char* sm = sm_raw + ((1024 - (smem_addr(sm_raw) & 1023)) & 1023);
    AtCtl& ctl = *reinterpret_cast<AtCtl*>(sm);
    unsigned char* qh = sm + kAtCtl;
    unsigned char* ql = qh + S::kQStage;
    unsigned char* ring = ql + S::kQStage;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sp = blockIdx.x, g = blockIdx.y, s = blockIdx.z;
    const int rep = nq / nkv, mq = rep * block_len;
    const int64_t row0 = (int64_t)s * block_len;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kAtSlots; ++i) {
            mbar_init(&ctl.full[i], 1);
            mbar_init(&ctl.empty[i], 1);
        }
        mbar_init(&ctl.s_full, 1);
        mbar_init(&ctl.s_free, kAtSoft);
        mbar_init(&ctl.q_ready, kAtSoft);
        mbar_init(&ctl.p_full, kAtSoft);
        mbar_init(&ctl.p_empty, 1);
        mbar_init(&ctl.fin, 1);
        ctl.abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kAtMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&ctl.tmem)),
                     "r"(S::kCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    at_fence_before();
    __syncthreads();
    at_fence_after();
    const uint32_t tmem = ctl.tmem;
    pdl_trigger();

    auto give_up = [&]() {
        atomicExch(err, 1);
        *reinterpret_cast<volatile int*>(&ctl.abort) = 1;
    };
    auto aborted = [&]() { return *reinterpret_cast<volatile int*>(&ctl.abort) != 0; };

    // the context view: ahead of the dependency wait only when the caller
    // vouches that the views and stores were final before the launch sequence
    if (!kv_ready) pdl_wait();
    const AttnSeq sq = seqs[s];
    const int total = sq.n + block_len;
    // this sequence's keys, the block's rows first, in nsplit equal shares;
    // a share that holds block rows starts with a step of them alone (written
    // by threads), then its context rows go by in 128-key steps (tensor copies)
    const int kps = (total + nsplit - 1) / nsplit;
    const int j0 = sp * kps, j1 = min(total, j0 + kps);
    const int nb = (j0 < j1 && j0 < block_len) ? 1 : 0;
    const int c0 = max(j0, block_len) - block_len, c1 = j1 - block_len;  // context rows [c0, c1) of the share
    const int nctx = c1 > c0 ? (c1 - c0 + kAtKeys - 1) / kAtKeys : 0;
    const int nsteps = nb + nctx;
    // step u: tile row 0's key and the end of the step's valid keys
    auto key0 = [&](int u) { return u < nb ? j0 : block_len + c0 + (u - nb) * kAtKeys; };
    auto keyend = [&](int u) { return u < nb ? min(block_len, j1) : j1; };
    // The ring's items in the order the MMAs take them: the keys of step 0,
    // then per step u the next step's keys (while there is one) and step u's
    // values -- K0, K1, V0, K2, V1, ..., V(n-1).  Item n goes to slot n % 3,
    // which the MMAs of item n - 3 have released.
    const int nitems = 2 * nsteps;
    auto item_v = [&](int n) { return n != 0 && (n == nitems - 1 || (n & 1) == 0); };
    auto item_u = [&](int n) {
        return n == 0 ? 0 : n == nitems - 1 ? nsteps - 1 : (n & 1) ? ((n - 1) >> 1) + 1 : (n - 1) >> 1;
    };

    if (warp >= kAtLoadWarp0) {
        // ------------------------------------------------------------ loads
        // Context steps: one thread issues the tensor copies of each item (128
        // rows x 64 columns a box, both planes) as soon as its slot is free.
        // The block step: two groups of two warps write its keys (normed and
        // rotated) and its values from qkv, zeros past the block's rows.
        const int grp = (warp - kAtLoadWarp0) / 2;                   // block step: 0 keys, 1 values
        const int lt = threadIdx.x - (kAtLoadWarp0 + 2 * grp) * 32;  // 0 .. 63
        const bool issuer = threadIdx.x == kAtLoadWarp0 * 32;
        auto is_block = [&](int n) { return item_u(n) < nb; };
        auto issue = [&](int n) {
            const CUtensorMap* map = reinterpret_cast<const CUtensorMap*>(sq.maps) + (item_v(n) ? 1 : 0);
            unsigned char* st = ring + (n % kAtSlots) * S::kItem;
            const int row = (int)sq.lo + c0 + (item_u(n) - nb) * kAtKeys;
            uint64_t* bar = &ctl.full[n % kAtSlots];
            mbar_arrive_expect_tx(bar, (uint32_t)S::kItem);
#pragma unroll
            for (int pl2 = 0; pl2 < 2; ++pl2)
#pragma unroll
                for (int kb = 0; kb < S::KB; ++kb)
                    at_tma_4d(st + pl2 * S::kPlane + kb * (kAtKeys * 128), map, kb * 64, row, g, pl2, bar);
        };
        int next = 0;  // the issuer's next item
        // the first items find their slots free
        if (issuer && kv_ready)
            for (; next < min(kAtSlots, nitems); ++next)
                if (!is_block(next)) issue(next);
        pdl_wait();
        if (nb) {
            // the block step: keys (item 0) or values (item 2, or 1 when it is the only step)
            const int n = grp ? (nsteps == 1 ? 1 : 2) : 0;
            unsigned char* st = ring + (n % kAtSlots) * S::kItem;
            const int lim = min(block_len, j1) - j0;
            for (int i = lt; i < (kAtKeys - lim) * (HD / 8); i += kAtLoaders) {
                const int kk = lim + i / (HD / 8), c = i % (HD / 8);
                const uint32_t off = (uint32_t)((c >> 3) * (kAtKeys * 128)) + at_swz(kk, c & 7);
                *reinterpret_cast<uint4*>(st + off) = make_uint4(0u, 0u, 0u, 0u);
                *reinterpret_cast<uint4*>(st + S::kPlane + off) = make_uint4(0u, 0u, 0u, 0u);
            }
            const int lw = (warp - kAtLoadWarp0) & 1, sub = lane / D4, d4 = lane % D4, d = 4 * d4;
            float4 gk = make_float4(1.f, 1.f, 1.f, 1.f);
            if (k_norm != nullptr && !grp) gk = *reinterpret_cast<const float4*>(k_norm + d);
#pragma unroll 1
            for (int kb0 = lw * RPW; kb0 < lim; kb0 += 2 * RPW) {
                const int kr = kb0 + sub, j = j0 + kr;
                const bool mine = kr < lim;
                float4 x = make_float4(0.f, 0.f, 0.f, 0.f), t01 = x, t23 = x;
                if (mine) {
                    x = *reinterpret_cast<const float4*>(qkv + (row0 + j) * ld + (int64_t)(nq + grp * nkv + g) * HD + d);
                    if (!grp && k_norm != nullptr && rope != nullptr) rope_pairs<HD>(rope, row0 + j, d4, t01, t23);
                }
                if (!grp && k_norm != nullptr) norm_rope4<HD>(x, mine, gk, t01, t23, d4, eps, rope != nullptr);
                if (mine) {
                    const uint32_t off = (uint32_t)((d >> 6) * (kAtKeys * 128)) + at_swz(kr, (d & 63) >> 3) + (d & 7) * 2;
                    split_store4(x, reinterpret_cast<__half*>(st + off), reinterpret_cast<__half*>(st + S::kPlane + off));
                }
            }
            fence_proxy_async_smem();
            asm volatile("bar.sync %0, %1;" ::"r"(2 + grp), "r"(kAtLoaders) : "memory");
            if (lt == 0) mbar_arrive(&ctl.full[n % kAtSlots]);
        }
        if (issuer) {
            for (; next < nitems; ++next) {
                if (is_block(next)) continue;
                if (aborted()) break;
                // the slot is free once the MMAs of item next - 3 are done
                if (next >= kAtSlots &&
                    !mbar_wait(&ctl.empty[next % kAtSlots], ((next / kAtSlots) - 1) & 1, kAtWait)) {
                    give_up();
                    break;
                }
                issue(next);
            }
            // no copy may still land in this CTA's memory after it exits
            for (int n = max(0, next - kAtSlots); n < next; ++n)
                if (!is_block(n)) mbar_wait(&ctl.full[n % kAtSlots], (n / kAtSlots) & 1, kAtWait);
        }
    } else if (warp == kAtMmaWarp) {
        // ------------------------------------------------------------ MMAs
        if (lane == 0 && nsteps > 0) {
            constexpr uint32_t idS = at_idesc(kAtM, kAtKeys, false), idO = at_idesc(kAtM, HD, true);
            // descriptors: built once; an operand's k16 slice is its base plus
            // the slice's byte offset / 16 (the start field never carries)
            const uint64_t dk0 = at_desc(smem_addr(ring), 16);
            const uint64_t dv0 = at_desc(smem_addr(ring), kAtKeys * 128);
            constexpr uint64_t kItemD = S::kItem >> 4, kPlaneD = S::kPlane >> 4;
            bool ok = mbar_wait(&ctl.q_ready, 0, kAtWait);
            int it = 0;  // the next ring item
            // S = Q K^T of the next item's keys
            auto scores = [&]() -> bool {
                const int n = it++;
                if (!mbar_wait(&ctl.full[n % kAtSlots], (n / kAtSlots) & 1, kAtWait)) return false;
                at_fence_after();
                const uint64_t kh = dk0 + (uint64_t)(n % kAtSlots) * kItemD, kl = kh + kPlaneD;
#pragma unroll
                for (int j = 0; j < HD / 16; ++j) {
                    // Q's k16 slice j: columns 8 j .. of its planes in tensor memory
                    const uint32_t qh_t = tmem + (uint32_t)(S::kColQ + 8 * j), ql_t = tmem + (uint32_t)(S::kColQl + 8 * j);
                    const uint64_t ko = (uint64_t)(((j >> 2) * (kAtKeys * 128) + (j & 3) * 32) >> 4);
                    at_mma_ts(tmem + S::kColS, qh_t, kh + ko, idS, j > 0 ? 1u : 0u);
                    at_mma_ts(tmem + S::kColS, qh_t, kl + ko, idS, 1u);
                    at_mma_ts(tmem + S::kColS, ql_t, kh + ko, idS, 1u);
                }
                at_commit(&ctl.empty[n % kAtSlots]);
                at_commit(&ctl.s_full);
                return true;
            };
            if (ok) ok = scores();
            for (int u = 0; ok && u < nsteps; ++u) {
                if (aborted()) break;
                if (u + 1 < nsteps) {
                    // S holds one step: the next one's scores once the softmax has read step u's
                    if (!(ok = mbar_wait(&ctl.s_free, u & 1, kAtWait))) break;
                    at_fence_after();
                    if (!(ok = scores())) break;
                }
                if (!(ok = mbar_wait(&ctl.p_full, u & 1, kAtWait))) break;
                const int n = it++;
                if (!(ok = mbar_wait(&ctl.full[n % kAtSlots], (n / kAtSlots) & 1, kAtWait))) break;
                at_fence_after();
                // O += P V of step u: V as stored, [key][dim], the MN-major B operand
                const uint64_t vh = dv0 + (uint64_t)(n % kAtSlots) * kItemD, vl = vh + kPlaneD;
#pragma unroll
                for (int j = 0; j < kAtKeys / 16; ++j) {
                    // P's k16 slice j (keys 16 j ..): columns 8 j .. of its planes
                    const uint32_t ph_t = tmem + (uint32_t)(S::kColP + 8 * j), pl_t = tmem + (uint32_t)(S::kColPl + 8 * j);
                    const uint64_t vo = (uint64_t)((j * 2048) >> 4);
                    at_mma_ts(tmem + S::kColO, ph_t, vh + vo, idO, (u > 0 || j > 0) ? 1u : 0u);
                    at_mma_ts(tmem + S::kColO, ph_t, vl + vo, idO, 1u);
                    at_mma_ts(tmem + S::kColO, pl_t, vh + vo, idO, 1u);
                }
                at_commit(&ctl.empty[n % kAtSlots]);
                at_commit(&ctl.p_empty);
            }
            if (!ok) give_up();
            // every MMA issued has completed before the CTA moves on
            at_commit(&ctl.fin);
            mbar_wait(&ctl.fin, 0, kAtWait);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ queries, softmax, epilogue
        pdl_wait();
        {
            // the unit's query rows, normed, rotated and split, staged kAtQRows
            // at a time and moved to tensor memory (the scores' A operand):
            // thread (row tq, half hq) moves dims [hq HD/2, (hq + 1) HD/2) of
            // its row, 8 dims a 16-byte chunk, 4 columns a chunk; rows past
            // the unit's are zeros
            const int sub = lane / D4, d4 = lane % D4, d = 4 * d4;
            float4 gq = make_float4(1.f, 1.f, 1.f, 1.f);
            if (q_norm != nullptr) gq = *reinterpret_cast<const float4*>(q_norm + d);
            const int tq = (warp & 3) * 32 + lane, hq = warp >> 2;
            const uint32_t qlane = tmem + ((uint32_t)((warp & 3) * 32) << 16);
            constexpr int kStride = kAtSoftWarps * RPW;  // rows between a warp's groups
            const int passes = (mq + kAtQRows - 1) / kAtQRows;
#pragma unroll 1
            for (int ps = 0; ps < kAtM / kAtQRows; ++ps) {
                const int rbase = ps * kAtQRows;
                const bool mine = tq >= rbase && tq < rbase + kAtQRows;  // (whole warps)
                if (ps < passes) {
                    // a warp takes RPW rows at once, four such groups a round
                    // with all their loads issued first
#pragma unroll 1
                    for (int rb = warp * RPW; rb < kAtQRows; rb += 4 * kStride) {
                        float4 qv[4], t01[4], t23[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int ii = rbase + rb + e * kStride + sub;
                            qv[e] = t01[e] = t23[e] = make_float4(0.f, 0.f, 0.f, 0.f);
                            if (ii < mq) {
                                const int head = g * rep + ii / block_len, r = ii % block_len;
                                qv[e] = *reinterpret_cast<const float4*>(qkv + (row0 + r) * ld + (int64_t)head * HD + d);
                                if (q_norm != nullptr && rope != nullptr) rope_pairs<HD>(rope, row0 + r, d4, t01[e], t23[e]);
                            }
                        }
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int li = rb + e * kStride + sub;
                            if (li >= kAtQRows) break;
                            if (q_norm != nullptr)
                                norm_rope4<HD>(qv[e], rbase + li < mq, gq, t01[e], t23[e], d4, eps, rope != nullptr);
                            const uint32_t off =
                                (uint32_t)((d >> 6) * (kAtQRows * 128)) + at_swz(li, (d & 63) >> 3) + (d & 7) * 2;
                            split_store4(qv[e], reinterpret_cast<__half*>(qh + off), reinterpret_cast<__half*>(ql + off));
                        }
                    }
                    asm volatile("bar.sync 1, %0;" ::"r"(kAtSoft) : "memory");  // the pass's rows written
                    if (mine) {
#pragma unroll
                        for (int pl2 = 0; pl2 < 2; ++pl2) {
                            const unsigned char* src = pl2 ? ql : qh;
#pragma unroll
                            for (int c4 = 0; c4 < HD / 64; ++c4) {
                                uint32_t w[16];
#pragma unroll
                                for (int k = 0; k < 4; ++k) {
                                    const int cq = hq * (HD / 16) + c4 * 4 + k;  // the row's 16-byte chunk
                                    const uint4 x = *reinterpret_cast<const uint4*>(src + (cq >> 3) * (kAtQRows * 128) +
                                                                                    at_swz(tq - rbase, cq & 7));
                                    w[4 * k] = x.x;
                                    w[4 * k + 1] = x.y;
                                    w[4 * k + 2] = x.z;
                                    w[4 * k + 3] = x.w;
                                }
                                at_st16(qlane + (uint32_t)((pl2 ? S::kColQl : S::kColQ) + hq * (HD / 4) + c4 * 16),
                                        *reinterpret_cast<const float(*)[16]>(w));
                            }
                        }
                    }
                    asm volatile("bar.sync 1, %0;" ::"r"(kAtSoft) : "memory");  // the staging area is read
                } else if (mine) {
                    const float zero[16] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f,
                                            0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int pl2 = 0; pl2 < 2; ++pl2)
#pragma unroll
                        for (int c4 = 0; c4 < HD / 64; ++c4)
                            at_st16(qlane + (uint32_t)((pl2 ? S::kColQl : S::kColQ) + hq * (HD / 4) + c4 * 16), zero);
                }
            }
            at_wait_st();
            at_fence_before();
            mbar_arrive(&ctl.q_ready);
        }
        // thread: query row t (tensor-memory lane t), key half h of each step
        // (keys 64 h .. 64 h + 63) and output columns h HD/2 .. of the row
        const int t = (warp & 3) * 32 + lane, h = warp >> 2;
        constexpr int KH = kAtKeys / 2, OH = HD / 2;
        const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        float m_ref = -INFINITY, l = 0.f;
        // the leading context rows this query row does not see (a windowed layer)
        int cut = kNoCut;
        if constexpr (WIN) cut = sq.cut + t % block_len;
        bool ok = true;
        for (int u = 0; u < nsteps; ++u) {
            // every exit below is decided by a barrier reduction over the
            // softmax warps: all of them leave the loop at the same step
            const bool got = mbar_wait(&ctl.s_full, u & 1, kAtWait);
            at_fence_after();
            float v[KH];
#pragma unroll
            for (int c = 0; c < KH; c += 16)
                at_ld16(lane_addr + (uint32_t)(S::kColS + h * KH + c), *reinterpret_cast<float(*)[16]>(v + c));
            at_wait_ld();
            // the scores are in registers: their columns may take the next step's
            at_fence_before();
            mbar_arrive(&ctl.s_free);
            const int jb = key0(u) + h * KH, jend = keyend(u);
            float rmax = -INFINITY;
            if (!WIN && jb + KH <= jend) {
#pragma unroll
                for (int c = 0; c < KH; ++c) {
                    v[c] *= scale_log2;
                    rmax = fmaxf(rmax, v[c]);
                }
            } else {
#pragma unroll
                for (int c = 0; c < KH; ++c) {
                    const int key = jb + c;
                    const bool seen = key < jend && (!WIN || key < block_len || key - block_len >= cut);
                    v[c] = seen ? v[c] * scale_log2 : -INFINITY;
                    rmax = fmaxf(rmax, v[c]);
                }
            }
            // the row's maximum over both halves (the partner thread's through
            // shared memory, between two named barriers of the softmax warps)
            ctl.xch[h][t] = rmax;
            if (at_bar_or(!got || aborted())) {
                ok = false;
                break;
            }
            rmax = fmaxf(rmax, ctl.xch[h ^ 1][t]);
            // the previous step's values are added (P is free and O final)
            const bool freed = u == 0 || mbar_wait(&ctl.p_empty, (u - 1) & 1, kAtWait);
            if (at_bar_or(!freed)) {
                ok = false;
                break;
            }
            // the row's reference moves only when its maximum passes it by
            // more than kAtLazy (P then stays within 2^kAtLazy)
            const float m_new = (rmax > m_ref + kAtLazy || (m_ref == -INFINITY && rmax > -INFINITY)) ? rmax : m_ref;
            const float f = (m_ref == -INFINITY) ? 0.f : exp2f(m_ref - m_new);
            at_fence_after();
            if (__any_sync(0xffffffffu, u > 0 && m_new != m_ref)) {
                // rescale this warp's half of its output rows in tensor memory
                const float fr = (m_new != m_ref) ? f : 1.f;
#pragma unroll 1
                for (int c = 0; c < OH; c += 16) {
                    float o[16];
                    at_ld16(lane_addr + (uint32_t)(S::kColO + h * OH + c), o);
                    at_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) o[i] *= fr;
                    at_st16(lane_addr + (uint32_t)(S::kColO + h * OH + c), o);
                }
                at_wait_st();
            }
            l *= f;
            m_ref = m_new;
            // P of the row's key half: (hi, lo) f16 pairs, two keys a
            // tensor-memory column (the A operand of O += P V), 32 keys a store
#pragma unroll
            for (int c32 = 0; c32 < KH / 32; ++c32) {
                uint32_t phw[16], plw[16];
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) {
                    float p[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float x = v[c32 * 32 + c8 * 8 + i];
                        p[i] = (x == -INFINITY) ? 0.f : at_exp2(x - m_ref);
                        l += p[i];
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const __half2 hh = __floats2half2_rn(p[2 * i], p[2 * i + 1]);
                        const float2 hf = __half22float2(hh);
                        const __half2 lo2 = __floats2half2_rn(p[2 * i] - hf.x, p[2 * i + 1] - hf.y);
                        phw[c8 * 4 + i] = *reinterpret_cast<const uint32_t*>(&hh);
                        plw[c8 * 4 + i] = *reinterpret_cast<const uint32_t*>(&lo2);
                    }
                }
                at_st16(lane_addr + (uint32_t)(S::kColP + h * (KH / 2) + c32 * 16), *reinterpret_cast<const float(*)[16]>(phw));
                at_st16(lane_addr + (uint32_t)(S::kColPl + h * (KH / 2) + c32 * 16),
                        *reinterpret_cast<const float(*)[16]>(plw));
            }
            at_wait_st();
            at_fence_before();
            mbar_arrive(&ctl.p_full);
        }
        // the row's softmax sum over both halves (every softmax thread gets
        // here: the loop's exits are uniform)
        ctl.xch[h][t] = l;
        asm volatile("bar.sync 1, %0;" ::"r"(kAtSoft) : "memory");
        if (__all_sync(0xffffffffu, ok && !aborted()) && nsteps > 0) {
            // the output: wait for the last values, rescale to 2^ref_log2 and add
            if (!__all_sync(0xffffffffu, mbar_wait(&ctl.p_empty, (nsteps - 1) & 1, kAtWait))) {
                ok = false;
            } else {
                at_fence_after();
                const float f = (m_ref == -INFINITY) ? 0.f : exp2f(m_ref - ref_log2);
                const bool live = t < mq;
                const int head = g * rep + t / block_len, r = t % block_len;
                float* dst = yacc + (row0 + r) * ((int64_t)nq * HD) + (int64_t)head * HD + h * OH;
#pragma unroll 1
                for (int c = 0; c < OH; c += 16) {
                    float o[16];
                    at_ld16(lane_addr + (uint32_t)(S::kColO + h * OH + c), o);
                    at_wait_ld();
                    if (live)
#pragma unroll
                        for (int i = 0; i < 16; i += 4)
                            red_add_v4(dst + c + i, o[i] * f, o[i + 1] * f, o[i + 2] * f, o[i + 3] * f);
                }
                if (live && h == 0) atomicAdd(lacc + (row0 + r) * nq + head, (ctl.xch[0][t] + ctl.xch[1][t]) * f);
            }
        }
        if (!ok) give_up();
    }
    at_fence_before();
    __syncthreads();
    if (warp == kAtMmaWarp) {
        at_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(S::kCols) : "memory");
    }
}

template <int HD, bool WIN>
static int attention_tc_hd(const float* qkv, int ld, int n_seqs, int block_len, const AttnSeq* seqs_dev, int nsplit,
                           int nq, int nkv, float scale, float* yacc, float* lacc, float ref_log2, cudaStream_t st,
                           const float* q_norm, const float* k_norm, const float2* rope, float eps, int kv_ready,
                           int* err) {
    static const cudaError_t attr = cudaFuncSetAttribute(attn_tc_kernel<HD, WIN>,
                                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                         (int)AtShape<HD>::kSmem);
    if (attr != cudaSuccess) return (int)attr;
    const float scale_log2 = scale * 1.4426950408889634f;
    return (int)launch(attn_tc_kernel<HD, WIN>, dim3(nsplit, nkv, n_seqs), dim3(kAtThreads), AtShape<HD>::kSmem, st,
                       qkv, ld, block_len, seqs_dev, nq, nkv, nsplit, scale_log2, yacc, lacc, ref_log2, q_norm, k_norm,
                       rope, eps, kv_ready, err);
}

int attn_tc_plan(int n_seqs, int block_len, int max_ctx, int nkv, int num_sms) {
    // one CTA a unit when the units fill the SMs; otherwise the keys of each
    // unit split over floor(SMs / units) CTAs (one wave)
    const int units = nkv * n_seqs;
    if (units >= num_sms) return 1;
    const int max_split = std::max(1, (max_ctx + block_len + kAtKeys - 1) / kAtKeys);
    return std::max(1, std::min(max_split, num_sms / units));
}


bool kv_tensor_maps(const __half* k, const __half* v, int nkv, int64_t cap, int hd, void* out) {
    EncodeTiledFn enc = encode_fn();
    if (!enc || (hd != 64 && hd != 128) || cap < 1 || (reinterpret_cast<uintptr_t>(out) & 63)) return false;
    // [plane][kv][cap][hd]: boxes of 64 head_dim columns x kAtKeys rows, one kv head and plane a box
    const cuuint64_t dims[4] = {(cuuint64_t)hd, (cuuint64_t)cap, (cuuint64_t)nkv, 2};
    const cuuint64_t strides[3] = {(cuuint64_t)hd * 2, (cuuint64_t)cap * hd * 2, (cuuint64_t)nkv * cap * hd * 2};
    const cuuint32_t box[4] = {64, (cuuint32_t)kAtKeys, 1, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    CUtensorMap* m = reinterpret_cast<CUtensorMap*>(out);
    for (int i = 0; i < 2; ++i)
        if (enc(m + i, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, const_cast<__half*>(i ? v : k), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    return true;
}

bool attention_tc_supported(int nq, int nkv, int hd, int block_len) {
    return (hd == 64 || hd == 128) && nq % nkv == 0 && (nq / nkv) * block_len <= kAtM && block_len <= kAtKeys;
}

int attention_tc(const float* qkv, int ld, int n_seqs, int block_len, const AttnSeq* seqs_dev, int nsplit, int nq,
                 int nkv, int hd, float scale, float* yacc, float* lacc, float ref_log2, cudaStream_t st,
                 const float* q_norm, const float* k_norm, const float2* rope, float eps, bool kv_ready, bool windowed,
                 int* err) {
    if (!attention_tc_supported(nq, nkv, hd, block_len) || !q_norm || !k_norm || !yacc || !lacc || nsplit < 1 ||
        (reinterpret_cast<uintptr_t>(yacc) & 15) || (reinterpret_cast<uintptr_t>(qkv) & 15) || ld % 4)
        return (int)cudaErrorInvalidValue;
    const int kr = kv_ready ? 1 : 0;
    if (hd == 128)
        return windowed ? attention_tc_hd<128, true>(qkv, ld, n_seqs, block_len, seqs_dev, nsplit, nq, nkv, scale, yacc,
                                                     lacc, ref_log2, st, q_norm, k_norm, rope, eps, kr, err)
                        : attention_tc_hd<128, false>(qkv, ld, n_seqs, block_len, seqs_dev, nsplit, nq, nkv, scale,
                                                      yacc, lacc, ref_log2, st, q_norm, k_norm, rope, eps, kr, err);
    return windowed ? attention_tc_hd<64, true>(qkv, ld, n_seqs, block_len, seqs_dev, nsplit, nq, nkv, scale, yacc, lacc,
                                                ref_log2, st, q_norm, k_norm, rope, eps, kr, err)
                    : attention_tc_hd<64, false>(qkv, ld, n_seqs, block_len, seqs_dev, nsplit, nq, nkv, scale, yacc,
                                                 lacc, ref_log2, st, q_norm, k_norm, rope, eps, kr, err);
}

}  // namespace dflash
