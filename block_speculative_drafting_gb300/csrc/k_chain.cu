// The chain: one persistent kernel (one CTA per SM) that runs a short program
// of the block's dependent steps -- the 4-bit matvecs of page "cortiq-engine
// 0.8.75 — src/gpu_wgpu/dflash_dev.rs" (`Dev::q4`) and the row steps between
// them of page "cortiq-engine 0.8.71 — src/dflash.rs" (`rms` then the int8
// quantisation of the matvec input; `Drafter::mlp`'s silu(gate) * up) -- with
// a grid-wide barrier between stages instead of a kernel boundary.
//
// Every warp owns a ring of bulk-copy slots and streams, in program order,
// its share of the weights of every matvec stage of the program: once it has
// consumed a slot it refills it with the next share, which may belong to a
// later stage, so the weights of the next matvec are already in shared memory
// while the row stage and the barriers before it run.  A matvec stage is the
// streaming kernel's loop (q4_stream in k_stream.cu: the CTA stages the
// activation codes of its K-block as exact f16, the products run on f16
// tensor-core MMAs of exact integers, each 64-row group's partial sums are
// added into y atomically); a row stage gives row i to CTA i, the other CTAs
// clear the buffer that a later matvec accumulates into.
//
// Every wait is bounded (1 s of %globaltimer): a barrier or a slot that does
// not complete raises the model's error flag, the CTA drains its copies in
// flight and leaves.
#include "common.cuh"
#include "kernels.cuh"

namespace dflash {

constexpr int kChWarps = 16;
constexpr int kChThreads = kChWarps * 32;
constexpr int kChSC = 4 * kQ4Chunk;              // super-chunk: four 16-row tiles x one k-step
constexpr int kChSlotSC = 2;                     // super-chunks per ring slot (one bulk copy)
constexpr int kChSlots = 2;                      // ring slots per warp
constexpr int kChRing = kChSlots * kChSlotSC * kChSC;
constexpr int kChActPad = 32;                    // halves of row pad of the staged codes
constexpr int kChMaxKbc = 32 * kQ4KStep;         // columns of the widest K-block
constexpr int kChBarBytes = 1024;
constexpr int kChRowNV = kChainRowMax / 4 / kChThreads;  // float4 of a row per thread
constexpr uint64_t kChWait = 1000000000ull;              // ns a wait may take before the kernel gives up
static_assert(kChRowNV * 4 * kChThreads == kChainRowMax, "row split");

constexpr int kChDumpBytes = 512;  // a warp's scratch for the vector reductions of a group
constexpr size_t kChActBytes = (size_t)16 * (kChMaxKbc + kChActPad) * sizeof(__half);
constexpr size_t kChSmem = (size_t)kChBarBytes + (size_t)kChWarps * kChRing + kChActBytes + (size_t)kChWarps * kChDumpBytes;

DF_DEV unsigned ld_acquire_gpu(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
DF_DEV int ld_volatile(const int* p) { return *reinterpret_cast<const volatile int*>(p); }

// codes4 out of line: the row stage calls it for up to 12 float4 a thread,
// and one copy of the IEEE divisions keeps the kernel's code small
__device__ __noinline__ uint32_t ch_codes4(float4 v, float sx) { return codes4(v, sx); }
__device__ __noinline__ float4 ch_silu_mul4(float4 g, float4 u) {
    return make_float4(silu_f(g.x) * u.x, silu_f(g.y) * u.y, silu_f(g.z) * u.z, silu_f(g.w) * u.w);
}

// The share of warp `warp` of this CTA in a matvec stage: the CTA's part of
// its K-block's span (as stream_geom, in 32-bit arithmetic: every count here
// is far below 2^31), then an equal contiguous sixteenth of it.
__device__ __noinline__ void ch_share(Q4Layout L, int g0, int ng, int warp, int& wlo, int& n, StreamGeom& sg) {
    const int nkb = L.ksteps / L.kb;
    const int G = gridDim.x, c = blockIdx.x;
    const int kblk = c * nkb / G;
    const int first = (kblk * G + nkb - 1) / nkb;
    const int nxt = ((kblk + 1) * G + nkb - 1) / nkb;
    const int cnt = nxt - first, lc = c - first;
    const int span = ng * L.kb;
    const int lo = span * lc / cnt, hi = span * (lc + 1) / cnt;
    sg.lo = lo;
    sg.hi = hi;
    sg.base = ((int64_t)kblk * L.ngroups + g0) * L.kb;
    sg.kblk = kblk;
    wlo = lo + (hi - lo) * warp / kChWarps;
    n = lo + (hi - lo) * (warp + 1) / kChWarps - wlo;
}

// Block-wide sum / max over the chain's 16 warps (red: 17 floats).
template <bool kMax>
DF_DEV float ch_reduce(float v, float* red) {
    v = kMax ? warp_max(v) : warp_sum(v);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    if (threadIdx.x < 32) {
        float u = threadIdx.x < kChWarps ? red[threadIdx.x] : 0.f;
        u = kMax ? warp_max(u) : warp_sum(u);
        if (threadIdx.x == 0) red[32] = u;
    }
    __syncthreads();
    const float r = red[32];
    __syncthreads();
    return r;
}

// Grid-wide barrier: every CTA adds one to *bar and waits (bounded) until
// *bar reaches `target`.  The fences on both sides order this CTA's writes
// before the arrival and the others' writes before what follows; the wait
// also ends at once when another CTA has raised the error flag.  Returns
// false (the same in every thread of the CTA) when it gave up.
DF_DEV bool grid_barrier(unsigned* bar, unsigned target, int* err, int* s_flag) {
    __syncthreads();
    if (threadIdx.x == 0) {
        int ok = 1;
        asm volatile("fence.acq_rel.gpu;\n\tred.release.gpu.global.add.u32 [%0], 1;" ::"l"(bar) : "memory");
        if (ld_acquire_gpu(bar) < target) {
            const uint64_t t0 = global_ns();
            while (ld_acquire_gpu(bar) < target) {
                if (ld_volatile(err) != 0 || global_ns() - t0 > kChWait) {
                    ok = 0;
                    atomicExch(err, 1);
                    break;
                }
            }
        }
        asm volatile("fence.acq_rel.gpu;" ::: "memory");
        *s_flag = ok;
    }
    __syncthreads();
    return *s_flag != 0;
}

// Row i of a row stage (NV float4 a thread; the row sits in registers from
// its single read to its codes).
template <int NV>
__device__ __noinline__ void ch_row(const ChainStage& s, int i, float* red) {
    const RowMap map = s.map;
    const int srow = (i / map.per) * map.stride + map.skip + (i % map.per);
    const int n = s.n, n4 = s.n / 4;
    const float* src = s.src + (int64_t)srow * s.ld_src;
    const float* wg = s.w;
    float4 v[NV];
    if (s.op == kChainSilu) {
        // a = silu(g) * u, g and u halves of the source row
        const float4* g4 = reinterpret_cast<const float4*>(src);
        const float4* u4 = reinterpret_cast<const float4*>(src + n);
#pragma unroll
        for (int u = 0; u < NV; ++u) {
            const int c = threadIdx.x + u * kChThreads;
            v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (c < n4) v[u] = ch_silu_mul4(__ldcg(g4 + c), __ldcg(u4 + c));
        }
    } else {
        const float4* x4 = reinterpret_cast<const float4*>(src);
        float ss = 0.f;
#pragma unroll
        for (int u = 0; u < NV; ++u) {
            const int c = threadIdx.x + u * kChThreads;
            v[u] = c < n4 ? __ldcg(x4 + c) : make_float4(0.f, 0.f, 0.f, 0.f);
            ss = fmaf(v[u].x, v[u].x, ss);
            ss = fmaf(v[u].y, v[u].y, ss);
            ss = fmaf(v[u].z, v[u].z, ss);
            ss = fmaf(v[u].w, v[u].w, ss);
        }
        if (wg) {
            ss = ch_reduce<false>(ss, red);
            const float sc = 1.f / sqrtf(ss / (float)n + s.eps);
            const float4* w4 = reinterpret_cast<const float4*>(wg);
#pragma unroll
            for (int u = 0; u < NV; ++u) {
                const int c = threadIdx.x + u * kChThreads;
                if (c < n4) {
                    const float4 g = w4[c];
                    v[u] = make_float4(v[u].x * sc * g.x, v[u].y * sc * g.y, v[u].z * sc * g.z, v[u].w * sc * g.w);
                }
            }
        }
    }
    float amax = 0.f;
#pragma unroll
    for (int u = 0; u < NV; ++u) amax = fmaxf(amax, amax4(v[u]));  // lanes past n hold zeros
    amax = ch_reduce<true>(amax, red);
    const float sx = __fdiv_rn(amax, 127.0f);
    uint32_t* q4 = reinterpret_cast<uint32_t*>(s.codes + (int64_t)i * s.ld_codes);
#pragma unroll
    for (int u = 0; u < NV; ++u) {
        const int c = threadIdx.x + u * kChThreads;
        if (c < n4) q4[c] = ch_codes4(v[u], sx);
    }
    if (threadIdx.x == 0) s.scale[i] = sx;
}

__global__ void __launch_bounds__(kChThreads, 1)
    chain_kernel(const __grid_constant__ ChainProgram prog, unsigned* bar, int* err) {
    extern __shared__ __align__(128) unsigned char sm[];
    __shared__ float red[33];
    __shared__ int s_flag, s_abort;
    // the program, copied once into shared memory: a stage's fields are then
    // plain shared loads (a dynamically indexed kernel parameter would be read
    // through the generic path on every use)
    __shared__ __align__(16) ChainProgram sp;
    {
        static_assert(sizeof(ChainProgram) % 4 == 0, "program copy");
        const int* src = reinterpret_cast<const int*>(&prog);
        int* dst = reinterpret_cast<int*>(&sp);
        for (int i = threadIdx.x; i < (int)(sizeof(ChainProgram) / 4); i += blockDim.x) dst[i] = src[i];
        __syncthreads();
    }
    const int nst = sp.n;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x;
    uint64_t* full = reinterpret_cast<uint64_t*>(sm) + warp * kChSlots;
    unsigned char* ring = sm + kChBarBytes + warp * kChRing;
    __half* act = reinterpret_cast<__half*>(sm + kChBarBytes + kChWarps * kChRing);
    float* dscr = reinterpret_cast<float*>(sm + kChBarBytes + kChWarps * kChRing + kChActBytes) + warp * (kChDumpBytes / 4);

    // this warp's share of a matvec stage: super-chunks [wlo, wlo + n) of the CTA's K-block span
    auto warp_share = [&](const ChainStage& s, int64_t& wlo, int& n, StreamGeom& sg) {
        int w0;
        ch_share(s.L, s.g0, s.ng, warp, w0, n, sg);
        wlo = w0;
    };

    // producer cursor (lane 0): stage ps, its next slot pj of pns, from psrc
    int ps = 0, pj = 0, pns = -1, pnsc = 0, issued = 0;
    const uint8_t* psrc = nullptr;
    auto issue_next = [&]() -> bool {
        if (!(pns >= 0 && pj < pns)) {
            while (ps < nst) {
                const ChainStage& s = sp.s[ps];
                if (s.op == kChainMatvec) {
                    if (pns < 0) {
                        int64_t wlo;
                        StreamGeom sg;
                        warp_share(s, wlo, pnsc, sg);
                        pns = (pnsc + kChSlotSC - 1) / kChSlotSC;
                        pj = 0;
                        psrc = s.wp + (sg.base + wlo) * kChSC;
                    }
                    if (pj < pns) break;
                }
                ++ps;
                pns = -1;
            }
            if (ps >= nst) return false;
        }
        const int slot = issued % kChSlots;
        const uint32_t bytes = (uint32_t)min(kChSlotSC, pnsc - pj * kChSlotSC) * kChSC;
        mbar_arrive_expect_tx(&full[slot], bytes);
        bulk_g2s(ring + slot * (kChSlotSC * kChSC), psrc + (int64_t)pj * (kChSlotSC * kChSC), bytes, &full[slot]);
        ++pj;
        ++issued;
        return true;
    };

    pdl_trigger();
    if (threadIdx.x == 0) s_abort = 0;
    if (lane == 0) {
        for (int i = 0; i < kChSlots; ++i) mbar_init(&full[i], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        // the first weights go out before the previous kernel has finished: they do not depend on it
        for (int i = 0; i < kChSlots; ++i)
            if (!issue_next()) break;
    }
    __syncwarp();
    pdl_wait();
    __syncthreads();

    const int gq = lane >> 2, tq = lane & 3;
    int cons = 0;  // slots this warp has consumed

    // ---- one matvec stage; false when a slot wait gave up (warp-uniform)
    auto matvec = [&](const ChainStage& s) -> bool {
        int64_t wlo;
        int n;
        StreamGeom sg;
        warp_share(s, wlo, n, sg);
        const int T = s.T, ldx = s.ldx, ldy = s.ldy, kb = s.L.kb;
        const int8_t* xc = s.xc;
        const float* xsp = s.xs;
        float* y = s.y;
        const int kbc = kb * kQ4KStep, ldact = kbc + kChActPad;
        {
            // the K-block's codes of the 16 rows as exact f16 (rows past T are zero)
            const int vec = kbc / 8, total = 16 * vec;
            constexpr int kBatch = 8;
            for (int base = threadIdx.x; base < total; base += kBatch * kChThreads) {
                uint2 v[kBatch];
#pragma unroll
                for (int u = 0; u < kBatch; ++u) {
                    const int i = base + u * kChThreads, r = i / vec, c = i - r * vec;
                    v[u] = make_uint2(0u, 0u);
                    if (i < total && r < T)
                        v[u] = __ldcg(reinterpret_cast<const uint2*>(xc + (int64_t)r * ldx + sg.kblk * kbc + c * 8));
                }
#pragma unroll
                for (int u = 0; u < kBatch; ++u) {
                    const int i = base + u * kChThreads, r = i / vec, c = i - r * vec;
                    if (i < total) {
                        uint4 h;
                        i8x4_to_half2x2(v[u].x, h.x, h.y);
                        i8x4_to_half2x2(v[u].y, h.z, h.w);
                        *reinterpret_cast<uint4*>(act + r * ldact + c * 8) = h;
                    }
                }
            }
            __syncthreads();
        }
        const __half* a_lo = act + gq * ldact + 8 * tq;
        const __half* a_hi = act + (gq + 8) * ldact + 8 * tq;
        float xs[2][2];
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int t = h * 8 + 2 * tq + e;
                xs[h][e] = t < T ? __ldcg(xsp + t) : 0.f;
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
        // one super-chunk: k-step ks of the current group
        auto sc_step = [&](const unsigned char* scp, int ks) {
            uint4 bq[2][2];
#pragma unroll
            for (int gi = 0; gi < 2; ++gi) {
                bq[gi][0] = *reinterpret_cast<const uint4*>(a_lo + ks * kQ4KStep + gi * 32);
                bq[gi][1] = *reinterpret_cast<const uint4*>(a_hi + ks * kQ4KStep + gi * 32);
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const uint4 wv = *reinterpret_cast<const uint4*>(scp + r * kQ4Chunk + lane * 16);
                const uint2 sv = *reinterpret_cast<const uint2*>(scp + r * kQ4Chunk + 512 + gq * 8);
                const uint32_t wds[4] = {wv.x, wv.y, wv.z, wv.w};
                const uint32_t svs[2] = {sv.x, sv.y};
#pragma unroll
                for (int gi = 0; gi < 2; ++gi) {
                    uint32_t a0[4], a1[4];
                    unpack_q4_word(wds[gi * 2 + 0], a0);
                    unpack_q4_word(wds[gi * 2 + 1], a1);
                    float d0[4], d1[4];
                    mma_f16_16816(d0, a0, bq[gi][0].x, bq[gi][0].y, zero);
                    mma_f16_16816(d0, a1, bq[gi][0].z, bq[gi][0].w, d0);
                    mma_f16_16816(d1, a0, bq[gi][1].x, bq[gi][1].y, zero);
                    mma_f16_16816(d1, a1, bq[gi][1].z, bq[gi][1].w, d1);
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

        // one flat loop over the warp's super-chunks (one copy of the step and
        // of the dump: the kernel's code stays small enough for the
        // instruction caches); k == n flushes the last group
        int ks = (int)(wlo % kb), grp = (int)(wlo / kb), cur = grp;
        const unsigned char* sb = ring;
#pragma unroll 1
        for (int k = 0; k <= n; ++k) {
            if (k == n || grp != cur) {
                if (k > 0) dump(cur);
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int e = 0; e < 4; ++e) acc[r][h][e] = 0.f;
                cur = grp;
                if (k == n) break;
            }
            const int u = k % kChSlotSC;
            if (u == 0) {
                const int slot = cons % kChSlots;
                const bool okw = __all_sync(0xffffffffu, mbar_wait(&full[slot], (cons / kChSlots) & 1, kChWait));
                if (!okw) return false;
                sb = ring + slot * (kChSlotSC * kChSC);
            }
            sc_step(sb + u * kChSC, ks);
            if (++ks == kb) {
                ks = 0;
                ++grp;
            }
            if (u == kChSlotSC - 1 || k == n - 1) {
                ++cons;
                // every lane has read the slot: refill it with the next share in program order
                __syncwarp();
                if (lane == 0) {
                    fence_proxy_async_smem();
                    issue_next();
                }
            }
        }
        return true;
    };

    // ---- a row stage: CTA i < rows takes row i, the others clear s.zero
    auto rows_stage = [&](const ChainStage& s) {
        const int i = blockIdx.x;
        const int rows = s.rows;
        if (i >= rows) {
            float* zero = s.zero;
            const int64_t zn = s.zero_n;
            if (zero && zn > 0) {
                const int64_t stride = (int64_t)(G - rows) * kChThreads;
                const int64_t first = (int64_t)(i - rows) * kChThreads + threadIdx.x;
                float4* z4 = reinterpret_cast<float4*>(zero);
                for (int64_t k = first; k < zn / 4; k += stride) z4[k] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (first < zn % 4) zero[zn / 4 * 4 + first] = 0.f;
            }
            return;
        }
        // the row's float4 per thread, rounded up to the variants below
        const int nv = (s.n / 4 + kChThreads - 1) / kChThreads;
        if (nv <= 2)
            ch_row<2>(s, i, red);
        else if (nv <= 6)
            ch_row<6>(s, i, red);
        else
            ch_row<kChRowNV>(s, i, red);
    };

    int nbar = 0;
    for (int si = 0; si < nst; ++si) {
        const ChainStage& s = sp.s[si];
        bool wok = true;
        if (s.op == kChainMatvec)
            wok = matvec(s);
        else
            rows_stage(s);
        if (!wok && lane == 0) {
            atomicExch(err, 1);
            s_abort = 1;
        }
        if (si + 1 < nst) {
            ++nbar;
            if (!grid_barrier(bar, (unsigned)(nbar * G), err, &s_flag)) s_abort = 1;
        }
        __syncthreads();
        if (s_abort) break;
    }
    if (s_abort) {
        // let no copy still land in this CTA's memory after it exits
        if (lane == 0)
            for (int k = cons; k < issued; ++k) mbar_wait(&full[k % kChSlots], (k / kChSlots) & 1, kChWait);
        return;
    }
    // the last CTA out returns the counter to zero for the next launch
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned v = atomicAdd(bar, 1u);
        if (v == (unsigned)((nbar + 1) * G - 1)) atomicExch(bar, 0u);
    }
}

int chain_run(const ChainProgram& p, int num_sms, unsigned* bar, int* err, cudaStream_t st) {
    if (p.n < 1 || p.n > kChainMaxStages || num_sms < 16) return (int)cudaErrorInvalidValue;
    auto al16 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15) == 0; };
    for (int i = 0; i < p.n; ++i) {
        const ChainStage& s = p.s[i];
        if (s.op == kChainMatvec) {
            if (s.T < 1 || s.T > 16 || s.L.kb * kQ4KStep > kChMaxKbc || s.L.ksteps / s.L.kb > num_sms ||
                s.ldy % 4 || (reinterpret_cast<uintptr_t>(s.y) & 15) ||
                s.g0 < 0 || s.ng < 1 || s.g0 + s.ng > s.L.ngroups || s.ldx % 8 || !s.wp || !s.xc || !s.xs || !s.y)
                return (int)cudaErrorInvalidValue;
        } else if (s.op == kChainRows || s.op == kChainSilu) {
            if (s.rows < 1 || s.rows >= num_sms || s.n % 4 || s.n > kChainRowMax || s.ld_src % 4 || !al16(s.src) ||
                (s.w && !al16(s.w)) || s.ld_codes % 4 || !s.codes || !s.scale ||
                (s.zero && s.zero_n > 0 && !al16(s.zero)) || (s.op == kChainSilu && (s.w || s.n % 4)))
                return (int)cudaErrorInvalidValue;
        } else {
            return (int)cudaErrorInvalidValue;
        }
    }
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kChSmem);
        if (e != cudaSuccess) return (int)e;
        attr = true;
    }
    return (int)launch(chain_kernel, dim3(num_sms), dim3(kChThreads), kChSmem, st, p, bar, err);
}

}  // namespace dflash
