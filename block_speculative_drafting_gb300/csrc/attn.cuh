// Device helpers shared by the attention kernels (warp-MMA and tcgen05
// forms) and the context append: the (hi, lo) f16 split of f32 values, the
// per-head RMSNorm and half-split rotation of a row spread over a warp's
// lanes, and 16-byte cp.async copies.
#pragma once

#include "common.cuh"

namespace dflash {

// f32 -> (hi, lo) f16 pair with hi + lo = x to about 2^-22 relative (the form
// the attention's tensor-core products take their operands in)
DF_DEV void split_f16(float x, __half& hi, __half& lo) {
    hi = __float2half_rn(x);
    lo = __float2half_rn(x - __half2float(hi));
}

DF_DEV void cp_async16(void* dst_smem, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst_smem)), "l"(src) : "memory");
}
DF_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
DF_DEV void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
DF_DEV void cp_async_wait_one() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

DF_DEV uint32_t pack_half2(__half a, __half b) {
    __half2 h = __halves2half2(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

// four consecutive f32 values as hi/lo f16 halves, one 8-byte store each
DF_DEV void split_store4(float4 v, __half* hi, __half* lo) {
    __half h0, l0, h1, l1, h2, l2, h3, l3;
    split_f16(v.x, h0, l0);
    split_f16(v.y, h1, l1);
    split_f16(v.z, h2, l2);
    split_f16(v.w, h3, l3);
    *reinterpret_cast<uint2*>(hi) = make_uint2(pack_half2(h0, h1), pack_half2(h2, h3));
    *reinterpret_cast<uint2*>(lo) = make_uint2(pack_half2(l0, l1), pack_half2(l2, l3));
}

// Per-head RMSNorm and half-split rotation of a row held as float4 by HD/4
// consecutive lanes (lane d4 holds dims 4 d4 .. 4 d4 + 3; the partner dims
// i +- HD/2 sit at lane d4 ^ HD/8).  Every lane runs the shuffles; the result
// replaces v where `apply`.  g: the gains of the lane's dims; t01 / t23: the
// (cos, sin) pairs of its frequencies i0 .. i0 + 3, i0 = 4 d4 mod HD/2
// (loaded by the caller, ahead of time).  rot false (a layer without the
// rotary position; the same for every thread): the norm alone.
template <int HD>
DF_DEV void norm_rope4(float4& v, bool apply, float4 g, float4 t01, float4 t23, int d4, float eps, bool rot = true) {
    constexpr int D4 = HD / 4;
    float ss = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, v.w * v.w)));
#pragma unroll
    for (int o = D4 / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float s = 1.0f / sqrtf(ss / (float)HD + eps);
    const float4 n = make_float4(v.x * s * g.x, v.y * s * g.y, v.z * s * g.z, v.w * s * g.w);
    if (!rot) {
        if (apply) v = n;
        return;
    }
    float4 pn;  // the partner lane's normed dims
    pn.x = __shfl_xor_sync(0xffffffffu, n.x, D4 / 2);
    pn.y = __shfl_xor_sync(0xffffffffu, n.y, D4 / 2);
    pn.z = __shfl_xor_sync(0xffffffffu, n.z, D4 / 2);
    pn.w = __shfl_xor_sync(0xffffffffu, n.w, D4 / 2);
    const bool lo_half = d4 < D4 / 2;
    const float cs[4] = {t01.x, t01.z, t23.x, t23.z}, sn[4] = {t01.y, t01.w, t23.y, t23.w};
    const float me[4] = {n.x, n.y, n.z, n.w}, other[4] = {pn.x, pn.y, pn.z, pn.w};
    float r[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        // lo' = lo cos - hi sin; hi' = hi cos + lo sin
        r[c] = lo_half ? me[c] * cs[c] - other[c] * sn[c] : me[c] * cs[c] + other[c] * sn[c];
    }
    if (apply) v = make_float4(r[0], r[1], r[2], r[3]);
}

// the (cos, sin) pairs a lane needs for row `row` of the rotation table
template <int HD>
DF_DEV void rope_pairs(const float2* __restrict__ rope, int64_t row, int d4, float4& t01, float4& t23) {
    const float4* t = reinterpret_cast<const float4*>(rope + row * (HD / 2) + (4 * d4) % (HD / 2));
    t01 = t[0];
    t23 = t[1];
}

}  // namespace dflash
