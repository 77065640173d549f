// tcgen05 and TMA building blocks shared by the tensor-core kernels: shared-
// memory matrix descriptors, tensor-memory loads, the bulk tensor copies
// between global and shared memory, and the host-side tensor maps of the
// operands (cuTensorMapEncodeTiled, reached through the runtime's driver
// entry point so that the library links against the runtime alone).
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>

#include "common.cuh"

namespace dflash {

// Shared-memory matrix descriptor: a K-major tile with 128-byte rows in the
// 128-byte swizzle (eight-row atoms of 1024 bytes, stride 1024 bytes between
// atoms), base 1024-aligned; the k16 slice j starts 32 j bytes into the rows.
DF_DEV uint64_t tc_desc_sw128(uint32_t saddr) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
DF_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
DF_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 16 consecutive f32 columns of this thread's tensor-memory lane (whole warp)
DF_DEV void tc_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
DF_DEV void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// a box of a tensor map fetched into L2 only (no shared memory, no barrier)
DF_DEV void tma_prefetch_2d(const CUtensorMap* map, int x, int y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(map), "r"(x), "r"(y)
                 : "memory");
}
// global -> this CTA's shared memory, completion counted on `bar`
DF_DEV void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_addr(dst)),
        "l"(map), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}
// shared -> global through a tensor map (elements outside the map's extents
// are not written): a plain store, or an f32 add into what is there
DF_DEV void tma_store_2d(const CUtensorMap* map, const void* src, int x, int y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(map), "r"(x),
                 "r"(y), "r"(smem_addr(src))
                 : "memory");
}
DF_DEV void tma_reduce_add_2d(const CUtensorMap* map, const void* src, int x, int y) {
    asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(map),
                 "r"(x), "r"(y), "r"(smem_addr(src))
                 : "memory");
}
DF_DEV void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// the issuing thread's bulk groups: at most N still reading shared memory / none outstanding
template <int N>
DF_DEV void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
DF_DEV void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// ---- host: tensor maps (k_tc.cu)
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_fn();  // nullptr where the driver has no entry point for it
// f16 codes [T][K] (activations) or [N][K] (a dense weight copy): 64-column x
// box_rows boxes in the 128-byte swizzle, rows past the extent read as zeros
bool act_map(CUtensorMap* map, const __half* codes, int K, int T, int box_rows);
bool dense_map(CUtensorMap* map, const __half* w, int K, int N, int box_rows);
// an f32 output [T][ldy] as a map of its first N columns: 32 x 32 boxes in the
// 128-byte swizzle; false where the rows are not 16-byte multiples or the base
// is not 16-aligned
bool out_map(CUtensorMap* map, float* y, int ldy, int N, int T);

}  // namespace dflash
