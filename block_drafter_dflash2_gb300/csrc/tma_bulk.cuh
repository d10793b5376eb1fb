// Inline-PTX copy-engine helpers beyond the tiled 2-D load of ptx.cuh: the L2 prefetch of a
// 2-D box, the 3-D tiled load and store, and the bulk async-group that tracks stores.
#pragma once

#include "ptx.cuh"

namespace df {

// Requests the 2-D box at (c0, c1) of `map` into L2 (no shared memory, no completion).
DF_DEV void tma_prefetch_2d(const CUtensorMap* map, int32_t c0, int32_t c1) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1)
               : "memory");
}

// The 3-D box at (c0, c1, c2) of `map` into shared memory (128-byte aligned), completing on
// `bar`; elements outside the tensor read as zero.
DF_DEV void tma_load_3d(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int32_t c0, int32_t c1, int32_t c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(
          smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// A 3-D box of shared memory (128-byte aligned) to (c0, c1, c2) of `map`; elements outside the
// tensor are not written. Tracked by the issuing thread's bulk async-group.
DF_DEV void tma_store_3d(const CUtensorMap* map, const void* smem_src, int32_t c0, int32_t c1, int32_t c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(smem_src)), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}

DF_DEV void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Waits until every bulk async-group the thread committed has completed: its shared memory is
// read and its global writes are performed.
DF_DEV void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

}  // namespace df
