// Device pieces shared by the merge and the walk kernels: the order-preserving key, 16-byte
// async copies, and the warp-wide K-round merge of per-partition sorted top-16 lists.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace df {

__device__ __forceinline__ bool better(float v, int32_t id, float bv, int32_t bid) {
  return v > bv || (v == bv && id < bid);
}

// Unsigned key with the same order as the float (negative values reversed).
__device__ __forceinline__ uint32_t order_key(float v) {
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst))),
               "l"(gmem_src)
               : "memory");
}

__device__ __forceinline__ void cp_async8(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst))),
               "l"(gmem_src)
               : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// One warp merges `parts` sorted lists of 16 (sv/si: [parts][16] in shared memory, head:
// [parts] zeroed) into the K best (logit desc, id asc). Lane l owns the lists p = l (mod 32)
// and caches its best head; a round is a redux.sync max over the order key, a redux.sync min
// over the ids of the lanes holding that key (ids are unique across lists), and a rescan by
// the winning lane only. emit(k, id, logit) is called by the winning lane.
template <class Emit>
__device__ __forceinline__ void warp_merge_lists(const float* sv, const int32_t* si, uint8_t* head, int parts,
                                                 int K, Emit emit) {
  const int lane = threadIdx.x & 31;
  float bv = -INFINITY;
  int32_t bid = 0x7fffffff;
  int bp = -1;
  auto rescan = [&]() {
    bv = -INFINITY;
    bid = 0x7fffffff;
    bp = -1;
    for (int p = lane; p < parts; p += 32) {
      const int h = head[p];
      if (h < 16) {
        const float v = sv[p * 16 + h];
        const int32_t id = si[p * 16 + h];
        if (bp < 0 || better(v, id, bv, bid)) {
          bv = v;
          bid = id;
          bp = p;
        }
      }
    }
  };
  rescan();
  for (int k = 0; k < K; ++k) {
    const uint32_t key = bp >= 0 ? order_key(bv) : 0u;
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, key);
    const bool tied = key == kmax && bp >= 0;
    const uint32_t wid = __reduce_min_sync(0xffffffffu, tied ? (uint32_t)bid : 0xffffffffu);
    const uint32_t win = __ballot_sync(0xffffffffu, tied && (uint32_t)bid == wid);
    if (lane == __ffs(win) - 1) {
      emit(k, bid, bv);
      head[bp] += 1;
      rescan();
    }
    __syncwarp();
  }
}

}  // namespace df
