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
// and keeps its best head; a round is a redux.sync max over the order key, a redux.sync min
// over the ids of the lanes holding that key (ids are unique across lists), and a ballot for
// the lowest such lane, which emits its head and advances that list. emit(k, id, logit) is
// called by the winning lane. Up to kMergeCache lists per lane (32 * kMergeCache partitions)
// the heads live in registers, so a round reads shared memory once (the winner's next entry);
// beyond that the winner rescans its lists' heads in shared memory.
constexpr int kMergeCache = 8;

template <class Emit>
__device__ __forceinline__ void warp_merge_lists(const float* sv, const int32_t* si, uint8_t* head, int parts,
                                                 int K, Emit emit) {
  const int lane = threadIdx.x & 31;
  float bv = -INFINITY;
  int32_t bid = 0x7fffffff;
  int bp = -1;  // the lane's best list (-1: none left)
  auto round = [&](auto&& advance) {
    for (int k = 0; k < K; ++k) {
      const uint32_t key = bp >= 0 ? order_key(bv) : 0u;
      const uint32_t kmax = __reduce_max_sync(0xffffffffu, key);
      const bool tied = key == kmax && bp >= 0;
      const uint32_t wid = __reduce_min_sync(0xffffffffu, tied ? (uint32_t)bid : 0xffffffffu);
      const uint32_t win = __ballot_sync(0xffffffffu, tied && (uint32_t)bid == wid);
      if (lane == __ffs(win) - 1) {
        emit(k, bid, bv);
        advance();
      }
      __syncwarp();
    }
  };
  if (parts <= 32 * kMergeCache) {
    // heads in registers: hv/hid the head entry of list lane + 32 m, hh its position (16: none)
    float hv[kMergeCache];
    int32_t hid[kMergeCache];
    int hh[kMergeCache];
#pragma unroll
    for (int m = 0; m < kMergeCache; ++m) {
      const int p = lane + 32 * m;
      const bool has = p < parts;
      hh[m] = has ? 0 : 16;
      hv[m] = has ? sv[p * 16] : -INFINITY;
      hid[m] = has ? si[p * 16] : 0x7fffffff;
    }
    auto pick = [&]() {  // the best head over the lane's lists, in list order (as a rescan would)
      bv = -INFINITY;
      bid = 0x7fffffff;
      bp = -1;
#pragma unroll
      for (int m = 0; m < kMergeCache; ++m) {
        if (hh[m] < 16 && (bp < 0 || better(hv[m], hid[m], bv, bid))) {
          bv = hv[m];
          bid = hid[m];
          bp = m;
        }
      }
    };
    pick();
    round([&]() {
#pragma unroll
      for (int m = 0; m < kMergeCache; ++m) {
        if (m == bp) {  // (a register array indexed by a constant)
          const int p = lane + 32 * m;
          const int h = ++hh[m];
          if (h < 16) {
            hv[m] = sv[p * 16 + h];
            hid[m] = si[p * 16 + h];
          }
        }
      }
      pick();
    });
  } else {
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
    round([&]() {
      head[bp] += 1;
      rescan();
    });
  }
}

}  // namespace df
