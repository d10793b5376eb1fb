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

// Inverse of order_key.
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// One warp merges `parts` sorted lists of 16 (sv/si: [parts][16] in shared memory, head:
// [parts] zeroed) into the K best (logit desc, id asc); lane k < K receives the k-th in
// (out_id, out_v) with out_ok set. Lane l owns the lists p = l (mod 32) and keeps its best head.
// A round is a redux.sync max over the order keys of the lanes' heads and, only when several
// lanes hold that key, a redux.sync min over their ids (ids are unique across lists); the lowest
// such lane wins, and every lane learns the round's value from the key and its id by a shuffle.
// Up to kMergeCache lists per lane the heads are kept in registers as 64-bit keys
// (order key << 32 | ~id: larger is better, 0 = list exhausted), every lane runs the same
// branch-free advance and tree pick (only the winner's state changes), so a round reads shared
// memory once; beyond that the winner rescans its lists' heads in shared memory.
constexpr int kMergeCache = 8;

__device__ __forceinline__ uint64_t entry_key(float v, int32_t id) {
  return ((uint64_t)order_key(v) << 32) | (uint32_t)(~id);
}

__device__ __forceinline__ void warp_merge_lists(const float* sv, const int32_t* si, uint8_t* head, int parts, int K,
                                                 int32_t& out_id, float& out_v, bool& out_ok) {
  const int lane = threadIdx.x & 31;
  out_ok = false;
  out_id = 0;
  out_v = -INFINITY;
  if (parts <= 32 * kMergeCache) {
    uint64_t hk[kMergeCache];  // head key of list lane + 32 m (0: none left)
    int hh[kMergeCache];       // its position in the list
#pragma unroll
    for (int m = 0; m < kMergeCache; ++m) {
      const int p = lane + 32 * m;
      const bool has = p < parts;
      hh[m] = 0;
      const float v0 = sv[has ? p * 16 : 0];
      const int32_t i0 = si[has ? p * 16 : 0];
      hk[m] = has ? entry_key(v0, i0) : 0ull;
    }
    uint64_t best = 0;
    int bm = 0;
    auto pick = [&]() {  // the largest key; the lower list on equal keys
      uint64_t k[kMergeCache];
      int mi[kMergeCache];
#pragma unroll
      for (int m = 0; m < kMergeCache; ++m) {
        k[m] = hk[m];
        mi[m] = m;
      }
#pragma unroll
      for (int w = 1; w < kMergeCache; w *= 2) {
#pragma unroll
        for (int a = 0; a < kMergeCache; a += 2 * w) {
          const bool gt = k[a + w] > k[a];
          k[a] = gt ? k[a + w] : k[a];
          mi[a] = gt ? mi[a + w] : mi[a];
        }
      }
      best = k[0];
      bm = mi[0];
    };
    pick();
    for (int k = 0; k < K; ++k) {
      const uint32_t key = (uint32_t)(best >> 32);
      const uint32_t kmax = __reduce_max_sync(0xffffffffu, key);
      const bool tied = key == kmax && best != 0ull;
      const uint32_t bid = ~(uint32_t)best;
      uint32_t win = __ballot_sync(0xffffffffu, tied);
      if (__popc(win) > 1) {  // (warp-uniform) equal values: the lowest id, then the lowest lane
        const uint32_t wid = __reduce_min_sync(0xffffffffu, tied ? bid : 0xffffffffu);
        win = __ballot_sync(0xffffffffu, tied && bid == wid);
      }
      const int wl = win ? __ffs(win) - 1 : 0;
      const uint32_t wid = __shfl_sync(0xffffffffu, bid, wl);
      if (win != 0u && lane == k) {
        out_id = (int32_t)wid;
        out_v = key_value(kmax);
        out_ok = true;
      }
      // the winner advances its list; every lane runs the same instructions
      const bool me = win != 0u && lane == wl;
      int h = 0;
#pragma unroll
      for (int m = 0; m < kMergeCache; ++m) h = (m == bm) ? hh[m] + 1 : h;
      const bool more = me && h < 16;
      const int p = lane + 32 * bm;
      const float nv = sv[more ? p * 16 + h : 0];
      const int32_t ni = si[more ? p * 16 + h : 0];
      const uint64_t nk = more ? entry_key(nv, ni) : 0ull;
#pragma unroll
      for (int m = 0; m < kMergeCache; ++m) {
        const bool upd = me && m == bm;
        hh[m] = upd ? h : hh[m];
        hk[m] = upd ? nk : hk[m];
      }
      pick();
    }
  } else {
    float bv = -INFINITY;
    int32_t bid = 0x7fffffff;
    int bp = -1;  // the lane's best list (-1: none left)
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
      if (win != 0u && lane == k) {
        out_id = (int32_t)wid;
        out_v = key_value(kmax);
        out_ok = true;
      }
      if (lane == __ffs(win) - 1) {
        head[bp] += 1;
        rescan();
      }
      __syncwarp();
    }
  }
}

}  // namespace df
