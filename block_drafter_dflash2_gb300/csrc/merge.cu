// Cross-partition merge: each column partition of the LM-head GEMM left, per row, its
// top-16 (logit desc, id asc) and its (max, sum of exp(l - max)). One warp per row merges
// them: lse = M + log(sum_p s_p * exp(m_p - M)), then K rounds of a warp-wide arg-max over
// the heads of the sorted partition lists (ties to the lower id).
#include <math.h>

#include "kernels.h"

namespace df {

namespace {
constexpr int kRowsPerBlock = 4;
constexpr int kMaxParts = 1024;

__device__ __forceinline__ bool better(float v, int32_t id, float bv, int32_t bid) {
  return v > bv || (v == bv && id < bid);
}

__global__ void __launch_bounds__(32 * kRowsPerBlock)
    topk_merge_kernel(const float* __restrict__ part_val, const int32_t* __restrict__ part_id,
                      const float2* __restrict__ part_ms, int parts, int M, int K, int32_t* __restrict__ cand_ids,
                      float* __restrict__ cand_lp, float* __restrict__ lse_out) {
  __shared__ uint8_t head[kRowsPerBlock][kMaxParts];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * kRowsPerBlock + warp;
  if (row >= M) return;  // warp-uniform
  for (int p = lane; p < parts; p += 32) head[warp][p] = 0;

  float m = -INFINITY;
  for (int p = lane; p < parts; p += 32) m = fmaxf(m, part_ms[(size_t)p * M + row].x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float s = 0.f;
  for (int p = lane; p < parts; p += 32) {
    const float2 ms = part_ms[(size_t)p * M + row];
    if (ms.y > 0.f) s += ms.y * expf(ms.x - m);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  const float lse = m + logf(s);
  if (lane == 0 && lse_out) lse_out[row] = lse;
  __syncwarp();

  for (int k = 0; k < K; ++k) {
    float bv = -INFINITY;
    int32_t bid = 0x7fffffff;
    int bp = -1;
    for (int p = lane; p < parts; p += 32) {
      const int h = head[warp][p];
      if (h < 16) {
        const size_t at = ((size_t)p * M + row) * 16 + h;
        const float v = part_val[at];
        const int32_t id = part_id[at];
        if (bp < 0 || better(v, id, bv, bid)) {
          bv = v;
          bid = id;
          bp = p;
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int32_t oid = __shfl_xor_sync(0xffffffffu, bid, o);
      const int op = __shfl_xor_sync(0xffffffffu, bp, o);
      if (op >= 0 && (bp < 0 || better(ov, oid, bv, bid))) {
        bv = ov;
        bid = oid;
        bp = op;
      }
    }
    if (bp >= 0 && lane == (bp & 31)) head[warp][bp] += 1;
    if (lane == 0) {
      cand_ids[(size_t)row * K + k] = bid;
      cand_lp[(size_t)row * K + k] = bv - lse;
    }
    __syncwarp();
  }
}
}  // namespace

cudaError_t launch_topk_merge(const float* part_val, const int32_t* part_id, const float* part_ms, int parts,
                              int M, int K, int32_t* cand_ids, float* cand_lp, float* lse, cudaStream_t s) {
  if (parts > kMaxParts) return cudaErrorInvalidValue;
  const int grid = (M + kRowsPerBlock - 1) / kRowsPerBlock;
  topk_merge_kernel<<<grid, 32 * kRowsPerBlock, 0, s>>>(part_val, part_id, reinterpret_cast<const float2*>(part_ms),
                                                        parts, M, K, cand_ids, cand_lp, lse);
  return cudaGetLastError();
}

}  // namespace df
