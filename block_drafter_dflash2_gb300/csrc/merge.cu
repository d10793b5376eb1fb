// Cross-partition merge: each column partition of the LM-head contraction left, per row, its
// top-16 (logit desc, id asc) and its (max, sum of exp(l - max)). One CTA per row stages the
// row's partials in shared memory with one batch of 16-byte loads, reduces
// lse = M + log(sum_p s_p * exp(m_p - M)) across the block, and warp 0 then takes K rounds of
// a warp-wide arg-max over the heads of the sorted partition lists (ties to the lower id).
// Each lane owns the lists p = lane (mod 32) and caches its best head; a round is one
// redux.sync max over an order-preserving key of the logit, a ballot of the lanes holding it
// and a redux.sync min over their ids; then only the winning lane rescans its own lists.
// The partials are staged with cp.async so every load of a row is in flight at once.
#include <math.h>

#include "kernels.h"
#include "launch_util.h"
#include "select.cuh"

namespace df {

namespace {
constexpr int kThreads = 128;
constexpr int kMaxParts = 1024;

__global__ void __launch_bounds__(kThreads)
    topk_merge_kernel(const float4* __restrict__ part_val, const int4* __restrict__ part_id,
                      const float2* __restrict__ part_ms, int parts, int M, int K, int32_t* __restrict__ cand_ids,
                      float* __restrict__ cand_lp, float* __restrict__ lse_out) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  float* sv = reinterpret_cast<float*>(smem_raw);              // [parts][16]
  int32_t* si = reinterpret_cast<int32_t*>(sv + parts * 16);   // [parts][16]
  uint8_t* head = reinterpret_cast<uint8_t*>(si + parts * 16);  // [parts]
  __shared__ float red_m[kThreads / 32], red_s[kThreads / 32];
  __shared__ float lse_s;
  const int row = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  for (int e = tid; e < parts * 4; e += kThreads) {
    const int p = e >> 2, q = e & 3;
    const size_t src = ((size_t)p * M + row) * 4 + q;
    cp_async16(reinterpret_cast<float4*>(sv) + e, part_val + src);
    cp_async16(reinterpret_cast<int4*>(si) + e, part_id + src);
  }
  cp_async_commit();
  for (int p = tid; p < parts; p += kThreads) head[p] = 0;

  float m = -INFINITY;
  for (int p = tid; p < parts; p += kThreads) m = fmaxf(m, part_ms[(size_t)p * M + row].x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) red_m[warp] = m;
  __syncthreads();
  m = red_m[0];
#pragma unroll
  for (int w = 1; w < kThreads / 32; ++w) m = fmaxf(m, red_m[w]);
  float s = 0.f;
  for (int p = tid; p < parts; p += kThreads) {
    const float2 ms = part_ms[(size_t)p * M + row];
    if (ms.y > 0.f) s += ms.y * expf(ms.x - m);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) red_s[warp] = s;
  __syncthreads();
  if (tid == 0) {
    float t = 0.f;
    for (int w = 0; w < kThreads / 32; ++w) t += red_s[w];
    lse_s = m + logf(t);
    if (lse_out) lse_out[row] = lse_s;
  }
  cp_async_wait_all();
  __syncthreads();
  if (warp != 0) return;
  const float lse = lse_s;

  int32_t id;
  float v;
  bool ok;
  warp_merge_lists(sv, si, head, parts, K, id, v, ok);
  const int k = threadIdx.x & 31;
  if (ok) {
    cand_ids[(size_t)row * K + k] = id;
    cand_lp[(size_t)row * K + k] = v - lse;
  }
}
}  // namespace

cudaError_t launch_topk_merge(const float* part_val, const int32_t* part_id, const float* part_ms, int parts,
                              int M, int K, int32_t* cand_ids, float* cand_lp, float* lse, cudaStream_t s) {
  if (parts > kMaxParts) return cudaErrorInvalidValue;
  const size_t smem = (size_t)parts * 16 * 8 + parts;
  if (smem > 48 * 1024) {
    static unsigned char smem_done[64];
    cudaError_t e = smem_opt_in(reinterpret_cast<const void*>(topk_merge_kernel), smem_done);
    if (e != cudaSuccess) return e;
  }
  topk_merge_kernel<<<M, kThreads, smem, s>>>(reinterpret_cast<const float4*>(part_val),
                                               reinterpret_cast<const int4*>(part_id),
                                               reinterpret_cast<const float2*>(part_ms), parts, M, K, cand_ids,
                                               cand_lp, lse);
  return cudaGetLastError();
}

}  // namespace df
