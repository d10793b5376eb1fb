// All conv layers in one cooperative launch, for a small number of rows (M <= 64, bf16).
//
// Each CTA owns a contiguous range of channel groups [g0, g1) for every layer (2-4 groups at
// the page shape: 320 groups over the SMs), i.e. projection rows 2*g0 .. 2*g1 of each layer's
// weight, which are contiguous in memory. Per layer:
//   1. taps: P[m][q] = x[m] . W[2*g0 + q] for every row m and the CTA's taps q. Each thread
//      takes 16-byte chunks of the hidden dimension (x from L2 with .cg loads, which skip the
//      non-coherent L1 since the buffers are rewritten between layers; the weight
//      slice from shared memory) and accumulates 8 rows x kTaps partial dot products; a
//      reduce-scatter across the warp (each step halves the values a lane keeps) and a sum over
//      the 8 warps in shared memory finish them;
//   2. mix: (a, b) = softmax(P[m][2j], P[m][2j+1]) (raw taps on request), and
//      y[m][c] = a * x[m-1][c] + b * x[m][c] for the group's 16 channels, x[-1] = 0 at each
//      block start, rounded to bf16 and written to the layer's output buffer;
//   3. a grid barrier (every CTA needs every channel of the next layer's input).
// The weight slices are double-buffered in shared memory by bulk async copies: layer l+2's
// slice is requested as soon as layer l's taps are done, so weight latency hides behind the
// mix and the barrier. The barrier is an atomic counter in the workspace (zeroed by the
// host before the launch) with a bounded spin: on timeout the kernel sets
// DFLASH2_DEVERR_WAIT_TIMEOUT and stops.
#include <cuda_bf16.h>
#include <math.h>

#include "../../include/dflash2.h"
#include "kernels.h"
#include "ptx.cuh"

namespace df {

namespace {
constexpr int kThreads = 256;
constexpr int kTaps = 8;    // taps per CTA at most (4 groups)
constexpr int kRowBlk = 8;  // rows per accumulation block
constexpr int kVals = kRowBlk * kTaps;  // partial sums per thread: 64 = 2 per lane after the scatter

DF_DEV void bulk_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(smem_dst)),
               "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

DF_DEV uint32_t ld_acquire(const unsigned* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Grid barrier number `round` (1, 2, ...): every CTA adds one, then waits for round * grid.
DF_DEV bool grid_barrier(unsigned* count, unsigned round, int32_t* err, volatile int* stop) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(count, 1u);
    const unsigned target = round * gridDim.x;
    const uint64_t t0 = globaltimer_ns();
    while (ld_acquire(count) < target) {
      __nanosleep(64);
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        flag_error(err, DFLASH2_DEVERR_WAIT_TIMEOUT);
        *stop = 1;
        break;
      }
    }
    __threadfence();
  }
  __syncthreads();
  return *stop == 0;
}

// accumulate acc += x . w over 8 bf16 pairs
DF_DEV float dot8(const uint4& a, const uint4& b, float acc) {
  const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
  const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 fa = __bfloat1622float2(a2[i]);
    const float2 fb = __bfloat1622float2(b2[i]);
    acc = fmaf(fa.x, fb.x, acc);
    acc = fmaf(fa.y, fb.y, acc);
  }
  return acc;
}

__global__ void __launch_bounds__(kThreads, 1)
    conv_chain_small_kernel(const __nv_bfloat16* __restrict__ x0, const __nv_bfloat16* __restrict__ W,
                            __nv_bfloat16* buf0, __nv_bfloat16* buf1, __nv_bfloat16* z_out, int M, int H, int T,
                            int NL, int raw, unsigned* bar_count, int32_t* err) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  __shared__ uint64_t wbar[2];
  __shared__ float red[kThreads / 32][kVals];
  __shared__ float taps_s[64][kTaps];
  __shared__ int stop;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = H / 16, P = 2 * G;
  const int g0 = (int)((int64_t)blockIdx.x * G / gridDim.x);
  const int g1 = (int)((int64_t)(blockIdx.x + 1) * G / gridDim.x);
  const int ntaps = 2 * (g1 - g0);
  const uint32_t slice_bytes = (uint32_t)ntaps * H * 2;
  __nv_bfloat16* wbuf[2] = {reinterpret_cast<__nv_bfloat16*>(smem_raw),
                            reinterpret_cast<__nv_bfloat16*>(smem_raw) + (size_t)kTaps * H};
  const int chunks = H / 8;

  int last_issued[2] = {-1, -1};  // thread 0: newest layer requested into each buffer
  if (tid == 0) {
    stop = 0;
    mbar_init(&wbar[0], 1);
    mbar_init(&wbar[1], 1);
    fence_barrier_init();
    for (int l = 0; l < 2 && l < NL; ++l) {
      mbar_arrive_expect_tx(&wbar[l], slice_bytes);
      bulk_g2s(wbuf[l], W + ((size_t)l * P + 2 * g0) * H, slice_bytes, &wbar[l]);
      last_issued[l] = l;
    }
  }
  __syncthreads();

  for (int l = 0; l < NL; ++l) {
    const __nv_bfloat16* xin = (l == 0) ? x0 : ((l - 1) % 2 == 0 ? buf0 : buf1);
    __nv_bfloat16* xout = (l == NL - 1) ? z_out : (l % 2 == 0 ? buf0 : buf1);
    const __nv_bfloat16* ws = wbuf[l & 1];
    if (!mbar_wait(&wbar[l & 1], (uint32_t)(l >> 1) & 1u, err, &stop)) break;

    // ---- 1. taps for every row
    for (int r0 = 0; r0 < M; r0 += kRowBlk) {
      float acc[kRowBlk][kTaps];
#pragma unroll
      for (int r = 0; r < kRowBlk; ++r)
#pragma unroll
        for (int q = 0; q < kTaps; ++q) acc[r][q] = 0.f;
      const int nrows = min(kRowBlk, M - r0);
      for (int c = tid; c < chunks; c += kThreads) {
        // every row's 16 bytes are requested before any is used
        uint4 xv[kRowBlk];
#pragma unroll
        for (int r = 0; r < kRowBlk; ++r)
          xv[r] = r < nrows ? __ldcg(reinterpret_cast<const uint4*>(xin + (size_t)(r0 + r) * H) + c)
                            : make_uint4(0, 0, 0, 0);
        uint4 wv[kTaps];
#pragma unroll
        for (int q = 0; q < kTaps; ++q)
          wv[q] = q < ntaps ? *reinterpret_cast<const uint4*>(ws + (size_t)q * H + c * 8) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int r = 0; r < kRowBlk; ++r)
#pragma unroll
          for (int q = 0; q < kTaps; ++q) acc[r][q] = dot8(xv[r], wv[q], acc[r][q]);
      }
      // reduce-scatter across the warp: after step s a lane keeps half of its values, summed
      // with its partner's; at the end lane l holds the warp sums of values 2l and 2l+1
      float v[kVals];
#pragma unroll
      for (int r = 0; r < kRowBlk; ++r)
#pragma unroll
        for (int q = 0; q < kTaps; ++q) v[r * kTaps + q] = acc[r][q];
#pragma unroll
      for (int step = 0; step < 5; ++step) {
        const int half = kVals >> (step + 1);  // 32, 16, 8, 4, 2
        const int off = 16 >> step;
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
          const float send = upper ? v[i] : v[i + half];
          const float keep = upper ? v[i + half] : v[i];
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
      }
      red[warp][2 * lane] = v[0];
      red[warp][2 * lane + 1] = v[1];
      __syncthreads();
      if (tid < kVals) {
        float t = 0.f;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) t += red[w][tid];
        const int r = tid / kTaps, q = tid % kTaps;
        if (r0 + r < M) taps_s[r0 + r][q] = t;
      }
      __syncthreads();
    }
    // the weight buffer of layer l is free: request layer l+2's slice into it
    if (tid == 0 && l + 2 < NL) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive_expect_tx(&wbar[l & 1], slice_bytes);
      bulk_g2s(wbuf[l & 1], W + ((size_t)(l + 2) * P + 2 * g0) * H, slice_bytes, &wbar[l & 1]);
      last_issued[l & 1] = l + 2;
    }

    // ---- 2. mix: 16-byte pieces (8 channels) of the CTA's channels, every row
    const int pieces = (g1 - g0) * 2;  // two 8-channel pieces per group
    for (int e = tid; e < M * pieces; e += kThreads) {
      const int m = e / pieces, pc = e % pieces;
      const int j = pc >> 1;  // group index within the CTA
      const float p0 = taps_s[m][2 * j], p1 = taps_s[m][2 * j + 1];
      float a, b;
      if (raw) {
        a = p0;
        b = p1;
      } else {
        const float mx = fmaxf(p0, p1);
        const float e0 = expf(p0 - mx), e1 = expf(p1 - mx);
        const float inv = 1.f / (e0 + e1);
        a = e0 * inv;
        b = e1 * inv;
      }
      const int c0 = (g0 + j) * 16 + (pc & 1) * 8;
      const uint4 cur = __ldcg(reinterpret_cast<const uint4*>(xin + (size_t)m * H + c0));
      const uint4 prv = (m % T) != 0 ? __ldcg(reinterpret_cast<const uint4*>(xin + (size_t)(m - 1) * H + c0))
                                     : make_uint4(0, 0, 0, 0);
      const __nv_bfloat162* c2 = reinterpret_cast<const __nv_bfloat162*>(&cur);
      const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&prv);
      uint4 out;
      __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(&out);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 cf = __bfloat1622float2(c2[k]);
        const float2 pf = __bfloat1622float2(p2[k]);
        o2[k] = __floats2bfloat162_rn(fmaf(a, pf.x, b * cf.x), fmaf(a, pf.y, b * cf.y));
      }
      *reinterpret_cast<uint4*>(xout + (size_t)m * H + c0) = out;
    }
    if (l + 1 < NL && !grid_barrier(bar_count, (unsigned)(l + 1), err, &stop)) break;
  }
  // no copy may still be landing in shared memory when the CTA exits
  if (tid == 0) {
    for (int b = 0; b < 2; ++b)
      if (last_issued[b] >= 0) mbar_wait(&wbar[b], (uint32_t)(last_issued[b] >> 1) & 1u, err, nullptr);
  }
  __syncthreads();
}
}  // namespace

size_t conv_chain_small_smem(int H) { return (size_t)2 * kTaps * H * 2; }

cudaError_t launch_conv_chain_small(const void* x, const void* conv_w, void* buf0, void* buf1, void* z, int M,
                                    int H, int T, int NL, int raw, unsigned* bar_count, int32_t* err, int grid,
                                    cudaStream_t s) {
  const size_t smem = conv_chain_small_smem(H);
  cudaError_t e = cudaFuncSetAttribute(conv_chain_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(bar_count, 0, sizeof(unsigned), s);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, conv_chain_small_kernel, reinterpret_cast<const __nv_bfloat16*>(x),
                         reinterpret_cast<const __nv_bfloat16*>(conv_w), reinterpret_cast<__nv_bfloat16*>(buf0),
                         reinterpret_cast<__nv_bfloat16*>(buf1), reinterpret_cast<__nv_bfloat16*>(z), M, H, T, NL, raw,
                         bar_count, err);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace df
