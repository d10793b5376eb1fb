// All conv layers in one cooperative launch, for a small number of rows (M <= 64, bf16).
//
// Each CTA owns a contiguous range of channel groups [g0, g1) for every layer (2-4 groups at
// the page shape: 320 groups over the SMs), i.e. projection rows 2*g0 .. 2*g1 of each layer's
// weight, which are contiguous in memory. Per layer:
//   1. taps: P[m][q] = x[m] . W[2*g0 + q] for every row m and the CTA's taps q, on the tensor
//      cores (mma.sync m16n8k16, bf16 in, fp32 accumulate); each warp takes 1/8 of the
//      hidden dimension and the 8 warps' partial tiles are summed in shared memory;
//   2. mix: (a, b) = softmax(P[m][2j], P[m][2j+1]) (raw taps on request), and
//      y[m][c] = a * x[m-1][c] + b * x[m][c] for the group's 16 channels, x[-1] = 0 at each
//      block start, rounded to bf16 and written to the layer's output buffer;
//   3. a grid barrier (every CTA needs every channel of the next layer's input).
// Weight slices arrive in shared memory by bulk async copies, requested as soon as the buffer
// they go to is free, so their latency hides behind the mix and the barrier.
// Two variants:
//   kStageX (M <= 16): the layer's whole input block x [M, H] (contiguous) is copied into
//     shared memory by one bulk copy after the barrier; taps and mix read it there. The weight
//     slice is single-buffered to make room.
//   otherwise: x is read from L2 with .cg loads (which skip the non-coherent L1, since the
//     buffers are rewritten between layers) and the weight slice is double-buffered.
// The barrier is an atomic counter in the workspace (zeroed by the host before the launch)
// with a bounded spin: on timeout the kernel sets DFLASH2_DEVERR_WAIT_TIMEOUT and stops.
#include <cuda_bf16.h>
#include <math.h>

#include "../../include/dflash2.h"
#include "kernels.h"
#include "ptx.cuh"

namespace df {

namespace {
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTaps = 8;       // taps per CTA at most (4 groups)
constexpr int kMaxRows = 64;
constexpr int kStageRows = 16;  // the staged variant's row limit

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
      __nanosleep(32);
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

// d += A(16x16 fragments a0..a3) * B(16x8 fragments b0, b1), bf16 in, fp32 out
DF_DEV void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                      uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <bool kStageX>
DF_DEV uint4 load_x16(const __nv_bfloat16* p) {
  if constexpr (kStageX) return *reinterpret_cast<const uint4*>(p);
  else return __ldcg(reinterpret_cast<const uint4*>(p));
}

template <bool kStageX>
__global__ void __launch_bounds__(kThreads, 1)
    conv_chain_small_kernel(const __nv_bfloat16* __restrict__ x0, const __nv_bfloat16* __restrict__ W,
                            __nv_bfloat16* buf0, __nv_bfloat16* buf1, __nv_bfloat16* z_out, int M, int H, int T,
                            int NL, int raw, int wtaps, unsigned* bar_count, int32_t* err) {
  constexpr int kRows = kStageX ? kStageRows : kMaxRows;
  constexpr int kMT = kRows / 16;  // row tiles of 16
  extern __shared__ __align__(128) uint8_t smem_raw[];
  __shared__ uint64_t wbar[2], xbar;
  __shared__ float red[kWarps][kRows * kTaps];
  __shared__ float taps_s[kRows][kTaps];
  __shared__ int stop;
  constexpr int kBufs = kStageX ? 1 : 2;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = H / 16, P = 2 * G;
  const int g0 = (int)((int64_t)blockIdx.x * G / gridDim.x);
  const int g1 = (int)((int64_t)(blockIdx.x + 1) * G / gridDim.x);
  const int ntaps = 2 * (g1 - g0);
  const uint32_t slice_bytes = (uint32_t)ntaps * H * 2;
  // weight buffers hold `wtaps` rows (the most any CTA owns); the staged x block follows them
  __nv_bfloat16* wbuf[2] = {reinterpret_cast<__nv_bfloat16*>(smem_raw),
                            reinterpret_cast<__nv_bfloat16*>(smem_raw) + (size_t)wtaps * H};
  __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(smem_raw) + (size_t)kBufs * wtaps * H;  // kStageX only
  const uint32_t x_bytes = (uint32_t)M * H * 2;

  int last_issued[2] = {-1, -1};  // thread 0: newest layer requested into each buffer
  if (tid == 0) {
    stop = 0;
    mbar_init(&wbar[0], 1);
    mbar_init(&wbar[1], 1);
    mbar_init(&xbar, 1);
    fence_barrier_init();
    for (int l = 0; l < kBufs && l < NL; ++l) {
      mbar_arrive_expect_tx(&wbar[l], slice_bytes);
      bulk_g2s(wbuf[l], W + ((size_t)l * P + 2 * g0) * H, slice_bytes, &wbar[l]);
      last_issued[l] = l;
    }
  }
  __syncthreads();

  uint32_t xphase = 0;
  for (int l = 0; l < NL; ++l) {
    const __nv_bfloat16* xin_g = (l == 0) ? x0 : ((l - 1) % 2 == 0 ? buf0 : buf1);
    __nv_bfloat16* xout = (l == NL - 1) ? z_out : (l % 2 == 0 ? buf0 : buf1);
    const int wb = l % kBufs;
    const __nv_bfloat16* ws = wbuf[wb];
    const __nv_bfloat16* xin = xin_g;
    if constexpr (kStageX) {
      if (tid == 0) {
        // the block was written by other CTAs' generic stores before the barrier; order them
        // before this async-proxy read
        asm volatile("fence.proxy.async.global;" ::: "memory");
        mbar_arrive_expect_tx(&xbar, x_bytes);
        bulk_g2s(xs, xin_g, x_bytes, &xbar);
      }
      xin = xs;
      if (!mbar_wait(&xbar, xphase, err, &stop)) break;
      xphase ^= 1u;
    }
    if (!mbar_wait(&wbar[wb], (uint32_t)(l / kBufs) & 1u, err, &stop)) break;

    // ---- 1. taps for every row on the tensor cores. Warp w takes the hidden range
    // [w*H/8, (w+1)*H/8) in chunks of 32. The 16 k-slots of one MMA may hold any 16 of the
    // chunk's positions as long as A and B agree, so lane (g = lane/4, j = lane%4) loads 8
    // consecutive positions 8j..8j+7 of rows g and g+8 (A) and of tap row g (B) as single
    // 16-byte loads: positions 8j..8j+3 feed the first MMA and 8j+4..8j+7 the second.
    {
      const int g = lane >> 2, j = lane & 3;
      const int kw = H / kWarps;
      const int kbeg = warp * kw;
      const int mtiles = (M + 15) / 16;  // at most kRows / 16
      float acc[kMT][4];
#pragma unroll
      for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[mt][e] = 0.f;
      // rows past M read row M-1 (their products land in accumulator rows that are dropped)
      int rlo[kMT], rhi[kMT];
#pragma unroll
      for (int mt = 0; mt < kMT; ++mt) {
        rlo[mt] = min(mt * 16 + g, M - 1);
        rhi[mt] = min(mt * 16 + g + 8, M - 1);
      }
      const bool tap_ok = g < ntaps;
      // unrolled so that several chunks' loads are in flight before their MMAs consume them
#pragma unroll 4
      for (int k0 = kbeg; k0 < kbeg + kw; k0 += 32) {
        const int kk = k0 + 8 * j;
        uint4 xa[kMT], xb[kMT];
#pragma unroll
        for (int mt = 0; mt < kMT; ++mt) {
          if (mt < mtiles) {
            xa[mt] = load_x16<kStageX>(xin + (size_t)rlo[mt] * H + kk);
            xb[mt] = load_x16<kStageX>(xin + (size_t)rhi[mt] * H + kk);
          }
        }
        const uint4 wv = tap_ok ? *reinterpret_cast<const uint4*>(ws + (size_t)g * H + kk) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int mt = 0; mt < kMT; ++mt) {
          if (mt < mtiles) {
            mma_16816(acc[mt], xa[mt].x, xb[mt].x, xa[mt].y, xb[mt].y, wv.x, wv.y);
            mma_16816(acc[mt], xa[mt].z, xb[mt].z, xa[mt].w, xb[mt].w, wv.z, wv.w);
          }
        }
      }
      // accumulator layout: acc[mt][0..1] = row mt*16+g, taps 2j, 2j+1; [2..3] = row +8
#pragma unroll
      for (int mt = 0; mt < kMT; ++mt) {
        if (mt < mtiles) {
          red[warp][(mt * 16 + g) * kTaps + 2 * j] = acc[mt][0];
          red[warp][(mt * 16 + g) * kTaps + 2 * j + 1] = acc[mt][1];
          red[warp][(mt * 16 + g + 8) * kTaps + 2 * j] = acc[mt][2];
          red[warp][(mt * 16 + g + 8) * kTaps + 2 * j + 1] = acc[mt][3];
        }
      }
      __syncthreads();
      for (int e = tid; e < M * kTaps; e += kThreads) {
        float t = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) t += red[w][e];
        taps_s[e / kTaps][e % kTaps] = t;
      }
      __syncthreads();
    }
    // the weight buffer of layer l is free: request layer l + kBufs's slice into it
    if (tid == 0 && l + kBufs < NL) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive_expect_tx(&wbar[wb], slice_bytes);
      bulk_g2s(wbuf[wb], W + ((size_t)(l + kBufs) * P + 2 * g0) * H, slice_bytes, &wbar[wb]);
      last_issued[wb] = l + kBufs;
    }

    // ---- 2. mix: 16-byte pieces (8 channels) of the CTA's channels, every row
    const int pieces = (g1 - g0) * 2;  // two 8-channel pieces per group
    for (int e = tid; e < M * pieces; e += kThreads) {
      const int m = e / pieces, pc = e % pieces;
      const int jg = pc >> 1;  // group index within the CTA
      const float p0 = taps_s[m][2 * jg], p1 = taps_s[m][2 * jg + 1];
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
      const int c0 = (g0 + jg) * 16 + (pc & 1) * 8;
      const uint4 cur = load_x16<kStageX>(xin + (size_t)m * H + c0);
      const uint4 prv = (m % T) != 0 ? load_x16<kStageX>(xin + (size_t)(m - 1) * H + c0) : make_uint4(0, 0, 0, 0);
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
    for (int b = 0; b < kBufs; ++b)
      if (last_issued[b] >= 0) mbar_wait(&wbar[b], (uint32_t)(last_issued[b] / kBufs) & 1u, err, nullptr);
  }
  __syncthreads();
}
}  // namespace

// Dynamic shared memory of one variant: the weight buffer(s) of `wtaps` rows, and for the
// staged variant the x block.
static size_t chain_smem(bool stage, int M, int H, int wtaps) {
  return (size_t)(stage ? 1 : 2) * wtaps * H * 2 + (stage ? (size_t)M * H * 2 : 0);
}

// Largest dynamic shared memory a variant may ask for: 227 KB minus its static arrays
// (reduction tiles and taps) and a margin for the barriers.
static size_t chain_smem_limit(bool stage) {
  const size_t rows = stage ? kStageRows : kMaxRows;
  return 227 * 1024 - (size_t)kWarps * rows * kTaps * 4 - rows * kTaps * 4 - 256;
}

bool conv_chain_small_fits(int M, int H, int wtaps) {
  if (M > kMaxRows || wtaps > kTaps || H % 256 != 0) return false;
  return chain_smem(false, M, H, wtaps) <= chain_smem_limit(false);
}

cudaError_t launch_conv_chain_small(const void* x, const void* conv_w, void* buf0, void* buf1, void* z, int M,
                                    int H, int T, int NL, int raw, int wtaps, unsigned* bar_count, int32_t* err,
                                    int grid, cudaStream_t s) {
  if (!conv_chain_small_fits(M, H, wtaps)) return cudaErrorInvalidValue;
  const bool stage = M <= kStageRows && chain_smem(true, M, H, wtaps) <= chain_smem_limit(true);
  const size_t smem = chain_smem(stage, M, H, wtaps);
  const void* fn = stage ? reinterpret_cast<const void*>(conv_chain_small_kernel<true>)
                         : reinterpret_cast<const void*>(conv_chain_small_kernel<false>);
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
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
  const __nv_bfloat16* xb = reinterpret_cast<const __nv_bfloat16*>(x);
  const __nv_bfloat16* wb = reinterpret_cast<const __nv_bfloat16*>(conv_w);
  __nv_bfloat16* b0 = reinterpret_cast<__nv_bfloat16*>(buf0);
  __nv_bfloat16* b1 = reinterpret_cast<__nv_bfloat16*>(buf1);
  __nv_bfloat16* zb = reinterpret_cast<__nv_bfloat16*>(z);
  e = stage ? cudaLaunchKernelEx(&cfg, conv_chain_small_kernel<true>, xb, wb, b0, b1, zb, M, H, T, NL, raw, wtaps,
                                 bar_count, err)
            : cudaLaunchKernelEx(&cfg, conv_chain_small_kernel<false>, xb, wb, b0, b1, zb, M, H, T, NL, raw, wtaps,
                                 bar_count, err);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace df
