// All conv layers in one cooperative launch (bf16), on the tensor cores through mma.sync.
//
// CTA (rb, gb) owns a block of rows [rb*RB, rb*RB + RB) and a contiguous range of channel
// groups [g0, g1) for every layer, i.e. projection rows 2*g0 .. 2*g1 of each layer's weight
// (contiguous in memory). RB is 16 or 64 rows (one or four 16-row tiles); row blocks are
// independent of each other, so each has its own grid barrier. Per layer:
//   1. taps: P[m][q] = x[m] . W[2*g0 + q] for the block's rows m and the CTA's taps q with
//      mma.sync m16n8k16 (bf16 in, fp32 accumulate). Warp w takes row tile w % MT and the
//      hidden slice w / MT of 8 / MT; the slices' partial tiles are summed in shared memory.
//      The 16 k-slots of one MMA may hold any 16 of a 32-wide chunk's positions as long as A
//      and B agree, so lane (g = lane/4, j = lane%4) feeds rows g, g+8 (A) and tap row g (B)
//      with one 16-byte load each for positions 8j..8j+7: 8j..8j+3 go to the first MMA and
//      8j+4..8j+7 to the second.
//   2. mix: (a, b) = softmax(P[m][2j], P[m][2j+1]) (raw taps on request), and
//      y[m][c] = a * x[m-1][c] + b * x[m][c] for the group's 16 channels, x[-1] = 0 at each
//      block start, rounded to bf16 and written to the layer's output buffer;
//   3. the row block's barrier (its CTAs need every channel of the next layer's input rows).
// Variants (template flags): the block's input rows x are staged in shared memory by bulk
// copies (one per row) after the barrier (kStageX, 16-row blocks), or read from L2 with .cg
// loads (which skip the non-coherent L1: the buffers are rewritten between layers); the weight
// slice is staged in shared memory by bulk copies requested as soon as the previous layer's
// taps are done (kStageW), or read from global memory after an L2 prefetch issued a layer
// ahead. Staged rows are padded by 64 bytes so the fragment loads are free of bank conflicts.
// Barriers are atomic counters in the workspace (zeroed by the host before the launch) with
// a bounded spin: on timeout the kernel sets DFLASH2_DEVERR_WAIT_TIMEOUT and stops.
#include <cuda_bf16.h>
#include <math.h>

#include "../../include/dflash2.h"
#include "kernels.h"
#include "grid_sync.cuh"
#include "launch_util.h"
#include "ptx.cuh"

namespace df {

namespace {
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRowPad = 32;  // bf16 elements of padding per staged row

DF_DEV void bulk_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(smem_dst)),
               "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

DF_DEV void prefetch_l2(const void* gmem_src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(gmem_src), "r"(bytes) : "memory");
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

template <bool kSmem>
DF_DEV uint4 ld16(const __nv_bfloat16* p) {
  if constexpr (kSmem) return *reinterpret_cast<const uint4*>(p);
  else return __ldcg(reinterpret_cast<const uint4*>(p));
}

template <bool kStageX, bool kStageW, int kMT, int kNT>
__global__ void __launch_bounds__(kThreads, 1)
    conv_chain_kernel(const __nv_bfloat16* __restrict__ x0, const __nv_bfloat16* __restrict__ W,
                      __nv_bfloat16* buf0, __nv_bfloat16* buf1, __nv_bfloat16* z_out, int M, int H, int T, int NL,
                      int raw, int GBn, int wtaps, unsigned* bar_counts, int32_t* err) {
  constexpr int RB = 16 * kMT;          // rows per block
  constexpr int kSlices = kWarps / kMT;  // hidden slices per row tile
  constexpr int TQ = kNT * 8;            // taps per CTA, padded
  constexpr int kAcc = kNT == 1 ? 4 : (kNT <= 3 ? 2 : 1);  // independent accumulator sets
  extern __shared__ __align__(128) uint8_t smem_raw[];
  __shared__ uint64_t wbar, xbar;
  __shared__ int stop;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rb = blockIdx.x / GBn, gb = blockIdx.x % GBn;
  const int r0 = rb * RB, nrows = min(RB, M - r0);
  const int G = H / 16, P = 2 * G;
  const int g0 = (int)((int64_t)gb * G / GBn);
  const int g1 = (int)((int64_t)(gb + 1) * G / GBn);
  const int ntaps = 2 * (g1 - g0);
  const uint32_t slice_bytes = (uint32_t)ntaps * H * 2;
  // staged rows are kRowPad elements longer than H (a 64-byte step modulo 128), so the
  // 16-byte fragment loads of lanes in different rows fall in different banks
  const int xstride = kStageX ? H + kRowPad : H;
  const int wstride = kStageW ? H + kRowPad : H;
  // shared memory: [weight slice (kStageW)] [x rows (kStageX)] [partial tiles] [taps]
  uint8_t* p = smem_raw;
  __nv_bfloat16* ws = reinterpret_cast<__nv_bfloat16*>(p);
  if constexpr (kStageW) p += (size_t)wtaps * (H + kRowPad) * 2;
  __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(p);
  if constexpr (kStageX) p += (size_t)RB * (H + kRowPad) * 2;
  float* red = reinterpret_cast<float*>(p);  // [kSlices][RB][TQ]
  p += (size_t)kSlices * RB * TQ * 4;
  float* taps_s = reinterpret_cast<float*>(p);  // [RB][TQ]
  unsigned* my_bar = bar_counts + rb;

  pdl_launch_dependents();  // the LM head may start its prologue as SMs free up
  if (tid == 0) {
    stop = 0;
    mbar_init(&wbar, 1);
    mbar_init(&xbar, 1);
    fence_barrier_init();
    if constexpr (kStageW) {
      mbar_arrive_expect_tx(&wbar, slice_bytes);
      for (int q = 0; q < ntaps; ++q) bulk_g2s(ws + (size_t)q * wstride, W + (size_t)(2 * g0 + q) * H, H * 2, &wbar);
    } else {
      prefetch_l2(W + (size_t)(2 * g0) * H, slice_bytes);
    }
  }
  __syncthreads();

  const int mt = warp % kMT, ks = warp / kMT;
  const int kw = H / kSlices;
  const int kbeg = ks * kw;
  const int g = lane >> 2, j = lane & 3;
  // rows past the block's end read its last row (their products land in dropped accumulator rows)
  const int rlo = min(mt * 16 + g, nrows - 1), rhi = min(mt * 16 + g + 8, nrows - 1);

  uint32_t wphase = 0, xphase = 0;
  bool w_pending = kStageW;  // thread 0 issued a weight copy not yet waited for
  for (int l = 0; l < NL; ++l) {
    const __nv_bfloat16* xin_g = (l == 0) ? x0 : ((l - 1) % 2 == 0 ? buf0 : buf1);
    __nv_bfloat16* xout = (l == NL - 1) ? z_out : (l % 2 == 0 ? buf0 : buf1);
    const __nv_bfloat16* wl = W + ((size_t)l * P + 2 * g0) * H;  // this layer's slice
    if (!kStageW && tid == 0 && l + 1 < NL) prefetch_l2(wl + (size_t)P * H, slice_bytes);
    const __nv_bfloat16* xb = xin_g + (size_t)r0 * H;  // the block's first row
    if constexpr (kStageX) {
      if (warp == 0) {
        // rows written by other CTAs' generic stores before the barrier; order them before
        // this async-proxy read. One bulk copy per row, spread over the lanes, so the rows
        // stream in parallel.
        if (lane == 0) mbar_arrive_expect_tx(&xbar, (uint32_t)nrows * H * 2);
        __syncwarp();
        asm volatile("fence.proxy.async.global;" ::: "memory");
        for (int m = lane; m < nrows; m += 32)
          bulk_g2s(xs + (size_t)m * xstride, xb + (size_t)m * H, (uint32_t)H * 2, &xbar);
      }
      if (!mbar_wait(&xbar, xphase, err, &stop)) break;
      xphase ^= 1u;
    }
    if constexpr (kStageW) {
      if (!mbar_wait(&wbar, wphase, err, &stop)) break;
      wphase ^= 1u;
      if (tid == 0) w_pending = false;
    }
    __syncwarp();  // the lanes left the waits at different times; mma.sync wants the warp converged
    const __nv_bfloat16* xa_base = kStageX ? xs : xb;
    const __nv_bfloat16* wb_base = kStageW ? ws : wl;

    // ---- 1. taps
    {
      // kAcc independent accumulator sets (32-wide chunks c go to set c % kAcc), so the
      // MMAs of consecutive chunks do not wait on each other; summed at the end
      float acc[kAcc][kNT][4];
#pragma unroll
      for (int a = 0; a < kAcc; ++a)
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[a][nt][e] = 0.f;
      bool tap_ok[kNT];
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt) tap_ok[nt] = nt * 8 + g < ntaps;
      const int kend = kbeg + kw;
      for (int k0 = kbeg; k0 < kend; k0 += 32 * kAcc) {
        uint4 xa[kAcc], xc[kAcc], wv[kAcc][kNT];
#pragma unroll
        for (int a = 0; a < kAcc; ++a) {
          const int kk = min(k0 + 32 * a, kend - 32) + 8 * j;  // a chunk past the end repeats the last one
          xa[a] = ld16<kStageX>(xa_base + (size_t)rlo * xstride + kk);
          xc[a] = ld16<kStageX>(xa_base + (size_t)rhi * xstride + kk);
#pragma unroll
          for (int nt = 0; nt < kNT; ++nt)
            wv[a][nt] =
                tap_ok[nt] ? ld16<kStageW>(wb_base + (size_t)(nt * 8 + g) * wstride + kk) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int a = 0; a < kAcc; ++a) {
          if (k0 + 32 * a >= kend) break;  // (uniform) the repeated chunk is not accumulated
#pragma unroll
          for (int nt = 0; nt < kNT; ++nt) {
            mma_16816(acc[a][nt], xa[a].x, xc[a].x, xa[a].y, xc[a].y, wv[a][nt].x, wv[a][nt].y);
            mma_16816(acc[a][nt], xa[a].z, xc[a].z, xa[a].w, xc[a].w, wv[a][nt].z, wv[a][nt].w);
          }
        }
      }
#pragma unroll
      for (int a = 1; a < kAcc; ++a)
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[0][nt][e] += acc[a][nt][e];
      // accumulator layout: acc[nt][0..1] = row mt*16+g, taps nt*8+2j, +1; [2..3] = row +8
      float* rw = red + (size_t)ks * RB * TQ;
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt) {
        rw[(mt * 16 + g) * TQ + nt * 8 + 2 * j] = acc[0][nt][0];
        rw[(mt * 16 + g) * TQ + nt * 8 + 2 * j + 1] = acc[0][nt][1];
        rw[(mt * 16 + g + 8) * TQ + nt * 8 + 2 * j] = acc[0][nt][2];
        rw[(mt * 16 + g + 8) * TQ + nt * 8 + 2 * j + 1] = acc[0][nt][3];
      }
      __syncthreads();
      for (int e = tid; e < nrows * TQ; e += kThreads) {
        float t = 0.f;
#pragma unroll
        for (int s = 0; s < kSlices; ++s) t += red[(size_t)s * RB * TQ + e];
        taps_s[e] = t;
      }
      __syncthreads();
    }
    // the staged weight slice is free: request the next layer's
    if (kStageW && warp == 0 && l + 1 < NL) {
      if (lane == 0) {
        mbar_arrive_expect_tx(&wbar, slice_bytes);
        w_pending = true;
      }
      __syncwarp();
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      for (int q = lane; q < ntaps; q += 32)
        bulk_g2s(ws + (size_t)q * wstride, wl + (size_t)(P + q) * H, H * 2, &wbar);
    }

    // ---- 2. mix: 16-byte pieces (8 channels) of the CTA's channels, every row of the block
    const int pieces = (g1 - g0) * 2;  // two 8-channel pieces per group
    for (int e = tid; e < nrows * pieces; e += kThreads) {
      const int m = e / pieces, pc = e % pieces;
      const int jg = pc >> 1;  // group index within the CTA
      const float p0 = taps_s[m * TQ + 2 * jg], p1 = taps_s[m * TQ + 2 * jg + 1];
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
      const uint4 cur = ld16<kStageX>(xa_base + (size_t)m * xstride + c0);
      uint4 prv = make_uint4(0, 0, 0, 0);
      if ((r0 + m) % T != 0)  // the previous row of the same sequence (outside the block if m == 0)
        prv = m > 0 ? ld16<kStageX>(xa_base + (size_t)(m - 1) * xstride + c0)
                    : __ldcg(reinterpret_cast<const uint4*>(xb - H + c0));
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
      *reinterpret_cast<uint4*>(xout + (size_t)(r0 + m) * H + c0) = out;
    }
    if (l + 1 < NL && !group_barrier(my_bar, (unsigned)(l + 1), (unsigned)GBn, err, &stop)) break;
  }
  // no copy may still be landing in shared memory when the CTA exits
  if (kStageW && tid == 0 && w_pending) mbar_wait(&wbar, wphase, err, nullptr);
  __syncthreads();
}

// Variants: (stage x, stage weights, row tiles, tap tiles).
struct Variant {
  bool sx, sw;
  int mt, nt;
};
constexpr Variant kVariants[] = {{true, true, 1, 1}, {true, false, 1, 3}, {false, true, 4, 3}, {false, false, 4, 9}};

size_t variant_smem(const Variant& v, int H, int wtaps) {
  const int RB = 16 * v.mt, slices = kWarps / v.mt, TQ = v.nt * 8;
  return (v.sw ? (size_t)wtaps * (H + kRowPad) * 2 : 0) + (v.sx ? (size_t)RB * (H + kRowPad) * 2 : 0) +
         (size_t)slices * RB * TQ * 4 +
         (size_t)RB * TQ * 4;
}

constexpr size_t kSmemLimit = 227 * 1024 - 256;  // minus the static barriers
}  // namespace

bool conv_chain_plan(int M, int H, int sms, ConvChainPlan* out) {
  if (H % 256 != 0 || M < 1 || sms < 1) return false;
  const int G = H / 16;
  // the first variant whose row tiles, tap capacity and shared memory fit
  for (int vi = 0; vi < 4; ++vi) {
    const Variant& v = kVariants[vi];
    const int RB = 16 * v.mt;
    if (vi == 0 && M > 16) continue;    // one 16-row block with all CTAs on the groups
    if (v.mt == 1 && M > 64) continue;  // 16-row blocks only for small M
    if (v.mt == 4 && M <= 64) continue;
    const int RBn = (M + RB - 1) / RB;
    if (RBn > sms) continue;
    int GBn = sms / RBn;
    if (GBn > G) GBn = G;
    const int taps = 2 * ((G + GBn - 1) / GBn);
    if (taps > v.nt * 8) continue;
    if (variant_smem(v, H, taps) > kSmemLimit) continue;
    out->variant = vi;
    out->row_blocks = RBn;
    out->group_blocks = GBn;
    out->wtaps = taps;
    out->smem = variant_smem(v, H, taps);
    return true;
  }
  return false;
}

cudaError_t launch_conv_chain(const ConvChainPlan& pl, const void* x, const void* conv_w, void* buf0, void* buf1,
                              void* z, int M, int H, int T, int NL, int raw, unsigned* bar_counts, int32_t* err,
                              cudaStream_t s) {
  const void* fns[4] = {reinterpret_cast<const void*>(conv_chain_kernel<true, true, 1, 1>),
                        reinterpret_cast<const void*>(conv_chain_kernel<true, false, 1, 3>),
                        reinterpret_cast<const void*>(conv_chain_kernel<false, true, 4, 3>),
                        reinterpret_cast<const void*>(conv_chain_kernel<false, false, 4, 9>)};
  if (pl.variant < 0 || pl.variant > 3) return cudaErrorInvalidValue;
  static unsigned char smem_done[4][64];
  cudaError_t e = smem_opt_in(fns[pl.variant], smem_done[pl.variant]);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(bar_counts, 0, sizeof(unsigned) * pl.row_blocks, s);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.row_blocks * pl.group_blocks);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = pl.smem;
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
  switch (pl.variant) {
    case 0:
      e = cudaLaunchKernelEx(&cfg, conv_chain_kernel<true, true, 1, 1>, xb, wb, b0, b1, zb, M, H, T, NL, raw,
                             pl.group_blocks, pl.wtaps, bar_counts, err);
      break;
    case 1:
      e = cudaLaunchKernelEx(&cfg, conv_chain_kernel<true, false, 1, 3>, xb, wb, b0, b1, zb, M, H, T, NL, raw,
                             pl.group_blocks, pl.wtaps, bar_counts, err);
      break;
    case 2:
      e = cudaLaunchKernelEx(&cfg, conv_chain_kernel<false, true, 4, 3>, xb, wb, b0, b1, zb, M, H, T, NL, raw,
                             pl.group_blocks, pl.wtaps, bar_counts, err);
      break;
    default:
      e = cudaLaunchKernelEx(&cfg, conv_chain_kernel<false, false, 4, 9>, xb, wb, b0, b1, zb, M, H, T, NL, raw,
                             pl.group_blocks, pl.wtaps, bar_counts, err);
      break;
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace df
