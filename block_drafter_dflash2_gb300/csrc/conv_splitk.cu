// All conv layers in one cooperative launch for larger row counts (bf16): the projection to
// the taps is split along the hidden dimension and runs on the tensor cores (tcgen05).
//
// Per layer l the taps are P[m][q] = x_l[m] . W_l[q] for the P = H/8 projection rows q
// (two per channel group of 16). CTA (rt, nt, ks) owns row tile rt (128 rows), tap tile nt
// (Nt projection rows) and K-slice ks (a range of 64-channel blocks):
//   A. TMA streams its (x rows, W rows) blocks of the slice through a 5-stage shared-memory
//      ring (128-byte swizzle, K-major); one thread issues tcgen05.mma (M = 128, N = Nt,
//      K = 16) into a TMEM accumulator; four epilogue warps (thread = TMEM lane = row) stage
//      the fp32 partial taps in the idle operand ring as [tap][row], and all 256 threads
//      write them to plane ks of [ks][q][m] with 16-byte stores (one scalar store per tap
//      and row from the epilogue threads alone would be limited by the stores a warp may
//      have in flight). Partials alternate between two sets of planes by layer parity.
//   grid barrier: every partial of the layer is written.
//   B. The NT CTAs sharing (rt, ks) split the channel groups of the slice. For each of its
//      (row, group) items a thread sums the group's two taps over the K-slices in slice
//      order (up to 20 slices loaded before any is added, the rows' channels issued
//      first), normalises them (softmax over the pair, unless raw), and writes
//      y[m, c] = a * x_l[m-1, c] + b * x_l[m, c] for the group's 16 channels (x[-1] = 0 at
//      each block start), rounded to bf16.
//   sibling barrier: the NT CTAs of (rt, ks) wait for each other, since the next layer's A
//      phase of each of them reads every channel of the slice for the tile's rows.
// Each CTA reads only its K-slice of the rows and of its tap rows, so the per-layer traffic
// is (M + P) * H * 2 bytes spread over the grid, plus the partial taps through L2; the older
// chain kernel, where each CTA reads every hidden channel of its rows, suits small M only.
// Every wait is bounded; on timeout the kernel sets DFLASH2_DEVERR_WAIT_TIMEOUT, lets copies
// in flight land, frees TMEM and returns.
#include <cuda_bf16.h>
#include <math.h>

#include "../../include/dflash2.h"
#include "grid_sync.cuh"
#include "kernels.h"
#include "launch_util.h"
#include "ptx.cuh"

namespace df {

namespace {
constexpr int kThreads = 256;
constexpr int kStages = 5;
constexpr uint32_t kABytes = 128 * 64 * 2;  // A region of a stage: the MMA reads 128 rows
constexpr int kMaxTile = 160;                // widest tap tile
constexpr int kC = 20;                       // K-slices whose partials a mix thread loads at once

struct SplitArgs {
  int M, H, T, NL, raw;
  int P;             // projection rows (taps) per layer = H / 8
  int RT, NT, KS;    // row tiles, tap tiles, K-slices
  int Nt;            // projection rows per tap tile (multiple of 16)
  int a_tail_rows;   // rows of the last row tile's TMA box (multiple of 8)
  int Mp;            // rows of a partial-tap plane (M rounded up to 4)
  float* part;       // [2][KS][P][Mp] fp32 partial taps
  const __nv_bfloat16* x0;
  __nv_bfloat16* buf0;
  __nv_bfloat16* buf1;
  __nv_bfloat16* z;
  unsigned* bar;     // [0]: grid barrier; [1 + rt * KS + ks]: barrier of the NT CTAs of (rt, ks)
  int32_t* err;
};

DF_DEV void tma_prefetch_2d(const CUtensorMap* map, int32_t c0, int32_t c1) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1)
               : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
    conv_splitk_kernel(const __grid_constant__ CUtensorMap map_x0, const __grid_constant__ CUtensorMap map_x0t,
                       const __grid_constant__ CUtensorMap map_b0, const __grid_constant__ CUtensorMap map_b0t,
                       const __grid_constant__ CUtensorMap map_b1, const __grid_constant__ CUtensorMap map_b1t,
                       const __grid_constant__ CUtensorMap map_w, const SplitArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(base);
  uint64_t* empty = full + kStages;
  uint64_t* tfull = empty + kStages;
  uint64_t* drain = tfull + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* stop = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* consumed_s = stop + 1;  // ring loads the MMA thread has waited for
  uint8_t* ring = base + 1024;
  float* stg = reinterpret_cast<float*>(ring);  // [Nt][128] fp32 tile of partials, in the idle ring

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nt = blockIdx.x % a.NT;
  const int sib = blockIdx.x / a.NT;  // rt * KS + ks
  const int ks = sib % a.KS, rt = sib / a.KS;
  const int nkb = a.H / 64;
  const int kb0 = ks * nkb / a.KS, kb1 = (ks + 1) * nkb / a.KS;
  const bool tail = rt == a.RT - 1;
  const uint32_t a_bytes = (uint32_t)(tail ? a.a_tail_rows : 128) * 128u;
  const uint32_t b_bytes = (uint32_t)a.Nt * 128u;
  const uint32_t stride = kABytes + ((b_bytes + 1023u) & ~1023u);
  const int rows = min(128, a.M - rt * 128);
  const uint32_t tmem_cols = a.Nt <= 32 ? 32u : (a.Nt <= 64 ? 64u : (a.Nt <= 128 ? 128u : 256u));
  const uint32_t idesc = idesc_bf16_f32(128, a.Nt);
  const size_t part_layer = (size_t)a.KS * a.P * a.Mp;

  pdl_launch_dependents();  // the LM head may start its prologue as SMs free up
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(drain, 1);
    *stop = 0;
    *consumed_s = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, tmem_cols);
    tmem_relinquish();
  }
  if (tid == 0) {
    tma_prefetch_desc(&map_w);
    tma_prefetch_desc(tail ? &map_x0t : &map_x0);
    // this CTA's weight blocks of every layer into L2 while the first layer runs
    for (int l = 0; l < a.NL; ++l)
      for (int kb = kb0; kb < kb1; ++kb) tma_prefetch_2d(&map_w, kb * 64, l * a.P + nt * a.Nt);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  uint32_t p_stage = 0, p_phase = 0, c_stage = 0, c_phase = 0;
  int issued = 0;  // producer thread: ring loads issued
  for (int l = 0; l < a.NL; ++l) {
    const CUtensorMap* mx = l == 0 ? (tail ? &map_x0t : &map_x0)
                                   : ((l - 1) % 2 == 0 ? (tail ? &map_b0t : &map_b0) : (tail ? &map_b1t : &map_b1));
    const __nv_bfloat16* xin = l == 0 ? a.x0 : ((l - 1) % 2 == 0 ? a.buf0 : a.buf1);
    __nv_bfloat16* xout = l == a.NL - 1 ? a.z : (l % 2 == 0 ? a.buf0 : a.buf1);
    float* part = a.part + (size_t)(l & 1) * part_layer;

    // ---- A. partial taps of the K-slice
    if (warp == 0) {
      if (lane == 0) {
        // the rows were written by other CTAs' generic stores before the last barrier, and
        // the ring held the previous layer's staged partials (generic accesses)
        if (l > 0) {
          asm volatile("fence.proxy.async.global;" ::: "memory");
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
        const uint64_t pol = l2_policy_evict_last();
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&empty[p_stage], p_phase ^ 1u, a.err, stop)) break;
          uint8_t* st = ring + (size_t)p_stage * stride;
          mbar_arrive_expect_tx(&full[p_stage], a_bytes + b_bytes);
          tma_load_2d(st, mx, &full[p_stage], kb * 64, rt * 128, pol);
          tma_load_2d(st + kABytes, &map_w, &full[p_stage], kb * 64, l * a.P + nt * a.Nt, pol);
          ++issued;
          if (++p_stage == kStages) {
            p_stage = 0;
            p_phase ^= 1u;
          }
        }
      }
    } else if (warp == 1) {
      if (lane == 0) {
        bool ok = true;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&full[c_stage], c_phase, a.err, stop)) {
            ok = false;
            break;
          }
          *consumed_s = *consumed_s + 1;
          tc_fence_after();
          const uint32_t sa = smem_u32(ring + (size_t)c_stage * stride);
          const uint64_t da = sdesc_k_sw128(sa);
          const uint64_t db = sdesc_k_sw128(sa + kABytes);
#pragma unroll
          for (int k = 0; k < 4; ++k)  // 16 bf16 = 32 B per MMA along K: +2 in 16-B units
            umma_bf16(tmem, da + 2 * k, db + 2 * k, idesc, (kb > kb0 || k > 0) ? 1u : 0u);
          umma_commit(&empty[c_stage]);
          if (++c_stage == kStages) {
            c_stage = 0;
            c_phase ^= 1u;
          }
        }
        if (ok) umma_commit(tfull);
      }
    } else if (warp >= 4) {
      // TMEM -> shared memory: the tile's partials as [tap][row] in the ring, which every
      // MMA of the layer has finished reading once tfull completes
      const int q = warp & 3;  // TMEM lane quadrant of this warp
      // lane 0 waits and the warp follows it converged: the TMEM loads are warp-wide
      // (.sync.aligned) and must not be reached by lanes leaving the wait at different times
      int ready = 0;
      if (lane == 0) ready = mbar_wait(tfull, (uint32_t)l & 1u, a.err, stop) ? 1 : 0;
      ready = __shfl_sync(0xffffffffu, ready, 0);
      __syncwarp();
      if (ready) {
        tc_fence_after();
        if (q * 32 < rows) {
          for (int c = 0; c < a.Nt; c += 32) {
            float v[32];
            tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)c, v);
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (c + i < a.Nt) stg[(c + i) * 128 + q * 32 + lane] = v[i];
          }
        }
        tc_fence_before();
      }
    }
    __syncthreads();
    // shared -> global by every thread, 16-byte stores: a warp instruction writes 32 x 4
    // consecutive rows of one tap (a few stores per thread instead of one per tap and row)
    {
      const int r4n = (rows + 3) / 4;
      const int ntaps = min(a.Nt, a.P - nt * a.Nt);
      float* dst0 = part + ((size_t)ks * a.P + nt * a.Nt) * a.Mp + rt * 128;
      for (int e = tid; e < ntaps * 32; e += kThreads) {
        const int tap = e >> 5, r4 = e & 31;
        if (r4 < r4n)
          __stcg(reinterpret_cast<float4*>(dst0 + (size_t)tap * a.Mp + r4 * 4),
                 *reinterpret_cast<const float4*>(stg + tap * 128 + r4 * 4));
      }
      // the next layer's TMA writes into this shared memory after the barriers
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (!group_barrier(&a.bar[0], (unsigned)(l + 1), gridDim.x, a.err, stop)) break;

    // ---- B. sum over the K-slices, normalise, mix
    {
      const int g_lo = kb0 * 4, ng = (kb1 - kb0) * 4;
      const int my_ng = (ng - nt + a.NT - 1) / a.NT;  // groups g_lo + nt, g_lo + nt + NT, ...
      const int items = rows * my_ng;
      const size_t sstride = (size_t)a.P * a.Mp;
      for (int it = tid; it < items; it += kThreads) {
        const int r = it % rows, gi = it / rows;
        const int g = g_lo + nt + gi * a.NT;
        const int row = rt * 128 + r;
        const int c0 = g * 16;
        // the rows' channels first, so their loads are in flight with the partials'
        const uint4* cur = reinterpret_cast<const uint4*>(xin + (size_t)row * a.H + c0);
        uint4 cv[2] = {__ldcg(cur), __ldcg(cur + 1)};
        uint4 pv[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
        if (row % a.T != 0) {
          pv[0] = __ldcg(cur - a.H / 8);  // the previous row
          pv[1] = __ldcg(cur - a.H / 8 + 1);
        }
        const float* p0 = part + (size_t)(2 * g) * a.Mp + row;
        // the partials of up to kC K-slices are loaded before any is added (one L2 round trip
        // for every plan up to kC slices); they are added in slice order
        float s0 = 0.f, s1 = 0.f;
        for (int sb = 0; sb < a.KS; sb += kC) {
          float v0[kC], v1[kC];
#pragma unroll
          for (int j = 0; j < kC; ++j) {
            if (sb + j < a.KS) {
              v0[j] = __ldcg(p0 + (size_t)(sb + j) * sstride);
              v1[j] = __ldcg(p0 + (size_t)(sb + j) * sstride + a.Mp);
            }
          }
#pragma unroll
          for (int j = 0; j < kC; ++j) {
            if (sb + j < a.KS) {
              s0 += v0[j];
              s1 += v1[j];
            }
          }
        }
        float wa, wb;
        if (a.raw) {
          wa = s0;
          wb = s1;
        } else {
          const float mx = fmaxf(s0, s1);
          const float e0 = expf(s0 - mx), e1 = expf(s1 - mx);
          const float inv = 1.f / (e0 + e1);
          wa = e0 * inv;
          wb = e1 * inv;
        }
        uint4 out[2];
        const __nv_bfloat162* c2 = reinterpret_cast<const __nv_bfloat162*>(cv);
        const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(pv);
        __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(out);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float2 cf = __bfloat1622float2(c2[k]);
          const float2 pf = __bfloat1622float2(p2[k]);
          o2[k] = __floats2bfloat162_rn(fmaf(wa, pf.x, wb * cf.x), fmaf(wa, pf.y, wb * cf.y));
        }
        uint4* dst = reinterpret_cast<uint4*>(xout + (size_t)row * a.H + c0);
        dst[0] = out[0];
        dst[1] = out[1];
      }
    }
    if (l + 1 < a.NL && !group_barrier(&a.bar[1 + sib], (unsigned)(l + 1), (unsigned)a.NT, a.err, stop)) break;
  }

  // ---- exit: no copy may still be landing and no MMA may still be running
  __syncthreads();
  if (warp == 0 && lane == 0) {
    for (int i = *consumed_s; i < issued; ++i)
      if (!mbar_wait(&full[i % kStages], (uint32_t)(i / kStages) & 1u, a.err, nullptr)) break;
  }
  if (warp == 1) {
    if (lane == 0) {
      umma_commit(drain);
      mbar_wait(drain, 0, a.err, nullptr);
    }
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, tmem_cols);
  }
}

size_t splitk_smem(int Nt) {
  const size_t b = ((size_t)Nt * 128 + 1023) & ~size_t(1023);
  return 1024 /*align*/ + 1024 /*barriers*/ + (size_t)kStages * (kABytes + b);
}
}  // namespace

bool conv_splitk_plan(int M, int H, int NL, int sms, ConvSplitPlan* out) {
  if (H % 64 != 0 || M < 1 || NL < 1 || sms < 1) return false;
  const int P = H / 8;
  const int NT = (P + kMaxTile - 1) / kMaxTile;
  const int Nt = (((P + NT - 1) / NT) + 15) / 16 * 16;
  const int RT = (M + 127) / 128;
  if (RT * NT > sms) return false;
  int KS = sms / (RT * NT);
  if (KS > H / 64) KS = H / 64;
  if (1 + RT * KS > 1024) return false;  // barrier counters in the workspace
  out->RT = RT;
  out->NT = NT;
  out->KS = KS;
  out->Nt = Nt;
  out->a_tail_rows = (M % 128 == 0) ? 128 : ((M % 128 + 7) / 8) * 8;
  out->grid = RT * NT * KS;
  out->smem = splitk_smem(Nt);
  out->Mp = (M + 3) / 4 * 4;
  out->part_bytes = 2 * (size_t)KS * P * out->Mp * sizeof(float);
  return true;
}

cudaError_t launch_conv_splitk(const ConvSplitPlan& pl, const CUtensorMap* maps, const void* x, void* buf0,
                               void* buf1, void* z, float* part, int M, int H, int T, int NL, int raw,
                               unsigned* bar_counts, int32_t* err, cudaStream_t s) {
  static unsigned char smem_done[64];
  cudaError_t e = smem_opt_in(reinterpret_cast<const void*>(conv_splitk_kernel), smem_done);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(bar_counts, 0, sizeof(unsigned) * (1 + (size_t)pl.RT * pl.KS), s);
  if (e != cudaSuccess) return e;
  SplitArgs a;
  a.M = M;
  a.H = H;
  a.T = T;
  a.NL = NL;
  a.raw = raw;
  a.P = H / 8;
  a.RT = pl.RT;
  a.NT = pl.NT;
  a.KS = pl.KS;
  a.Nt = pl.Nt;
  a.a_tail_rows = pl.a_tail_rows;
  a.Mp = pl.Mp;
  a.part = part;
  a.x0 = reinterpret_cast<const __nv_bfloat16*>(x);
  a.buf0 = reinterpret_cast<__nv_bfloat16*>(buf0);
  a.buf1 = reinterpret_cast<__nv_bfloat16*>(buf1);
  a.z = reinterpret_cast<__nv_bfloat16*>(z);
  a.bar = bar_counts;
  a.err = err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, conv_splitk_kernel, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], maps[6],
                         a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace df
