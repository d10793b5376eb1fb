// All conv layers in one cooperative launch for larger row counts (bf16): the projection to
// the taps is split along the hidden dimension and runs on the tensor cores (tcgen05).
//
// Per layer l the taps are P[m][q] = x_l[m] . W_l[q] for the P = H/8 projection rows q
// (two per channel group of 16). CTA (rt, nt, ks) owns row tile rt (128 rows), tap tile nt
// (Nt projection rows) and K-slice ks (a range of 64-channel blocks):
//   A. TMA streams its (x rows, W rows) blocks of the slice through a 5-stage shared-memory
//      ring (128-byte swizzle, K-major); one thread issues tcgen05.mma (M = 128, N = Nt,
//      K = 16) into a TMEM accumulator; four epilogue warps (thread = TMEM lane = row) stage
//      the fp32 partial taps in the idle operand ring as [tap][row], and one TMA store writes
//      them to plane ks of [ks][q][m] (clipped at the tensor's edges). Partials alternate
//      between two sets of planes by layer parity.
//   grid barrier: every partial of the layer is written.
//   B. The NT CTAs sharing (rt, ks) split the channel groups of the slice into contiguous
//      ranges. In chunks that fit the idle ring, one 3-D TMA load brings the chunk's taps of
//      every K-slice ([ks][tap][row]), and 2-D loads the tile's rows of the chunk's channels
//      (when a CTA's groups make one chunk and shared memory has room, those row boxes have
//      their own region and load while phase A runs: this CTA wrote them itself in the
//      previous layer). From shared memory a thread per (row, group) sums the two taps over
//      the K-slices in slice order, normalises them (softmax over the pair, unless raw), and
//      writes y[m, c] = a * x_l[m-1, c] + b * x_l[m, c] for the group's 16 channels
//      (x[-1] = 0 at each block start; the row above the tile, another tile's, comes from
//      global memory into shared memory while the boxes land), rounded to bf16.
//   sibling barrier: the NT CTAs of (rt, ks) wait for each other, since the next layer's A
//      phase of each of them reads every channel of the slice for the tile's rows.
// Each CTA reads only its K-slice of the rows and of its tap rows, so the per-layer traffic
// is (M + P) * H * 2 bytes spread over the grid, plus the partial taps through L2, moved by
// the copy engine both ways; the older chain kernel, where each CTA reads every hidden channel
// of its rows, suits small M only.
// Every wait is bounded; on timeout the kernel sets DFLASH2_DEVERR_WAIT_TIMEOUT, lets copies
// in flight land, frees TMEM and returns.
#include <cuda_bf16.h>
#include <math.h>

#include "../../include/dflash2.h"
#include "grid_sync.cuh"
#include "kernels.h"
#include "launch_util.h"
#include "ptx.cuh"
#include "tma_bulk.cuh"

namespace df {

namespace {
constexpr int kThreads = 256;
constexpr int kStages = 5;
constexpr uint32_t kABytes = 128 * 64 * 2;  // A region of a stage: the MMA reads 128 rows
constexpr int kMaxTile = 160;                // widest tap tile
constexpr int kMaxSmem = 227 * 1024;         // dynamic shared memory a CTA may take

struct SplitArgs {
  int M, H, T, NL, raw;
  int P;             // projection rows (taps) per layer = H / 8
  int RT, NT, KS;    // row tiles, tap tiles, K-slices
  int Nt;            // projection rows per tap tile (multiple of 16)
  int a_tail_rows;   // rows of the last row tile's TMA box (multiple of 8)
  int Mp;            // rows of a partial-tap plane (M rounded up to 4)
  int gc;            // channel groups per mix chunk
  int br;            // rows of the partial-tap and row boxes: 128, or the rows of a single tile
  int xb, nxs;       // channels per row box of the mix (br rows), row boxes per chunk
  uint32_t pbox_bytes, xbox_bytes;  // a chunk's partial-tap box, one row box
  int x_early;       // the row boxes have their own region and are loaded as the layer starts
  uint32_t xoff;     // byte offset of the row boxes from the ring's start
  uint32_t aboff;    // byte offset of the chunk's row above the tile ([gc][16] bf16) from the ring's start
  const __nv_bfloat16* x0;
  __nv_bfloat16* buf0;
  __nv_bfloat16* buf1;
  __nv_bfloat16* z;
  unsigned* bar;     // [0]: grid barrier; [1 + rt * KS + ks]: barrier of the NT CTAs of (rt, ks)
  int32_t* err;
};

__global__ void __launch_bounds__(kThreads, 1)
    conv_splitk_kernel(const __grid_constant__ CUtensorMap map_x0, const __grid_constant__ CUtensorMap map_x0t,
                       const __grid_constant__ CUtensorMap map_b0, const __grid_constant__ CUtensorMap map_b0t,
                       const __grid_constant__ CUtensorMap map_b1, const __grid_constant__ CUtensorMap map_b1t,
                       const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_pst,
                       const __grid_constant__ CUtensorMap map_pld, const __grid_constant__ CUtensorMap map_r0,
                       const __grid_constant__ CUtensorMap map_r1, const __grid_constant__ CUtensorMap map_r2,
                       const SplitArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(base);
  uint64_t* empty = full + kStages;
  uint64_t* tfull = empty + kStages;
  uint64_t* drain = tfull + 1;
  uint64_t* mixfull = drain + 1;  // a mix chunk's boxes have landed
  uint64_t* rowsfull = mixfull + 1;  // the layer's row boxes have landed (x_early)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(rowsfull + 1);
  volatile int* stop = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* consumed_s = stop + 1;  // ring loads the MMA thread has waited for
  uint8_t* ring = base + 1024;
  float* stg = reinterpret_cast<float*>(ring);  // [Nt][br] fp32 tile of partials, in the idle ring

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

  pdl_launch_dependents();  // the LM head may start its prologue as SMs free up
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(drain, 1);
    mbar_init(mixfull, 1);
    mbar_init(rowsfull, 1);
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
  int issued = 0;     // producer thread: ring loads issued
  uint32_t mixes = 0; // thread 0: mix chunks whose loads were issued
  int rows_loaded = 0;  // thread 0: layers whose row boxes were loaded early
  // this CTA's contiguous range of the slice's channel groups in the mix
  const int g0 = kb0 * 4 + nt * ((kb1 - kb0) * 4) / a.NT, g1 = kb0 * 4 + (nt + 1) * ((kb1 - kb0) * 4) / a.NT;
  const uint32_t xbox_tx = (uint32_t)(a.nxs * a.br * a.xb * 2);  // bytes of a chunk's row boxes
  const uint32_t pbox_tx = (uint32_t)(a.br * 2 * a.gc * a.KS * 4);  // bytes of a chunk's partial-tap box
  uint8_t* xboxes = ring + a.xoff;                                  // [nxs][br][xb] bf16
  uint4* above = reinterpret_cast<uint4*>(ring + a.aboff);       // [gc][2] the row above the tile
  for (int l = 0; l < a.NL; ++l) {
    const CUtensorMap* mx = l == 0 ? (tail ? &map_x0t : &map_x0)
                                   : ((l - 1) % 2 == 0 ? (tail ? &map_b0t : &map_b0) : (tail ? &map_b1t : &map_b1));
    const CUtensorMap* mrows = l == 0 ? &map_r0 : ((l - 1) % 2 == 0 ? &map_r1 : &map_r2);  // x_l, row boxes
    const __nv_bfloat16* xin = l == 0 ? a.x0 : ((l - 1) % 2 == 0 ? a.buf0 : a.buf1);
    __nv_bfloat16* xout = l == a.NL - 1 ? a.z : (l % 2 == 0 ? a.buf0 : a.buf1);
    const int pset = (l & 1) * a.KS;  // this layer's set of partial-tap planes

    // ---- A. partial taps of the K-slice
    if (warp == 0) {
      if (lane == 0) {
        // the rows were written by other CTAs' generic stores before the last barrier, and
        // the ring held the previous layer's staged partials (generic accesses)
        if (l > 0) {
          asm volatile("fence.proxy.async.global;" ::: "memory");
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
        if (a.x_early && g1 > g0) {  // (the mix waits for these rows only when it has groups)
          // the mix's rows of this tile for this CTA's groups: this CTA wrote them in the
          // previous layer (the row above the tile, another tile's, is read in the mix itself)
          mbar_arrive_expect_tx(rowsfull, xbox_tx);
          for (int j = 0; j < a.nxs; ++j)
            tma_load_2d(xboxes + (size_t)j * a.xbox_bytes, mrows, rowsfull, g0 * 16 + j * a.xb, rt * 128,
                        l2_policy_evict_first());
          ++rows_loaded;
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
              if (c + i < a.Nt && q * 32 + lane < a.br) stg[(c + i) * a.br + q * 32 + lane] = v[i];
          }
        }
        // generic writes that the TMA store below reads
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        tc_fence_before();
      }
    }
    __syncthreads();
    // staged partials -> plane ks of this layer's set: one TMA store of the [Nt][br] tile
    // (taps past P and rows past the plane are not written); complete before the release
    if (tid == 0 && *stop == 0) {
      tma_store_3d(&map_pst, stg, rt * 128, nt * a.Nt, pset + ks);
      bulk_commit();
      bulk_wait_all();
      asm volatile("fence.proxy.async.global;" ::: "memory");
    }
    if (!group_barrier(&a.bar[0], (unsigned)(l + 1), gridDim.x, a.err, stop)) break;

    // ---- B. sum over the K-slices, normalise, mix: this CTA's groups [g0, g1) in chunks of
    //      a.gc groups; the chunk's partial taps (and, unless loaded early, its row boxes) are
    //      staged in the idle ring by TMA
    {
      const float* pbox = reinterpret_cast<const float*>(ring);  // [KS][2 gc][br] fp32
      const int kstride = 2 * a.gc * a.br;
      bool ok = true;
      for (int c0 = g0; c0 < g1; c0 += a.gc) {
        const int gn = min(a.gc, g1 - c0);
        if (tid == 0) {
          // the planes were written by other CTAs' TMA stores and the rows by generic stores;
          // the ring last held generic accesses (the staged partials, the previous chunk)
          asm volatile("fence.proxy.async.global;" ::: "memory");
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          mbar_arrive_expect_tx(mixfull, pbox_tx + (a.x_early ? 0u : xbox_tx));
          tma_load_3d(ring, &map_pld, mixfull, rt * 128, 2 * c0, pset);
          if (!a.x_early)
            for (int j = 0; j < a.nxs; ++j)
              tma_load_2d(xboxes + (size_t)j * a.xbox_bytes, mrows, mixfull, c0 * 16 + j * a.xb, rt * 128,
                          l2_policy_evict_first());
          ++mixes;
        }
        // the row above the tile (another tile's, written before the grid barrier) for the
        // chunk's groups, one 16-byte load per thread while the boxes land; zero where the
        // tile's first row starts a block
        if (tid < 2 * gn) {
          const int above_row = rt * 128 - 1;
          uint4 v = make_uint4(0, 0, 0, 0);
          if (above_row >= 0 && (above_row + 1) % a.T != 0)
            v = __ldcg(reinterpret_cast<const uint4*>(xin + (size_t)above_row * a.H + (c0 + (tid >> 1)) * 16) +
                       (tid & 1));
          above[tid] = v;
        }
        if (tid == 0 && mbar_wait(mixfull, (mixes - 1) & 1u, a.err, stop) && a.x_early && c0 == g0)
          mbar_wait(rowsfull, (uint32_t)(rows_loaded - 1) & 1u, a.err, stop);
        __syncthreads();
        if (*stop) {
          ok = false;
          break;
        }
        const int items = rows * gn;
        for (int it = tid; it < items; it += kThreads) {
          const int r = it % rows, gi = it / rows;
          const int row = rt * 128 + r;
          // the two taps summed over the K-slices in slice order, loads batched
          const float* p0 = pbox + (size_t)(2 * gi) * a.br + r;
          float s0 = 0.f, s1 = 0.f;
          int k = 0;
          for (; k + 8 <= a.KS; k += 8) {
            float v0[8], v1[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              v0[j] = p0[(size_t)(k + j) * kstride];
              v1[j] = p0[(size_t)(k + j) * kstride + a.br];
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              s0 += v0[j];
              s1 += v1[j];
            }
          }
          for (; k < a.KS; ++k) {
            s0 += p0[(size_t)k * kstride];
            s1 += p0[(size_t)k * kstride + a.br];
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
          // box row r is row `row`; the previous row is box row r - 1, or for the tile's first
          // row the last row of the tile above (x[-1] = 0 at each block start)
          const int sub = (gi * 16) / a.xb, cc = (gi * 16) % a.xb;  // the boxes start at group c0
          const __nv_bfloat16* xs = reinterpret_cast<const __nv_bfloat16*>(xboxes + (size_t)sub * a.xbox_bytes);
          const uint4* cur = reinterpret_cast<const uint4*>(xs + (size_t)r * a.xb + cc);
          uint4 cv[2] = {cur[0], cur[1]};
          uint4 pv[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
          if (row % a.T != 0) {
            const uint4* prv = r > 0 ? reinterpret_cast<const uint4*>(xs + (size_t)(r - 1) * a.xb + cc) : above + 2 * gi;
            pv[0] = prv[0];
            pv[1] = prv[1];
          }
          uint4 out[2];
          const __nv_bfloat162* c2 = reinterpret_cast<const __nv_bfloat162*>(cv);
          const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(pv);
          __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(out);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float2 cf = __bfloat1622float2(c2[q]);
            const float2 pf = __bfloat1622float2(p2[q]);
            o2[q] = __floats2bfloat162_rn(fmaf(wa, pf.x, wb * cf.x), fmaf(wa, pf.y, wb * cf.y));
          }
          uint4* dst = reinterpret_cast<uint4*>(xout + (size_t)row * a.H + (c0 + gi) * 16);
          dst[0] = out[0];
          dst[1] = out[1];
        }
        __syncthreads();  // the next chunk's copies overwrite the boxes
      }
      if (!ok) break;
    }
    if (l + 1 < a.NL && !group_barrier(&a.bar[1 + sib], (unsigned)(l + 1), (unsigned)a.NT, a.err, stop)) break;
  }

  // ---- exit: no copy may still be landing and no MMA may still be running
  __syncthreads();
  if (warp == 0 && lane == 0) {
    for (int i = *consumed_s; i < issued; ++i)
      if (!mbar_wait(&full[i % kStages], (uint32_t)(i / kStages) & 1u, a.err, nullptr)) break;
    if (mixes > 0) mbar_wait(mixfull, (mixes - 1) & 1u, a.err, nullptr);  // the last mix chunk's copies
    if (rows_loaded > 0) mbar_wait(rowsfull, (uint32_t)(rows_loaded - 1) & 1u, a.err, nullptr);
    bulk_wait_all();                                                     // and the partials' store
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
  // box rows: a single row tile's (a multiple of 8), else 128 (the last tile's box reads zeros
  // past the tensor)
  const int br = RT == 1 ? out->a_tail_rows : 128;
  out->br = br;
  // mix chunks: the most channel groups whose partial taps (2 per group, every K-slice, br rows
  // of fp32) and row boxes (br rows of 16 channels) fit the operand ring
  const size_t ring = (size_t)kStages * (kABytes + ((Nt * 128 + 1023) & ~1023));
  const int ng_max = 4 * ((H / 64 + KS - 1) / KS);  // groups of the widest K-slice
  const int g_cta = (ng_max + NT - 1) / NT;          // groups of one CTA, at most
  int gc = g_cta < 128 ? g_cta : 128;
  for (; gc >= 1; --gc) {
    const int xb = 16 * (gc < 8 ? gc : 8);
    const int nxs = (16 * gc + xb - 1) / xb;
    const size_t xbox = (size_t)br * xb * 2;                                // a multiple of 256
    const size_t pbox = ((size_t)br * 2 * gc * KS * 4 + 127) & ~size_t(127);  // 128-B aligned
    if (pbox + nxs * xbox <= ring) {
      out->gc = gc;
      out->xb = xb;
      out->nxs = nxs;
      out->pbox_bytes = (uint32_t)pbox;
      out->xbox_bytes = (uint32_t)xbox;
      // one chunk per CTA and room past the ring: the row boxes get their own region, loaded
      // while the layer's taps are contracted
      const size_t above = ((size_t)gc * 32 + 127) & ~size_t(127);  // the row above the tile
      out->x_early = gc == g_cta && out->smem + nxs * xbox + above <= (size_t)kMaxSmem;
      out->xoff = out->x_early ? (uint32_t)ring : (uint32_t)pbox;
      if (out->x_early) out->smem += nxs * xbox;
      out->aboff = (uint32_t)(out->smem - 2048);  // past the ring and the early row boxes
      out->smem += above;
      return out->smem <= (size_t)kMaxSmem;
    }
  }
  return false;
}

cudaError_t launch_conv_splitk(const ConvSplitPlan& pl, const CUtensorMap* maps, const void* x, void* buf0,
                               void* buf1, void* z, int M, int H, int T, int NL, int raw, unsigned* bar_counts,
                               int32_t* err, cudaStream_t s) {
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
  a.gc = pl.gc;
  a.br = pl.br;
  a.xb = pl.xb;
  a.nxs = pl.nxs;
  a.pbox_bytes = pl.pbox_bytes;
  a.xbox_bytes = pl.xbox_bytes;
  a.x_early = pl.x_early;
  a.xoff = pl.xoff;
  a.aboff = pl.aboff;
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
                         maps[7], maps[8], maps[9], maps[10], maps[11], a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace df
