// Transition tiles and the walk from the anchor, one CTA (8 warps) per sequence; and the
// same walk fused with the top-K merge for the whole-tail call.
//
// For slot boundary t the previous candidates are the anchor (t = 0, repeated K times) or
// slot t-1's candidates; the current ones are slot t's. Warp t % 8 gathers the 16 U-rows
// (previous) and 16 V-rows (current) with 16-byte cp.async copies (all in flight at once)
// into padded shared memory, in chunks of up to 256 columns, and forms the 16x16 tile
// tau_t(i, j) = <U[prev_i], V[cur_j]> with mma.sync m16n8k16 (bf16 in, fp32 accumulate).
// Warp 0 then runs the recursion over the tiles: lane j holds delta(j); each step takes,
// for every j, the max over i of delta(i) + tau(i, j) with the lowest i on ties, adds
// lp_t(j), and keeps the back-pointer; a shuffle arg-max (lowest index on ties) picks the
// final state and lane 0 reads the path back.
//
// Sampling (optional, temperature > 0): instead of the best path, warp 0 draws one from
// P(path) ~ exp(score / temperature) by forward filtering (log-sum-exp over the previous
// candidates) and backward inverse-CDF draws on the caller's uniforms; or, with the greedy walk,
// draws each step from the softmax of that step's scores given the previous draw.
//
// Context gate (optional): tau_t(i, j) = sum_r U[prev_i][r] g_t[r] V[cur_j][r] with g_t the gate
// of slot t (fp32, [B*T, R]). The warp that builds tile t forms V[cur_j][r] g_t[r] in fp32 and
// splits it into two bf16 parts, hi = bf16(v g) and lo = bf16(v g - hi) (together within about
// 2^-17 of the fp32 product), and contracts U with both (fp32 accumulation); fp32 embeddings keep
// the product in fp32.
//
// Score on the raw logits (optional, whole-tail calls): the Viterbi / greedy score is reported
// as sum_t logit_t(j_t) + transitions, i.e. the log-softmax score plus the slots' lse.
//
// Slots and rows: a sequence has T slots; its candidate (or LM-head) rows are rows_per_seq
// apart and slot t is row first + t of them (first = 1 when row 0 of each block is the
// anchor's position). Outputs are per slot.
//
// The fused kernel first merges the sequence's T slot rows (warp t % 8 takes slot t): the row's
// per-partition top-16 lists and (max, sum) pairs are staged with cp.async, lse is reduced
// across the warp and the K best candidates are picked by the warp-wide merge; they stay in
// shared memory for the walk (and are also written out).
#include <cuda_bf16.h>

#include "../../include/dflash2.h"
#include "kernels.h"
#include "launch_util.h"
#include "ptx.cuh"
#include "select.cuh"

namespace df {

namespace {
constexpr int kWarps = 8;
constexpr int kKP = 16;         // candidate slots per tile (K padded to 16)
constexpr int kRChunk = 256;    // embedding columns staged per pass
constexpr int kRowPad = kRChunk + 8;  // bf16 per staged row: 528 B (33 x 16 B), keeps ldmatrix conflict-free
constexpr int kMaxT = 32;

struct SmemWalk {
  int32_t ids[kMaxT][kKP];
  float lp[kMaxT][kKP];
  float tau[kMaxT][kKP][kKP];
  float alpha[kMaxT][kKP];  // sampling: forward log-weights
  float lse[kMaxT];         // each slot's lse (for the score on raw logits)
  int8_t bp[kMaxT][kKP];
  int32_t anchor;
  int32_t dry_ids[kMaxT];   // outputs of the fused kernel's dry run (discarded)
  int32_t dry_idx[kMaxT];
  float dry_score;
};

// Sampling parameters of the walk: u == nullptr is the Viterbi / greedy walk; otherwise a path
// is drawn at temperature 1 / inv_temp with the uniforms u [B, T] (slot t's draw in u[b, t]).
struct SampleArgs {
  const float* u;
  float inv_temp;
};

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ int32_t clamp_id(int32_t id, int vocab, int32_t* err, int bit) {
  if (id < 0 || id >= vocab) {
    if (err) atomicOr(err, bit);
    return id < 0 ? 0 : vocab - 1;
  }
  return id;
}

// 16 x 16 products of the rows staged in stA (16 x rc) and stB (16 x rc), accumulated into acc.
__device__ __forceinline__ void tile_mma(const __nv_bfloat16* stA, const __nv_bfloat16* stB, int rc,
                                         float (&acc)[2][4]) {
  const int lane = threadIdx.x & 31;
  for (int k0 = 0; k0 < rc; k0 += 16) {
    uint32_t a[4], b[4];
    {
      const int r = (lane & 7) + ((lane >> 3) & 1) * 8;
      const int c = k0 + (lane >> 4) * 8;
      ldmatrix_x4(static_cast<uint32_t>(__cvta_generic_to_shared(stA + r * kRowPad + c)), a[0], a[1], a[2], a[3]);
    }
    {
      const int n = (lane & 7) + (lane >> 4) * 8;
      const int c = k0 + ((lane >> 3) & 1) * 8;
      ldmatrix_x4(static_cast<uint32_t>(__cvta_generic_to_shared(stB + n * kRowPad + c)), b[0], b[1], b[2], b[3]);
    }
    mma_bf16_16816(acc[0], a, b[0], b[1]);
    mma_bf16_16816(acc[1], a, b[2], b[3]);
  }
}

__device__ __forceinline__ void store_tau(const float (&acc)[2][4], float (&tau)[kKP][kKP]) {
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, c2 = (lane & 3) * 2;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    tau[g][nt * 8 + c2] = acc[nt][0];
    tau[g][nt * 8 + c2 + 1] = acc[nt][1];
    tau[g + 8][nt * 8 + c2] = acc[nt][2];
    tau[g + 8][nt * 8 + c2 + 1] = acc[nt][3];
  }
}

// Gated 16 x 16 products: acc += stA * (stB (.) g)^T over rc columns (g: the gate from the first
// staged column). Per 64-column chunk each lane forms V g in fp32 for its pieces and splits it
// into hi = bf16(V g) and lo = bf16(V g - hi); hi is written over the staged V rows and
// contracted, then lo, so no extra shared memory is needed. The staged V rows are consumed.
__device__ __forceinline__ void tile_mma_gated(const __nv_bfloat16* stA, __nv_bfloat16* stB, int rc, const float* g,
                                               float (&acc)[2][4]) {
  const int lane = threadIdx.x & 31;
  for (int c0 = 0; c0 < rc; c0 += 64) {
    const int cw = min(64, rc - c0);  // a multiple of 16
    const int vpr = cw / 8;           // 16-byte pieces per row in this chunk
    uint4 lo[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int v = lane + 32 * i;
      if (v < kKP * vpr) {
        const int row = v / vpr, cv = v % vpr;
        uint4* p = reinterpret_cast<uint4*>(stB + row * kRowPad + c0 + cv * 8);
        const float4 g0 = *reinterpret_cast<const float4*>(g + c0 + cv * 8);  // global or staged in shared memory
        const float4 g1 = *reinterpret_cast<const float4*>(g + c0 + cv * 8 + 4);
        const float gg[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
        uint4 x = *p;
        __nv_bfloat162* x2 = reinterpret_cast<__nv_bfloat162*>(&x);
        __nv_bfloat162* l2 = reinterpret_cast<__nv_bfloat162*>(&lo[i]);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 f = __bfloat1622float2(x2[k]);
          const float p0 = f.x * gg[2 * k], p1 = f.y * gg[2 * k + 1];
          const __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
          const float2 hf = __bfloat1622float2(h);
          l2[k] = __floats2bfloat162_rn(p0 - hf.x, p1 - hf.y);
          x2[k] = h;
        }
        *p = x;
      }
    }
    __syncwarp();
    tile_mma(stA + c0, stB + c0, cw, acc);
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int v = lane + 32 * i;
      if (v < kKP * vpr) {
        const int row = v / vpr, cv = v % vpr;
        *reinterpret_cast<uint4*>(stB + row * kRowPad + c0 + cv * 8) = lo[i];
      }
    }
    __syncwarp();
    tile_mma(stA + c0, stB + c0, cw, acc);
    __syncwarp();
  }
}

// Issues (without waiting) the 16-byte copies of rows ids[0..15] of E (R <= kRChunk columns)
// into the 16 padded rows at st.
__device__ __forceinline__ void gather_rows(const __nv_bfloat16* __restrict__ E, int R, const int32_t* ids,
                                            __nv_bfloat16* st) {
  const int lane = threadIdx.x & 31;
  const int vec_per_row = R / 8;
  for (int v = lane; v < kKP * vec_per_row; v += 32) {
    const int row = v / vec_per_row, cv = v % vec_per_row;
    cp_async16(st + row * kRowPad + cv * 8, E + (size_t)ids[row] * R + cv * 8);
  }
}

// tau tile for one boundary, bf16 embeddings, on one warp.
__device__ void tile_bf16(const __nv_bfloat16* __restrict__ U, const __nv_bfloat16* __restrict__ V, int R,
                          const int32_t* prev, const int32_t* cur, const float* g, __nv_bfloat16* stA,
                          __nv_bfloat16* stB, float (&tau)[kKP][kKP]) {
  const int lane = threadIdx.x & 31;
  float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  for (int r0 = 0; r0 < R; r0 += kRChunk) {
    const int rc = min(kRChunk, R - r0);  // multiple of 16
    const int vec_per_row = rc / 8;       // 16-byte vectors per staged row
    __syncwarp();
    // every 16-byte piece of the 32 gathered rows is issued before any is waited for
    for (int v = lane; v < kKP * vec_per_row; v += 32) {
      const int row = v / vec_per_row, cv = v % vec_per_row;
      cp_async16(stA + row * kRowPad + cv * 8, U + (size_t)prev[row] * R + r0 + cv * 8);
      cp_async16(stB + row * kRowPad + cv * 8, V + (size_t)cur[row] * R + r0 + cv * 8);
    }
    cp_async_commit();
    cp_async_wait_all();
    __syncwarp();
    if (g) tile_mma_gated(stA, stB, rc, g + r0, acc);
    else tile_mma(stA, stB, rc, acc);
  }
  store_tau(acc, tau);
}

// tau tile for one boundary, fp32 embeddings (small instantiation): 8 entries per lane.
__device__ void tile_f32(const float* __restrict__ U, const float* __restrict__ V, int R, const int32_t* prev,
                         const int32_t* cur, const float* g, float (&tau)[kKP][kKP]) {
  const int lane = threadIdx.x & 31;
  for (int e = lane; e < kKP * kKP; e += 32) {
    const int i = e / kKP, j = e % kKP;
    const float* u = U + (size_t)prev[i] * R;
    const float* v = V + (size_t)cur[j] * R;
    float s = 0.f;
    if (g)
      for (int r = 0; r < R; ++r) s = fmaf(u[r], v[r] * g[r], s);
    else
      for (int r = 0; r < R; ++r) s = fmaf(u[r], v[r], s);
    tau[i][j] = s;
  }
}

// Pads candidate slots K..15 of every slot with a valid id and -inf score (call after the
// real candidates are in sw, then __syncthreads).
__device__ void pad_candidates(SmemWalk& sw, int T, int K) {
  for (int e = threadIdx.x; e < T * kKP; e += blockDim.x) {
    const int t = e / kKP, j = e % kKP;
    if (j >= K) {
      sw.ids[t][j] = sw.ids[t][0];
      sw.lp[t][j] = -INFINITY;
    }
  }
}

// All T transition tiles of one sequence; warp w builds the tiles t = w, w + 8, ...
// gate_b: the sequence's gate rows [T, R] (nullptr: no gate).
template <bool kBf16>
__device__ void build_tiles(SmemWalk& sw, int T, int R, const void* Uv, const void* Vv, const float* gate_b,
                            __nv_bfloat16* stage) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __shared__ int32_t prev_s[kWarps][kKP];
  for (int t = warp; t < T; t += kWarps) {
    const int32_t* cur = sw.ids[t];
    // previous candidates of this boundary: the anchor for slot 0, else slot t-1's list
    if (lane < kKP) prev_s[warp][lane] = (t == 0) ? sw.anchor : sw.ids[t - 1][lane];
    __syncwarp();
    if constexpr (kBf16) {
      __nv_bfloat16* stA = stage + (size_t)warp * 2 * kKP * kRowPad;
      __nv_bfloat16* stB = stA + kKP * kRowPad;
      tile_bf16(reinterpret_cast<const __nv_bfloat16*>(Uv), reinterpret_cast<const __nv_bfloat16*>(Vv), R,
                prev_s[warp], cur, gate_b ? gate_b + (size_t)t * R : nullptr, stA, stB, sw.tau[t]);
    } else {
      tile_f32(reinterpret_cast<const float*>(Uv), reinterpret_cast<const float*>(Vv), R, prev_s[warp], cur,
               gate_b ? gate_b + (size_t)t * R : nullptr, sw.tau[t]);
    }
    __syncwarp();
  }
}

// One inverse-CDF draw on warp 0: lane i < K holds the log-weight lw (-inf elsewhere); returns
// the smallest index whose cumulative weight exceeds u times the total (index order), and the
// log of its probability. Every lane returns the same values.
__device__ __forceinline__ int draw_index(float lw, int K, float u, float& logp) {
  const int lane = threadIdx.x & 31;
  float m = lw;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const float w = lane < K ? expf(lw - m) : 0.f;
  float c = w;  // inclusive prefix sum over lanes
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, c, o);
    if (lane >= o) c += y;
  }
  const float total = __shfl_sync(0xffffffffu, c, 31);
  const uint32_t above = __ballot_sync(0xffffffffu, lane < K && c > u * total);
  const int k = above ? (__ffs(above) - 1) : K - 1;
  const float wk = __shfl_sync(0xffffffffu, w, k);
  logp = logf(wk / total);
  return k;
}

// Forward filtering and backward sampling on warp 0 (fp32): P(path) = exp(score(path) * inv_temp)
// / Z. alpha_0(j) = (lp_0(j) + tau_0(0, j)) inv_temp; alpha_t(j) = lp_t(j) inv_temp +
// logsumexp_i (alpha_{t-1}(i) + tau_t(i, j) inv_temp). Then j_{T-1} ~ alpha_{T-1} and
// j_{t-1} ~ alpha_{t-1}(i) + tau_t(i, j_t) inv_temp, each by inverse CDF on u[b, t]. score[b]
// receives log P(path).
__device__ void sample_warp0(SmemWalk& sw, int b, int T, int K, const SampleArgs& sa, int32_t* __restrict__ path_ids,
                             int32_t* __restrict__ path_idx, float* __restrict__ score) {
  const int lane = threadIdx.x & 31;
  const int j = lane;
  const bool live = j < K;
  const float it = sa.inv_temp;
  __shared__ float ash[kKP];
  float a = live ? (sw.lp[0][j] + sw.tau[0][0][j]) * it : -INFINITY;
  if (lane < kKP) sw.alpha[0][lane] = a;
  for (int t = 1; t < T; ++t) {
    if (lane < kKP) ash[lane] = a;
    __syncwarp();
    if (live) {
      float m = -INFINITY;
      for (int i = 0; i < K; ++i) m = fmaxf(m, ash[i] + sw.tau[t][i][j] * it);
      float s = 0.f;
      for (int i = 0; i < K; ++i) s += expf(ash[i] + sw.tau[t][i][j] * it - m);
      a = sw.lp[t][j] * it + (m + logf(s));
    }
    if (lane < kKP) sw.alpha[t][lane] = a;
    __syncwarp();
  }
  const float* u = sa.u + (size_t)b * T;
  float lp_sum = 0.f, lpk;
  int cj = draw_index(live ? sw.alpha[T - 1][j] : -INFINITY, K, u[T - 1], lpk);
  lp_sum += lpk;
  if (lane == 0) {
    path_idx[(size_t)b * T + T - 1] = cj;
    path_ids[(size_t)b * T + T - 1] = sw.ids[T - 1][cj];
  }
  for (int t = T - 1; t > 0; --t) {
    const float lw = live ? sw.alpha[t - 1][j] + sw.tau[t][j][cj] * it : -INFINITY;
    cj = draw_index(lw, K, u[t - 1], lpk);
    lp_sum += lpk;
    if (lane == 0) {
      path_idx[(size_t)b * T + t - 1] = cj;
      path_ids[(size_t)b * T + t - 1] = sw.ids[t - 1][cj];
    }
  }
  if (lane == 0) score[b] = lp_sum;
}

// Per-step sampling along the greedy walk on warp 0: j_0 ~ softmax_j ((lp_0(j) + tau_0(0, j)) / T),
// j_t ~ softmax_j ((lp_t(j) + tau_t(j_{t-1}, j)) / T), each by inverse CDF on u[b, t]; score[b]
// receives the log-probability of the drawn path, sum_t log p_t(j_t).
__device__ void greedy_sample_warp0(SmemWalk& sw, int b, int T, int K, const SampleArgs& sa,
                                    int32_t* __restrict__ path_ids, int32_t* __restrict__ path_idx,
                                    float* __restrict__ score) {
  const int lane = threadIdx.x & 31;
  const bool live = lane < K;
  const float* u = sa.u + (size_t)b * T;
  float lp_sum = 0.f, lpk;
  int pj = 0;
  for (int t = 0; t < T; ++t) {
    const float lw = live ? (sw.lp[t][lane] + sw.tau[t][pj][lane]) * sa.inv_temp : -INFINITY;
    pj = draw_index(lw, K, u[t], lpk);
    lp_sum += lpk;
    if (lane == 0) {
      path_idx[(size_t)b * T + t] = pj;
      path_ids[(size_t)b * T + t] = sw.ids[t][pj];
    }
  }
  if (lane == 0) score[b] = lp_sum;
}

// Sum of the slots' lse, added to a Viterbi / greedy score reported on the raw logits.
__device__ __forceinline__ float lse_sum(const SmemWalk& sw, int T) {
  float s = 0.f;
  for (int t = 0; t < T; ++t) s += sw.lse[t];
  return s;
}

// The walk for sequence b on warp 0 (the other warps return before calling it).
__device__ __noinline__ void walk_warp0(SmemWalk& sw, int b, int T, int K, int flags, const SampleArgs& sa,
                           int32_t* __restrict__ path_ids, int32_t* __restrict__ path_idx,
                           float* __restrict__ score) {
  const int lane = threadIdx.x & 31;
  const int j = lane;
  const bool live = j < K;
  const bool greedy = (flags & kWalkFlagGreedy) != 0;
  if (sa.u) {
    if (greedy) greedy_sample_warp0(sw, b, T, K, sa, path_ids, path_idx, score);
    else sample_warp0(sw, b, T, K, sa, path_ids, path_idx, score);
  } else if (!greedy) {
    // Viterbi in fp32: delta_0 = lp_0 + tau_0(0, j); delta_t = lp_t + max_i (delta_{t-1}(i) + tau_t(i, j)).
    // Each step, lane j loads its column of tau_t into registers, receives delta(i) by shuffles
    // and takes the max over i as a tree on registers: the right operand replaces the left only
    // if strictly greater, so the lowest i wins ties (as a scan in i order with strict > would).
    // Candidates i >= K enter as -inf and are never chosen over a live one.
    float delta = live ? sw.lp[0][j] + sw.tau[0][0][j] : -INFINITY;
    const int jc = j & (kKP - 1);  // lanes past the candidates read a valid column, unused
    for (int t = 1; t < T; ++t) {
      float v[kKP];
      int ai[kKP];
#pragma unroll
      for (int i = 0; i < kKP; ++i) {
        const float tc = sw.tau[t][i][jc];
        const float di = __shfl_sync(0xffffffffu, delta, i);  // every lane, every i: no branch
        v[i] = i < K ? di + tc : -INFINITY;
        ai[i] = i;
      }
#pragma unroll
      for (int w = 1; w < kKP; w *= 2) {
#pragma unroll
        for (int a = 0; a < kKP; a += 2 * w) {
          if (v[a + w] > v[a]) {
            v[a] = v[a + w];
            ai[a] = ai[a + w];
          }
        }
      }
      if (live) {
        delta = sw.lp[t][j] + v[0];
        sw.bp[t][j] = (int8_t)ai[0];
      }
    }
    __syncwarp();
    // arg-max over lanes, lowest index on ties
    float bv = delta;
    int bj = live ? j : 0x7fffffff;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oj = __shfl_xor_sync(0xffffffffu, bj, o);
      if (oj < 0x7fffffff && (bj == 0x7fffffff || ov > bv || (ov == bv && oj < bj))) {
        bv = ov;
        bj = oj;
      }
    }
    __syncwarp();
    if (lane == 0) {
      int cj = bj;
      for (int t = T - 1; t >= 0; --t) {
        path_idx[(size_t)b * T + t] = cj;
        path_ids[(size_t)b * T + t] = sw.ids[t][cj];
        if (t > 0) cj = sw.bp[t][cj];
      }
      score[b] = (flags & kWalkFlagScoreLogits) ? bv + lse_sum(sw, T) : bv;
    }
  } else {
    // Greedy: j_t = argmax_j (lp_t(j) + tau_t(j_{t-1}, j)); the score follows the Viterbi
    // recursion's order on the chosen path: delta_t = lp_t(j_t) + (delta_{t-1} + tau_t(j_{t-1}, j_t)).
    // Lane c evaluates candidate c and a shuffle arg-max picks the best, lowest index on ties.
    float delta = 0.f;
    int pj = 0;
    for (int t = 0; t < T; ++t) {
      const int row = t == 0 ? 0 : pj;
      float bv = live ? sw.lp[t][j] + sw.tau[t][row][j] : -INFINITY;
      int bj = live ? j : 0x7fffffff;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oj = __shfl_xor_sync(0xffffffffu, bj, o);
        if (oj < 0x7fffffff && (bj == 0x7fffffff || ov > bv || (ov == bv && oj < bj))) {
          bv = ov;
          bj = oj;
        }
      }
      delta = (t == 0) ? sw.lp[0][bj] + sw.tau[0][0][bj] : sw.lp[t][bj] + (delta + sw.tau[t][pj][bj]);
      if (lane == 0) {
        path_idx[(size_t)b * T + t] = bj;
        path_ids[(size_t)b * T + t] = sw.ids[t][bj];
      }
      pj = bj;
    }
    if (lane == 0) score[b] = (flags & kWalkFlagScoreLogits) ? delta + lse_sum(sw, T) : delta;
  }
}

template <bool kBf16>
__global__ void __launch_bounds__(32 * kWarps)
    transition_walk_kernel(const int32_t* __restrict__ anchor, const int32_t* __restrict__ cand_ids,
                           const float* __restrict__ cand_lp, const void* __restrict__ Uv,
                           const void* __restrict__ Vv, const float* __restrict__ gate,
                           const float* __restrict__ lse_rows, int T, int cand_rows, int first, int K, int R,
                           int vocab, int walk_flags, SampleArgs sa,
                           int32_t* __restrict__ path_ids,
                           int32_t* __restrict__ path_idx, float* __restrict__ score, int32_t* err) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  SmemWalk& sw = *reinterpret_cast<SmemWalk*>(smem_raw);
  __nv_bfloat16* stage = reinterpret_cast<__nv_bfloat16*>(smem_raw + ((sizeof(SmemWalk) + 127) & ~size_t(127)));
  const int b = blockIdx.x;

  if (threadIdx.x == 0) sw.anchor = clamp_id(anchor[b], vocab, err, DFLASH2_DEVERR_ANCHOR_RANGE);
  for (int e = threadIdx.x; e < T * kKP; e += blockDim.x) {
    const int t = e / kKP, j = e % kKP;
    if (j < K) {
      const size_t at = ((size_t)b * cand_rows + first + t) * K + j;  // slot t's candidate row
      sw.ids[t][j] = clamp_id(cand_ids[at], vocab, err, DFLASH2_DEVERR_CANDIDATE_RANGE);
      sw.lp[t][j] = cand_lp[at];
    }
  }
  for (int t = threadIdx.x; t < T; t += blockDim.x)
    sw.lse[t] = lse_rows ? lse_rows[(size_t)b * cand_rows + first + t] : 0.f;
  __syncthreads();
  pad_candidates(sw, T, K);
  __syncthreads();
  build_tiles<kBf16>(sw, T, R, Uv, Vv, gate ? gate + ((size_t)b * cand_rows + first) * R : nullptr, stage);
  __syncthreads();
  if ((threadIdx.x >> 5) != 0) return;
  walk_warp0(sw, b, T, K, walk_flags, sa, path_ids, path_idx, score);
}

// Bytes of one warp's merge staging: values and ids [parts][16], (max, sum) [parts], heads.
__host__ __device__ inline size_t merge_stage_bytes(int parts) {
  return (((size_t)parts * 16 * 8 + (size_t)parts * 8 + (size_t)parts) + 127) & ~size_t(127);
}

// Per-warp region of the fused kernel: the merge staging of one row, later the gathered
// V rows of its slot, the U rows that feed the next slot's tile and the slot's gate row.
constexpr size_t kTileStageBytes = (size_t)2 * kKP * kRowPad * sizeof(__nv_bfloat16);
constexpr size_t kGateStageBytes = (size_t)kRChunk * sizeof(float);
constexpr size_t kAnchorStageBytes = (size_t)kKP * kRowPad * sizeof(__nv_bfloat16);
__host__ __device__ inline size_t select_region_stride(int parts) {
  const size_t m = merge_stage_bytes(parts);
  return m > kTileStageBytes + kGateStageBytes ? m : kTileStageBytes + kGateStageBytes;
}

// lse and the K-way merge of one staged row (warp-wide), with the candidates written to sw and,
// where the pointers are given, to global memory. Out of line, so that the dry call the fused
// kernel makes while it waits for the LM head runs the same instructions as the real one.
__device__ __noinline__ void merge_staged_row(const float* sv, const int32_t* si, const float2* sms, uint8_t* head,
                                              int parts, int K, int vocab, int32_t* err, SmemWalk& sw, int t,
                                              int slot, float* lse_out, int32_t* cand_ids, float* cand_lp) {
  const int lane = threadIdx.x & 31;
  float m = -INFINITY;
  for (int p = lane; p < parts; p += 32) m = fmaxf(m, sms[p].x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float s = 0.f;
  for (int p = lane; p < parts; p += 32)
    if (sms[p].y > 0.f) s += sms[p].y * expf(sms[p].x - m);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  const float lse = m + logf(s);
  if (lane == 0) {
    sw.lse[t] = lse;
    if (lse_out) lse_out[slot] = lse;
  }
  {
    int32_t id;
    float v;
    bool ok;
    warp_merge_lists(sv, si, head, parts, K, id, v, ok);
    if (ok) {  // lane k holds the k-th candidate
      const int k = lane;
      const float lp = v - lse;
      // every merged id indexes U and V below: a partial that held no column would carry an
      // out-of-range id, so clamp (and flag) as for the caller's candidates
      id = clamp_id(id, vocab, err, DFLASH2_DEVERR_CANDIDATE_RANGE);
      sw.ids[t][k] = id;
      sw.lp[t][k] = lp;
      if (cand_ids) cand_ids[(size_t)slot * K + k] = id;
      if (cand_lp) cand_lp[(size_t)slot * K + k] = lp;
    }
  }
}

template <bool kBf16>
__global__ void __launch_bounds__(32 * kWarps)
    select_walk_kernel(const float* __restrict__ part_val, const int32_t* __restrict__ part_id,
                       const float2* __restrict__ part_ms, int parts, int M, const int32_t* __restrict__ anchor,
                       const void* __restrict__ Uv, const void* __restrict__ Vv, const float* __restrict__ gate,
                       int T, int rows_per_seq, int first, int K, int R, int vocab,
                       int walk_flags, SampleArgs sa, int32_t* __restrict__ cand_ids, float* __restrict__ cand_lp,
                       float* __restrict__ lse_out, int32_t* __restrict__ path_ids, int32_t* __restrict__ path_idx,
                       float* __restrict__ score, int32_t* err) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  SmemWalk& sw = *reinterpret_cast<SmemWalk*>(smem_raw);
  uint8_t* region = smem_raw + ((sizeof(SmemWalk) + 127) & ~size_t(127));
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t wstride = select_region_stride(parts);
  // One slot per warp and the rank in one staged chunk (the page shape): each warp gathers its
  // slot's embedding rows as soon as its merge is done, while the other warps still merge, and
  // the anchor's U row (tile 0's A operand, the same for all 16 rows) is fetched first.
  const bool early = kBf16 && T <= kWarps && R <= kRChunk;
  __nv_bfloat16* a0 = reinterpret_cast<__nv_bfloat16*>(region + kWarps * wstride);

  if (warp == 0) {
    int32_t anc = 0;
    if (lane == 0) {
      anc = clamp_id(anchor[b], vocab, err, DFLASH2_DEVERR_ANCHOR_RANGE);
      sw.anchor = anc;
    }
    anc = __shfl_sync(0xffffffffu, anc, 0);
    if (early) {
      const __nv_bfloat16* U = reinterpret_cast<const __nv_bfloat16*>(Uv);
      const int vec_per_row = R / 8;
      for (int v = lane; v < kKP * vec_per_row; v += 32)
        cp_async16(a0 + (v / vec_per_row) * kRowPad + (v % vec_per_row) * 8, U + (size_t)anc * R + (v % vec_per_row) * 8);
      cp_async_commit();
    }
  }
  // Dry run while the LM head still runs (this kernel is its programmatic dependent, placed as
  // the LM head's CTAs leave their SMs): the merge and the walk run once on placeholder lists in
  // shared memory, every output kept in shared memory, so that the instructions of the real run
  // below are in this SM's caches when the partials arrive (cold, each phase's first pass costs
  // thousands of cycles of instruction fetch). Only for a few sequences: their CTAs take the first
  // SMs the LM head frees, tens of microseconds before it ends; with many, the last ones placed
  // would still be in the dry run when the partials are ready (measured: B = 1 -3 us, B = 32 +2.5).
  if (gridDim.x <= kWarps) {
    float* sv = reinterpret_cast<float*>(region + warp * wstride);
    int32_t* si = reinterpret_cast<int32_t*>(sv + parts * 16);
    float2* sms = reinterpret_cast<float2*>(si + parts * 16);
    uint8_t* head = reinterpret_cast<uint8_t*>(sms + parts);
    if (warp < T) {
      for (int e = lane; e < parts * 16; e += 32) {
        sv[e] = -(float)(e & 15);
        si[e] = e;
      }
      for (int p = lane; p < parts; p += 32) {
        sms[p] = make_float2(0.f, 1.f);
        head[p] = 0;
      }
      __syncwarp();
      merge_staged_row(sv, si, sms, head, parts, K, vocab, nullptr, sw, warp, 0, nullptr, nullptr, nullptr);
    }
    __syncthreads();
    if (warp == 0) walk_warp0(sw, 0, T, K, walk_flags, sa, sw.dry_ids, sw.dry_idx, &sw.dry_score);
    __syncthreads();
  }
  // the partials are the LM head's output (launched as its programmatic dependent, the
  // prologue above overlaps its end)
  pdl_wait();
  {
    float* sv = reinterpret_cast<float*>(region + warp * wstride);
    int32_t* si = reinterpret_cast<int32_t*>(sv + parts * 16);
    float2* sms = reinterpret_cast<float2*>(si + parts * 16);
    uint8_t* head = reinterpret_cast<uint8_t*>(sms + parts);
    for (int t = warp; t < T; t += kWarps) {
      const int row = b * rows_per_seq + first + t;  // slot t's row of the LM-head pass
      const int slot = b * T + t;
      // the row's lists and (max, sum) pairs in one batch of async copies
      for (int e = lane; e < parts * 4; e += 32) {
        const int p = e >> 2, q = e & 3;
        const size_t src = ((size_t)p * M + row) * 16 + q * 4;
        cp_async16(sv + e * 4, part_val + src);
        cp_async16(si + e * 4, part_id + src);
      }
      for (int p = lane; p < parts; p += 32) {
        cp_async8(sms + p, part_ms + (size_t)p * M + row);
        head[p] = 0;
      }
      cp_async_commit();
      cp_async_wait_all();
      __syncwarp();
      merge_staged_row(sv, si, sms, head, parts, K, vocab, err, sw, t, slot, lse_out, cand_ids, cand_lp);
      __syncwarp();
      if (early) {
        // pad the slot (as pad_candidates does) and start its gathers into this warp's
        // region, whose merge staging is no longer needed: V rows for tile t, U rows for t+1
        if (lane >= K && lane < kKP) {
          sw.ids[t][lane] = sw.ids[t][0];
          sw.lp[t][lane] = -INFINITY;
        }
        __syncwarp();
        __nv_bfloat16* stB = reinterpret_cast<__nv_bfloat16*>(region + warp * wstride);
        gather_rows(reinterpret_cast<const __nv_bfloat16*>(Vv), R, sw.ids[t], stB);
        if (t + 1 < T) gather_rows(reinterpret_cast<const __nv_bfloat16*>(Uv), R, sw.ids[t], stB + kKP * kRowPad);
        if (gate) {  // the slot's gate row, read by the tile's hi / lo split
          float* gs = reinterpret_cast<float*>(region + warp * wstride + kTileStageBytes);
          const float* gsrc = gate + ((size_t)b * rows_per_seq + first + t) * R;
          for (int v = lane; v < R / 4; v += 32) cp_async16(gs + v * 4, gsrc + v * 4);
        }
        cp_async_commit();
      }
    }
  }
  if (early) {
    cp_async_wait_all();
    __syncthreads();  // every warp's gathers have landed
    if (warp < T) {
      const __nv_bfloat16* stA =
          warp == 0 ? a0 : reinterpret_cast<const __nv_bfloat16*>(region + (warp - 1) * wstride) + kKP * kRowPad;
      __nv_bfloat16* stB = reinterpret_cast<__nv_bfloat16*>(region + warp * wstride);
      float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      if (gate) tile_mma_gated(stA, stB, R, reinterpret_cast<const float*>(region + warp * wstride + kTileStageBytes), acc);
      else tile_mma(stA, stB, R, acc);
      store_tau(acc, sw.tau[warp]);
    }
    __syncthreads();
  } else {
    __syncthreads();
    pad_candidates(sw, T, K);
    __syncthreads();
    build_tiles<kBf16>(sw, T, R, Uv, Vv, gate ? gate + ((size_t)b * rows_per_seq + first) * R : nullptr,
                       reinterpret_cast<__nv_bfloat16*>(region));
    __syncthreads();
  }
  if (warp != 0) return;
  walk_warp0(sw, b, T, K, walk_flags, sa, path_ids, path_idx, score);
}

constexpr size_t kWalkStageBytes = (size_t)kWarps * 2 * kKP * kRowPad * sizeof(__nv_bfloat16);

}  // namespace

size_t select_walk_smem(int parts) {
  const size_t base = (sizeof(SmemWalk) + 127) & ~size_t(127);
  return base + (size_t)kWarps * select_region_stride(parts) + kAnchorStageBytes;
}

cudaError_t launch_select_walk(bool bf16, const float* part_val, const int32_t* part_id, const float* part_ms,
                               int parts, int M, const int32_t* anchor, const void* U, const void* V,
                               const float* gate, int B, int T, int rows_per_seq, int first, int K, int R,
                               int vocab, int walk_flags, const float* uniforms, float inv_temp, int32_t* cand_ids,
                               float* cand_lp, float* lse, int32_t* path_ids, int32_t* path_idx, float* score,
                               int32_t* err, cudaStream_t s) {
  if (first < 0 || first + T > rows_per_seq) return cudaErrorInvalidValue;
  const SampleArgs sa{uniforms, inv_temp};
  if (T > kMaxT || K > kKP) return cudaErrorInvalidValue;
  const size_t smem = select_walk_smem(parts);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  cudaError_t e;
  const float2* ms = reinterpret_cast<const float2*>(part_ms);
  // a programmatic dependent of the LM head: it reads the partials after griddepcontrol.wait
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(B);
  cfg.blockDim = dim3(32 * kWarps);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (bf16) {
    static unsigned char smem_done[64];
    e = smem_opt_in(reinterpret_cast<const void*>(select_walk_kernel<true>), smem_done);
    if (e != cudaSuccess) return e;
    e = cudaLaunchKernelEx(&cfg, select_walk_kernel<true>, part_val, part_id, ms, parts, M, anchor, U, V, gate, T,
                           rows_per_seq, first, K, R, vocab, walk_flags, sa, cand_ids, cand_lp, lse, path_ids,
                           path_idx, score, err);
    if (e != cudaSuccess) return e;
  } else {
    static unsigned char smem_done[64];
    e = smem_opt_in(reinterpret_cast<const void*>(select_walk_kernel<false>), smem_done);
    if (e != cudaSuccess) return e;
    e = cudaLaunchKernelEx(&cfg, select_walk_kernel<false>, part_val, part_id, ms, parts, M, anchor, U, V, gate, T,
                           rows_per_seq, first, K, R, vocab, walk_flags, sa, cand_ids, cand_lp, lse, path_ids,
                           path_idx, score, err);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

cudaError_t launch_transition_walk(bool bf16, const int32_t* anchor, const int32_t* cand_ids,
                                   const float* cand_lp, const void* U, const void* V, const float* gate,
                                   const float* lse_rows, int B, int T, int cand_rows, int first, int K, int R,
                                   int vocab, int walk_flags,
                                   const float* uniforms, float inv_temp, int32_t* path_ids, int32_t* path_idx,
                                   float* score, int32_t* err, cudaStream_t s) {
  if (first < 0 || first + T > cand_rows) return cudaErrorInvalidValue;
  const SampleArgs sa{uniforms, inv_temp};
  if (T > kMaxT || K > kKP) return cudaErrorInvalidValue;
  const size_t base = (sizeof(SmemWalk) + 127) & ~size_t(127);
  const size_t smem = base + (bf16 ? kWalkStageBytes : 0);
  cudaError_t e;
  if (bf16) {
    static unsigned char smem_done[64];
    e = smem_opt_in(reinterpret_cast<const void*>(transition_walk_kernel<true>), smem_done);
    if (e != cudaSuccess) return e;
    transition_walk_kernel<true><<<B, 32 * kWarps, smem, s>>>(anchor, cand_ids, cand_lp, U, V, gate, lse_rows, T,
                                                               cand_rows, first, K, R, vocab, walk_flags, sa,
                                                               path_ids, path_idx, score, err);
  } else {
    static unsigned char smem_done[64];
    e = smem_opt_in(reinterpret_cast<const void*>(transition_walk_kernel<false>), smem_done);
    if (e != cudaSuccess) return e;
    transition_walk_kernel<false><<<B, 32 * kWarps, smem, s>>>(anchor, cand_ids, cand_lp, U, V, gate, lse_rows, T,
                                                                cand_rows, first, K, R, vocab, walk_flags, sa,
                                                                path_ids, path_idx, score, err);
  }
  return cudaGetLastError();
}

}  // namespace df
