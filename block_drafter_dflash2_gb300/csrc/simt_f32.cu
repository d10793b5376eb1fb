// fp32 instantiation of the conv layer and of the LM-head top-K/lse partials, for small
// shapes (rows <= 64, hidden <= 4096). Same per-row state and partial layout as the bf16
// tensor-core path, so the same merge kernel finishes both.
#include <math.h>

#include "kernels.h"
#include "tc_gemm.cuh"

namespace df {

namespace {

// One CTA per row: warp w computes group g's two taps p_j = x[row] . w[2g + j] for
// g = w, w + 8, ...; lanes 0..15 then write the group's 16 channels.
__global__ void __launch_bounds__(256) conv_layer_f32_kernel(const float* __restrict__ x, const float* __restrict__ w,
                                                             float* __restrict__ y, int H, int T, int raw) {
  const int row = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = H / 16;
  const float* xr = x + (size_t)row * H;
  const bool has_prev = (row % T) != 0;
  for (int g = warp; g < G; g += 8) {
    const float* w0 = w + (size_t)(2 * g) * H;
    const float* w1 = w0 + H;
    float p0 = 0.f, p1 = 0.f;
    for (int h = lane; h < H; h += 32) {
      p0 = fmaf(xr[h], w0[h], p0);
      p1 = fmaf(xr[h], w1[h], p1);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      p0 += __shfl_xor_sync(0xffffffffu, p0, o);
      p1 += __shfl_xor_sync(0xffffffffu, p1, o);
    }
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
    if (lane < 16) {
      const int c = g * 16 + lane;
      const float xp = has_prev ? xr[c - H] : 0.f;
      y[(size_t)row * H + c] = fmaf(a, xp, b * xr[c]);
    }
  }
}

// Column partition per CTA (same split as the tensor-core path). For each tile of 128
// columns, thread t computes column t's logits for every row into shared memory; thread r
// then feeds row r's 128 values, in column order, through the same top-K/lse state.
constexpr int kTileCols = 128;
constexpr int kMaxRows = 64;

// gw: the context gate's weights [gate_cols, H] (the gate partition's rows), or nullptr.
__global__ void __launch_bounds__(128) lmhead_topk_f32_kernel(const float* __restrict__ z,
                                                               const float* __restrict__ w,
                                                               const float* __restrict__ gw, TcGemmArgs args,
                                                               EpiTopK::Params ep) {
  __shared__ float tile[kMaxRows][kTileCols + 1];
  const int part = blockIdx.x;
  if (part >= args.parts) return;
  const TileRange tr = tile_range(args, part);
  const bool gate_part = is_gate_part(args, part);
  const int t = threadIdx.x;
  const int M = args.M, H = args.K;
  EpiTopK::State st;
  EpiTopK::init(st);
  for (int c0 = tr.u0 * 16; c0 < tr.col_end; c0 += kTileCols) {
    const int col = c0 + t;
    const bool col_ok = col < tr.col_end;
    for (int r = 0; r < M; ++r) {
      float s = 0.f;
      if (col_ok) {
        const float* wr = gate_part ? gw + (size_t)(col - args.gate_base) * H : w + (size_t)col * H;
        const float* zr = z + (size_t)r * H;
        for (int h = 0; h < H; ++h) s = fmaf(zr[h], wr[h], s);
      }
      tile[r][t] = s;
    }
    __syncthreads();
    if (t < M) {
      for (int c = 0; c < kTileCols; c += 32) {
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = tile[t][c + i];
        EpiTopK::consume(st, ep, v, t, true, c0 + c, 32, tr.col_end);
      }
    }
    __syncthreads();
  }
  if (t < M) EpiTopK::finish(st, ep, t, true, part);
}

}  // namespace

cudaError_t launch_conv_layer_f32(const float* x, const float* w, float* y, int M, int H, int T, int raw,
                                  cudaStream_t s) {
  conv_layer_f32_kernel<<<M, 256, 0, s>>>(x, w, y, H, T, raw);
  return cudaGetLastError();
}

cudaError_t launch_lmhead_topk_f32(const float* z, const float* w, const float* gate_w, const TcGemmArgs& args,
                                   float* part_val, int32_t* part_id, float* part_ms, float* gate_out,
                                   cudaStream_t s) {
  if (args.M > kMaxRows) return cudaErrorInvalidValue;
  if (args.gate_cols > 0 && (gate_w == nullptr || gate_out == nullptr || args.parts < 2 ||
                             args.gate_base < args.n_total))
    return cudaErrorInvalidValue;
  EpiTopK::Params ep{part_val, part_id, part_ms, args.M, args.n_total, gate_out, args.gate_base, args.gate_cols};
  lmhead_topk_f32_kernel<<<args.parts, 128, 0, s>>>(z, w, gate_w, args, ep);
  return cudaGetLastError();
}

}  // namespace df
