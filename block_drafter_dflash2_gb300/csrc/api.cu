// C ABI of the DFlash2 draft tail: host-side validation, workspace layout, TMA tensor-map
// encoding and the launch sequence. No allocation, no synchronisation (except
// dflash2_read_device_error).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "../../include/dflash2.h"
#include "kernels.h"

namespace {

using df::TcGemmArgs;

constexpr int kMaxDevices = 64;

int g_sm_count[kMaxDevices];
std::once_flag g_encode_once;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  if (g_sm_count[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_sm_count[dev] = n;
  }
  return g_sm_count[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

// Encoded maps are cached per host thread (32 entries, round robin): a call re-encodes only
// maps it has not seen with the same base, type, shape and box. Encoding costs microseconds of
// host time per map, which an eager caller pays on every call.
struct MapKey {
  const void* base;
  int dtype, rank, swizzle;
  uint64_t dims[3];
  uint32_t box[3];
};
constexpr int kMapCache = 32;
struct MapCache {
  MapKey key[kMapCache];
  CUtensorMap map[kMapCache];
  int n = 0, next = 0;
};
thread_local MapCache t_maps;

bool same_key(const MapKey& a, const MapKey& b) {
  if (a.base != b.base || a.dtype != b.dtype || a.rank != b.rank || a.swizzle != b.swizzle) return false;
  for (int i = 0; i < a.rank; ++i)
    if (a.dims[i] != b.dims[i] || a.box[i] != b.box[i]) return false;
  return true;
}

// A dense row-major tensor (innermost dimension first in dims) as a tiled TMA map with the
// given box, unit element strides and zero fill out of bounds; cached.
bool encode_map(CUtensorMap* map, CUtensorMapDataType dtype, int esize, int rank, const void* base,
                const uint64_t* dims, const uint32_t* box, CUtensorMapSwizzle swizzle) {
  MapKey k{base, (int)dtype, rank, (int)swizzle, {0, 0, 0}, {0, 0, 0}};
  for (int i = 0; i < rank; ++i) {
    k.dims[i] = dims[i];
    k.box[i] = box[i];
  }
  for (int i = 0; i < t_maps.n; ++i)
    if (same_key(t_maps.key[i], k)) {
      *map = t_maps.map[i];
      return true;
    }
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t gdims[3], gstrides[2];
  cuuint32_t gbox[3], estr[3] = {1, 1, 1};
  uint64_t stride = (uint64_t)esize;
  for (int i = 0; i < rank; ++i) {
    gdims[i] = dims[i];
    gbox[i] = box[i];
    stride *= dims[i];
    if (i + 1 < rank) gstrides[i] = stride;
  }
  if (enc(map, dtype, (cuuint32_t)rank, const_cast<void*>(base), gdims, gstrides, gbox, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  const int slot = t_maps.next;
  t_maps.key[slot] = k;
  t_maps.map[slot] = *map;
  t_maps.next = (slot + 1) % kMapCache;
  if (t_maps.n < kMapCache) ++t_maps.n;
  return true;
}

// Row-major bf16 matrix [rows, inner] as a 2-D TMA map with a (64 x box_rows) box,
// 128-byte swizzle, zero fill out of bounds.
bool encode_bf16_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows) {
  const uint64_t dims[2] = {inner, rows};
  const uint32_t box[2] = {64, box_rows};
  return encode_map(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 2, base, dims, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Row counts up to this use the chain kernel that reads whole rows per CTA; above it the
// split-K chain, whose per-CTA traffic does not grow with the row count as fast.
constexpr int kChainMaxRows = 16;

struct Plan {
  int B, T, H, V, K, R, NL, P, M;
  bool bf16;
  size_t esz;
  int n_rc;
  int a_tail_rows;  // rows of the last 128-row chunk, rounded up to 8
  bool lm_pair;     // LM head on CTA pairs (more than one row chunk)
  int lm_parts;
  int conv_parts;
  bool chain;                // all conv layers in one cooperative launch (small M)
  df::ConvChainPlan chain_plan;
  bool split;                // all conv layers in one cooperative launch, split-K (larger M)
  df::ConvSplitPlan split_plan;
  bool raw, greedy, score_logits;
  int first;  // 1: row 0 of each block is the anchor's position (DFLASH2_FIRST_SLOT_1), else 0
  int S;      // slots per sequence: T - first
};

dflash2_status_t make_plan(const dflash2_shape_t* s, Plan& p) {
  if (!s) return DFLASH2_ERR_INVALID_ARGUMENT;
  if (s->batch < 1 || s->block < 1 || s->hidden < 1 || s->vocab < 1 || s->top_k < 1 || s->rank < 1 ||
      s->conv_layers < 0)
    return DFLASH2_ERR_INVALID_ARGUMENT;
  if (s->dtype != DFLASH2_BF16 && s->dtype != DFLASH2_FP32) return DFLASH2_ERR_INVALID_ARGUMENT;
  if (s->flags & ~(uint32_t)(DFLASH2_CONV_TAPS_RAW | DFLASH2_WALK_GREEDY | DFLASH2_FIRST_SLOT_1 |
                             DFLASH2_SCORE_LOGITS))
    return DFLASH2_ERR_INVALID_ARGUMENT;
  if ((s->flags & DFLASH2_FIRST_SLOT_1) && s->block < 2) return DFLASH2_ERR_INVALID_ARGUMENT;
  if (s->hidden % 64 != 0 || s->conv_group_size != 16 || s->conv_kernel_size != 2 || s->top_k > 16 ||
      s->top_k > s->vocab || s->rank % 16 != 0 || s->rank > 1024 || s->block > 32 || s->conv_layers > 16)
    return DFLASH2_ERR_UNSUPPORTED;
  const int64_t M = (int64_t)s->batch * s->block;
  if (M > (1 << 20) || (int64_t)s->hidden * s->vocab > (int64_t)1 << 40) return DFLASH2_ERR_UNSUPPORTED;
  p.B = s->batch;
  p.T = s->block;
  p.H = s->hidden;
  p.V = s->vocab;
  p.K = s->top_k;
  p.R = s->rank;
  p.NL = s->conv_layers;
  p.P = 2 * s->hidden / 16;
  p.M = (int)M;
  p.bf16 = s->dtype == DFLASH2_BF16;
  p.esz = p.bf16 ? 2 : 4;
  p.raw = (s->flags & DFLASH2_CONV_TAPS_RAW) != 0;
  p.greedy = (s->flags & DFLASH2_WALK_GREEDY) != 0;
  p.score_logits = (s->flags & DFLASH2_SCORE_LOGITS) != 0;
  p.first = (s->flags & DFLASH2_FIRST_SLOT_1) ? 1 : 0;
  p.S = p.T - p.first;
  if (!p.bf16 && (p.M > 64 || p.H > 4096)) return DFLASH2_ERR_UNSUPPORTED;
  const int sms = sm_count();
  if (sms <= 0) return DFLASH2_ERR_CUDA;
  const int v_units = (p.V + 15) / 16;
  const int p_units = (p.P + 15) / 16;
  if (p.bf16) {
    p.n_rc = (p.M + 127) / 128;
    p.a_tail_rows = (p.M % 128 == 0) ? 128 : ((p.M % 128 + 7) / 8) * 8;
    const int per = sms / p.n_rc > 0 ? sms / p.n_rc : 1;
    // More than one row chunk: the LM head runs on CTA pairs, two row chunks per pair sharing
    // each weight tile (each SM loads half of it), so a column range has one pair per two chunks
    p.lm_pair = p.n_rc >= 2;
    if (p.lm_pair) {
      const int n_prc = (p.n_rc + 1) / 2;
      const int per_pair = sms / (2 * n_prc) > 0 ? sms / (2 * n_prc) : 1;
      const int pair_units = (p.V + 31) / 32;
      p.lm_parts = per_pair < pair_units ? per_pair : pair_units;
    } else {
      p.lm_parts = per < v_units ? per : v_units;
    }
    p.conv_parts = per < p_units ? per : p_units;
    p.split = p.M > kChainMaxRows && p.NL > 0 && df::conv_splitk_plan(p.M, p.H, p.NL, sms, &p.split_plan);
    p.chain = !p.split && df::conv_chain_plan(p.M, p.H, sms, &p.chain_plan);
  } else {
    p.n_rc = 1;
    p.lm_pair = false;
    p.a_tail_rows = 0;
    p.lm_parts = sms < v_units ? sms : v_units;
    p.conv_parts = 0;
    p.chain = false;
    p.split = false;
  }
  if (p.lm_parts > 1024) p.lm_parts = 1024;
  return DFLASH2_OK;
}

size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

// Partitions of a gated LM-head pass: the vocabulary's, less one, plus the gate's own (at least
// one of each). The workspace holds partials for this many.
int gated_parts(const Plan& p) { return p.lm_parts >= 2 ? p.lm_parts : 2; }

struct Ws {
  int32_t* err;
  unsigned* bar;
  void* conv0;
  void* conv1;
  float* conv_part;
  float* part_val;
  int32_t* part_id;
  float* part_ms;
  int32_t* cand_ids;
  float* cand_lp;
  float* lse;
  float* gate;  // [M, R] fp32 context gate of the gated tail
  size_t total;
};

Ws carve(const Plan& p, void* base) {
  Ws w{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    void* q = base ? static_cast<char*>(base) + off : nullptr;
    off += up256(bytes);
    return q;
  };
  const size_t act = (size_t)p.M * p.H * p.esz;
  w.err = static_cast<int32_t*>(take(256));
  w.bar = static_cast<unsigned*>(take(4096));  // one barrier counter per conv row block
  w.conv0 = take(act);
  w.conv1 = take(act);
  w.conv_part = static_cast<float*>(take(p.split ? p.split_plan.part_bytes : 0));
  const size_t np = (size_t)gated_parts(p);
  w.part_val = static_cast<float*>(take(np * p.M * 16 * 4));
  w.part_id = static_cast<int32_t*>(take(np * p.M * 16 * 4));
  w.part_ms = static_cast<float*>(take(np * p.M * 2 * 4));
  w.cand_ids = static_cast<int32_t*>(take((size_t)p.M * p.K * 4));
  w.cand_lp = static_cast<float*>(take((size_t)p.M * p.K * 4));
  w.gate = static_cast<float*>(take((size_t)p.M * p.R * 4));
  w.lse = static_cast<float*>(take((size_t)p.M * 4));
  w.total = off;
  return w;
}

dflash2_status_t check_ws(const Plan& p, void* ws, size_t ws_bytes, Ws& w) {
  if (!ws || !aligned16(ws)) return DFLASH2_ERR_INVALID_ARGUMENT;
  w = carve(p, ws);
  if (ws_bytes < w.total) return DFLASH2_ERR_WORKSPACE_TOO_SMALL;
  return DFLASH2_OK;
}

dflash2_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? DFLASH2_OK : DFLASH2_ERR_CUDA; }

// ---- stages (arguments already validated)

dflash2_status_t run_conv(const Plan& p, const void* x, const void* conv_w, void* y, const Ws& w,
                          cudaStream_t s) {
  const size_t act = (size_t)p.M * p.H * p.esz;
  if (p.NL == 0) return cuda_status(cudaMemcpyAsync(y, x, act, cudaMemcpyDeviceToDevice, s));
  if (p.bf16 && p.split) {
    const df::ConvSplitPlan& sp = p.split_plan;
    CUtensorMap maps[12];
    const void* srcs[3] = {x, w.conv0, w.conv1};
    for (int i = 0; i < 3; ++i)
      if (!encode_bf16_2d(&maps[2 * i], srcs[i], p.H, p.M, 128) ||
          !encode_bf16_2d(&maps[2 * i + 1], srcs[i], p.H, p.M, sp.a_tail_rows))
        return DFLASH2_ERR_CUDA;
    if (!encode_bf16_2d(&maps[6], conv_w, p.H, (uint64_t)p.NL * p.P, sp.Nt)) return DFLASH2_ERR_CUDA;
    const uint64_t pdims[3] = {(uint64_t)sp.Mp, (uint64_t)p.P, 2 * (uint64_t)sp.KS};
    const uint32_t pst_box[3] = {(uint32_t)sp.br, (uint32_t)sp.Nt, 1};
    const uint32_t pld_box[3] = {(uint32_t)sp.br, 2 * (uint32_t)sp.gc, (uint32_t)sp.KS};
    if (!encode_map(&maps[7], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, 3, w.conv_part, pdims, pst_box,
                    CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_map(&maps[8], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, 3, w.conv_part, pdims, pld_box,
                    CU_TENSOR_MAP_SWIZZLE_NONE))
      return DFLASH2_ERR_CUDA;
    const uint64_t xdims[2] = {(uint64_t)p.H, (uint64_t)p.M};
    const uint32_t xbox[2] = {(uint32_t)sp.xb, (uint32_t)sp.br};
    for (int i = 0; i < 3; ++i)
      if (!encode_map(&maps[9 + i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 2, srcs[i], xdims, xbox,
                      CU_TENSOR_MAP_SWIZZLE_NONE))
        return DFLASH2_ERR_CUDA;
    return cuda_status(df::launch_conv_splitk(sp, maps, x, w.conv0, w.conv1, y, p.M, p.H, p.T, p.NL, p.raw ? 1 : 0,
                                              w.bar, w.err, s));
  }
  if (p.bf16 && p.chain)
    return cuda_status(df::launch_conv_chain(p.chain_plan, x, conv_w, w.conv0, w.conv1, y, p.M, p.H, p.T, p.NL,
                                             p.raw ? 1 : 0, w.bar, w.err, s));
  const void* cur = x;
  for (int l = 0; l < p.NL; ++l) {
    void* out = (l == p.NL - 1) ? y : ((l % 2 == 0) ? w.conv0 : w.conv1);
    const char* wl = static_cast<const char*>(conv_w) + (size_t)l * p.P * p.H * p.esz;
    if (p.bf16) {
      CUtensorMap ma, mat, mb128, mb16;
      if (!encode_bf16_2d(&ma, cur, p.H, p.M, 128) || !encode_bf16_2d(&mat, cur, p.H, p.M, p.a_tail_rows) ||
          !encode_bf16_2d(&mb128, wl, p.H, p.P, 128) || !encode_bf16_2d(&mb16, wl, p.H, p.P, 16))
        return DFLASH2_ERR_CUDA;
      TcGemmArgs a{p.M, p.H, p.P, p.n_rc, p.conv_parts, p.a_tail_rows, 8, 0, w.err};
      if (df::launch_conv_layer_bf16(ma, mat, mb128, mb16, a, cur, out, p.T, p.raw ? 1 : 0, s) != cudaSuccess)
        return DFLASH2_ERR_CUDA;
    } else {
      if (df::launch_conv_layer_f32(static_cast<const float*>(cur), reinterpret_cast<const float*>(wl),
                                    static_cast<float*>(out), p.M, p.H, p.T, p.raw ? 1 : 0, s) != cudaSuccess)
        return DFLASH2_ERR_CUDA;
    }
    cur = out;
  }
  return DFLASH2_OK;
}

// gate_w [R, H] (bf16; nullptr: no gate): the context gate's weights, contracted with the rows
// in the same pass as gate columns past the vocabulary; gate_out [M, R] fp32 receives them.
dflash2_status_t run_partials(const Plan& p, const void* rows, const void* lm_head, const Ws& w, cudaStream_t s,
                              const void* gate_w = nullptr, float* gate_out = nullptr) {
  // 256-column tiles once the row tile is not small: each stage's row-tile box is then shared
  // by twice the weight columns (the copy engine issues box rows at a fixed rate; at 8 rows the
  // stream is HBM-bound either way), and several row chunks re-read each row tile half as often
  TcGemmArgs a{p.M, p.H, p.V, p.n_rc, p.lm_parts, p.a_tail_rows, (p.n_rc > 1 || p.M >= 32) ? 16 : 8,
               p.lm_pair ? 1 : 0, w.err};
  if (gate_w) {
    // the gate rows are one more partition: the last CTA's (the vocabulary keeps the others)
    if (!gate_out) return DFLASH2_ERR_INVALID_ARGUMENT;
    a.parts = gated_parts(p);
    a.gate_base = (p.V + 31) / 32 * 32;
    a.gate_cols = p.R;
  }
  if (p.bf16) {
    CUtensorMap ma, mat, mb128, mb16, mg128, mg16;
    if (!encode_bf16_2d(&ma, rows, p.H, p.M, 128) || !encode_bf16_2d(&mat, rows, p.H, p.M, p.a_tail_rows) ||
        !encode_bf16_2d(&mb128, lm_head, p.H, p.V, 128) || !encode_bf16_2d(&mb16, lm_head, p.H, p.V, 16))
      return DFLASH2_ERR_CUDA;
    if (gate_w) {
      if (!encode_bf16_2d(&mg16, gate_w, p.H, p.R, 16)) return DFLASH2_ERR_CUDA;
      if (p.R >= 128) {
        if (!encode_bf16_2d(&mg128, gate_w, p.H, p.R, 128)) return DFLASH2_ERR_CUDA;
      } else {
        mg128 = mg16;  // unused below 128 gate rows
      }
    } else {
      mg128 = mb128;
      mg16 = mb16;
    }
    if (df::launch_lmhead_topk_bf16(ma, mat, mb128, mb16, mg128, mg16, a, p.V, w.part_val, w.part_id, w.part_ms,
                                    gate_w ? gate_out : nullptr, s) != cudaSuccess)
      return DFLASH2_ERR_CUDA;
  } else {
    if (df::launch_lmhead_topk_f32(static_cast<const float*>(rows), static_cast<const float*>(lm_head),
                                   static_cast<const float*>(gate_w), a, w.part_val, w.part_id, w.part_ms,
                                   gate_w ? gate_out : nullptr, s) != cudaSuccess)
      return DFLASH2_ERR_CUDA;
  }
  return DFLASH2_OK;
}

// parts: the partitions the LM-head pass wrote (gated_parts(p) after a gated pass)
dflash2_status_t run_merge(const Plan& p, int32_t* ids, float* lp, float* lse, const Ws& w, cudaStream_t s,
                           int parts = 0) {
  return cuda_status(df::launch_topk_merge(w.part_val, w.part_id, w.part_ms, parts > 0 ? parts : p.lm_parts, p.M,
                                           p.K, ids, lp, lse ? lse : w.lse, s));
}

// Walk flags of the kernels for this plan.
int walk_flags(const Plan& p) {
  return (p.greedy ? df::kWalkFlagGreedy : 0) | (p.score_logits ? df::kWalkFlagScoreLogits : 0);
}

// The walk over p.S slots. ids / lp / gate / lse_rows hold cand_rows rows per sequence and slot t
// is row first + t (the caller's per-slot arrays: cand_rows = S, first = 0). uniforms [B, S]
// (nullptr: the Viterbi / greedy walk) and inv_temp: draw a path instead.
dflash2_status_t run_walk(const Plan& p, const int32_t* anchor, const int32_t* ids, const float* lp,
                          const void* U, const void* V, const float* gate, const float* lse_rows, int32_t* path_ids,
                          int32_t* path_idx, float* score, const Ws& w, cudaStream_t s, const float* uniforms,
                          float inv_temp, int cand_rows, int first) {
  return cuda_status(df::launch_transition_walk(p.bf16, anchor, ids, lp, U, V, gate, lse_rows, p.B, p.S, cand_rows,
                                                first, p.K, p.R, p.V, walk_flags(p), uniforms, inv_temp, path_ids,
                                                path_idx, score, w.err, s));
}

// ---- scratch for dflash2_select_topk_noalloc: a fixed device array instead of a caller
// workspace. Every device that loads the library holds it until the process exits. Host
// code sees only a host-side stand-in for the symbol; its device address is looked up once
// per device with cudaGetSymbolAddress, with that device current.
constexpr size_t kStaticScratchBytes = 4u << 20;  // 4 MiB

std::mutex g_scratch_mu;
void* g_scratch_dev[kMaxDevices];

}  // namespace

static __device__ __align__(256) unsigned char g_select_scratch[kStaticScratchBytes];

namespace {

dflash2_status_t static_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DFLASH2_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_dev[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_select_scratch) != cudaSuccess || ptr == nullptr) return DFLASH2_ERR_CUDA;
    g_scratch_dev[dev] = ptr;
  }
  *out = g_scratch_dev[dev];
  return DFLASH2_OK;
}

// The part of the workspace layout that the top-K selection uses: error word and partials.
Ws carve_select(const Plan& p, void* base) {
  Ws w{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    void* q = base ? static_cast<char*>(base) + off : nullptr;
    off += up256(bytes);
    return q;
  };
  w.err = static_cast<int32_t*>(take(256));
  w.part_val = static_cast<float*>(take((size_t)p.lm_parts * p.M * 16 * 4));
  w.part_id = static_cast<int32_t*>(take((size_t)p.lm_parts * p.M * 16 * 4));
  w.part_ms = static_cast<float*>(take((size_t)p.lm_parts * p.M * 2 * 4));
  w.total = off;
  return w;
}

}  // namespace

extern "C" {

size_t dflash2_workspace_size(const dflash2_shape_t* shape) {
  Plan p;
  if (make_plan(shape, p) != DFLASH2_OK) return 0;
  return carve(p, nullptr).total;
}

dflash2_status_t dflash2_conv(const dflash2_shape_t* shape, const void* x, const void* conv_w, void* y, void* ws,
                              size_t ws_bytes, void* stream) {
  Plan p;
  dflash2_status_t st = make_plan(shape, p);
  if (st != DFLASH2_OK) return st;
  if (!x || !y || (p.NL > 0 && !conv_w) || x == y) return DFLASH2_ERR_INVALID_ARGUMENT;
  if (!aligned16(x) || !aligned16(y) || (conv_w && !aligned16(conv_w))) return DFLASH2_ERR_INVALID_ARGUMENT;
  Ws w;
  if ((st = check_ws(p, ws, ws_bytes, w)) != DFLASH2_OK) return st;
  return run_conv(p, x, conv_w, y, w, static_cast<cudaStream_t>(stream));
}

dflash2_status_t dflash2_select_topk(const dflash2_shape_t* shape, const void* rows, const void* lm_head,
                                     int32_t* cand_ids, float* cand_lp, float* lse, void* ws, size_t ws_bytes,
                                     void* stream) {
  return dflash2_select_topk_gated(shape, rows, lm_head, nullptr, cand_ids, cand_lp, lse, nullptr, ws, ws_bytes,
                                   stream);
}

dflash2_status_t dflash2_select_topk_gated(const dflash2_shape_t* shape, const void* rows, const void* lm_head,
                                           const void* gate_w, int32_t* cand_ids, float* cand_lp, float* lse,
                                           float* gate, void* ws, size_t ws_bytes, void* stream) {
  Plan p;
  dflash2_status_t st = make_plan(shape, p);
  if (st != DFLASH2_OK) return st;
  if (!rows || !lm_head || !cand_ids || !cand_lp || (gate_w && !gate)) return DFLASH2_ERR_INVALID_ARGUMENT;
  if (!aligned16(rows) || !aligned16(lm_head) || (gate_w && !aligned16(gate_w))) return DFLASH2_ERR_INVALID_ARGUMENT;
  Ws w;
  if ((st = check_ws(p, ws, ws_bytes, w)) != DFLASH2_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if ((st = run_partials(p, rows, lm_head, w, s, gate_w, gate)) != DFLASH2_OK) return st;
  return run_merge(p, cand_ids, cand_lp, lse, w, s, gate_w ? gated_parts(p) : p.lm_parts);
}

dflash2_status_t dflash2_select_topk_noalloc(const dflash2_shape_t* shape, const void* rows, const void* lm_head,
                                             int32_t* cand_ids, float* cand_lp, float* lse, void* stream) {
  Plan p;
  dflash2_status_t st = make_plan(shape, p);
  if (st != DFLASH2_OK) return st;
  if (!rows || !lm_head || !cand_ids || !cand_lp) return DFLASH2_ERR_INVALID_ARGUMENT;
  if (!aligned16(rows) || !aligned16(lm_head)) return DFLASH2_ERR_INVALID_ARGUMENT;
  if (carve_select(p, nullptr).total > kStaticScratchBytes) return DFLASH2_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  if ((st = static_scratch(&scratch)) != DFLASH2_OK) return st;
  const Ws w = carve_select(p, scratch);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the error word must start at zero; the partials are overwritten in full by every call
  if (cudaMemsetAsync(w.err, 0, sizeof(int32_t), s) != cudaSuccess) return DFLASH2_ERR_CUDA;
  if ((st = run_partials(p, rows, lm_head, w, s)) != DFLASH2_OK) return st;
  return run_merge(p, cand_ids, cand_lp, lse, w, s);
}

dflash2_status_t dflash2_lmhead_partials(const dflash2_shape_t* shape, const void* rows, const void* lm_head,
                                         void* ws, size_t ws_bytes, void* stream) {
  Plan p;
  dflash2_status_t st = make_plan(shape, p);
  if (st != DFLASH2_OK) return st;
  if (!rows || !lm_head) return DFLASH2_ERR_INVALID_ARGUMENT;
  if (!aligned16(rows) || !aligned16(lm_head)) return DFLASH2_ERR_INVALID_ARGUMENT;
  Ws w;
  if ((st = check_ws(p, ws, ws_bytes, w)) != DFLASH2_OK) return st;
  return run_partials(p, rows, lm_head, w, static_cast<cudaStream_t>(stream));
}

dflash2_status_t dflash2_merge_partials(const dflash2_shape_t* shape, int32_t* cand_ids, float* cand_lp, float* lse,
                                        void* ws, size_t ws_bytes, void* stream) {
  Plan p;
  dflash2_status_t st = make_plan(shape, p);
  if (st != DFLASH2_OK) return st;
  if (!cand_ids || !cand_lp) return DFLASH2_ERR_INVALID_ARGUMENT;
  Ws w;
  if ((st = check_ws(p, ws, ws_bytes, w)) != DFLASH2_OK) return st;
  return run_merge(p, cand_ids, cand_lp, lse, w, static_cast<cudaStream_t>(stream));
}

dflash2_status_t dflash2_viterbi(const dflash2_shape_t* shape, const int32_t* anchor, const int32_t* cand_ids,
                                 const float* cand_lp, const void* U, const void* V, int32_t* path_ids,
                                 int32_t* path_idx, float* score, void* ws, size_t ws_bytes, void* stream) {
  return dflash2_viterbi_gated(shape, anchor, cand_ids, cand_lp, U, V, nullptr, path_ids, path_idx, score, ws,
                               ws_bytes, stream);
}

dflash2_status_t dflash2_viterbi_gated(const dflash2_shape_t* shape, const int32_t* anchor, const int32_t* cand_ids,
                                       const float* cand_lp, const void* U, const void* V, const float* gate,
                                       int32_t* path_ids, int32_t* path_idx, float* score, void* ws,
                                       size_t ws_bytes, void* stream) {
  return dflash2_sample_walk(shape, anchor, cand_ids, cand_lp, U, V, gate, 0.f, nullptr, path_ids, path_idx, score,
                             ws, ws_bytes, stream);
}

dflash2_status_t dflash2_sample_walk(const dflash2_shape_t* shape, const int32_t* anchor, const int32_t* cand_ids,
                                     const float* cand_lp, const void* U, const void* V, const float* gate,
                                     float temperature, const float* uniforms, int32_t* path_ids, int32_t* path_idx,
                                     float* score, void* ws, size_t ws_bytes, void* stream) {
  Plan p;
  dflash2_status_t st = make_plan(shape, p);
  if (st != DFLASH2_OK) return st;
  if (!anchor || !cand_ids || !cand_lp || !U || !V || !path_ids || !path_idx || !score)
    return DFLASH2_ERR_INVALID_ARGUMENT;
  if (!aligned16(U) || !aligned16(V) || (gate && !aligned16(gate))) return DFLASH2_ERR_INVALID_ARGUMENT;
  if (uniforms && !(temperature > 0.f && temperature < 1e30f)) return DFLASH2_ERR_INVALID_ARGUMENT;
  // the score on raw logits needs each slot's lse, which only the whole-tail calls have
  if (p.score_logits) return DFLASH2_ERR_UNSUPPORTED;
  Ws w;
  if ((st = check_ws(p, ws, ws_bytes, w)) != DFLASH2_OK) return st;
  return run_walk(p, anchor, cand_ids, cand_lp, U, V, gate, nullptr, path_ids, path_idx, score, w,
                  static_cast<cudaStream_t>(stream), uniforms, uniforms ? 1.f / temperature : 0.f, p.S, 0);
}

dflash2_status_t dflash2_draft_tail(const dflash2_shape_t* shape, const void* hidden, const void* lm_head,
                                    const void* U, const void* V, const void* conv_w, const int32_t* anchor,
                                    int32_t* path_ids, int32_t* path_idx, float* score, int32_t* cand_ids,
                                    float* cand_lp, float* lse, void* ws, size_t ws_bytes, void* stream) {
  return dflash2_draft_tail_gated(shape, hidden, lm_head, U, V, conv_w, nullptr, anchor, path_ids, path_idx, score,
                                  cand_ids, cand_lp, lse, nullptr, ws, ws_bytes, stream);
}

dflash2_status_t dflash2_draft_tail_gated(const dflash2_shape_t* shape, const void* hidden, const void* lm_head,
                                          const void* U, const void* V, const void* conv_w, const void* gate_w,
                                          const int32_t* anchor, int32_t* path_ids, int32_t* path_idx, float* score,
                                          int32_t* cand_ids, float* cand_lp, float* lse, float* gate,
                                          void* ws, size_t ws_bytes, void* stream) {
  return dflash2_draft_tail_sampled(shape, hidden, lm_head, U, V, conv_w, gate_w, anchor, 0.f, nullptr, path_ids,
                                    path_idx, score, cand_ids, cand_lp, lse, gate, ws, ws_bytes, stream);
}

dflash2_status_t dflash2_draft_tail_sampled(const dflash2_shape_t* shape, const void* hidden, const void* lm_head,
                                            const void* U, const void* V, const void* conv_w, const void* gate_w,
                                            const int32_t* anchor, float temperature, const float* uniforms,
                                            int32_t* path_ids, int32_t* path_idx, float* score, int32_t* cand_ids,
                                            float* cand_lp, float* lse, float* gate, void* ws, size_t ws_bytes,
                                            void* stream) {
  Plan p;
  dflash2_status_t st = make_plan(shape, p);
  if (st != DFLASH2_OK) return st;
  if (!hidden || !lm_head || !U || !V || (p.NL > 0 && !conv_w) || !anchor || !path_ids || !path_idx || !score)
    return DFLASH2_ERR_INVALID_ARGUMENT;
  if (!aligned16(hidden) || !aligned16(lm_head) || !aligned16(U) || !aligned16(V) ||
      (conv_w && !aligned16(conv_w)) || (gate_w && !aligned16(gate_w)))
    return DFLASH2_ERR_INVALID_ARGUMENT;
  if (gate && !aligned16(gate)) return DFLASH2_ERR_INVALID_ARGUMENT;
  if (uniforms && !(temperature > 0.f && temperature < 1e30f)) return DFLASH2_ERR_INVALID_ARGUMENT;
  Ws w;
  if ((st = check_ws(p, ws, ws_bytes, w)) != DFLASH2_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const float inv_temp = uniforms ? 1.f / temperature : 0.f;
  // z: the last conv layer's output lands in conv0/conv1 (never the caller's hidden)
  const void* z = hidden;
  if (p.NL > 0) {
    // Layers l < NL-1 write conv0 (even l) / conv1 (odd l); the last layer writes the buffer that
    // layer NL-2 did not write, so no layer reads and writes the same buffer.
    void* zbuf = (p.NL % 2 == 1) ? w.conv0 : w.conv1;
    if ((st = run_conv(p, hidden, conv_w, zbuf, w, s)) != DFLASH2_OK) return st;
    z = zbuf;
  }
  // the gate rows: the caller's buffer when given, else the workspace's
  float* g = gate_w ? (gate ? gate : w.gate) : nullptr;
  if ((st = run_partials(p, z, lm_head, w, s, gate_w, g)) != DFLASH2_OK) return st;
  const int parts = gate_w ? gated_parts(p) : p.lm_parts;
  if (df::select_walk_smem(parts) <= 227 * 1024)  // merge fused with the walk
    return cuda_status(df::launch_select_walk(p.bf16, w.part_val, w.part_id, w.part_ms, parts, p.M, anchor, U,
                                              V, g, p.B, p.S, p.T, p.first, p.K, p.R, p.V, walk_flags(p),
                                              uniforms, inv_temp, cand_ids, cand_lp, lse, path_ids, path_idx, score,
                                              w.err, s));
  // merge every row into the workspace, walk the slot rows, and copy the slot rows out
  if ((st = run_merge(p, w.cand_ids, w.cand_lp, w.lse, w, s, parts)) != DFLASH2_OK) return st;
  if ((st = run_walk(p, anchor, w.cand_ids, w.cand_lp, U, V, g, w.lse, path_ids, path_idx, score, w, s, uniforms,
                     inv_temp, p.T, p.first)) != DFLASH2_OK)
    return st;
  const size_t k4 = (size_t)p.K * 4;
  if (cand_ids && cudaMemcpy2DAsync(cand_ids, p.S * k4, w.cand_ids + (size_t)p.first * p.K, p.T * k4, p.S * k4, p.B,
                                    cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return DFLASH2_ERR_CUDA;
  if (cand_lp && cudaMemcpy2DAsync(cand_lp, p.S * k4, w.cand_lp + (size_t)p.first * p.K, p.T * k4, p.S * k4, p.B,
                                   cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return DFLASH2_ERR_CUDA;
  if (lse && cudaMemcpy2DAsync(lse, (size_t)p.S * 4, w.lse + p.first, (size_t)p.T * 4, (size_t)p.S * 4, p.B,
                               cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return DFLASH2_ERR_CUDA;
  return DFLASH2_OK;
}

dflash2_status_t dflash2_read_device_error(void* ws, void* stream, int32_t* code_out) {
  if (!ws || !code_out) return DFLASH2_ERR_INVALID_ARGUMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t host = 0;
  if (cudaMemcpyAsync(&host, ws, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return DFLASH2_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return DFLASH2_ERR_CUDA;
  *code_out = host;
  if (host != 0) {
    if (cudaMemsetAsync(ws, 0, sizeof(int32_t), s) != cudaSuccess) return DFLASH2_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return DFLASH2_ERR_CUDA;
  }
  return DFLASH2_OK;
}

const char* dflash2_status_string(dflash2_status_t status) {
  switch (status) {
    case DFLASH2_OK: return "ok";
    case DFLASH2_ERR_INVALID_ARGUMENT: return "invalid argument (null, misaligned or bad size)";
    case DFLASH2_ERR_UNSUPPORTED: return "shape outside the supported set";
    case DFLASH2_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case DFLASH2_ERR_CUDA: return "CUDA runtime or launch error";
    case DFLASH2_ERR_DEVICE: return "device error word set";
  }
  return "unknown status";
}

int32_t dflash2_version(void) { return 100; }

}  // extern "C"
