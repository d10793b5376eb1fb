// Persistent tcgen05 GEMM with a fused epilogue: D = A * B^T, A = rows [M, K] bf16, B = [N, K] bf16.
//
// Layout: rows sit on the MMA M dimension (128 TMEM lanes), columns on N. One epilogue
// thread owns one row and sees that row's N values of a tile in its registers, so a per-row
// reduction (top-K, log-sum-exp, the conv's per-group tap softmax) is sequential per thread
// with no cross-thread exchange.
//
// Work split: CTA c takes row chunk c % n_rc (128 rows) and column partition c / n_rc of
// `parts` contiguous ranges (in units of 16 columns, balanced to one unit). A range is walked
// in tiles of `tile_units` units (128 or 256 columns: wider tiles re-read the row tile less
// often when several row chunks share a column range); the last tile of a range is narrower
// and fetched in 16-row TMA boxes, so no column outside the range is ever loaded.
//
// Roles (192 threads): warp 0 = TMA producer (one thread), warp 1 = MMA issuer (one thread)
// and TMEM owner, warps 2..5 = epilogue (thread = TMEM lane = row). Shared memory holds a
// ring of (A, B) bf16 stages, K = 64 each, in the 128-byte swizzled K-major layout. The A
// box of the last row chunk covers only its real rows (rounded up to 8), so a small M does
// not pay for TMA zero-fill, and the ring is cut into as many stages as fit, so small tiles
// keep many more loads in flight. The MMA reads 128 A rows regardless; rows past the box hold
// stale data and only feed TMEM lanes no epilogue thread reads. TMEM holds two fp32
// accumulators as wide as a tile, so the epilogue of tile t overlaps the MMAs of tile t+1.
//
// Gate columns: the LM-head launch can add the rows of a second matrix (the context gate's
// [R, H] weights) as extra columns past the vocabulary, numbered from gate_base. They form a
// partition of their own, the last CTA's, fetched through the gate's own tensor maps, and the
// vocabulary is balanced over the other partitions; so no tile straddles the two matrices (a
// tile that did, fetched in 16-row boxes, measured 130 us slower). The epilogue stores the
// gate columns' fp32 values instead of ranking them.
#pragma once

#include "ptx.cuh"
#include "tc_gemm_args.h"

namespace df {

constexpr int kBK = 64;   // K per stage: one 128-byte swizzle row of bf16
constexpr int kBM = 128;  // rows per tile (MMA M)
constexpr int kBN = 128;  // widest tile with 8-unit tiles (MMA N); 16-unit tiles are 256 wide
constexpr int kMaxStages = 48;
constexpr int kRingBytes = 200 * 1024;           // smem ring, split into as many stages as fit
constexpr int kASlackBytes = kBM * kBK * 2;       // the MMA always reads 128 A rows from a stage
constexpr int kBarrierBytes = 1024;
constexpr int kGemmThreads = 192;
constexpr int kGemmSmemBytes = 1024 /*align*/ + kBarrierBytes + kRingBytes + kASlackBytes;

struct TileRange {
  int u0, u1;      // unit range [u0, u1) of 16 columns
  int col_end;     // min(u1 * 16, n_total)
  int num_tiles;
};

DF_DEV bool is_gate_part(const TcGemmArgs& a, int part) { return a.gate_cols > 0 && part == a.parts - 1; }

DF_DEV TileRange tile_range(const TcGemmArgs& a, int part) {
  TileRange r;
  if (is_gate_part(a, part)) {
    r.u0 = a.gate_base / 16;
    r.u1 = r.u0 + (a.gate_cols + 15) / 16;
    r.col_end = a.gate_base + a.gate_cols;
  } else {
    const int units = (a.n_total + 15) / 16;
    const int vparts = a.gate_cols > 0 ? a.parts - 1 : a.parts;
    r.u0 = (int)((int64_t)part * units / vparts);
    r.u1 = (int)((int64_t)(part + 1) * units / vparts);
    r.col_end = min(r.u1 * 16, a.n_total);
  }
  r.num_tiles = (r.u1 - r.u0 + a.tile_units - 1) / a.tile_units;
  return r;
}

// Stage geometry of one CTA: the A box is the row chunk's real rows (padded to 8; 128 for full
// chunks), the B tile is as wide as this CTA's widest tile. Stages are as many as fit the ring.
struct StageGeom {
  uint32_t a_bytes;  // bytes of this CTA's A box per stage
  uint32_t b_off;    // offset of the B tile in a stage
  uint32_t stride;   // bytes per stage
  int stages;
};

DF_DEV StageGeom stage_geom(const TcGemmArgs& a, int rc, const TileRange& tr) {
  StageGeom g;
  const int rows = (rc == a.n_rc - 1) ? a.a_tail_rows : kBM;
  g.a_bytes = (uint32_t)rows * kBK * 2;
  const int nmax = min(a.tile_units, tr.u1 - tr.u0) * 16;
  g.b_off = g.a_bytes;
  g.stride = (g.a_bytes + (uint32_t)nmax * kBK * 2 + 1023u) & ~1023u;
  g.stages = min(kMaxStages, (int)(kRingBytes / g.stride));
  return g;
}

template <class Epi>
__global__ void __launch_bounds__(kGemmThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_a_tail,
                   const __grid_constant__ CUtensorMap map_b128, const __grid_constant__ CUtensorMap map_b16,
                   const __grid_constant__ CUtensorMap map_g128, const __grid_constant__ CUtensorMap map_g16,
                   const TcGemmArgs args, const typename Epi::Params ep) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(base);
  uint64_t* empty = full + kMaxStages;
  uint64_t* tfull = empty + kMaxStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint8_t* ring = base + kBarrierBytes;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rc = blockIdx.x % args.n_rc;
  const int part = blockIdx.x / args.n_rc;
  if (part >= args.parts) return;  // whole CTA idle (uniform)
  const TileRange tr = tile_range(args, part);
  const StageGeom sg = stage_geom(args, rc, tr);
  const int kblocks = args.K / kBK;
  const bool tail_chunk = (rc == args.n_rc - 1);
  const int TU = args.tile_units;                   // tile width in 16-column units (8 or 16)
  const uint32_t tmem_cols = (uint32_t)(2 * TU * 16);  // two accumulators: 256 or 512 columns

  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < sg.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);  // released by the MMA warp's commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 128);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, tmem_cols);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    tma_prefetch_desc(tail_chunk ? &map_a_tail : &map_a);
    tma_prefetch_desc(&map_b128);
    tma_prefetch_desc(&map_b16);
    if (is_gate_part(args, part)) {
      tma_prefetch_desc(&map_g16);
      if (args.gate_cols >= 128) tma_prefetch_desc(&map_g128);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      const uint64_t pol_a = l2_policy_evict_last();   // row tiles are re-read for every column tile
      const uint64_t pol_b = l2_policy_evict_first();  // column tiles (weights) stream through once
      const CUtensorMap* ma = tail_chunk ? &map_a_tail : &map_a;
      // B: the vocabulary, or the gate matrix for the gate partition (its rows from gate_base)
      const bool gate_part = is_gate_part(args, part);
      const CUtensorMap* mb128 = gate_part ? &map_g128 : &map_b128;
      const CUtensorMap* mb16 = gate_part ? &map_g16 : &map_b16;
      const int row0 = gate_part ? args.gate_base : 0;
      // The rows are the previous kernel's output (launched as its programmatic dependent,
      // this kernel's prologue overlaps its end): wait for it before the first load.
      pdl_wait();
      int stage = 0;
      uint32_t phase = 0;
      uint64_t issued = 0, issued_phase = 0;  // per-stage bits: ever issued / parity of last issue
      bool ok = true;
      for (int t = 0; t < tr.num_tiles && ok; ++t) {
        const int cu0 = tr.u0 + t * TU;
        const int nu = min(TU, tr.u1 - cu0);
        const int n0 = cu0 * 16;
        const uint32_t bytes = sg.a_bytes + (uint32_t)nu * 16 * kBK * 2;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, args.err, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* sa = ring + (size_t)stage * sg.stride;
          uint8_t* sb = sa + sg.b_off;
          mbar_arrive_expect_tx(&full[stage], bytes);
          tma_load_2d(sa, ma, &full[stage], kb * kBK, rc * kBM, pol_a);
          if (nu % 8 == 0) {
            for (int j = 0; j < nu / 8; ++j)
              tma_load_2d(sb + j * 128 * kBK * 2, mb128, &full[stage], kb * kBK, n0 - row0 + 128 * j, pol_b);
          } else {
            for (int j = 0; j < nu; ++j)
              tma_load_2d(sb + j * 16 * kBK * 2, mb16, &full[stage], kb * kBK, n0 - row0 + 16 * j, pol_b);
          }
          issued |= 1ull << stage;
          issued_phase = (issued_phase & ~(1ull << stage)) | ((uint64_t)phase << stage);
          if (++stage == sg.stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // Aborted: let every copy still in flight land before the CTA can exit.
        // (one timeout ends the drain: a copy that has not landed by then is not coming)
        for (int s = 0; s < sg.stages; ++s)
          if ((issued & (1ull << s)) && !mbar_wait(&full[s], (uint32_t)(issued_phase >> s) & 1u, args.err, nullptr))
            break;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int t = 0; t < tr.num_tiles && ok; ++t) {
        const int acc = t & 1;
        const uint32_t acc_phase = (uint32_t)(t >> 1) & 1u;
        const int nu = min(TU, tr.u1 - (tr.u0 + t * TU));
        const uint32_t idesc = idesc_bf16_f32(kBM, nu * 16);
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, args.err, abort_flag)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * TU * 16);
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(&full[stage], phase, args.err, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(ring + (size_t)stage * sg.stride);
          const uint64_t da = sdesc_k_sw128(sa);
          const uint64_t db = sdesc_k_sw128(sa + sg.b_off);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)  // 16 bf16 = 32 B per MMA along K: +2 in 16-B units
            umma_bf16(d_tmem, da + 2 * k, db + 2 * k, idesc, (kb | k) != 0 ? 1u : 0u);
          umma_commit(&empty[stage]);
          if (++stage == sg.stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) umma_commit(&tfull[acc]);
      }
      // Make sure no MMA is still running before TMEM is released.
      umma_commit(drain);
      mbar_wait(drain, 0, args.err, nullptr);
    }
  } else {
    // ---------------- epilogue: thread = TMEM lane = row of the chunk
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const int row = rc * kBM + q * 32 + lane;
    const bool row_ok = row < args.M;
    const bool warp_rows = rc * kBM + q * 32 < args.M;
    typename Epi::State st;
    Epi::init(st);
    for (int t = 0; t < tr.num_tiles; ++t) {
      const int acc = t & 1;
      const uint32_t acc_phase = (uint32_t)(t >> 1) & 1u;
      const int n0 = (tr.u0 + t * TU) * 16;
      const int nt = min(TU, tr.u1 - (tr.u0 + t * TU)) * 16;
      // lane 0 waits and the warp follows it converged (the TMEM loads are warp-wide)
      int ready = 0;
      if (lane == 0) ready = mbar_wait(&tfull[acc], acc_phase, args.err, abort_flag) ? 1 : 0;
      ready = __shfl_sync(0xffffffffu, ready, 0);
      __syncwarp();
      if (!ready) break;
      tc_fence_after();
      if (warp_rows) {
        for (int c = 0; c < nt; c += 32) {
          float v[32];
          tmem_ld32(tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * TU * 16 + c), v);
          Epi::consume(st, ep, v, row, row_ok, n0 + c, min(32, nt - c), tr.col_end);
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
    }
    if (!*abort_flag) Epi::finish(st, ep, row, row_ok, part);
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, tmem_cols);
  }
}

// ---------------------------------------------------------------------------
// CTA-pair form, for more than one row chunk. The two CTAs of a cluster (ranks 0 and 1) take row
// chunks 2k and 2k + 1 of the same column range and run each tile as one MMA of M = 256 rows
// (tcgen05 cta_group::2, issued by rank 0): each CTA loads its own 128 A rows and half of the
// tile's columns of B (rank 0 the first half), so each weight byte crosses into one SM, not two,
// and a stage is 32 KB per SM instead of 48 (7 stages in the ring instead of 4). Each CTA's TMEM
// holds its 128 rows of the accumulator over the tile's full width, so the epilogue is the same
// thread-per-row reduction as above. Both CTAs' copies of a stage complete on rank 0's full
// barrier; rank 0's MMA thread commits every stage to the empty barriers of both CTAs and every
// tile to both CTAs' TMEM-full barriers; each CTA's epilogue releases the accumulator with one
// arrival on rank 0's TMEM-empty barrier. Ranges are balanced in units of 32 columns so every
// tile splits evenly (a range's last tile may run up to 16 columns past the vocabulary or the gate
// matrix: those rows are outside the tensor maps, read as zeros and never ranked or stored).
// ---------------------------------------------------------------------------
constexpr int kPairRingBytes = 224 * 1024;
constexpr int kPairKps = 2;  // K blocks of 64 per ring stage: fewer, larger stages move more bytes per SM
constexpr int kPairProducer2 = 6;                 // warp of the second TMA producer
constexpr int kPairThreads = kGemmThreads + 32;  // the single-CTA roles plus that warp
constexpr int kPairSmemBytes = 1024 /*align*/ + kBarrierBytes + kPairRingBytes;

DF_DEV TileRange tile_range_pair(const TcGemmArgs& a, int part) {
  TileRange r;
  if (is_gate_part(a, part)) {
    r.u0 = a.gate_base / 16;
    r.u1 = r.u0 + 2 * ((a.gate_cols + 31) / 32);
    r.col_end = a.gate_base + a.gate_cols;
  } else {
    const int pairs = (a.n_total + 31) / 32;
    const int vparts = a.gate_cols > 0 ? a.parts - 1 : a.parts;
    r.u0 = 2 * (int)((int64_t)part * pairs / vparts);
    r.u1 = 2 * (int)((int64_t)(part + 1) * pairs / vparts);
    r.col_end = min(r.u1 * 16, a.n_total);
  }
  r.num_tiles = (r.u1 - r.u0 + a.tile_units - 1) / a.tile_units;
  return r;
}

template <class Epi>
__global__ void __launch_bounds__(kPairThreads, 1)
    tc_gemm_pair_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_a_tail,
                        const __grid_constant__ CUtensorMap map_b128, const __grid_constant__ CUtensorMap map_b16,
                        const __grid_constant__ CUtensorMap map_g128, const __grid_constant__ CUtensorMap map_g16,
                        const TcGemmArgs args, const typename Epi::Params ep) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(base);
  uint64_t* empty = full + kMaxStages;
  uint64_t* tfull = empty + kMaxStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint8_t* ring = base + kBarrierBytes;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs; 1: its peer
  const int n_prc = (args.n_rc + 1) / 2;
  const int cl = (int)(blockIdx.x >> 1);
  const int prc = cl % n_prc, part = cl / n_prc;
  if (part >= args.parts) return;  // both CTAs of the pair (same cluster) leave together
  const int rc = 2 * prc + (int)rank;       // this CTA's row chunk (>= n_rc: none)
  const int peer_rc = 2 * prc + (int)(rank ^ 1u);
  const TileRange tr = tile_range_pair(args, part);
  const int kblocks = args.K / kBK;
  const int TU = args.tile_units;  // even: tiles are whole pairs of 16-column units
  // identical stage layout in both CTAs: kPairKps K blocks, each 128 A rows then the widest
  // tile's half of B
  const uint32_t b_off = (uint32_t)kBM * kBK * 2;
  const int half_max = min(TU, tr.u1 - tr.u0) * 8;
  const uint32_t sub = (b_off + (uint32_t)half_max * kBK * 2 + 1023u) & ~1023u;
  const uint32_t stride = sub * kPairKps;
  const int stages = min(kMaxStages, (int)(kPairRingBytes / stride));
  const int ksteps = (kblocks + kPairKps - 1) / kPairKps;
  auto a_rows = [&](int chunk) {
    return chunk >= args.n_rc ? 0 : (chunk == args.n_rc - 1 ? args.a_tail_rows : kBM);
  };
  const uint32_t own_a = (uint32_t)a_rows(rc) * kBK * 2;
  const uint32_t peer_a = (uint32_t)a_rows(peer_rc) * kBK * 2;
  const uint32_t tmem_cols = (uint32_t)(2 * TU * 16);

  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);   // rank 0's producer arrives with both CTAs' bytes
      mbar_init(&empty[s], 1);  // rank 0's MMA commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 2);  // one arrival per CTA of the pair
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, tmem_cols);
    tmem_relinquish_pair();
  }
  if (threadIdx.x == 0) {
    tma_prefetch_desc(rc == args.n_rc - 1 ? &map_a_tail : &map_a);
    tma_prefetch_desc(&map_b128);
    tma_prefetch_desc(&map_b16);
    if (is_gate_part(args, part)) {
      tma_prefetch_desc(&map_g16);
      if (args.gate_cols >= 128) tma_prefetch_desc(&map_g128);
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_barrier();  // both CTAs' barriers exist before either signals the other's
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t lead_full = mapa_shared(smem_u32(full), 0);      // + 8 s: rank 0's full[s]
  const uint32_t peer_empty = mapa_shared(smem_u32(empty), 1);    // + 8 s: rank 1's empty[s]
  const uint32_t peer_tfull = mapa_shared(smem_u32(tfull), 1);    // + 8 b
  const uint32_t lead_tempty = mapa_shared(smem_u32(tempty), 0);  // + 8 b

  if (warp == 0 || warp == kPairProducer2) {
    if (lane == 0) {
      // ---------------- TMA producers (both CTAs): warp 0 loads K block 0 of every stage and
      // posts the stage's bytes; the second producer loads K block 1. Two issuing threads move
      // more bytes into the SM than one. Its copies may land before the byte count is posted:
      // the count goes below zero and the phase still waits for the posting arrival.
      const int j = warp == 0 ? 0 : 1;
      const uint64_t pol_a = l2_policy_evict_last();
      const uint64_t pol_b = l2_policy_evict_first();
      const bool tail_chunk = rc == args.n_rc - 1;
      const CUtensorMap* ma = tail_chunk ? &map_a_tail : &map_a;
      const bool gate_part = is_gate_part(args, part);
      const CUtensorMap* mb128 = gate_part ? &map_g128 : &map_b128;
      const CUtensorMap* mb16 = gate_part ? &map_g16 : &map_b16;
      const int row0 = gate_part ? args.gate_base : 0;
      pdl_wait();
      int stage = 0;
      uint32_t phase = 0;
      uint64_t issued = 0, issued_phase = 0;
      bool ok = true;
      for (int t = 0; t < tr.num_tiles && ok; ++t) {
        const int cu0 = tr.u0 + t * TU;
        const int nu = min(TU, tr.u1 - cu0);  // even
        const int half = nu * 8;              // columns of B this CTA loads
        const int my_n0 = cu0 * 16 + (int)rank * half;
        const uint32_t bytes = own_a + peer_a + 2u * (uint32_t)half * kBK * 2;  // per K block
        for (int ks = 0; ks < ksteps; ++ks) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, args.err, abort_flag)) {
            ok = false;
            break;
          }
          const int nkb = min(kPairKps, kblocks - ks * kPairKps);
          const uint32_t fb = lead_full + 8u * (uint32_t)stage;
          if (j == 0 && rank == 0) mbar_arrive_expect_tx(&full[stage], (uint32_t)nkb * bytes);
          if (j < nkb) {
            const int kb = ks * kPairKps + j;
            uint8_t* sa = ring + (size_t)stage * stride + (size_t)j * sub;
            uint8_t* sb = sa + b_off;
            if (own_a) tma_load_2d_pair(sa, ma, fb, kb * kBK, rc * kBM, pol_a);
            if (half == 128) {
              tma_load_2d_pair(sb, mb128, fb, kb * kBK, my_n0 - row0, pol_b);
            } else {
              for (int i = 0; i < half / 16; ++i)
                tma_load_2d_pair(sb + i * 16 * kBK * 2, mb16, fb, kb * kBK, my_n0 - row0 + 16 * i, pol_b);
            }
          }
          issued |= 1ull << stage;
          issued_phase = (issued_phase & ~(1ull << stage)) | ((uint64_t)phase << stage);
          if (++stage == stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // Aborted. Rank 0's first producer lets the stages it posted land (their bytes include
        // the peer's and the second producer's; a stage whose other copies were never issued
        // gives up at the wait's time limit); the others cannot see their copies complete
        // (they signal rank 0's barrier), so they wait a fixed 50 us.
        if (rank == 0 && j == 0) {
          for (int s = 0; s < stages; ++s)
            if ((issued & (1ull << s)) && !mbar_wait(&full[s], (uint32_t)(issued_phase >> s) & 1u, args.err, nullptr))
              break;
        } else {
          const uint64_t t0 = globaltimer_ns();
          while (globaltimer_ns() - t0 < 50000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---------------- MMA issuer (rank 0 only)
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int t = 0; t < tr.num_tiles && ok; ++t) {
        const int acc = t & 1;
        const uint32_t acc_phase = (uint32_t)(t >> 1) & 1u;
        const int nu = min(TU, tr.u1 - (tr.u0 + t * TU));
        const uint32_t idesc = idesc_bf16_f32(2 * kBM, nu * 16);
        if (!mbar_wait_cluster(&tempty[acc], acc_phase ^ 1u, args.err, abort_flag)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * TU * 16);
        for (int ks = 0; ks < ksteps; ++ks) {
          if (!mbar_wait(&full[stage], phase, args.err, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int nkb = min(kPairKps, kblocks - ks * kPairKps);
          for (int j = 0; j < nkb; ++j) {
            const uint32_t sa = smem_u32(ring + (size_t)stage * stride + (size_t)j * sub);
            const uint64_t da = sdesc_k_sw128(sa);
            const uint64_t db = sdesc_k_sw128(sa + b_off);
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k)
              umma_bf16_pair(d_tmem, da + 2 * k, db + 2 * k, idesc, (ks | j | k) != 0 ? 1u : 0u);
          }
          umma_commit_pair(smem_u32(&empty[stage]));
          umma_commit_pair(peer_empty + 8u * (uint32_t)stage);
          if (++stage == stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) {
          umma_commit_pair(smem_u32(&tfull[acc]));
          umma_commit_pair(peer_tfull + 8u * (uint32_t)acc);
        }
      }
      // no MMA may still be running (in either CTA) when the pair frees TMEM
      umma_commit_pair(smem_u32(drain));
      mbar_wait(drain, 0, args.err, nullptr);
    }
  } else {
    // ---------------- epilogue (both CTAs): thread = TMEM lane = row of this CTA's chunk
    const int q = warp & 3;
    const int row = rc * kBM + q * 32 + lane;
    const bool row_ok = rc < args.n_rc && row < args.M;
    const bool warp_rows = rc < args.n_rc && rc * kBM + q * 32 < args.M;
    typename Epi::State st;
    Epi::init(st);
    for (int t = 0; t < tr.num_tiles; ++t) {
      const int acc = t & 1;
      const uint32_t acc_phase = (uint32_t)(t >> 1) & 1u;
      const int n0 = (tr.u0 + t * TU) * 16;
      const int nt = min(TU, tr.u1 - (tr.u0 + t * TU)) * 16;
      // lane 0 waits and its warp follows (the TMEM loads are warp-wide); the four warps then
      // agree at the barrier whether any of them gave up
      int ready = 0;
      if (lane == 0) ready = mbar_wait(&tfull[acc], acc_phase, args.err, abort_flag) ? 1 : 0;
      ready = __shfl_sync(0xffffffffu, ready, 0);
      if (ready) {
        tc_fence_after();
        if (warp_rows) {
          for (int c = 0; c < nt; c += 32) {
            float v[32];
            tmem_ld32(tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * TU * 16 + c), v);
            Epi::consume(st, ep, v, row, row_ok, n0 + c, min(32, nt - c), tr.col_end);
          }
        }
        tc_fence_before();
      }
      __syncwarp();
      if (named_barrier_or(1, 128, !ready)) break;  // the accumulator was read by all four warps
      if (warp == 2 && lane == 0) {
        if (rank == 0) mbar_arrive(&tempty[acc]);
        else mbar_arrive_remote(lead_tempty + 8u * (uint32_t)acc);
      }
    }
    if (!*abort_flag) Epi::finish(st, ep, row, row_ok, part);
  }

  __syncthreads();
  cluster_barrier();  // rank 0 has drained its MMAs, which write both CTAs' TMEM and read both rings
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, tmem_cols);
  }
}

// ---------------------------------------------------------------------------
// Epilogue 1: running top-16 (logit desc, id asc) and online log-sum-exp per row.
// Each thread sees its row's columns in increasing id order, so inserting only values
// strictly above the current 16th keeps equal logits in id order. Per 32-column chunk, only the
// chunk's columns above the 16th are visited, lowest first, one per iteration of a loop the warp
// runs as often as its busiest lane needs (a per-column branch would make the warp run an
// insertion for every column that any of its lanes keeps).
// ---------------------------------------------------------------------------
constexpr int kKeep = 16;
constexpr float kLog2e = 1.4426950408889634f;

struct EpiTopK {
  struct Params {
    float* part_val;    // [parts][M][16]
    int32_t* part_id;   // [parts][M][16]
    float* part_ms;     // [parts][M][2]  (running max, sum of exp(l - max))
    int M;
    int vocab;          // columns ranked (the vocabulary; every launcher must set it)
    float* gate_out;    // [M][gate_cols] fp32: the gate columns' values (gate_cols > 0)
    int gate_base, gate_cols;
  };
  struct State {
    float m, s;
    float v[kKeep];
    int32_t id[kKeep];
  };
  static DF_DEV void init(State& st) {
    st.m = -INFINITY;
    st.s = 0.f;
#pragma unroll
    for (int i = 0; i < kKeep; ++i) {
      st.v[i] = -INFINITY;
      st.id[i] = 0x7fffffff;
    }
  }
  static DF_DEV void insert(State& st, float x, int32_t id) {
    // x > st.v[15]: positions below the insertion point shift down by one.
#pragma unroll
    for (int i = kKeep - 1; i >= 1; --i) {
      const bool down = x > st.v[i - 1];
      const bool here = x > st.v[i];
      st.v[i] = down ? st.v[i - 1] : (here ? x : st.v[i]);
      st.id[i] = down ? st.id[i - 1] : (here ? id : st.id[i]);
    }
    if (x > st.v[0]) {
      st.v[0] = x;
      st.id[0] = id;
    }
  }
  static DF_DEV void consume(State& st, const Params& p, const float (&v)[32], int row, bool row_ok, int col0,
                             int ncols, int col_end) {
    if (!row_ok) return;
    if (col0 + 32 > p.vocab) {
      // past the vocabulary: store the gate columns of this chunk; rank only the vocabulary
      if (p.gate_cols > 0) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          // only this partition's columns (a chunk may run past the partition's end)
          const int c = col0 + i - p.gate_base;
          if (i < ncols && col0 + i < col_end && c >= 0 && c < p.gate_cols)
            p.gate_out[(size_t)row * p.gate_cols + c] = v[i];
        }
      }
      col_end = min(col_end, p.vocab);
    }
    const int nvalid = min(ncols, col_end - col0);
    float cm = -INFINITY;
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i < nvalid) cm = fmaxf(cm, v[i]);
    if (cm == -INFINITY) return;
    if (cm > st.m) {
      st.s *= ex2_approx((st.m - cm) * kLog2e);
      st.m = cm;
    }
    // exp(l - max) as 2^((l - max) log2 e): the difference first, so that the rounding of a large
    // max times log2 e cannot leave a residual that overflows (a fused l log2 e - max log2 e would)
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i < nvalid) acc += ex2_approx((v[i] - st.m) * kLog2e);
    st.s += acc;
    if (cm > st.v[kKeep - 1]) {
      uint32_t cand = 0;  // the chunk's columns above the 16th kept entry
#pragma unroll
      for (int i = 0; i < 32; ++i) cand |= (i < nvalid && v[i] > st.v[kKeep - 1]) ? (1u << i) : 0u;
      while (cand) {
        const int i = __ffs(cand) - 1;
        cand &= cand - 1;
        // v[i] without indexing registers: a tree on the bits of i
        float t[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) t[k] = (i & 1) ? v[2 * k + 1] : v[2 * k];
#pragma unroll
        for (int k = 0; k < 8; ++k) t[k] = (i & 2) ? t[2 * k + 1] : t[2 * k];
#pragma unroll
        for (int k = 0; k < 4; ++k) t[k] = (i & 4) ? t[2 * k + 1] : t[2 * k];
#pragma unroll
        for (int k = 0; k < 2; ++k) t[k] = (i & 8) ? t[2 * k + 1] : t[2 * k];
        const float x = (i & 16) ? t[1] : t[0];
        if (x > st.v[kKeep - 1]) insert(st, x, col0 + i);  // (the 16th rises as entries enter)
      }
    }
  }
  static DF_DEV void finish(const State& st, const Params& p, int row, bool row_ok, int part) {
    if (!row_ok) return;
    const size_t base = ((size_t)part * p.M + row);
    float4* pv = reinterpret_cast<float4*>(p.part_val + base * kKeep);
    int4* pi = reinterpret_cast<int4*>(p.part_id + base * kKeep);
#pragma unroll
    for (int i = 0; i < kKeep / 4; ++i) {
      pv[i] = make_float4(st.v[4 * i], st.v[4 * i + 1], st.v[4 * i + 2], st.v[4 * i + 3]);
      pi[i] = make_int4(st.id[4 * i], st.id[4 * i + 1], st.id[4 * i + 2], st.id[4 * i + 3]);
    }
    reinterpret_cast<float2*>(p.part_ms)[base] = make_float2(st.m, st.s);
  }
};

// ---------------------------------------------------------------------------
// Epilogue 2: one conv layer. Columns are the projection outputs (taps); column pair
// (2g, 2g+1) gives group g's taps for this row's position t. The epilogue normalises them
// (softmax over the pair, unless raw) and writes y[t, c] = a * x[t-1, c] + b * x[t, c]
// for the group's 16 channels, rounded to bf16, with x[-1] = 0 at each block start.
// ---------------------------------------------------------------------------
struct EpiConv {
  struct Params {
    const __nv_bfloat16* x;  // [M, H] layer input
    __nv_bfloat16* y;        // [M, H] layer output
    int M, H, T;
    int raw;                 // 1: taps unnormalised
  };
  struct State {};
  static DF_DEV void init(State&) {}
  static DF_DEV void consume(State&, const Params& p, const float (&v)[32], int row, bool row_ok, int col0,
                             int ncols, int col_end) {
    if (!row_ok) return;
    const bool has_prev = (row % p.T) != 0;
    const __nv_bfloat16* xr = p.x + (size_t)row * p.H;
    const __nv_bfloat16* xp = xr - p.H;
    __nv_bfloat16* yr = p.y + (size_t)row * p.H;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int tap = col0 + 2 * i;
      if (2 * i < ncols && tap < col_end) {
        float a, b;
        const float p0 = v[2 * i], p1 = v[2 * i + 1];
        if (p.raw) {
          a = p0;
          b = p1;
        } else {
          const float mx = fmaxf(p0, p1);
          const float e0 = expf(p0 - mx), e1 = expf(p1 - mx);
          const float inv = 1.f / (e0 + e1);
          a = e0 * inv;
          b = e1 * inv;
        }
        const int c0 = (tap >> 1) * 16;
        const uint4* cur = reinterpret_cast<const uint4*>(xr + c0);
        uint4 cv[2] = {cur[0], cur[1]};
        uint4 pv[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
        if (has_prev) {
          const uint4* prv = reinterpret_cast<const uint4*>(xp + c0);
          pv[0] = prv[0];
          pv[1] = prv[1];
        }
        uint4 out[2];
        const __nv_bfloat162* c2 = reinterpret_cast<const __nv_bfloat162*>(cv);
        const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(pv);
        __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(out);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float2 cf = __bfloat1622float2(c2[k]);
          const float2 pf = __bfloat1622float2(p2[k]);
          const float y0 = fmaf(a, pf.x, b * cf.x);
          const float y1 = fmaf(a, pf.y, b * cf.y);
          o2[k] = __floats2bfloat162_rn(y0, y1);
        }
        uint4* dst = reinterpret_cast<uint4*>(yr + c0);
        dst[0] = out[0];
        dst[1] = out[1];
      }
    }
  }
  static DF_DEV void finish(const State&, const Params&, int, bool, int) {}
};

}  // namespace df
