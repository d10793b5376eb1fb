// Work description of one tcgen05 GEMM launch (host and device).
#pragma once

#include <stdint.h>

namespace df {

struct TcGemmArgs {
  int M;         // rows in total
  int K;         // contraction length, multiple of 64
  int n_total;   // columns in total
  int n_rc;      // row chunks of 128
  int parts;     // column partitions per row chunk
  int a_tail_rows;  // TMA box rows of the last row chunk: its rows rounded up to 8 (128 if full)
  int tile_units;   // columns per tile in units of 16: 8 (128) or 16 (256)
  int pair;         // 1: CTA pairs (cta_group::2) over row-chunk pairs; parts = column ranges per pair
  int32_t* err;  // device error word
  // Extra columns from a second matrix (the context gate): with gate_cols > 0 the last of
  // `parts` partitions holds columns [gate_base, gate_base + gate_cols), rows 0.. of the gate
  // matrix, and the vocabulary [0, n_total) is split over the other parts - 1. gate_base is a
  // multiple of 16 and >= n_total; gate_cols = 0: no gate partition.
  int gate_base = 0;
  int gate_cols = 0;
};

}  // namespace df
