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
  int32_t* err;  // device error word
};

}  // namespace df
