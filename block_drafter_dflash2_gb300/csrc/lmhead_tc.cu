// bf16 instantiations of the tcgen05 GEMM: LM head with the top-K/lse epilogue, and one
// conv layer with the tap-mix epilogue.
#include "kernels.h"
#include "launch_util.h"
#include "tc_gemm.cuh"

namespace df {

namespace {
// CTA pairs (more than one row chunk): clusters of two, one per (row-chunk pair, column range).
// The launch waits for the previous kernel as usual.
template <class Epi>
cudaError_t launch_gemm_pair(const CUtensorMap& a, const CUtensorMap& a_tail, const CUtensorMap& b128,
                             const CUtensorMap& b16, const CUtensorMap& g128, const CUtensorMap& g16,
                             const TcGemmArgs& args, const typename Epi::Params& ep, cudaStream_t s) {
  if (!args.pair || args.tile_units % 2 != 0 || args.gate_base % 32 != 0) return cudaErrorInvalidValue;
  static unsigned char smem_done[64];
  cudaError_t e = smem_opt_in(reinterpret_cast<const void*>(tc_gemm_pair_kernel<Epi>), smem_done);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * ((args.n_rc + 1) / 2) * args.parts));
  cfg.blockDim = dim3(kPairThreads);
  cfg.dynamicSmemBytes = kPairSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, tc_gemm_pair_kernel<Epi>, a, a_tail, b128, b16, g128, g16, args, ep);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <class Epi>
cudaError_t launch_gemm(const CUtensorMap& a, const CUtensorMap& a_tail, const CUtensorMap& b128,
                        const CUtensorMap& b16, const CUtensorMap& g128, const CUtensorMap& g16,
                        const TcGemmArgs& args, const typename Epi::Params& ep, cudaStream_t s) {
  if (args.pair) return cudaErrorInvalidValue;
  static unsigned char smem_done[64];
  cudaError_t e = smem_opt_in(reinterpret_cast<const void*>(tc_gemm_kernel<Epi>), smem_done);
  if (e != cudaSuccess) return e;
  const int grid = args.n_rc * args.parts;
  // With one row chunk the launch is a programmatic dependent of the previous kernel: the
  // producer waits for it (griddepcontrol.wait) before reading the rows, so the prologue
  // overlaps its end (2-9 us saved at 8-64 rows). With several chunks the CTAs would be placed
  // in the order the previous kernel's CTAs leave their SMs, which measured 30-50 us slower at
  // 256 rows; those launches wait for the previous kernel as usual.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = kGemmSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = args.n_rc == 1 ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, tc_gemm_kernel<Epi>, a, a_tail, b128, b16, g128, g16, args, ep);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_lmhead_topk_bf16(const CUtensorMap& a, const CUtensorMap& a_tail, const CUtensorMap& b128,
                                    const CUtensorMap& b16, const CUtensorMap& g128, const CUtensorMap& g16,
                                    const TcGemmArgs& args, int vocab, float* part_val, int32_t* part_id,
                                    float* part_ms, float* gate_out, cudaStream_t s) {
  if (args.gate_cols > 0 && (args.gate_base < vocab || args.gate_base % 16 != 0 || gate_out == nullptr ||
                             args.n_total != vocab || args.parts < 2))
    return cudaErrorInvalidValue;
  EpiTopK::Params ep{part_val, part_id, part_ms, args.M, vocab, gate_out, args.gate_base, args.gate_cols};
  if (args.pair) return launch_gemm_pair<EpiTopK>(a, a_tail, b128, b16, g128, g16, args, ep, s);
  return launch_gemm<EpiTopK>(a, a_tail, b128, b16, g128, g16, args, ep, s);
}

cudaError_t launch_conv_layer_bf16(const CUtensorMap& a, const CUtensorMap& a_tail, const CUtensorMap& b128,
                                   const CUtensorMap& b16, const TcGemmArgs& args, const void* x, void* y, int T,
                                   int raw, cudaStream_t s) {
  EpiConv::Params ep{reinterpret_cast<const __nv_bfloat16*>(x), reinterpret_cast<__nv_bfloat16*>(y), args.M,
                     args.K, T, raw};
  return launch_gemm<EpiConv>(a, a_tail, b128, b16, b128, b16, args, ep, s);
}

}  // namespace df
