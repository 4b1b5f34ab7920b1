// gemm_f16_f32out.cu -- launchers of the tcgen05 half-precision GEMM kernel
// (gemm_f16_tc_kernel.cuh) with an fp32 C: half operands, fp32 accumulation,
// and the epilogue alpha*acc + beta*C kept in fp32 (the WMMA kernel of the
// "Tensorcore_wmma_vs_fp32 test code" page stores its fp32 accumulator
// fragment to a float C).  Kept apart from gemm_f16_tc.cu so that the two
// sets of kernel instances compile in parallel.
#include "gemm_f16_tc_kernel.cuh"

namespace gb300 {

cudaError_t launch_gemm_f16_tc_f32(int bn, int load_mode, const CUtensorMap& tmA,
                                   const CUtensorMap& tmB, const TcArgs& args, int grid,
                                   cudaStream_t stream) {
  const CUtensorMap& c = tmA;   // no C map: C is written from registers
  const bool tma = load_mode == kLoadTma;
  switch (bn) {
    case 256:
      return tma ? launch_one<256, kLoadTma, kEpiF32, false>(tmA, tmB, c, args, grid, stream)
                 : launch_one<256, kLoadManual, kEpiF32, false>(tmA, tmB, c, args, grid, stream);
    case 128:
      return tma ? launch_one<128, kLoadTma, kEpiF32, false>(tmA, tmB, c, args, grid, stream)
                 : launch_one<128, kLoadManual, kEpiF32, false>(tmA, tmB, c, args, grid, stream);
    case 64:
      return tma ? launch_one<64, kLoadTma, kEpiF32, false>(tmA, tmB, c, args, grid, stream)
                 : launch_one<64, kLoadManual, kEpiF32, false>(tmA, tmB, c, args, grid, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

cudaError_t launch_gemm_f16_tc_pair_f32(int epi_mode, const CUtensorMap& tmA,
                                        const CUtensorMap& tmB, const CUtensorMap& tmC,
                                        const TcArgs& args, int grid, cudaStream_t stream) {
  if (epi_mode == kEpiF32Tma)
    return launch_one<256, kLoadTma, kEpiF32Tma, true>(tmA, tmB, tmC, args, grid, stream);
  return launch_one<256, kLoadTma, kEpiF32, true>(tmA, tmB, tmA, args, grid, stream);
}

int tc_pair_max_clusters_f32(int epi_mode) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  return epi_mode == kEpiF32Tma ? pair_max_clusters<kEpiF32Tma>(dev) : pair_max_clusters<kEpiF32>(dev);
}

}  // namespace gb300
