// gemm_f16_pair_narrow.cu -- launchers of the CTA-pair tcgen05 half-precision
// GEMM (gemm_f16_tc_kernel.cuh) with 224- and 192-wide pair tiles, for shapes
// whose 256-wide tiles would leave a partial last wave of pairs (at 4096^3:
// 256 tiles of 256 x 256 on 76 pairs, but 304 = 4 x 76 tiles of 256 x 224).
// Kept apart from gemm_f16_tc.cu so that these instances compile in parallel.
#include "gemm_f16_tc_kernel.cuh"

namespace gb300 {

cudaError_t launch_gemm_f16_tc_pair_narrow(int bn, int epi_mode, const CUtensorMap& tmA,
                                           const CUtensorMap& tmB, const CUtensorMap& tmC,
                                           const TcArgs& args, int grid, cudaStream_t stream) {
  if (bn == 224) {
    if (epi_mode == kEpiTma)
      return launch_one<224, kLoadTma, kEpiTma, true>(tmA, tmB, tmC, args, grid, stream);
    if (epi_mode == kEpiManual)
      return launch_one<224, kLoadTma, kEpiManual, true>(tmA, tmB, tmC, args, grid, stream);
  } else if (bn == 192) {
    if (epi_mode == kEpiTma)
      return launch_one<192, kLoadTma, kEpiTma, true>(tmA, tmB, tmC, args, grid, stream);
    if (epi_mode == kEpiManual)
      return launch_one<192, kLoadTma, kEpiManual, true>(tmA, tmB, tmC, args, grid, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace gb300
