// gemm_f16_skinny.cu -- launchers of the tcgen05 half-precision GEMM kernel
// (gemm_f16_tc_kernel.cuh) for the bandwidth-bound shapes: at most 64 rows,
// where each k-block stages only 32 or 64 rows of A, so the ring has more
// stages and keeps more of B in flight (these shapes stream B from HBM once);
// and tall shapes on 64-row tiles (tcgen05.mma with M = 64), which doubles
// their tiles so that whole-K units fill the SMs.  Kept apart from the other
// instances so that they compile in parallel.
#include "gemm_f16_tc_kernel.cuh"

namespace gb300 {
namespace {

template <int AM>
cudaError_t launch_am(int epi, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c,
                      const TcArgs& args, int grid, cudaStream_t s) {
  switch (epi) {
    case kEpiTma: return launch_one<128, kLoadTma, kEpiTma, false, AM>(a, b, c, args, grid, s);
    case kEpiManual: return launch_one<128, kLoadTma, kEpiManual, false, AM>(a, b, c, args, grid, s);
    case kEpiF32: return launch_one<128, kLoadTma, kEpiF32, false, AM>(a, b, c, args, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_gemm_f16_tc_skinny(int am, int epi_mode, const CUtensorMap& tmA,
                                      const CUtensorMap& tmB, const CUtensorMap& tmC,
                                      const TcArgs& args, int grid, cudaStream_t stream) {
  if (am == 32) return launch_am<32>(epi_mode, tmA, tmB, tmC, args, grid, stream);
  if (am == 64) return launch_am<64>(epi_mode, tmA, tmB, tmC, args, grid, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_gemm_f16_tc_m64(const CUtensorMap& tmA, const CUtensorMap& tmB,
                                   const CUtensorMap& tmC, const TcArgs& args, int grid,
                                   cudaStream_t stream) {
  return launch_one<64, kLoadTma, kEpiTma, false, 64, 64>(tmA, tmB, tmC, args, grid, stream);
}

}  // namespace gb300
