// gemm_f16_tc.cu -- launchers of the tcgen05 half-precision GEMM kernel
// (gemm_f16_tc_kernel.cuh) for half-precision C: TMA, predicated and
// partial-sum epilogues, single CTAs and CTA pairs.
#include "gemm_f16_tc_kernel.cuh"

namespace gb300 {
namespace {

template <int BN>
cudaError_t launch_bn(int load, int epi, const CUtensorMap& a, const CUtensorMap& b,
                      const CUtensorMap& c, const TcArgs& args, int grid, cudaStream_t s) {
  if (load == kLoadTma) {
    if (epi == kEpiTma) return launch_one<BN, kLoadTma, kEpiTma, false>(a, b, c, args, grid, s);
    if (epi == kEpiManual)
      return launch_one<BN, kLoadTma, kEpiManual, false>(a, b, c, args, grid, s);
    return launch_one<BN, kLoadTma, kEpiPartial, false>(a, b, c, args, grid, s);
  }
  if (epi == kEpiTma) return launch_one<BN, kLoadManual, kEpiTma, false>(a, b, c, args, grid, s);
  if (epi == kEpiManual)
    return launch_one<BN, kLoadManual, kEpiManual, false>(a, b, c, args, grid, s);
  return launch_one<BN, kLoadManual, kEpiPartial, false>(a, b, c, args, grid, s);
}

}  // namespace

cudaError_t launch_gemm_f16_tc(int bn, int load_mode, int epi_mode, const CUtensorMap& tmA,
                               const CUtensorMap& tmB, const CUtensorMap& tmC, const TcArgs& args,
                               int grid, cudaStream_t stream, int kpb) {
  if (epi_mode == kEpiF32)
    return launch_gemm_f16_tc_f32(bn, load_mode, tmA, tmB, args, grid, stream);
  // two k-blocks per ring stage: 64-wide tiles with TMA loads and epilogue
  if (kpb == 2)
    return bn == 64 && load_mode == kLoadTma && epi_mode == kEpiTma
               ? launch_one<64, kLoadTma, kEpiTma, false, 128, 128, 2>(tmA, tmB, tmC, args, grid,
                                                                        stream)
               : cudaErrorInvalidValue;
  switch (bn) {
    case 256: return launch_bn<256>(load_mode, epi_mode, tmA, tmB, tmC, args, grid, stream);
    case 128: return launch_bn<128>(load_mode, epi_mode, tmA, tmB, tmC, args, grid, stream);
    case 64: return launch_bn<64>(load_mode, epi_mode, tmA, tmB, tmC, args, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_gemm_f16_tc_pair(int bn, int epi_mode, const CUtensorMap& tmA,
                                    const CUtensorMap& tmB, const CUtensorMap& tmC,
                                    const TcArgs& args, int grid, cudaStream_t stream, int kpb) {
  if (epi_mode == kEpiF32 || epi_mode == kEpiF32Tma)
    return bn == 256 ? launch_gemm_f16_tc_pair_f32(epi_mode, tmA, tmB, tmC, args, grid, stream)
                     : cudaErrorInvalidValue;
  if (bn != 256)
    return launch_gemm_f16_tc_pair_narrow(bn, epi_mode, tmA, tmB, tmC, args, grid, stream);
  if (epi_mode == kEpiTma)
    return kpb == 2 ? launch_one<256, kLoadTma, kEpiTma, true, 128, 128, 2>(tmA, tmB, tmC, args,
                                                                             grid, stream)
                    : launch_one<256, kLoadTma, kEpiTma, true>(tmA, tmB, tmC, args, grid, stream);
  if (kpb == 2) return cudaErrorInvalidValue;
  if (epi_mode == kEpiManual)
    return launch_one<256, kLoadTma, kEpiManual, true>(tmA, tmB, tmC, args, grid, stream);
  return cudaErrorInvalidValue;
}

int tc_pair_max_clusters(int epi_mode) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (epi_mode == kEpiF32 || epi_mode == kEpiF32Tma) return tc_pair_max_clusters_f32(epi_mode);
  return epi_mode == kEpiTma ? pair_max_clusters<kEpiTma>(dev) : pair_max_clusters<kEpiManual>(dev);
}

int tc_threads(int load_mode) {
  return load_mode == kLoadTma ? Roles<kLoadTma>::kThreads : Roles<kLoadManual>::kThreads;
}

int tc_epilogue_tile_cols() { return kSubCols; }

}  // namespace gb300
