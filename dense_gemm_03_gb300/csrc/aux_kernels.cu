// aux_kernels.cu -- HBM-bound helper kernels of the GEMM path:
//   * split-K reduction: C = half(alpha * sum_s P_s + beta * C), slices summed
//     in ascending order (deterministic), fp32 arithmetic, one rounding;
//   * scale-only update for alpha == 0 or K == 0: C := beta*C (C := 0 when
//     beta == 0, without reading C -- the convention of the "LeetGPU GEMM T4"
//     WMMA sections and the "advanced SGEMM" page for beta == 0).
// Grid-stride loops over rows x column groups; 4-wide vectors where the
// row stride and the base pointer allow it.
#include <cuda_fp16.h>

#include "internal.h"

namespace gb300 {
namespace {

__device__ __forceinline__ float half_bits_to_float(uint16_t b) {
  return __half2float(__ushort_as_half(b));
}
__device__ __forceinline__ uint16_t float_to_half_bits(float x) {
  return __half_as_ushort(__float2half_rn(x));
}

// One thread per group of 4 consecutive columns of one row.
__global__ void splitk_reduce_f16_kernel(const float* __restrict__ ws, long long ws_ld, int splits,
                                         uint16_t* __restrict__ C, long long ldc, int M, int N,
                                         float alpha, float beta) {
  const int groups = (N + 3) >> 2;
  const long long total = static_cast<long long>(M) * groups;
  const long long slice = static_cast<long long>(M) * ws_ld;
  const bool has_c = beta != 0.0f;
  for (long long g = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; g < total;
       g += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int row = static_cast<int>(g / groups);
    const int col = static_cast<int>(g % groups) * 4;
    const float* w = ws + static_cast<long long>(row) * ws_ld + col;
    float4 s = *reinterpret_cast<const float4*>(w);   // ws_ld % 4 == 0, 16-byte aligned
    for (int k = 1; k < splits; ++k) {
      const float4 v = *reinterpret_cast<const float4*>(w + k * slice);
      s.x += v.x;
      s.y += v.y;
      s.z += v.z;
      s.w += v.w;
    }
    const float acc[4] = {s.x, s.y, s.z, s.w};
    uint16_t* c = C + static_cast<long long>(row) * ldc + col;
    const int n = min(4, N - col);
    for (int i = 0; i < n; ++i) {
      const float o = has_c ? __fmaf_rn(alpha, acc[i], beta * half_bits_to_float(c[i]))
                            : alpha * acc[i];
      c[i] = float_to_half_bits(o);
    }
  }
}

__global__ void scale_f16_kernel(uint16_t* __restrict__ C, long long ldc, int M, int N,
                                 float beta) {
  const long long total = static_cast<long long>(M) * N;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int row = static_cast<int>(i / N), col = static_cast<int>(i % N);
    uint16_t* c = C + static_cast<long long>(row) * ldc + col;
    *c = (beta == 0.0f) ? float_to_half_bits(0.0f) : float_to_half_bits(beta * half_bits_to_float(*c));
  }
}

__global__ void scale_f32_kernel(float* __restrict__ C, long long ldc, int M, int N, float beta) {
  const long long total = static_cast<long long>(M) * N;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int row = static_cast<int>(i / N), col = static_cast<int>(i % N);
    float* c = C + static_cast<long long>(row) * ldc + col;
    *c = (beta == 0.0f) ? 0.0f : beta * *c;
  }
}

}  // namespace

cudaError_t launch_splitk_reduce_f16(const float* ws, long long ws_ld, int splits, uint16_t* C,
                                     long long ldc, int M, int N, float alpha, float beta,
                                     int grid, cudaStream_t stream) {
  splitk_reduce_f16_kernel<<<grid, 256, 0, stream>>>(ws, ws_ld, splits, C, ldc, M, N, alpha, beta);
  return cudaGetLastError();
}

cudaError_t launch_scale_f16(uint16_t* C, long long ldc, int M, int N, float beta, int grid,
                             cudaStream_t stream) {
  scale_f16_kernel<<<grid, 256, 0, stream>>>(C, ldc, M, N, beta);
  return cudaGetLastError();
}

cudaError_t launch_scale_f32(float* C, long long ldc, int M, int N, float beta, int grid,
                             cudaStream_t stream) {
  scale_f32_kernel<<<grid, 256, 0, stream>>>(C, ldc, M, N, beta);
  return cudaGetLastError();
}

}  // namespace gb300
