// aux_kernels.cu -- HBM-bound helper kernels of the GEMM path:
//   * split-K reduction: C = half(alpha * sum_s P_s + beta * C), slices summed
//     in ascending order (deterministic), fp32 arithmetic, one rounding;
//   * realignment of an operand whose rows are not 16-byte aligned into an
//     aligned copy, so that the tensor-core kernel can load it by TMA;
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

// 16 bytes starting `m` bytes (m even, 2..14) into the 32 bytes lo|hi.
__device__ __forceinline__ uint4 shift_bytes(uint4 lo, uint4 hi, uint32_t m) {
  const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
  const uint32_t sh = (m & 3u) * 8u;
  uint32_t o[4];
  switch (m >> 2) {
#define GB300_SEL(Q)                                                          \
  case Q:                                                                     \
    for (int i = 0; i < 4; ++i) o[i] = __funnelshift_r(w[Q + i], w[Q + i + 1], sh); \
    break;
    GB300_SEL(0)
    GB300_SEL(1)
    GB300_SEL(2)
    default:
      for (int i = 0; i < 4; ++i) o[i] = __funnelshift_r(w[3 + i], w[4 + i], sh);
      break;
#undef GB300_SEL
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// dst[r][c] = src[r][c] for c < cols, 0 for cols <= c < ldd (ldd % 8 == 0,
// dst 16-byte aligned).  One thread writes 8 halves.  A fully valid source
// piece at any 2-byte alignment is read as the (at most two) 16-byte-aligned
// blocks that contain it -- blocks that hold at least one element of the
// piece, so the reads never leave memory the caller owns -- and shifted into
// place; the ragged end of a row uses element loads.
__global__ void realign_f16_kernel(const uint16_t* __restrict__ src, long long lds,
                                   uint16_t* __restrict__ dst, long long ldd, int rows, int cols) {
  const long long groups = ldd / 8;
  const long long total = static_cast<long long>(rows) * groups;
  for (long long g = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; g < total;
       g += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int r = static_cast<int>(g / groups);
    const int c0 = static_cast<int>(g % groups) * 8;
    const uint16_t* p = src + static_cast<long long>(r) * lds + c0;
    uint4 v;
    if (c0 + 8 <= cols) {
      const uintptr_t a = reinterpret_cast<uintptr_t>(p);
      const uint32_t m = static_cast<uint32_t>(a & 15u);
      const uint4* blk = reinterpret_cast<const uint4*>(a - m);
      // m is even: half pointers are 2-byte aligned (checked by the host)
      v = (m == 0) ? __ldg(blk) : shift_bytes(__ldg(blk), __ldg(blk + 1), m);
    } else {
      uint32_t h[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) h[i] = (c0 + i < cols) ? static_cast<uint32_t>(__ldg(p + i)) : 0u;
      v = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16),
                     h[6] | (h[7] << 16));
    }
    *reinterpret_cast<uint4*>(dst + static_cast<long long>(r) * ldd + c0) = v;
  }
}

}  // namespace

cudaError_t launch_realign_f16(const uint16_t* src, long long lds, uint16_t* dst, long long ldd,
                               int rows, int cols, int grid, cudaStream_t stream) {
  realign_f16_kernel<<<grid, 256, 0, stream>>>(src, lds, dst, ldd, rows, cols);
  return cudaGetLastError();
}

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
