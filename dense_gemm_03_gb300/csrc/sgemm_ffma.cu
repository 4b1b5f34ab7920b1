// sgemm_ffma.cu -- fp32 SGEMM on the CUDA cores (FFMA), C := alpha*A*B + beta*C.
//
// Design follows the "advanced SGEMM on NVIDIA GPUs" page (section on tiling
// and data movement), re-derived for sm_103a:
//   * 128 x 128 output tile per 256-thread block, k-slices of 16, two blocks
//     per SM (at most 128 registers a thread: 16 warps per SM keep the FMA
//     pipe busy where one block of 8 warps with double-buffered fragments and
//     146 registers left it idle a third of the time);
//   * the A slice (128 x 16) goes through registers (two 16-byte loads a
//     thread) and is stored TRANSPOSED in shared memory with a padded leading
//     dimension of 132 floats, so each thread reads 4 consecutive rows with one
//     16-byte load and the transposing stores are free of bank conflicts; the
//     B slice (16 x 128) is copied as is by cp.async (no registers on the
//     way); both are double-buffered in shared memory, one barrier per slice;
//   * 8 warps each own a 32 x 64 sub-tile; a thread owns an 8 x 8 block made
//     of four 4 x 4 pieces (rows tm*4 and 16+tm*4, columns tn*4 and 32+tn*4
//     of its warp's sub-tile), with tm = lane % 4 and tn = lane / 4, so a
//     16-byte B fragment is shared by at most 4 consecutive lanes and an A
//     fragment by lanes 4 apart;
//   * the products use the packed two-lane FMA of sm_100-class GPUs
//     (fma.rn.f32x2, one instruction for two adjacent columns of a row; each
//     lane is an ordinary fp32 fused multiply-add, so the result is the same
//     as with scalar FMAs in the same k order), which halves the FMA
//     instructions per k step;
//   * with that thread layout every 16-byte store of C from a warp covers
//     four full 128-byte row segments, so C is written (and, when beta != 0,
//     read) coalesced straight from registers;
//   * beta == 0: C is not read.
// VEC selects 16-byte global loads/copies/stores (aligned base pointers and
// leading dimensions that are multiples of 4 floats -- the run-time check of
// the same page's kernel-selection section); otherwise every access is a
// predicated 4-byte one.  Ragged M, N, K are zero-filled on load (a copy of
// zero source bytes for B) and masked on store.
#include "internal.h"

namespace gb300 {
namespace {

constexpr int kBM = 128, kBN = 128, kBK = 16;
constexpr int kLdA = kBM + 4;   // padded, transposed A slice

// Global -> shared copies that bypass registers; a false `pred` copies zero
// source bytes (the destination is zero-filled) from a valid address.
__device__ __forceinline__ void cp_async16(uint32_t dst, const float* src, bool pred) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(pred ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const float* src, bool pred) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(pred ? 4 : 0)
               : "memory");
}

template <bool VEC>
__global__ void __launch_bounds__(256, 2) sgemm_ffma_kernel(const SgemmArgs p) {
  __shared__ __align__(16) float As[2][kBK][kLdA];
  __shared__ __align__(16) float Bs[2][kBK][kBN];

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int wm = warp >> 1, wn = warp & 1;            // 4 x 2 warps
  const int tm = lane & 3, tn = lane >> 2;            // 4 x 8 lanes
  const int m0 = blockIdx.y * kBM, n0 = blockIdx.x * kBN;

  // copy assignment: A row a_r, k a_k .. +3 and a_k + 8 .. +11 (through
  // registers); B k rows b_k and b_k + 8, columns b_c .. +3 (cp.async)
  const int a_r = tid >> 1, a_k = (tid & 1) * 4;
  const int b_k = tid >> 5, b_c = (tid & 31) * 4;
  const int M = p.M, N = p.N, K = p.K;

  float4 a_st, a_st2;
  auto ld4 = [&](int k0) -> float4 {
    const int row = m0 + a_r, kk = k0;
    float4 v;
    if (VEC && row < M && kk + 4 <= K) {
      v = __ldg(reinterpret_cast<const float4*>(p.A + static_cast<long long>(row) * p.lda + kk));
    } else {
      const float* ar = p.A + static_cast<long long>(row) * p.lda;
      const bool rok = row < M;
      v.x = (rok && kk + 0 < K) ? __ldg(ar + kk + 0) : 0.f;
      v.y = (rok && kk + 1 < K) ? __ldg(ar + kk + 1) : 0.f;
      v.z = (rok && kk + 2 < K) ? __ldg(ar + kk + 2) : 0.f;
      v.w = (rok && kk + 3 < K) ? __ldg(ar + kk + 3) : 0.f;
    }
    return v;
  };
  auto load_tile = [&](int k0) {
    a_st = ld4(k0 + a_k);
    a_st2 = ld4(k0 + a_k + 8);
  };
  auto copy_b1 = [&](int k0, int buf, int bk) {
    const int kr = k0 + bk, col = n0 + b_c;
    const bool kok = kr < K;
    const float* br = p.B + static_cast<long long>(kok ? kr : 0) * p.ldb;
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(&Bs[buf][bk][b_c]));
    if (VEC && kok && col + 4 <= N) {
      cp_async16(d, br + col, true);
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const bool ok = kok && col + j < N;
        cp_async4(d + 4 * j, ok ? br + col + j : p.B, ok);
      }
    }
  };
  auto copy_b = [&](int k0, int buf) {
    copy_b1(k0, buf, b_k);
    copy_b1(k0, buf, b_k + 8);
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  auto store_tile = [&](int buf) {
    As[buf][a_k + 0][a_r] = a_st.x;
    As[buf][a_k + 1][a_r] = a_st.y;
    As[buf][a_k + 2][a_r] = a_st.z;
    As[buf][a_k + 3][a_r] = a_st.w;
    As[buf][a_k + 8][a_r] = a_st2.x;
    As[buf][a_k + 9][a_r] = a_st2.y;
    As[buf][a_k + 10][a_r] = a_st2.z;
    As[buf][a_k + 11][a_r] = a_st2.w;
  };

  const int a_off0 = wm * 32 + tm * 4, a_off1 = a_off0 + 16;
  const int b_off0 = wn * 64 + tn * 4, b_off1 = b_off0 + 32;
  float4 fa[2], fb[2];
  // one k step's fragments (single-buffered: the second block on the SM
  // hides their latency)
  auto load_frag = [&](int buf, int k) {
    fa[0] = *reinterpret_cast<const float4*>(&As[buf][k][a_off0]);
    fa[1] = *reinterpret_cast<const float4*>(&As[buf][k][a_off1]);
    fb[0] = *reinterpret_cast<const float4*>(&Bs[buf][k][b_off0]);
    fb[1] = *reinterpret_cast<const float4*>(&Bs[buf][k][b_off1]);
  };

  // acc[i][q] holds columns 2q and 2q+1 of row i: one packed two-lane FMA
  // (fma.rn.f32x2) updates both, so a k step is 32 instructions, not 64.
  float2 acc[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[i][q] = make_float2(0.f, 0.f);

  const int nkt = (K + kBK - 1) / kBK;
  load_tile(0);
  copy_b(0, 0);
  store_tile(0);
  asm volatile("cp.async.wait_group 0;" ::: "memory");   // this thread's copies of B
  __syncthreads();
  int buf = 0;

  for (int kt = 0; kt < nkt; ++kt) {
    const bool has_next = kt + 1 < nkt;
    if (has_next) {
      load_tile((kt + 1) * kBK);
      copy_b((kt + 1) * kBK, buf ^ 1);
    }
#pragma unroll
    for (int k = 0; k < kBK; ++k) {
      load_frag(buf, k);
      const float a[8] = {fa[0].x, fa[0].y, fa[0].z, fa[0].w, fa[1].x, fa[1].y, fa[1].z, fa[1].w};
      const float2 b[4] = {make_float2(fb[0].x, fb[0].y), make_float2(fb[0].z, fb[0].w),
                           make_float2(fb[1].x, fb[1].y), make_float2(fb[1].z, fb[1].w)};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float2 ai = make_float2(a[i], a[i]);
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[i][q] = __ffma2_rn(ai, b[q], acc[i][q]);
      }
    }
    if (has_next) {
      store_tile(buf ^ 1);
      asm volatile("cp.async.wait_group 0;" ::: "memory");
      __syncthreads();
      buf ^= 1;
    }
  }

  // epilogue: alpha*acc (+ beta*C), straight from registers
  auto elem = [&](int i, int j) { return (j & 1) ? acc[i][j >> 1].y : acc[i][j >> 1].x; };
  const bool has_c = p.beta != 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int row = m0 + (i < 4 ? a_off0 + i : a_off1 + (i - 4));
    if (row >= M) continue;
    float* crow = p.C + static_cast<long long>(row) * p.ldc;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int col = n0 + (h == 0 ? b_off0 : b_off1);
      float o[4];
      if (VEC && col + 4 <= N) {
        float4 c = make_float4(0.f, 0.f, 0.f, 0.f);
        if (has_c) c = *reinterpret_cast<const float4*>(crow + col);
        const float cv[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
          o[j] = has_c ? fmaf(p.alpha, elem(i, h * 4 + j), p.beta * cv[j]) : p.alpha * elem(i, h * 4 + j);
        *reinterpret_cast<float4*>(crow + col) = make_float4(o[0], o[1], o[2], o[3]);
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (col + j < N) {
            const float a = elem(i, h * 4 + j);
            crow[col + j] = has_c ? fmaf(p.alpha, a, p.beta * crow[col + j]) : p.alpha * a;
          }
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_sgemm_ffma(bool vec, const SgemmArgs& args, cudaStream_t stream) {
  const dim3 grid((args.N + kBN - 1) / kBN, (args.M + kBM - 1) / kBM);
  if (grid.y > 65535u) return cudaErrorInvalidConfiguration;
  if (vec)
    sgemm_ffma_kernel<true><<<grid, 256, 0, stream>>>(args);
  else
    sgemm_ffma_kernel<false><<<grid, 256, 0, stream>>>(args);
  return counted_launch(cudaGetLastError());
}

}  // namespace gb300
