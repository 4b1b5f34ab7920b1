// sgemm_ffma.cu -- fp32 SGEMM on the CUDA cores (FFMA), C := alpha*A*B + beta*C.
//
// Design follows the "advanced SGEMM on NVIDIA GPUs" page (section on tiling
// and data movement), re-derived for sm_103a:
//   * 128 x 128 output tile per 256-thread block, k-slices of 8;
//   * the A slice (128 x 8) is stored TRANSPOSED in shared memory with a
//     padded leading dimension of 132 floats, so each thread reads 4
//     consecutive rows with one 16-byte load and the transposing stores are
//     free of bank conflicts; the B slice (8 x 128) is stored as is;
//   * both slices are double-buffered in shared memory (one barrier per
//     k-slice) and the per-thread fragments are double-buffered in registers;
//   * 8 warps each own a 32 x 64 sub-tile; a thread owns an 8 x 8 block made
//     of four 4 x 4 pieces (rows tm*4 and 16+tm*4, columns tn*4 and 32+tn*4
//     of its warp's sub-tile), with tm = lane % 4 and tn = lane / 4, so a
//     16-byte B fragment is shared by at most 4 consecutive lanes and an A
//     fragment by lanes 4 apart;
//   * the products use the packed two-lane FMA of sm_100-class GPUs
//     (fma.rn.f32x2, one instruction for two adjacent columns of a row; each
//     lane is an ordinary fp32 fused multiply-add, so the result is the same
//     as with scalar FMAs in the same k order), which halves the FMA
//     instructions per k step; the kernel then needs ~146 registers and runs
//     one 256-thread block per SM;
//   * with that thread layout every 16-byte store of C from a warp covers
//     four full 128-byte row segments, so C is written (and, when beta != 0,
//     read) coalesced straight from registers;
//   * beta == 0: C is not read.
// VEC selects 16-byte global loads/stores (aligned base pointers and leading
// dimensions that are multiples of 4 floats -- the run-time check of the same
// page's kernel-selection section); otherwise every access is a predicated
// scalar access.  Ragged M, N, K are zero-filled on load and masked on store.
#include "internal.h"

namespace gb300 {
namespace {

constexpr int kBM = 128, kBN = 128, kBK = 8;
constexpr int kLdA = kBM + 4;   // padded, transposed A slice

template <bool VEC>
__global__ void __launch_bounds__(256, 1) sgemm_ffma_kernel(const SgemmArgs p) {
  __shared__ __align__(16) float As[2][kBK][kLdA];
  __shared__ __align__(16) float Bs[2][kBK][kBN];

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int wm = warp >> 1, wn = warp & 1;            // 4 x 2 warps
  const int tm = lane & 3, tn = lane >> 2;            // 4 x 8 lanes
  const int m0 = blockIdx.y * kBM, n0 = blockIdx.x * kBN;

  // global -> register staging assignment
  const int a_r = tid >> 1, a_k = (tid & 1) * 4;      // A: row, first of 4 k
  const int b_k = tid >> 5, b_c = (tid & 31) * 4;     // B: k row, first of 4 columns
  const int M = p.M, N = p.N, K = p.K;

  float4 a_st, b_st;
  auto load_tile = [&](int k0) {
    const int row = m0 + a_r, kk = k0 + a_k;
    if (VEC && row < M && kk + 4 <= K) {
      a_st = __ldg(reinterpret_cast<const float4*>(p.A + static_cast<long long>(row) * p.lda + kk));
    } else {
      const float* ar = p.A + static_cast<long long>(row) * p.lda;
      const bool rok = row < M;
      a_st.x = (rok && kk + 0 < K) ? __ldg(ar + kk + 0) : 0.f;
      a_st.y = (rok && kk + 1 < K) ? __ldg(ar + kk + 1) : 0.f;
      a_st.z = (rok && kk + 2 < K) ? __ldg(ar + kk + 2) : 0.f;
      a_st.w = (rok && kk + 3 < K) ? __ldg(ar + kk + 3) : 0.f;
    }
    const int kr = k0 + b_k, col = n0 + b_c;
    if (VEC && kr < K && col + 4 <= N) {
      b_st = __ldg(reinterpret_cast<const float4*>(p.B + static_cast<long long>(kr) * p.ldb + col));
    } else {
      const float* br = p.B + static_cast<long long>(kr) * p.ldb;
      const bool kok = kr < K;
      b_st.x = (kok && col + 0 < N) ? __ldg(br + col + 0) : 0.f;
      b_st.y = (kok && col + 1 < N) ? __ldg(br + col + 1) : 0.f;
      b_st.z = (kok && col + 2 < N) ? __ldg(br + col + 2) : 0.f;
      b_st.w = (kok && col + 3 < N) ? __ldg(br + col + 3) : 0.f;
    }
  };
  auto store_tile = [&](int buf) {
    As[buf][a_k + 0][a_r] = a_st.x;
    As[buf][a_k + 1][a_r] = a_st.y;
    As[buf][a_k + 2][a_r] = a_st.z;
    As[buf][a_k + 3][a_r] = a_st.w;
    *reinterpret_cast<float4*>(&Bs[buf][b_k][b_c]) = b_st;
  };

  const int a_off0 = wm * 32 + tm * 4, a_off1 = a_off0 + 16;
  const int b_off0 = wn * 64 + tn * 4, b_off1 = b_off0 + 32;
  float4 fa[2][2], fb[2][2];
  auto load_frag = [&](int buf, int k, int slot) {
    fa[slot][0] = *reinterpret_cast<const float4*>(&As[buf][k][a_off0]);
    fa[slot][1] = *reinterpret_cast<const float4*>(&As[buf][k][a_off1]);
    fb[slot][0] = *reinterpret_cast<const float4*>(&Bs[buf][k][b_off0]);
    fb[slot][1] = *reinterpret_cast<const float4*>(&Bs[buf][k][b_off1]);
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
  store_tile(0);
  __syncthreads();
  int buf = 0;
  load_frag(0, 0, 0);

  for (int kt = 0; kt < nkt; ++kt) {
    const bool has_next = kt + 1 < nkt;
    if (has_next) load_tile((kt + 1) * kBK);
#pragma unroll
    for (int k = 0; k < kBK; ++k) {
      if (k + 1 < kBK) load_frag(buf, k + 1, (k + 1) & 1);
      const int s = k & 1;
      const float a[8] = {fa[s][0].x, fa[s][0].y, fa[s][0].z, fa[s][0].w,
                          fa[s][1].x, fa[s][1].y, fa[s][1].z, fa[s][1].w};
      const float2 b[4] = {make_float2(fb[s][0].x, fb[s][0].y), make_float2(fb[s][0].z, fb[s][0].w),
                           make_float2(fb[s][1].x, fb[s][1].y), make_float2(fb[s][1].z, fb[s][1].w)};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float2 ai = make_float2(a[i], a[i]);
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[i][q] = __ffma2_rn(ai, b[q], acc[i][q]);
      }
    }
    if (has_next) {
      store_tile(buf ^ 1);
      __syncthreads();
      buf ^= 1;
      load_frag(buf, 0, 0);
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
