// splitk_static.cu -- an allocation-free form of the split-K half-precision
// GEMM.
//
// The split-K path of gemm_f16_ld keeps its fp32 partial sums in a workspace
// that the library allocates with cudaMalloc the first time a shape needs it.
// Some callers cannot allow that: code that must not allocate device memory
// once it is running -- because cudaMalloc may synchronise the whole device
// and can fail at run time, or because every device allocation must come from
// the caller's own memory planner or a fixed budget set at start-up.  For
// them, gemm_f16_splitk_noalloc runs the same two kernels (tensor-core partial
// GEMM, then the fixed-order reduction with the alpha/beta epilogue) on a
// scratch area that is a file-scope device array of GEMM_STATIC_SCRATCH_BYTES.
// That array exists on every GPU that loads this library, for as long as the
// library stays loaded; the entry point itself never calls cudaMalloc,
// cudaFree or any other allocating routine.
//
// Set-up: the first call on each device (with that device current) looks up
// the device address of the array with cudaGetSymbolAddress and keeps it; in
// host code the array's name is only a host-side stand-in and must never be
// handed to a kernel.  Make that first call before any stream capture.
//
// Sharing: every call uses the same array and it keeps the last call's
// contents.  Nothing in it has to start at zero: each partial sum the
// reduction uses is written by the same call first.  Calls whose kernels
// overlap on the GPU (for example on two streams without ordering) race on
// the array and give wrong results; order them on one stream or with events.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "gemm.h"
#include "internal.h"

namespace gb300 {
namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr size_t kScratchFloats = GEMM_STATIC_SCRATCH_BYTES / sizeof(float);

// The scratch: fp32 partial sums [splits][M][roundup4(N)].
static __device__ __align__(256) float g_static_scratch[kScratchFloats];

struct ScratchSetup {
  bool ready = false;
  float* device_ptr = nullptr;
};

std::mutex g_setup_mu;
ScratchSetup g_setup[64];

// Device address of the scratch array on the current device (looked up once).
int scratch_on_current_device(float** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GEMM_ERR_CUDA;
  if (dev < 0 || dev >= 64) return GEMM_ERR_DEVICE;
  std::lock_guard<std::mutex> lk(g_setup_mu);
  ScratchSetup& s = g_setup[dev];
  if (!s.ready) {
    float* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(&ptr), g_static_scratch);
    if (e != cudaSuccess || ptr == nullptr) return GEMM_ERR_CUDA;
    s.device_ptr = ptr;
    s.ready = true;
  }
  *out = s.device_ptr;
  return GEMM_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace gb300

using namespace gb300;

extern "C" int gemm_f16_splitk_noalloc(const uint16_t* A, const uint16_t* B, uint16_t* C, int M,
                                       int N, int K, int lda, int ldb, int ldc, float alpha,
                                       float beta, int splits, cudaStream_t stream) {
  if (M < 0 || N < 0 || K < 0 || splits < 0) return M < 0 || N < 0 || K < 0 ? GEMM_ERR_DIM : GEMM_ERR_ARG;
  if (M == 0 || N == 0) {
    set_last_path("noop");
    return GEMM_OK;
  }
  if (ldc < N || (K > 0 && (lda < K || ldb < N))) return GEMM_ERR_LD;
  if (C == nullptr) return GEMM_ERR_NULL;
  if (K > 0 && alpha != 0.0f && (A == nullptr || B == nullptr)) return GEMM_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) |
       reinterpret_cast<uintptr_t>(C)) & 1u)
    return GEMM_ERR_ARG;   // half pointers must be 2-byte aligned

  int sm_count = 0;
  DeviceStatus* status = nullptr;
  unsigned long long wait_limit = 0;
  if (int rc = query_device(&sm_count, &status, &wait_limit)) return rc;
  float* scratch = nullptr;
  if (int rc = scratch_on_current_device(&scratch)) return rc;

  if (alpha == 0.0f || K == 0) {   // no products: C := beta*C, scratch unused
    set_last_path("f16.scale.noalloc");
    const long long blocks = (1ll * M * N + 255) / 256;
    const int grid = static_cast<int>(std::max(1ll, std::min<long long>(blocks, 8ll * sm_count)));
    return launch_scale_f16(C, ldc, M, N, beta, grid, stream) == cudaSuccess ? GEMM_OK
                                                                             : GEMM_ERR_CUDA;
  }

  const int bn = N <= 64 ? 64 : (N <= 128 ? 128 : 256);
  TcArgs a{};
  a.A = A;
  a.B = B;
  a.C = C;
  a.M = M;
  a.N = N;
  a.K = K;
  a.lda = lda;
  a.ldb = ldb;
  a.ldc = ldc;
  a.alpha = alpha;
  a.beta = beta;
  a.tiles_m = (M + kBM - 1) / kBM;
  a.tiles_n = (N + bn - 1) / bn;
  a.kb_total = (K + kBK - 1) / kBK;
  a.group_m = 8;
  a.wait_limit_ns = wait_limit;
  a.status = status;
  const long long tiles = 1ll * a.tiles_m * a.tiles_n;
  int s = splits;
  if (s == 0)
    s = static_cast<int>(std::min<long long>(
        {std::max(1ll, sm_count / tiles), static_cast<long long>(a.kb_total / 4), 16ll}));
  s = std::max(1, std::min(s, a.kb_total));
  a.kb_per_split = (a.kb_total + s - 1) / s;
  s = (a.kb_total + a.kb_per_split - 1) / a.kb_per_split;   // no empty slice
  a.splits = s;
  a.ws_ld = (N + 3) / 4 * 4;
  const double need = static_cast<double>(s) * M * static_cast<double>(a.ws_ld);
  if (need > static_cast<double>(kScratchFloats) || tiles * s > 0x7fffffffll) return GEMM_ERR_ARG;
  a.num_units = static_cast<int>(tiles * s);
  a.ws = scratch;
  a.dp_tiles = static_cast<int>(tiles);   // every tile split; no tail balancing
  a.tail_splits = 1;
  a.tail_kb_per_split = a.kb_total;

  const bool ab_tma = aligned16(A) && aligned16(B) && (1ll * lda * 2) % 16 == 0 &&
                      (1ll * ldb * 2) % 16 == 0;
  CUtensorMap tmA{}, tmB{}, tmC{};
  if (ab_tma) {
    if (int rc = encode_map_f16(&tmA, A, M, K, lda, 64, kBM)) return rc;
    if (int rc = encode_map_f16(&tmB, B, K, N, ldb, 64, 64)) return rc;
  }
  const int grid = static_cast<int>(std::min<long long>(a.num_units, sm_count));
  set_last_path(ab_tma ? "f16.splitk.noalloc.tma" : "f16.splitk.noalloc.manual");
  if (launch_gemm_f16_tc(bn, ab_tma ? kLoadTma : kLoadManual, kEpiPartial, tmA, tmB, tmC, a, grid,
                         stream) != cudaSuccess)
    return GEMM_ERR_CUDA;
  const long long groups = 1ll * M * ((N + 3) / 4);
  const int rgrid =
      static_cast<int>(std::max(1ll, std::min<long long>((groups + 255) / 256, 8ll * sm_count)));
  if (launch_splitk_reduce_f16(scratch, a.ws_ld, s, C, ldc, M, N, alpha, beta, rgrid, stream) !=
      cudaSuccess)
    return GEMM_ERR_CUDA;
  return GEMM_OK;
}
