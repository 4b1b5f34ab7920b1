// api.cu -- the C ABI of libgemm.so (declared in include/gemm.h): argument
// checks, path choice, tensor-map construction, workspace management and
// kernel launches on the caller's stream.
//
// Path choice for the half-precision GEMM (gemm_f16_ld, gemm_f16_f32out):
//   1. M == 0 or N == 0                 -> nothing to do
//   2. alpha == 0 or K == 0             -> scale-only kernel, C := beta*C
//   3. tile width BN from N (64 / 128 / 256; 128 when one row of 256-wide
//      tiles could not fill the SMs)
//   4. operand loads: TMA when A and B start on 16-byte boundaries and
//      lda*2, ldb*2 are multiples of 16 bytes (the run-time alignment check
//      of the "advanced SGEMM" page, kernel selection section, extended to
//      the 16-byte rule of TMA); an operand that breaks it is first copied to
//      16-byte rows (one launch for all), else predicated element loads
//   5. epilogue: TMA for a half C under the same rule when N is a multiple of
//      8; otherwise C is copied to 16-byte rows in the same launch (when
//      beta != 0), the TMA epilogue writes the copy and a last kernel copies
//      it back; predicated accesses when that is forced or too large; a float
//      C is written from registers
//   6. few tiles for many SMs with a long K: stream-K over all tiles when it
//      is expected to beat half-width units, or one wave of whole tiles for
//      64-wide tiles (few_tiles_prefer_stream_k)
//   7. CTA pairs (256 x 256 tiles) for 256-wide TMA shapes with at least two
//      tile rows; 32 or 64 rows of A staged per k-block when M <= 64
//   8. the tiles of the last, partial wave are shared out as stream-K pieces
//      (each worker runs the piece that starts a tile first and the piece that
//      ends a tile last, plan_tail_stream_k) when that is expected to beat two
//      half-width units per tile, which are used otherwise when the halves fit
//      in one wave
// The fp32 GEMM (sgemm_f32_ld) takes the tensor-core path for K >= 64: three
// products of operands split into two scaled half parts (3xFP16; 3xTF32 with
// tf32 parts when forced), with K slices when few tiles meet a long K
// (plan_tf32_slices); else the FFMA kernel.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <initializer_list>
#include <mutex>
#include <unordered_map>

#include "gemm.h"
#include "internal.h"
#include "ptx.cuh"

namespace gb300 {

__device__ DeviceStatus g_device_status;

namespace {

constexpr int kMaxDevices = 64;
constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kHostBlocks = 4;   // row blocks of the pipelined host-buffer forms

// Scratch of one stream: fp32 partial sums (split-K or tail tiles) and the
// tail-tile arrival counters.  Kernels on one stream run in order, so giving
// each stream its own scratch keeps concurrent streams apart.
struct StreamWs {
  void* ptr = nullptr;
  size_t bytes = 0;
  void* counters = nullptr;     // unsigned long long[]
  size_t counter_bytes = 0;
  unsigned int epoch = 0;       // launches that used the counters
  void* realigned = nullptr;    // aligned copies of unaligned operands
  size_t realigned_bytes = 0;
  void* split = nullptr;        // big/small tf32 parts of fp32 operands
  size_t split_bytes = 0;
};

struct DevState {
  bool init = false;
  int err = 0;
  int sm_count = 0;
  int l2_bytes = 0;
  DeviceStatus* status = nullptr;
  std::unordered_map<uintptr_t, StreamWs> ws;   // per stream
  void* flush = nullptr;        // L2 flush buffer
  size_t flush_bytes = 0;
  void* host_buf[3] = {nullptr, nullptr, nullptr};  // staging for the host-buffer forms
  size_t host_bytes[3] = {0, 0, 0};
  // host forms: copy-in and copy-back streams, and per row block an "in"
  // event (operands on the device) and a "done" event (block computed), plus
  // the call's entry and exit events
  cudaStream_t copy_in = nullptr, copy_back = nullptr;
  cudaEvent_t host_ev[2 * kHostBlocks + 2] = {};
};

std::mutex g_mu;
std::mutex g_host_mu;   // host-buffer forms share their staging buffers: one call at a time
DevState g_dev[kMaxDevices];
std::atomic<int> g_force_path{0};
std::atomic<int> g_stage_kblocks{0};   // 0 = automatic
std::atomic<int> g_force_splits{0};
std::atomic<long long> g_wait_limit_ns{2000000000ll};
std::atomic<long long> g_launches{0};
thread_local const char* t_last_path = "none";

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

int encode_fn(EncodeTiledFn* out) {
  if (g_encode) {
    *out = g_encode;
    return GEMM_OK;
  }
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q{};
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || fn == nullptr)
    return GEMM_ERR_CUDA;
  g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  *out = g_encode;
  return GEMM_OK;
}

// Per-device set-up: capability check, SM count, L2 size, status word.
int device_state(DevState** out, int* dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GEMM_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return GEMM_ERR_DEVICE;
  std::lock_guard<std::mutex> lk(g_mu);
  DevState& d = g_dev[dev];
  if (!d.init) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.l2_bytes, cudaDevAttrL2CacheSize, dev) != cudaSuccess)
      return GEMM_ERR_CUDA;
    if (major != 10 || minor != 3) {
      d.err = GEMM_ERR_DEVICE;
    } else {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return GEMM_ERR_CUDA;
      d.status = static_cast<DeviceStatus*>(p);
    }
    d.init = true;
  }
  if (d.err) return d.err;
  *out = &d;
  if (dev_out) *dev_out = dev;
  return GEMM_OK;
}

// Grows a library-owned device buffer (synchronising the device before a
// buffer that may be in use is replaced).
int ensure_buffer(void** buf, size_t* have, size_t need) {
  if (*have >= need && *buf) return GEMM_OK;
  if (*buf) {
    if (cudaDeviceSynchronize() != cudaSuccess) return GEMM_ERR_CUDA;
    cudaFree(*buf);
    *buf = nullptr;
    *have = 0;
  }
  size_t sz = std::max(need, static_cast<size_t>(1) << 20);
  if (cudaMalloc(buf, sz) != cudaSuccess) {
    *buf = nullptr;
    return GEMM_ERR_CUDA;
  }
  *have = sz;
  return GEMM_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Scratch of `stream` with at least `bytes` of partials and `counters`
// arrival counters (fresh counters start at zero).  Caller holds g_mu.
int stream_scratch(DevState* d, cudaStream_t stream, size_t bytes, size_t counters,
                   StreamWs** out) {
  StreamWs& w = d->ws[reinterpret_cast<uintptr_t>(stream)];
  if (bytes) {
    if (int rc = ensure_buffer(&w.ptr, &w.bytes, bytes)) return rc;
  }
  if (counters) {
    const size_t cb = counters * sizeof(unsigned long long);
    if (w.counter_bytes < cb || !w.counters) {
      if (int rc = ensure_buffer(&w.counters, &w.counter_bytes, cb)) return rc;
      if (cudaMemsetAsync(w.counters, 0, w.counter_bytes, stream) != cudaSuccess)
        return GEMM_ERR_CUDA;
      w.epoch = 0;
    }
  }
  *out = &w;
  return GEMM_OK;
}

// K slices for the fp32 tensor-core kernel when few pair tiles leave most
// pairs idle: the slice count in [2, cap] (slices of whole 4-k-block chunks)
// with the least estimated time, or 1 when whole-K half-width units are
// expected to be faster.  Estimates measured on GB300: a whole-K half-width
// unit runs ~0.6 us per k-block, a full-width slice ~0.75 us, and publishing
// plus adding up S slices' partial sums costs ~8 + 1.5 S us; slices must be
// estimated at least 10% faster.  `forced` takes the largest count up to
// `cap` whatever the estimate.
struct TailSplit {
  int splits = 1;
  int kb_per_split = 0;
};
TailSplit plan_tf32_slices(int kb_total, int cap, bool forced) {
  TailSplit best;
  double best_us = 0.9 * 0.6 * kb_total;
  for (int want = 2; want <= cap; ++want) {
    const int per = ((kb_total + want - 1) / want + 3) / 4 * 4;
    const int s = (kb_total + per - 1) / per;   // no empty slice
    if (s < 2) continue;
    const double us = 0.75 * per + 8.0 + 1.5 * s;
    if (forced || us < best_us) {
      best_us = us;
      best.splits = s;
      best.kb_per_split = per;
    }
  }
  return best;
}

// The K-slice plan of the fp32 tensor-core path: slices only when the tiles
// fill at most half the pairs and K has at least two chunks; `fs` > 1 forces
// that many slices (fs == 1: none).
TailSplit tf32_slice_plan(long long tiles, long long pairs, int kb_total, int fs) {
  if (fs == 1 || tiles <= 0 || 2 * tiles > pairs || kb_total < 8) return TailSplit{};
  const long long fit = pairs / tiles;
  const int cap = static_cast<int>(std::min<long long>({fs > 1 ? fs : fit, kb_total / 4, 16}));
  return plan_tf32_slices(kb_total, cap, fs > 1);
}

// Tail plan for `tiles` whole tiles on `ctas` persistent CTAs: the number of K
// slices (1 = none) that minimises the number of tile-times, counting a tile
// cut into s slices as 1/s of a tile-time per slice plus a small fix-up cost.
int plan_tail_splits(long long tiles, long long ctas, int kb_total) {
  if (tiles <= ctas || ctas <= 0) return 1;
  const long long full = tiles / ctas, rem = tiles % ctas;
  if (rem == 0) return 1;
  int best = 1;
  double best_t = static_cast<double>(full + 1);
  // A sliced tile is finished by one extra pass over its partial sums (about
  // as long as a 32-k-block main loop): only long slices, at most two, pay.
  for (int s = 2; s <= 2; ++s) {
    if (kb_total / s < 32) break;
    // each extra slice costs a little: its partial sums go through L2 once
    const double t = static_cast<double>(full) +
                     static_cast<double>((rem * s + ctas - 1) / ctas) / static_cast<double>(s) +
                     0.03 * (s - 1);
    if (t < best_t - 1e-9) {
      best_t = t;
      best = s;
    }
  }
  return best;
}

// Stream-K plan for `tiles` tiles of kb k-blocks on at most `slots`
// concurrent workers (CTAs or CTA pairs).
//  * all_tiles (few tiles, many SMs): every tile's k-blocks are shared out,
//    at least kSkMinKb per worker;
//  * otherwise, when the tiles do not fill a whole number of waves, the
//    last partial wave and the full wave before it are shared out, so every
//    worker ends at the same k-block count; the earlier waves stay whole
//    tiles.  Taken only when it beats whole tiles by more than the cost of
//    finishing a shared tile (about kSkFixKb k-blocks of main loop).
// A worker's range then spans at most ceil(kb / range) + 1 tiles' pieces.
struct SkPlan {
  long long dp_tiles = 0, sk_tiles = 0, workers = 0, max_pieces = 0;
};
constexpr long long kSkMinKb = 4;
constexpr long long kSkFixKb = 8;

SkPlan plan_stream_k(long long tiles, long long slots, int kb, bool all_tiles) {
  SkPlan p;
  if (tiles <= 0 || slots <= 0 || kb <= 0) return p;
  long long dp = 0;
  if (!all_tiles) {
    if (tiles <= slots || tiles % slots == 0) return p;
    const long long full = tiles / slots;
    dp = (full - 1) * slots;
    const long long whole = (full + 1) * kb;
    const long long shared = (full - 1) * kb + ((tiles - dp) * kb + slots - 1) / slots + kSkFixKb;
    if (shared >= whole) return p;
  }
  const long long iters = (tiles - dp) * kb;
  if (iters >= (1ll << 31)) return p;   // the kernel counts k-blocks in 32 bits
  const long long workers = std::min(slots, iters / kSkMinKb);
  if (workers < 2) return p;
  const long long range = iters / workers;   // shortest range
  p.dp_tiles = dp;
  p.sk_tiles = tiles - dp;
  p.workers = workers;
  p.max_pieces = (kb + range - 1) / range + 1;
  return p;
}

// Stream-K over the last, partial wave only, in the order of sk_order 1:
// the `tiles` % `slots` tiles after the whole waves are shared out as k-block
// ranges over up to kTailPieces workers per tile (no range longer than a
// tile, none shorter than kSkMinKb k-blocks).  Each worker runs the part of its range
// that starts a tile before its whole tiles and the part that ends a tile
// after them, so the piece that finishes a tile finds the others published.
constexpr long long kTailPieces = 4;

SkPlan plan_tail_stream_k(long long tiles, long long slots, int kb) {
  SkPlan p;
  if (tiles <= slots || slots <= 0 || kb < 2 * kSkMinKb) return p;
  const long long rem = tiles % slots;
  if (rem == 0) return p;
  const long long iters = rem * kb;
  if (iters >= (1ll << 31)) return p;
  const long long workers = std::min({slots, rem * kTailPieces, iters / kSkMinKb});
  if (workers <= rem) return p;   // no range may be longer than a tile
  const long long range = iters / workers;   // shortest range
  p.dp_tiles = tiles - rem;
  p.sk_tiles = rem;
  p.workers = workers;
  p.max_pieces = (kb + range - 1) / range + 1;
  return p;
}

// The last, partial wave as two K slices per tile, publisher first: the
// first slice of each of its tiles is the first unit of one worker (it
// publishes fp32 partial sums), the second is the last unit of another worker
// (it finishes the tile, reading the first slice's partial sums back, which
// are long published by then and prefetched into L2 while its main loop
// runs).  Returns the k-blocks of the first slice, or 0 when the shape does
// not suit: at least one whole wave before the tail, the two slices of every
// tail tile on different workers (2 x tail tiles <= slots), and at least 48
// k-blocks (measured: with 32 or 16, half-width units are faster -- 4096^2 x
// 2048 55.6 against 57.3 us, 2560^2 x 1024 24.6 against 27.1 us).  The finishing slice is kTailReadKb k-blocks shorter, for the
// read-back of the other slice (measured on GB300: ~2.5 us against 0.32 us
// per k-block of a pair tile).
constexpr int kTailReadKb = 8;

int tail_first_slice(long long tiles, long long slots, int kb) {
  if (tiles <= slots || slots <= 0 || kb < 48) return 0;
  const long long rem = tiles % slots;
  if (rem == 0 || 2 * rem > slots) return 0;
  return std::min(kb - 4, (kb + kTailReadKb + 1) / 2);
}

// Whether stream-K over all of a few tiles (plan_stream_k's all_tiles form)
// is expected to beat half-width whole-K units, in k-block times of one
// tile: stream-K takes the longest range plus a fix-up for every extra piece
// of a tile, in proportion to the partial sums each publishes and the
// finisher re-reads (about 8 k-blocks for 128 full rows of a 128-wide tile);
// a wave of half-width units takes about 3/4 of a tile's k-blocks (measured:
// they stage 3/4 of the operand bytes for half the FLOPs).  Measured: 1024^3
// (32 tiles of 16 k-blocks) half-width units 16 us, stream-K 24 us;
// 1000x1001x4096 (32 tiles of 64) 38 us and 61 us; 16x8192x8192 (64 tiles of
// 128, 16 rows) stream-K 42 us, equal K slices 51 us.
// 64-wide TMA tiles have no half-width units; there stream-K is weighed
// against one wave of whole-K tiles.  A whole-K CTA takes ~0.25 us per
// k-block whatever the tile's height or the number of CTAs (its TMA ring
// completes about one stage per DRAM round trip, whatever the stage's size),
// and ~4% less with two k-blocks per stage, which such tiles take from
// kWholeTwoKb k-blocks on (whole_stage_kblocks).  Stream-K's ranges can go no
// faster than HBM streams A: per k-block of a range, the time HBM takes for
// the k-blocks of about 96 128-row tiles.  Measured over M = 512..9728, N = 32
// and 64, K = 512..16384 (second-half mean of 24 replays after the page's
// flush): whole tiles win for K <= 2048 (8192x64x1024 14.1 against 18.5 us)
// and at K = 4096 for most M (8192x64x4096 24.4 against 26.1 us), stream-K
// for K >= 8192 (4096x64x8192 26.9 against 43.1 us); the estimate is within
// 1 us of the faster one at 81 of 84 shapes.
constexpr int kWholeTwoKb = 16;

int whole_stage_kblocks(int kb) { return kb >= kWholeTwoKb ? 2 : 1; }

bool few_tiles_prefer_stream_k(long long tiles, long long slots, int kb, bool halves_ok,
                               bool whole_ok, int rows, int bn) {
  const SkPlan sk = plan_stream_k(tiles, slots, kb, true);
  if (sk.sk_tiles == 0) return false;
  const long long range = (sk.sk_tiles * kb + sk.workers - 1) / sk.workers;
  const long long per_piece = std::max(1ll, 8ll * std::min(rows, kBM) * bn / (kBM * 128));
  if (!halves_ok) {
    if (!whole_ok) return true;
    const long long floor_kb = (sk.sk_tiles * kb * std::min(rows, kBM) + 96 * kBM - 1) / (96 * kBM);
    const long long whole_cost = whole_stage_kblocks(kb) == 2 ? kb * 24 / 25 : kb;
    return std::max(range, floor_kb) + kSkFixKb + per_piece * (sk.max_pieces - 1) < whole_cost;
  }
  const long long sk_cost = range + kSkFixKb + per_piece * (sk.max_pieces - 1);
  const long long waves = (2 * tiles + slots - 1) / slots;
  const long long halves_cost = (3 * kb * waves + 3) / 4;
  return sk_cost < halves_cost;
}

// Tensor maps encode only host-side facts (address, shape, stride, box,
// swizzle), so a map built once for a key stays valid for every later call
// with the same key, whatever happened to the memory in between.  Each host
// thread keeps the last kMapCache maps it encoded and reuses them: repeated
// calls on the same operands skip cuTensorMapEncodeTiled (the run-time
// dispatch stays cheap, as the kernel-selection section of the "advanced
// SGEMM" page asks of it).
struct MapKey {
  const void* ptr;
  long long ld;
  int rows, cols, box_cols, box_rows;
  int dtype, swizzle;
  bool operator==(const MapKey& o) const {
    return ptr == o.ptr && ld == o.ld && rows == o.rows && cols == o.cols &&
           box_cols == o.box_cols && box_rows == o.box_rows && dtype == o.dtype &&
           swizzle == o.swizzle;
  }
};
constexpr int kMapCache = 16;
struct MapCache {
  MapKey key[kMapCache];
  CUtensorMap map[kMapCache];
  int used = 0, next = 0;
};
thread_local MapCache t_maps;

// Width of the CTA-pair tiles: 256 unless forced (paths 12 / 13: 224 / 192).
// Measured on GB300 (same-box A/B, alpha 1.5 beta 0.5): a k-block of a
// 256 x 224 or 256 x 192 pair tile takes as long as one of a 256 x 256 tile,
// and so does a half-width unit (N = 128; 4096^3 as 512 half-width units in
// 7 rounds: 139 us, against 20.5 us per full round), so narrower tiles only
// move the partial last wave: 4096^3 (304 tiles of 224 = 4 waves) 91.7 us
// against 92.2 us for 256-wide tiles with a half-width tail; 8192x8192x4096
// 351 against 315 us, 6144^2 x 4096 197 against 184 us, 192-wide slower
// still.  A narrower tile never wins once its per-tile time equals the
// 256-wide one, so the automatic choice keeps 256 and balances the last wave
// along K instead (plan_tail_stream_k).
int pair_width(int force) { return force == 12 ? 224 : (force == 13 ? 192 : 256); }

int make_map(CUtensorMap* map, CUtensorMapDataType dtype, size_t elem, const void* ptr, int rows,
             int cols, long long ld, int box_cols, int box_rows, CUtensorMapSwizzle swizzle) {
  const MapKey k{ptr, ld, rows, cols, box_cols, box_rows, static_cast<int>(dtype),
                 static_cast<int>(swizzle)};
  MapCache& c = t_maps;
  for (int i = 0; i < c.used; ++i)
    if (c.key[i] == k) {
      *map = c.map[i];
      return GEMM_OK;
    }
  EncodeTiledFn enc = nullptr;
  if (int rc = encode_fn(&enc)) return rc;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * elem};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1u, 1u};
  const CUresult r = enc(map, dtype, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return GEMM_ERR_CUDA;
  const int slot = c.used < kMapCache ? c.used++ : c.next;
  c.next = (slot + 1) % kMapCache;
  c.key[slot] = k;
  c.map[slot] = *map;
  return GEMM_OK;
}

int make_map_f16(CUtensorMap* map, const void* ptr, int rows, int cols, long long ld,
                 int box_cols, int box_rows, CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  return make_map(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, ptr, rows, cols, ld, box_cols, box_rows,
                  swizzle);
}

int make_map_f32(CUtensorMap* map, const void* ptr, int rows, int cols, long long ld,
                 int box_cols, int box_rows, CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  return make_map(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, ptr, rows, cols, ld, box_cols, box_rows,
                  swizzle);
}

// Blocks of 256 threads for `elems` work items, at most `per_sm` blocks per SM
// (grid-stride kernels loop over the rest).
int scale_grid(const DevState& d, long long elems, int per_sm = 8) {
  const long long blocks = (elems + 255) / 256;
  return static_cast<int>(
      std::max(1ll, std::min<long long>(blocks, static_cast<long long>(per_sm) * d.sm_count)));
}

// [bn index][load][epilogue: TMA, predicated, fp32 partial sums (split-K)]
const char* kPathNames[3][2][3] = {
    // [bn index][load][epi]
    {{"f16.tc.bn64.tma.epi_tma", "f16.tc.bn64.tma.epi_manual", "f16.tc.bn64.tma.splitk"},
     {"f16.tc.bn64.manual.epi_tma", "f16.tc.bn64.manual.epi_manual", "f16.tc.bn64.manual.splitk"}},
    {{"f16.tc.bn128.tma.epi_tma", "f16.tc.bn128.tma.epi_manual", "f16.tc.bn128.tma.splitk"},
     {"f16.tc.bn128.manual.epi_tma", "f16.tc.bn128.manual.epi_manual",
      "f16.tc.bn128.manual.splitk"}},
    {{"f16.tc.bn256.tma.epi_tma", "f16.tc.bn256.tma.epi_manual", "f16.tc.bn256.tma.splitk"},
     {"f16.tc.bn256.manual.epi_tma", "f16.tc.bn256.manual.epi_manual",
      "f16.tc.bn256.manual.splitk"}},
};

int check_common(const void* A, const void* B, const void* C, int M, int N, int K, long long lda,
                 long long ldb, long long ldc, float alpha, size_t elem = 1) {
  if (M < 0 || N < 0 || K < 0) return GEMM_ERR_DIM;
  if (M == 0 || N == 0) return GEMM_OK;
  if (ldc < N || (K > 0 && (lda < K || ldb < N))) return GEMM_ERR_LD;
  if (C == nullptr) return GEMM_ERR_NULL;
  if (K > 0 && alpha != 0.0f && (A == nullptr || B == nullptr)) return GEMM_ERR_NULL;
  // element pointers must at least be aligned to their element size
  const uintptr_t mis = (reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) |
                         reinterpret_cast<uintptr_t>(C)) & (elem - 1);
  if (mis) return GEMM_ERR_ARG;
  return GEMM_OK;
}

thread_local char t_path_buf[96];

// Half-precision operands, fp32 accumulation; C is half (c_f32 false) or
// float (c_f32 true).
int gemm_f16_impl(const uint16_t* A, const uint16_t* B, void* C, bool c_f32, int M, int N, int K,
                  long long lda, long long ldb, long long ldc, float alpha, float beta,
                  cudaStream_t stream) {
  if (int rc = check_common(A, B, C, M, N, K, lda, ldb, ldc, alpha, 2)) return rc;
  if (c_f32 && (reinterpret_cast<uintptr_t>(C) & 3u)) return GEMM_ERR_ARG;
  if (M == 0 || N == 0) {
    t_last_path = "noop";
    return GEMM_OK;
  }
  DevState* d = nullptr;
  if (int rc = device_state(&d, nullptr)) return rc;

  if (alpha == 0.0f || K == 0) {
    t_last_path = c_f32 ? "f16f32.scale" : "f16.scale";
    const int g = scale_grid(*d, 1ll * M * N);
    const cudaError_t e =
        c_f32 ? launch_scale_f32(static_cast<float*>(C), ldc, M, N, beta, g, stream)
              : launch_scale_f16(static_cast<uint16_t*>(C), ldc, M, N, beta, g, stream);
    return e == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
  }

  const int force = g_force_path.load();
  int bn = N <= 64 ? 64 : (N <= 128 ? 128 : 256);
  // A single row of 256-wide tiles that cannot fill the SMs: narrower tiles
  // give more of them, so fewer K slices are needed.
  if (bn == 256 && M <= kBM && 1ll * ((N + 255) / 256) * 2 <= d->sm_count) bn = 128;
  const bool a_tma = aligned16(A) && (lda * 2) % 16 == 0;
  const bool b_tma = aligned16(B) && (ldb * 2) % 16 == 0;
  // A TMA store writes whole 16-byte pieces of a row: when N is not a multiple
  // of 8 halves it would also write the elements just past column N (measured
  // on GB300), which may belong to the caller.
  bool c_tma = !c_f32 && aligned16(C) && (ldc * 2) % 16 == 0 && N % 8 == 0;
  // An operand whose rows break the 16-byte rule is first copied into an
  // aligned layout (one bandwidth-bound launch for all of them) unless the
  // predicated path is forced or the copies would be very large.  Such a half
  // C is copied in (when beta != 0), written by the TMA epilogue into its
  // aligned copy (rows padded to a multiple of 8, so the pieces past N land
  // in the padding) and copied back by a last kernel.
  const char* how = "";
  bool prepass = false;         // a realignment kernel was launched just before the GEMM
  uint16_t* c_user = nullptr;   // the caller's C when the GEMM writes an aligned copy
  long long ldc_user = 0;
  if ((!a_tma || !b_tma || (!c_f32 && !c_tma)) && force != 2) {
    const long long lda2 = (K + 7) / 8 * 8, ldb2 = (N + 7) / 8 * 8, ldc2 = (N + 7) / 8 * 8;
    auto round256 = [](size_t x) { return (x + 255) / 256 * 256; };
    const size_t a_bytes = a_tma ? 0 : round256(static_cast<size_t>(M) * lda2 * 2);
    const size_t b_bytes = b_tma ? 0 : round256(static_cast<size_t>(K) * ldb2 * 2);
    const size_t c_bytes = (c_f32 || c_tma) ? 0 : round256(static_cast<size_t>(M) * ldc2 * 2);
    if (a_bytes + b_bytes + c_bytes <= (static_cast<size_t>(1) << 31)) {
      std::lock_guard<std::mutex> lk(g_mu);
      StreamWs& w = d->ws[reinterpret_cast<uintptr_t>(stream)];
      if (int rc = ensure_buffer(&w.realigned, &w.realigned_bytes, a_bytes + b_bytes + c_bytes))
        return rc;
      uint8_t* buf = static_cast<uint8_t*>(w.realigned);
      RealignBatch batch{};
      auto add = [&](const RealignJob& j, long long groups) {
        batch.job[batch.n] = j;
        batch.end[batch.n] = (batch.n ? batch.end[batch.n - 1] : 0) + scale_grid(*d, groups);
        ++batch.n;
      };
      if (!a_tma) {
        uint16_t* dst = reinterpret_cast<uint16_t*>(buf);
        add(RealignJob{A, lda, dst, lda2, M, K}, 1ll * M * lda2 / 8);
        A = dst;
        lda = lda2;
        buf += a_bytes;
      }
      if (!b_tma) {
        uint16_t* dst = reinterpret_cast<uint16_t*>(buf);
        add(RealignJob{B, ldb, dst, ldb2, K, N}, 1ll * K * ldb2 / 8);
        B = dst;
        ldb = ldb2;
        buf += b_bytes;
      }
      if (c_bytes) {
        uint16_t* dst = reinterpret_cast<uint16_t*>(buf);
        if (beta != 0.0f)
          add(RealignJob{static_cast<uint16_t*>(C), ldc, dst, ldc2, M, N}, 1ll * M * ldc2 / 8);
        c_user = static_cast<uint16_t*>(C);
        ldc_user = ldc;
        C = dst;
        ldc = ldc2;
        c_tma = true;
      }
      if (batch.n > 0) {
        if (launch_realign_f16(batch, stream) != cudaSuccess) return GEMM_ERR_CUDA;
        prepass = true;
      }
      how = c_user ? (batch.n > 0 ? ".realigned.c" : ".c") : ".realigned";
    }
  }
  const bool ab_tma = aligned16(A) && aligned16(B) && (lda * 2) % 16 == 0 && (ldb * 2) % 16 == 0;
  int load = (ab_tma && force != 2) ? kLoadTma : kLoadManual;
  int epi = c_f32 ? kEpiF32 : ((c_tma && force != 2) ? kEpiTma : kEpiManual);

  TcArgs a{};
  a.pdl = prepass;   // the realignment copy was launched just before
  a.A = A;
  a.B = B;
  a.C = c_f32 ? nullptr : static_cast<uint16_t*>(C);
  a.Cf = c_f32 ? static_cast<float*>(C) : nullptr;
  a.vec_c = c_f32 && aligned16(C) && ldc % 4 == 0;
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
  a.wait_limit_ns = static_cast<unsigned long long>(g_wait_limit_ns.load());
  a.status = d->status;

  const long long tiles = 1ll * a.tiles_m * a.tiles_n;
  int splits = 1;
  const int fs = g_force_splits.load();
  // Few tiles for many SMs: the k-blocks of all tiles are shared out evenly
  // over the SMs (stream-K); the forced split-K path cuts every tile into
  // equal K slices instead.
  // Few tiles for many SMs: stream-K over all tiles when it beats half-width
  // whole-K units (few_sk; then one CTA per worker, no pairs).
  const bool few = tiles * 2 <= d->sm_count && a.kb_total >= 8;
  // Tall shapes (one column of 64-wide tiles): 64-row tiles (M = 64 MMAs)
  // double the tiles, so that whole-K units fill one wave without stream-K
  // partial sums.
  const long long tiles64 = 1ll * ((M + 63) / 64) * a.tiles_n;
  const bool m64 = force == 17 && load == kLoadTma && epi == kEpiTma && bn == 64 &&
                   tiles64 <= d->sm_count;
  if (m64) a.tiles_m = (M + 63) / 64;
  const bool few_sk = !m64 &&
      (few && force == 0 &&
       few_tiles_prefer_stream_k(tiles, d->sm_count, a.kb_total, load == kLoadTma && bn >= 128,
                                 load == kLoadTma && bn == 64, M, bn)) ||
      force == 11;
  if (force == 3) {
    // as many K slices as fit in ONE wave of CTAs (a second, partial wave would
    // double the time of these bandwidth-bound shapes)
    splits = fs > 0 ? fs
                    : static_cast<int>(std::min<long long>(
                          {std::max(1ll, d->sm_count / tiles), static_cast<long long>(a.kb_total / 4),
                           16ll}));
    splits = std::max(1, std::min(splits, a.kb_total));
  }
  if (splits > 1) {
    a.kb_per_split = (a.kb_total + splits - 1) / splits;
    splits = (a.kb_total + a.kb_per_split - 1) / a.kb_per_split;  // no empty slice
  } else {
    a.kb_per_split = a.kb_total;
  }
  a.splits = splits;
  if (tiles * splits * 4 > 0x7fffffffll) return GEMM_ERR_ARG;

  // CTA pairs (256 x 256 tiles on clusters of 2 sharing each MMA) for the
  // large aligned shapes: each SM then stages half as much of B per MMA.
  int pair_slots = 0;
  const bool pair = splits == 1 && !few_sk && force != 6 && bn == 256 &&
                    load == kLoadTma && a.tiles_m >= 2 &&
                    (pair_slots = tc_pair_max_clusters(epi)) > 0;
  // forced narrower pair tiles (the tile-family comparison)
  if (pair && !c_f32 && (force == 12 || force == 13)) {
    bn = pair_width(force);
    a.tiles_n = (N + bn - 1) / bn;
  }
  // fp32 C on CTA pairs goes through shared memory and TMA when its rows are
  // 16-byte aligned and N is a multiple of 4 (a TMA store writes whole 16-byte
  // pieces of a row)
  if (epi == kEpiF32 && pair && a.vec_c && N % 4 == 0) epi = kEpiF32Tma;
  long long units_tiles = m64 ? tiles64 : tiles;   // tiles in units of the worker (CTA or pair)
  long long slots = d->sm_count;   // workers that can run at once
  if (pair) {
    a.tiles_m = (M + 2 * kBM - 1) / (2 * kBM);
    units_tiles = 1ll * a.tiles_m * a.tiles_n;
    slots = pair_slots;
  }
  long long workers = std::min<long long>(units_tiles, slots);
  // an operand that only one row (column) of single-CTA tiles reads -- B of a
  // skinny shape, A of a tall one -- is streamed once: loaded evict-first
  a.stream_a = !pair && a.tiles_n == 1;
  a.stream_b = !pair && a.tiles_m == 1;

  a.dp_tiles = static_cast<int>(units_tiles);
  a.tail_splits = 1;
  a.tail_kb_per_split = a.kb_total;
  const char* cut = "";
  // scratch for partial sums: `parts` 128-row tile parts x `pieces` each
  auto take_scratch = [&](long long parts, long long pieces) -> int {
    const size_t need = sizeof(float) * static_cast<size_t>(parts) * pieces * kBM * bn;
    std::lock_guard<std::mutex> lk(g_mu);
    StreamWs* w = nullptr;
    if (int rc = stream_scratch(d, stream, need, static_cast<size_t>(parts) * 8, &w)) return rc;
    a.tail_ws = static_cast<float*>(w->ptr);
    a.tail_counters = static_cast<unsigned long long*>(w->counters);
    a.epoch = ++w->epoch;
    if (a.epoch == 0) a.epoch = ++w->epoch;   // 0 marks never-used counters
    return GEMM_OK;
  };
  if (splits > 1) {
    // Every tile is cut into `splits` K slices: each slice publishes fp32
    // partial sums and the last one of a tile to finish adds them up (in slice
    // order) and runs the epilogue -- no second kernel.
    a.dp_tiles = 0;
    a.tail_splits = splits;
    a.tail_kb_per_split = a.kb_per_split;
    a.kb_per_split = a.kb_total;
    splits = 1;
    a.splits = 1;
    if (int rc = take_scratch(tiles, a.tail_splits)) return rc;
    cut = ".splitk";
  } else if (force == 9) {
    // Two equal K slices for each tile of the last, partial wave.
    int ts = plan_tail_splits(units_tiles, workers, a.kb_total);
    if (ts > 1) {
      const long long tail_tiles = units_tiles % workers;
      a.tail_kb_per_split = (a.kb_total + ts - 1) / ts;
      ts = (a.kb_total + a.tail_kb_per_split - 1) / a.tail_kb_per_split;   // no empty slice
      a.dp_tiles = static_cast<int>(units_tiles - tail_tiles);
      a.tail_splits = ts;
      if (int rc = take_scratch(tail_tiles * (pair ? 2 : 1), ts)) return rc;
      cut = ".tail";
    }
  } else if (force == 10) {
    // stream-K over the last waves (k-block ranges shared out evenly)
    const SkPlan sk = plan_stream_k(units_tiles, slots, a.kb_total, false);
    if (sk.sk_tiles > 0) {
      a.dp_tiles = static_cast<int>(sk.dp_tiles);
      a.sk_tile0 = static_cast<int>(sk.dp_tiles);
      a.sk_tiles = static_cast<int>(sk.sk_tiles);
      a.sk_workers = static_cast<int>(sk.workers);
      a.sk_iters = sk.sk_tiles * a.kb_total;
      a.tail_splits = static_cast<int>(sk.max_pieces);
      workers = sk.workers;
      if (int rc = take_scratch(sk.sk_tiles * (pair ? 2 : 1), sk.max_pieces)) return rc;
      cut = ".sk";
    }
  } else if (!m64 && force != 5 && force != 12 && force != 13 && !few_sk) {
    // The tiles of the last, partial wave: two K slices each, the first slice
    // a worker's first unit and the second another worker's last
    // (tail_first_slice); else two half-width units each (whole K, no partial
    // sums) when the halves fit in one wave.  Forced path 14 shares them out
    // as stream-K pieces instead (plan_tail_stream_k), 15 takes half-width
    // units.
    const long long rem = units_tiles % slots;
    const SkPlan sk = force == 14 ? plan_tail_stream_k(units_tiles, slots, a.kb_total) : SkPlan{};
    const int first_kb =
        (force == 14 || force == 15) ? 0 : tail_first_slice(units_tiles, slots, a.kb_total);
    if (first_kb > 0) {
      a.dp_tiles = static_cast<int>(units_tiles - rem);
      a.tail_splits = 2;
      a.tail_kb_per_split = first_kb;
      a.tail_first = 1;
      workers = slots;
      if (int rc = take_scratch(rem * (pair ? 2 : 1), 2)) return rc;
      cut = ".ktail";
    } else if (sk.sk_tiles > 0) {
      a.dp_tiles = static_cast<int>(sk.dp_tiles);
      a.sk_tile0 = static_cast<int>(sk.dp_tiles);
      a.sk_tiles = static_cast<int>(sk.sk_tiles);
      a.sk_workers = static_cast<int>(sk.workers);
      a.sk_iters = sk.sk_tiles * a.kb_total;
      a.sk_order = 1;
      a.tail_splits = static_cast<int>(sk.max_pieces);
      workers = slots;
      if (int rc = take_scratch(sk.sk_tiles * (pair ? 2 : 1), sk.max_pieces)) return rc;
      cut = ".sktail";
    } else if (load == kLoadTma && (bn == 128 || bn == 256) && rem > 0 && 2 * rem <= slots) {
      a.dp_tiles = static_cast<int>(units_tiles - rem);
      a.tail_splits = 2;
      a.tail_halves = 1;
      workers = std::min<long long>(slots, a.dp_tiles > 0 ? slots : 2 * rem);
      cut = ".halves";
    }
  } else if (force != 5 && few_sk) {
    const SkPlan sk = plan_stream_k(units_tiles, slots, a.kb_total, true);
    if (sk.sk_tiles > 0) {
      a.dp_tiles = static_cast<int>(sk.dp_tiles);
      a.sk_tile0 = static_cast<int>(sk.dp_tiles);
      a.sk_tiles = static_cast<int>(sk.sk_tiles);
      a.sk_workers = static_cast<int>(sk.workers);
      a.sk_iters = sk.sk_tiles * a.kb_total;
      // no range longer than a tile (fewer tiles than workers): each worker
      // runs the piece that starts a tile first and the piece that ends one
      // last, so a tile's finishing piece finds the others published (and
      // brings their partial sums into L2 while its own main loop runs)
      a.sk_order = sk.sk_tiles <= sk.workers ? 1 : 0;
      a.tail_splits = static_cast<int>(sk.max_pieces);
      workers = sk.workers;
      if (int rc = take_scratch(sk.sk_tiles * (pair ? 2 : 1), sk.max_pieces)) return rc;
      cut = ".sk";
    }
  }

  a.num_units = a.sk_tiles > 0
                    ? a.dp_tiles
                    : static_cast<int>(a.dp_tiles * static_cast<long long>(splits) +
                                       (units_tiles - a.dp_tiles) * a.tail_splits);

  // k-blocks per ring stage: two for one wave of whole 64-wide tiles with a
  // long enough K (whole_stage_kblocks), or where forced and the kernel has
  // that form (64-wide single-CTA tiles, 256-wide pairs, TMA epilogue)
  int kpb = 1;
  const int fk = g_stage_kblocks.load();
  const bool two_ok = load == kLoadTma && epi == kEpiTma && !m64 &&
                      ((pair && bn == 256) || (!pair && bn == 64));
  if (fk == 2 && two_ok) {
    kpb = 2;
  } else if (fk == 0 && two_ok && !pair && few && a.sk_tiles == 0 && a.tail_splits == 1 &&
             a.splits == 1 && a.num_units == tiles) {
    kpb = whole_stage_kblocks(a.kb_total);
  }

  // At most 64 rows on 128-wide single-CTA tiles: stage only the A rows that
  // exist (32 or 64), which leaves room for more stages of B.
  const int am = m64 ? 64
                     : ((load == kLoadTma && !pair && bn == 128 && M <= 64) ? (M <= 32 ? 32 : 64)
                                                                           : kBM);
  CUtensorMap tmA{}, tmB{}, tmC{};
  if (load == kLoadTma) {
    if (int rc = make_map_f16(&tmA, A, M, K, lda, 64, am)) return rc;
    if (int rc = make_map_f16(&tmB, B, K, N, ldb, 64, 64)) return rc;
  }
  if (epi == kEpiTma) {
    // epilogue staging tile: 32 rows (16 on 64-row tiles) x 32 halves, 64-byte swizzle
    if (int rc = make_map_f16(&tmC, a.C, M, N, ldc, 32, m64 ? 16 : 32, CU_TENSOR_MAP_SWIZZLE_64B))
      return rc;
  } else if (epi == kEpiF32Tma) {
    // the same 64-byte rows: 32 rows x 16 floats
    if (int rc = make_map_f32(&tmC, a.Cf, M, N, ldc, 16, 32, CU_TENSOR_MAP_SWIZZLE_64B)) return rc;
  }
  // a C with rows off the 16-byte grid: the kernel wrote its aligned copy,
  // which goes back to the caller's C last
  auto copy_back = [&]() -> int {
    if (!c_user) return GEMM_OK;
    const RealignJob j{a.C, ldc, c_user, ldc_user, M, N};
    return launch_unalign_f16(j, scale_grid(*d, 1ll * M * (N / 8 + 2)), stream) == cudaSuccess
               ? GEMM_OK
               : GEMM_ERR_CUDA;
  };
  // one CTA (pair) per worker; with stream-K over all tiles or the last waves
  // exactly sk_workers of them, with the stream-K tail every worker
  const long long nw = a.sk_tiles > 0 ? (a.sk_order ? workers : a.sk_workers)
                                      : std::min<long long>(a.num_units, workers);
  if (pair) {
    const int grid = 2 * static_cast<int>(nw);
    snprintf(t_path_buf, sizeof(t_path_buf), "f16.tc.pair.bn%d.tma.%s%s%s%s", bn,
             epi == kEpiF32Tma ? "epi_f32_tma"
                               : (epi == kEpiF32 ? "epi_f32" : (epi == kEpiTma ? "epi_tma" : "epi_manual")),
             kpb == 2 ? ".kb2" : "", cut, how);
    t_last_path = t_path_buf;
    if (launch_gemm_f16_tc_pair(bn, epi, tmA, tmB, tmC, a, grid, stream, kpb) != cudaSuccess)
      return GEMM_ERR_CUDA;
    return copy_back();
  }
  const int grid = static_cast<int>(nw);
  const int bi = bn == 64 ? 0 : (bn == 128 ? 1 : 2);
  const char* rows = m64 ? ".m64" : (am == 32 ? ".a32" : (am == 64 ? ".a64" : (kpb == 2 ? ".kb2" : "")));
  if (c_f32)
    snprintf(t_path_buf, sizeof(t_path_buf), "f16.tc.bn%d.%s.epi_f32%s%s%s", bn,
             load == kLoadTma ? "tma" : "manual", rows, cut, how);
  else
    snprintf(t_path_buf, sizeof(t_path_buf), "%s%s%s%s", kPathNames[bi][load][epi], rows, cut,
             how);
  t_last_path = t_path_buf;
  const cudaError_t e =
      m64 ? launch_gemm_f16_tc_m64(tmA, tmB, tmC, a, grid, stream)
          : (am < kBM ? launch_gemm_f16_tc_skinny(am, epi, tmA, tmB, tmC, a, grid, stream)
                      : launch_gemm_f16_tc(bn, load, epi, tmA, tmB, tmC, a, grid, stream, kpb));
  if (e != cudaSuccess) return GEMM_ERR_CUDA;
  return copy_back();
}

int gemm_f16_device(const uint16_t* A, const uint16_t* B, uint16_t* C, int M, int N, int K,
                    long long lda, long long ldb, long long ldc, float alpha, float beta,
                    cudaStream_t stream) {
  return gemm_f16_impl(A, B, C, false, M, N, K, lda, ldb, ldc, alpha, beta, stream);
}

int sgemm_f32_device(const float* A, const float* B, float* C, int M, int N, int K, long long lda,
                     long long ldb, long long ldc, float alpha, float beta, cudaStream_t stream) {
  if (int rc = check_common(A, B, C, M, N, K, lda, ldb, ldc, alpha, 4)) return rc;
  if (M == 0 || N == 0) {
    t_last_path = "noop";
    return GEMM_OK;
  }
  DevState* d = nullptr;
  if (int rc = device_state(&d, nullptr)) return rc;
  if (alpha == 0.0f || K == 0) {
    t_last_path = "f32.scale";
    return launch_scale_f32(C, ldc, M, N, beta, scale_grid(*d, 1ll * M * N), stream) == cudaSuccess
               ? GEMM_OK
               : GEMM_ERR_CUDA;
  }
  const int force = g_force_path.load();
  // Three tensor-core products of split operands whenever K has at least 64
  // elements: measured faster than the FFMA kernel at every M and N tried,
  // skinny and tiny shapes included (3xTF32: 16 x 8192 x 8192 274 us against
  // 830 us; 128^3: 14 us against 18 us); a shorter K stays on the FFMA kernel.
  // The parts are scaled halves (3xFP16, twice the tf32 rate) unless the
  // product is tiny (M*N*K at most 256^3), where the 3xTF32 form's simpler
  // pre-pass is as fast or faster (measured, same box, L2 flushed: 128^3
  // 17.0 us against 14.9 for 3xTF32, 200^3 19.0 / 17.0, 256^3 19.0 / 18.7,
  // 512^3 21.5 / 25.2, 1024^3 29.6 / 39.5, 16 x 8192 x 1024 37.5 / 53.9,
  // 8192 x 64 x 4096 111 / 136, 4096^3 302 / 502).  Path 8 forces 3xTF32,
  // path 16 3xFP16.
  if (force != 4 && force != 7 && (force == 8 || force == 16 || K >= 64)) {
    const int pairs = sgemm_3xtf32_max_pairs();
    const bool x16 = force == 16 ||
                     (force != 8 && static_cast<double>(M) * N * K > 256.0 * 256.0 * 256.0);
    auto round256 = [](size_t x) { return (x + 255) / 256 * 256; };
    const long long K2 = (K + 3) / 4 * 4;
    const long long lda2 = (K + 7) / 8 * 8, ldb2 = (N + 7) / 8 * 8;
    const size_t a_part = x16 ? round256(static_cast<size_t>(M) * lda2 * 2)
                              : static_cast<size_t>(M) * K2 * 4;
    const size_t b_part = x16 ? round256(static_cast<size_t>(K) * ldb2 * 2)
                              : static_cast<size_t>(N) * K2 * 4;
    // 3xFP16 exponents per K chunk: ea M x kchunks, eb kchunks x ldeb
    const int kchunks = (K + kF16x3ChunkK - 1) / kF16x3ChunkK;
    const long long ldeb = (N + 3) / 4 * 4 + 4;
    const size_t ea_bytes = round256(static_cast<size_t>(M) * kchunks * 4);
    const size_t e_bytes =
        x16 ? ea_bytes + round256(static_cast<size_t>(kchunks) * static_cast<size_t>(ldeb) * 4) : 0;
    const size_t need = 2 * (a_part + b_part) + e_bytes + 1024;
    if (pairs > 0 && need <= (static_cast<size_t>(16) << 30)) {
      uint8_t* buf = nullptr;
      {
        std::lock_guard<std::mutex> lk(g_mu);
        StreamWs& w = d->ws[reinterpret_cast<uintptr_t>(stream)];
        if (int rc = ensure_buffer(&w.split, &w.split_bytes, need)) return rc;
        buf = static_cast<uint8_t*>(w.split);
      }
      Tf32Args t{};
      t.pdl = true;   // the split pre-pass was launched just before
      CUtensorMap m1{}, m2{}, m3{}, m4{}, m5{}, m6{};
      if (x16) {
        F16x3Parts parts{};
        parts.A1 = reinterpret_cast<uint16_t*>(buf);
        parts.A2 = reinterpret_cast<uint16_t*>(buf + a_part);
        parts.B1 = reinterpret_cast<uint16_t*>(buf + 2 * a_part);
        parts.B2 = reinterpret_cast<uint16_t*>(buf + 2 * a_part + b_part);
        uint8_t* const eptr = buf + 2 * (a_part + b_part);
        parts.ea = reinterpret_cast<int*>(eptr);
        parts.eb = reinterpret_cast<int*>(eptr + ea_bytes);
        parts.ldeb = ldeb;
        parts.lda2 = lda2;
        parts.ldb2 = ldb2;
        // one launch: a block per (K chunk, 128 columns) of B, a warp per
        // (row, K chunk) of A
        const long long b_items = 1ll * kchunks * ((N + 127) / 128);
        const int grid_b = static_cast<int>(std::min<long long>(b_items, 2ll * d->sm_count));
        const int grid_a = static_cast<int>(
            std::max(1ll, std::min<long long>((1ll * M * kchunks + 31) / 32, 2ll * d->sm_count)));
        if (launch_f16x3_split(A, lda, B, ldb, parts, M, N, K, grid_a, grid_b, stream) !=
            cudaSuccess)
          return GEMM_ERR_CUDA;
        // k-blocks of 32 halves: A parts in 64-byte rows, B parts as 64-column
        // boxes of 32 k-rows
        if (int rc = make_map_f16(&m1, parts.A1, M, K, lda2, 32, 128, CU_TENSOR_MAP_SWIZZLE_64B))
          return rc;
        if (int rc = make_map_f16(&m2, parts.A2, M, K, lda2, 32, 128, CU_TENSOR_MAP_SWIZZLE_64B))
          return rc;
        if (int rc = make_map_f16(&m3, parts.B1, K, N, ldb2, 64, 32)) return rc;
        if (int rc = make_map_f16(&m4, parts.B2, K, N, ldb2, 64, 32)) return rc;
        t.ea = parts.ea;
        t.eb = parts.eb;
        t.ldeb = ldeb;
        t.kchunks = kchunks;
        t.kb_total = (K + 31) / 32;
      } else {
        float* Ab = reinterpret_cast<float*>(buf);
        float* As = Ab + a_part / 4;
        float* Bb = As + a_part / 4;
        float* Bs = Bb + b_part / 4;
        // one launch splits both operands, the blocks shared in proportion to the bytes
        const long long ttiles = ((K2 + 31) / 32) * ((N + 31) / 32);
        const int grid_a = scale_grid(*d, 1ll * M * K2 / 4);
        const int grid_b = static_cast<int>(std::min<long long>(ttiles, 8ll * d->sm_count));
        if (launch_split_tf32_ab(A, lda, Ab, As, B, ldb, Bb, Bs, K2, M, N, K, grid_a, grid_b,
                                 stream) != cudaSuccess)
          return GEMM_ERR_CUDA;
        // k-blocks of 16 floats: every part in 64-byte rows
        const CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_64B;
        if (int rc = make_map_f32(&m1, Ab, M, K, K2, 16, 128, sw)) return rc;
        if (int rc = make_map_f32(&m2, As, M, K, K2, 16, 128, sw)) return rc;
        if (int rc = make_map_f32(&m3, Bb, N, K, K2, 16, 128, sw)) return rc;
        if (int rc = make_map_f32(&m4, Bs, N, K, K2, 16, 128, sw)) return rc;
        if (int rc = make_map_f32(&m5, Bb, N, K, K2, 16, 64, sw)) return rc;
        if (int rc = make_map_f32(&m6, Bs, N, K, K2, 16, 64, sw)) return rc;
        t.Ab = Ab;
        t.As = As;
        t.Bb = Bb;
        t.Bs = Bs;
        t.kb_total = (K + 15) / 16;
      }
      t.C = C;
      t.M = M;
      t.N = N;
      t.K = K;
      t.ldc = ldc;
      t.alpha = alpha;
      t.beta = beta;
      t.tiles_m = (M + 255) / 256;
      t.tiles_n = (N + 255) / 256;
      const int tiles = t.tiles_m * t.tiles_n;
      // Few tiles for the pairs and a long K: every tile is cut into equal K
      // slices (whole 4-k-block chunks) that fill about one wave; each slice
      // publishes fp32 partial sums and the last to finish adds them up.
      // Otherwise the tiles of the last, partial wave run as two half-width
      // units each when the halves fit in one wave.  The plan counts in
      // 128-byte rows of K (32 floats or 64 halves, the same MMA work for
      // either kind): two of the kernel's 64-byte k-blocks, four of them one
      // accumulation chunk.  gemm_force_splits: 1 keeps whole-K units, > 1
      // sets the slice count.
      const int fs = g_force_splits.load();
      int splits = 1;
      if (force != 5) {
        const TailSplit ts = tf32_slice_plan(tiles, pairs, (t.kb_total + 1) / 2, fs);
        if (ts.splits > 1) {
          splits = ts.splits;
          t.kb_per_split = 2 * ts.kb_per_split;
        }
      }
      bool halves = false;
      t.splits = 1;
      // partial sums of `sliced` tiles cut into `per` slices: per tile 2 CTAs x
      // 8 epilogue warps x slices x (32 rows x 128 fp32)
      auto slice_scratch = [&](long long sliced, int per) -> int {
        const size_t wneed = static_cast<size_t>(sliced) * per * 2 * 8 * 32 * 128 * sizeof(float);
        std::lock_guard<std::mutex> lk(g_mu);
        StreamWs* w = nullptr;
        if (int rc = stream_scratch(d, stream, wneed, static_cast<size_t>(sliced) * 16, &w))
          return rc;
        t.part_ws = static_cast<float4*>(w->ptr);
        t.counters = static_cast<unsigned long long*>(w->counters);
        t.epoch = ++w->epoch;
        if (t.epoch == 0) t.epoch = ++w->epoch;   // 0 marks never-used counters
        return GEMM_OK;
      };
      const int rem = tiles % pairs;
      const int chunks = (t.kb_total + kSplitChunkKb - 1) / kSplitChunkKb;
      if (splits > 1) {
        t.splits = splits;
        t.dp_tiles = tiles;
        t.num_units = tiles * splits;
        if (int rc = slice_scratch(tiles, splits)) return rc;
      } else if (force != 5 && force != 15 && tiles > pairs && rem > 0 && 2 * rem <= pairs &&
                 chunks >= 6) {
        // The tiles of the last, partial wave as two K slices each, publisher
        // first (tail_first): the first slice (about 56% of the chunks, the
        // first wave's loads being the slow ones) is a worker's first unit,
        // the second a worker's last.  Half-width units instead took nearly a
        // full tile's time for half the work (3xFP16, same box: 4096^3 302 ->
        // 288 us, 5120^3 553 -> 536 us; first slices of 50% or 62% of the
        // chunks were slower than 56%).
        t.tail_first = 1;
        t.kb_per_split = std::min(chunks - 1, (chunks + 2) / 2) * kSplitChunkKb;
        t.dp_tiles = tiles - rem;
        t.num_units = t.dp_tiles + 2 * rem;
        if (int rc = slice_scratch(rem, 2)) return rc;
      } else {
        halves = force != 5 && rem > 0 && 2 * rem <= pairs;
        t.dp_tiles = halves ? tiles - rem : tiles;
        t.num_units = t.dp_tiles + 2 * (tiles - t.dp_tiles);
        t.kb_per_split = t.kb_total;
      }
      t.group_m = 8;
      t.vec_c = aligned16(C) && ldc % 4 == 0;
      t.wait_limit_ns = static_cast<unsigned long long>(g_wait_limit_ns.load());
      t.status = d->status;
      const int grid = 2 * std::min(t.num_units, pairs);
      if (x16)
        t_last_path = splits > 1 ? "f32.3xf16.pair.ksplit"
                      : t.tail_first ? "f32.3xf16.pair.ktail"
                                     : (halves ? "f32.3xf16.pair.halves" : "f32.3xf16.pair");
      else
        t_last_path = splits > 1 ? "f32.3xtf32.pair.ksplit"
                      : t.tail_first ? "f32.3xtf32.pair.ktail"
                                     : (halves ? "f32.3xtf32.pair.halves" : "f32.3xtf32.pair");
      const cudaError_t e = x16 ? launch_sgemm_3xf16(m1, m2, m3, m4, t, grid, stream)
                                : launch_sgemm_3xtf32(m1, m2, m3, m4, m5, m6, t, grid, stream);
      return e == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
    }
  }
  const bool vec = force != 4 && aligned16(A) && aligned16(B) && aligned16(C) && lda % 4 == 0 &&
                   ldb % 4 == 0 && ldc % 4 == 0;
  SgemmArgs s{A, B, C, M, N, K, lda, ldb, ldc, alpha, beta};
  t_last_path = vec ? "f32.ffma.vec" : "f32.ffma.scalar";
  return launch_sgemm_ffma(vec, s, stream) == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

size_t extent_bytes(int rows, int cols, long long ld, size_t elem) {
  if (rows <= 0 || cols <= 0) return 0;
  return (static_cast<size_t>(rows - 1) * static_cast<size_t>(ld) + static_cast<size_t>(cols)) *
         elem;
}

template <typename T, typename Fn>
int host_form(const T* A, const T* B, T* C, int M, int N, int K, int lda, int ldb, int ldc,
              float alpha, float beta, cudaStream_t stream, Fn device_fn) {
  if (int rc = check_common(A, B, C, M, N, K, lda, ldb, ldc, alpha)) return rc;
  if (M == 0 || N == 0) return GEMM_OK;
  DevState* d = nullptr;
  if (int rc = device_state(&d, nullptr)) return rc;
  std::lock_guard<std::mutex> host_lk(g_host_mu);
  const bool read_ab = alpha != 0.0f && K > 0;
  const bool read_c = beta != 0.0f || ldc > N;   // ldc > N: the padding must come back unchanged
  const size_t ba = read_ab ? extent_bytes(M, K, lda, sizeof(T)) : 0;
  const size_t bb = read_ab ? extent_bytes(K, N, ldb, sizeof(T)) : 0;
  const size_t bc = extent_bytes(M, N, ldc, sizeof(T));
  T *dA = nullptr, *dB = nullptr, *dC = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (read_ab) {
      if (int rc = ensure_buffer(&d->host_buf[0], &d->host_bytes[0], ba)) return rc;
      if (int rc = ensure_buffer(&d->host_buf[1], &d->host_bytes[1], bb)) return rc;
      dA = static_cast<T*>(d->host_buf[0]);
      dB = static_cast<T*>(d->host_buf[1]);
    }
    if (int rc = ensure_buffer(&d->host_buf[2], &d->host_bytes[2], bc)) return rc;
    dC = static_cast<T*>(d->host_buf[2]);
    for (cudaStream_t* st : {&d->copy_in, &d->copy_back})
      if (!*st && cudaStreamCreateWithFlags(st, cudaStreamNonBlocking) != cudaSuccess)
        return GEMM_ERR_CUDA;
    for (cudaEvent_t& e : d->host_ev)
      if (!e && cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess)
        return GEMM_ERR_CUDA;
  }
  cudaEvent_t* const ev_in = d->host_ev;                    // [kHostBlocks]
  cudaEvent_t* const ev_done = d->host_ev + kHostBlocks;    // [kHostBlocks]
  cudaEvent_t const ev_entry = d->host_ev[2 * kHostBlocks];
  cudaEvent_t const ev_exit = d->host_ev[2 * kHostBlocks + 1];
  // Blocks of rows of A and C, on three streams: the copy-in stream brings B
  // and then block after block of A and C; `stream` computes block j once it
  // is in; the copy-back stream returns block j's C once it is computed.  So
  // copies in, GEMMs and copies back of different blocks overlap (the two
  // directions of the host link run concurrently).  Blocks are multiples of
  // 256 rows: whole output tiles of the big kernels.
  const int nblk = (read_ab && M >= 2048) ? kHostBlocks : 1;
  const int rb = (M + nblk - 1) / nblk;
  const int rows_per = nblk == 1 ? M : (rb + 255) / 256 * 256;
  // the copies follow whatever the caller queued on `stream` before this call
  if (cudaEventRecord(ev_entry, stream) != cudaSuccess ||
      cudaStreamWaitEvent(d->copy_in, ev_entry, 0) != cudaSuccess)
    return GEMM_ERR_CUDA;
  if (read_ab && cudaMemcpyAsync(dB, B, bb, cudaMemcpyHostToDevice, d->copy_in) != cudaSuccess)
    return GEMM_ERR_CUDA;
  int j = 0;
  for (int r0 = 0; r0 < M; r0 += rows_per, ++j) {
    const int mr = std::min(rows_per, M - r0);
    const size_t a_off = static_cast<size_t>(r0) * lda, c_off = static_cast<size_t>(r0) * ldc;
    if (read_ab && cudaMemcpyAsync(dA + a_off, A + a_off, extent_bytes(mr, K, lda, sizeof(T)),
                                   cudaMemcpyHostToDevice, d->copy_in) != cudaSuccess)
      return GEMM_ERR_CUDA;
    const size_t cbytes = extent_bytes(mr, N, ldc, sizeof(T));
    if (read_c && cudaMemcpyAsync(dC + c_off, C + c_off, cbytes, cudaMemcpyHostToDevice,
                                  d->copy_in) != cudaSuccess)
      return GEMM_ERR_CUDA;
    if (cudaEventRecord(ev_in[j], d->copy_in) != cudaSuccess ||
        cudaStreamWaitEvent(stream, ev_in[j], 0) != cudaSuccess)
      return GEMM_ERR_CUDA;
    if (int rc = device_fn(read_ab ? dA + a_off : nullptr, dB, dC + c_off, mr, N, K, lda, ldb, ldc,
                           alpha, beta, stream))
      return rc;
    if (cudaEventRecord(ev_done[j], stream) != cudaSuccess ||
        cudaStreamWaitEvent(d->copy_back, ev_done[j], 0) != cudaSuccess ||
        cudaMemcpyAsync(C + c_off, dC + c_off, cbytes, cudaMemcpyDeviceToHost, d->copy_back) !=
            cudaSuccess)
      return GEMM_ERR_CUDA;
  }
  // the caller's stream (and so the next call) waits for the last copy back
  if (cudaEventRecord(ev_exit, d->copy_back) != cudaSuccess ||
      cudaStreamWaitEvent(stream, ev_exit, 0) != cudaSuccess)
    return GEMM_ERR_CUDA;
  return cudaStreamSynchronize(stream) == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

}  // namespace

// Device facts and the tensor-map encoder, for entry points defined in other
// files of the library.
int query_device(int* sm_count, DeviceStatus** status, unsigned long long* wait_limit_ns) {
  DevState* d = nullptr;
  if (int rc = device_state(&d, nullptr)) return rc;
  *sm_count = d->sm_count;
  *status = d->status;
  *wait_limit_ns = static_cast<unsigned long long>(g_wait_limit_ns.load());
  return GEMM_OK;
}

int encode_map_f16(CUtensorMap* map, const void* ptr, int rows, int cols, long long ld,
                   int box_cols, int box_rows) {
  return make_map_f16(map, ptr, rows, cols, ld, box_cols, box_rows);
}

void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

void set_last_path(const char* path) { t_last_path = path; }

int stage_kblocks() { return g_stage_kblocks.load() == 2 ? 2 : 1; }

}  // namespace gb300

using namespace gb300;

extern "C" {

int gemm_f16(const uint16_t* A, const uint16_t* B, uint16_t* C, int M, int N, int K, float alpha,
             float beta, cudaStream_t stream) {
  return gemm_f16_device(A, B, C, M, N, K, K, N, N, alpha, beta, stream);
}

int gemm_f16_ld(const uint16_t* A, const uint16_t* B, uint16_t* C, int M, int N, int K, int lda,
                int ldb, int ldc, float alpha, float beta, cudaStream_t stream) {
  return gemm_f16_device(A, B, C, M, N, K, lda, ldb, ldc, alpha, beta, stream);
}

int gemm_f16_f32out(const uint16_t* A, const uint16_t* B, float* C, int M, int N, int K, int lda,
                    int ldb, int ldc, float alpha, float beta, cudaStream_t stream) {
  return gemm_f16_impl(A, B, C, true, M, N, K, lda, ldb, ldc, alpha, beta, stream);
}

int gemm_f32_to_f16(const float* src, uint16_t* dst, long long n, cudaStream_t stream) {
  if (n < 0) return GEMM_ERR_DIM;
  if (n == 0) return GEMM_OK;
  if (src == nullptr || dst == nullptr) return GEMM_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(src) & 3u) || (reinterpret_cast<uintptr_t>(dst) & 1u))
    return GEMM_ERR_ARG;
  DevState* d = nullptr;
  if (int rc = device_state(&d, nullptr)) return rc;
  t_last_path = "f32_to_f16";
  // up to 64 blocks per SM: about one step per thread, so the block scheduler
  // balances the SMs (22.5 -> 20.5 us for 4096 x 4096 against 8 per SM)
  return launch_f32_to_f16(src, dst, n, scale_grid(*d, (n + 7) / 8, 64), stream) == cudaSuccess
             ? GEMM_OK
             : GEMM_ERR_CUDA;
}

int sgemm_f32(const float* A, const float* B, float* C, int M, int N, int K, float alpha,
              float beta, cudaStream_t stream) {
  return sgemm_f32_device(A, B, C, M, N, K, K, N, N, alpha, beta, stream);
}

int sgemm_f32_ld(const float* A, const float* B, float* C, int M, int N, int K, int lda, int ldb,
                 int ldc, float alpha, float beta, cudaStream_t stream) {
  return sgemm_f32_device(A, B, C, M, N, K, lda, ldb, ldc, alpha, beta, stream);
}

int gemm_f16_host(const uint16_t* A, const uint16_t* B, uint16_t* C, int M, int N, int K, int lda,
                  int ldb, int ldc, float alpha, float beta, cudaStream_t stream) {
  return host_form<uint16_t>(A, B, C, M, N, K, lda, ldb, ldc, alpha, beta, stream,
                             [](const uint16_t* a, const uint16_t* b, uint16_t* c, int m, int n,
                                int k, long long la, long long lb, long long lc, float al,
                                float be, cudaStream_t s) {
                               return gemm_f16_device(a, b, c, m, n, k, la, lb, lc, al, be, s);
                             });
}

int sgemm_f32_host(const float* A, const float* B, float* C, int M, int N, int K, int lda, int ldb,
                   int ldc, float alpha, float beta, cudaStream_t stream) {
  return host_form<float>(A, B, C, M, N, K, lda, ldb, ldc, alpha, beta, stream,
                          [](const float* a, const float* b, float* c, int m, int n, int k,
                             long long la, long long lb, long long lc, float al, float be,
                             cudaStream_t s) {
                            return sgemm_f32_device(a, b, c, m, n, k, la, lb, lc, al, be, s);
                          });
}

int gemm_l2_flush(size_t bytes, cudaStream_t stream) {
  DevState* d = nullptr;
  if (int rc = device_state(&d, nullptr)) return rc;
  const size_t n = bytes ? bytes : 2 * static_cast<size_t>(d->l2_bytes);
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (int rc = ensure_buffer(&d->flush, &d->flush_bytes, n)) return rc;
  }
  return cudaMemsetAsync(d->flush, 0, n, stream) == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

int gemm_force_path(int path) {
  if (path < 0 || path > 17) return GEMM_ERR_ARG;
  return g_force_path.exchange(path);
}

int gemm_stage_kblocks(int kblocks) {
  if (kblocks < 0 || kblocks > 2) return GEMM_ERR_ARG;
  return g_stage_kblocks.exchange(kblocks);
}

int gemm_force_splits(int splits) {
  if (splits < 0) return GEMM_ERR_ARG;
  return g_force_splits.exchange(splits);
}

long long gemm_set_wait_limit_ns(long long ns) {
  return g_wait_limit_ns.exchange(ns > 0 ? ns : 2000000000ll);
}

int gemm_debug_status(void) {
  DevState* d = nullptr;
  if (int rc = device_state(&d, nullptr)) return rc;
  if (cudaDeviceSynchronize() != cudaSuccess) return GEMM_ERR_CUDA;
  DeviceStatus s{};
  if (cudaMemcpy(&s, d->status, sizeof(s), cudaMemcpyDeviceToHost) != cudaSuccess)
    return GEMM_ERR_CUDA;
  const DeviceStatus zero{};
  if (cudaMemcpy(d->status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
    return GEMM_ERR_CUDA;
  return s.code;
}

const char* gemm_last_path(void) { return t_last_path; }

int gemm_debug_wait_probe(long long limit_ns, cudaStream_t stream) {
  if (limit_ns <= 0) return GEMM_ERR_ARG;
  DevState* d = nullptr;
  if (int rc = device_state(&d, nullptr)) return rc;
  t_last_path = "wait_probe";
  return launch_wait_probe(static_cast<unsigned long long>(limit_ns), d->status, stream) ==
                 cudaSuccess
             ? GEMM_OK
             : GEMM_ERR_CUDA;
}

int gemm_plan_stream_k(long long tiles, long long slots, int kb, int all_tiles, long long* out) {
  if (out == nullptr) return GEMM_ERR_NULL;
  const SkPlan p = all_tiles == 2 ? plan_tail_stream_k(tiles, slots, kb)
                                  : plan_stream_k(tiles, slots, kb, all_tiles != 0);
  out[0] = p.dp_tiles;
  out[1] = p.sk_tiles;
  out[2] = p.workers;
  out[3] = p.max_pieces;
  return GEMM_OK;
}

int gemm_plan_tf32_slices(long long tiles, long long pairs, int kb, int forced_slices,
                          long long* out) {
  if (out == nullptr) return GEMM_ERR_NULL;
  if (tiles < 0 || pairs < 0 || kb < 0 || forced_slices < 0) return GEMM_ERR_ARG;
  const TailSplit ts = tf32_slice_plan(tiles, pairs, kb, forced_slices);
  out[0] = ts.splits;
  out[1] = ts.splits > 1 ? ts.kb_per_split : kb;
  return GEMM_OK;
}

long long gemm_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char* gemm_strerror(int code) {
  switch (code) {
    case GEMM_OK: return "ok";
    case GEMM_ERR_NULL: return "null pointer";
    case GEMM_ERR_DIM: return "negative dimension";
    case GEMM_ERR_LD: return "leading dimension smaller than the row length";
    case GEMM_ERR_CUDA: return "CUDA call or kernel launch failed";
    case GEMM_ERR_DEVICE: return "device is not compute capability 10.3 (sm_103a)";
    case GEMM_ERR_TIMEOUT: return "a kernel gave up waiting (time limit reached)";
    case GEMM_ERR_ARG: return "invalid argument";
    default: return "unknown error";
  }
}

int gemm_release(void) {
  std::lock_guard<std::mutex> host_lk(g_host_mu);
  std::lock_guard<std::mutex> lk(g_mu);
  int prev = 0;
  if (cudaGetDevice(&prev) != cudaSuccess) return GEMM_ERR_CUDA;
  int rc = GEMM_OK;
  for (int dev = 0; dev < kMaxDevices; ++dev) {
    DevState& d = g_dev[dev];
    void** bufs[4] = {&d.flush, &d.host_buf[0], &d.host_buf[1], &d.host_buf[2]};
    size_t* sizes[4] = {&d.flush_bytes, &d.host_bytes[0], &d.host_bytes[1], &d.host_bytes[2]};
    bool any = !d.ws.empty();
    for (void** b : bufs) any = any || *b != nullptr;
    if (!any) continue;
    if (cudaSetDevice(dev) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
      rc = GEMM_ERR_CUDA;
      continue;
    }
    for (int i = 0; i < 4; ++i) {
      if (*bufs[i]) cudaFree(*bufs[i]);
      *bufs[i] = nullptr;
      *sizes[i] = 0;
    }
    for (auto& kv : d.ws) {
      if (kv.second.ptr) cudaFree(kv.second.ptr);
      if (kv.second.counters) cudaFree(kv.second.counters);
      if (kv.second.realigned) cudaFree(kv.second.realigned);
      if (kv.second.split) cudaFree(kv.second.split);
    }
    d.ws.clear();
    for (cudaStream_t* st : {&d.copy_in, &d.copy_back}) {
      if (*st) cudaStreamDestroy(*st);
      *st = nullptr;
    }
    for (cudaEvent_t& e : d.host_ev) {
      if (e) cudaEventDestroy(e);
      e = nullptr;
    }
  }
  cudaSetDevice(prev);
  return rc;
}

}  // extern "C"
