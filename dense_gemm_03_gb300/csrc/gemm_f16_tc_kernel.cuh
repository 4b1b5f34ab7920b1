// gemm_f16_tc_kernel.cuh -- fp16-in / fp32-accumulate GEMM on the 5th-generation
// tensor cores (tcgen05) of sm_103a.
//
// Computes C := alpha*A*B + beta*C with A (M x K) and B (K x N) row-major fp16,
// an fp32 accumulator in tensor memory (TMEM), and an fp32 epilogue rounded to
// fp16 ("LeetGPU GEMM T4" page: baseline section for the formula, WMMA
// sections for the half-operand / float-accumulator split and the skipped
// load of C when beta == 0).  The three-phase structure -- stage tiles of A
// and B in shared memory along K, multiply-accumulate, write back the C tile
// -- and the double-buffered staging are those of the "advanced SGEMM" page
// (section on tiling and data movement); on sm_103a they become a
// multi-stage mbarrier ring fed by TMA and drained by tcgen05.mma.
//
// One CTA per SM (or one CTA pair per two SMs), persistent over work units,
// warp-specialised:
//   producer warp(s)  TMA tile loads (or, for unaligned operands, 4 warps of
//                     predicated element loads written in the same layout)
//   MMA warp          one thread issues tcgen05.mma (M=128, or M=256 on a CTA
//                     pair, or M=64 on 64-row tiles; N=BN or BN/2; K=16) into
//                     a double-buffered TMEM accumulator (2 x BN fp32 columns)
//   8 epilogue warps  warp (q, h) owns TMEM lanes 32q..32q+31 (= tile rows;
//                     on 64-row tiles the first 16 of them hold rows
//                     16q..16q+15) and the h-th half of the unit's columns; in 32-column
//                     sub-chunks it loads the accumulator (the next sub-chunk's
//                     load in flight), applies alpha/beta in fp32, rounds to
//                     fp16 and stores by TMA through 2 KB staging tiles (on
//                     CTA pairs C itself is TMA-loaded into those tiles during
//                     the main loop), or stores fp16/fp32 from registers with
//                     predicated accesses, or publishes fp32 partial sums.
// The epilogue of one unit overlaps the main loop of the next.
//
// A unit is a whole output tile, half of one (its columns split in two, for
// the last partial wave), a split-K slice, or a piece of a stream-K range.
// Pieces of a shared tile publish fp32 partial sums; the piece that finishes
// last (counted per launch) adds them up in k order and runs the epilogue, so
// no CTA ever waits for another.
//
// Shared-memory operand layouts (128-byte swizzle, 1024-byte aligned; a ring
// stage holds one k-block, or two, the second's A and B parts after the
// first's):
//   A stage: 128 rows x 64 halves, K-major; row r at r*128 B, 16-byte chunk c
//            of the row stored at chunk (c ^ (r % 8)).  SBO = 1024 B.
//   B stage: BN/64 column blocks of 64 (k) rows x 64 halves, N-major (MN-major
//            operand); k-row at k*128 B inside its block, same swizzle.
//            LBO = 8 KB (next 64 columns), SBO = 1024 B (next 8 k-rows).
// Epilogue staging tile: 32 rows x 32 halves, 64-byte swizzle: row r at r*64 B,
//            16-byte chunk c stored at chunk (c ^ ((r / 2) % 4)).
#pragma once
#include "internal.h"
#include "ptx.cuh"

namespace gb300 {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;                       // halves per k-block: one 128-byte swizzle row
constexpr int kUmmaK = 16;                   // K of one tcgen05.mma kind::f16
constexpr int kABytes = BM * BK * 2;         // 16 KB
constexpr int kBBlockBytes = BK * 128;       // one 64-column block of a B stage: 8 KB
constexpr int kSubCols = 32;                 // epilogue sub-chunk width
constexpr int kEpiBufBytes = 32 * kSubCols * 2;   // 2 KB staging tile
constexpr unsigned long long kDrainLimitNs = 1000000000ull;
// C staging tiles per epilogue warp in the CTA-pair kernel (2: six stages of
// A/B fit beside them; 4: the warp's whole C part, five stages).
constexpr int kCsBufs = 2;

// PAIR: two CTAs of a cluster share each tcgen05.mma.cta_group::2 (M = 256);
// each CTA stages its own 128 rows of A and half of the BN columns of B.  A
// pair tile is 256 wide, or 224 / 192 wide (the tile-family comparison: the
// MMA takes N = BN; B is still staged in whole 64-column boxes, of which the
// MMA reads the first BN/2 columns).
// AM: rows of A staged per k-block.  128 normally; 32 or 64 for shapes with
// M <= AM, whose stages then hold more of B (the MMA still reads 128 rows of
// A: the rows past AM come from the stage's B region and only produce
// accumulator rows >= M, which are never stored).
// KPB: k-blocks per ring stage (1 or 2).  A stage holds KPB consecutive
// k-blocks, each as its A part followed by its B part, and is loaded and
// released as one: a CTA's TMA ring completes about one stage per ~0.4 us of
// DRAM latency whatever the stage's size, so two k-blocks per stage move
// about 1.5x the bytes per CTA in the same time.
template <int BN, bool PAIR, bool CS = false, int AM = 128, int KPB = 1>
struct TcCfg {
  static constexpr int kBLoadCols = PAIR ? BN / 2 : BN;   // B columns this CTA gives the MMA
  static constexpr int kBStageCols = (kBLoadCols + 63) / 64 * 64;   // staged: whole boxes
  static constexpr int kBBytes = kBStageCols * BK * 2;
  static constexpr int kAStageBytes = AM * BK * 2;
  static constexpr int kKbBytes = kAStageBytes + kBBytes;   // one k-block of A and B
  static constexpr int kStageBytes = KPB * kKbBytes;
  // skinny stages: as many as fit beside the epilogue tiles, at most 16 k-blocks
  static constexpr int kSkinnyStages = (232448 - 1024 - 1024 - 8 * 2 * kEpiBufBytes) / kStageBytes;
  static constexpr int kStages1 =
      AM < 128 ? (kSkinnyStages < 16 / KPB ? kSkinnyStages : 16 / KPB)
               : (PAIR ? ((CS && kCsBufs > 2) ? 5 : 6) : ((BN == 256) ? 4 : (BN == 128 ? 6 : 8)));
  static constexpr int kStages = AM < 128 ? kStages1 : kStages1 / KPB;
  // TMEM columns per accumulator (a power of two) and for both of them
  static constexpr int kAccStride = BN <= 64 ? 64 : (BN <= 128 ? 128 : 256);
  static constexpr int kTmemCols = 2 * kAccStride;
  static_assert(PAIR ? (BN == 256 || BN == 224 || BN == 192) : (BN == 64 || BN == 128 || BN == 256),
                "tile width");
  static_assert(AM == 128 || (!PAIR && kKbBytes >= kABytes), "skinny stages span 128 A rows");
  static_assert(KPB == 1 || KPB == 2, "k-blocks per stage");
};

// Warp roles.  With TMA loads: 1 producer, 1 MMA and 8 epilogue warps (two
// per TMEM lane quadrant, each on half of the columns).  With predicated loads:
// 4 producer warps, 1 MMA and 4 epilogue warps (each on all columns), so that
// no sub-partition runs more than 3 warps and every thread keeps 168 registers.
template <int LOAD>
struct Roles {
  static constexpr int kProdWarps = (LOAD == kLoadTma) ? 1 : 4;
  static constexpr int kEpiWarps = (LOAD == kLoadTma) ? 8 : 4;
  static constexpr int kMmaWarp = kProdWarps;
  static constexpr int kEpiWarp0 = kProdWarps + 1;
  static constexpr int kWarps = kProdWarps + 1 + kEpiWarps;
  static constexpr int kThreads = kWarps * 32;
};

// Counters per tail tile: one per epilogue warp (at most 8).
constexpr int kTailCounters = 8;

template <int BN, int EPI, bool PAIR, int AM = 128, int KPB = 1>
struct Smem {
  // C read by TMA into the epilogue's staging tiles: the CTA-pair kernel with
  // TMA stores
  static constexpr bool kCs = PAIR && (EPI == kEpiTma || EPI == kEpiF32Tma);
  using Cfg = TcCfg<BN, PAIR, kCs, AM, KPB>;
  // 32 x 32 staging tiles per epilogue warp
  static constexpr int kBufs = kCs ? kCsBufs : 2;
  static constexpr int kWarpEpiBytes = kBufs * kEpiBufBytes;
  static constexpr int kEpiOff = Cfg::kStages * Cfg::kStageBytes;
  static constexpr int kEpiBytes = (EPI == kEpiPartial || EPI == kEpiF32) ? 0 : 8 * kWarpEpiBytes;
  static constexpr int kBarOff = kEpiOff + kEpiBytes;
  // full[S], empty[S], acc_full[2], acc_empty[2], mma_done, tmem_free,
  // c_full[8 warps][kBufs staging tiles]
  static constexpr int kNumBars = 2 * Cfg::kStages + 2 + 2 + 1 + 1 + 8 * kBufs;
  static constexpr int kTmemPtrOff = kBarOff + kNumBars * 8;
  static constexpr int kUsed = kTmemPtrOff + 16;
  static constexpr int kAlloc = kUsed + 1024;  // the dynamic base is aligned up to 1024 B
  static_assert(kAlloc <= 232448, "shared memory budget");
};

struct Unit {
  int m0, n0, kb0, kb1, split;
  int tail;       // 1 for a K slice of a tail tile (or a piece of a shared stream-K tile)
  int tail_idx;   // index of the tail tile (tail units only)
  int npieces;    // slices or pieces the tile is cut into (tail units only)
  int ncols;      // columns of the unit: BN, or BN/2 for a half-width tail unit
};

// Output tile index (in visiting order) -> first row and column.  Tiles are
// visited in groups of group_m tile-rows so that concurrently running CTAs
// share B panels in L2.
__device__ __forceinline__ void tile_origin(const TcArgs& p, int tile, int bn, int bm_tile,
                                            int rank, Unit& x) {
  const int group = p.group_m * p.tiles_n;
  const int g = tile / group;
  const int first_m = g * p.group_m;
  const int gm = min(p.tiles_m - first_m, p.group_m);
  const int r = tile - g * group;
  x.m0 = (first_m + r % gm) * bm_tile + rank * BM;
  x.n0 = (r / gm) * bn;
}

// Work unit u -> output tile and K range.  Units [0, dp_tiles*splits) are
// whole tiles (or split-K slices); the rest are K slices of the tail tiles.
__device__ __forceinline__ Unit decode_unit(const TcArgs& p, int u, int bn, int bm_tile = BM,
                                           int rank = 0) {
  Unit x;
  int tile, kpb;
  const int dp_units = p.dp_tiles * p.splits;
  if (p.tail_first) {
    // The T tiles cut in two are the first T in visiting order (so that the
    // first wave, their first slices beside the first whole tiles, reads the
    // same panels of A and B as a wave of whole tiles would).  Units [0, T)
    // are their first slices, [T, T + dp_tiles) the whole tiles T, T + 1, ...,
    // then come their second slices.
    const int T = (p.num_units - p.dp_tiles) >> 1;
    x.split = 0;
    x.ncols = bn;
    if (u >= T && u < T + p.dp_tiles) {
      tile_origin(p, u, bn, bm_tile, rank, x);
      x.tail = 0;
      x.tail_idx = 0;
      x.npieces = 1;
      x.kb0 = 0;
      x.kb1 = p.kb_total;
      return x;
    }
    x.tail_idx = u < T ? u : u - T - p.dp_tiles;
    x.split = u < T ? 0 : 1;
    x.tail = 1;
    x.npieces = 2;
    tile_origin(p, x.tail_idx, bn, bm_tile, rank, x);
    x.kb0 = x.split ? p.tail_kb_per_split : 0;
    x.kb1 = x.split ? p.kb_total : p.tail_kb_per_split;
    return x;
  }
  if (u < dp_units) {
    tile = u / p.splits;
    x.split = u - tile * p.splits;
    kpb = p.kb_per_split;
    x.tail = 0;
    x.tail_idx = 0;
    x.npieces = 1;
    x.ncols = bn;
  } else if (p.tail_halves) {
    // two half-width units per tail tile, each over the whole K
    const int v = u - dp_units;
    tile = p.dp_tiles + (v >> 1);
    tile_origin(p, tile, bn, bm_tile, rank, x);
    x.n0 += (v & 1) * (bn / 2);
    x.ncols = bn / 2;
    x.split = 0;
    x.tail = 0;
    x.tail_idx = 0;
    x.npieces = 1;
    x.kb0 = 0;
    x.kb1 = p.kb_total;
    return x;
  } else {
    const int v = u - dp_units;
    x.tail_idx = v / p.tail_splits;
    x.split = v - x.tail_idx * p.tail_splits;
    tile = p.dp_tiles + x.tail_idx;
    kpb = p.tail_kb_per_split;
    x.tail = 1;
    x.npieces = p.tail_splits;
    x.ncols = bn;
  }
  tile_origin(p, tile, bn, bm_tile, rank, x);
  x.kb0 = x.split * kpb;
  x.kb1 = min(p.kb_total, x.kb0 + kpb);
  return x;
}

// Stream-K: first k-block of worker w's range, and the worker whose range
// holds k-block x (the largest w with sk_begin(w) <= x).
__device__ __forceinline__ int sk_begin(const TcArgs& p, int w) {
  return static_cast<int>(static_cast<long long>(w) * p.sk_iters / p.sk_workers);
}
__device__ __forceinline__ int sk_owner(const TcArgs& p, int x) {
  return static_cast<int>((static_cast<long long>(x + 1) * p.sk_workers - 1) / p.sk_iters);
}

// Position of one worker in its sequence of units.  sk_order 0: first the
// units worker, worker + nworkers, ... below num_units, then the pieces of its
// stream-K range [x, x_end).  sk_order 1: first the piece [x, x_end) (part of
// a tile that another worker finishes), then the units, then the piece
// [fx, fx_end) that ends its tile.
struct UnitCursor {
  int u, x, x_end, fx, fx_end;   // the host keeps sk_iters below 2^31
};

__device__ __forceinline__ UnitCursor first_unit(const TcArgs& p, int worker) {
  UnitCursor c;
  c.u = worker;
  c.x = c.x_end = c.fx = c.fx_end = 0;
  if (p.sk_tiles > 0 && worker < p.sk_workers) {
    const int x0 = sk_begin(p, worker), x1 = sk_begin(p, worker + 1);
    if (p.sk_order == 0) {
      c.x = x0;
      c.x_end = x1;
    } else {
      // the range is no longer than a tile: it ends the tile holding x0 (and
      // may start the next one), or it lies inside one tile
      const int tile_end = (x0 / p.kb_total + 1) * p.kb_total;
      if (x1 >= tile_end) {
        c.fx = x0;
        c.fx_end = tile_end;
        c.x = tile_end;
        c.x_end = x1;
      } else {
        c.x = x0;
        c.x_end = x1;
      }
    }
  }
  return c;
}

// The stream-K piece starting at k-block x of the shared region (at most
// x_end, within one tile) into t; returns the k-blocks it covers.
__device__ __forceinline__ int sk_piece(const TcArgs& p, int x, int x_end, int worker, int bn,
                                        int bm_tile, int rank, Unit& t) {
  const int kb = p.kb_total;
  const int s = x / kb;   // stream-K tile
  t.kb0 = x - s * kb;
  t.kb1 = min(kb, t.kb0 + (x_end - x));
  const int first = sk_owner(p, s * kb);
  const int last = sk_owner(p, (s + 1) * kb - 1);
  t.npieces = last - first + 1;
  t.split = worker - first;
  t.tail = t.npieces > 1 ? 1 : 0;
  t.tail_idx = s;
  t.ncols = bn;
  tile_origin(p, p.sk_tile0 + s, bn, bm_tile, rank, t);
  return t.kb1 - t.kb0;
}

// The worker's next unit into t; false when it has none left.
__device__ __forceinline__ bool next_unit(const TcArgs& p, UnitCursor& c, int worker,
                                          int nworkers, int bn, int bm_tile, int rank, Unit& t) {
  if (p.sk_order != 0 && c.x < c.x_end) {
    c.x += sk_piece(p, c.x, c.x_end, worker, bn, bm_tile, rank, t);
    return true;
  }
  if (c.u < p.num_units) {
    t = decode_unit(p, c.u, bn, bm_tile, rank);
    c.u += nworkers;
    return true;
  }
  if (p.sk_order != 0) {
    if (c.fx >= c.fx_end) return false;
    c.fx += sk_piece(p, c.fx, c.fx_end, worker, bn, bm_tile, rank, t);
    return true;
  }
  if (c.x >= c.x_end) return false;
  c.x += sk_piece(p, c.x, c.x_end, worker, bn, bm_tile, rank, t);
  return true;
}

// Partial sums of one K slice of a tail tile: BN/4 column quads x 128 rows of
// float4, so that the 32 lanes of a warp (32 consecutive rows) touch 512
// contiguous bytes.  Private to this kernel.
__device__ __forceinline__ float4* tail_partials(const TcArgs& p, int tail_idx, int split, int bn) {
  return reinterpret_cast<float4*>(p.tail_ws) +
         (static_cast<long long>(tail_idx) * p.tail_splits + split) * (bn / 4) * BM;
}

// Waits that must not give up early because another thread failed: used only
// to let copies and MMAs already in flight finish before the CTA exits.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, DeviceStatus* st,
                                           int where) {
  if (mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return;
    if (globaltimer_ns() - t0 > kDrainLimitNs) {
      if (atomicCAS(&st->code, 0, kStatusTimeout) == 0) st->where = where;
      return;
    }
  }
}

// Eight consecutive halves row[col .. col+7] (zero outside [0, ncols) or when
// the row is out of range), with the widest load the address allows.
__device__ __forceinline__ uint4 load8_pred(const uint16_t* row, int col, int ncols, bool row_ok) {
  uint4 v = make_uint4(0u, 0u, 0u, 0u);
  if (!row_ok || col >= ncols) return v;
  const uint16_t* ptr = row + col;
  const uintptr_t a = reinterpret_cast<uintptr_t>(ptr);
  if (col + 8 <= ncols) {
    if ((a & 15u) == 0) return __ldg(reinterpret_cast<const uint4*>(ptr));
    if ((a & 7u) == 0) {
      const uint2 x = __ldg(reinterpret_cast<const uint2*>(ptr));
      const uint2 y = __ldg(reinterpret_cast<const uint2*>(ptr) + 1);
      return make_uint4(x.x, x.y, y.x, y.y);
    }
    if ((a & 3u) == 0) {
      const uint32_t* q = reinterpret_cast<const uint32_t*>(ptr);
      return make_uint4(__ldg(q), __ldg(q + 1), __ldg(q + 2), __ldg(q + 3));
    }
  }
  uint32_t h[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    h[i] = (col + i < ncols) ? static_cast<uint32_t>(__ldg(ptr + i)) : 0u;
  v.x = h[0] | (h[1] << 16);
  v.y = h[2] | (h[3] << 16);
  v.z = h[4] | (h[5] << 16);
  v.w = h[6] | (h[7] << 16);
  return v;
}

__device__ __forceinline__ float2 half2_bits_to_float2(uint32_t bits) {
  __half2 h;
  memcpy(&h, &bits, 4);
  return __half22float2(h);
}

__device__ __forceinline__ uint32_t float2_to_half2_bits(float x, float y) {
  const __half2 h = __floats2half2_rn(x, y);
  uint32_t bits;
  memcpy(&bits, &h, 4);
  return bits;
}

// alpha*acc (+ beta*c) for 8 accumulator columns -> 8 packed halves.
__device__ __forceinline__ uint4 epilogue8(const uint32_t* acc, uint4 cbits, bool has_c,
                                           float alpha, float beta) {
  float c[8];
  if (has_c) {
    const float2 c0 = half2_bits_to_float2(cbits.x), c1 = half2_bits_to_float2(cbits.y);
    const float2 c2 = half2_bits_to_float2(cbits.z), c3 = half2_bits_to_float2(cbits.w);
    c[0] = c0.x; c[1] = c0.y; c[2] = c1.x; c[3] = c1.y;
    c[4] = c2.x; c[5] = c2.y; c[6] = c3.x; c[7] = c3.y;
  }
  float o[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float a = __uint_as_float(acc[i]);
    o[i] = has_c ? __fmaf_rn(alpha, a, beta * c[i]) : alpha * a;
  }
  return make_uint4(float2_to_half2_bits(o[0], o[1]), float2_to_half2_bits(o[2], o[3]),
                    float2_to_half2_bits(o[4], o[5]), float2_to_half2_bits(o[6], o[7]));
}

// alpha*acc (+ beta*c) for 4 accumulator columns -> 4 floats (16 bytes).
__device__ __forceinline__ uint4 epilogue4f(const uint32_t* acc, uint4 cbits, bool has_c,
                                            float alpha, float beta) {
  const float c[4] = {__uint_as_float(cbits.x), __uint_as_float(cbits.y), __uint_as_float(cbits.z),
                      __uint_as_float(cbits.w)};
  float o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float a = __uint_as_float(acc[i]);
    o[i] = has_c ? __fmaf_rn(alpha, a, beta * c[i]) : alpha * a;
  }
  return make_uint4(__float_as_uint(o[0]), __float_as_uint(o[1]), __float_as_uint(o[2]),
                    __float_as_uint(o[3]));
}

// C values of one row for a 32-column sub-chunk (4 groups of 8 halves), read
// straight into registers with streaming loads; zero outside the matrix.  Used
// by the TMA epilogue, where rows of C are 16-byte aligned and N % 8 == 0.
__device__ __forceinline__ void load_c_sub(const TcArgs& p, int row, int col0, uint4 (&dst)[4]) {
  const bool rok = row < p.M;
  const uint4* src =
      reinterpret_cast<const uint4*>(p.C + static_cast<long long>(row) * p.ldc + col0);
#pragma unroll
  for (int g = 0; g < 4; ++g)
    dst[g] = (rok && col0 + 8 * g < p.N) ? __ldcs(src + g) : make_uint4(0u, 0u, 0u, 0u);
}

// Byte offset of 16-byte chunk c (0..3) of row r in a 64-byte-swizzled staging tile.
__device__ __forceinline__ uint32_t sw64_chunk(int r, int c) {
  return static_cast<uint32_t>(r * 64 + ((c ^ ((r >> 1) & 3)) << 4));
}

// Byte offset of column c (0..31) of row r in the same tile.
__device__ __forceinline__ uint32_t sw64_elem(int r, int c) {
  return sw64_chunk(r, c >> 3) + static_cast<uint32_t>((c & 7) << 1);
}

// The 32 registers of an in-flight tcgen05.ld become readable here; listing
// them as operands keeps every use after this wait.
__device__ __forceinline__ void tmem_wait_regs(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                 "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                 "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}

// Adds one tail slice's partial sums for a 32-column sub-chunk into acc.
__device__ __forceinline__ void add_partials(uint32_t (&acc)[32], const float4* src, bool assign) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 v = __ldcg(src + i * BM);
    if (assign) {
      acc[4 * i] = __float_as_uint(v.x);
      acc[4 * i + 1] = __float_as_uint(v.y);
      acc[4 * i + 2] = __float_as_uint(v.z);
      acc[4 * i + 3] = __float_as_uint(v.w);
    } else {
      acc[4 * i] = __float_as_uint(__uint_as_float(acc[4 * i]) + v.x);
      acc[4 * i + 1] = __float_as_uint(__uint_as_float(acc[4 * i + 1]) + v.y);
      acc[4 * i + 2] = __float_as_uint(__uint_as_float(acc[4 * i + 2]) + v.z);
      acc[4 * i + 3] = __float_as_uint(__uint_as_float(acc[4 * i + 3]) + v.w);
    }
  }
}

template <int BN, int LOAD, int EPI, bool PAIR, int AM = 128, int MM = 128, int KPB = 1>
__global__ void __launch_bounds__(Roles<LOAD>::kThreads, 1)
    gemm_f16_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmC, const TcArgs p) {
  using R = Roles<LOAD>;
  using L = Smem<BN, EPI, PAIR, AM, KPB>;
  using Cfg = typename L::Cfg;
  constexpr bool kCs = L::kCs;
  constexpr int kAB = Cfg::kAStageBytes;   // A bytes per stage
  static_assert(AM == 128 || LOAD == kLoadTma, "skinny stages take TMA loads");
  static_assert(KPB == 1 || LOAD == kLoadTma, "two k-blocks per stage take TMA loads");
  constexpr int S = Cfg::kStages;
  static_assert(!PAIR || (LOAD == kLoadTma && EPI != kEpiPartial), "pair configuration");
  // MM = 64: 64-row tiles (tcgen05.mma with M = 64), whole-K units only, TMA
  // loads of 64 rows of A and the TMA epilogue
  static_assert(MM == 128 || (MM == 64 && AM == 64 && !PAIR && EPI == kEpiTma), "64-row tiles");
  // Units are handed out per CTA, or per CTA pair (cluster of 2).
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  const int worker = PAIR ? static_cast<int>(cluster_id_x()) : static_cast<int>(blockIdx.x);
  const int nworkers = PAIR ? static_cast<int>(cluster_count_x()) : static_cast<int>(gridDim.x);
  const int bm_tile = PAIR ? 2 * BM : MM;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - raw_addr);

  const int warp = warp_id_uniform();
  const int lane = static_cast<int>(lane_id());
  const uint32_t bars = base + L::kBarOff;
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (S + s); };
  auto accf_bar = [&](uint32_t b) { return bars + 8u * (2 * S + b); };
  auto acce_bar = [&](uint32_t b) { return bars + 8u * (2 * S + 2 + b); };
  const uint32_t done_bar = bars + 8u * (2 * S + 4);
  const uint32_t tmem_free_bar = bars + 8u * (2 * S + 5);   // epilogue warps done with TMEM
  // C sub-tile landed in staging tile b of epilogue warp w
  auto cfull_bar = [&](int w, int b) { return bars + 8u * (2 * S + 6 + L::kBufs * w + b); };
  auto stage_a = [&](int s) { return base + static_cast<uint32_t>(s * Cfg::kStageBytes); };
  auto stage_b = [&](int s) { return stage_a(s) + kAB; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), LOAD == kLoadTma ? 1u : 128u);
      mbar_init(empty_bar(s), 1u);
    }
    for (uint32_t b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1u);
      mbar_init(acce_bar(b), static_cast<uint32_t>((PAIR ? 2 : 1) * R::kEpiWarps));
    }
    mbar_init(done_bar, 1u);
    mbar_init(tmem_free_bar, static_cast<uint32_t>(R::kEpiWarps));
    for (int w = 0; w < 8; ++w)
      for (int b = 0; b < L::kBufs; ++b) mbar_init(cfull_bar(w, b), 1u);
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == R::kMmaWarp) {
    if (PAIR) {
      tmem_alloc_pair(base + L::kTmemPtrOff, Cfg::kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(base + L::kTmemPtrOff, Cfg::kTmemCols);
      tmem_relinquish();
    }
  }
  if (LOAD == kLoadTma && warp == 0 && lane == 0) {
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
  }
  if ((EPI == kEpiTma || EPI == kEpiF32Tma) && warp == R::kEpiWarp0 && lane == 0)
    prefetch_tensormap(&tmC);
  tc_fence_before();
  __syncwarp();
  if (PAIR)
    cluster_sync();   // the peer's barriers are initialised before any remote use
  else
    __syncthreads();
  tc_fence_after();
  // everything above touched only this CTA's shared and tensor memory; from
  // here on global memory is read and written, once a pre-pass launched just
  // before this kernel has completed
  griddep_wait();
  // a copy-back kernel launched after this one may be scheduled now (it waits
  // for this kernel's completion before reading anything this kernel writes)
  griddep_launch_dependents();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(base_ptr + L::kTmemPtrOff);

  const unsigned long long limit = p.wait_limit_ns;
  DeviceStatus* const st = p.status;

  if (warp < R::kProdWarps) {
    // ------------------------------------------------------------ producer
    if (LOAD == kLoadTma) {
      if (lane == 0) {
        int stage = 0;
        uint32_t phase = 0, issued = 0;
        bool ok = true;
        const uint64_t evict_first = l2_evict_first_policy();
        UnitCursor cur = first_unit(p, worker);
        Unit t;
        while (ok && next_unit(p, cur, worker, nworkers, BN, bm_tile, rank, t)) {
          for (int kb = t.kb0; kb < t.kb1; kb += KPB) {
            if (!wait_parity(empty_bar(stage), phase ^ 1u, limit, st, 1)) {
              ok = false;
              break;
            }
            // k-blocks of this stage (the unit's last stage may hold one)
            const int nk = KPB == 1 ? 1 : min(KPB, t.kb1 - kb);
            // B columns this CTA gives the MMA (a half-width unit needs half of
            // them), staged in whole 64-column boxes
            const int bcols = PAIR ? t.ncols / 2 : t.ncols;
            const uint32_t bytes =
                static_cast<uint32_t>(nk * (kAB + ((bcols + 63) / 64) * kBBlockBytes));
            if (PAIR) {
              // Both CTAs' bytes are counted on the leader's barrier; only the
              // leader arms it (for the pair's total), the peer's copies just
              // signal it.
              const uint32_t fb = map_to_cta(full_bar(stage), 0);
              if (leader) mbar_arrive_expect_tx(full_bar(stage), 2 * bytes);
              for (int j = 0; j < nk; ++j) {
                const uint32_t sa = stage_a(stage) + j * Cfg::kKbBytes, sb = sa + kAB;
                const int k0 = (kb + j) * BK;
                tma_load_2d_pair(sa, &tmA, fb, k0, t.m0);
#pragma unroll
                for (int c = 0; c < Cfg::kBStageCols / 64; ++c)
                  if (64 * c < bcols)
                    tma_load_2d_pair(sb + c * kBBlockBytes, &tmB, fb,
                                     t.n0 + static_cast<int>(rank) * bcols + 64 * c, k0);
              }
            } else {
              mbar_arrive_expect_tx(full_bar(stage), bytes);
              for (int j = 0; j < nk; ++j) {
                const uint32_t sa = stage_a(stage) + j * Cfg::kKbBytes, sb = sa + kAB;
                const int k0 = (kb + j) * BK;
                if (p.stream_a)
                  tma_load_2d_hint(sa, &tmA, full_bar(stage), k0, t.m0, evict_first);
                else
                  tma_load_2d(sa, &tmA, full_bar(stage), k0, t.m0);
#pragma unroll
                for (int c = 0; c < BN / 64; ++c)
                  if (64 * c < bcols) {
                    if (p.stream_b)
                      tma_load_2d_hint(sb + c * kBBlockBytes, &tmB, full_bar(stage),
                                       t.n0 + 64 * c, k0, evict_first);
                    else
                      tma_load_2d(sb + c * kBBlockBytes, &tmB, full_bar(stage), t.n0 + 64 * c,
                                  k0);
                  }
              }
            }
            ++issued;
            if (++stage == S) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
        // The last loads (at most one per stage) must land before the CTA exits.
        // With pairs the completion is counted in the leader, so wait instead for
        // the MMAs that consumed them (which also guarantees that every commit
        // the leader multicasts into this CTA's stage barriers has arrived).
        const uint32_t n = issued < static_cast<uint32_t>(S) ? issued : static_cast<uint32_t>(S);
        for (uint32_t i = issued - n; i < issued; ++i) {
          if (PAIR)
            drain_wait(empty_bar(static_cast<int>(i % S)), (i / S) & 1u, st, 15);
          else
            drain_wait(full_bar(static_cast<int>(i % S)), (i / S) & 1u, st, 11);
        }
      }
      __syncwarp();
    } else {
      const int tp = static_cast<int>(threadIdx.x);  // 0..127
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      UnitCursor cur = first_unit(p, worker);
      Unit t;
      while (ok && next_unit(p, cur, worker, nworkers, BN, bm_tile, rank, t)) {
        for (int kb = t.kb0; kb < t.kb1; ++kb) {
          if (!wait_parity(empty_bar(stage), phase ^ 1u, limit, st, 2)) {
            ok = false;
            break;
          }
          uint8_t* const sa = base_ptr + stage * Cfg::kStageBytes;
          uint8_t* const sb = sa + kAB;
          const int k0 = kb * BK;
          // A: 128 rows x 8 chunks of 8 halves.
#pragma unroll 4
          for (int i = 0; i < 8; ++i) {
            const int id = tp + 128 * i;
            const int r = id >> 3, kc = id & 7;
            const int row = t.m0 + r;
            const uint4 v = load8_pred(p.A + static_cast<long long>(row) * p.lda, k0 + 8 * kc, p.K,
                                       row < p.M);
            *reinterpret_cast<uint4*>(sa + r * 128 + ((kc ^ (r & 7)) << 4)) = v;
          }
          // B: 64 k-rows x BN/8 chunks of 8 halves.
          constexpr int kBChunks = BK * BN / 8;
#pragma unroll 4
          for (int i = 0; i < kBChunks / 128; ++i) {
            const int id = tp + 128 * i;
            const int k = id / (BN / 8), nc = id % (BN / 8);
            const int krow = k0 + k;
            const uint4 v = load8_pred(p.B + static_cast<long long>(krow) * p.ldb, t.n0 + 8 * nc,
                                       p.N, krow < p.K);
            *reinterpret_cast<uint4*>(sb + (nc >> 3) * kBBlockBytes + k * 128 +
                                      (((nc & 7) ^ (k & 7)) << 4)) = v;
          }
          fence_proxy_async_smem();   // generic-proxy writes -> tensor-core reads
          mbar_arrive(full_bar(stage));
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp == R::kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && leader) {
      constexpr uint32_t idesc_full = make_idesc(0u, PAIR ? 2 * BM : MM, BN, 0u, 1u);
      constexpr uint32_t idesc_half = make_idesc(0u, PAIR ? 2 * BM : MM, BN / 2, 0u, 1u);
      int stage = 0;
      uint32_t phase = 0, local = 0;
      bool ok = true;
      UnitCursor cur = first_unit(p, worker);
      Unit t;
      while (ok && next_unit(p, cur, worker, nworkers, BN, bm_tile, rank, t)) {
        const uint32_t buf = local & 1u, use = local >> 1;
        if (!wait_parity(acce_bar(buf), (use & 1u) ^ 1u, limit, st, 3)) break;
        tc_fence_after();
        const uint32_t idesc = t.ncols == BN ? idesc_full : idesc_half;
        const uint32_t d_tmem = tmem_base + buf * Cfg::kAccStride;
        for (int kb = t.kb0; kb < t.kb1; kb += KPB) {
          if (!wait_parity(full_bar(stage), phase, limit, st, 4)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int nk = KPB == 1 ? 1 : min(KPB, t.kb1 - kb);
          for (int j = 0; j < nk; ++j) {
            const uint32_t a0 = stage_a(stage) + j * Cfg::kKbBytes, b0 = a0 + kAB;
#pragma unroll
            for (int kk = 0; kk < BK / kUmmaK; ++kk) {
              const uint64_t ad = smem_desc_sw128(a0 + kk * (kUmmaK * 2), 16u, 1024u);
              const uint64_t bd = smem_desc_sw128(b0 + kk * (kUmmaK * 128), kBBlockBytes, 1024u);
              const uint32_t acc = (kb > t.kb0 || j > 0 || kk > 0) ? 1u : 0u;
              if (PAIR)
                mma_f16_ss_pair(d_tmem, ad, bd, idesc, acc);
              else
                mma_f16_ss(d_tmem, ad, bd, idesc, acc);
            }
          }
          // frees the stage (in both CTAs of a pair) once these MMAs finish
          if (PAIR)
            mma_commit_pair_multicast(empty_bar(stage), 3);
          else
            mma_commit(empty_bar(stage));
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        // accumulator ready for the epilogue(s)
        if (PAIR)
          mma_commit_pair_multicast(accf_bar(buf), 3);
        else
          mma_commit(accf_bar(buf));
        ++local;
      }
      // Every MMA issued above must complete before TMEM is released.
      if (PAIR)
        mma_commit_pair_multicast(done_bar, 3);
      else
        mma_commit(done_bar);
      drain_wait(done_bar, 0u, st, 12);
      if (PAIR) {
        // The last accumulator releases (from both CTAs) must have arrived
        // before this CTA may leave.
        const uint32_t first = local > 2u ? local - 2u : 0u;
        for (uint32_t j = first; j < local; ++j) drain_wait(acce_bar(j & 1u), (j >> 1) & 1u, st, 16);
      }
    } else if (PAIR && lane == 0) {
      drain_wait(done_bar, 0u, st, 12);   // the leader's MMAs also wrote this CTA's TMEM
    }
    // Every epilogue warp of this CTA must be done reading TMEM before it is released.
    if (lane == 0) drain_wait(tmem_free_bar, 0u, st, 14);
    __syncwarp();
    tc_fence_after();
    if (PAIR)
      tmem_dealloc_pair(tmem_base, Cfg::kTmemCols);
    else
      tmem_dealloc(tmem_base, Cfg::kTmemCols);
  } else {
    // ------------------------------------------------------------ epilogue
    // The 32-column sub-chunks of a unit are shared out between the kParts
    // warps of each TMEM lane quadrant: part h takes chunks [lo, hi) (the first
    // part takes the odd one of a 224-wide tile).  kSubs: most chunks of a warp.
    constexpr int kParts = R::kEpiWarps / 4;
    constexpr int kSubs = (BN / kSubCols + kParts - 1) / kParts;
    const int ew = warp - R::kEpiWarp0;   // 0 .. kEpiWarps-1
    const int q = warp & 3;               // TMEM lane quadrant -> rows 32q .. 32q+31
    // Tile rows per lane quadrant: 32 (row 32q + l in TMEM lane 32q + l), or
    // 16 on 64-row tiles, whose M = 64 accumulator holds row 16q + l in lane
    // 32q + l for l < 16 only (the other lanes are not written; their threads
    // take a row past M, so that they neither read nor write C).
    constexpr int kQRows = MM / 4;
    const int h = ew >> 2;                // column part of the tile
    // first column (within the unit) and number of sub-chunks of this warp
    auto warp_cols = [&](const Unit& u, int& first, int& nchunks) {
      const int nch = u.ncols / kSubCols;
      const int lo = (h * nch + kParts - 1) / kParts;
      const int hi = ((h + 1) * nch + kParts - 1) / kParts;
      first = lo * kSubCols;
      nchunks = hi - lo;
    };
    const bool has_c = p.beta != 0.0f;
    const uint32_t sbuf0 = base + L::kEpiOff + ew * L::kWarpEpiBytes;
    uint8_t* const sptr0 = base_ptr + L::kEpiOff + ew * L::kWarpEpiBytes;
    uint32_t local = 0, nstore = 0;
    // kCs: C sub-tiles (32 rows x 64 bytes: 32 halves or 16 floats) are read
    // by TMA into the staging tiles, where the result replaces them and is
    // stored by TMA.  The first kBufs sub-tiles of a unit are requested while
    // its main loop runs; sub-tile j + kBufs as soon as the store of sub-tile
    // j has read its tile.  c_loads[b] counts the loads into tile b (the
    // parity of its barrier).
    constexpr int NB = L::kBufs;
    constexpr int kTc = (EPI == kEpiF32Tma) ? 16 : 32;   // columns per staging sub-tile
    constexpr int kTpc = kSubCols / kTc;                  // staging sub-tiles per TMEM chunk
    uint32_t c_loads[NB];
    bool c_pending[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      c_loads[b] = 0u;
      c_pending[b] = false;
    }
    auto load_c_sub_tma = [&](int b, int col, int r0) {
      if (lane == 0) {
        bulk_wait_group_read<0>();   // stores issued from the staging tiles have read them
        mbar_arrive_expect_tx(cfull_bar(ew, b), static_cast<uint32_t>(kEpiBufBytes));
        tma_load_2d(sbuf0 + b * kEpiBufBytes, &tmC, cfull_bar(ew, b), col, r0);
      }
      ++c_loads[b];
      c_pending[b] = true;
    };
    auto wait_c_sub = [&](int b) -> bool {
      if (!c_pending[b]) return true;
      // on failure the load stays pending and is drained before the CTA exits
      if (!wait_parity(cfull_bar(ew, b), (c_loads[b] - 1u) & 1u, limit, st, 9)) return false;
      c_pending[b] = false;
      return true;
    };
    auto load_c_head = [&](const Unit& u2) {   // the first NB sub-tiles of a unit
      int first2, nch2;
      warp_cols(u2, first2, nch2);
      const int wc = nch2 * kSubCols;
      const int r0 = u2.m0 + kQRows * q, cw = u2.n0 + first2;
      if (!has_c || r0 >= p.M || cw >= p.N) return;
#pragma unroll
      for (int j = 0; j < NB; ++j)
        if (kTc * j < wc && cw + kTc * j < p.N) load_c_sub_tma(j, cw + kTc * j, r0);
    };
    UnitCursor cur = first_unit(p, worker);
    Unit t, tn;
    bool have = next_unit(p, cur, worker, nworkers, BN, bm_tile, rank, t);
    if (kCs && have) load_c_head(t);
    while (have) {
      // kCs looks one unit ahead (its C tile is loaded during the next main loop)
      const bool have_next = kCs && next_unit(p, cur, worker, nworkers, BN, bm_tile, rank, tn);
      const uint32_t buf = local & 1u, use = local >> 1;
      const int row0 = t.m0 + kQRows * q;
      // tail bookkeeping is per CTA: the rows of one CTA of a pair form their own part
      const int tail_part = PAIR ? 2 * t.tail_idx + static_cast<int>(rank) : t.tail_idx;
      int wcol0, nsub;                              // this warp's columns of the unit
      warp_cols(t, wcol0, nsub);
      const int wcols = nsub * kSubCols;
      const int colw = t.n0 + wcol0;                // first column of this warp
      const int row = lane < kQRows ? row0 + lane : p.M;   // this thread's row
      bool finish = nsub > 0 && row0 < p.M && colw < p.N;   // this warp has outputs to produce
      if (EPI != kEpiPartial && has_c && finish && row < p.M) {
        // While this unit's main loop runs, bring this row's part of C into
        // L2, so that the epilogue's reads of C wait on L2 and not on DRAM.
        const int ncols = min(wcols, p.N - colw);
        const long long e0 = static_cast<long long>(row) * p.ldc + colw;
        constexpr bool kF32C = EPI == kEpiF32 || EPI == kEpiF32Tma;
        const uintptr_t c0 = kF32C ? reinterpret_cast<uintptr_t>(p.Cf + e0)
                                            : reinterpret_cast<uintptr_t>(p.C + e0);
        const uintptr_t first = c0 & ~static_cast<uintptr_t>(127);
        const uintptr_t last = c0 + static_cast<uintptr_t>(ncols) * (kF32C ? 4 : 2) - 1;
        for (uintptr_t a = first; a <= last; a += 128) prefetch_l2(reinterpret_cast<const void*>(a));
      }
      // A tile's last slice reads the others' partial sums back: bring them
      // into L2 while its main loop runs (its lane's column quad, 512 bytes
      // per warp and slice).
      if (EPI != kEpiPartial && t.tail && t.split == t.npieces - 1 && finish &&
          lane < wcols / 4) {
        for (int s2 = 0; s2 + 1 < t.npieces; ++s2) {
          const float4* part =
              tail_partials(p, tail_part, s2, BN) + (wcol0 / 4 + lane) * BM + 32 * q;
#pragma unroll
          for (int l = 0; l < 4; ++l) prefetch_l2(part + 8 * l);
        }
      }
      // C of the first sub-chunk is requested before the accumulator is ready.
      uint4 c_next[4];
      if (!kCs && EPI == kEpiTma && has_c && finish && !t.tail) load_c_sub(p, row, colw, c_next);
      if (!wait_parity(accf_bar(buf), use & 1u, limit, st, 5)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(32 * q) << 16) +
                             buf * Cfg::kAccStride + static_cast<uint32_t>(wcol0);

      if (EPI != kEpiPartial && t.tail && finish) {
        unsigned long long* cnt = p.tail_counters + tail_part * kTailCounters + h * 4 + q;
        // If every other slice of the tile has already published, this one
        // finishes the tile straight from TMEM and need not publish.
        uint32_t before = 0;
        if (lane == 0) {
          const unsigned long long c0 = ld_acquire_gpu_u64(cnt);
          before = (static_cast<unsigned int>(c0 >> 32) == p.epoch)
                       ? static_cast<uint32_t>(c0 & 0xFFFFFFFFull)
                       : 0u;
        }
        before = __shfl_sync(0xffffffffu, before, 0);
        if (before + 1u == static_cast<uint32_t>(t.npieces)) {
          __threadfence();
          if (!kCs && EPI == kEpiTma && has_c) load_c_sub(p, row, colw, c_next);
        } else {
          // Publish this slice's partial sums, then count the slice in; the last
          // slice to arrive finishes the tile.
          float4* mine = tail_partials(p, tail_part, t.split, BN) + 32 * q + lane;
          for (int k = 0; k < kSubs; ++k) {
            if (k >= nsub || colw + kSubCols * k >= p.N) break;
            uint32_t acc[32];
            tmem_ld_32x32b_x32(tbase + kSubCols * k, acc);
            tmem_wait_regs(acc);
            const int cq0 = (wcol0 + kSubCols * k) / 4;
#pragma unroll
            for (int i = 0; i < 8; ++i)
              __stcg(mine + (cq0 + i) * BM,
                     make_float4(__uint_as_float(acc[4 * i]), __uint_as_float(acc[4 * i + 1]),
                                 __uint_as_float(acc[4 * i + 2]), __uint_as_float(acc[4 * i + 3])));
          }
          __threadfence();
          __syncwarp();
          uint32_t arrived = 0;
          if (lane == 0) {
            unsigned long long cv = *reinterpret_cast<volatile unsigned long long*>(cnt);
            for (;;) {
              const unsigned long long next =
                  (static_cast<unsigned int>(cv >> 32) == p.epoch)
                      ? cv + 1ull
                      : ((static_cast<unsigned long long>(p.epoch) << 32) | 1ull);
              const unsigned long long prev = atomicCAS(cnt, cv, next);
              if (prev == cv) {
                arrived = static_cast<uint32_t>(next & 0xFFFFFFFFull);
                break;
              }
              cv = prev;
            }
          }
          arrived = __shfl_sync(0xffffffffu, arrived, 0);
          finish = arrived == static_cast<uint32_t>(t.npieces);
          if (finish) {
            __threadfence();
            if (!kCs && EPI == kEpiTma && has_c) load_c_sub(p, row, colw, c_next);
          }
        }
        // Every other piece of the tile has counted in: the finisher clears the
        // counter, so the next launch starts from zero whatever its epoch (a
        // replayed CUDA graph repeats the captured epoch).
        if (finish && lane == 0) *reinterpret_cast<volatile unsigned long long*>(cnt) = 0ull;
      }

      if (kCs && !finish) {   // unused C retired
        bool ok_c = true;
#pragma unroll
        for (int b = 0; b < NB; ++b) ok_c = wait_c_sub(b) && ok_c;
        if (!ok_c) break;
      }
      if (finish) {
        uint32_t acc_a[32], acc_b[32];
        if (!t.tail) {
          tmem_ld_32x32b_x32(tbase, acc_a);
          tmem_wait_regs(acc_a);
        }
#pragma unroll
        for (int k = 0; k < kSubs; ++k) {
          uint32_t(&cur)[32] = (k & 1) ? acc_b : acc_a;
          uint32_t(&nxt)[32] = (k & 1) ? acc_a : acc_b;
          const int col0 = colw + kSubCols * k;
          if (k >= nsub || col0 >= p.N) break;
          const bool more = k + 1 < nsub && col0 + kSubCols < p.N;
          if (more && !t.tail) tmem_ld_32x32b_x32(tbase + kSubCols * (k + 1), nxt);   // in flight
          uint4 c_cur[4];
          if (!kCs && EPI == kEpiTma) {
#pragma unroll
            for (int g = 0; g < 4; ++g) c_cur[g] = c_next[g];
            if (has_c && more) load_c_sub(p, row, col0 + kSubCols, c_next);
          }
          if (EPI != kEpiPartial && t.tail) {
            // cur := sum of every slice's partial sums in slice order; this
            // slice's own term is still in TMEM (bit-identical to what it
            // published), so only the other slices are read back.
            const int cq0 = (wcol0 + kSubCols * k) / 4;
            const float4* part = tail_partials(p, tail_part, 0, BN) + 32 * q + lane + cq0 * BM;
            const long long slice = static_cast<long long>(BN / 4) * BM;
            if (t.split == 0) {
              tmem_ld_32x32b_x32(tbase + kSubCols * k, cur);
              tmem_wait_regs(cur);
            } else {
              add_partials(cur, part, true);
            }
            for (int s2 = 1; s2 < t.npieces; ++s2) {
              if (s2 == t.split) {
                tmem_ld_32x32b_x32(tbase + kSubCols * k, nxt);
                tmem_wait_regs(nxt);
#pragma unroll
                for (int i = 0; i < 32; ++i)
                  cur[i] = __float_as_uint(__uint_as_float(cur[i]) + __uint_as_float(nxt[i]));
              } else {
                add_partials(cur, part + s2 * slice, false);
              }
            }
          }
          if (EPI == kEpiPartial) {
            if (row < p.M) {
              float* wrow = p.ws + (static_cast<long long>(t.split) * p.M + row) * p.ws_ld;
#pragma unroll
              for (int c = 0; c < kSubCols; c += 4) {
                const int col = col0 + c;
                const float4 v = make_float4(__uint_as_float(cur[c]), __uint_as_float(cur[c + 1]),
                                             __uint_as_float(cur[c + 2]),
                                             __uint_as_float(cur[c + 3]));
                if (col + 4 <= p.N) {
                  *reinterpret_cast<float4*>(wrow + col) = v;
                } else {
                  if (col < p.N) wrow[col] = v.x;
                  if (col + 1 < p.N) wrow[col + 1] = v.y;
                  if (col + 2 < p.N) wrow[col + 2] = v.z;
                }
              }
            }
          } else if (EPI == kEpiF32) {
            // fp32 C straight from registers: each thread writes 32 consecutive
            // floats of its row (eight 16-byte pieces)
            if (row < p.M) {
              float* crow = p.Cf + static_cast<long long>(row) * p.ldc;
              if (p.vec_c && col0 + kSubCols <= p.N) {
                float4 cv[8];
#pragma unroll
                for (int g = 0; g < 8; ++g)
                  cv[g] = has_c ? __ldcs(reinterpret_cast<const float4*>(crow + col0) + g)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int g = 0; g < 8; ++g) {
                  const float c4[4] = {cv[g].x, cv[g].y, cv[g].z, cv[g].w};
                  float o[4];
#pragma unroll
                  for (int j = 0; j < 4; ++j) {
                    const float a = __uint_as_float(cur[4 * g + j]);
                    o[j] = has_c ? __fmaf_rn(p.alpha, a, p.beta * c4[j]) : p.alpha * a;
                  }
                  __stcs(reinterpret_cast<float4*>(crow + col0) + g,
                         make_float4(o[0], o[1], o[2], o[3]));
                }
              } else {
#pragma unroll
                for (int j = 0; j < kSubCols; ++j) {
                  const int col = col0 + j;
                  if (col < p.N) {
                    const float a = __uint_as_float(cur[j]);
                    crow[col] = has_c ? __fmaf_rn(p.alpha, a, p.beta * crow[col]) : p.alpha * a;
                  }
                }
              }
            }
          } else if (kCs) {
            // staging sub-tile j in tile j % NB -> result in place -> TMA store
            bool c_ok = true;
#pragma unroll
            for (int e = 0; e < kTpc; ++e) {
              const int j = k * kTpc + e;
              const int colt = col0 + e * kTc;
              if (colt >= p.N) break;
              const int b = j % NB;
              uint8_t* const sptr = sptr0 + b * kEpiBufBytes;
              if (has_c) {
                if (!wait_c_sub(b)) {
                  c_ok = false;
                  break;
                }
              } else {
                // the store issued from this tile NB sub-tiles ago must have read it
                if (lane == 0) bulk_wait_group_read<NB - 1>();
                __syncwarp();
              }
#pragma unroll
              for (int g = 0; g < 4; ++g) {
                uint8_t* const ep = sptr + sw64_chunk(lane, g);
                const uint4 cv =
                    has_c ? *reinterpret_cast<const uint4*>(ep) : make_uint4(0u, 0u, 0u, 0u);
                *reinterpret_cast<uint4*>(ep) =
                    (EPI == kEpiF32Tma)
                        ? epilogue4f(cur + e * kTc + 4 * g, cv, has_c, p.alpha, p.beta)
                        : epilogue8(cur + 8 * g, cv, has_c, p.alpha, p.beta);
              }
              fence_proxy_async_smem();   // generic writes -> TMA store reads
              __syncwarp();
              if (lane == 0) {
                tma_store_2d(&tmC, sbuf0 + b * kEpiBufBytes, colt, row0);
                bulk_commit_group();
              }
              if (has_c && j + NB < nsub * kTpc && colt + NB * kTc < p.N)
                load_c_sub_tma(b, colt + NB * kTc, row0);
            }
            if (!c_ok) break;
          } else if (EPI == kEpiTma) {
            const uint32_t b = nstore & 1u;
            const uint32_t sbuf = sbuf0 + b * kEpiBufBytes;
            uint8_t* const sptr = sptr0 + b * kEpiBufBytes;
            // the store issued from this buffer two sub-chunks ago must have read it
            if (lane == 0) bulk_wait_group_read<1>();
            __syncwarp();
#pragma unroll
            for (int g = 0; g < 4; ++g)
              *reinterpret_cast<uint4*>(sptr + sw64_chunk(lane, g)) =
                  epilogue8(cur + 8 * g, c_cur[g], has_c, p.alpha, p.beta);
            fence_proxy_async_smem();   // generic writes -> TMA store reads
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmC, sbuf, col0, row0);
              bulk_commit_group();
            }
            ++nstore;
          } else {  // kEpiManual: C through shared memory with predicated accesses
            uint8_t* const sptr = sptr0;
            const int col = col0 + lane;   // this lane's column in the row-wise passes
            const bool col_ok = col < p.N;
            const uint16_t* __restrict__ cbase = p.C + static_cast<long long>(row0) * p.ldc + col;
            if (has_c) {
              // all 32 loads are issued before any is written to shared memory
              uint16_t v[32];
#pragma unroll
              for (int r = 0; r < 32; ++r)
                v[r] = (row0 + r < p.M && col_ok) ? __ldg(cbase + static_cast<long long>(r) * p.ldc)
                                                  : static_cast<uint16_t>(0);
#pragma unroll
              for (int r = 0; r < 32; ++r)
                *reinterpret_cast<uint16_t*>(sptr + sw64_elem(r, lane)) = v[r];
              __syncwarp();
            }
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              const uint32_t off = sw64_chunk(lane, g);
              const uint4 cv = has_c ? *reinterpret_cast<const uint4*>(sptr + off)
                                     : make_uint4(0u, 0u, 0u, 0u);
              *reinterpret_cast<uint4*>(sptr + off) =
                  epilogue8(cur + 8 * g, cv, has_c, p.alpha, p.beta);
            }
            __syncwarp();
            uint16_t o[32];
#pragma unroll
            for (int r = 0; r < 32; ++r)
              o[r] = *reinterpret_cast<const uint16_t*>(sptr + sw64_elem(r, lane));
            uint16_t* const cout = p.C + static_cast<long long>(row0) * p.ldc + col;
#pragma unroll
            for (int r = 0; r < 32; ++r)
              if (row0 + r < p.M && col_ok) cout[static_cast<long long>(r) * p.ldc] = o[r];
            __syncwarp();
          }
          if (more && !t.tail) tmem_wait_regs(nxt);
        }
      }
      tc_fence_before();
      __syncwarp();
      // the accumulator may be overwritten (with pairs: counted on the leader)
      if (lane == 0) {
        if (PAIR)
          mbar_arrive_cluster(map_to_cta(acce_bar(buf), 0));
        else
          mbar_arrive(acce_bar(buf));
      }
      ++local;
      if (kCs) {
        if (have_next) load_c_head(tn);
        t = tn;
        have = have_next;
      } else {
        have = next_unit(p, cur, worker, nworkers, BN, bm_tile, rank, t);
      }
    }
    // C loads still in flight (a wait above gave up) must land before exit
    for (int b = 0; b < NB; ++b)
      if (kCs && c_pending[b] && lane == 0)
        drain_wait(cfull_bar(ew, b), (c_loads[b] - 1u) & 1u, st, 17);
    if ((EPI == kEpiTma || kCs) && lane == 0) bulk_wait_group<0>();   // stores done reading smem
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(tmem_free_bar);
  }
  if (PAIR) {
    // Neither CTA of a pair leaves while the other may still touch its shared
    // memory (remote barrier arrivals, multicast commits).
    __syncwarp();
    cluster_sync();
  }
  // No CTA-wide barrier at the end: every role has already waited for its own
  // asynchronous work (TMA loads, MMAs, TMA stores), and TMEM is released by
  // the MMA warp only after all epilogue warps have signalled tmem_free.
}

template <int BN, int LOAD, int EPI, bool PAIR, int AM = 128, int MM = 128, int KPB = 1>
cudaError_t configure(int dev) {
  using L = Smem<BN, EPI, PAIR, AM, KPB>;
  static bool configured[64] = {};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(gemm_f16_tc_kernel<BN, LOAD, EPI, PAIR, AM, MM, KPB>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               L::kAlloc);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  return cudaSuccess;
}

template <int BN, int LOAD, int EPI, bool PAIR, int AM = 128, int MM = 128, int KPB = 1>
cudaError_t launch_one(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                       const TcArgs& args, int grid, cudaStream_t stream) {
  using L = Smem<BN, EPI, PAIR, AM, KPB>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = configure<BN, LOAD, EPI, PAIR, AM, MM, KPB>(dev)) != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(Roles<LOAD>::kThreads, 1, 1);
  cfg.dynamicSmemBytes = L::kAlloc;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  unsigned int nattr = 0;
  if (PAIR) {
    attr[nattr].id = cudaLaunchAttributeClusterDimension;
    attr[nattr].val.clusterDim.x = 2;
    attr[nattr].val.clusterDim.y = 1;
    attr[nattr].val.clusterDim.z = 1;
    ++nattr;
  }
  if (args.pdl) {
    attr[nattr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[nattr].val.programmaticStreamSerializationAllowed = 1;
    ++nattr;
  }
  cfg.attrs = nattr ? attr : nullptr;
  cfg.numAttrs = nattr;
  e = cudaLaunchKernelEx(&cfg, gemm_f16_tc_kernel<BN, LOAD, EPI, PAIR, AM, MM, KPB>, tmA, tmB,
                         tmC, args);
  if (e != cudaSuccess) return e;
  return counted_launch(cudaGetLastError());
}

// Largest number of CTA pairs of this configuration that can be resident at
// once (pairs must sit in one GPC), cached per device.
template <int EPI>
int pair_max_clusters(int dev) {
  static int cached[64] = {};
  if (dev < 0 || dev >= 64) return 0;
  if (cached[dev] > 0) return cached[dev];
  using L = Smem<256, EPI, true>;
  if (configure<256, kLoadTma, EPI, true>(dev) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(Roles<kLoadTma>::kThreads, 1, 1);
  cfg.dynamicSmemBytes = L::kAlloc;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, gemm_f16_tc_kernel<256, kLoadTma, EPI, true>, &cfg) !=
      cudaSuccess)
    return 0;
  cached[dev] = n;
  return n;
}

}  // namespace
}  // namespace gb300
