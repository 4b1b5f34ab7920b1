// sgemm_split.cu -- fp32 SGEMM on the tensor cores as three products of split
// operands (3xTF32: tf32 parts; 3xFP16: scaled half parts).
//
// C := alpha*A*B + beta*C in fp32.  Each operand is split (by a pre-pass) into
// a tf32 "big" part (low 13 mantissa bits cleared) and a tf32 "small" part
// (the remainder, rounded to tf32), so that A = Ab + As and B = Bb + Bs up to
// about 2^-22 relative.  The product keeps the three largest terms,
//     A*B ~= Ab*Bb + Ab*Bs + As*Bb;
// the dropped As*Bs term is below 2^-20 of |A||B|.
//
// Accumulation.  The tensor core's fp32 accumulation does not round to
// nearest: summed over a long K in tensor memory, the result drifts toward
// zero by a bias that grows like K*|C| (measured: at K = 16384 it exceeds the
// fp32 error bound).  So the MMA accumulates only chunks of 128 along K (256
// for the 3xFP16 form below) into tensor memory, alternating between two
// buffers, and the epilogue warps add each chunk into fp32 registers with
// ordinary round-to-nearest adds; the result is then as accurate as the FFMA
// kernel's.
//
// Kernel: CTA pairs (clusters of 2) share tcgen05.mma.cta_group::2.kind::tf32
// with M = 256 (128 rows of A in each CTA) and N = 256 (each CTA stages 128 of
// the columns of B); per 16-deep k-block each CTA stages Ab, As (128 x 16) and
// Bb, Bs (128 columns x 16) by TMA into a 6-stage ring (32 KB per stage; three
// stages of 64 KB ran at the same speed), and the leader issues 3 MMAs per
// 8-deep K step.  Warp roles and barriers follow the fp16 tensor-core kernel;
// the 8 epilogue warps keep fp32 row sums in registers and write C through a
// small shared-memory tile each, so that stores cover whole 64-byte row
// pieces.  Both operands are K-major (the pre-pass stores the B parts
// transposed): 64-byte swizzle, 16 floats per row, SBO 512 B.
//
// Units: whole 256 x 256 tiles; the tiles of a last, partial wave as two K
// slices each, publisher first (the first slice a worker's first unit, the
// second a worker's last; see slice_of), or, with a short K, as two
// half-width units each; or, when few tiles meet a long K, equal K slices of
// every tile (whole accumulation chunks).  The fp32 partial sums of a tile's
// slices are added up in slice order by the slice that arrives last, before
// it writes C.
//
// 3xFP16 (the same kernel, F16 = true): the parts are halves instead of tf32
// values -- x * 2^e = h1 + h2 with e a power-of-two exponent per row of A and
// per column of B within each 256-deep K chunk that keeps the parts inside the
// half range (the same 11 + 11 significand bits as the tf32 split), written
// by the split pre-pass -- and
// the three products run as kind::f16 MMAs at twice the tf32 rate.  A k-block
// is then 32 deep (one 64-byte row of halves), B is staged N-major as 64-
// column blocks of 32 k-rows (128-byte swizzle, no transpose), chunks are 8
// k-blocks (256 deep: a 128-deep chunk left the fold of the chunks into
// registers, not the MMAs, setting the pace), and the
// epilogue undoes the scaling chunk by chunk (the exponents are per 256-deep K
// chunk; each chunk's sums are multiplied by 2^-(e_row + e_col) as they are
// folded into the registers, exactly).
#include "internal.h"
#include "ptx.cuh"

namespace gb300 {
namespace {

constexpr int BM = 128;                     // rows per CTA
constexpr int BN = 256;                     // pair tile width
constexpr int kRowBytes = 64;               // bytes of K per k-block row: 16 floats or 32 halves
constexpr int kATile = BM * kRowBytes;      // 8 KB per part (128 rows of 64 bytes)
constexpr int kBCols = BN / 2;              // B columns staged by each CTA
constexpr int kBTile = kBCols * kRowBytes;  // 8 KB per part
constexpr int kBBlock = 32 * 128;           // 3xFP16: one 64-column block of a B part (32 k-rows)
constexpr int kStageBytes = 2 * kATile + 2 * kBTile;
constexpr int kStages = 6;
constexpr int kEpiWarps = 8;
constexpr int kCols = BN / 2;               // accumulator columns per epilogue thread
constexpr int kChunkKb = kSplitChunkKb;     // k-blocks per TMEM chunk: 128 floats / 256 halves
constexpr int kThreads = (2 + kEpiWarps) * 32;
constexpr int kTmemCols = 2 * BN;
constexpr int kBarOff = kStages * kStageBytes;
constexpr int kNumBars = 2 * kStages + 2 + 2 + 1 + 1;   // full, empty, accf, acce, done, tmem_free
constexpr int kTmemPtrOff = kBarOff + kNumBars * 8;
// per epilogue warp a 32-row x 16-float staging tile that turns the row-owned
// sums into row-contiguous stores of C
constexpr int kEpiOff = (kTmemPtrOff + 16 + 127) / 128 * 128;
constexpr int kEpiTileF4 = 32 * 4;
// 3xFP16: per epilogue warp the exponents of its 128 columns (32 int4)
constexpr int kEpiExpOff = kEpiOff + kEpiWarps * kEpiTileF4 * 16;
constexpr int kSmemAlloc = kEpiExpOff + kEpiWarps * 32 * 16 + 1024;
constexpr unsigned long long kDrainLimitNs = 1000000000ull;
static_assert(kSmemAlloc <= 232448, "shared memory budget");
static_assert(kChunkKb * 32 == kF16x3ChunkK, "3xFP16 exponent chunks are the accumulation chunks");

__device__ __forceinline__ void drain(uint32_t bar, uint32_t parity, DeviceStatus* st, int where) {
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

__device__ __forceinline__ void tmem_wait_regs32(uint32_t (&r)[32]) {
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

// 32 lanes x 16 consecutive columns (the 3xFP16 fold: half the registers of
// the 32-column load, which leaves room for the chunk's exponents).
__device__ __forceinline__ void tmem_ld16_wait(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// Partial sums of one K slice for one epilogue warp: [32 column quads][32
// rows] of float4, so a warp's stores and loads are contiguous.
constexpr long long kSliceF4 = (kCols / 4) * 32;
constexpr int kSumQuads = 16;   // column quads the finisher sums at a time

// One K slice of a tile, for one epilogue warp (32 rows x 128 columns of its
// CTA's half of the tile, the row sums in `acc`): publishes the slice's
// partial sums and counts it in.  Returns true (warp-uniform) in the slice
// that arrives last, which then owns the tile's sum: `part` points at slice
// 0 of this warp's partial sums, the slices following at kSliceF4 apart; the
// finisher adds them in slice order, so the result does not depend on which
// slice finishes.  The finisher also clears the counter, so the next launch
// starts from zero whatever its epoch.
__device__ __forceinline__ bool publish_slice(const Tf32Args& p, int tile, int slice, int nslices,
                                              int rank, int ew, int lane,
                                              const float (&acc)[kCols], const float4*& part) {
  const long long slot = (static_cast<long long>(tile) * 2 + rank) * kEpiWarps + ew;
  unsigned long long* const cnt = p.counters + slot;
  float4* const mine = p.part_ws + (slot * nslices + slice) * kSliceF4 + lane;
#pragma unroll
  for (int g = 0; g < kCols / 4; ++g)
    __stcg(mine + g * 32, make_float4(acc[4 * g], acc[4 * g + 1], acc[4 * g + 2], acc[4 * g + 3]));
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
  if (arrived != static_cast<uint32_t>(nslices)) return false;
  __threadfence();
  if (lane == 0) *reinterpret_cast<volatile unsigned long long*>(cnt) = 0ull;
  part = p.part_ws + slot * nslices * kSliceF4 + lane;
  return true;
}

// Unit u's shared tile, if it is one K slice of a tile: the tile's index among
// the sliced tiles, the slice and the slices per tile (nslices = 1: a whole
// tile or half-width unit).  K slices of every tile (splits > 1): unit = tile
// * splits + slice.  Two-slice tail (tail_first): units [0, T) are the first
// slices of the tiles [0, T) (visiting order), [T, T + dp_tiles) whole tiles,
// then the second slices -- a first slice is a worker's first unit, a second
// slice its last, long after the first was published.
__device__ __forceinline__ void slice_of(const Tf32Args& p, int u, int& tile, int& slice,
                                         int& nslices) {
  tile = u;
  slice = 0;
  nslices = 1;
  if (p.splits > 1) {
    tile = u / p.splits;
    slice = u - tile * p.splits;
    nslices = p.splits;
  } else if (p.tail_first) {
    const int T = (p.num_units - p.dp_tiles) >> 1;
    if (u < T) {
      nslices = 2;
    } else if (u >= T + p.dp_tiles) {
      tile = u - T - p.dp_tiles;
      slice = 1;
      nslices = 2;
    }
  }
}


template <bool F16>
__global__ void __launch_bounds__(kThreads, 1)
    sgemm_split_kernel(const __grid_constant__ CUtensorMap tmAb,
                        const __grid_constant__ CUtensorMap tmAs,
                        const __grid_constant__ CUtensorMap tmBb,
                        const __grid_constant__ CUtensorMap tmBs,
                        const __grid_constant__ CUtensorMap tmBbh,
                        const __grid_constant__ CUtensorMap tmBsh, const Tf32Args p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - raw_addr);
  const int warp = warp_id_uniform();
  const int lane = static_cast<int>(lane_id());
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int worker = static_cast<int>(cluster_id_x());
  const int nworkers = static_cast<int>(cluster_count_x());

  const uint32_t bars = base + kBarOff;
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (kStages + s); };
  auto accf_bar = [&](uint32_t b) { return bars + 8u * (2 * kStages + b); };
  auto acce_bar = [&](uint32_t b) { return bars + 8u * (2 * kStages + 2 + b); };
  const uint32_t done_bar = bars + 8u * (2 * kStages + 4);
  const uint32_t tmem_free_bar = bars + 8u * (2 * kStages + 5);
  auto stage = [&](int s) { return base + static_cast<uint32_t>(s * kStageBytes); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1u);
      mbar_init(empty_bar(s), 1u);
    }
    for (uint32_t b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1u);
      mbar_init(acce_bar(b), 2u * kEpiWarps);
    }
    mbar_init(done_bar, 1u);
    mbar_init(tmem_free_bar, static_cast<uint32_t>(kEpiWarps));
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc_pair(base + kTmemPtrOff, kTmemCols);
    tmem_relinquish_pair();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmAb);
    prefetch_tensormap(&tmAs);
    prefetch_tensormap(&tmBb);
    prefetch_tensormap(&tmBs);
    prefetch_tensormap(&tmBbh);
    prefetch_tensormap(&tmBsh);
  }
  tc_fence_before();
  __syncwarp();
  cluster_sync();
  tc_fence_after();
  // global memory (the split operand parts, C) only after the split pre-pass,
  // which may still run when this kernel starts, has completed
  griddep_wait();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(base_ptr + kTmemPtrOff);
  const unsigned long long limit = p.wait_limit_ns;
  DeviceStatus* const st = p.status;

  // unit -> (m0 of this CTA, n0, columns, k-block range); groups of group_m
  // tile-rows share B in L2; units past dp_tiles are the two column halves of
  // a tile; with K slices a unit is one slice of a whole tile
  auto tile_of = [&](int u, int& m0, int& n0, int& ncols, int& kb0, int& kb1) {
    int tile = u, half = -1;
    kb0 = 0;
    kb1 = p.kb_total;
    if (p.splits > 1) {
      tile = u / p.splits;
      kb0 = (u - tile * p.splits) * p.kb_per_split;
      kb1 = min(kb0 + p.kb_per_split, p.kb_total);
    } else if (p.tail_first) {
      int slice, nslices;
      slice_of(p, u, tile, slice, nslices);
      if (nslices > 1) {
        kb0 = slice ? p.kb_per_split : 0;
        kb1 = slice ? p.kb_total : p.kb_per_split;
      }
    } else if (u >= p.dp_tiles) {
      tile = p.dp_tiles + ((u - p.dp_tiles) >> 1);
      half = (u - p.dp_tiles) & 1;
    }
    const int group = p.group_m * p.tiles_n;
    const int g = tile / group;
    const int first_m = g * p.group_m;
    const int gm = min(p.tiles_m - first_m, p.group_m);
    const int r = tile - g * group;
    m0 = (first_m + r % gm) * (2 * BM) + static_cast<int>(rank) * BM;
    n0 = (r / gm) * BN + (half > 0 ? BN / 2 : 0);
    ncols = half < 0 ? BN : BN / 2;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int s = 0;
      uint32_t phase = 0, issued = 0;
      bool ok = true;
      for (int u = worker; ok && u < p.num_units; u += nworkers) {
        int m0, n0, ncols, kb0, kb1;
        tile_of(u, m0, n0, ncols, kb0, kb1);
        // B rows (columns of B) this CTA stages: half of the unit's
        const int bcols = ncols / 2;
        const uint32_t bytes = static_cast<uint32_t>(2 * kATile + 2 * bcols * kRowBytes);
        const CUtensorMap* mb = bcols == kBCols ? &tmBb : &tmBbh;
        const CUtensorMap* ms = bcols == kBCols ? &tmBs : &tmBsh;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!wait_parity(empty_bar(s), phase ^ 1u, limit, st, 21)) {
            ok = false;
            break;
          }
          const uint32_t fb = map_to_cta(full_bar(s), 0);
          if (leader) mbar_arrive_expect_tx(full_bar(s), 2 * bytes);
          const uint32_t sa = stage(s);
          constexpr int kbk = F16 ? 32 : 16;   // elements per k-block
          tma_load_2d_pair(sa, &tmAb, fb, kb * kbk, m0);
          tma_load_2d_pair(sa + kATile, &tmAs, fb, kb * kbk, m0);
          const int nb = n0 + static_cast<int>(rank) * bcols;
          if (F16) {
            // B parts N-major: one 64-column block (32 k-rows) per box
            for (int c = 0; c < bcols / 64; ++c) {
              tma_load_2d_pair(sa + 2 * kATile + c * kBBlock, &tmBb, fb, nb + 64 * c, kb * kbk);
              tma_load_2d_pair(sa + 2 * kATile + kBTile + c * kBBlock, &tmBs, fb, nb + 64 * c,
                               kb * kbk);
            }
          } else {
            tma_load_2d_pair(sa + 2 * kATile, mb, fb, kb * kbk, nb);
            tma_load_2d_pair(sa + 2 * kATile + kBTile, ms, fb, kb * kbk, nb);
          }
          ++issued;
          if (++s == kStages) {
            s = 0;
            phase ^= 1u;
          }
        }
      }
      const uint32_t n = issued < static_cast<uint32_t>(kStages) ? issued : kStages;
      for (uint32_t i = issued - n; i < issued; ++i)
        drain(empty_bar(static_cast<int>(i % kStages)), (i / kStages) & 1u, st, 22);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader)
    // Chunks of kChunkKb k-blocks alternate between the two TMEM buffers; each
    // chunk starts a fresh accumulation and the epilogue folds it into its
    // fp32 register accumulators.
    if (lane == 0 && leader) {
      // tf32: both operands K-major; f16: B N-major
      constexpr uint32_t idesc_full = F16 ? make_idesc(0u, 2 * BM, BN, 0u, 1u)
                                          : make_idesc(2u, 2 * BM, BN, 0u, 0u);
      constexpr uint32_t idesc_half = F16 ? make_idesc(0u, 2 * BM, BN / 2, 0u, 1u)
                                          : make_idesc(2u, 2 * BM, BN / 2, 0u, 0u);
      constexpr int kChunk = kChunkKb;
      int s = 0;
      uint32_t phase = 0, chunk = 0;
      bool ok = true;
      for (int u = worker; ok && u < p.num_units; u += nworkers) {
        int m0, n0, ncols, kb0, kb1;
        tile_of(u, m0, n0, ncols, kb0, kb1);
        const uint32_t idesc = ncols == BN ? idesc_full : idesc_half;
        for (int kc = kb0; ok && kc < kb1; kc += kChunk, ++chunk) {
          const uint32_t buf = chunk & 1u, use = chunk >> 1;
          if (!wait_parity(acce_bar(buf), (use & 1u) ^ 1u, limit, st, 23)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem_base + buf * BN;
          const int kend = min(kc + kChunk, kb1);
          for (int kb = kc; kb < kend; ++kb) {
            if (!wait_parity(full_bar(s), phase, limit, st, 24)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a_big = stage(s), a_small = a_big + kATile;
            const uint32_t b_big = a_big + 2 * kATile, b_small = b_big + kBTile;
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {   // 2 MMA K steps per 64-byte k-block
              // K-major parts (64-byte swizzle, 8-row groups 512 bytes apart)
              // advance 32 bytes per step (8 floats or 16 halves); an N-major
              // B part (128-byte swizzle) advances 16 k-rows (2 KB)
              const uint64_t adb = smem_desc_sw64(a_big + kk * 32, 16u, 512u);
              const uint64_t ads = smem_desc_sw64(a_small + kk * 32, 16u, 512u);
              const uint64_t bdb = F16 ? smem_desc_sw128(b_big + kk * 2048, kBBlock, 1024u)
                                       : smem_desc_sw64(b_big + kk * 32, 16u, 512u);
              const uint64_t bds = F16 ? smem_desc_sw128(b_small + kk * 2048, kBBlock, 1024u)
                                       : smem_desc_sw64(b_small + kk * 32, 16u, 512u);
              // the two small terms first, then the big one
              if (F16) {
                mma_f16_ss_pair(d, ads, bdb, idesc, (kb > kc || kk > 0) ? 1u : 0u);
                mma_f16_ss_pair(d, adb, bds, idesc, 1u);
                mma_f16_ss_pair(d, adb, bdb, idesc, 1u);
              } else {
                mma_tf32_ss_pair(d, ads, bdb, idesc, (kb > kc || kk > 0) ? 1u : 0u);
                mma_tf32_ss_pair(d, adb, bds, idesc, 1u);
                mma_tf32_ss_pair(d, adb, bdb, idesc, 1u);
              }
            }
            mma_commit_pair_multicast(empty_bar(s), 3);
            if (++s == kStages) {
              s = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          mma_commit_pair_multicast(accf_bar(buf), 3);
        }
      }
      mma_commit_pair_multicast(done_bar, 3);
      drain(done_bar, 0u, st, 25);
      const uint32_t first = chunk > 2u ? chunk - 2u : 0u;
      for (uint32_t j = first; j < chunk; ++j) drain(acce_bar(j & 1u), (j >> 1) & 1u, st, 26);
    } else if (lane == 0) {
      drain(done_bar, 0u, st, 25);
    }
    if (lane == 0) drain(tmem_free_bar, 0u, st, 27);
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  } else {
    // ------------------------------------------------------------ epilogue
    // Warp (q, h) owns TMEM lanes 32q..32q+31 (rows) and columns h*128..+127;
    // each thread keeps its row's 128 sums in fp32 registers.
    const int ew = warp - 2;
    const int q = warp & 3;
    const int h = ew >> 2;
    const bool has_c = p.beta != 0.0f;
    uint32_t chunk = 0;
    bool ok = true;
    for (int u = worker; ok && u < p.num_units; u += nworkers) {
      int m0, n0, ncols, kb0, kb1;
      tile_of(u, m0, n0, ncols, kb0, kb1);
      const int wcols = ncols / 2;   // this warp's columns of the unit
      const int row0 = m0 + 32 * q;
      const int row = row0 + lane;
      const int colw = n0 + h * wcols;
      const bool active = row0 < p.M && colw < p.N;   // warp-uniform
      // 3xFP16: each chunk's sums leave the scaled domain as they are folded,
      // multiplied by 2^-(e_row + e_col) with the chunk's exponents: e_row
      // for the thread's row, and for the warp's columns 2^-e_col as float
      // bits to add to 2^-e_row's (-(e_col << 23); lane l holds columns
      // colw + 4l .. +3 in shared memory).  Both are read before the chunk's
      // accumulator is waited for.  When every e_row + e_col of the warp is
      // within +-126 the factor is one normal power of two and the fold one
      // fused multiply-add (exact product, one rounding, as the plain add);
      // otherwise two normal factors.
      int4* const e_col = reinterpret_cast<int4*>(base_ptr + kEpiExpOff) + ew * 32;
      float acc[kCols];
#pragma unroll
      for (int j = 0; j < kCols; ++j) acc[j] = 0.0f;
      for (int kc = kb0; kc < kb1; kc += kChunkKb, ++chunk) {
        const uint32_t buf = chunk & 1u, use = chunk >> 1;
        int e_row = 0, rbits = 0;
        bool fast = true;
        if (F16 && active) {
          const int ci = kc / kChunkKb;
          if (row < p.M) e_row = __ldg(p.ea + static_cast<long long>(row) * p.kchunks + ci);
          int4 ec = make_int4(0, 0, 0, 0);
          if (4 * lane < wcols && colw + 4 * lane < p.N)   // eb rows hold N + 4 entries or more
            ec = __ldg(reinterpret_cast<const int4*>(p.eb + ci * p.ldeb + colw + 4 * lane));
          const int lo = __reduce_min_sync(0xffffffffu, min(min(ec.x, ec.y), min(ec.z, ec.w))) +
                         __reduce_min_sync(0xffffffffu, e_row);
          const int hi = __reduce_max_sync(0xffffffffu, max(max(ec.x, ec.y), max(ec.z, ec.w))) +
                         __reduce_max_sync(0xffffffffu, e_row);
          fast = lo >= -126 && hi <= 126;
          rbits = (127 - e_row) << 23;
          e_col[lane] = make_int4(-(ec.x << 23), -(ec.y << 23), -(ec.z << 23), -(ec.w << 23));
          __syncwarp();
        }
        if (!wait_parity(accf_bar(buf), use & 1u, limit, st, 28)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (active) {
          const uint32_t tbase =
              tmem_base + (static_cast<uint32_t>(32 * q) << 16) + buf * BN + h * wcols;
#pragma unroll
          for (int k = 0; k < kCols / 32; ++k) {
            if (32 * k >= wcols) break;
            if (!F16) {
              uint32_t t[32];
              tmem_ld_32x32b_x32(tbase + 32 * k, t);
              tmem_wait_regs32(t);
#pragma unroll
              for (int j = 0; j < 32; ++j) acc[32 * k + j] += __uint_as_float(t[j]);
              continue;
            }
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {   // 16 columns at a time
              uint32_t t[16];
              tmem_ld16_wait(tbase + 32 * k + 16 * hh, t);
              if (fast) {
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                  const int4 cb = e_col[8 * k + 4 * hh + g];
                  const int b4[4] = {cb.x, cb.y, cb.z, cb.w};
#pragma unroll
                  for (int i = 0; i < 4; ++i) {
                    float& a = acc[32 * k + 16 * hh + 4 * g + i];
                    a = fmaf(__uint_as_float(t[4 * g + i]), __int_as_float(rbits + b4[i]), a);
                  }
                }
                continue;
              }
#pragma unroll
              for (int g = 0; g < 4; ++g) {
                const int4 cb = e_col[8 * k + 4 * hh + g];
                const int b4[4] = {cb.x, cb.y, cb.z, cb.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  // 2^-E as two normal powers of two: exact whenever the result
                  // is a normal float (an intermediate that leaves the range
                  // means the result does too)
                  const int E = e_row - (b4[i] >> 23);
                  const int e1 = max(-126, min(126, E));
                  const int e2 = max(-126, min(126, E - e1));
                  acc[32 * k + 16 * hh + 4 * g + i] += (__uint_as_float(t[4 * g + i]) *
                                                        __int_as_float((127 - e1) << 23)) *
                                                       __int_as_float((127 - e2) << 23);
                }
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(map_to_cta(acce_bar(buf), 0));
      }
      if (!ok || !active) continue;
      float* const crow = p.C + static_cast<long long>(row) * p.ldc;
      // C[row][colw + 4g ..] := alpha * v + beta * C (columns past N and rows
      // past M are not written)
      float4* const tile = reinterpret_cast<float4*>(base_ptr + kEpiOff) + ew * kEpiTileF4;
      auto store_quad = [&](int g, float4 v) {
        const int col = colw + 4 * g;
        if (row >= p.M || 4 * g >= wcols || col >= p.N) return;
        float o[4] = {v.x, v.y, v.z, v.w};
        if (p.vec_c && col + 4 <= p.N) {
          float4 c = make_float4(0.f, 0.f, 0.f, 0.f);
          if (has_c) c = __ldcs(reinterpret_cast<const float4*>(crow + col));
          const float cv[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
          for (int j = 0; j < 4; ++j)
            o[j] = has_c ? fmaf(p.alpha, o[j], p.beta * cv[j]) : p.alpha * o[j];
          __stcs(reinterpret_cast<float4*>(crow + col), make_float4(o[0], o[1], o[2], o[3]));
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (col + j < p.N)
              crow[col + j] = has_c ? fmaf(p.alpha, o[j], p.beta * crow[col + j]) : p.alpha * o[j];
        }
      };
      // Columns colw + 16j .. +15 (quads 4j .. 4j+3) through the staging tile:
      // lane r writes its row's four quads (slot q ^ ((r >> 1) & 3): eight
      // lanes fill 128 distinct bytes), then every store instruction covers 8
      // rows x 64 contiguous bytes of C.  Groups that cross N, or a C that
      // breaks the 16-byte rule, are written row by row.  Warp-uniform.
      auto store_group = [&](int j, const float4 (&v)[4]) {
        const int col0 = colw + 16 * j;
        if (16 * j >= wcols || col0 >= p.N) return;
        if (!p.vec_c || col0 + 16 > p.N) {
#pragma unroll
          for (int q2 = 0; q2 < 4; ++q2) store_quad(4 * j + q2, v[q2]);
          return;
        }
        const int sw = (lane >> 1) & 3;
#pragma unroll
        for (int q2 = 0; q2 < 4; ++q2) tile[lane * 4 + (q2 ^ sw)] = v[q2];
        __syncwarp();
        const int rq = lane & 3;
        float* const cq = p.C + static_cast<long long>(row0 + (lane >> 2)) * p.ldc + col0 + 4 * rq;
        const long long row8 = 8 * p.ldc;   // eight rows further
        float4 val[4], cv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = 8 * i + (lane >> 2);
          val[i] = tile[r * 4 + (rq ^ ((r >> 1) & 3))];
          cv[i] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (has_c && row0 + r < p.M) cv[i] = __ldcs(reinterpret_cast<const float4*>(cq + i * row8));
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (row0 + 8 * i + (lane >> 2) >= p.M) continue;
          const float4 o =
              has_c ? make_float4(fmaf(p.alpha, val[i].x, p.beta * cv[i].x),
                                  fmaf(p.alpha, val[i].y, p.beta * cv[i].y),
                                  fmaf(p.alpha, val[i].z, p.beta * cv[i].z),
                                  fmaf(p.alpha, val[i].w, p.beta * cv[i].w))
                    : make_float4(p.alpha * val[i].x, p.alpha * val[i].y, p.alpha * val[i].z,
                                  p.alpha * val[i].w);
          __stcs(reinterpret_cast<float4*>(cq + i * row8), o);
        }
        __syncwarp();
      };
      int stile, sslice, nslices;
      slice_of(p, u, stile, sslice, nslices);
      if (nslices > 1) {
        // K slices: publish; the last slice of the tile to arrive adds all
        // slices up in slice order, kSumQuads column quads at a time (as many
        // loads in flight per slice), and writes C from the sums
        const float4* part = nullptr;
        if (!publish_slice(p, stile, sslice, nslices, static_cast<int>(rank), ew, lane, acc, part))
          continue;
#pragma unroll
        for (int gb = 0; gb < kCols / 4 / kSumQuads; ++gb) {
          float4 sum[kSumQuads];
#pragma unroll
          for (int i = 0; i < kSumQuads; ++i) sum[i] = __ldcg(part + (kSumQuads * gb + i) * 32);
          for (int s2 = 1; s2 < nslices; ++s2) {
            float4 v[kSumQuads];
#pragma unroll
            for (int i = 0; i < kSumQuads; ++i)
              v[i] = __ldcg(part + s2 * kSliceF4 + (kSumQuads * gb + i) * 32);
#pragma unroll
            for (int i = 0; i < kSumQuads; ++i) {
              sum[i].x += v[i].x;
              sum[i].y += v[i].y;
              sum[i].z += v[i].z;
              sum[i].w += v[i].w;
            }
          }
#pragma unroll
          for (int jj = 0; jj < kSumQuads / 4; ++jj) {
            const int g0 = kSumQuads * gb + 4 * jj;
            const float4 v4[4] = {sum[4 * jj], sum[4 * jj + 1], sum[4 * jj + 2], sum[4 * jj + 3]};
            store_group(kSumQuads / 4 * gb + jj, v4);
          }
        }
        continue;
      }
#pragma unroll
      for (int j = 0; j < kCols / 16; ++j) {
        float4 v4[4];
#pragma unroll
        for (int q2 = 0; q2 < 4; ++q2) {
          const int g = 4 * j + q2;
          v4[q2] = make_float4(acc[4 * g], acc[4 * g + 1], acc[4 * g + 2], acc[4 * g + 3]);
        }
        store_group(j, v4);
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(tmem_free_bar);
  }
  __syncwarp();
  cluster_sync();
}

cudaLaunchConfig_t pair_config(int grid, cudaStream_t stream, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemAlloc;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

cudaError_t configure(int dev) {
  static bool done[64] = {};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(sgemm_split_kernel<false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(sgemm_split_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemAlloc);
    if (e != cudaSuccess) return e;
    done[dev] = true;
  }
  return cudaSuccess;
}

template <bool F16>
cudaError_t launch_split(const CUtensorMap& a1, const CUtensorMap& a2, const CUtensorMap& b1,
                         const CUtensorMap& b2, const CUtensorMap& b1h, const CUtensorMap& b2h,
                         const Tf32Args& args, int grid, cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = configure(dev)) != cudaSuccess) return e;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = pair_config(grid, stream, attr);
  if (args.pdl) {
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 2;
  }
  e = cudaLaunchKernelEx(&cfg, sgemm_split_kernel<F16>, a1, a2, b1, b2, b1h, b2h, args);
  if (e != cudaSuccess) return e;
  return counted_launch(cudaGetLastError());
}

}  // namespace

int sgemm_3xtf32_max_pairs() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || configure(dev) != cudaSuccess) return 0;
  static int cached[64] = {};
  if (cached[dev] > 0) return cached[dev];
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pair_config(2, nullptr, attr);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, sgemm_split_kernel<false>, &cfg) != cudaSuccess) return 0;
  cached[dev] = n;
  return n;
}

cudaError_t launch_sgemm_3xtf32(const CUtensorMap& tmAb, const CUtensorMap& tmAs,
                                const CUtensorMap& tmBb, const CUtensorMap& tmBs,
                                const CUtensorMap& tmBbh, const CUtensorMap& tmBsh,
                                const Tf32Args& args, int grid, cudaStream_t stream) {
  return launch_split<false>(tmAb, tmAs, tmBb, tmBs, tmBbh, tmBsh, args, grid, stream);
}

cudaError_t launch_sgemm_3xf16(const CUtensorMap& tmA1, const CUtensorMap& tmA2,
                               const CUtensorMap& tmB1, const CUtensorMap& tmB2,
                               const Tf32Args& args, int grid, cudaStream_t stream) {
  return launch_split<true>(tmA1, tmA2, tmB1, tmB2, tmB1, tmB2, args, grid, stream);
}

}  // namespace gb300
