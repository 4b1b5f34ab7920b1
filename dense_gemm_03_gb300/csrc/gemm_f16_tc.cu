// gemm_f16_tc.cu -- fp16-in / fp32-accumulate GEMM on the 5th-generation
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
// One CTA per SM, persistent over output tiles (BM x BN = 128 x {64,128,256}),
// warp-specialised:
//   producer warp(s)  TMA tile loads (or, for unaligned operands, predicated
//                     element loads written in the same swizzled layout)
//   MMA warp          one thread issues tcgen05.mma (M=128, N=BN, K=16) into a
//                     double-buffered TMEM accumulator (2 x BN fp32 columns)
//   4 epilogue warps  tcgen05.ld the accumulator (warp w owns TMEM lanes
//                     32*(w%4) .. +31 = tile rows), apply alpha/beta in fp32,
//                     round to fp16 and store (TMA, predicated stores, or raw
//                     fp32 partials for split-K)
// The epilogue of tile i overlaps the main loop of tile i+1.
//
// Shared-memory operand layouts (128-byte swizzle, 1024-byte aligned):
//   A stage: 128 rows x 64 halves, K-major; row r at r*128 B, 16-byte chunk c
//            of the row stored at chunk (c ^ (r % 8)).  SBO = 1024 B.
//   B stage: BN/64 column blocks of 64 (k) rows x 64 halves, N-major (MN-major
//            operand); k-row at k*128 B inside its block, same swizzle.
//            LBO = 8 KB (next 64 columns), SBO = 1024 B (next 8 k-rows).
#include "internal.h"
#include "ptx.cuh"

namespace gb300 {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;                       // halves per k-block: one 128-byte swizzle row
constexpr int kUmmaK = 16;                   // K of one tcgen05.mma kind::f16
constexpr int kABytes = BM * BK * 2;         // 16 KB
constexpr int kBBlockBytes = BK * 128;       // one 64-column block of a B stage: 8 KB
constexpr int kEpiBufBytes = 32 * 128;       // 32 rows x 64 halves
constexpr unsigned long long kDrainLimitNs = 1000000000ull;

template <int BN>
struct TcCfg {
  static constexpr int kBBytes = BN * BK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = (BN == 256) ? 4 : (BN == 128 ? 6 : 8);
  static constexpr int kTmemCols = 2 * BN;   // two accumulators
  static constexpr int kChunks = BN / 64;    // epilogue column chunks
  static_assert(BN == 64 || BN == 128 || BN == 256, "tile width");
};

template <int LOAD>
struct Roles {
  static constexpr int kProdWarps = (LOAD == kLoadTma) ? 1 : 4;
  static constexpr int kMmaWarp = kProdWarps;
  static constexpr int kEpiWarp0 = kProdWarps + 1;
  static constexpr int kWarps = kProdWarps + 5;
  static constexpr int kThreads = kWarps * 32;
};

template <int BN, int EPI>
struct Smem {
  using Cfg = TcCfg<BN>;
  static constexpr int kEpiOff = Cfg::kStages * Cfg::kStageBytes;
  static constexpr int kEpiBytes = (EPI == kEpiPartial) ? 0 : 4 * 2 * kEpiBufBytes;
  static constexpr int kBarOff = kEpiOff + kEpiBytes;
  // full[S], empty[S], acc_full[2], acc_empty[2], c_load[4][2], mma_done
  static constexpr int kNumBars = 2 * Cfg::kStages + 2 + 2 + 8 + 1;
  static constexpr int kTmemPtrOff = kBarOff + kNumBars * 8;
  static constexpr int kUsed = kTmemPtrOff + 16;
  static constexpr int kAlloc = kUsed + 1024;  // the dynamic base is aligned up to 1024 B
  static_assert(kAlloc <= 232448, "shared memory budget");
};

struct Unit {
  int m0, n0, kb0, kb1, split;
  int tail;       // 1 for a K slice of a tail tile
  int tail_idx;   // index of the tail tile (tail units only)
};

// Work unit u -> output tile and K range.  Units [0, dp_tiles*splits) are
// whole tiles (or split-K slices); the rest are K slices of the tail tiles.
// Tiles are visited in groups of group_m tile-rows so that concurrently
// running CTAs share B panels in L2.
__device__ __forceinline__ Unit decode_unit(const TcArgs& p, int u, int bn) {
  Unit x;
  int tile, kpb;
  const int dp_units = p.dp_tiles * p.splits;
  if (u < dp_units) {
    tile = u / p.splits;
    x.split = u - tile * p.splits;
    kpb = p.kb_per_split;
    x.tail = 0;
    x.tail_idx = 0;
  } else {
    const int v = u - dp_units;
    x.tail_idx = v / p.tail_splits;
    x.split = v - x.tail_idx * p.tail_splits;
    tile = p.dp_tiles + x.tail_idx;
    kpb = p.tail_kb_per_split;
    x.tail = 1;
  }
  const int group = p.group_m * p.tiles_n;
  const int g = tile / group;
  const int first_m = g * p.group_m;
  const int gm = min(p.tiles_m - first_m, p.group_m);
  const int r = tile - g * group;
  x.m0 = (first_m + r % gm) * BM;
  x.n0 = (r / gm) * bn;
  x.kb0 = x.split * kpb;
  x.kb1 = min(p.kb_total, x.kb0 + kpb);
  return x;
}

// Waits that must not give up early because another thread failed: used only
// to let copies already in flight land before the CTA exits.
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

// Byte offset of (row r, column c) inside a 128-byte-swizzled 32 x 64 half tile.
__device__ __forceinline__ uint32_t sw128_off(int r, int c) {
  return static_cast<uint32_t>(r * 128 + ((((c >> 3) ^ (r & 7)) & 7) << 4) + ((c & 7) << 1));
}

template <int BN, int LOAD, int EPI>
__global__ void __launch_bounds__(Roles<LOAD>::kThreads, 1)
    gemm_f16_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmC, const TcArgs p) {
  using Cfg = TcCfg<BN>;
  using R = Roles<LOAD>;
  using L = Smem<BN, EPI>;
  constexpr int S = Cfg::kStages;

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
  auto cload_bar = [&](int w, uint32_t b) { return bars + 8u * (2 * S + 4 + 2 * w + b); };
  const uint32_t done_bar = bars + 8u * (2 * S + 12);
  auto stage_a = [&](int s) { return base + static_cast<uint32_t>(s * Cfg::kStageBytes); };
  auto stage_b = [&](int s) { return stage_a(s) + kABytes; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), LOAD == kLoadTma ? 1u : 128u);
      mbar_init(empty_bar(s), 1u);
    }
    for (uint32_t b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1u);
      mbar_init(acce_bar(b), 4u);
    }
    for (int w = 0; w < 4; ++w)
      for (uint32_t b = 0; b < 2; ++b) mbar_init(cload_bar(w, b), 1u);
    mbar_init(done_bar, 1u);
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == R::kMmaWarp) {
    tmem_alloc(base + L::kTmemPtrOff, Cfg::kTmemCols);
    tmem_relinquish();
  }
  if (LOAD == kLoadTma && warp == 0 && lane == 0) {
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
  }
  if (EPI == kEpiTma && warp == R::kEpiWarp0 && lane == 0) prefetch_tensormap(&tmC);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
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
        for (int u = blockIdx.x; ok && u < p.num_units; u += gridDim.x) {
          const Unit t = decode_unit(p, u, BN);
          for (int kb = t.kb0; kb < t.kb1; ++kb) {
            if (!wait_parity(empty_bar(stage), phase ^ 1u, limit, st, 1)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(full_bar(stage), Cfg::kStageBytes);
            tma_load_2d(stage_a(stage), &tmA, full_bar(stage), kb * BK, t.m0);
#pragma unroll
            for (int c = 0; c < Cfg::kChunks; ++c)
              tma_load_2d(stage_b(stage) + c * kBBlockBytes, &tmB, full_bar(stage), t.n0 + 64 * c,
                          kb * BK);
            ++issued;
            if (++stage == S) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
        // The last loads (at most one per stage) must land before the CTA exits.
        const uint32_t n = issued < static_cast<uint32_t>(S) ? issued : static_cast<uint32_t>(S);
        for (uint32_t i = issued - n; i < issued; ++i)
          drain_wait(full_bar(static_cast<int>(i % S)), (i / S) & 1u, st, 11);
      }
      __syncwarp();
    } else {
      const int tp = static_cast<int>(threadIdx.x);  // 0..127
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < p.num_units; u += gridDim.x) {
        const Unit t = decode_unit(p, u, BN);
        for (int kb = t.kb0; kb < t.kb1; ++kb) {
          if (!wait_parity(empty_bar(stage), phase ^ 1u, limit, st, 2)) {
            ok = false;
            break;
          }
          uint8_t* const sa = base_ptr + stage * Cfg::kStageBytes;
          uint8_t* const sb = sa + kABytes;
          const int k0 = kb * BK;
          // A: 128 rows x 8 chunks of 8 halves.
#pragma unroll
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
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc(0u, BM, BN, 0u, 1u);
      int stage = 0;
      uint32_t phase = 0, local = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < p.num_units; u += gridDim.x) {
        const Unit t = decode_unit(p, u, BN);
        const uint32_t buf = local & 1u, use = local >> 1;
        if (!wait_parity(acce_bar(buf), (use & 1u) ^ 1u, limit, st, 3)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * BN;
        for (int kb = t.kb0; kb < t.kb1; ++kb) {
          if (!wait_parity(full_bar(stage), phase, limit, st, 4)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = stage_a(stage), b0 = stage_b(stage);
#pragma unroll
          for (int kk = 0; kk < BK / kUmmaK; ++kk) {
            const uint64_t ad = smem_desc_sw128(a0 + kk * (kUmmaK * 2), 16u, 1024u);
            const uint64_t bd = smem_desc_sw128(b0 + kk * (kUmmaK * 128), kBBlockBytes, 1024u);
            mma_f16_ss(d_tmem, ad, bd, idesc, (kb > t.kb0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(empty_bar(stage));  // frees the stage once these MMAs finish
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(accf_bar(buf));       // accumulator ready for the epilogue
        ++local;
      }
      // Every MMA issued above must complete before TMEM is released.
      mma_commit(done_bar);
      drain_wait(done_bar, 0u, st, 12);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - R::kEpiWarp0;   // buffer set 0..3
    const int q = warp & 3;               // TMEM lane quadrant -> rows 32q .. 32q+31
    const bool has_c = p.beta != 0.0f;
    uint32_t local = 0, cc = 0;
    for (int u = blockIdx.x; u < p.num_units; u += gridDim.x) {
      const Unit t = decode_unit(p, u, BN);
      const uint32_t buf = local & 1u, use = local >> 1;
      if (!wait_parity(accf_bar(buf), use & 1u, limit, st, 5)) break;
      tc_fence_after();
      const int row0 = t.m0 + 32 * q;
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + buf * BN;
      bool ok = true;
      bool finish = row0 < p.M;   // this warp produces final values for its rows
      if (EPI != kEpiPartial && t.tail && finish) {
        // Publish this slice's partial sums (tile-local rows 32q+lane, all BN
        // columns), then count the slice in.  The last slice finishes the tile.
        float* mine = p.tail_ws +
                      ((static_cast<long long>(t.tail_idx) * p.tail_splits + t.split) * BM +
                       32 * q + lane) * BN;
        for (int j = 0; j < Cfg::kChunks; ++j) {
          if (t.n0 + 64 * j >= p.N) break;
          uint32_t acc[64];
          tmem_ld_32x32b_x32(tbase + 64 * j, *reinterpret_cast<uint32_t(*)[32]>(acc));
          tmem_ld_32x32b_x32(tbase + 64 * j + 32, *reinterpret_cast<uint32_t(*)[32]>(acc + 32));
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 64; c += 4)
            __stcg(reinterpret_cast<float4*>(mine + 64 * j + c),
                   make_float4(__uint_as_float(acc[c]), __uint_as_float(acc[c + 1]),
                               __uint_as_float(acc[c + 2]), __uint_as_float(acc[c + 3])));
        }
        __threadfence();
        __syncwarp();
        uint32_t arrived = 0;
        if (lane == 0) {
          unsigned long long* cnt = p.tail_counters + t.tail_idx * 4 + q;
          unsigned long long cur = *reinterpret_cast<volatile unsigned long long*>(cnt);
          for (;;) {
            const unsigned long long next =
                (static_cast<unsigned int>(cur >> 32) == p.epoch)
                    ? cur + 1ull
                    : ((static_cast<unsigned long long>(p.epoch) << 32) | 1ull);
            const unsigned long long prev = atomicCAS(cnt, cur, next);
            if (prev == cur) {
              arrived = static_cast<uint32_t>(next & 0xFFFFFFFFull);
              break;
            }
            cur = prev;
          }
        }
        arrived = __shfl_sync(0xffffffffu, arrived, 0);
        finish = arrived == static_cast<uint32_t>(p.tail_splits);
        if (finish) __threadfence();
      }
      if (finish) {
        for (int j = 0; j < Cfg::kChunks && ok; ++j) {
          const int col0 = t.n0 + 64 * j;
          if (col0 >= p.N) break;
          uint32_t acc[64];
          if (EPI == kEpiTma) {
            // wait until the store issued from this buffer two chunks ago has read it
            if (lane == 0) bulk_wait_group_read<1>();
            __syncwarp();
            if (has_c && lane == 0) {
              const uint32_t b = cc & 1u;
              const uint32_t sbuf = base + L::kEpiOff + (ew * 2 + b) * kEpiBufBytes;
              mbar_arrive_expect_tx(cload_bar(ew, b), kEpiBufBytes);
              tma_load_2d(sbuf, &tmC, cload_bar(ew, b), col0, row0);
            }
          }
          tmem_ld_32x32b_x32(tbase + 64 * j, *reinterpret_cast<uint32_t(*)[32]>(acc));
          tmem_ld_32x32b_x32(tbase + 64 * j + 32, *reinterpret_cast<uint32_t(*)[32]>(acc + 32));
          tmem_wait_ld();
          if (EPI != kEpiPartial && t.tail) {
            // acc := sum over slices in slice order (own slice from TMEM)
            float sum[64];
            for (int s2 = 0; s2 < p.tail_splits; ++s2) {
              const float* src = p.tail_ws +
                                 ((static_cast<long long>(t.tail_idx) * p.tail_splits + s2) * BM +
                                  32 * q + lane) * BN + 64 * j;
#pragma unroll
              for (int c = 0; c < 64; c += 4) {
                float4 v;
                if (s2 == t.split)
                  v = make_float4(__uint_as_float(acc[c]), __uint_as_float(acc[c + 1]),
                                  __uint_as_float(acc[c + 2]), __uint_as_float(acc[c + 3]));
                else
                  v = __ldcg(reinterpret_cast<const float4*>(src + c));
                if (s2 == 0) {
                  sum[c] = v.x; sum[c + 1] = v.y; sum[c + 2] = v.z; sum[c + 3] = v.w;
                } else {
                  sum[c] += v.x; sum[c + 1] += v.y; sum[c + 2] += v.z; sum[c + 3] += v.w;
                }
              }
            }
#pragma unroll
            for (int c = 0; c < 64; ++c) acc[c] = __float_as_uint(sum[c]);
          }
          if (EPI == kEpiPartial) {
            const int row = row0 + lane;
            if (row < p.M) {
              float* wrow = p.ws + (static_cast<long long>(t.split) * p.M + row) * p.ws_ld;
#pragma unroll
              for (int c = 0; c < 64; c += 4) {
                const int col = col0 + c;
                const float4 v = make_float4(__uint_as_float(acc[c]), __uint_as_float(acc[c + 1]),
                                             __uint_as_float(acc[c + 2]),
                                             __uint_as_float(acc[c + 3]));
                if (col + 4 <= p.N) {
                  *reinterpret_cast<float4*>(wrow + col) = v;
                } else {
                  if (col < p.N) wrow[col] = v.x;
                  if (col + 1 < p.N) wrow[col + 1] = v.y;
                  if (col + 2 < p.N) wrow[col + 2] = v.z;
                }
              }
            }
          } else if (EPI == kEpiTma) {
            const uint32_t b = cc & 1u;
            const int boff = L::kEpiOff + (ew * 2 + static_cast<int>(b)) * kEpiBufBytes;
            const uint32_t sbuf = base + boff;
            uint8_t* const sptr = base_ptr + boff;
            if (has_c && !wait_parity(cload_bar(ew, b), (cc >> 1) & 1u, limit, st, 6)) {
              drain_wait(cload_bar(ew, b), (cc >> 1) & 1u, st, 13);
              ok = false;
              break;
            }
#pragma unroll
            for (int g = 0; g < 8; ++g) {
              const uint32_t off = static_cast<uint32_t>(lane * 128 + ((g ^ (lane & 7)) << 4));
              const uint4 cv = has_c ? *reinterpret_cast<const uint4*>(sptr + off)
                                     : make_uint4(0u, 0u, 0u, 0u);
              *reinterpret_cast<uint4*>(sptr + off) =
                  epilogue8(acc + 8 * g, cv, has_c, p.alpha, p.beta);
            }
            fence_proxy_async_smem();   // generic writes -> TMA store reads
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmC, sbuf, col0, row0);
              bulk_commit_group();
            }
            ++cc;
          } else {  // kEpiManual
            uint8_t* const sptr = base_ptr + L::kEpiOff + (ew * 2) * kEpiBufBytes;
            const int cl = 2 * lane;   // this lane's column pair inside the chunk
            if (has_c) {
              for (int r = 0; r < 32; ++r) {
                const int row = row0 + r, col = col0 + cl;
                uint32_t h0 = 0, h1 = 0;
                if (row < p.M) {
                  const uint16_t* crow = p.C + static_cast<long long>(row) * p.ldc;
                  if (col < p.N) h0 = crow[col];
                  if (col + 1 < p.N) h1 = crow[col + 1];
                }
                *reinterpret_cast<uint32_t*>(sptr + sw128_off(r, cl)) = h0 | (h1 << 16);
              }
              __syncwarp();
            }
#pragma unroll
            for (int g = 0; g < 8; ++g) {
              const uint32_t off = static_cast<uint32_t>(lane * 128 + ((g ^ (lane & 7)) << 4));
              const uint4 cv = has_c ? *reinterpret_cast<const uint4*>(sptr + off)
                                     : make_uint4(0u, 0u, 0u, 0u);
              *reinterpret_cast<uint4*>(sptr + off) =
                  epilogue8(acc + 8 * g, cv, has_c, p.alpha, p.beta);
            }
            __syncwarp();
            for (int r = 0; r < 32; ++r) {
              const int row = row0 + r, col = col0 + cl;
              if (row < p.M) {
                const uint32_t v = *reinterpret_cast<const uint32_t*>(sptr + sw128_off(r, cl));
                uint16_t* crow = p.C + static_cast<long long>(row) * p.ldc;
                if (col < p.N) crow[col] = static_cast<uint16_t>(v & 0xFFFFu);
                if (col + 1 < p.N) crow[col + 1] = static_cast<uint16_t>(v >> 16);
              }
            }
            __syncwarp();
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acce_bar(buf));   // accumulator may be overwritten
      ++local;
      if (!ok) break;
    }
    if (EPI == kEpiTma && lane == 0) bulk_wait_group<0>();
    __syncwarp();
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (warp == R::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}

template <int BN, int LOAD, int EPI>
cudaError_t launch_one(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                       const TcArgs& args, int grid, cudaStream_t stream) {
  using L = Smem<BN, EPI>;
  auto kernel = gemm_f16_tc_kernel<BN, LOAD, EPI>;
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  kernel<<<grid, Roles<LOAD>::kThreads, L::kAlloc, stream>>>(tmA, tmB, tmC, args);
  return cudaGetLastError();
}

template <int BN>
cudaError_t launch_bn(int load, int epi, const CUtensorMap& a, const CUtensorMap& b,
                      const CUtensorMap& c, const TcArgs& args, int grid, cudaStream_t s) {
  if (load == kLoadTma) {
    if (epi == kEpiTma) return launch_one<BN, kLoadTma, kEpiTma>(a, b, c, args, grid, s);
    if (epi == kEpiManual) return launch_one<BN, kLoadTma, kEpiManual>(a, b, c, args, grid, s);
    return launch_one<BN, kLoadTma, kEpiPartial>(a, b, c, args, grid, s);
  }
  if (epi == kEpiTma) return launch_one<BN, kLoadManual, kEpiTma>(a, b, c, args, grid, s);
  if (epi == kEpiManual) return launch_one<BN, kLoadManual, kEpiManual>(a, b, c, args, grid, s);
  return launch_one<BN, kLoadManual, kEpiPartial>(a, b, c, args, grid, s);
}

}  // namespace

cudaError_t launch_gemm_f16_tc(int bn, int load_mode, int epi_mode, const CUtensorMap& tmA,
                               const CUtensorMap& tmB, const CUtensorMap& tmC, const TcArgs& args,
                               int grid, cudaStream_t stream) {
  switch (bn) {
    case 256: return launch_bn<256>(load_mode, epi_mode, tmA, tmB, tmC, args, grid, stream);
    case 128: return launch_bn<128>(load_mode, epi_mode, tmA, tmB, tmC, args, grid, stream);
    case 64: return launch_bn<64>(load_mode, epi_mode, tmA, tmB, tmC, args, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

int tc_smem_bytes(int bn, int epi_mode) {
  const bool part = epi_mode == kEpiPartial;
  switch (bn) {
    case 256: return part ? Smem<256, kEpiPartial>::kAlloc : Smem<256, kEpiTma>::kAlloc;
    case 128: return part ? Smem<128, kEpiPartial>::kAlloc : Smem<128, kEpiTma>::kAlloc;
    default: return part ? Smem<64, kEpiPartial>::kAlloc : Smem<64, kEpiTma>::kAlloc;
  }
}

int tc_threads(int load_mode) {
  return load_mode == kLoadTma ? Roles<kLoadTma>::kThreads : Roles<kLoadManual>::kThreads;
}

}  // namespace gb300
