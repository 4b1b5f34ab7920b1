// internal.h -- declarations shared by the host dispatcher and the kernel
// translation units.  Not part of the public ABI.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace gb300 {

// Every kernel launch of the library goes through counted_launch: a
// successful launch adds one to a process-wide counter (gemm_launch_count).
void note_launch();
// Records the path the current call on this thread takes (a static string);
// gemm_last_path() returns it.
void set_last_path(const char* path);
inline cudaError_t counted_launch(cudaError_t e) {
  if (e == cudaSuccess) note_launch();
  return e;
}

struct DeviceStatus;

// Operand-load modes of the tensor-core kernel.
enum LoadMode : int { kLoadTma = 0, kLoadManual = 1 };
// Epilogue modes: TMA load/store of C, predicated element access of C, or
// raw fp32 partial sums to the split-K workspace.
// kEpiF32: fp32 C from registers; kEpiF32Tma: fp32 C through shared memory
// and TMA (CTA pairs, C 16-byte aligned, N % 4 == 0).
enum EpiMode : int { kEpiTma = 0, kEpiManual = 1, kEpiPartial = 2, kEpiF32 = 3, kEpiF32Tma = 4 };

struct TcArgs {
  const uint16_t* A;
  const uint16_t* B;
  uint16_t* C;
  int M, N, K;
  long long lda, ldb, ldc;
  float alpha, beta;
  int tiles_m, tiles_n;
  int splits;         // number of K slices (1 = no split)
  int kb_total;       // ceil(K / 64)
  int kb_per_split;   // K blocks per slice (every slice non-empty)
  int num_units;      // dp_tiles * splits + tail tiles * tail_splits
  int group_m;        // tile-order grouping along M (L2 reuse of B panels)
  float* ws;          // split-K partials [splits][M][ws_ld]
  long long ws_ld;
  // Tail balancing (splits == 1 only): the first dp_tiles tiles (in visiting
  // order) are computed whole; each remaining tile is cut into tail_splits
  // K slices whose fp32 partial sums go to tail_ws; the last slice to finish
  // (counted in tail_counters under this launch's epoch) adds them up in
  // slice order and runs the epilogue.
  int dp_tiles;
  int tail_splits;
  int tail_kb_per_split;
  float* tail_ws;                      // [tail tile][slice][128][BN]
  unsigned long long* tail_counters;   // [tail tile][8 epilogue warps]: epoch << 32 | arrivals
  unsigned int epoch;
  // Stream-K region (sk_tiles > 0, after the units above): the tiles
  // sk_tile0 .. sk_tile0 + sk_tiles - 1 (in visiting order) are treated as
  // sk_iters = sk_tiles * kb_total k-blocks, and worker w of sk_workers takes
  // k-blocks [w*sk_iters/sk_workers, (w+1)*sk_iters/sk_workers), cut at tile
  // boundaries into pieces.  A tile covered by several pieces is finished like
  // a tail tile; tail_splits is then the most pieces any tile can have (the
  // stride of tail_ws).
  int sk_tile0, sk_tiles, sk_workers;
  long long sk_iters;
  // sk_order 0: a worker takes its stream-K pieces after its whole tiles, in
  // k order.  sk_order 1 (the stream-K tiles are the last, partial wave and no
  // range is longer than a tile, so a range touches at most two tiles): the
  // piece that ends a tile (it finishes the tile) runs last, after the whole
  // tiles, and the other piece runs first, so that a tile's other pieces have
  // long published when its finisher ends.
  int sk_order;
  // kEpiF32: C is fp32 (Cf, ldc in floats) and written straight from
  // registers, with 16-byte accesses when vec_c (Cf and ldc 16-byte aligned)
  // and predicated element accesses otherwise.
  float* Cf;
  int vec_c;
  // tail_halves != 0 (TMA loads, BN >= 128): the tiles after dp_tiles are
  // computed as two units of BN/2 columns each (whole K, an MMA of N = BN/2)
  // instead of K slices.
  int tail_halves;
  // tail_first != 0 (splits == 1, tail_splits == 2, K slices of
  // tail_kb_per_split k-blocks and the rest): the first T tiles in visiting
  // order are cut in two; units [0, T) are their first K slices, then come the
  // dp_tiles whole tiles T, T + 1, ..., then the second slices.  Workers take
  // units worker, worker + nworkers, ..., so a first slice (it publishes its
  // partial sums) is its worker's first unit and a second slice (it finishes
  // the tile) its worker's last, long after the first was published.
  int tail_first;
  // single-CTA kernels: A (B) is read by one column (row) of tiles only, i.e.
  // streamed once -- loaded evict-first, so it does not push out of L2 lines
  // that are still useful (or dirty lines that would be written back)
  int stream_a, stream_b;
  unsigned long long wait_limit_ns;
  DeviceStatus* status;
  // host only: the launch directly follows this call's pre-pass kernel on the
  // same stream, so it may start early (programmatic dependent launch; the
  // kernel waits for the pre-pass before touching global memory)
  bool pdl;
};

// Tensor-core fp16 GEMM (tcgen05).  Maps are ignored by the modes that do not
// use them.  kpb: k-blocks per ring stage, 1, or 2 for 64-wide tiles with TMA
// loads and epilogue.  Returns a cudaError_t from the launch.
cudaError_t launch_gemm_f16_tc(int bn, int load_mode, int epi_mode, const CUtensorMap& tmA,
                               const CUtensorMap& tmB, const CUtensorMap& tmC, const TcArgs& args,
                               int grid, cudaStream_t stream, int kpb = 1);
int tc_threads(int load_mode);

// The same GEMM with an fp32 C (epilogue kEpiF32; gemm_f16_f32out.cu).
cudaError_t launch_gemm_f16_tc_f32(int bn, int load_mode, const CUtensorMap& tmA,
                                   const CUtensorMap& tmB, const TcArgs& args, int grid,
                                   cudaStream_t stream);
cudaError_t launch_gemm_f16_tc_pair_f32(int epi_mode, const CUtensorMap& tmA,
                                        const CUtensorMap& tmB, const CUtensorMap& tmC,
                                        const TcArgs& args, int grid, cudaStream_t stream);
int tc_pair_max_clusters_f32(int epi_mode);

// The same GEMM (128-wide tiles, TMA loads, one CTA per tile) for M <= am,
// staging am = 32 or 64 rows of A per k-block (gemm_f16_skinny.cu).
cudaError_t launch_gemm_f16_tc_skinny(int am, int epi_mode, const CUtensorMap& tmA,
                                      const CUtensorMap& tmB, const CUtensorMap& tmC,
                                      const TcArgs& args, int grid, cudaStream_t stream);
// 64-wide tiles of 64 rows (tcgen05.mma with M = 64), TMA loads and epilogue,
// whole-K units only (gemm_f16_skinny.cu); C's map has 32 x 16-row boxes.
cudaError_t launch_gemm_f16_tc_m64(const CUtensorMap& tmA, const CUtensorMap& tmB,
                                   const CUtensorMap& tmC, const TcArgs& args, int grid,
                                   cudaStream_t stream);

// One thread waits on an mbarrier that nothing arrives on, so the bounded wait
// runs out after limit_ns and records GEMM_ERR_TIMEOUT in *status.
cudaError_t launch_wait_probe(unsigned long long limit_ns, DeviceStatus* status,
                              cudaStream_t stream);

// fp32 -> fp16 conversion of n elements, round to nearest even.
cudaError_t launch_f32_to_f16(const float* src, uint16_t* dst, long long n, int grid,
                              cudaStream_t stream);

// The same GEMM on CTA pairs (clusters of 2 sharing tcgen05.mma.cta_group::2):
// 256 x bn output tiles (bn = 256, or 224 / 192 with a half C), TMA operand
// loads only, epilogue kEpiTma or kEpiManual (or the fp32-C ones, bn = 256).
// tiles_m counts 256-row tiles; grid = 2 x (number of pairs).  kpb: k-blocks
// per ring stage, 1, or 2 for bn = 256 with the TMA epilogue.
cudaError_t launch_gemm_f16_tc_pair(int bn, int epi_mode, const CUtensorMap& tmA,
                                    const CUtensorMap& tmB, const CUtensorMap& tmC,
                                    const TcArgs& args, int grid, cudaStream_t stream,
                                    int kpb = 1);
// The 224- and 192-wide instances (gemm_f16_pair_narrow.cu).
cudaError_t launch_gemm_f16_tc_pair_narrow(int bn, int epi_mode, const CUtensorMap& tmA,
                                           const CUtensorMap& tmB, const CUtensorMap& tmC,
                                           const TcArgs& args, int grid, cudaStream_t stream);
// Pairs of the 256-wide configuration that fit on the device at once (0 on
// error); the narrower tiles stage the same bytes, so the same number fits.
int tc_pair_max_clusters(int epi_mode);

// Split-K reduction: C = half(alpha * sum_s ws[s] + beta * C).
cudaError_t launch_splitk_reduce_f16(const float* ws, long long ws_ld, int splits, uint16_t* C,
                                     long long ldc, int M, int N, float alpha, float beta,
                                     int grid, cudaStream_t stream);

// Copies a rows x cols half matrix with any leading dimension and alignment
// into a 16-byte-aligned one with ldd = cols rounded up to 8 (zero padding).
struct RealignJob {
  const uint16_t* src;
  long long lds;
  uint16_t* dst;
  long long ldd;
  int rows, cols;
};
// One launch for up to three copies: blocks [end[i-1], end[i]) copy jobs[i].
struct RealignBatch {
  RealignJob job[3];
  int end[3];
  int n;
};
cudaError_t launch_realign_f16(const RealignBatch& batch, cudaStream_t stream);

// The copy back: dst (rows x cols, any 2-byte alignment and leading dimension
// ldd) := src (16-byte-aligned rows, lds >= cols rounded up to 8).  Launched
// after the kernel that writes src, which it may overlap (programmatic
// dependent launch; it waits for that kernel's completion before reading).
cudaError_t launch_unalign_f16(const RealignJob& job, int grid, cudaStream_t stream);

// Both splits of a 3xTF32 product in one launch: A (M x K) into Ab, As and
// B^T (B is K x N) into Bb, Bs, all with leading dimension ld2 (>= K, % 4 == 0);
// grid_a blocks work on A, grid_b on B^T.
cudaError_t launch_split_tf32_ab(const float* A, long long lda, float* Ab, float* As,
                                 const float* B, long long ldb, float* Bb, float* Bs, long long ld2,
                                 int M, int N, int K, int grid_a, int grid_b, cudaStream_t stream);

// The fp16 parts of the 3xFP16 SGEMM, x * 2^e = h1 + h2 (+ 2^-22 relative):
// 3xFP16 operand parts: A1, A2 (M x lda2 halves) and B1, B2 (K x ldb2), and
// the power-of-two exponents they were scaled by, per K chunk of
// kF16x3ChunkK: ea[row][chunk] (M x kchunks), eb[chunk][col] (kchunks x ldeb,
// ldeb >= N + 4).
constexpr int kF16x3ChunkK = 256;
struct F16x3Parts {
  uint16_t *A1, *A2, *B1, *B2;
  long long lda2, ldb2;
  int* ea;
  int* eb;
  long long ldeb;
};
// One launch of 1024-thread blocks: blocks [0, grid_b) split B by (chunk,
// 128 columns), the other grid_a blocks A by (row, chunk), one warp an item.
cudaError_t launch_f16x3_split(const float* A, long long lda, const float* B, long long ldb,
                               const F16x3Parts& parts, int M, int N, int K, int grid_a,
                               int grid_b, cudaStream_t stream);

// 3xTF32 SGEMM on CTA pairs: C = alpha*(Ab*Bb + Ab*Bs + As*Bb) + beta*C with
// the split operands dense and K-contiguous: A parts M x roundup(K,4), B parts
// transposed, N x roundup(K,4).
// k-blocks (64 bytes of K per row) in one TMEM accumulation chunk of the
// split-operand kernel: 128 floats (3xTF32) or 256 halves (3xFP16).
constexpr int kSplitChunkKb = 8;
struct Tf32Args {
  const float* Ab;
  const float* As;
  const float* Bb;
  const float* Bs;
  float* C;
  int M, N, K;
  long long ldc;
  float alpha, beta;
  int tiles_m, tiles_n;   // 256 x 256 pair tiles
  int kb_total;           // ceil(K / 32)
  // units [0, dp_tiles) are whole tiles; each tile after them (the last,
  // partial wave) runs as two half-width units of 128 columns
  int dp_tiles;
  int num_units;
  int group_m;
  bool vec_c;             // C 16-byte aligned with ldc % 4 == 0
  unsigned long long wait_limit_ns;
  DeviceStatus* status;
  // splits > 1: every unit is one K slice of a whole tile (unit = tile *
  // splits + slice, slice s covering k-blocks [s * kb_per_split, ...), a
  // multiple of the 4-k-block accumulation chunk); each slice publishes fp32
  // partial sums and the last one of a tile to finish adds them up in slice
  // order and writes C
  int splits;
  int kb_per_split;
  float4* part_ws;                  // [tile][rank][warp][slice][32 column quads][32 rows]
  unsigned long long* counters;     // [tile][rank][warp]: (epoch << 32) | arrivals
  unsigned int epoch;
  bool pdl;                         // host only: as TcArgs::pdl (after the split pre-pass)
  // Two-slice tail (splits == 1): the tail tiles -- T = (num_units -
  // dp_tiles) / 2 of them, the first T in visiting order -- are cut into a
  // first slice of kb_per_split k-blocks (whole accumulation chunks), a
  // worker's first unit, and a second slice, a worker's last; the slice that
  // arrives last adds both up, as with K slices.
  int tail_first;
  // 3xFP16 only: the power-of-two exponents the parts were scaled by, per K
  // chunk of kF16x3ChunkK (the accumulation chunk): ea[row * kchunks + c],
  // eb[c * ldeb + col] (ldeb >= N + 4)
  const int* ea;
  const int* eb;
  long long ldeb;
  int kchunks;
};
// tmBbh / tmBsh: the B parts with 64-row boxes, for the half-width units.
cudaError_t launch_sgemm_3xtf32(const CUtensorMap& tmAb, const CUtensorMap& tmAs,
                                const CUtensorMap& tmBb, const CUtensorMap& tmBs,
                                const CUtensorMap& tmBbh, const CUtensorMap& tmBsh,
                                const Tf32Args& args, int grid, cudaStream_t stream);
int sgemm_3xtf32_max_pairs();
// The same kernel on the 3xFP16 parts (A1, A2: M x lda2 halves, boxes of 64
// columns x 128 rows; B1, B2: K x ldb2 halves, boxes of 64 columns x 64 rows);
// k-blocks of 64.
cudaError_t launch_sgemm_3xf16(const CUtensorMap& tmA1, const CUtensorMap& tmA2,
                               const CUtensorMap& tmB1, const CUtensorMap& tmB2,
                               const Tf32Args& args, int grid, cudaStream_t stream);

// C := beta * C (C := 0 when beta == 0): the alpha == 0 / K == 0 case.
cudaError_t launch_scale_f16(uint16_t* C, long long ldc, int M, int N, float beta, int grid,
                             cudaStream_t stream);
cudaError_t launch_scale_f32(float* C, long long ldc, int M, int N, float beta, int grid,
                             cudaStream_t stream);

// FFMA SGEMM.  vec = 16-byte vector loads allowed (aligned pointers, ld % 4 == 0).
struct SgemmArgs {
  const float* A;
  const float* B;
  float* C;
  int M, N, K;
  long long lda, ldb, ldc;
  float alpha, beta;
};
cudaError_t launch_sgemm_ffma(bool vec, const SgemmArgs& args, cudaStream_t stream);

// Current device: SM count, status word and wait limit (library set-up done
// on first use).  Returns a GEMM_* code.
int query_device(int* sm_count, DeviceStatus** status, unsigned long long* wait_limit_ns);

// 2-D fp16 tensor map with 128-byte swizzle (rows x cols, row stride ld).
int encode_map_f16(CUtensorMap* map, const void* ptr, int rows, int cols, long long ld,
                   int box_cols, int box_rows);

}  // namespace gb300
