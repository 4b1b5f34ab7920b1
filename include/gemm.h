/*
 * gemm.h -- C ABI of the GB300 dense GEMM library (libgemm.so).
 *
 * Every entry point computes, or supports the computation of,
 *
 *     C := alpha * A * B + beta * C
 *
 * on row-major operands: A is M x K, B is K x N, C is M x N, and element
 * (r, c) of an operand with leading dimension ld lives at ptr[r*ld + c]
 * ("advanced SGEMM on NVIDIA GPUs" summary page: introduction for the
 * formula, section on memory layout and PTX for row-major storage and the
 * lda/ldb/ldc convention).  The half-precision entry points follow the
 * LeetGPU statement on the "LeetGPU GEMM T4" page (baseline section): half
 * operands, a float accumulator, and the result acc*alpha + C*beta rounded to
 * half.
 *
 * Common rules
 *   Pointers   A, B, C are DEVICE pointers owned by the caller; the library
 *              never frees them.  A and B are read-only; C is read (unless
 *              beta == 0) and written.  C must not overlap A or B (not
 *              checked; the result is undefined).
 *   Layout     row-major; the non-_ld forms mean lda = K, ldb = N, ldc = N.
 *              Pointers must be aligned to their element (2 bytes for half,
 *              4 for float; else GEMM_ERR_ARG).  Beyond that any alignment is
 *              accepted: a half operand whose rows are not 16-byte aligned is
 *              first copied into an aligned scratch layout (or, with
 *              gemm_force_path(2), loaded with predicated element loads), and
 *              such a C is written with predicated element stores.
 *   Types      half = IEEE binary16 (bits in a uint16_t); float = binary32.
 *   Numerics   products accumulate in fp32; the epilogue alpha*acc + beta*c
 *              is evaluated in fp32 and rounded once, to nearest even, to the
 *              type of C.  Accumulation order is unspecified but fixed for a
 *              given shape and device, so repeated calls are bitwise equal.
 *   beta == 0  C is not read (it may hold NaN or Inf); C := alpha*A*B.
 *   alpha == 0 or K == 0
 *              A and B are not read; C := beta*C (C := 0 when beta == 0).
 *   M == 0 or N == 0
 *              nothing is done; returns GEMM_OK.
 *   Streams    work is enqueued on `stream` (NULL = the legacy default
 *              stream) and the call returns without synchronising.  Calls on
 *              different streams that write the same C race.
 *   Scratch    some shapes split K over several thread blocks and need an
 *              fp32 workspace (few tiles with a long K: stream-K for half
 *              operands, K slices for fp32 ones; the forced split paths);
 *              unaligned half operands need an aligned copy;
 *              the fp32 path keeps its tf32 operand parts.  The library owns
 *              this scratch, per device and stream, grows it on first need
 *              (that call may allocate device memory) and frees it in
 *              gemm_release().
 *   Graphs     a call may be captured in a CUDA graph on `stream` once the
 *              same shape has run on that stream outside the capture (so
 *              that no scratch has to be allocated inside it); replays give
 *              the same results as direct calls.
 *   Errors     a negative return code (below) and nothing enqueued, except
 *              GEMM_ERR_CUDA, which reports a failed launch.  Kernels never
 *              trap: a wait that runs past its time limit sets a device
 *              status word that gemm_debug_status() reads.
 */
#ifndef GB300_GEMM_H
#define GB300_GEMM_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
#define GEMM_OK               0
#define GEMM_ERR_NULL        -1  /* a needed pointer is NULL                          */
#define GEMM_ERR_DIM         -2  /* M, N or K is negative                             */
#define GEMM_ERR_LD          -3  /* lda < K, ldb < N or ldc < N (for a non-empty op)   */
#define GEMM_ERR_CUDA        -4  /* a CUDA runtime/driver call or a launch failed     */
#define GEMM_ERR_DEVICE      -5  /* current device is not compute capability 10.3     */
#define GEMM_ERR_TIMEOUT     -6  /* a kernel gave up waiting (gemm_debug_status)      */
#define GEMM_ERR_ARG         -7  /* another invalid argument (see the function)       */

/*
 * Half-precision GEMM: fp16 A, B, C; fp32 accumulation; fp16 result.
 * ("LeetGPU GEMM T4" page, baseline section: the solve(A, B, C, M, N, K,
 * alpha, beta) statement, with a stream argument and a status return added.)
 */
int gemm_f16(const uint16_t* A, const uint16_t* B, uint16_t* C,
             int M, int N, int K, float alpha, float beta, cudaStream_t stream);

/* As gemm_f16, with explicit leading dimensions in elements
 * (lda >= K, ldb >= N, ldc >= N; "advanced SGEMM" page, memory-layout
 * section). */
int gemm_f16_ld(const uint16_t* A, const uint16_t* B, uint16_t* C,
                int M, int N, int K, int lda, int ldb, int ldc,
                float alpha, float beta, cudaStream_t stream);

/*
 * C := alpha*A*B + beta*C with half A and B and a FLOAT C: fp32 accumulation
 * and an fp32 epilogue, with no rounding to half.  This is the WMMA kernel of
 * the "Tensorcore_wmma_vs_fp32 test code" page (section on the WMMA tensor
 * core GEMM kernel), which stores its fp32 accumulator fragment to a float C;
 * alpha = 1, beta = 0 gives exactly that product.  Leading dimensions in
 * elements (lda >= K, ldb >= N, ldc >= N).  C must be 4-byte aligned
 * (GEMM_ERR_ARG otherwise); with beta == 0 C is not read.  Otherwise the
 * rules of gemm_f16_ld apply (same kernels and scheduling).
 */
int gemm_f16_f32out(const uint16_t* A, const uint16_t* B, float* C,
                    int M, int N, int K, int lda, int ldb, int ldc,
                    float alpha, float beta, cudaStream_t stream);

/*
 * dst[i] := src[i] rounded to the nearest half, ties to even, for 0 <= i < n
 * (the float-to-half kernel of the same page, section on the float - half
 * conversion kernel): values beyond the half range become +-Inf, NaN stays
 * NaN.  Device pointers, src 4-byte and dst 2-byte aligned (GEMM_ERR_ARG
 * otherwise); 16-byte aligned pointers take the vectorised path.  n < 0 is
 * GEMM_ERR_DIM, n == 0 a no-op.  Asynchronous on `stream`.
 */
int gemm_f32_to_f16(const float* src, uint16_t* dst, long long n, cudaStream_t stream);

/* Single-precision GEMM (SGEMM, "advanced SGEMM" page): fp32 operands and
 * result, within the fp32 bound 1e-6 * K * max|A| * max|B| per element.
 * Shapes with K >= 64 run on the tensor cores as three products of split
 * operands with fp32 accumulation: within each 256-deep K chunk, each row of
 * A and each column of B is scaled by a power of two that brings its largest
 * magnitude into [2^14, 2^15) and split into two halves, x * 2^e = h1 + h2
 * (11 + 11 significand bits), so A*B ~= A1*B1 + A1*B2 + A2*B1 (the A2*B2 term,
 * about 2^-22 of |A||B|, is dropped); each chunk's products are scaled back
 * exactly as they are added up (3xFP16, for M*N*K above 256^3; tiny products
 * take tf32 parts instead, 3xTF32, at half the rate, as does
 * gemm_force_path(8)).  A pre-pass writes the parts to library-owned scratch (few output
 * tiles with a long K: every tile cut into K slices whose fp32 partial sums
 * are added in slice order, so results are reproducible run to run); a
 * shorter K uses an FFMA kernel (exact fp32 products).  An Inf or NaN operand
 * makes every output of its row or column NaN on the tensor-core path (its
 * remainder part is Inf - Inf); the FFMA kernel follows IEEE. */
int sgemm_f32(const float* A, const float* B, float* C,
              int M, int N, int K, float alpha, float beta, cudaStream_t stream);

int sgemm_f32_ld(const float* A, const float* B, float* C,
                 int M, int N, int K, int lda, int ldb, int ldc,
                 float alpha, float beta, cudaStream_t stream);

/*
 * Host-buffer forms: A, B, C are HOST pointers (pinned memory gives the
 * fastest copies and lets them overlap; pageable memory works).  On a
 * library-owned copy-in stream the call copies B, then A and C (C when
 * beta != 0 or ldc > N) in blocks of rows to library-owned device buffers;
 * each block is computed on `stream` as soon as it is in, and copied back on
 * a library-owned copy-back stream as soon as it is computed (M >= 2048: four
 * blocks of a multiple of 256 rows; else one), so copies in, GEMMs and copies
 * back of different blocks overlap.  The copies in wait for the work already
 * queued on `stream`; the call returns after `stream` has synchronised with
 * the last copy back.  A blocked call
 * may round differently in the last bit from the device form on the same
 * operands (each block is its own GEMM, with its own tile schedule).  Calls
 * are serialised process-wide (they share the staging buffers).  The device
 * buffers are kept for reuse and freed by gemm_release().
 */
int gemm_f16_host(const uint16_t* A, const uint16_t* B, uint16_t* C,
                  int M, int N, int K, int lda, int ldb, int ldc,
                  float alpha, float beta, cudaStream_t stream);

int sgemm_f32_host(const float* A, const float* B, float* C,
                   int M, int N, int K, int lda, int ldb, int ldc,
                   float alpha, float beta, cudaStream_t stream);

/*
 * Allocation-free split-K GEMM.  The paper has no counterpart: this entry
 * point is a service of this library.  Same computation and conventions as
 * gemm_f16_ld, always through the split-K path, for callers that must not
 * allocate device memory while they run (cudaMalloc may synchronise the
 * device and may fail; some callers must draw every allocation from their
 * own planner or a budget fixed at start-up).  The fp32 partial sums live in
 * a fixed device array of GEMM_STATIC_SCRATCH_BYTES that every GPU loading
 * this library holds until the library is unloaded; this call itself never
 * allocates or frees.
 *   splits   number of K slices, 0 = automatic (enough to fill the SMs)
 *   returns  GEMM_ERR_ARG, with nothing enqueued, when
 *            slices * M * roundup(N, 4) * 4 bytes exceed the array
 *            (e.g. M=16, N=8192: up to 16 slices; M=8192, N=64: up to 4)
 * The first call on each device (with that device current) looks up the
 * array's device address; make it before any stream capture.  All calls share
 * the array and it keeps the previous call's contents (nothing needs to start
 * at zero); calls whose kernels overlap on the GPU race on it.
 */
#define GEMM_STATIC_SCRATCH_BYTES (8u << 20)
int gemm_f16_splitk_noalloc(const uint16_t* A, const uint16_t* B, uint16_t* C,
                            int M, int N, int K, int lda, int ldb, int ldc,
                            float alpha, float beta, int splits, cudaStream_t stream);

/*
 * L2 flush used between timed replays ("advanced SGEMM" page, benchmark
 * section: a cudaMemsetAsync of an L2-sized buffer before each replay).
 * Enqueues a memset of a library-owned buffer of `bytes` bytes (0 = twice
 * the device's L2 size) on `stream`.
 */
int gemm_l2_flush(size_t bytes, cudaStream_t stream);

/*
 * Kernel path selection, for tests and benchmarks.  0 = automatic (default);
 * 1 = tensor-memory-accelerator operand loads; 2 = predicated element loads
 * (the path taken when strides or pointers are not 16-byte aligned);
 * 3 = split-K (every tile cut into equal K slices); 4 = (fp32 only) FFMA
 * kernel with predicated scalar loads; 5 = whole tiles only (no stream-K, no
 * splitting of the last wave); 6 = no CTA pairs (one
 * CTA per 128-row tile); 7 = (fp32) FFMA kernel only, no tensor cores;
 * 8 = (fp32) the 3xTF32 tensor-core kernel (tf32 parts) whatever the shape; 9 = the last,
 * partial wave of tiles cut into two equal K slices (instead of two
 * half-width units); 10 = stream-K over the last waves of tiles (k-block
 * ranges shared out evenly); 11 = stream-K over all tiles, one CTA per worker
 * (chosen automatically for few tiles when it is expected to beat half-width
 * units); 12 / 13 = CTA-pair tiles 224 / 192 columns wide for a half C
 * (whole tiles; the automatic choice keeps 256); 14 = the tiles of the last,
 * partial wave shared out as stream-K pieces, each worker taking the piece
 * that starts a tile first and the piece that ends a tile last.  The
 * automatic choice (fp16 and fp32 tensor-core kernels alike; for fp32 when K
 * holds at least 6 accumulation chunks) cuts the tiles of a last, partial
 * wave that fills at most half the workers into two K slices each, the first slice one worker's
 * first unit and the second another worker's last (it adds the first one's
 * partial sums, published long before); else it runs them as half-width
 * units; 15 = half-width units for them; 16 = (fp32) the 3xFP16 tensor-core
 * kernel whatever the shape (8 = 3xTF32); 17 = 64-row tiles (tcgen05.mma with
 * M = 64) for a half C at most 64 columns wide with TMA loads and epilogue,
 * whole-K tiles in one wave (at most one per SM; the automatic choice keeps
 * 128-row tiles, which run as fast: a CTA's time goes with its k-blocks, not
 * with its rows).
 * A forced path that cannot serve a call (e.g. TMA
 * loads on unaligned operands) falls back to the automatic choice.  Process
 * wide; returns the previous value, or GEMM_ERR_ARG for an unknown value.
 */
int gemm_force_path(int path);

/* k-blocks (of 64 elements of K) per stage of the operand ring of the
 * half-precision tensor-core kernels: 0 = automatic (two for one wave of
 * whole 64-wide tiles with at least 16 k-blocks, else one), 1, or 2 (taken
 * only where the kernel has that form: 64-wide single-CTA tiles and 256-wide
 * CTA pairs, with TMA loads and the TMA epilogue).  Results do not depend on
 * it.  For tests and benchmarks; process wide; returns the previous value, or
 * GEMM_ERR_ARG for an unknown value. */
int gemm_stage_kblocks(int kblocks);

/* Fixes the split count of the split-K path (0 = automatic).  On the fp32
 * tensor-core path it also sets the K slices of few-tile shapes: 1 keeps
 * whole-K units, > 1 asks for that many slices (fewer when a slice would be
 * empty).  Process wide; returns the previous value. */
int gemm_force_splits(int splits);

/* Limit, in nanoseconds, of every wait inside the kernels (0 = default of
 * two seconds).  Returns the previous value. */
long long gemm_set_wait_limit_ns(long long ns);

/*
 * Synchronises the device and returns, then clears, the device status word:
 * GEMM_OK, or GEMM_ERR_TIMEOUT if a kernel abandoned a wait since the last
 * call.
 */
int gemm_debug_status(void);

/*
 * Failure-detection probe: launches one thread that waits, through the same
 * bounded wait every kernel of the library uses, on an mbarrier that nothing
 * ever arrives on.  After `limit_ns` nanoseconds the wait gives up, records
 * GEMM_ERR_TIMEOUT in the device status word and the kernel returns normally
 * (no trap; the context stays usable), so the next gemm_debug_status() call
 * returns GEMM_ERR_TIMEOUT.  limit_ns <= 0 is GEMM_ERR_ARG.  Asynchronous.
 */
int gemm_debug_wait_probe(long long limit_ns, cudaStream_t stream);

/* Describes the path the last call on this thread took (static string). */
const char* gemm_last_path(void);

/*
 * The stream-K plan the half-precision path would use for `tiles` output
 * tiles of `kb` k-blocks on at most `slots` concurrent workers (CTAs or CTA
 * pairs); `all_tiles` = 1 asks for the few-tiles form (every tile's k-blocks
 * shared out), 2 for the tail form (the tiles of the last, partial wave
 * shared out over at most 4 workers per tile, no range longer than a tile),
 * 0 for the last two waves.  Writes out[0] = whole tiles computed first, out[1] = tiles
 * whose k-blocks are shared out (0 = no stream-K), out[2] = workers sharing
 * them, out[3] = most pieces one tile can be cut into.  Worker w of W takes
 * k-blocks [w*I/W, (w+1)*I/W) of the I = out[1]*kb shared ones.  Host-only
 * (no device call); returns GEMM_OK, or GEMM_ERR_NULL for a null `out`.
 */
int gemm_plan_stream_k(long long tiles, long long slots, int kb, int all_tiles, long long* out);

/*
 * The K-slice plan of the fp32 tensor-core path for `tiles` 256x256 output
 * tiles of `kb` planning k-blocks (128 bytes of K per row: 32 floats, or 64
 * halves for 3xFP16; the kernel runs each as two 64-byte k-blocks) on `pairs`
 * concurrent CTA pairs, as the automatic choice makes it (`forced_slices` > 1
 * plays gemm_force_splits).  Writes out[0] = slices per tile (1 = whole-K
 * units, no slicing) and out[1] = planning k-blocks per slice (a multiple of
 * 4; the last slice may be shorter).  Host-only; returns GEMM_OK, GEMM_ERR_NULL for a null `out`, or
 * GEMM_ERR_ARG for a negative argument.
 */
int gemm_plan_tf32_slices(long long tiles, long long pairs, int kb, int forced_slices,
                          long long* out);

/* Number of kernels the library has launched in this process (all threads,
 * all devices; launches that failed are not counted).  Nothing else --
 * memset, copies, L2 flushes -- is counted. */
long long gemm_launch_count(void);

/* Text for a return code (static string). */
const char* gemm_strerror(int code);

/* Frees every library-owned device buffer on every device (workspace,
 * host-form staging buffers, L2-flush buffer).  Synchronises each device
 * that has such buffers. */
int gemm_release(void);

#ifdef __cplusplus
}
#endif

#endif /* GB300_GEMM_H */
