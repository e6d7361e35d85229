/*
 * sptgemm.h -- C ABI of the software-pipelined tiled GEMM library for
 * NVIDIA GB300 (sm_103a).
 *
 * The operation is the tiled matrix multiply C = A * B of "Hiding Memory
 * Latency in CUDA: Asynchronous Loads and Software Pipelines" (opening
 * section: load A and B tiles, stage them in shared memory, multiply on the
 * tensor cores, advance to the next K tile), software-pipelined so that the
 * load of K-tile k+1 overlaps the multiply-accumulate of K-tile k (same
 * page, sections 1, 5 and 11; "Pipeline GPU Kernel", Step 3). Pipelining
 * reorders loads and leaves the arithmetic alone ("Pipeline GPU Kernel",
 * Step 5 item 4): the result is the plain product.
 *
 * Layouts (all dense, leading dimensions implied by the shape):
 *   A  row-major    M x K : element (i, k) at A[i*K + k]
 *   B  column-major K x N : element (k, j) at B[j*K + k]
 *   C  row-major    M x N : element (i, j) at C[i*N + j]
 *
 * Ownership: the caller owns A, B and C, which are device pointers (any
 * allocation the CUDA runtime can address on the current device). The
 * library keeps no pointer past a call. It owns one cached scratch area per
 * (device, stream) for the paths that need one (int8 operand conversion,
 * split-K partial sums), grown on demand and released at unload.
 *
 * Streams: every call is asynchronous on `stream` (a cudaStream_t; NULL is
 * the legacy default stream) and never synchronizes. Inputs must stay valid
 * and C untouched by others until the stream reaches the call.
 *
 * Errors: functions return an int status, 0 on success, a negative
 * SPTG_ERR_* code otherwise. No call aborts the process and there is no CPU
 * fallback: on a machine without an sm_103 device the call fails.
 */
#ifndef SPTGEMM_H
#define SPTGEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Input/output element pairs. Float inputs accumulate in fp32; int8 inputs
 * accumulate exactly and return int32. */
typedef enum {
  SPTG_F16_F32 = 0,   /* binary16 A, B -> fp32 C                 */
  SPTG_F16_F16 = 1,   /* binary16 A, B -> binary16 C (RN-even)   */
  SPTG_S8_S32 = 2,    /* int8 A, B -> int32 C, bit-exact while the
                         sum fits int32 (any inputs for K < 131072);
                         beyond, it wraps modulo 2^32               */
  SPTG_BF16_BF16 = 3, /* bfloat16 A, B -> bfloat16 C (RN-even)   */
  SPTG_BF16_F32 = 4,  /* bfloat16 A, B -> fp32 C                 */
  /* range markers, not dtypes: they make sptg_dtype span every 32-bit int,
     so any value a caller passes is representable and is rejected with
     SPTG_ERR_ARG unless it names one of the pairs above */
  SPTG_DTYPE_RANGE_MIN_ = -2147483647 - 1,
  SPTG_DTYPE_RANGE_MAX_ = 2147483647
} sptg_dtype;

enum {
  SPTG_OK = 0,
  SPTG_ERR_ARG = -1,         /* null pointer with a nonzero extent, negative or
                                too-large dimension, unknown dtype or option   */
  SPTG_ERR_ALIGN = -2,       /* a pointer not 16-byte aligned, or a row pitch
                                (K*sizeof(in), N*sizeof(out)) not a multiple
                                of 16 bytes, as the tensor-copy engine needs  */
  SPTG_ERR_UNSUPPORTED = -3, /* no CUDA device of compute capability 10.3    */
  SPTG_ERR_LAUNCH = -4,      /* a CUDA runtime error; see sptg_last_error()  */
  SPTG_ERR_TIMEOUT = -5,     /* a kernel gave up a bounded wait (reported by
                                sptg_device_error); C's contents are then
                                unspecified                                   */
  SPTG_ERR_NOMEM = -6,       /* scratch memory could not be allocated        */
  SPTG_ERR_CONFIG = -7       /* a forced configuration does not fit          */
};

/*
 * C = A * B.  M, N, K >= 0.  M == 0 or N == 0: nothing is done.  K == 0:
 * C is set to zero (the empty sum).  Shapes need not be multiples of any
 * tile: edges are zero-filled on load and clipped on store.
 *
 * Alignment: A, B, C 16-byte aligned; K * sizeof(input) and
 * N * sizeof(output) multiples of 16 bytes.  Otherwise SPTG_ERR_ALIGN.
 */
int sptg_gemm(int64_t M, int64_t N, int64_t K, sptg_dtype dtype,
              const void* A, const void* B, void* C, void* stream);

/* Kernel selection for sptg_gemm_ex; fields left at 0 mean "choose". */
typedef struct {
  int kernel;   /* 0 auto, 1 square, 2 skinny swap-AB with stream-K split,
                   3 skinny swap-AB with the K split across a cluster of
                   CTAs (splits = cluster size, 1, 2 or 4), 4 skinny
                   (M <= 64, float) with one CTA per strip of output columns
                   over the whole of K (bn = strip width), 5 skinny swap-AB
                   (M <= 256, float) on CTA pairs with the 2-SM MMA over the
                   whole of K (bn = output columns per CTA)                  */
  int bn;       /* square: tile columns, 112 to 256 in steps of 16 for
                   float types (int8: 128, 160, 192, 224 or 256), or 512 for
                   float CTA pairs; skinny column strips (kernel 4):
                   a multiple of 8 from 8 to 256; skinny CTA pairs (kernel
                   5): a multiple of 8 from 8 to 128                         */
  int stages;   /* shared-memory ring depth (1 = synchronous load/compute)  */
  int splits;   /* square: cap on persistent workers; skinny stream-K: CTAs
                   sharing the work (0 = SM count); skinny cluster: cluster
                   size                                                      */
  int timeout_ms; /* bounded-wait limit inside the kernel (0 = default 2000) */
  int inject_stall; /* test hook: 1 makes the producer withhold one k-tile so
                       the consumer's bounded wait runs out; 0 = off          */
  int cta_pair; /* square: 0 choose, 1 one CTA (128-row tiles), 2 a CTA pair on
                   two SMs with the 2-SM MMA (256-row tiles); every CTA
                   copies its own operand tiles (no multicast copies)       */
  int no_overlap; /* 1: launch without programmatic dependent launch (the
                     kernel then starts only after the previous one ends)    */
  void* trace;  /* optional device buffer of SPTG_TRACE_WORDS uint64 (8-byte
                   aligned, zeroed by the caller): word [8*cta + e] is the
                   %globaltimer ns of event e of CTA cta (first 1024 CTAs):
                   0 set-up done, 1 first copy issued, 2 first stage full at
                   the MMA issuer, 3 last copy issued, 4 last MMA committed,
                   5 epilogue done, 6 exit, 7 last split-K reduction; then
                   for CTA 0, the issue time of K-tiles 0..63 (words 8192..)
                   and the time the MMA issuer found each full (8256..);
                   NULL = off                                               */
  int stream_k; /* square kernel: 0 choose (the tiles of a partial last
                   round are cut along K over all workers), 1 never, 2 every
                   tile (a test setting)                                    */
} sptg_config;

#define SPTG_TRACE_WORDS (8 * 1024 + 2 * 64)

/* sptg_gemm with an explicit configuration (NULL = sptg_gemm). */
int sptg_gemm_ex(int64_t M, int64_t N, int64_t K, sptg_dtype dtype,
                 const void* A, const void* B, void* C, void* stream,
                 const sptg_config* cfg);

/*
 * sptg_gemm_ex on matrices inside larger row-pitched buffers ("Pipeline GPU
 * Kernel", pitfalls: boundary handling; the tiles are read and written
 * through the row pitch, never past a row's K or N elements).
 *
 *   lda  elements between rows of A        (>= K)
 *   ldb  elements between the K-long columns of B, i.e. rows of the N x K
 *        array Bcm                          (>= K)
 *   ldc  elements between rows of C        (>= N)
 *
 * Besides the alignment rules of sptg_gemm (which still apply to K and N),
 * lda * sizeof(in), ldb * sizeof(in) and ldc * sizeof(out) must be multiples
 * of 16 bytes (SPTG_ERR_ALIGN), and each leading dimension must be below
 * 2^31 (SPTG_ERR_ARG). Elements between N and ldc of a row of C are never
 * written. lda = ldb = K and ldc = N give sptg_gemm_ex.
 */
int sptg_gemm_strided(int64_t M, int64_t N, int64_t K, sptg_dtype dtype,
                      const void* A, int64_t lda, const void* B, int64_t ldb,
                      void* C, int64_t ldc, void* stream, const sptg_config* cfg);

/*
 * sptg_gemm_ex on HOST buffers: A (M x K), B (the N x K array Bcm) and C
 * (M x N), dense, in host memory. The call enqueues on `stream` the copies of
 * A and B to device buffers the library owns (one set per device and stream,
 * grown on demand and freed in stream order), the product, and the copy of
 * C back to the host, and returns without waiting. The caller keeps A, B and
 * C alive and leaves C alone until the stream has reached this point.
 * Page-locked (pinned) host memory makes the copies asynchronous; pageable
 * memory works but the driver then stages it and the call may block. The
 * pitch rules of sptg_gemm apply (SPTG_ERR_ALIGN); the pointers themselves
 * need no alignment. The pages have no counterpart: this is the call a
 * caller whose data lives in host memory makes, and bench.py's end-to-end
 * measurement goes through it.
 */
int sptg_gemm_host(int64_t M, int64_t N, int64_t K, sptg_dtype dtype,
                   const void* A, const void* B, void* C, void* stream,
                   const sptg_config* cfg);

/*
 * The software-pipelined ring on its own: out[i] = alpha * in[i] for
 * i < n, binary32, one rounding per element. This is the minimal working
 * example of "Hiding Memory Latency in CUDA: Asynchronous Loads and Software
 * Pipelines" (section 8: a vector streamed through a multi-stage
 * shared-memory ring and scaled by two), here for any alpha; it measures the
 * copy pipeline against memory bandwidth.
 *
 * in and out are device pointers, 16-byte aligned (else SPTG_ERR_ALIGN),
 * and may be the same buffer (in place); they must not otherwise overlap.
 * n >= 0 of any size (n == 0: nothing). Asynchronous on `stream`.
 */
int sptg_stream_scale(int64_t n, float alpha, const float* in, float* out, void* stream);

/* sptg_stream_scale with the timeout_ms, inject_stall, no_overlap and trace
 * fields of a configuration (the others are ignored; NULL = defaults). */
int sptg_stream_scale_ex(int64_t n, float alpha, const float* in, float* out, void* stream,
                         const sptg_config* cfg);

/* Static text for a status code. */
const char* sptg_status_string(int status);

/* Text of the last CUDA runtime error seen by this thread ("" if none). */
const char* sptg_last_error(void);

/* Writes "kernel=... bm=... bn=... bk=... stages=... ..." for the last call
 * made by this thread into buf (NUL-terminated, truncated to len).
 * Returns the length the full text needs. */
int sptg_last_config(char* buf, size_t len);

/* Synchronizes `stream`, then reads and clears the current device's error
 * word written by timed-out waits. Returns SPTG_OK or SPTG_ERR_TIMEOUT
 * (or SPTG_ERR_LAUNCH if synchronization itself failed). */
int sptg_device_error(void* stream);

/*
 * Allocation-free variant of the skinny (M <= 64) kernel.
 *
 * This call has no counterpart in the paper. It exists for callers that
 * cannot let a library allocate device memory: a serving process that reserves the GPU's
 * memory for its own pool up front (a library cudaMalloc would then fail or
 * fragment that pool), and latency-critical code that cannot accept the
 * device-wide synchronisation a cudaMalloc or cudaFree may imply.
 *
 * It computes exactly what sptg_gemm computes for the same arguments, with
 * the same kernel, but keeps its split-K partial sums and arrival counters in
 * one fixed array compiled into the library (SPTG_NOALLOC_PARTIAL_BYTES +
 * SPTG_NOALLOC_COUNTER_BYTES of device memory, held on every GPU that loads
 * the library until the process exits). It calls no cudaMalloc, cudaFree or
 * other allocating routine.
 *
 *  - dtype: the float pairs only (not SPTG_S8_S32), and M <= 64; otherwise
 *    SPTG_ERR_CONFIG. A, B, C, stream, alignment and return codes as for
 *    sptg_gemm.
 *  - A shape whose split needs more partial-tile bytes (column tiles of 128 x
 *    contributing CTAs x 32 KiB) or counter bytes than the fixed array holds
 *    is rejected with SPTG_ERR_CONFIG; sptg_last_error() gives the sizes.
 *  - The first call on a device looks up the array's device address (with
 *    that device current); make that first call before any stream capture.
 *  - Every call uses the same array, which keeps the last call's partial
 *    sums and counters. Each call tags the counters it uses with a new call
 *    number, so whatever an earlier call left there (even one whose kernel
 *    gave up a wait) is never taken for this call's. Calls whose kernels
 *    overlap on the GPU (two streams, or two threads) race on the array:
 *    serialise them.
 */
#define SPTG_NOALLOC_PARTIAL_BYTES (8u << 20)
#define SPTG_NOALLOC_COUNTER_BYTES (64u << 10)
int sptg_gemm_skinny_noalloc(int64_t M, int64_t N, int64_t K, sptg_dtype dtype,
                             const void* A, const void* B, void* C, void* stream);

/* Library ABI version (major*100 + minor). */
int sptg_version(void);

/*
 * The square kernel's plan for a shape, computed on the host alone (no
 * device is touched), for a GPU of `sm_count` SMs: the tile shape and the
 * schedule sptg_gemm_ex would choose with configuration `cfg` (NULL =
 * defaults), before any fallback for a missing ring depth. On success
 * out[0..6] = tile columns BN, tile mode (0 one CTA, 1 CTA pair), tiles of
 * the schedule, workers (CTAs or pairs), tiles cut along K (stream-K),
 * workers sharing them, and the most contributors one cut tile can have. The
 * worker count assumes every SM holds one CTA; the library itself asks the
 * device how many pairs fit. SPTG_ERR_ARG for a non-positive dimension, fewer
 * than 2 SMs, an unknown dtype or an invalid field; SPTG_ERR_CONFIG when a
 * forced width does not exist for the dtype and pairing.
 */
int sptg_plan_square(int64_t M, int64_t N, int64_t K, sptg_dtype dtype, int sm_count,
                     const sptg_config* cfg, int* out);

/*
 * The whole kernel choice sptg_gemm_ex would make for a shape with
 * configuration `cfg` (NULL = defaults) on a GPU of `sm_count` SMs, computed
 * on the host alone (no device is touched). On success out[0..5] = kernel
 * (1 square, 2 skinny stream-K, 3 skinny cluster split, 4 skinny column
 * strips, 5 skinny CTA pairs -- the sptg_config.kernel numbering), tile width
 * (square: BN; 2 and 3: 128; 4: strip width; 5: output columns per CTA),
 * CTAs launched, CTAs per cluster (1, 2 or 4), the rows of A on a skinny
 * MMA's N side (64, 128 or 256; 0 for the square kernel) and, for the square
 * kernel, the tiles cut along K. Assumes every SM holds one CTA and every
 * cluster of the chosen size fits the GPU (the library asks the device; a
 * cluster split it cannot place goes to stream-K or the square kernel).
 * Errors as for sptg_plan_square; SPTG_ERR_CONFIG when a forced kernel does
 * not take the shape.
 */
int sptg_plan(int64_t M, int64_t N, int64_t K, sptg_dtype dtype, int sm_count,
              const sptg_config* cfg, int* out);

#ifdef __cplusplus
}
#endif

#endif /* SPTGEMM_H */
