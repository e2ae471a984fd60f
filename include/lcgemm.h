/*
 * lcgemm -- half-precision GEMM for GB300 (sm_103a): plain tiled GEMM and the
 * low-complexity (LCMA / Strassen) path, behind a plain C ABI.
 *
 * Operation (every entry point): C = A . B with FP16 or BF16 inputs, FP32
 * accumulation and one round-to-nearest-even cast to the input type.
 *   - plain:     one persistent tensor-core kernel.
 *   - strassen1: one-level Strassen -- 7 block products instead of 8, the A and
 *                B sub-blocks combined before the products and the products
 *                recombined into the four quadrants of C (FalconGEMM write-up,
 *                hyper.ai news 54396, section "从 Strassen 出发"; the
 *                combine / product / recombine pipeline and its fusion are in
 *                section "从 LCMA 到 FalconGEMM").
 *   - strassen2: two-level Strassen, 49 block products over a 4x4 block grid
 *                (same section: 49 instead of 64 block multiplications); the
 *                seven outer products each run as one pass of the fused
 *                one-level kernel over the inner blocks, and the outer level
 *                is combined in FP32 before the one cast.
 *   - auto:      a roofline-style cost model picks one of the above per shape
 *                (section "从缓存重排到 Cost Model").
 * The one-level scheme is the textbook Strassen (1969) formulas:
 *   M1=(A11+A22)(B11+B22) M2=(A21+A22)B11 M3=A11(B12-B22) M4=A22(B21-B11)
 *   M5=(A11+A12)B22 M6=(A21-A11)(B11+B12) M7=(A12-A22)(B21+B22)
 *   C11=M1+M4-M5+M7 C12=M3+M5 C21=M2+M4 C22=M1-M2+M3+M6
 *
 * Layouts (element type = dtype for A, B and C):
 *   A : row-major M x K, element (i,k) at A[i*lda + k], lda >= K
 *   B : the K x N operand stored column-major, element (k,j) at B[j*ldb + k],
 *       ldb >= K (both operands are K-contiguous)
 *   C : row-major M x N, element (i,j) at C[i*ldc + j], ldc >= N
 *
 * Alignment (the tensor-memory-access engine reads A and B): A, B and C must
 * be 16-byte aligned and lda, ldb, ldc multiples of 8 elements.  There is no
 * fallback path: misaligned calls fail with LCGEMM_ERR_ALIGN.
 *
 * Errors: every entry point returns an int, 0 = LCGEMM_OK, negative on
 * failure; nothing is thrown across the ABI.  Argument checks happen on the
 * host before anything is launched.  Device-side waits are bounded; a wait
 * that gives up records LCGEMM_ERR_TIMEOUT, which the NEXT lcgemm_run on the
 * handle or lcgemm_sync_status returns (and clears).
 *
 * Numerics: NaN and Inf propagate per IEEE with no checks on the hot path.
 * In the Strassen paths an Inf in one block can turn into NaN in other
 * blocks (Inf - Inf in the operand sums or the recombination).
 *
 * Threading: a handle may be used by one host thread at a time, and runs
 * through one handle must not overlap on different streams (they share the
 * handle's workspace).
 *
 * CUDA graphs: lcgemm_run and lcgemm_run_epilogue may be captured into a graph
 * (stream capture) and the graph replayed, provided each captured shape has
 * run once on the handle outside the capture, so that the workspace and the
 * other handle-owned buffers already have their size (a call that would grow
 * one returns LCGEMM_ERR_CAPTURE and captures nothing).  Device pointers and
 * sizes are fixed in the graph; replays read the buffers' current contents.
 * lcgemm_run_host cannot be captured.
 */
#ifndef LCGEMM_H
#define LCGEMM_H

#include <stdint.h>

#if defined(__GNUC__)
#define LCGEMM_API __attribute__((visibility("default")))
#else
#define LCGEMM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct lcgemm_ctx* lcgemm_t;

/* element type of A, B and C */
enum { LCGEMM_F16 = 0, LCGEMM_BF16 = 1 };

/* algorithm */
enum {
  LCGEMM_PLAIN = 0,             /* persistent tiled GEMM                                  */
  LCGEMM_STRASSEN1 = 1,         /* one-level Strassen: combine pre-pass + fused products  */
  LCGEMM_STRASSEN2 = 2,         /* two-level Strassen (49 products, fused hierarchically) */
  LCGEMM_AUTO = 3,              /* cost model chooses among the three above               */
  LCGEMM_STRASSEN1_UNFUSED = 4  /* ablation: combine, 7 products written to HBM in FP32,
                                   separate recombination kernel (the basic pipeline)     */
};

/* status codes */
enum {
  LCGEMM_OK = 0,
  LCGEMM_ERR_ARG = -1,          /* null pointer, negative size, ld too small, bad enum    */
  LCGEMM_ERR_ALIGN = -2,        /* pointer not 16-byte aligned or ld not a multiple of 8  */
  LCGEMM_ERR_UNSUPPORTED = -3,  /* shape outside an entry point's range (allocation-free
                                   entry point on dimensions it cannot split)             */
  LCGEMM_ERR_ALIAS = -4,        /* C overlaps A or B                                      */
  LCGEMM_ERR_CUDA = -5,         /* a CUDA runtime/driver call or launch failed            */
  LCGEMM_ERR_TIMEOUT = -6,      /* a bounded device-side wait gave up (earlier launch)    */
  LCGEMM_ERR_NOMEM = -7,        /* workspace or staging allocation failed                 */
  LCGEMM_ERR_TOO_LARGE = -8,    /* problem exceeds lcgemm_strassen1_noalloc's fixed scratch */
  LCGEMM_ERR_CAPTURE = -9       /* the stream is capturing a CUDA graph and the call would have
                                   to grow a handle buffer (or it is lcgemm_run_host)       */
};

/* options for lcgemm_set_option */
enum {
  LCGEMM_OPT_WAIT_TIMEOUT_US = 1,  /* bound on every device-side wait, microseconds (default 2000000) */
  LCGEMM_OPT_GROUP_ORDER = 2,      /* one-level Strassen on CTA pairs: 1 (default) every pair walks
                                      its Groups' seven products in one order, so a wave streams one
                                      product's operands at a time (only the split tail mixes);
                                      0: odd pairs take another order, so every wave mixes two product
                                      types (an ablation; the result is the same bit for bit)        */
  LCGEMM_OPT_SPLIT = 3,            /* 1: split tail Groups across two CTAs (default), 0: off          */
  LCGEMM_OPT_MAX_CTAS = 4,         /* cap on the persistent grid (default 0 = one CTA per SM)         */
  LCGEMM_OPT_PEAK_GFLOPS = 5,      /* cost model: dense FP16/BF16 tensor peak, GFLOP/s                */
  LCGEMM_OPT_HBM_GBPS = 6,         /* cost model: HBM bandwidth, GB/s                                 */
  LCGEMM_OPT_DEBUG_DROP_SIGNAL = 7, /* test hook: a split Group's partner (Strassen) or a split tail
                                      tile's second K half (plain CTA-pair kernel) never signals, so
                                      the waiting side's bounded wait runs out (no fault, no hang)   */
  LCGEMM_OPT_PLAIN_KERNEL = 8,      /* plain GEMM kernel: 0 choose (default: the GEMV for M <= 2; CTA
                                      pairs when M, N > 128 and their 256x256 tiles fill a quarter of
                                      the pairs; else single-CTA tiles with split-K), 1 single-CTA
                                      128x256 tiles, 2 CTA-pair (cta_group::2) 256x256 tiles, 3 the
                                      stream-K skinny kernel (M <= 256), 4 the CUDA-core GEMV
                                      (M <= 4), 5 CTA-pair 256x512 tiles (0 takes them for long main
                                      loops without a fused epilogue); for 3 and 4 larger M choose   */
  LCGEMM_OPT_LCMA_KERNEL = 9,       /* fused one-level Strassen kernel: 0 choose (default), 1
                                      single-CTA 128x128 Groups, 2 CTA-pair 256x256 Groups           */
  LCGEMM_OPT_PDL = 10               /* 1 (default): launch the GEMM kernels (plain tiles, GEMV,
                                      skinny, Strassen products) as programmatic dependents of the
                                      kernel before them: their prologue (barriers, tensor memory,
                                      descriptors) overlaps that kernel's tail and they touch no
                                      global memory before it completes; 0: plain stream order.
                                      The GEMM kernels let their own dependents start early: a
                                      kernel the caller launches after a run with programmatic
                                      stream serialization must wait for its prerequisite grid
                                      (cudaGridDependencySynchronize) before reading C; ordinary
                                      launches, copies and events are ordered as usual.            */
};

/* `device` value of a planning handle (see lcgemm_create). */
#define LCGEMM_PLANNING_DEVICE (-1)

/*
 * Create a handle bound to CUDA device `device`.  Allocates only a few bytes
 * (the mapped error word); the Strassen workspace grows on first use.
 * Reads environment overrides LCGEMM_PEAK_GFLOPS and LCGEMM_HBM_GBPS.
 * Returns LCGEMM_ERR_ARG for a null `out` or an invalid device.
 * device = LCGEMM_PLANNING_DEVICE creates a planning handle that makes no CUDA
 * call at all: it answers lcgemm_select / lcgemm_estimate for a GB300 (152
 * SMs; LCGEMM_OPT_MAX_CTAS lowers that) and rejects every run with
 * LCGEMM_ERR_ARG.
 */
LCGEMM_API int lcgemm_create(lcgemm_t* out, int device);

/* Synchronise the device, free the workspace and the handle.  Null is a no-op. */
LCGEMM_API int lcgemm_destroy(lcgemm_t h);

/*
 * C = A . B, asynchronous on `cuda_stream` (a cudaStream_t; NULL = legacy
 * default stream).  A, B, C are device pointers owned by the caller; C is
 * overwritten (beta = 0).  M = 0 or N = 0 is a no-op; K = 0 writes zeros.
 * Every algorithm takes any shape.  Strassen splits M and N into 2 (one level)
 * or 4 (two levels) blocks and K into blocks of a multiple of 8; when a
 * dimension does not divide (M, N by 2 resp. 4, K by 16 resp. 32), A and B
 * are first copied into zero-padded buffers owned by the handle (the padding
 * multiplies to zero) and only C's M x N elements are written.
 */
LCGEMM_API int lcgemm_run(lcgemm_t h, int64_t M, int64_t N, int64_t K,
               const void* A, int64_t lda, const void* B, int64_t ldb,
               void* C, int64_t ldc, int dtype, int algo, void* cuda_stream);

/*
 * Same operation on HOST buffers (same layouts): copies A and B to device
 * staging buffers owned by the handle, runs lcgemm_run, copies C back, all
 * enqueued on `cuda_stream`.  The call returns once the work is enqueued;
 * synchronise the stream before reading C.  Page-locked host memory gives
 * asynchronous copies; pageable memory works but the copies block.
 */
LCGEMM_API int lcgemm_run_host(lcgemm_t h, int64_t M, int64_t N, int64_t K,
                    const void* A, int64_t lda, const void* B, int64_t ldb,
                    void* C, int64_t ldc, int dtype, int algo, void* cuda_stream);

/* activation of the fused epilogue (lcgemm_epilogue.act) */
enum {
  LCGEMM_ACT_NONE = 0,
  LCGEMM_ACT_RELU = 1,       /* x > 0 ? x : +0                                             */
  LCGEMM_ACT_GELU = 2,       /* x * Phi(x) = x/2 (1 + erf(x / sqrt 2)); Phi from the
                                Abramowitz-Stegun 7.1.26 erfc form (absolute error of the
                                result below 1e-7 |x|)                                     */
  LCGEMM_ACT_GELU_TANH = 3   /* x/2 (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))), hardware
                                tanh approximation (absolute error of tanh below 2^-10)   */
};

/*
 * Element-wise epilogue fused into the GEMM (DeepGEMM tuning blog, kwkr.cn
 * news 553926, section 3.3: bias add and GeLU applied to the finished tile in
 * registers before the single store; "Kernel 与性能", wineandchord.com
 * kernels-performance, section "Fusion": bias + activation, residual add):
 *
 *     C[i,j] = act( sum_k A[i,k] B[k,j] + bias[j] ) + residual[i,j]
 *
 * evaluated in FP32 from the FP32 accumulator and rounded once to dtype.
 *   bias     : device pointer to N values of dtype (one per column of C), or
 *              NULL; 16-byte aligned; must not overlap C.
 *   residual : device pointer to an M x N matrix of dtype, element (i,j) at
 *              residual[i*ldr + j], or NULL; 16-byte aligned, ldr >= N and a
 *              multiple of 8.  It may be C itself (same pointer, ldr == ldc:
 *              an in-place residual add); any other overlap with C is
 *              LCGEMM_ERR_ALIAS.
 *   act      : LCGEMM_ACT_*.
 * Both buffers are owned by the caller and only read.
 */
typedef struct {
  const void* bias;
  const void* residual;
  int64_t ldr;
  int act;
} lcgemm_epilogue;

/*
 * lcgemm_run with a fused epilogue (`ep` NULL or all-empty: plain lcgemm_run).
 * Every algorithm applies it where an element of C becomes final: the plain
 * kernels after the K loop (or the split-K / split-tail sum), the Strassen
 * kernels after the quadrant recombination.  K = 0 gives act(bias) + residual.
 * Errors: those of lcgemm_run, plus LCGEMM_ERR_ARG for an unknown act or a
 * residual with ldr < N, LCGEMM_ERR_ALIGN for a misaligned bias / residual or
 * an ldr that is not a multiple of 8, LCGEMM_ERR_ALIAS as stated above.
 */
LCGEMM_API int lcgemm_run_epilogue(lcgemm_t h, int64_t M, int64_t N, int64_t K,
                        const void* A, int64_t lda, const void* B, int64_t ldb,
                        void* C, int64_t ldc, int dtype, int algo,
                        const lcgemm_epilogue* ep, void* cuda_stream);

/* Algorithm the last successful lcgemm_run on this handle executed (LCGEMM_PLAIN..). */
LCGEMM_API int lcgemm_last_algo(lcgemm_t h);

/* Algorithm LCGEMM_AUTO would execute for this shape (>= 0), or a negative status. */
LCGEMM_API int lcgemm_select(lcgemm_t h, int64_t M, int64_t N, int64_t K, int dtype);

/* Cost-model time estimate in seconds for `algo` on this shape (no launch). */
LCGEMM_API int lcgemm_estimate(lcgemm_t h, int64_t M, int64_t N, int64_t K, int dtype, int algo,
                    double* seconds);

/* Synchronise `cuda_stream`, then return and clear the device error word. */
LCGEMM_API int lcgemm_sync_status(lcgemm_t h, void* cuda_stream);

/* Set an LCGEMM_OPT_* option.  Returns LCGEMM_ERR_ARG for unknown keys or bad values. */
LCGEMM_API int lcgemm_set_option(lcgemm_t h, int option, int64_t value);

/*
 * One-level Strassen (the same kernels as LCGEMM_STRASSEN1) that allocates
 * nothing.  The paper has no counterpart to this entry point.
 *
 * For callers that must not allocate device memory while they run -- a
 * framework whose caching allocator already owns the device's memory, so a
 * cudaMalloc from a library would compete for the same pool, or a service or
 * safety-critical process that only allocates at start-up.  It needs no
 * handle; its scratch (the summed operand blocks) is a fixed 16 MiB array that
 * every device holds from the moment the library is loaded until the process
 * exits, and the call makes no cudaMalloc, cudaFree or other allocating call.
 *
 * Arguments, layouts and alignment rules are those of lcgemm_run; requires M,
 * N even and K a multiple of 16 (else LCGEMM_ERR_UNSUPPORTED); K = 0 fills C
 * with zeros (no kernel but a 2-D memset; A and B are then not read and may be
 * NULL).  The summed operands take
 * 2.5 * K * (M + N) bytes plus alignment; larger problems fail with
 * LCGEMM_ERR_TOO_LARGE (e.g. M = N = K = 1792 fits, 2048 does not).
 * Runs asynchronously on `cuda_stream`.  All calls on a device share the one
 * array: calls that overlap on the GPU (other streams, other threads) race and
 * must be serialised by the caller.  The array keeps the previous call's data.
 * A bounded device-side wait that runs out ends the kernel early (C is then
 * partly written) and sets the array's error word, which stays set until
 * lcgemm_noalloc_status reads and clears it.  The first call on each device
 * looks up the array's device address (with that device current); make that
 * first call before any stream capture.
 */
LCGEMM_API int lcgemm_strassen1_noalloc(int64_t M, int64_t N, int64_t K,
                                        const void* A, int64_t lda, const void* B, int64_t ldb,
                                        void* C, int64_t ldc, int dtype, void* cuda_stream);

/*
 * Status of lcgemm_strassen1_noalloc on the current device, without
 * allocating: synchronises `cuda_stream`, reads the fixed array's error word
 * with a synchronous copy into a host integer, clears it, and returns
 * LCGEMM_ERR_TIMEOUT if any call since the last query had a device-side wait
 * run out (LCGEMM_OK otherwise; LCGEMM_ERR_CUDA if the synchronisation or the
 * copy fails).  The paper has no counterpart to this entry point.
 */
LCGEMM_API int lcgemm_noalloc_status(void* cuda_stream);

/*
 * Test hook: sets the error word of lcgemm_strassen1_noalloc on the current
 * device as a wait that ran out would (synchronous, allocates nothing), so a
 * caller's error handling can be exercised without a device-side failure.
 */
LCGEMM_API int lcgemm_noalloc_debug_fail(void);

/* Static description of a status code (never NULL). */
LCGEMM_API const char* lcgemm_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* LCGEMM_H */
