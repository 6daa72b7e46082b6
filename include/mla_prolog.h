/*
 * mla_prolog.h -- C ABI of the GB300 (sm_103a) Multi-Head Latent Attention prolog.
 *
 * The operation is the one "aclnnMlaPrologV2WeightNz" defines (Function: Formula):
 *
 *   c^Q  = RmsNorm(x . W^DQ)              q^C = c^Q . W^UQ,   q^N = q^C . W^UK  (per head)
 *   q^R  = ROPE(c^Q . W^QR)
 *   c^KV = RmsNorm(x . W^DKV)             k^C = Cache(c^KV)   (written at cacheIndex)
 *   k^R  = Cache(ROPE(x . W^KR))                              (second cache, same slots)
 *   optional: dequantScaleQNope = RowMax(|q^N|) / 127,  q^N = round(q^N / dequantScaleQNope)
 *
 * RmsNorm(x) = gamma * x_i / sqrt(mean(x^2) + eps) (same page, Function: RmsNorm formula);
 * ROPE is the "half" rotation of "aclnnMlaPreprocess" (Constraints: RoPE mode):
 * out = v * cos + rotate_half(v) * sin with rotate_half(v) = [-v[Dr/2:], v[:Dr/2]].
 *
 * The call sequence follows the page's two-phase statement (Function Prototype):
 * first mla_prolog_workspace_size(), then mla_prolog() with a device workspace of at
 * least that many bytes.  There is no executor object: the second call takes the same
 * tensor arguments again.
 *
 * Conventions for every entry point
 *  - Tensors are described by mla_tensor: a DEVICE pointer (CUDA global memory of the
 *    current device), a dtype and a row-major, contiguous shape.  Non-contiguous tensors
 *    are not supported (the page's parameter table marks them "x").
 *  - Ownership: the caller allocates and frees every buffer, including the workspace.
 *    The library allocates no device memory in these calls and keeps no pointer after a
 *    call returns.  kvCache and krCache are updated in place, only at the rows named by
 *    cacheIndex; queryOut, queryRopeOut and dequantScaleQNopeOut are fully overwritten.
 *  - mla_prolog() is asynchronous on `stream` (a cudaStream_t, passed as void*; NULL is
 *    the legacy default stream).  The workspace and all tensors belong to the call until
 *    the stream passes it.  Calls never synchronise the stream and never trap.
 *  - Errors use the codes of the page's return-value table: 161001 a required pointer is
 *    NULL; 161002 a shape, dtype or scenario is outside what the operation accepts;
 *    361001 the CUDA runtime failed (a launch, a device query); 561002 the shapes are valid
 *    for the operation but not for the kernels' tiling (see mla_prolog_workspace_size).
 *  - Problems only the device can see (a cacheIndex value outside [0, BlockNum*BlockSize),
 *    a pipeline wait that gave up) do not fault: the kernels skip the affected writes and
 *    set bits in a status word inside the workspace, read by mla_prolog_device_status().
 */
#ifndef MLA_PROLOG_H
#define MLA_PROLOG_H

#include <stdint.h>

#if defined(__GNUC__)
#define MLA_API __attribute__((visibility("default")))
#else
#define MLA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes ("aclnnMlaPrologV2WeightNz", Return Value table). */
typedef enum {
    MLA_OK = 0,
    MLA_ERR_PARAM_NULLPTR = 161001, /* a required tensor, its data pointer, or an out-pointer is NULL */
    MLA_ERR_PARAM_INVALID = 161002, /* shape / dtype / optional-argument pattern not accepted */
    MLA_ERR_RUNTIME = 361001,       /* a CUDA runtime call failed */
    MLA_ERR_TILING = 561002,        /* valid operation, but outside the kernels' tiling rules */
    MLA_ERR_SCRATCH_LIMIT = 561003  /* mla_prolog_no_alloc only: the call needs more scratch than
                                       MLA_NO_ALLOC_SCRATCH_BYTES (no counterpart on the pages) */
} mla_status;

typedef enum {
    MLA_DT_BF16 = 0,
    MLA_DT_INT8 = 1,
    MLA_DT_FP32 = 2,
    MLA_DT_INT64 = 3,
    MLA_DT_FP16 = 4, /* aclnnMlaPreprocess only */
    MLA_DT_INT32 = 5 /* aclnnMlaPreprocess only */
} mla_dtype;

/* A dense, row-major, contiguous device tensor. */
typedef struct {
    void* data;       /* device address of element 0 (may be NULL only when the tensor is empty) */
    int32_t dtype;    /* an mla_dtype */
    int32_t ndim;     /* 1..4 */
    int64_t shape[4]; /* extents, outermost first; entries past ndim are ignored */
} mla_tensor;

/* Bits of the device status word (mla_prolog_device_status). */
#define MLA_DEV_CACHE_INDEX_RANGE 0x1u /* a cacheIndex value was outside [0, BlockNum*BlockSize):
                                          that token's cache rows were not written */
#define MLA_DEV_WAIT_TIMEOUT 0x2u      /* a kernel pipeline wait exceeded its time limit; the
                                          kernel stopped early and its outputs are incomplete */

/*
 * Phase 1 ("aclnnMlaPrologV2WeightNz", Function Prototype: ...GetWorkspaceSize).
 *
 * Validates every argument and returns in *workspaceSize the bytes of device workspace
 * mla_prolog() needs for these shapes on the current CUDA device.  Argument meaning,
 * shapes and dtypes follow the page's parameter table, with (k, n) weight orientation
 * and ND (row-major) layout for every weight:
 *
 *   tokenX        (T, He) or (B, S, He)        bf16 | int8
 *   weightDq      (He, Hcq)                    bf16 | int8
 *   weightUqQr    (Hcq, N*(D+Dr))              bf16 | int8   column n*(D+Dr)+j: head n, D
 *                                                            columns of W^UQ then Dr of W^QR
 *   weightUk      (N, D, Hckv)                 bf16
 *   weightDkvKr   (He, Hckv+Dr)                bf16 | int8   columns [W^DKV | W^KR]
 *   rmsnormGammaCq (Hcq), rmsnormGammaCkv (Hckv)  bf16
 *   ropeSin, ropeCos (T, Dr) or (B, S, Dr)      bf16          full-width tables
 *   cacheIndex    (T) or (B, S)                int64         flat slot in [0, BlockNum*BlockSize)
 *   kvCache       (BlockNum, BlockSize, 1, Hckv)  bf16 | int8 updated in place
 *   krCache       (BlockNum, BlockSize, 1, Dr)    bf16 | int8 updated in place
 *   dequantScaleX (T, 1) or (T)                fp32   int8 tokenX only
 *   dequantScaleWDq (1, Hcq), dequantScaleWUqQr (1, N*(D+Dr)), dequantScaleWDkvKr (1, Hckv+Dr)
 *                                              fp32   per-output-column weight scales
 *   quantScaleCkv (1, Hckv), quantScaleCkr (1, Dr) fp32   int8 caches: code = round(v * scale)
 *   smoothScalesCq (1, Hcq)                    fp32   int8 weightUqQr only, may be NULL
 *   rmsnormEpsilonCq, rmsnormEpsilonCkv        epsilon of each RmsNorm (1e-5 recommended)
 *   cacheMode                                  NULL or "PA_BSND" (the only mode built)
 *   queryOut      (T, N, Hckv) or (B, S, N, Hckv)  bf16 | int8 (int8 = dynamic quantisation)
 *   queryRopeOut  (T, N, Dr) or (B, S, N, Dr)      bf16
 *   dequantScaleQNopeOut (T, N, 1)             fp32   required iff queryOut is int8
 *
 * Scenarios (the page's scenario table; the optional-argument pattern selects one):
 *   non-quantised:     all bf16, every optional NULL;
 *   partial quant:     weightUqQr int8 + dequantScaleWUqQr (+ smoothScalesCq); with an int8
 *                      kvCache also quantScaleCkv, and krCache int8 with quantScaleCkr;
 *   int8 full quant:   tokenX, weightDq, weightUqQr, weightDkvKr int8 + all four dequant
 *                      scales (+ smoothScalesCq); an int8 kvCache needs quantScaleCkv and
 *                      keeps krCache bf16;
 *   queryOut int8 turns on the dynamic quantisation of q^N in any scenario.
 *
 * Empty inputs (same page, Constraints): T = 0 is valid and does nothing;
 * BlockNum * BlockSize = 0 is valid: queryOut and queryRopeOut are computed and no
 * cache is written.
 *
 * Tiling rules (561002 when broken): He % 8 == 0, Hcq % 64 == 0, D % 8 == 0, Dr even,
 * N*(D+Dr) % 8 == 0, (Hckv+Dr) % 8 == 0, Hckv % 8 == 0, Hcq + Hckv + Dr <= 12288,
 * and Hckv <= 512 when queryOut is int8.
 * Every device pointer must be 16-byte aligned.
 */
MLA_API mla_status mla_prolog_workspace_size(
    const mla_tensor* tokenX, const mla_tensor* weightDq, const mla_tensor* weightUqQr,
    const mla_tensor* weightUk, const mla_tensor* weightDkvKr,
    const mla_tensor* rmsnormGammaCq, const mla_tensor* rmsnormGammaCkv,
    const mla_tensor* ropeSin, const mla_tensor* ropeCos, const mla_tensor* cacheIndex,
    const mla_tensor* kvCache, const mla_tensor* krCache,
    const mla_tensor* dequantScaleX, const mla_tensor* dequantScaleWDq,
    const mla_tensor* dequantScaleWUqQr, const mla_tensor* dequantScaleWDkvKr,
    const mla_tensor* quantScaleCkv, const mla_tensor* quantScaleCkr,
    const mla_tensor* smoothScalesCq,
    double rmsnormEpsilonCq, double rmsnormEpsilonCkv, const char* cacheMode,
    const mla_tensor* queryOut, const mla_tensor* queryRopeOut,
    const mla_tensor* dequantScaleQNopeOut,
    uint64_t* workspaceSize);

/*
 * Phase 2 ("aclnnMlaPrologV2WeightNz", Function Prototype: aclnnMlaPrologV2WeightNz).
 *
 * Same tensor and scalar arguments as phase 1, then a device workspace of at least the
 * size phase 1 returned (16-byte aligned; its contents need no initialisation) and the
 * CUDA stream.  Validates again, then enqueues the prolog's kernels on `stream` and
 * returns without waiting.  Two calls may not share a workspace while both are in flight.
 * The result is deterministic: the same inputs give the same output bits.
 * Returns 161001 / 161002 / 561002 as phase 1, 161002 if workspaceSize is too small, and
 * 361001 if a launch fails.
 */
MLA_API mla_status mla_prolog(
    const mla_tensor* tokenX, const mla_tensor* weightDq, const mla_tensor* weightUqQr,
    const mla_tensor* weightUk, const mla_tensor* weightDkvKr,
    const mla_tensor* rmsnormGammaCq, const mla_tensor* rmsnormGammaCkv,
    const mla_tensor* ropeSin, const mla_tensor* ropeCos, const mla_tensor* cacheIndex,
    const mla_tensor* kvCache, const mla_tensor* krCache,
    const mla_tensor* dequantScaleX, const mla_tensor* dequantScaleWDq,
    const mla_tensor* dequantScaleWUqQr, const mla_tensor* dequantScaleWDkvKr,
    const mla_tensor* quantScaleCkv, const mla_tensor* quantScaleCkr,
    const mla_tensor* smoothScalesCq,
    double rmsnormEpsilonCq, double rmsnormEpsilonCkv, const char* cacheMode,
    const mla_tensor* queryOut, const mla_tensor* queryRopeOut,
    const mla_tensor* dequantScaleQNopeOut,
    void* workspace, uint64_t workspaceSize, void* stream);

/*
 * Diagnostic: waits for `stream`, then copies the status word of the last mla_prolog()
 * call that used `workspace` into *bits (MLA_DEV_* flags; 0 = clean).  The first kernel of
 * every mla_prolog() call clears the word.  No counterpart on the pages (their kernels
 * report through return codes only).  Returns 161001 for NULL arguments, 161002 when
 * workspaceSize is below the status word's size, 361001 if the copy fails.
 */
MLA_API mla_status mla_prolog_device_status(const void* workspace, uint64_t workspaceSize, void* stream,
                                    uint32_t* bits);

/*
 * Diagnostic for failure detection, no counterpart on the pages: enqueues on `stream` one small
 * kernel whose wait nothing can satisfy -- which = 0: the flag wait of the persistent decode
 * kernel on a flag that never holds its tag (limit 2 s); which = 1: an mbarrier wait that
 * nothing arrives on (limit 10 ms).  The wait gives up at its limit, the kernel sets
 * MLA_DEV_WAIT_TIMEOUT in the workspace's status word (cleared first) and returns, so the
 * context stays usable; mla_prolog_device_status() then reads the bit.  Needs a workspace of at
 * least 1 KB (16-byte aligned).  Returns 161001 for a NULL workspace, 161002 for a short or
 * misaligned workspace or another `which`, 361001 if the launch fails.
 */
MLA_API mla_status mla_prolog_debug_wait_probe(void* workspace, uint64_t workspaceSize, int which, void* stream);

/*
 * Per-kernel timing, a diagnostic with no counterpart on the pages.  While enabled
 * (process-wide, from the next mla_prolog() call on), each call records a CUDA event on
 * its stream before its first kernel and after every kernel, and launches the kernels
 * without programmatic-dependent overlap so that each interval is one kernel alone.
 * mla_prolog_timing_read() waits for the last event of the most recent timed call and
 * fills up to `capacity` entries (kernel name, milliseconds), setting *count to the number
 * of kernels of that call.  Returns 161001 for NULL pointers, 361001 if an event call fails,
 * 161002 if no call was timed yet.  Not thread-safe: time one caller at a time.
 */
typedef struct {
    char name[32];
    float ms;
} mla_kernel_time;

MLA_API mla_status mla_prolog_timing_enable(int enable);
MLA_API mla_status mla_prolog_timing_read(mla_kernel_time* out, int capacity, int* count);

/*
 * mla_prolog without a caller-supplied workspace.  The pages have no counterpart: their
 * operator always takes a workspace from the caller.
 *
 * Some callers have no way to obtain device memory on their own: a plugin whose host
 * process owns the whole device memory budget and hands out no allocator, or a runtime
 * that plans every buffer once at start-up and may not call cudaMalloc afterwards.  They
 * can provide the inputs and outputs, but not the workspace mla_prolog() needs.  This
 * entry point takes the same tensor and scalar arguments (no workspace) and runs the same
 * kernels, with the workspace placed in one fixed scratch buffer that the library itself
 * holds in device memory: MLA_NO_ALLOC_SCRATCH_BYTES bytes, reserved on every GPU that
 * loads the library, for the life of the process.
 *
 * - Size limit: calls whose workspace (as mla_prolog_workspace_size reports it) exceeds
 *   MLA_NO_ALLOC_SCRATCH_BYTES return MLA_ERR_SCRATCH_LIMIT and launch nothing.  16 MiB
 *   covers bf16 decode batches of up to 128 tokens with DeepSeek-V3 shapes; prefill-sized
 *   calls (hundreds of tokens and more) do not fit.
 * - No allocation: the call makes no cudaMalloc / cudaFree and no allocating library call.
 *   The first call on each device looks up the scratch buffer's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call before any
 *   stream capture on the device.  The address is tied to the CUDA context it was found in:
 *   after cudaDeviceReset (or when another context is current) the next call looks it up
 *   again, so that call too belongs before any capture.
 * - Sharing: every call on a device uses the same scratch buffer, which keeps the previous
 *   call's contents.  The call clears the part that must start at zero (the status word)
 *   on `stream` before its kernels run.  Calls whose kernels overlap on the GPU (other
 *   streams, or other host threads) race on the scratch buffer and give wrong results:
 *   order them on one stream or with events.
 * - The device status word (out-of-range cacheIndex rows, which are skipped, and pipeline
 *   waits that gave up) lives in the scratch buffer; mla_prolog_no_alloc_status() reads it.
 *
 * Returns the codes of mla_prolog(), plus MLA_ERR_SCRATCH_LIMIT, and 361001 if the scratch
 * buffer's address cannot be obtained.
 */
#define MLA_NO_ALLOC_SCRATCH_BYTES (16ull << 20)

MLA_API mla_status mla_prolog_no_alloc(
    const mla_tensor* tokenX, const mla_tensor* weightDq, const mla_tensor* weightUqQr,
    const mla_tensor* weightUk, const mla_tensor* weightDkvKr,
    const mla_tensor* rmsnormGammaCq, const mla_tensor* rmsnormGammaCkv,
    const mla_tensor* ropeSin, const mla_tensor* ropeCos, const mla_tensor* cacheIndex,
    const mla_tensor* kvCache, const mla_tensor* krCache,
    const mla_tensor* dequantScaleX, const mla_tensor* dequantScaleWDq,
    const mla_tensor* dequantScaleWUqQr, const mla_tensor* dequantScaleWDkvKr,
    const mla_tensor* quantScaleCkv, const mla_tensor* quantScaleCkr,
    const mla_tensor* smoothScalesCq,
    double rmsnormEpsilonCq, double rmsnormEpsilonCkv, const char* cacheMode,
    const mla_tensor* queryOut, const mla_tensor* queryRopeOut,
    const mla_tensor* dequantScaleQNopeOut, void* stream);

/*
 * The device status bits (MLA_DEV_* flags) of the last mla_prolog_no_alloc() call on the
 * current device: waits for `stream`, then copies the status word out of the library's
 * scratch buffer into *bits.  No allocation.  Like the buffer itself, the word belongs to
 * whichever call ran last; read it before the next call.  Returns 161001 for a NULL `bits`,
 * 361001 if a CUDA call fails.
 */
MLA_API mla_status mla_prolog_no_alloc_status(void* stream, uint32_t* bits);

/* A constant, human-readable name for a return code. */
MLA_API const char* mla_prolog_status_string(mla_status status);

#ifdef __cplusplus
}
#endif

#endif /* MLA_PROLOG_H */
