/*
 * mla_preprocess.h -- C ABI of the "aclnnMlaPreprocess" variant of the MLA prolog on GB300.
 *
 * The operation is the one "aclnnMlaPreprocess" defines (Function description; Formula):
 *
 *   x'   = RmsNormQuant(x)            (gamma0, beta0, quantScale0, quantOffset0; int8)
 *   y    = x' . W^DQKV                (int8 x int8; + bias0, * deScale0 per output column)
 *   path 1: c = RmsNormQuant(y[:Hcq]) (gamma1, beta1, quantScale1, quantOffset1; int8)
 *           z = c . W^UQ              (int8 x int8; + bias1, * deScale1), viewed (N, D + 64)
 *   path 3: q^N = z[n, :D] . W^UK[n]  (per head)
 *   path 4: q^R = ROPE(z[n, D:])
 *   path 5: k^N = RmsNorm(y[Hcq : Hcq + 512])  (gamma2), written to the cache
 *   path 6: k^R = ROPE(y[Hcq + 512 : Hcq + 576]), written to the cache
 *
 * RmsNorm(x) = gamma * x_i / sqrt(mean(x^2) + epsilon), RmsNormQuant(x) =
 * (RmsNorm(x) + beta) * quantScale (same page, Formula), and the int8 code of a value v is
 * clamp(round_half_away(v * quantScale) + quantOffset, -128, 127) (quantMode 0: per-tensor
 * static asymmetric).  With doRmsNorm false the input is only quantised: the code of x
 * itself (beta0 belongs to the norm and is not added).  ROPE is the half rotation of the
 * page's Constraints (RoPE mode): out = v * cos + rotate_half(v) * sin.
 *
 * Conventions are those of mla_prolog.h: mla_tensor descriptors of contiguous row-major
 * DEVICE tensors, caller-owned buffers (the library allocates nothing and keeps no
 * pointer), the same return codes, an asynchronous call on `stream`, no synchronisation,
 * no trap.  The workspace begins with the same status word as mla_prolog()'s, so
 * mla_prolog_device_status() reads it (MLA_DEV_CACHE_INDEX_RANGE: a slotMapping value
 * outside [0, blockNum*blockSize) -- that token's cache row is not written).
 *
 * Arguments, in the page's order (aclnnMlaPreprocessGetWorkspaceSize, parameter table).
 * "F" is the input's dtype, bf16 or fp16; it is also the dtype of every F tensor below.
 *
 *   input         (T, He)                 F       tokenNum T in [0, 256]
 *   gamma0, beta0 (He)                    F
 *   quantScale0   (1)                     F
 *   quantOffset0  (1)                     int8
 *   wdqkv         (Hcq + 576, He)         int8    one row per output column ("transposeWdq"
 *                                                 true); columns [W^DQ | W^DKV (512) | W^KR (64)];
 *                                                 row-major (the page's NZ tiling is Ascend's)
 *   deScale0      (Hcq + 576)             fp32    per output column
 *   bias0         (Hcq + 576)             int32   may be NULL or empty (then 0)
 *   gamma1, beta1 (Hcq)                   F       qLoraDim Hcq in [1, 4096]
 *   quantScale1   (1)                     F
 *   quantOffset1  (1)                     int8
 *   wuq           (N * (D + 64), Hcq)     int8    one row per output column; head n owns rows
 *                                                 n*(D+64) .. : D of W^UQ, then 64 of W^QR
 *   deScale1      (N * (D + 64))          fp32
 *   bias1         (N * (D + 64))          int32   may be NULL or empty
 *   gamma2        (512)                   F
 *   cos, sin      (T, 64)                 F       full-width tables
 *   wuk           (N, D, 512)             F
 *   kvCache       cacheMode 0: (blockNum, blockSize, 1, 576)  F   row = [k^N | k^R]
 *                 cacheMode 1: (blockNum, blockSize, 1, 512)  F   row = k^N
 *   kvCacheRope   cacheMode 1: (blockNum, blockSize, 1, 64)   F   row = k^R; NULL in mode 0
 *   slotMapping   (T)                     int32   flat slot in [0, blockNum * blockSize)
 *   ctkvScale, qNopeScale                 must be NULL (cacheMode 2 only)
 *   wdqDim == Hcq; qRopeDim == kRopeDim == 64; qRotaryCoeff == kRotaryCoeff == 2;
 *   transposeWdq, transposeWuq, transposeWuk nonzero; cacheMode 0 or 1; quantMode 0;
 *   wdkvSplitCount 1 (the only values the page accepts, except cacheMode 2 and 3, whose
 *   NZ cache layouts and per-head static quantisation are not built here: 161002)
 *   epsilon       one epsilon for all three norms
 *   doRmsNorm     nonzero: RmsNormQuant of the input; zero: quantisation only
 *   qOut          cacheMode 0: (T, N, 576) F, row = [q^N | q^R]; cacheMode 1: (T, N, 512) F
 *   kvCacheOut    the same tensor as kvCache (same data pointer), updated in place
 *   qRopeOut      cacheMode 1: (T, N, 64) F; NULL in mode 0
 *   krCacheOut    cacheMode 1: the same tensor as kvCacheRope; NULL in mode 0
 *
 * Only the cache rows named by slotMapping change.  blockNum * blockSize = 0 is valid: the
 * q outputs are computed and no cache is written.  T = 0 does nothing.  Distinct slots are
 * the caller's contract (with duplicates the surviving row is unspecified).
 *
 * Tiling rules (561002 when broken): He % 64 == 0, Hcq % 64 == 0, D % 16 == 0 with
 * 16 <= D <= 256, N in [1, 128].  Every device pointer must be 16-byte aligned.
 *
 * Determinism: the same inputs give the same output bits (the page: deterministic by
 * default).
 */
#ifndef MLA_PREPROCESS_H
#define MLA_PREPROCESS_H

#include "mla_prolog.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Phase 1 ("aclnnMlaPreprocess", Function prototype: aclnnMlaPreprocessGetWorkspaceSize).
 * Validates every argument and returns in *workspaceSize the device workspace bytes that
 * mla_preprocess() needs for these shapes.  161001: a required tensor or out-pointer is
 * NULL; 161002: a shape, dtype, scalar or optional-argument pattern outside the above;
 * 561002: the tiling rules.
 */
MLA_API mla_status mla_preprocess_workspace_size(
    const mla_tensor* input, const mla_tensor* gamma0, const mla_tensor* beta0,
    const mla_tensor* quantScale0, const mla_tensor* quantOffset0, const mla_tensor* wdqkv,
    const mla_tensor* deScale0, const mla_tensor* bias0, const mla_tensor* gamma1,
    const mla_tensor* beta1, const mla_tensor* quantScale1, const mla_tensor* quantOffset1,
    const mla_tensor* wuq, const mla_tensor* deScale1, const mla_tensor* bias1,
    const mla_tensor* gamma2, const mla_tensor* cos, const mla_tensor* sin, const mla_tensor* wuk,
    const mla_tensor* kvCache, const mla_tensor* kvCacheRope, const mla_tensor* slotMapping,
    const mla_tensor* ctkvScale, const mla_tensor* qNopeScale,
    int64_t wdqDim, int64_t qRopeDim, int64_t kRopeDim, double epsilon,
    int64_t qRotaryCoeff, int64_t kRotaryCoeff, int32_t transposeWdq, int32_t transposeWuq,
    int32_t transposeWuk, int64_t cacheMode, int64_t quantMode, int32_t doRmsNorm,
    int64_t wdkvSplitCount,
    const mla_tensor* qOut, const mla_tensor* kvCacheOut, const mla_tensor* qRopeOut,
    const mla_tensor* krCacheOut,
    uint64_t* workspaceSize);

/*
 * Phase 2 ("aclnnMlaPreprocess", Function prototype: aclnnMlaPreprocess).  Same arguments,
 * then a device workspace of at least the phase-1 size (16-byte aligned, no initialisation
 * needed) and the CUDA stream.  Validates again and enqueues the kernels on `stream`.
 * Returns the phase-1 codes, 161002 if workspaceSize is too small, 361001 if a launch fails.
 */
MLA_API mla_status mla_preprocess(
    const mla_tensor* input, const mla_tensor* gamma0, const mla_tensor* beta0,
    const mla_tensor* quantScale0, const mla_tensor* quantOffset0, const mla_tensor* wdqkv,
    const mla_tensor* deScale0, const mla_tensor* bias0, const mla_tensor* gamma1,
    const mla_tensor* beta1, const mla_tensor* quantScale1, const mla_tensor* quantOffset1,
    const mla_tensor* wuq, const mla_tensor* deScale1, const mla_tensor* bias1,
    const mla_tensor* gamma2, const mla_tensor* cos, const mla_tensor* sin, const mla_tensor* wuk,
    const mla_tensor* kvCache, const mla_tensor* kvCacheRope, const mla_tensor* slotMapping,
    const mla_tensor* ctkvScale, const mla_tensor* qNopeScale,
    int64_t wdqDim, int64_t qRopeDim, int64_t kRopeDim, double epsilon,
    int64_t qRotaryCoeff, int64_t kRotaryCoeff, int32_t transposeWdq, int32_t transposeWuq,
    int32_t transposeWuk, int64_t cacheMode, int64_t quantMode, int32_t doRmsNorm,
    int64_t wdkvSplitCount,
    const mla_tensor* qOut, const mla_tensor* kvCacheOut, const mla_tensor* qRopeOut,
    const mla_tensor* krCacheOut,
    void* workspace, uint64_t workspaceSize, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA_PREPROCESS_H */
