// C ABI of the MLA prolog: argument validation, tile planning, workspace layout, TMA
// descriptors and kernel launches.  Declarations and argument documentation: mla_prolog.h.
//
// Pipeline of one call (all kernels on the caller's stream, chained with programmatic
// dependent launch so each grid's prologue overlaps the previous grid's tail):
//   [int8 tokenX only] widen the int8 codes of tokenX to fp16 in the workspace
//   K1  x . [W^DQ | W^DKV | W^KR]        -> fp32 partials (decode) or fp32 rows (prefill); int8
//                                           weights stream as int8 and are widened in shared memory
//   F1  sum partials, RmsNorm, RoPE(k^R), kv/kr cache writes, c^Q (bf16, or int8 codes as fp16)
//   K2  c^Q . W^UqQr                      -> fused RoPE epilogue, or (int8 W^UqQr, widened in
//                                           shared memory) fp32 rows + F2
//   K3  q^C[:, n, :] . W^UK[n] per head   -> queryOut bf16, or int8 + dequantScaleQNope
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <atomic>
#include <mutex>
#include <random>

#include "mla_prolog.h"
#include "decode_persist.cuh"
#include "finalize.cuh"
#include "gemm_tc.cuh"
#include "gemm_pair.cuh"
#include "preprocess.cuh"
#include "gemm_w8.cuh"

using namespace mla;

namespace {

// ---------------------------------------------------------------- validation

struct Dims {
    int64_t T, He, Hcq, N, D, Dr, Hckv, block_num, block_size;
};

struct Scenario {
    bool x_i8;      // int8 tokenX, weightDq, weightDkvKr
    bool uqqr_i8;   // int8 weightUqQr
    bool kv_i8;
    bool kr_i8;
    bool q_i8;      // queryOut int8: dynamic quantisation of q^N
};

struct Args {
    const mla_tensor *x, *wdq, *wuqqr, *wuk, *wdkvkr, *gcq, *gckv, *sin, *cos, *idx, *kv, *kr;
    const mla_tensor *sx, *swdq, *swuqqr, *swdkvkr, *qckv, *qckr, *smooth;
    double eps_cq, eps_ckv;
    const char* cache_mode;
    const mla_tensor *qout, *qrope, *qscale;
};

int64_t numel(const mla_tensor* t) {
    int64_t n = 1;
    for (int i = 0; i < t->ndim; ++i) n *= t->shape[i];
    return n;
}

bool shape_is(const mla_tensor* t, std::initializer_list<int64_t> s) {
    if (t->ndim != (int)s.size()) return false;
    int i = 0;
    for (int64_t v : s)
        if (t->shape[i++] != v) return false;
    return true;
}

bool aligned16(const mla_tensor* t) {
    return t->data == nullptr || (reinterpret_cast<uintptr_t>(t->data) & 15u) == 0;
}

// A per-token tensor: (T, rest...) or (B, S, rest...).  Returns T or -1.
int64_t tokens_of(const mla_tensor* t, int rest_dims) {
    const int lead = t->ndim - rest_dims;
    if (lead != 1 && lead != 2) return -1;
    int64_t T = t->shape[0];
    if (lead == 2) T *= t->shape[1];
    return T;
}

bool rest_is(const mla_tensor* t, int rest_dims, std::initializer_list<int64_t> s) {
    if ((int)s.size() != rest_dims) return false;
    int i = t->ndim - rest_dims;
    for (int64_t v : s)
        if (t->shape[i++] != v) return false;
    return true;
}

// A (1, n) or (n) fp32 vector.
bool vec_f32(const mla_tensor* t, int64_t n) {
    if (t->dtype != MLA_DT_FP32) return false;
    return shape_is(t, {n}) || shape_is(t, {1, n});
}

mla_status validate(const Args& a, Dims& d, Scenario& sc) {
    const mla_tensor* req[] = {a.x, a.wdq, a.wuqqr, a.wuk, a.wdkvkr, a.gcq, a.gckv, a.sin, a.cos,
                               a.idx, a.kv, a.kr, a.qout, a.qrope};
    for (const mla_tensor* t : req)
        if (t == nullptr) return MLA_ERR_PARAM_NULLPTR;
    const mla_tensor* all[] = {a.x, a.wdq, a.wuqqr, a.wuk, a.wdkvkr, a.gcq, a.gckv, a.sin, a.cos, a.idx, a.kv,
                               a.kr, a.qout, a.qrope, a.sx, a.swdq, a.swuqqr, a.swdkvkr, a.qckv, a.qckr,
                               a.smooth, a.qscale};
    for (const mla_tensor* t : all) {
        if (t == nullptr) continue;
        if (t->ndim < 1 || t->ndim > 4) return MLA_ERR_PARAM_INVALID;
        for (int i = 0; i < t->ndim; ++i)
            if (t->shape[i] < 0) return MLA_ERR_PARAM_INVALID;
        if (t->data == nullptr && numel(t) > 0) return MLA_ERR_PARAM_NULLPTR;
        if (!aligned16(t)) return MLA_ERR_PARAM_INVALID;
    }

    // tokenX (T, He) or (B, S, He)
    if (a.x->dtype != MLA_DT_BF16 && a.x->dtype != MLA_DT_INT8) return MLA_ERR_PARAM_INVALID;
    d.T = tokens_of(a.x, 1);
    if (d.T < 0) return MLA_ERR_PARAM_INVALID;
    d.He = a.x->shape[a.x->ndim - 1];
    sc.x_i8 = a.x->dtype == MLA_DT_INT8;
    // weightUk (N, D, Hckv)
    if (a.wuk->dtype != MLA_DT_BF16 || a.wuk->ndim != 3) return MLA_ERR_PARAM_INVALID;
    d.N = a.wuk->shape[0];
    d.D = a.wuk->shape[1];
    d.Hckv = a.wuk->shape[2];
    // weightDq (He, Hcq)
    if (a.wdq->ndim != 2 || a.wdq->shape[0] != d.He) return MLA_ERR_PARAM_INVALID;
    d.Hcq = a.wdq->shape[1];
    // weightUqQr (Hcq, N*(D+Dr))
    if (a.wuqqr->ndim != 2 || a.wuqqr->shape[0] != d.Hcq || d.N <= 0) return MLA_ERR_PARAM_INVALID;
    if (a.wuqqr->shape[1] % d.N != 0) return MLA_ERR_PARAM_INVALID;
    d.Dr = a.wuqqr->shape[1] / d.N - d.D;
    if (d.He <= 0 || d.Hcq <= 0 || d.D <= 0 || d.Dr <= 0 || d.Hckv <= 0) return MLA_ERR_PARAM_INVALID;
    // weightDkvKr (He, Hckv + Dr)
    if (!shape_is(a.wdkvkr, {d.He, d.Hckv + d.Dr})) return MLA_ERR_PARAM_INVALID;
    // dtype pattern of the weights
    sc.uqqr_i8 = a.wuqqr->dtype == MLA_DT_INT8;
    if (a.wuqqr->dtype != MLA_DT_BF16 && !sc.uqqr_i8) return MLA_ERR_PARAM_INVALID;
    const int32_t xdt = a.x->dtype;
    if (a.wdq->dtype != xdt || a.wdkvkr->dtype != xdt) return MLA_ERR_PARAM_INVALID;
    if (sc.x_i8 && !sc.uqqr_i8) return MLA_ERR_PARAM_INVALID;
    // gammas
    if (a.gcq->dtype != MLA_DT_BF16 || !(shape_is(a.gcq, {d.Hcq}) || shape_is(a.gcq, {1, d.Hcq})))
        return MLA_ERR_PARAM_INVALID;
    if (a.gckv->dtype != MLA_DT_BF16 || !(shape_is(a.gckv, {d.Hckv}) || shape_is(a.gckv, {1, d.Hckv})))
        return MLA_ERR_PARAM_INVALID;
    // rope tables, cacheIndex
    for (const mla_tensor* t : {a.sin, a.cos}) {
        if (t->dtype != MLA_DT_BF16 || tokens_of(t, 1) != d.T || !rest_is(t, 1, {d.Dr})) return MLA_ERR_PARAM_INVALID;
        if (t->ndim == 3 && (t->shape[0] != a.x->shape[0] || a.x->ndim != 3)) return MLA_ERR_PARAM_INVALID;
    }
    if (a.idx->dtype != MLA_DT_INT64 || tokens_of(a.idx, 0) != d.T) return MLA_ERR_PARAM_INVALID;
    // caches (BlockNum, BlockSize, Nkv = 1, H)
    if (a.kv->ndim != 4 || a.kr->ndim != 4) return MLA_ERR_PARAM_INVALID;
    d.block_num = a.kv->shape[0];
    d.block_size = a.kv->shape[1];
    if (!shape_is(a.kv, {d.block_num, d.block_size, 1, d.Hckv})) return MLA_ERR_PARAM_INVALID;
    if (!shape_is(a.kr, {d.block_num, d.block_size, 1, d.Dr})) return MLA_ERR_PARAM_INVALID;
    sc.kv_i8 = a.kv->dtype == MLA_DT_INT8;
    sc.kr_i8 = a.kr->dtype == MLA_DT_INT8;
    if (a.kv->dtype != MLA_DT_BF16 && !sc.kv_i8) return MLA_ERR_PARAM_INVALID;
    if (a.kr->dtype != MLA_DT_BF16 && !sc.kr_i8) return MLA_ERR_PARAM_INVALID;
    // outputs
    if (a.qout->dtype != MLA_DT_BF16 && a.qout->dtype != MLA_DT_INT8) return MLA_ERR_PARAM_INVALID;
    if (tokens_of(a.qout, 2) != d.T || !rest_is(a.qout, 2, {d.N, d.Hckv})) return MLA_ERR_PARAM_INVALID;
    if (a.qrope->dtype != MLA_DT_BF16 || tokens_of(a.qrope, 2) != d.T || !rest_is(a.qrope, 2, {d.N, d.Dr}))
        return MLA_ERR_PARAM_INVALID;
    sc.q_i8 = a.qout->dtype == MLA_DT_INT8;
    if (sc.q_i8) {
        if (a.qscale == nullptr) return MLA_ERR_PARAM_NULLPTR;
        if (a.qscale->dtype != MLA_DT_FP32) return MLA_ERR_PARAM_INVALID;
        const bool ok = (a.qscale->ndim == 3 && a.qscale->shape[0] == d.T && a.qscale->shape[1] == d.N &&
                         a.qscale->shape[2] == 1) ||
                        (a.qscale->ndim == 2 && a.qscale->shape[0] == d.T && a.qscale->shape[1] == d.N);
        if (!ok) return MLA_ERR_PARAM_INVALID;
    } else if (a.qscale != nullptr && numel(a.qscale) > 1) {
        return MLA_ERR_PARAM_INVALID;
    }

    // optional-argument pattern of each scenario (page: scenario / dtype table)
    const int64_t W = d.N * (d.D + d.Dr);
    if (sc.x_i8) {
        if (!a.sx || !a.swdq || !a.swuqqr || !a.swdkvkr) return MLA_ERR_PARAM_NULLPTR;
        if (a.sx->dtype != MLA_DT_FP32 || !(shape_is(a.sx, {d.T, 1}) || shape_is(a.sx, {d.T})))
            return MLA_ERR_PARAM_INVALID;
        if (!vec_f32(a.swdq, d.Hcq) || !vec_f32(a.swdkvkr, d.Hckv + d.Dr)) return MLA_ERR_PARAM_INVALID;
        if (sc.kr_i8 || a.qckr) return MLA_ERR_PARAM_INVALID;  // krCache stays bf16 in full quantisation
    } else {
        if (a.sx || a.swdq || a.swdkvkr) return MLA_ERR_PARAM_INVALID;
    }
    if (sc.uqqr_i8) {
        if (!a.swuqqr) return MLA_ERR_PARAM_NULLPTR;
        if (!vec_f32(a.swuqqr, W)) return MLA_ERR_PARAM_INVALID;
        if (a.smooth && !vec_f32(a.smooth, d.Hcq)) return MLA_ERR_PARAM_INVALID;
    } else {
        if (a.swuqqr || a.smooth) return MLA_ERR_PARAM_INVALID;
    }
    if (sc.kv_i8) {
        if (!sc.uqqr_i8) return MLA_ERR_PARAM_INVALID;   // a quantised cache needs a quantised scenario
        if (!a.qckv) return MLA_ERR_PARAM_NULLPTR;
        if (!vec_f32(a.qckv, d.Hckv)) return MLA_ERR_PARAM_INVALID;
        if (!sc.x_i8) {
            // partial quantisation with quantised caches: both caches are int8
            if (!sc.kr_i8) return MLA_ERR_PARAM_INVALID;
            if (!a.qckr) return MLA_ERR_PARAM_NULLPTR;
            if (!vec_f32(a.qckr, d.Dr)) return MLA_ERR_PARAM_INVALID;
        }
    } else {
        if (a.qckv || a.qckr || sc.kr_i8) return MLA_ERR_PARAM_INVALID;
    }
    if (!std::isfinite(a.eps_cq) || !std::isfinite(a.eps_ckv) || a.eps_cq < 0 || a.eps_ckv < 0)
        return MLA_ERR_PARAM_INVALID;
    if (a.cache_mode != nullptr && std::strcmp(a.cache_mode, "PA_BSND") != 0) return MLA_ERR_PARAM_INVALID;

    // tiling rules of the kernels
    if (d.He % 8 || d.Hcq % 64 || d.D % 8 || (d.Dr & 1) || W % 8 || (d.Hckv + d.Dr) % 8 || d.Hckv % 8)
        return MLA_ERR_TILING;
    if (sc.q_i8 && d.Hckv > 512) return MLA_ERR_TILING;
    if ((d.Hcq + d.Hckv + d.Dr) * 4 > 48 * 1024) return MLA_ERR_TILING;   // one fp32 row in shared memory
    if (d.T > (int64_t)INT32_MAX || d.He > (int64_t)INT32_MAX || W > (int64_t)INT32_MAX) return MLA_ERR_TILING;
    return MLA_OK;
}

// ---------------------------------------------------------------------- plan

// One GEMM launch: tile shape, work split and grid.
struct GemmPlan {
    int msub = 1, grid = 0, m_tiles = 1, n_tiles = 0, kblocks = 0, bn = 192, ksplit = 1, a_box_rows = 128;
};

struct Plan {
    GemmPlan g1, g2, g3;
    bool g2_fused = false;   // K2 epilogue does RoPE and q^C (no finalize_up)
    bool g2_wide = false;    // K2 with 256 x 256 tiles on SM pairs (prefill)
    bool g1_pair = false;    // K1 with 256 x 256 tiles on SM pairs (prefill)
    bool fold_cq = false;    // K1 writes bf16(gamma_cq * y) and row sums of squares, K2 applies 1 / RMS
    size_t off_ss = 0;       // fold_cq: T x kFoldSums row sums of squares
    bool persist = false;    // decode-sized bf16 call: the one persistent kernel of decode_persist.cuh
    int p_n1 = 0, p_s1 = 0, p_wst = 0, p_arows = 0, p_na3 = 0, p_pf = 0;
    size_t p_smem = 0, off_pbar = 0;
    int64_t ncols1 = 0, ncols2 = 0;
    size_t off_cq = 0, off_cqs = 0, off_qc = 0, off_y1 = 0, off_y2 = 0, off_xb = 0, bytes = 0;
};

constexpr size_t kStatusBytes = 1024;
constexpr int kDecodeRows = 256;   // up to this many tokens: one row tile, weight streaming
constexpr int kPairKps = 2;         // k-blocks per stage of the prefill GEMMs on SM pairs
constexpr int kFoldSums = 16;       // row sums of squares per token in the folded c^Q RmsNorm (at most)

size_t up1024(size_t v) { return (v + 1023) & ~size_t(1023); }

int device_sms(int* out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) return -1;
    *out = sms;
    return 0;
}

// Tiles of bn columns; at decode-sized T one row tile of MSUB*128 rows and, when asked,
// k ranges so that (tiles x ranges) covers the SMs.
void plan_gemm(GemmPlan& g, int64_t T, int64_t ncols, int64_t K, int sms, int bn, bool allow_ksplit) {
    g.bn = bn;
    g.kblocks = (int)((K + kBK - 1) / kBK);
    g.n_tiles = (int)((ncols + bn - 1) / bn);
    if (T <= kDecodeRows) {
        g.msub = T <= 128 ? 1 : 2;
        g.m_tiles = 1;
        g.a_box_rows = g.msub == 1 ? (int)((T + 7) / 8 * 8) : 128;
        int S = allow_ksplit ? sms / g.n_tiles : 1;
        if (S > g.kblocks) S = g.kblocks;
        if (S > 16) S = 16;
        g.ksplit = S < 1 ? 1 : S;
    } else {
        g.msub = 2;
        g.m_tiles = (int)((T + 255) / 256);
        g.a_box_rows = 128;
        g.ksplit = 1;
    }
    const long long units = (long long)g.m_tiles * g.n_tiles * g.ksplit;
    g.grid = (int)(units < sms ? units : sms);
}

Plan make_plan(const Dims& d, const Scenario& sc, int sms) {
    Plan p;
    const int64_t T = d.T;
    p.ncols1 = d.Hcq + d.Hckv + d.Dr;
    p.ncols2 = d.N * (d.D + d.Dr);
    // Down-projection: at decode, 64-column tiles x k ranges; two 128-row sub-tiles use
    // 192-column tiles; prefill 256-column tiles (2112 columns: nine tiles per 256 rows, so that
    // 8192 tokens make two waves on 152 SMs instead of three).
    // int8 weights (widened in shared memory, MN-major int8 boxes of one BN-byte row per k): 192
    // columns per tile (a tile must not straddle W^DQ | W^DkvKr)
    const int bn1_i8 = d.Hcq % 192 == 0 ? 192 : 64;
    plan_gemm(p.g1, T, p.ncols1, d.He, sms, sc.x_i8 ? bn1_i8 : (T <= 128 ? 64 : (T <= kDecodeRows ? 192 : 256)), true);
    // prefill: 256 x 256 tiles on SM pairs (W^DQ's columns split into whole 128-column halves)
    p.g1_pair = !sc.x_i8 && p.g1.bn == 256 && p.g1.ksplit == 1 && d.Hcq % 128 == 0 && (d.Hckv + d.Dr) % 64 == 0 &&
                (d.He / 64) % kPairKps == 0 && p.ncols1 % 4 == 0;
    if (p.g1_pair) {
        p.g1.msub = 2;
        p.g1.m_tiles = (int)((T + 255) / 256);
        p.g1.a_box_rows = 128;
        p.g1.grid = 0;   // pairs: sized at launch
    }
    // Up-projection: one head (192 columns) per tile, full K, fused RoPE epilogue; prefill with
    // the 128 + 64 head layout uses 256 x 256 tiles on SM pairs (their epilogue sorts 64-column
    // blocks into q^C and rope blocks).
    p.g2_fused = d.D == 128 && d.Dr == 64;
    p.g2_wide = p.g2_fused && T > kDecodeRows && p.ncols2 % 256 == 0 && !sc.uqqr_i8;
    // The RmsNorm of c^Q folded into the two prefill GEMMs (bf16 operands): no row pass over c^Q.
    // (the row pass that then handles only c^KV | k^R is the warp-per-token one)
    p.fold_cq = p.g1_pair && p.g2_wide && !sc.x_i8 && d.Hcq % 256 == 0 && d.Hcq / 256 * 2 <= kFoldSums &&
                d.Dr == 64 && d.Hckv % 64 == 0 && d.Hcq <= 64 * kWQ && d.Hckv <= 64 * kWKV;
    plan_gemm(p.g2, T, p.ncols2, d.Hcq, sms, p.g2_wide ? 256 : 192, false);
    if (p.g2_wide) {
        p.g2.msub = 2;
        p.g2.m_tiles = (int)((T + 255) / 256);
        p.g2.a_box_rows = 128;
        p.g2.grid = 0;   // pairs: sized at launch from the co-resident clusters
    }
    // K3: per head, 128-row tiles; an int8 output needs the whole Hckv row in one tile.
    p.g3.bn = sc.q_i8 ? 512 : 256;
    p.g3.kblocks = (int)((d.D + kBK - 1) / kBK);
    const int tph = (int)((d.Hckv + p.g3.bn - 1) / p.g3.bn);
    p.g3.n_tiles = (int)(d.N * tph);
    p.g3.m_tiles = (int)((T + 127) / 128);
    p.g3.msub = 1;
    p.g3.a_box_rows = T < 128 ? (int)((T + 7) / 8 * 8) : 128;
    {
        const long long tiles = (long long)p.g3.m_tiles * p.g3.n_tiles;
        p.g3.grid = (int)(tiles < sms ? tiles : sms);
    }

    // The persistent decode kernel: bf16 operands and outputs, 128 + 64 head layout, 512-wide
    // c^KV, every head on its own CTA.
    {
        const int64_t ncols1 = p.ncols1;
        const int n1 = (int)(ncols1 / 192);
        const int kb1 = (int)(d.He / 64);
        const int arows = (int)((T + 7) / 8 * 8);
        const size_t a_bytes = (size_t)arows * 128;
        const PersistSlots ps = persist_slots((int)a_bytes, (int)(d.Hcq / 64), kSmemLimit);
        const int wst = ps.wst;
        int s1 = n1 > 0 ? sms / n1 : 0;
        if (s1 > kb1) s1 = kb1;
        if (s1 > kPMaxS) s1 = kPMaxS;
        if (!sc.x_i8 && !sc.uqqr_i8 && !sc.kv_i8 && !sc.kr_i8 && !sc.q_i8 && T >= 1 && T <= kPMaxT &&
            d.D == 128 && d.Dr == 64 && d.Hckv == 512 && d.Hcq % 384 == 0 && d.He % 64 == 0 && ncols1 % 192 == 0 &&
            d.Hcq / kPChunk <= 128 && d.N >= 1 && d.N <= sms && s1 >= 1 &&
            ps.na3 >= 2 && wst >= kPMinW) {   // P4 staging needs its six stages in distinct slots
            p.persist = true;
            p.p_n1 = n1;
            p.p_s1 = s1;
            p.p_wst = wst;
            p.p_na3 = ps.na3;
            p.p_pf = ps.pf;
            p.p_arows = arows;
            p.p_smem = persist_smem_bytes((int)a_bytes, ps.na3, wst);
        }
    }

    size_t off = kStatusBytes;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = up1024(off + bytes);
        return o;
    };
    p.off_cq = take((size_t)T * d.Hcq * 2);
    p.off_cqs = take((size_t)T * 4);
    p.off_qc = take((size_t)T * d.N * d.D * 2);
    int y1_slots = p.g1.ksplit > 1 ? p.g1.ksplit : 1;
    if (p.persist && p.p_s1 > y1_slots) y1_slots = p.p_s1;
    p.off_y1 = take((size_t)y1_slots * T * p.ncols1 * 4);
    if (p.fold_cq) p.off_ss = take((size_t)T * kFoldSums * 4);
    // per P1 tile: a flag and a counter; per 16-column c^Q chunk: a flag and T sums of squares
    if (p.persist) p.off_pbar = take((size_t)p.p_n1 * (8 + 4) + 8 + (size_t)(d.Hcq / kPChunk) * (8 + 4 * T));
    if (!p.g2_fused) p.off_y2 = take((size_t)T * p.ncols2 * 4);
    if (sc.x_i8) p.off_xb = take((size_t)T * d.He * 2);   // tokenX's int8 codes as fp16
    p.bytes = off;
    return p;
}

// A per-call tag for the persistent kernel's dependency flags.  It starts at a random value
// so that flags left in a reused workspace by earlier calls never match.
unsigned long long next_tag() {
    static std::atomic<unsigned long long> ctr{[] {
        std::random_device rd;
        return ((unsigned long long)rd() << 32) ^ (unsigned long long)rd();
    }()};
    return ctr.fetch_add(1) + 1;
}

// --------------------------------------------------------------- tensor maps

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encoder() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode != nullptr;
}

// bf16 map with a 64-element (128-byte) inner box and 128-byte swizzle.
bool encode_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
                const uint32_t* box, CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
    cuuint64_t gd[3];
    cuuint64_t gs[2];
    cuuint32_t bx[3];
    cuuint32_t es[3] = {1, 1, 1};
    for (int i = 0; i < rank; ++i) {
        gd[i] = dims[i];
        bx[i] = box[i];
    }
    for (int i = 0; i < rank - 1; ++i) gs[i] = strides_bytes[i];
    const CUresult r = g_encode(m, dtype, (cuuint32_t)rank, const_cast<void*>(base), gd, gs,
                                bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Row-major (rows, cols) bf16 matrix.  Activations use a 128-row box, weights a 64-row box.
bool map_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    const uint64_t dims[2] = {cols, rows};
    const uint64_t strides[1] = {cols * 2};
    const uint32_t box[2] = {64, box_rows};
    return encode_map(m, base, 2, dims, strides, box);
}

// Row-major (rows, cols) bf16 matrix viewed as (64 columns, rows, cols/64 column blocks): a box
// {64, box_rows, nblk} brings nblk 64-column blocks of box_rows rows, block after block, in one
// request (cols must be a multiple of 64).
bool map_colblocks(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows, uint32_t nblk) {
    const uint64_t dims[3] = {64, rows, cols / 64};
    const uint64_t strides[2] = {cols * 2, 128};
    const uint32_t box[3] = {64, box_rows, nblk};
    return encode_map(m, base, 3, dims, strides, box);
}

// --------------------------------------------------------------------- timing

struct Timing {
    bool enabled = false;
    bool have = false;
    int n = 0;                        // kernels recorded in the last timed call
    cudaEvent_t ev[16] = {};
    const char* name[16] = {};
};
Timing g_timing;
std::mutex g_timing_mu;

// Records the event that closes the interval of the kernel just launched.
// Inside stream capture the record must be "external" to become a graph node.
void timing_record(cudaEvent_t ev, cudaStream_t st) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
        cudaEventRecordWithFlags(ev, st, cudaEventRecordExternal);
    else
        cudaEventRecord(ev, st);
}

void timing_mark(cudaStream_t st, const char* name) {
    if (!g_timing.enabled || g_timing.n >= 15) return;
    if (!g_timing.ev[g_timing.n + 1] && cudaEventCreate(&g_timing.ev[g_timing.n + 1]) != cudaSuccess) return;
    g_timing.name[g_timing.n] = name;
    timing_record(g_timing.ev[g_timing.n + 1], st);
    ++g_timing.n;
}

void timing_begin(cudaStream_t st) {
    if (!g_timing.enabled) return;
    g_timing.n = 0;
    g_timing.have = false;
    if (!g_timing.ev[0] && cudaEventCreate(&g_timing.ev[0]) != cudaSuccess) return;
    timing_record(g_timing.ev[0], st);
}

// --------------------------------------------------------------------- launch

// cudaFuncSetAttribute only when the (kernel, attribute, device) value changes: the setting
// persists, and the call costs microseconds of host time that a decode step cannot spare.
cudaError_t set_attr(const void* fn, cudaFuncAttribute attr, int value) {
    struct Entry {
        const void* fn;
        int attr, value, dev;
    };
    static std::mutex mu;
    static Entry done[256];
    static int ndone = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    int slot = -1;   // the entry holding the attribute's current value
    for (int i = 0; i < ndone && slot < 0; ++i)
        if (done[i].fn == fn && done[i].attr == (int)attr && done[i].dev == dev) slot = i;
    if (slot >= 0 && done[slot].value == value) return cudaSuccess;
    e = cudaFuncSetAttribute(fn, attr, value);
    if (e != cudaSuccess) return e;
    if (slot >= 0)
        done[slot].value = value;
    else if (ndone < 256)
        done[ndone++] = {fn, (int)attr, value, dev};
    return e;
}
template <typename Kernel>
cudaError_t set_attr(Kernel* k, cudaFuncAttribute attr, int value) {
    return set_attr(reinterpret_cast<const void*>(k), attr, value);
}

template <typename Kernel, typename... ArgsT>
cudaError_t launch(Kernel k, int grid, int block, size_t smem, cudaStream_t st, ArgsT... args) {
    // Every kernel of the prolog runs with the same (maximum) shared-memory carve-out, so the
    // SMs never re-partition L1 / shared memory between consecutive kernels.
    cudaError_t e = set_attr(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                                         (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = g_timing.enabled ? 0 : 1;
    return cudaLaunchKernelEx(&cfg, k, args...);
}

// Launches one GEMM instantiation; fills in the ring depth and dynamic shared memory.
template <int BN, int MSUB, int MAXST, int EPI, int OUTB = 0, int KPS = 1, int EPW = 1>
cudaError_t launch_gemm(int grid, cudaStream_t st, const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                        GemmArgs args, const CUtensorMap* out = nullptr, const CUtensorMap* out2 = nullptr) {
    using C = GemmCfg<BN, MSUB, MAXST, OUTB, KPS, EPW>;
    auto k = gemm_tc_kernel<BN, MSUB, MAXST, EPI, OUTB, KPS, EPW>;
    CUtensorMap mo, mo2;
    std::memset(&mo, 0, sizeof mo);
    std::memset(&mo2, 0, sizeof mo2);
    if (out != nullptr) mo = *out;
    if (out2 != nullptr) mo2 = *out2;
    args.stages = C::max_stages(args.a_box_rows);
    if (args.stages < 2) return cudaErrorInvalidConfiguration;
    const size_t smem = C::smem_bytes(args.stages, args.a_box_rows);
    cudaError_t e = set_attr(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemLimit);
    if (e != cudaSuccess) return e;
    return launch(k, grid, gemm_threads(EPW), smem, st, a, b0, b1, mo, mo2, args);
}

// Launches one int8-weight GEMM instantiation (gemm_w8.cuh); b8b holds the columns from
// args.b_split_col on (MN-major only).
template <int BN, int MSUB, int MAXST, bool MN = false, int EPI = EPI_F32, bool A8 = false>
cudaError_t launch_gemm_w8(int grid, cudaStream_t st, const CUtensorMap& a, const CUtensorMap& b8,
                           const CUtensorMap& b8b, GemmArgs args) {
    using C = W8Cfg<BN, MSUB, MAXST, MN, A8>;
    auto k = gemm_w8_kernel<BN, MSUB, MAXST, MN, EPI, A8>;
    args.stages = C::max_stages(args.a_box_rows);
    if (args.stages < 2) return cudaErrorInvalidConfiguration;
    cudaError_t e = set_attr(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemLimit);
    if (e != cudaSuccess) return e;
    return launch(k, grid, kW8Threads, C::smem_bytes(args.stages, args.a_box_rows), st, a, b8, b8b, args);
}
template <int BN, int MSUB, int MAXST>
cudaError_t launch_gemm_w8(int grid, cudaStream_t st, const CUtensorMap& a, const CUtensorMap& b8, GemmArgs args) {
    return launch_gemm_w8<BN, MSUB, MAXST, false>(grid, st, a, b8, b8, args);
}

// int8 (K, cols) row-major weight in the (k, n) orientation: boxes of box_cols columns (one
// box_cols-byte row per k, no swizzle) x 64 * kW8Kb k rows; rows and columns past the end read
// as zero.
bool map_w8_cols(CUtensorMap* m, const void* base, uint64_t K, uint64_t cols, uint32_t box_cols) {
    const cuuint64_t gd[2] = {cols, K};
    const cuuint64_t gs[1] = {cols};
    const cuuint32_t bx[2] = {box_cols, (cuuint32_t)(64 * kW8Kb)};
    const cuuint32_t es[2] = {1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), gd, gs, bx, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// int8 (rows, K) row-major matrix, one row per output column (the variant's weights) or per
// token (int8 tokenX): boxes of 64 * kW8Kb k (no swizzle) x box_rows rows; rows and columns past
// the end read as zero.
bool map_w8_rows(CUtensorMap* m, const void* base, uint64_t rows, uint64_t K, uint32_t box_rows) {
    const cuuint64_t gd[2] = {K, rows};
    const cuuint64_t gs[1] = {K};
    const cuuint32_t bx[2] = {(cuuint32_t)(64 * kW8Kb), box_rows};
    const cuuint32_t es[2] = {1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), gd, gs, bx, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Launches one pair-CTA GEMM instantiation (clusters of two CTAs): as many pairs as the GPU
// holds at once, at most one per 256-row tile.
template <int BN, int MAXST, int EPI, int OUTB, int EPW, int KPS>
cudaError_t launch_gemm_pair(cudaStream_t st, const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                             GemmArgs args, const CUtensorMap& out, const CUtensorMap& out2) {
    using C = PairCfg<BN, MAXST, OUTB, EPW, KPS>;
    auto k = gemm_pair_kernel<BN, MAXST, EPI, OUTB, EPW, KPS>;
    if (args.kblocks % KPS != 0) return cudaErrorInvalidValue;
    args.stages = C::max_stages();
    if (args.stages < 2) return cudaErrorInvalidConfiguration;
    const size_t smem = C::smem_bytes(args.stages);
    cudaError_t e = set_attr(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemLimit);
    if (e != cudaSuccess) return e;
    e = set_attr(k, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3((unsigned)gemm_threads(EPW));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = g_timing.enabled ? 1 : 2;
    // co-resident pairs of this instantiation on this device (queried once per device)
    static int s_pairs[64] = {};
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (s_pairs[dev] == 0) {
        int clusters = 0;
        cfg.gridDim = dim3(2);
        e = cudaOccupancyMaxActiveClusters(&clusters, k, &cfg);
        if (e != cudaSuccess) return e;
        if (clusters < 1) return cudaErrorInvalidConfiguration;
        s_pairs[dev] = clusters;
    }
    const long long units = (long long)args.m_tiles * args.n_tiles;
    const int pairs = (int)(units < s_pairs[dev] ? units : s_pairs[dev]);
    if (pairs < 1) return cudaSuccess;
    cfg.gridDim = dim3((unsigned)(2 * pairs));
    return cudaLaunchKernelEx(&cfg, k, a, b0, b1, out, out2, args);
}

// A second stream per device for work that nothing later in the call reads (the cache rows of
// a folded prefill call): it runs beside the tensor-core kernels instead of between them.  The
// fork and join are event edges, so stream capture records them as graph edges.  The mutex
// keeps two host threads from interleaving on the shared events.
struct SideStream {
    cudaStream_t s = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};
std::mutex g_side_mu;
SideStream g_side[64];

cudaError_t side_stream(SideStream** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    SideStream& sd = g_side[dev];
    if (sd.s == nullptr) {
        if ((e = cudaStreamCreateWithFlags(&sd.s, cudaStreamNonBlocking)) != cudaSuccess) return e;
        if ((e = cudaEventCreateWithFlags(&sd.fork, cudaEventDisableTiming)) != cudaSuccess) return e;
        if ((e = cudaEventCreateWithFlags(&sd.join, cudaEventDisableTiming)) != cudaSuccess) return e;
    }
    *out = &sd;
    return cudaSuccess;
}

struct Launched {
    const Args* a;
    Dims d;
    Scenario sc;
    Plan p;
    uint8_t* ws;
    cudaStream_t st;
    int sms;
};

GemmArgs gemm_args(const GemmPlan& g, int T, int64_t ncols, uint32_t* status) {
    GemmArgs a = {};
    a.T = T;
    a.kblocks = g.kblocks;
    a.ncols = (int)ncols;
    a.n_tiles = g.n_tiles;
    a.m_tiles = g.m_tiles;
    a.ksplit = g.ksplit;
    a.b_split_col = INT32_MAX;
    a.a_box_rows = g.a_box_rows;
    a.status = status;
    return a;
}

mla_status run(const Launched& L) {
    const Args& a = *L.a;
    const Dims& d = L.d;
    const Scenario& sc = L.sc;
    const Plan& p = L.p;
    uint8_t* ws = L.ws;
    cudaStream_t st = L.st;
    uint32_t* status = reinterpret_cast<uint32_t*>(ws);
    const int T = (int)d.T;
    if (!get_encoder()) return MLA_ERR_RUNTIME;
    SideStream* side = nullptr;   // set once work is forked onto the side stream
    std::unique_lock<std::mutex> side_lock(g_side_mu, std::defer_lock);

    // int8 tokenX: its codes widened to fp16 (exact), the A operand of the int8-weight GEMM; the
    // int8 weights stay int8 in HBM and are widened in shared memory.
    const void* x_bf = a.x->data;
    const void* wdq_bf = a.wdq->data;
    const void* wdkvkr_bf = a.wdkvkr->data;
    const void* wuqqr_bf = a.wuqqr->data;
    // When its fp16 A slots leave room for three stages (one row tile, T <= 64 at these shapes)
    // the down-projection loads tokenX as int8 and widens it in shared memory beside the
    // weights: no widening launch.
    const bool x_a8 = sc.x_i8 && p.g1.msub == 1 &&
                      (p.g1.bn == 192 ? W8Cfg<192, 1, 16, true, true>::max_stages(p.g1.a_box_rows)
                                      : W8Cfg<64, 1, 16, true, true>::max_stages(p.g1.a_box_rows)) >= 3;
    if (sc.x_i8 && !x_a8) {
        const long long n = (long long)d.T * d.He;
        const long long blocks = (n / 16 + 255) / 256;
        const int grid = (int)(blocks < 4096 ? (blocks > 0 ? blocks : 1) : 4096);
        if (launch(convert_i8_to_f16_kernel, grid, 256, 0, st, static_cast<const int8_t*>(a.x->data),
                   reinterpret_cast<__half*>(ws + p.off_xb), n) != cudaSuccess)
            return MLA_ERR_RUNTIME;
        timing_mark(st, "widen_x");
        x_bf = ws + p.off_xb;
    }

    DownArgs f1 = {};
    f1.T = T;
    f1.Hcq = (int)d.Hcq;
    f1.Hckv = (int)d.Hckv;
    f1.Dr = (int)d.Dr;
    float* y1 = reinterpret_cast<float*>(ws + p.off_y1);
    f1.src = {y1, (int)p.ncols1, p.g1.ksplit, (size_t)d.T * p.ncols1};
    if (sc.x_i8) {
        f1.scale_x = static_cast<const float*>(a.sx->data);
        f1.scale_w_dq = static_cast<const float*>(a.swdq->data);
        f1.scale_w_dkvkr = static_cast<const float*>(a.swdkvkr->data);
    }
    f1.gamma_cq = static_cast<const __nv_bfloat16*>(a.gcq->data);
    f1.gamma_ckv = static_cast<const __nv_bfloat16*>(a.gckv->data);
    f1.eps_cq = (float)a.eps_cq;
    f1.eps_ckv = (float)a.eps_ckv;
    f1.rope_cos = static_cast<const __nv_bfloat16*>(a.cos->data);
    f1.rope_sin = static_cast<const __nv_bfloat16*>(a.sin->data);
    f1.cache_index = static_cast<const long long*>(a.idx->data);
    f1.nslots = d.block_num * d.block_size;
    f1.kv_cache = a.kv->data;
    f1.kv_int8 = sc.kv_i8;
    f1.quant_scale_ckv = a.qckv ? static_cast<const float*>(a.qckv->data) : nullptr;
    f1.kr_cache = a.kr->data;
    f1.kr_int8 = sc.kr_i8;
    f1.quant_scale_ckr = a.qckr ? static_cast<const float*>(a.qckr->data) : nullptr;
    f1.c_q = reinterpret_cast<__nv_bfloat16*>(ws + p.off_cq);
    f1.cq_quant = sc.uqqr_i8;
    f1.smooth_cq = a.smooth ? static_cast<const float*>(a.smooth->data) : nullptr;
    f1.c_q_scale = reinterpret_cast<float*>(ws + p.off_cqs);
    f1.cq_done = p.fold_cq ? 1 : 0;
    f1.status = status;
    const float* row_scale = sc.uqqr_i8 ? reinterpret_cast<const float*>(ws + p.off_cqs) : nullptr;
    const float* col_scale = sc.uqqr_i8 ? static_cast<const float*>(a.swuqqr->data) : nullptr;
    __nv_bfloat16* qc = reinterpret_cast<__nv_bfloat16*>(ws + p.off_qc);
    cudaError_t e;

    // The 3D map of q^C (one head's T x D slice per box) and of W^UK (one head's D x Hckv).
    // Row tiles of 128 tokens take both k-blocks of D = 128 in one stage.
    CUtensorMap mA3, mB3;
    const bool kps3 = !sc.q_i8 && p.g3.m_tiles > 1 && p.g3.kblocks % 2 == 0;   // 512-column int8 tiles: no room
    const bool blocks3 = d.D % 64 == 0 && d.Hckv % 64 == 0;   // whole-k-block boxes of all column blocks
    const uint32_t a3_rows = (uint32_t)p.g3.a_box_rows;
    {
        const uint64_t dims[3] = {(uint64_t)d.D, (uint64_t)d.N, (uint64_t)d.T};
        const uint64_t strides[2] = {(uint64_t)d.D * 2, (uint64_t)d.N * d.D * 2};
        const uint32_t box[3] = {64, 1, a3_rows};
        if (!encode_map(&mA3, qc, 3, dims, strides, box)) return MLA_ERR_RUNTIME;
        if (blocks3) {
            // W^UK as (64 columns, N * D rows, Hckv / 64 blocks): one box per stage brings every
            // column block of the tile (8 KB boxes move far fewer bytes per SM per second)
            if (!map_colblocks(&mB3, a.wuk->data, (uint64_t)d.N * d.D, d.Hckv, kps3 ? 128u : 64u,
                               (uint32_t)(p.g3.bn / 64)))
                return MLA_ERR_RUNTIME;
        } else {
            const uint64_t dimsb[3] = {(uint64_t)d.Hckv, (uint64_t)d.D, (uint64_t)d.N};
            const uint64_t stridesb[2] = {(uint64_t)d.Hckv * 2, (uint64_t)d.D * d.Hckv * 2};
            const uint32_t boxb[3] = {64, kps3 ? 128u : 64u, 1};
            if (!encode_map(&mB3, a.wuk->data, 3, dimsb, stridesb, boxb)) return MLA_ERR_RUNTIME;
        }
    }

    if (p.persist) {
        // ---- the whole prolog in one persistent kernel
        const uint32_t rows = (uint32_t)p.p_arows;
        // weights as (64 columns, k rows, 64-column blocks): one box brings a 192-column stage
        CUtensorMap mx, mwdq, mwdkvkr, mcq, mwuqqr, mwuk, mo;
        const uint64_t ocols = (uint64_t)d.N * (uint64_t)d.Hckv;
        const uint64_t odims[2] = {ocols, (uint64_t)d.T};
        const uint64_t ostrides[1] = {ocols * 2};
        const uint32_t obox[2] = {64, (uint32_t)((d.T + 3) / 4)};   // one lane quarter's tokens
        if (!map_2d(&mx, x_bf, d.T, d.He, rows) || !map_colblocks(&mwdq, wdq_bf, d.He, d.Hcq, 64, 3) ||
            !map_colblocks(&mwdkvkr, wdkvkr_bf, d.He, d.Hckv + d.Dr, 64, 3) ||
            !map_2d(&mcq, ws + p.off_cq, d.T, d.Hcq, rows) || !map_colblocks(&mwuqqr, wuqqr_bf, d.Hcq, p.ncols2, 64, 3) ||
            !map_colblocks(&mwuk, a.wuk->data, d.N * d.D, d.Hckv, 64, 3) ||
            !encode_map(&mo, a.qout->data, 2, odims, ostrides, obox))
            return MLA_ERR_RUNTIME;
        PersistArgs pa = {};
        pa.T = T;
        pa.a_rows = (int)rows;
        pa.a_bytes = (int)rows * 128;
        pa.wst = p.p_wst;
        pa.na3 = p.p_na3;
        pa.pf = p.p_pf;
        pa.hcq = (int)d.Hcq;
        pa.hckv = (int)d.Hckv;
        pa.dr = (int)d.Dr;
        pa.ncols1 = (int)p.ncols1;
        pa.n1 = p.p_n1;
        pa.s1 = p.p_s1;
        pa.kb1 = (int)(d.He / 64);
        pa.y = y1;
        pa.zflags = reinterpret_cast<unsigned long long*>(ws + p.off_pbar);
        pa.cnt = reinterpret_cast<unsigned int*>(ws + p.off_pbar + (size_t)p.p_n1 * 8);
        pa.cqflags = reinterpret_cast<unsigned long long*>(ws + p.off_pbar + (((size_t)p.p_n1 * 12 + 7) & ~(size_t)7));
        pa.ss = reinterpret_cast<float*>(pa.cqflags + d.Hcq / kPChunk);
        pa.cq = f1.c_q;
        pa.gamma_cq = f1.gamma_cq;
        pa.gamma_ckv = f1.gamma_ckv;
        pa.eps_cq = f1.eps_cq;
        pa.eps_ckv = f1.eps_ckv;
        pa.cache_index = f1.cache_index;
        pa.nslots = f1.nslots;
        pa.kv_cache = static_cast<__nv_bfloat16*>(a.kv->data);
        pa.kr_cache = static_cast<__nv_bfloat16*>(a.kr->data);
        pa.rope_cos = f1.rope_cos;
        pa.rope_sin = f1.rope_sin;
        pa.N = (int)d.N;
        pa.kb2 = (int)(d.Hcq / 64);
        pa.q_rope = static_cast<__nv_bfloat16*>(a.qrope->data);
        pa.q_out = static_cast<__nv_bfloat16*>(a.qout->data);
        pa.tag = next_tag();
        pa.status = status;
        e = set_attr(decode_persist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.p_smem);
        if (e != cudaSuccess) return MLA_ERR_RUNTIME;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)L.sms);
        cfg.blockDim = dim3((unsigned)kPThreads);
        cfg.dynamicSmemBytes = p.p_smem;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;   // all CTAs co-resident: the grid barriers need it
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, decode_persist_kernel, mx, mwdq, mwdkvkr, mcq, mwuqqr, mwuk, mo, pa);
        if (e == cudaSuccess) {
            timing_mark(st, "decode_persist");
            if (g_timing.enabled) g_timing.have = true;
            return MLA_OK;
        }
        // Not every CTA can be resident (another context holds SMs): run the kernel-per-step path.
        if (e != cudaErrorCooperativeLaunchTooLarge) return MLA_ERR_RUNTIME;
        (void)cudaGetLastError();
    }

    // ---- K1: down-projection x . [W^DQ | W^DKV | W^KR] -> fp32 rows Y1
    CUtensorMap mA1, mB1a, mB1b;
    if (sc.x_i8) {
        // int8 weights streamed as int8 and widened in shared memory (fp16 x fp16 -> fp32, exact
        // integer sums); F1 applies tokenX's and the weights' dequant scales
        constexpr int BN = 192;
        if (p.g1.bn != BN && p.g1.bn != 64) return MLA_ERR_TILING;
        if (!(x_a8 ? map_w8_rows(&mA1, a.x->data, d.T, d.He, (uint32_t)p.g1.a_box_rows)
                   : map_2d(&mA1, x_bf, d.T, d.He, (uint32_t)p.g1.a_box_rows)) ||
            !map_w8_cols(&mB1a, a.wdq->data, d.He, d.Hcq, (uint32_t)p.g1.bn) ||
            !map_w8_cols(&mB1b, a.wdkvkr->data, d.He, d.Hckv + d.Dr, (uint32_t)p.g1.bn))
            return MLA_ERR_RUNTIME;
        GemmArgs g1 = gemm_args(p.g1, T, p.ncols1, status);
        g1.b_split_col = (int)d.Hcq;
        g1.clear_status = 1;
        g1.out_f32 = y1;
        g1.a_ready = x_a8 ? 1 : 0;   // int8 tokenX is read as passed
        if (p.g1.bn == BN)
            e = x_a8                ? launch_gemm_w8<BN, 1, 16, true, EPI_F32, true>(p.g1.grid, st, mA1, mB1a, mB1b, g1)
                : p.g1.msub == 1 ? launch_gemm_w8<BN, 1, 16, true>(p.g1.grid, st, mA1, mB1a, mB1b, g1)
                                 : launch_gemm_w8<BN, 2, 16, true>(p.g1.grid, st, mA1, mB1a, mB1b, g1);
        else
            e = x_a8                ? launch_gemm_w8<64, 1, 16, true, EPI_F32, true>(p.g1.grid, st, mA1, mB1a, mB1b, g1)
                : p.g1.msub == 1 ? launch_gemm_w8<64, 1, 16, true>(p.g1.grid, st, mA1, mB1a, mB1b, g1)
                                 : launch_gemm_w8<64, 2, 16, true>(p.g1.grid, st, mA1, mB1a, mB1b, g1);
    } else {
    // 256-row tiles store their fp32 rows through shared memory with TMA (32 x 32 boxes of the
    // T x ncols1 matrix, or of the ksplit slots stacked when T is a multiple of 32); other k
    // ranges use plain stores into their slots.
    const bool tma1 = p.g1.msub == 2 && p.ncols1 % 4 == 0 && (p.g1.ksplit == 1 || d.T % 32 == 0);
    // 256-column tiles: one 256-row activation box and one column-blocked weight box per k-block
    const bool big1 = !p.g1_pair && p.g1.bn == 256 && d.Hcq % 256 == 0 && (d.Hckv + d.Dr) % 64 == 0;
    if (p.g1_pair) {
        if (!map_colblocks(&mA1, x_bf, d.T, d.He, 128, kPairKps) ||
            !map_colblocks(&mB1a, wdq_bf, d.He, d.Hcq, 64 * kPairKps, 2) ||
            !map_colblocks(&mB1b, wdkvkr_bf, d.He, d.Hckv + d.Dr, 64 * kPairKps, 2))
            return MLA_ERR_RUNTIME;
    } else if (big1) {
        if (!map_2d(&mA1, x_bf, d.T, d.He, 256) || !map_colblocks(&mB1a, wdq_bf, d.He, d.Hcq, 64, 4) ||
            !map_colblocks(&mB1b, wdkvkr_bf, d.He, d.Hckv + d.Dr, 64, 4))
            return MLA_ERR_RUNTIME;
    } else if (!map_2d(&mA1, x_bf, d.T, d.He, (uint32_t)p.g1.a_box_rows) || !map_2d(&mB1a, wdq_bf, d.He, d.Hcq, 64) ||
               !map_2d(&mB1b, wdkvkr_bf, d.He, d.Hckv + d.Dr, 64)) {
        return MLA_ERR_RUNTIME;
    }
    GemmArgs g1 = gemm_args(p.g1, T, p.ncols1, status);
    g1.b_split_col = (int)d.Hcq;
    g1.clear_status = 1;
    g1.a_ready = 1;   // bf16 tokenX is read as passed
    g1.a_one_box = big1 ? 1 : 0;
    g1.b_blocks = big1 ? 1 : 0;
    CUtensorMap mO1;
    if (tma1) {
        const uint64_t dims[2] = {(uint64_t)p.ncols1, (uint64_t)d.T * (uint64_t)p.g1.ksplit};
        const uint64_t strides[1] = {(uint64_t)p.ncols1 * 4};
        const uint32_t box[2] = {32, 32};
        g1.tma_out = encode_map(&mO1, y1, 2, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_FLOAT32) ? 1 : 0;
    }
    g1.out_f32 = y1;
    if (p.g1_pair && !g1.tma_out) return MLA_ERR_RUNTIME;   // pair tiles store only through TMA
    g1.n_fastest = 1;   // x (T x He) is larger than the weights: read each row tile once
    if (p.fold_cq) {
        CUtensorMap mCq;
        const uint64_t dims[2] = {(uint64_t)d.Hcq, (uint64_t)d.T};
        const uint64_t strides[1] = {(uint64_t)d.Hcq * 2};
        const uint32_t box[2] = {64, 32};
        if (!encode_map(&mCq, ws + p.off_cq, 2, dims, strides, box)) return MLA_ERR_RUNTIME;
        g1.cq_cols = (int)d.Hcq;
        g1.gamma_cq = f1.gamma_cq;
        g1.ss_out = reinterpret_cast<float*>(ws + p.off_ss);
        g1.nss = (int)(d.Hcq / 256) * 2;
        e = launch_gemm_pair<256, 8, EPI_DOWN, 1, 2, kPairKps>(st, mA1, mB1a, mB1b, g1, mO1, mCq);
    } else if (p.g1_pair)
        e = launch_gemm_pair<256, 8, EPI_F32, 1, 2, kPairKps>(st, mA1, mB1a, mB1b, g1, mO1, mO1);
    else if (p.g1.bn == 64)
        e = launch_gemm<64, 1, 32, EPI_F32>(p.g1.grid, st, mA1, mB1a, mB1b, g1);
    else
        e = p.g1.bn == 256 ? (g1.tma_out && big1
                                  ? launch_gemm<256, 2, 4, EPI_F32, 1, 1, 2>(p.g1.grid, st, mA1, mB1a, mB1b, g1, &mO1)
                                  : launch_gemm<256, 2, 4, EPI_F32>(p.g1.grid, st, mA1, mB1a, mB1b, g1))
                           : (g1.tma_out ? launch_gemm<192, 2, 4, EPI_F32, 2>(p.g1.grid, st, mA1, mB1a, mB1b, g1, &mO1)
                                         : launch_gemm<192, 2, 4, EPI_F32>(p.g1.grid, st, mA1, mB1a, mB1b, g1));
    }
    if (e != cudaSuccess) return MLA_ERR_RUNTIME;
    timing_mark(st, "k1_down_proj");

    // ---- F1: RmsNorm, RoPE(k^R), cache writes, c^Q
    if (T > kDecodeRows && p.g1.ksplit == 1 && d.Dr == 64 && d.Hcq % 64 == 0 && d.Hckv % 64 == 0 &&
        d.Hcq <= 64 * kWQ && d.Hckv <= 64 * kWKV) {
        // many tokens: one warp per token, the row in registers
        const int wpc = kWarpRowThreads / 32;
        if (p.fold_cq && !g_timing.enabled) {
            // only the cache rows are left, and no later kernel of the call reads them: on the
            // side stream, beside K2 / K3
            SideStream* sd = nullptr;
            if (side_stream(&sd) != cudaSuccess) return MLA_ERR_RUNTIME;
            side_lock.lock();
            side = sd;
            if (cudaEventRecord(sd->fork, st) != cudaSuccess || cudaStreamWaitEvent(sd->s, sd->fork, 0) != cudaSuccess)
                return MLA_ERR_RUNTIME;
            e = launch(finalize_down_warp_kernel, (T + wpc - 1) / wpc, kWarpRowThreads, 0, sd->s, f1);
            if (e != cudaSuccess || cudaEventRecord(sd->join, sd->s) != cudaSuccess) return MLA_ERR_RUNTIME;
        } else {
            e = launch(finalize_down_warp_kernel, (T + wpc - 1) / wpc, kWarpRowThreads, 0, st, f1);
            if (e != cudaSuccess) return MLA_ERR_RUNTIME;
            timing_mark(st, "f1_norm_rope_cache");
        }
    } else {
        const int grid = T < 16 * L.sms ? T : 16 * L.sms;
        const size_t fsmem = down_smem_bytes((int)d.Hcq, (int)d.Hckv, (int)d.Dr);
        // decode-sized T: 512 threads per token, each with all k-range partials of its five
        // columns in flight at once (the k ranges number at most 16 there); many rows: fewer
        // loads in flight, so that more rows fit on an SM
        const bool wide = T <= kDecodeRows && p.g1.ksplit <= 16;
        auto fk = wide ? finalize_down_kernel<5, 512, 16> : finalize_down_kernel<3>;
        e = set_attr(fk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)fsmem);
        if (e != cudaSuccess) return MLA_ERR_RUNTIME;
        e = launch(fk, grid, wide ? 512 : kRowThreads, fsmem, st, f1);
        if (e != cudaSuccess) return MLA_ERR_RUNTIME;
        timing_mark(st, "f1_norm_rope_cache");
    }

    // ---- K2: up-projection c^Q . W^UqQr -> RoPE(q^R) and q^C
    CUtensorMap mA2, mB2;
    // Prefill tiles without dequant scales store q^C and q^R through shared memory with TMA.
    const bool tma2 = p.g2_fused && (p.g2.msub == 2 || p.g2_wide) && !sc.uqqr_i8;
    // SM-pair tiles: per k-block each CTA takes one 128-row activation box and one box of its
    // 128 weight columns (two 64-column blocks)
    if (p.g2_wide) {
        if (!map_colblocks(&mA2, ws + p.off_cq, d.T, d.Hcq, 128, kPairKps) ||
            !map_colblocks(&mB2, wuqqr_bf, d.Hcq, p.ncols2, 64 * kPairKps, 2))
            return MLA_ERR_RUNTIME;
    } else if (sc.uqqr_i8) {
        // int8 W^UqQr streamed as int8 and widened in shared memory; c^Q's int8 codes as fp16
        if (!map_2d(&mA2, ws + p.off_cq, d.T, d.Hcq, (uint32_t)p.g2.a_box_rows) ||
            !map_w8_cols(&mB2, a.wuqqr->data, d.Hcq, p.ncols2, 192))
            return MLA_ERR_RUNTIME;
    } else if (!map_2d(&mA2, ws + p.off_cq, d.T, d.Hcq, (uint32_t)p.g2.a_box_rows) ||
               !map_2d(&mB2, wuqqr_bf, d.Hcq, p.ncols2, 64)) {
        return MLA_ERR_RUNTIME;
    }
    GemmArgs g2 = gemm_args(p.g2, T, p.ncols2, status);
    g2.a_one_box = p.g2_wide ? 1 : 0;
    g2.b_blocks = p.g2_wide ? 1 : 0;
    CUtensorMap mO2c, mO2r;
    if (tma2) {
        const uint64_t dc[2] = {(uint64_t)d.N * d.D, (uint64_t)d.T};
        const uint64_t sc2[1] = {(uint64_t)d.N * d.D * 2};
        const uint64_t dr[2] = {(uint64_t)d.N * d.Dr, (uint64_t)d.T};
        const uint64_t sr[1] = {(uint64_t)d.N * d.Dr * 2};
        const uint32_t box[2] = {64, 32};
        g2.tma_out = encode_map(&mO2c, qc, 2, dc, sc2, box) && encode_map(&mO2r, a.qrope->data, 2, dr, sr, box) ? 1 : 0;
    }
    if (p.g2_wide && !g2.tma_out) return MLA_ERR_RUNTIME;   // 256-column tiles store only through TMA
    g2.N = (int)d.N;
    g2.q_c = qc;
    g2.q_rope = static_cast<__nv_bfloat16*>(a.qrope->data);
    g2.rope_cos = f1.rope_cos;
    g2.rope_sin = f1.rope_sin;
    if (p.fold_cq) {
        g2.ss_in = reinterpret_cast<const float*>(ws + p.off_ss);
        g2.nss = (int)(d.Hcq / 256) * 2;
        g2.hcq = (int)d.Hcq;
        g2.eps_cq = f1.eps_cq;
    }
    g2.row_scale = row_scale;
    g2.col_scale = col_scale;
    g2.out_f32 = reinterpret_cast<float*>(ws + p.off_y2);
    if (sc.uqqr_i8) {
        if (p.g2.bn != 192) return MLA_ERR_TILING;
        g2.b_split_col = (int)p.ncols2;   // every column from the one map
        if (p.g2_fused)
            e = (p.g2.msub == 1)
                    ? launch_gemm_w8<192, 1, 16, true, EPI_QROPE>(p.g2.grid, st, mA2, mB2, mB2, g2)
                    : launch_gemm_w8<192, 2, 16, true, EPI_QROPE>(p.g2.grid, st, mA2, mB2, mB2, g2);
        else
            e = (p.g2.msub == 1) ? launch_gemm_w8<192, 1, 16, true>(p.g2.grid, st, mA2, mB2, mB2, g2)
                                 : launch_gemm_w8<192, 2, 16, true>(p.g2.grid, st, mA2, mB2, mB2, g2);
    } else if (p.g2_fused) {
        if (p.g2_wide)
            e = launch_gemm_pair<256, 8, EPI_QROPE, 1, 2, kPairKps>(st, mA2, mB2, mB2, g2, mO2c, mO2r);
        else if (p.g2.msub == 1)
            e = launch_gemm<192, 1, 16, EPI_QROPE>(p.g2.grid, st, mA2, mB2, mB2, g2);
        else
            e = g2.tma_out ? launch_gemm<192, 2, 4, EPI_QROPE, 2>(p.g2.grid, st, mA2, mB2, mB2, g2, &mO2c, &mO2r)
                           : launch_gemm<192, 2, 4, EPI_QROPE>(p.g2.grid, st, mA2, mB2, mB2, g2);
    } else {
        e = (p.g2.msub == 1) ? launch_gemm<192, 1, 16, EPI_F32>(p.g2.grid, st, mA2, mB2, mB2, g2)
                             : launch_gemm<192, 2, 4, EPI_F32>(p.g2.grid, st, mA2, mB2, mB2, g2);
    }
    if (e != cudaSuccess) return MLA_ERR_RUNTIME;
    timing_mark(st, "k2_up_proj");
    if (!p.g2_fused) {
        UpArgs f2 = {};
        f2.T = T;
        f2.N = (int)d.N;
        f2.D = (int)d.D;
        f2.Dr = (int)d.Dr;
        f2.src = {reinterpret_cast<const float*>(ws + p.off_y2), (int)p.ncols2, 1, (size_t)d.T * p.ncols2};
        f2.row_scale = row_scale;
        f2.col_scale = col_scale;
        f2.rope_cos = f1.rope_cos;
        f2.rope_sin = f1.rope_sin;
        f2.q_c = qc;
        f2.q_rope = static_cast<__nv_bfloat16*>(a.qrope->data);
        const int grid = T < 16 * L.sms ? T : 16 * L.sms;
        e = launch(finalize_up_kernel, grid, kRowThreads, 0, st, f2);
        if (e != cudaSuccess) return MLA_ERR_RUNTIME;
        timing_mark(st, "f2_rope_qc");
    }

    // ---- K3: per-head W^UK contraction
    GemmArgs g3 = gemm_args(p.g3, T, d.Hckv, status);
    g3.head_mode = 1;
    g3.b_blocks = blocks3 ? 1 : 0;
    g3.head_rows = (int)d.D;
    g3.tiles_per_head = p.g3.n_tiles / (int)d.N;
    g3.N = (int)d.N;
    g3.Hckv = (int)d.Hckv;
    // queryOut as a (T, N * Hckv) matrix for TMA stores of 32-row x 128-byte boxes (whole boxes
    // stay inside one head when Hckv is a multiple of the box width).
    CUtensorMap mO3;
    {
        const uint64_t cols = (uint64_t)d.N * (uint64_t)d.Hckv;
        if (sc.q_i8) {
            const uint64_t dims[2] = {cols, (uint64_t)d.T};
            const uint64_t strides[1] = {cols};
            const uint32_t box[2] = {128, 32};
            g3.tma_out = d.Hckv % 128 == 0 && encode_map(&mO3, a.qout->data, 2, dims, strides, box,
                                                          CU_TENSOR_MAP_DATA_TYPE_UINT8);
        } else {
            const uint64_t dims[2] = {cols, (uint64_t)d.T};
            const uint64_t strides[1] = {cols * 2};
            const uint32_t box[2] = {64, 32};
            g3.tma_out = d.Hckv % 64 == 0 && encode_map(&mO3, a.qout->data, 2, dims, strides, box);
        }
    }
    if (sc.q_i8) {
        g3.q_out_i8 = static_cast<int8_t*>(a.qout->data);
        g3.q_scale = static_cast<float*>(a.qscale->data);
        // two warps per TMEM lane quarter, each with 256 of the 512 columns (TMA-stored boxes)
        e = g3.tma_out ? launch_gemm<512, 1, 4, EPI_QN, 1, 1, 2>(p.g3.grid, st, mA3, mB3, mB3, g3, &mO3)
                       : launch_gemm<512, 1, 4, EPI_QN, 2>(p.g3.grid, st, mA3, mB3, mB3, g3, nullptr);
    } else {
        g3.q_out_bf16 = static_cast<__nv_bfloat16*>(a.qout->data);
        e = kps3 ? launch_gemm<256, 1, 8, EPI_QN, 2, 2>(p.g3.grid, st, mA3, mB3, mB3, g3, g3.tma_out ? &mO3 : nullptr)
                 : launch_gemm<256, 1, 8, EPI_QN, 2>(p.g3.grid, st, mA3, mB3, mB3, g3, g3.tma_out ? &mO3 : nullptr);
    }
    if (e != cudaSuccess) return MLA_ERR_RUNTIME;
    timing_mark(st, "k3_absorb_uk");
    if (side != nullptr && cudaStreamWaitEvent(st, side->join, 0) != cudaSuccess) return MLA_ERR_RUNTIME;
    if (g_timing.enabled) g_timing.have = true;
    return MLA_OK;
}

}  // namespace

// ====================================================================== C ABI

#define MLA_TENSOR_PARAMS                                                                                      \
    const mla_tensor *tokenX, const mla_tensor *weightDq, const mla_tensor *weightUqQr,                        \
        const mla_tensor *weightUk, const mla_tensor *weightDkvKr, const mla_tensor *rmsnormGammaCq,          \
        const mla_tensor *rmsnormGammaCkv, const mla_tensor *ropeSin, const mla_tensor *ropeCos,              \
        const mla_tensor *cacheIndex, const mla_tensor *kvCache, const mla_tensor *krCache,                   \
        const mla_tensor *dequantScaleX, const mla_tensor *dequantScaleWDq,                                   \
        const mla_tensor *dequantScaleWUqQr, const mla_tensor *dequantScaleWDkvKr,                            \
        const mla_tensor *quantScaleCkv, const mla_tensor *quantScaleCkr, const mla_tensor *smoothScalesCq,   \
        double rmsnormEpsilonCq, double rmsnormEpsilonCkv, const char *cacheMode, const mla_tensor *queryOut, \
        const mla_tensor *queryRopeOut, const mla_tensor *dequantScaleQNopeOut

static Args pack_args(MLA_TENSOR_PARAMS) {
    Args a;
    a.x = tokenX;
    a.wdq = weightDq;
    a.wuqqr = weightUqQr;
    a.wuk = weightUk;
    a.wdkvkr = weightDkvKr;
    a.gcq = rmsnormGammaCq;
    a.gckv = rmsnormGammaCkv;
    a.sin = ropeSin;
    a.cos = ropeCos;
    a.idx = cacheIndex;
    a.kv = kvCache;
    a.kr = krCache;
    a.sx = dequantScaleX;
    a.swdq = dequantScaleWDq;
    a.swuqqr = dequantScaleWUqQr;
    a.swdkvkr = dequantScaleWDkvKr;
    a.qckv = quantScaleCkv;
    a.qckr = quantScaleCkr;
    a.smooth = smoothScalesCq;
    a.eps_cq = rmsnormEpsilonCq;
    a.eps_ckv = rmsnormEpsilonCkv;
    a.cache_mode = cacheMode;
    a.qout = queryOut;
    a.qrope = queryRopeOut;
    a.qscale = dequantScaleQNopeOut;
    return a;
}

#define MLA_TENSOR_ARGS                                                                                          \
    tokenX, weightDq, weightUqQr, weightUk, weightDkvKr, rmsnormGammaCq, rmsnormGammaCkv, ropeSin, ropeCos,     \
        cacheIndex, kvCache, krCache, dequantScaleX, dequantScaleWDq, dequantScaleWUqQr, dequantScaleWDkvKr,    \
        quantScaleCkv, quantScaleCkr, smoothScalesCq, rmsnormEpsilonCq, rmsnormEpsilonCkv, cacheMode, queryOut, \
        queryRopeOut, dequantScaleQNopeOut

extern "C" mla_status mla_prolog_workspace_size(MLA_TENSOR_PARAMS, uint64_t* workspaceSize) {
    if (workspaceSize == nullptr) return MLA_ERR_PARAM_NULLPTR;
    const Args a = pack_args(MLA_TENSOR_ARGS);
    Dims d;
    Scenario sc;
    const mla_status s = validate(a, d, sc);
    if (s != MLA_OK) return s;
    if (d.T == 0) {
        *workspaceSize = kStatusBytes;
        return MLA_OK;
    }
    int sms = 0;
    if (device_sms(&sms) != 0) return MLA_ERR_RUNTIME;
    *workspaceSize = make_plan(d, sc, sms).bytes;
    return MLA_OK;
}

extern "C" mla_status mla_prolog(MLA_TENSOR_PARAMS, void* workspace, uint64_t workspaceSize, void* stream) {
    const Args a = pack_args(MLA_TENSOR_ARGS);
    Dims d;
    Scenario sc;
    const mla_status s = validate(a, d, sc);
    if (s != MLA_OK) return s;
    if (d.T == 0) return MLA_OK;
    if (workspace == nullptr) return MLA_ERR_PARAM_NULLPTR;
    if ((reinterpret_cast<uintptr_t>(workspace) & 15u) != 0) return MLA_ERR_PARAM_INVALID;
    int sms = 0;
    if (device_sms(&sms) != 0) return MLA_ERR_RUNTIME;
    Launched L{&a, d, sc, make_plan(d, sc, sms), static_cast<uint8_t*>(workspace),
               static_cast<cudaStream_t>(stream), sms};
    if (workspaceSize < L.p.bytes) return MLA_ERR_PARAM_INVALID;
    timing_begin(L.st);
    return run(L);
}

// ------------------------------------------------------- no-allocation variant

// The workspace of mla_prolog_no_alloc(): one buffer per device, part of the library's
// device image.  Host code must not use this name as a device address; the address is
// looked up once per device with cudaGetSymbolAddress.
static __device__ __align__(256) uint8_t g_no_alloc_scratch[MLA_NO_ALLOC_SCRATCH_BYTES];

static constexpr int kMaxDevices = 64;
static std::mutex g_scratch_mu;
static void* g_scratch_addr[kMaxDevices] = {};
static unsigned long long g_scratch_ctx[kMaxDevices] = {};   // id of the context the address belongs to

// The unique id of the calling thread's current CUDA context (driver entry points, looked up
// once); false when there is no current context or the driver does not offer the calls.
typedef CUresult (*PFN_ctx_current)(CUcontext*);
typedef CUresult (*PFN_ctx_id)(CUcontext, unsigned long long*);
static PFN_ctx_current g_ctx_current = nullptr;
static PFN_ctx_id g_ctx_id = nullptr;
static std::once_flag g_ctx_once;

static bool current_context_id(unsigned long long* id) {
    std::call_once(g_ctx_once, [] {
        void* f1 = nullptr;
        void* f2 = nullptr;
        cudaDriverEntryPointQueryResult q1, q2;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1) == cudaSuccess &&
            q1 == cudaDriverEntryPointSuccess &&
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) == cudaSuccess &&
            q2 == cudaDriverEntryPointSuccess) {
            g_ctx_current = reinterpret_cast<PFN_ctx_current>(f1);
            g_ctx_id = reinterpret_cast<PFN_ctx_id>(f2);
        }
    });
    if (g_ctx_current == nullptr || g_ctx_id == nullptr) return false;
    CUcontext ctx = nullptr;
    if (g_ctx_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
    return g_ctx_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the scratch buffer on the current device.  Looked up on the first call on
// a device, and again whenever the current context is not the one the address was found in
// (after cudaDeviceReset the module is loaded anew and the buffer may move).  Without the
// context-id calls the address is looked up on every call.
static mla_status no_alloc_scratch(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MLA_ERR_RUNTIME;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    unsigned long long id = 0;
    const bool have_id = current_context_id(&id);
    if (g_scratch_addr[dev] == nullptr || !have_id || g_scratch_ctx[dev] != id) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_no_alloc_scratch) != cudaSuccess || p == nullptr) return MLA_ERR_RUNTIME;
        g_scratch_addr[dev] = p;
        // the lookup made the device's primary context current if no context was
        unsigned long long id2 = 0;
        g_scratch_ctx[dev] = current_context_id(&id2) ? id2 : 0;
    }
    *out = g_scratch_addr[dev];
    return MLA_OK;
}

extern "C" mla_status mla_prolog_no_alloc(MLA_TENSOR_PARAMS, void* stream) {
    const Args a = pack_args(MLA_TENSOR_ARGS);
    Dims d;
    Scenario sc;
    const mla_status s = validate(a, d, sc);
    if (s != MLA_OK) return s;
    if (d.T == 0) return MLA_OK;
    int sms = 0;
    if (device_sms(&sms) != 0) return MLA_ERR_RUNTIME;
    const Plan plan = make_plan(d, sc, sms);
    if (plan.bytes > MLA_NO_ALLOC_SCRATCH_BYTES) return MLA_ERR_SCRATCH_LIMIT;
    void* ws = nullptr;
    const mla_status ss = no_alloc_scratch(&ws);
    if (ss != MLA_OK) return ss;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // The status word starts at zero; everything else the kernels read they write first.
    if (cudaMemsetAsync(ws, 0, kStatusBytes, st) != cudaSuccess) return MLA_ERR_RUNTIME;
    Launched L{&a, d, sc, plan, static_cast<uint8_t*>(ws), st, sms};
    timing_begin(L.st);
    return run(L);
}

extern "C" mla_status mla_prolog_no_alloc_status(void* stream, uint32_t* bits) {
    if (bits == nullptr) return MLA_ERR_PARAM_NULLPTR;
    void* ws = nullptr;
    const mla_status ss = no_alloc_scratch(&ws);
    if (ss != MLA_OK) return ss;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MLA_ERR_RUNTIME;
    if (cudaMemcpy(bits, ws, sizeof(uint32_t), cudaMemcpyDeviceToHost) != cudaSuccess) return MLA_ERR_RUNTIME;
    return MLA_OK;
}

extern "C" mla_status mla_prolog_device_status(const void* workspace, uint64_t workspaceSize, void* stream,
                                               uint32_t* bits) {
    if (workspace == nullptr || bits == nullptr) return MLA_ERR_PARAM_NULLPTR;
    if (workspaceSize < sizeof(uint32_t)) return MLA_ERR_PARAM_INVALID;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return MLA_ERR_RUNTIME;
    if (cudaMemcpy(bits, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost) != cudaSuccess) return MLA_ERR_RUNTIME;
    return MLA_OK;
}

extern "C" mla_status mla_prolog_debug_wait_probe(void* workspace, uint64_t workspaceSize, int which, void* stream) {
    if (workspace == nullptr) return MLA_ERR_PARAM_NULLPTR;
    if (workspaceSize < kStatusBytes || (reinterpret_cast<uintptr_t>(workspace) & 15u) != 0 || (which != 0 && which != 1))
        return MLA_ERR_PARAM_INVALID;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    // the status word cleared, and the flag (bytes 8..15) zero: it never holds the probe's tag
    if (cudaMemsetAsync(ws, 0, 16, st) != cudaSuccess) return MLA_ERR_RUNTIME;
    wait_probe_kernel<<<1, 128, 0, st>>>(reinterpret_cast<const unsigned long long*>(ws + 8),
                                         reinterpret_cast<uint32_t*>(ws), which);
    return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_RUNTIME;
}

extern "C" mla_status mla_prolog_timing_enable(int enable) {
    std::lock_guard<std::mutex> lk(g_timing_mu);
    g_timing.enabled = enable != 0;
    g_timing.have = false;
    return MLA_OK;
}

extern "C" mla_status mla_prolog_timing_read(mla_kernel_time* out, int capacity, int* count) {
    if (out == nullptr || count == nullptr) return MLA_ERR_PARAM_NULLPTR;
    std::lock_guard<std::mutex> lk(g_timing_mu);
    if (!g_timing.have || g_timing.n == 0) return MLA_ERR_PARAM_INVALID;
    if (cudaEventSynchronize(g_timing.ev[g_timing.n]) != cudaSuccess) return MLA_ERR_RUNTIME;
    *count = g_timing.n;
    for (int i = 0; i < g_timing.n && i < capacity; ++i) {
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, g_timing.ev[i], g_timing.ev[i + 1]) != cudaSuccess) return MLA_ERR_RUNTIME;
        std::memset(out[i].name, 0, sizeof out[i].name);
        std::strncpy(out[i].name, g_timing.name[i], sizeof out[i].name - 1);
        out[i].ms = ms;
    }
    return MLA_OK;
}

extern "C" const char* mla_prolog_status_string(mla_status status) {
    switch (status) {
        case MLA_OK: return "MLA_OK";
        case MLA_ERR_PARAM_NULLPTR: return "MLA_ERR_PARAM_NULLPTR (161001): a required pointer is NULL";
        case MLA_ERR_PARAM_INVALID: return "MLA_ERR_PARAM_INVALID (161002): shape, dtype or scenario not accepted";
        case MLA_ERR_RUNTIME: return "MLA_ERR_RUNTIME (361001): a CUDA runtime call failed";
        case MLA_ERR_TILING: return "MLA_ERR_TILING (561002): shapes outside the kernels' tiling rules";
        case MLA_ERR_SCRATCH_LIMIT:
            return "MLA_ERR_SCRATCH_LIMIT (561003): the call needs more workspace than the fixed "
                   "no-allocation scratch buffer (MLA_NO_ALLOC_SCRATCH_BYTES) holds";
    }
    return "unknown mla_status";
}

// ====================================================================== aclnnMlaPreprocess variant

#include "preprocess_api.cuh"
