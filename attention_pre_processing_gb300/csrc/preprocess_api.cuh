// C ABI of the "aclnnMlaPreprocess" variant: validation, plan, workspace layout, launches.
// Declarations and argument documentation: mla_preprocess.h.  Part of the translation unit of
// mla_prolog_api.cu (it uses that file's launch helpers and tensor-map encoders).
//
// Pipeline of one call (the caller's stream, programmatic dependent launch between kernels):
//   Q0  RmsNormQuant(x) -> int8 codes as fp16 (T, He)
//   G1  codes . wdqkv^T -> fp32 k-range partials (T, Hcq + 576)      (gemm_w8: int8 weights
//       widened in shared memory, split-K)
//   M1  + bias0, * deScale0; RmsNormQuant(c^Q part) -> fp16 codes (T, Hcq); RmsNorm(kv) and
//       RoPE(kr) -> cache row at slotMapping[t]
//   G2  codes . wuq^T -> fp32 (T, n2)                                 (gemm_w8)
//   U2  + bias1, * deScale1 -> q^C (T, N, D) 16-bit; RoPE(q^R) -> q output
//   G3  q^C[:, n, :] . W^UK[n] -> q^N into qOut (row stride 576 or 512 per head)

#include "mla_preprocess.h"

namespace {

struct PpArgs {
    const mla_tensor *x, *g0, *b0, *qs0, *qo0, *w1, *de0, *bias0, *g1, *b1, *qs1, *qo1, *w2, *de1, *bias1, *g2,
        *cos, *sin, *wuk, *kv, *kr, *slots, *ctkv, *qns;
    int64_t wdq_dim, q_rope_dim, k_rope_dim;
    double eps;
    int64_t q_rot, k_rot;
    int32_t tr_wdq, tr_wuq, tr_wuk;
    int64_t cache_mode, quant_mode;
    int32_t do_norm;
    int64_t split;
    const mla_tensor *qout, *kv_out, *qrope, *kr_out;
};

struct PpDims {
    int64_t T, He, Hcq, N, D, Dr, Hckv, nslots;
    bool f16;
    int mode;
};

struct PpPlan {
    GemmPlan g1, g2, g3;
    int64_t n1 = 0, n2 = 0;
    bool kps3 = false;
    size_t off_a0 = 0, off_y1 = 0, off_a1 = 0, off_y2 = 0, off_qc = 0, bytes = 0;
};

bool pp_absent(const mla_tensor* t) { return t == nullptr || numel(t) == 0; }

mla_status pp_validate(const PpArgs& a, PpDims& d) {
    const mla_tensor* req[] = {a.x,  a.g0,  a.b0, a.qs0, a.qo0, a.w1,  a.de0,   a.g1,   a.b1,    a.qs1,
                               a.qo1, a.w2, a.de1, a.g2,  a.cos, a.sin, a.wuk, a.kv, a.slots, a.qout, a.kv_out};
    for (const mla_tensor* t : req)
        if (t == nullptr) return MLA_ERR_PARAM_NULLPTR;
    const mla_tensor* all[] = {a.x,   a.g0,  a.b0,  a.qs0, a.qo0, a.w1,    a.de0,  a.bias0, a.g1,   a.b1,
                               a.qs1, a.qo1, a.w2,  a.de1, a.bias1, a.g2,  a.cos,  a.sin,   a.wuk,  a.kv,
                               a.kr,  a.slots, a.qout, a.kv_out, a.qrope, a.kr_out};
    for (const mla_tensor* t : all) {
        if (t == nullptr) continue;
        if (t->ndim < 1 || t->ndim > 4) return MLA_ERR_PARAM_INVALID;
        for (int i = 0; i < t->ndim; ++i)
            if (t->shape[i] < 0) return MLA_ERR_PARAM_INVALID;
        if (!aligned16(t)) return MLA_ERR_PARAM_INVALID;
        if (t->data == nullptr && numel(t) > 0) return MLA_ERR_PARAM_NULLPTR;
    }
    // scalars: the only values the page accepts (cacheMode 2 / 3 are not built)
    if (a.cache_mode != 0 && a.cache_mode != 1) return MLA_ERR_PARAM_INVALID;
    if (a.quant_mode != 0 || a.split != 1 || a.q_rope_dim != 64 || a.k_rope_dim != 64 || a.q_rot != 2 ||
        a.k_rot != 2 || !a.tr_wdq || !a.tr_wuq || !a.tr_wuk)
        return MLA_ERR_PARAM_INVALID;
    if (!(a.eps >= 0.0) || !std::isfinite(a.eps)) return MLA_ERR_PARAM_INVALID;
    if (a.ctkv != nullptr || a.qns != nullptr) return MLA_ERR_PARAM_INVALID;   // cacheMode 2 only

    const int F = a.x->dtype;
    if (F != MLA_DT_BF16 && F != MLA_DT_FP16) return MLA_ERR_PARAM_INVALID;
    d.f16 = F == MLA_DT_FP16;
    d.mode = (int)a.cache_mode;
    d.Dr = 64;
    d.Hckv = 512;
    if (a.x->ndim != 2) return MLA_ERR_PARAM_INVALID;
    d.T = a.x->shape[0];
    d.He = a.x->shape[1];
    if (d.T > 256) return MLA_ERR_PARAM_INVALID;   // tokenNum in [0, 256]
    auto is = [](const mla_tensor* t, int dt, std::initializer_list<int64_t> s) {
        return t->dtype == dt && shape_is(t, s);
    };
    if (!is(a.g0, F, {d.He}) || !is(a.b0, F, {d.He}) || !is(a.qs0, F, {1}) || !is(a.qo0, MLA_DT_INT8, {1}))
        return MLA_ERR_PARAM_INVALID;
    if (a.w1->dtype != MLA_DT_INT8 || a.w1->ndim != 2 || a.w1->shape[1] != d.He) return MLA_ERR_PARAM_INVALID;
    const int64_t n1 = a.w1->shape[0];
    d.Hcq = n1 - d.Hckv - d.Dr;
    if (d.Hcq < 1 || d.Hcq > 4096 || a.wdq_dim != d.Hcq) return MLA_ERR_PARAM_INVALID;   // qLoraDim <= 4096
    if (!is(a.de0, MLA_DT_FP32, {n1})) return MLA_ERR_PARAM_INVALID;
    if (!pp_absent(a.bias0) && !is(a.bias0, MLA_DT_INT32, {n1})) return MLA_ERR_PARAM_INVALID;
    if (!is(a.g1, F, {d.Hcq}) || !is(a.b1, F, {d.Hcq}) || !is(a.qs1, F, {1}) || !is(a.qo1, MLA_DT_INT8, {1}))
        return MLA_ERR_PARAM_INVALID;
    if (a.wuk->dtype != F || a.wuk->ndim != 3 || a.wuk->shape[2] != d.Hckv) return MLA_ERR_PARAM_INVALID;
    d.N = a.wuk->shape[0];
    d.D = a.wuk->shape[1];
    if (d.N < 1 || d.N > 128 || d.D < 1) return MLA_ERR_PARAM_INVALID;   // headNum in [1, 128]
    const int64_t n2 = d.N * (d.D + d.Dr);
    if (!is(a.w2, MLA_DT_INT8, {n2, d.Hcq}) || !is(a.de1, MLA_DT_FP32, {n2})) return MLA_ERR_PARAM_INVALID;
    if (!pp_absent(a.bias1) && !is(a.bias1, MLA_DT_INT32, {n2})) return MLA_ERR_PARAM_INVALID;
    if (!is(a.g2, F, {d.Hckv}) || !is(a.cos, F, {d.T, d.Dr}) || !is(a.sin, F, {d.T, d.Dr}) ||
        !is(a.slots, MLA_DT_INT32, {d.T}))
        return MLA_ERR_PARAM_INVALID;
    // caches and outputs by cacheMode
    const int64_t kv_w = d.mode == 0 ? d.Hckv + d.Dr : d.Hckv;
    if (a.kv->dtype != F || a.kv->ndim != 4 || a.kv->shape[2] != 1 || a.kv->shape[3] != kv_w)
        return MLA_ERR_PARAM_INVALID;
    const int64_t bn = a.kv->shape[0], bs = a.kv->shape[1];
    d.nslots = bn * bs;
    if (a.kv_out->data != a.kv->data || !is(a.kv_out, F, {bn, bs, 1, kv_w})) return MLA_ERR_PARAM_INVALID;
    if (d.mode == 0) {
        if (a.kr != nullptr || a.kr_out != nullptr || a.qrope != nullptr) return MLA_ERR_PARAM_INVALID;
        if (!is(a.qout, F, {d.T, d.N, d.Hckv + d.Dr})) return MLA_ERR_PARAM_INVALID;
    } else {
        if (a.kr == nullptr || a.kr_out == nullptr || a.qrope == nullptr) return MLA_ERR_PARAM_NULLPTR;
        if (!is(a.kr, F, {bn, bs, 1, d.Dr}) || a.kr_out->data != a.kr->data || !is(a.kr_out, F, {bn, bs, 1, d.Dr}))
            return MLA_ERR_PARAM_INVALID;
        if (!is(a.qout, F, {d.T, d.N, d.Hckv}) || !is(a.qrope, F, {d.T, d.N, d.Dr})) return MLA_ERR_PARAM_INVALID;
    }
    // the kernels' tiling
    if (d.He % 64 != 0 || d.Hcq % 64 != 0 || d.D % 16 != 0 || d.D < 16 || d.D > 256) return MLA_ERR_TILING;
    return MLA_OK;
}

PpPlan pp_plan(const PpDims& d, int sms) {
    PpPlan p;
    const int64_t T = d.T;
    p.n1 = d.Hcq + d.Hckv + d.Dr;
    p.n2 = d.N * (d.D + d.Dr);
    // the down-projection: 128-column tiles x k ranges up to 128 tokens (17 x 8 at 2112 columns:
    // 14 k-blocks per CTA; with 64-column tiles each CTA walked 28, and the pipeline's per-k-block
    // latency, not the bytes, set the time: 21.5 -> 17.4 us per launch at T = 32), 192-column
    // tiles above
    plan_gemm(p.g1, T, p.n1, d.He, sms, T <= 128 ? 128 : 192, true);
    // the up-projection: 192-column tiles, whole K
    plan_gemm(p.g2, T, p.n2, d.Hcq, sms, 192, false);
    // W^UK: up to 128 tokens one 512-column tile per head (N tiles: one wave on the SMs for
    // N <= 152), above that two 256-column tiles per head and row tile
    p.g3.m_tiles = (int)((T + 127) / 128);
    p.g3.bn = p.g3.m_tiles == 1 ? 512 : 256;
    p.g3.kblocks = (int)((d.D + kBK - 1) / kBK);
    p.g3.n_tiles = (int)(d.N * (512 / p.g3.bn));
    p.g3.msub = 1;
    p.g3.a_box_rows = T < 128 ? (int)((T + 7) / 8 * 8) : 128;
    const long long tiles = (long long)p.g3.m_tiles * p.g3.n_tiles;
    p.g3.grid = (int)(tiles < sms ? tiles : sms);
    p.kps3 = p.g3.m_tiles > 1 && p.g3.kblocks % 2 == 0;

    size_t off = kStatusBytes;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = up1024(off + bytes);
        return o;
    };
    p.off_a0 = take((size_t)T * d.He * 2);
    p.off_y1 = take((size_t)p.g1.ksplit * T * p.n1 * 4);
    p.off_a1 = take((size_t)T * d.Hcq * 2);
    p.off_y2 = take((size_t)T * p.n2 * 4);
    p.off_qc = take((size_t)T * d.N * d.D * 2);
    p.bytes = off;
    return p;
}

mla_status pp_run(const PpArgs& a, const PpDims& d, const PpPlan& p, uint8_t* ws, cudaStream_t st) {
    if (!get_encoder()) return MLA_ERR_RUNTIME;
    uint32_t* status = reinterpret_cast<uint32_t*>(ws);
    const int T = (int)d.T;
    auto* a0 = reinterpret_cast<__nv_bfloat16*>(ws + p.off_a0);
    auto* y1 = reinterpret_cast<float*>(ws + p.off_y1);
    auto* a1 = reinterpret_cast<__nv_bfloat16*>(ws + p.off_a1);
    auto* y2 = reinterpret_cast<float*>(ws + p.off_y2);
    uint8_t* qc = ws + p.off_qc;
    cudaError_t e;

    // ---- Q0: the input's int8 codes
    PpQuantArgs q = {};
    q.x = a.x->data;
    q.gamma = a.g0->data;
    q.beta = a.b0->data;
    q.qscale = a.qs0->data;
    q.qoffset = static_cast<const int8_t*>(a.qo0->data);
    q.out = a0;
    q.He = (int)d.He;
    q.eps_h = (float)a.eps;
    q.eps_l = (float)(a.eps - (double)q.eps_h);
    q.do_norm = a.do_norm ? 1 : 0;
    e = launch(d.f16 ? pp_quant_x_kernel<true> : pp_quant_x_kernel<false>, T, kPpRowThreads, 0, st, q);
    if (e != cudaSuccess) return MLA_ERR_RUNTIME;
    timing_mark(st, "pp_quant_x");

    // ---- G1: down-projection
    CUtensorMap mA1, mB1;
    if (!map_2d(&mA1, a0, d.T, d.He, (uint32_t)p.g1.a_box_rows) ||
        !map_w8_rows(&mB1, a.w1->data, p.n1, d.He, (uint32_t)p.g1.bn))
        return MLA_ERR_RUNTIME;
    GemmArgs g1 = gemm_args(p.g1, T, p.n1, status);
    g1.clear_status = 1;
    g1.out_f32 = y1;
    e = p.g1.bn == 128 ? launch_gemm_w8<128, 1, 16>(p.g1.grid, st, mA1, mB1, g1)
                      : launch_gemm_w8<192, 2, 16>(p.g1.grid, st, mA1, mB1, g1);
    if (e != cudaSuccess) return MLA_ERR_RUNTIME;
    timing_mark(st, "pp_down_proj");

    // ---- M1: dequant, RmsNormQuant of c^Q, the cache row
    PpMidArgs m = {};
    m.y = y1;
    m.ksplit = p.g1.ksplit;
    m.slot_stride = (size_t)d.T * p.n1;
    m.n1 = (int)p.n1;
    m.Hcq = (int)d.Hcq;
    m.Hckv = (int)d.Hckv;
    m.Dr = (int)d.Dr;
    m.bias0 = pp_absent(a.bias0) ? nullptr : static_cast<const int*>(a.bias0->data);
    m.de0 = static_cast<const float*>(a.de0->data);
    m.gamma1 = a.g1->data;
    m.beta1 = a.b1->data;
    m.qscale1 = a.qs1->data;
    m.qoffset1 = static_cast<const int8_t*>(a.qo1->data);
    m.codes1 = a1;
    m.gamma2 = a.g2->data;
    m.cos = a.cos->data;
    m.sin = a.sin->data;
    m.slots = static_cast<const int*>(a.slots->data);
    m.nslots = d.nslots;
    m.kv = a.kv->data;
    m.kv_ld = (int)(d.mode == 0 ? d.Hckv + d.Dr : d.Hckv);
    m.kr = d.mode == 0 ? nullptr : a.kr->data;
    m.eps_h = (float)a.eps;
    m.eps_l = (float)(a.eps - (double)m.eps_h);
    m.status = status;
    e = launch(d.f16 ? pp_mid_kernel<true> : pp_mid_kernel<false>, T, kPpRowThreads, (size_t)p.n1 * 8, st, m);
    if (e != cudaSuccess) return MLA_ERR_RUNTIME;
    timing_mark(st, "pp_norm_quant_cache");

    // ---- G2: up-projection
    CUtensorMap mA2, mB2;
    if (!map_2d(&mA2, a1, d.T, d.Hcq, (uint32_t)p.g2.a_box_rows) ||
        !map_w8_rows(&mB2, a.w2->data, p.n2, d.Hcq, (uint32_t)p.g2.bn))
        return MLA_ERR_RUNTIME;
    GemmArgs g2 = gemm_args(p.g2, T, p.n2, status);
    g2.out_f32 = y2;
    e = p.g2.msub == 1 ? launch_gemm_w8<192, 1, 16>(p.g2.grid, st, mA2, mB2, g2)
                       : launch_gemm_w8<192, 2, 16>(p.g2.grid, st, mA2, mB2, g2);
    if (e != cudaSuccess) return MLA_ERR_RUNTIME;
    timing_mark(st, "pp_up_proj");

    // ---- U2: q^C and RoPE(q^R)
    PpUpArgs u = {};
    u.z = y2;
    u.N = (int)d.N;
    u.D = (int)d.D;
    u.Dr = (int)d.Dr;
    u.bias1 = pp_absent(a.bias1) ? nullptr : static_cast<const int*>(a.bias1->data);
    u.de1 = static_cast<const float*>(a.de1->data);
    u.cos = a.cos->data;
    u.sin = a.sin->data;
    u.qc = qc;
    if (d.mode == 0) {
        u.qr = static_cast<uint16_t*>(a.qout->data) + d.Hckv;   // after q^N in each 576-wide row
        u.qr_ld = (int)(d.Hckv + d.Dr);
    } else {
        u.qr = a.qrope->data;
        u.qr_ld = (int)d.Dr;
    }
    const int up_grid = T * (int)((d.N + kPpUpHeads - 1) / kPpUpHeads);
    e = launch(d.f16 ? pp_up_kernel<true> : pp_up_kernel<false>, up_grid, kPpThreads, 0, st, u);
    if (e != cudaSuccess) return MLA_ERR_RUNTIME;
    timing_mark(st, "pp_dequant_rope_q");

    // ---- G3: per-head W^UK contraction into qOut
    const CUtensorMapDataType tdt = d.f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    CUtensorMap mA3, mB3, mO3;
    {
        const uint64_t dims[3] = {(uint64_t)d.D, (uint64_t)d.N, (uint64_t)d.T};
        const uint64_t strides[2] = {(uint64_t)d.D * 2, (uint64_t)d.N * d.D * 2};
        const uint32_t box[3] = {64, 1, (uint32_t)p.g3.a_box_rows};
        if (!encode_map(&mA3, qc, 3, dims, strides, box, tdt)) return MLA_ERR_RUNTIME;
        const uint64_t dimsb[3] = {(uint64_t)d.Hckv, (uint64_t)d.D, (uint64_t)d.N};
        const uint64_t stridesb[2] = {(uint64_t)d.Hckv * 2, (uint64_t)d.D * d.Hckv * 2};
        const uint32_t boxb[3] = {64, p.kps3 ? 128u : 64u, 1};
        if (!encode_map(&mB3, a.wuk->data, 3, dimsb, stridesb, boxb, tdt)) return MLA_ERR_RUNTIME;
    }
    const int64_t q_ld = d.mode == 0 ? d.Hckv + d.Dr : d.Hckv;
    GemmArgs g3 = gemm_args(p.g3, T, d.Hckv, status);
    g3.head_mode = 1;
    g3.tiles_per_head = 512 / p.g3.bn;
    g3.N = (int)d.N;
    g3.Hckv = (int)d.Hckv;
    g3.q_ld = (int)q_ld;
    g3.f16 = d.f16 ? 1 : 0;
    g3.q_out_bf16 = static_cast<__nv_bfloat16*>(a.qout->data);
    {
        // qOut as a (T, N * q_ld) matrix: 32-row x 64-column boxes, whole boxes inside one head's q^N
        const uint64_t dims[2] = {(uint64_t)(d.N * q_ld), (uint64_t)d.T};
        const uint64_t strides[1] = {(uint64_t)(d.N * q_ld) * 2};
        const uint32_t box[2] = {64, 32};
        g3.tma_out = encode_map(&mO3, a.qout->data, 2, dims, strides, box, tdt) ? 1 : 0;
    }
    // one 512-column tile per head: four epilogue warps per TMEM lane quarter, 128 columns each
    // (at T = 32 every row sits in the first lane quarter, which one warp alone drained in ~1.5 us more)
    e = p.g3.bn == 512 ? launch_gemm<512, 1, 4, EPI_QN, 1, 1, 4>(p.g3.grid, st, mA3, mB3, mB3, g3, g3.tma_out ? &mO3 : nullptr)
        : p.kps3 ? launch_gemm<256, 1, 8, EPI_QN, 2, 2>(p.g3.grid, st, mA3, mB3, mB3, g3, g3.tma_out ? &mO3 : nullptr)
               : launch_gemm<256, 1, 8, EPI_QN, 2>(p.g3.grid, st, mA3, mB3, mB3, g3, g3.tma_out ? &mO3 : nullptr);
    if (e != cudaSuccess) return MLA_ERR_RUNTIME;
    timing_mark(st, "pp_absorb_uk");
    if (g_timing.enabled) g_timing.have = true;
    return MLA_OK;
}

}  // namespace

#define MLA_PP_PARAMS                                                                                         \
    const mla_tensor *input, const mla_tensor *gamma0, const mla_tensor *beta0, const mla_tensor *quantScale0, \
        const mla_tensor *quantOffset0, const mla_tensor *wdqkv, const mla_tensor *deScale0,                  \
        const mla_tensor *bias0, const mla_tensor *gamma1, const mla_tensor *beta1,                           \
        const mla_tensor *quantScale1, const mla_tensor *quantOffset1, const mla_tensor *wuq,                 \
        const mla_tensor *deScale1, const mla_tensor *bias1, const mla_tensor *gamma2, const mla_tensor *cos,  \
        const mla_tensor *sin, const mla_tensor *wuk, const mla_tensor *kvCache, const mla_tensor *kvCacheRope, \
        const mla_tensor *slotMapping, const mla_tensor *ctkvScale, const mla_tensor *qNopeScale,              \
        int64_t wdqDim, int64_t qRopeDim, int64_t kRopeDim, double epsilon, int64_t qRotaryCoeff,              \
        int64_t kRotaryCoeff, int32_t transposeWdq, int32_t transposeWuq, int32_t transposeWuk,                \
        int64_t cacheMode, int64_t quantMode, int32_t doRmsNorm, int64_t wdkvSplitCount,                       \
        const mla_tensor *qOut, const mla_tensor *kvCacheOut, const mla_tensor *qRopeOut,                     \
        const mla_tensor *krCacheOut

#define MLA_PP_ARGS                                                                                            \
    input, gamma0, beta0, quantScale0, quantOffset0, wdqkv, deScale0, bias0, gamma1, beta1, quantScale1,       \
        quantOffset1, wuq, deScale1, bias1, gamma2, cos, sin, wuk, kvCache, kvCacheRope, slotMapping, ctkvScale, \
        qNopeScale, wdqDim, qRopeDim, kRopeDim, epsilon, qRotaryCoeff, kRotaryCoeff, transposeWdq, transposeWuq, \
        transposeWuk, cacheMode, quantMode, doRmsNorm, wdkvSplitCount, qOut, kvCacheOut, qRopeOut, krCacheOut

static PpArgs pp_pack(MLA_PP_PARAMS) {
    PpArgs a;
    a.x = input;
    a.g0 = gamma0;
    a.b0 = beta0;
    a.qs0 = quantScale0;
    a.qo0 = quantOffset0;
    a.w1 = wdqkv;
    a.de0 = deScale0;
    a.bias0 = bias0;
    a.g1 = gamma1;
    a.b1 = beta1;
    a.qs1 = quantScale1;
    a.qo1 = quantOffset1;
    a.w2 = wuq;
    a.de1 = deScale1;
    a.bias1 = bias1;
    a.g2 = gamma2;
    a.cos = cos;
    a.sin = sin;
    a.wuk = wuk;
    a.kv = kvCache;
    a.kr = kvCacheRope;
    a.slots = slotMapping;
    a.ctkv = ctkvScale;
    a.qns = qNopeScale;
    a.wdq_dim = wdqDim;
    a.q_rope_dim = qRopeDim;
    a.k_rope_dim = kRopeDim;
    a.eps = epsilon;
    a.q_rot = qRotaryCoeff;
    a.k_rot = kRotaryCoeff;
    a.tr_wdq = transposeWdq;
    a.tr_wuq = transposeWuq;
    a.tr_wuk = transposeWuk;
    a.cache_mode = cacheMode;
    a.quant_mode = quantMode;
    a.do_norm = doRmsNorm;
    a.split = wdkvSplitCount;
    a.qout = qOut;
    a.kv_out = kvCacheOut;
    a.qrope = qRopeOut;
    a.kr_out = krCacheOut;
    return a;
}

extern "C" mla_status mla_preprocess_workspace_size(MLA_PP_PARAMS, uint64_t* workspaceSize) {
    if (workspaceSize == nullptr) return MLA_ERR_PARAM_NULLPTR;
    const PpArgs a = pp_pack(MLA_PP_ARGS);
    PpDims d;
    const mla_status s = pp_validate(a, d);
    if (s != MLA_OK) return s;
    if (d.T == 0) {
        *workspaceSize = kStatusBytes;
        return MLA_OK;
    }
    int sms = 0;
    if (device_sms(&sms) != 0) return MLA_ERR_RUNTIME;
    *workspaceSize = pp_plan(d, sms).bytes;
    return MLA_OK;
}

extern "C" mla_status mla_preprocess(MLA_PP_PARAMS, void* workspace, uint64_t workspaceSize, void* stream) {
    const PpArgs a = pp_pack(MLA_PP_ARGS);
    PpDims d;
    const mla_status s = pp_validate(a, d);
    if (s != MLA_OK) return s;
    if (d.T == 0) return MLA_OK;
    if (workspace == nullptr) return MLA_ERR_PARAM_NULLPTR;
    if ((reinterpret_cast<uintptr_t>(workspace) & 15u) != 0) return MLA_ERR_PARAM_INVALID;
    int sms = 0;
    if (device_sms(&sms) != 0) return MLA_ERR_RUNTIME;
    const PpPlan p = pp_plan(d, sms);
    if (workspaceSize < p.bytes) return MLA_ERR_PARAM_INVALID;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    timing_begin(st);
    return pp_run(a, d, p, static_cast<uint8_t*>(workspace), st);
}
