// Row kernels of the "aclnnMlaPreprocess" variant (the two int8 contractions run on gemm_w8,
// the W^UK contraction on gemm_tc):
//   pp_quant_x_kernel   RmsNormQuant of the input (or the quantiser alone) -> int8 codes held
//                       as fp16, the A operand of the down-projection
//   pp_mid_kernel       per token after the down-projection: add the k-range slots, + bias0,
//                       * deScale0; RmsNormQuant of the c^Q part -> codes (A of the
//                       up-projection); RmsNorm of the kv part and RoPE of the rope part ->
//                       the cache row at slotMapping[t]
//   pp_up_kernel        per token after the up-projection: + bias1, * deScale1; q^C (16-bit,
//                       A of the W^UK contraction) and RoPE(q^R) into the q output
// Every kernel waits for the previous grid before touching memory (programmatic dependent
// launch) and lets the next one start its prologue at once.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "finalize.cuh"
#include "gemm_tc.cuh"
#include "ptx.cuh"

namespace mla {

constexpr int kPpThreads = 256;
// The per-token row kernels (one CTA per token) run 1024 threads: at decode sizes they are
// latency-bound, and more warps per token hide more of it.
constexpr int kPpRowThreads = 1024;

// 16-bit element <-> float for the input dtype (bf16 or fp16).
template <bool F16>
struct Half16;
template <>
struct Half16<false> {
    using T = __nv_bfloat16;
    static __device__ __forceinline__ float load(const void* p, size_t i) {
        return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
    }
    static __device__ __forceinline__ void store(void* p, size_t i, float v) {
        static_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
    }
    static __device__ __forceinline__ float lo(uint32_t w) { return bf16_lo(w); }
    static __device__ __forceinline__ float hi(uint32_t w) { return bf16_hi(w); }
};
template <>
struct Half16<true> {
    using T = __half;
    static __device__ __forceinline__ float load(const void* p, size_t i) {
        return __half2float(static_cast<const __half*>(p)[i]);
    }
    static __device__ __forceinline__ void store(void* p, size_t i, float v) {
        static_cast<__half*>(p)[i] = __float2half_rn(v);
    }
    static __device__ __forceinline__ float lo(uint32_t w) {
        return __half2float(__ushort_as_half((unsigned short)(w & 0xFFFFu)));
    }
    static __device__ __forceinline__ float hi(uint32_t w) {
        return __half2float(__ushort_as_half((unsigned short)(w >> 16)));
    }
};

// Error-free float transformations: s + e == a + b and p + e == a * b exactly.  two_sum is
// Knuth's branch-free TwoSum (The Art of Computer Programming, vol. 2, section 4.2.2); two_prod
// forms the product's rounding error with one fused multiply-add (the FMA form of Dekker's
// exact product).
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}
__device__ __forceinline__ void two_prod(float a, float b, float& p, float& e) {
    p = __fmul_rn(a, b);
    e = fmaf(a, b, -p);
}
// Float pairs (hi + lo, |lo| <= ulp(hi) / 2) carry ~48 significant bits: the double-length
// arithmetic of Dekker ("A floating-point technique for extending the available precision",
// Numerische Mathematik 18, 1971), with quotient and square root corrected by one residual step.
__device__ __forceinline__ void ff_norm(float& hi, float& lo) {
    const float s = __fadd_rn(hi, lo);
    lo = __fsub_rn(lo, __fsub_rn(s, hi));
    hi = s;
}
// (hi, lo) += (vh, vl)
__device__ __forceinline__ void ff_add(float& hi, float& lo, float vh, float vl) {
    float s, e;
    two_sum(hi, vh, s, e);
    e = __fadd_rn(e, __fadd_rn(lo, vl));
    hi = s;
    lo = e;
    ff_norm(hi, lo);
}
// (ah, al) * f
__device__ __forceinline__ void ff_mul_f(float ah, float al, float f, float& h, float& l) {
    two_prod(ah, f, h, l);
    l = fmaf(al, f, l);
    ff_norm(h, l);
}
// (ah, al) / (bh, bl); the residual a - q * b is formed exactly from the product's error term
__device__ __forceinline__ void ff_div(float ah, float al, float bh, float bl, float& h, float& l) {
    h = __fdiv_rn(ah, bh);
    float p, e;
    two_prod(h, bh, p, e);
    const float rem = __fsub_rn(__fadd_rn(__fsub_rn(__fsub_rn(ah, p), e), al), __fmul_rn(h, bl));
    l = __fdiv_rn(rem, bh);
    ff_norm(h, l);
}
// sqrt(ah + al)
__device__ __forceinline__ void ff_sqrt(float ah, float al, float& h, float& l) {
    h = __fsqrt_rn(ah);
    float p, e;
    two_prod(h, h, p, e);
    l = __fdiv_rn(__fadd_rn(__fsub_rn(__fsub_rn(ah, p), e), al), __fmul_rn(2.f, h));
    ff_norm(h, l);
}

// The int8 code of the page's static asymmetric quantiser,
//   code = clamp(round_half_away(v * qs) + qo, -128, 127),  v = (gamma * y) / r + beta  (norm)
//                                                            v = y                     (no norm)
// with r = sqrt(mean(y^2) + eps), evaluated in the definition's operation order.  The fp32
// estimate decides unless it lies within its error bound of a rounding boundary (a
// half-integer); the bound is a few fp32 roundings (2^-24 relative each) of terms no larger than
// (|gamma * y / r| + |beta|) * |qs|, and 1e-5 of that is a wide margin.  Near a boundary the same
// expression is evaluated in float pairs (~48 bits), which decide like exact arithmetic unless the
// value lies within ~1e-13 of the half-integer (GB300 runs doubles at a small fraction of its
// float rate, and a double path there cost microseconds per kernel).  y arrives as a float pair
// (yl = 0 when y is a float); PpNorm holds r as a float pair and its fp32 reciprocal.
struct PpNorm {
    float rh, rl;   // r = sqrt(sum / nfeat + eps) as a float pair
    float inv;      // fp32 estimate of 1 / r
};
// r from the sum of squares (sh, sl) over nfeat features and eps = eh + el.
__device__ __forceinline__ PpNorm pp_norm(float sh, float sl, int nfeat, float eh, float el) {
    float mh, ml;
    ff_div(sh, sl, (float)nfeat, 0.f, mh, ml);   // nfeat <= 2^24: exact as a float
    ff_add(mh, ml, eh, el);
    PpNorm n;
    ff_sqrt(mh, ml, n.rh, n.rl);
    n.inv = __fdiv_rn(1.f, n.rh);
    return n;
}
__device__ __forceinline__ float pp_code(float yh, float yl, float g, float b, bool norm, const PpNorm& nr, float qs,
                                         int qo) {
    const float a = norm ? g * yh * nr.inv : yh;
    const float sf = (a + (norm ? b : 0.f)) * qs;
    const float margin = 1e-5f * (fabsf(a) + (norm ? fabsf(b) : 0.f)) * fabsf(qs) + 1e-30f;
    float q;
    if (fabsf(sf - floorf(sf) - 0.5f) <= margin) {
        float vh = yh, vl = yl;
        if (norm) {
            float ph, pl;
            ff_mul_f(yh, yl, g, ph, pl);
            ff_div(ph, pl, nr.rh, nr.rl, vh, vl);
            ff_add(vh, vl, b, 0.f);
        }
        float sh, sl;
        ff_mul_f(vh, vl, qs, sh, sl);
        // round half away from zero: compare |s| with the half-integer next to it
        const float sg = sh < 0.f ? -1.f : 1.f;
        sh *= sg;
        sl *= sg;
        const float m = floorf(sh);
        const float d = __fadd_rn(__fsub_rn(sh, m + 0.5f), sl);
        q = sg * (m + (d >= 0.f ? 1.f : 0.f));
    } else {
        q = roundf(sf);
    }
    return fminf(fmaxf(q + (float)qo, -128.f), 127.f);
}

// Deterministic sum of float pairs over the CTA of NT threads (fixed shuffle tree, then the
// warps in order); red holds NT / 32 + 1 pairs.
template <int NT>
__device__ __forceinline__ float2 pp_block_sum(float hi, float lo, float2* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float oh = __shfl_xor_sync(0xffffffffu, hi, o), ol = __shfl_xor_sync(0xffffffffu, lo, o);
        ff_add(hi, lo, oh, ol);
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) red[warp] = make_float2(hi, lo);
    __syncthreads();
    if (warp == 0) {
        float2 r = lane < NT / 32 ? red[lane] : make_float2(0.f, 0.f);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float oh = __shfl_xor_sync(0xffffffffu, r.x, o), ol = __shfl_xor_sync(0xffffffffu, r.y, o);
            ff_add(r.x, r.y, oh, ol);
        }
        if (lane == 0) red[NT / 32] = r;
    }
    __syncthreads();
    return red[NT / 32];
}

// Four 16-bit values from four floats, as one 8-byte word.
template <bool F16>
__device__ __forceinline__ uint2 pp_pack4(float a, float b, float c, float d) {
    if constexpr (F16)
        return make_uint2(pack_f16(a, b), pack_f16(c, d));
    else
        return make_uint2(pack_bf16(a, b), pack_bf16(c, d));
}

// ---------------------------------------------------------------- input quantisation

struct PpQuantArgs {
    const void* x;          // (T, He) F
    const void* gamma;      // (He) F
    const void* beta;       // (He) F
    const void* qscale;     // (1) F
    const int8_t* qoffset;  // (1)
    __nv_bfloat16* out;     // (T, He): codes as fp16 (exact), the A operand of gemm_w8
    int He;
    float eps_h, eps_l;     // epsilon as a float pair
    int do_norm;
};

// One CTA per token.  He % 8 == 0.
template <bool F16>
__global__ void __launch_bounds__(kPpRowThreads) pp_quant_x_kernel(const PpQuantArgs a) {
    using H = Half16<F16>;
    __shared__ float2 red[kPpRowThreads / 32 + 1];
    pdl_launch_dependents();
    pdl_wait();
    const int t = blockIdx.x, tid = threadIdx.x;
    const uint4* xr = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.x) + (size_t)t * a.He);
    const int n8 = a.He / 8;
    PpNorm nr = {1.f, 0.f, 1.f};
    if (a.do_norm) {
        // squares of 16-bit values are exact floats; each thread adds its squares as a float
        // pair, the CTA adds the pairs in double
        float sh = 0.f, sl = 0.f;
        for (int i = tid; i < n8; i += kPpRowThreads) {
            const uint4 v = xr[i];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float lo = H::lo(w[e]), hi = H::hi(w[e]);
                ff_add(sh, sl, lo * lo, 0.f);
                ff_add(sh, sl, hi * hi, 0.f);
            }
        }
        const float2 ss = pp_block_sum<kPpRowThreads>(sh, sl, red);
        nr = pp_norm(ss.x, ss.y, a.He, a.eps_h, a.eps_l);
    }
    const float qs = H::load(a.qscale, 0);
    const int qo = (int)a.qoffset[0];
    const uint4* gr = reinterpret_cast<const uint4*>(a.gamma);
    const uint4* br = reinterpret_cast<const uint4*>(a.beta);
    uint4* outr = reinterpret_cast<uint4*>(a.out + (size_t)t * a.He);
    for (int i = tid; i < n8; i += kPpRowThreads) {
        const uint4 v = xr[i];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t gw[4] = {0, 0, 0, 0}, bw[4] = {0, 0, 0, 0};
        if (a.do_norm) {
            const uint4 g = gr[i], b = br[i];
            gw[0] = g.x, gw[1] = g.y, gw[2] = g.z, gw[3] = g.w;
            bw[0] = b.x, bw[1] = b.y, bw[2] = b.z, bw[3] = b.w;
        }
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const bool nm = a.do_norm != 0;
            o[e] = pack_f16(pp_code(H::lo(w[e]), 0.f, H::lo(gw[e]), H::lo(bw[e]), nm, nr, qs, qo),
                            pp_code(H::hi(w[e]), 0.f, H::hi(gw[e]), H::hi(bw[e]), nm, nr, qs, qo));
        }
        outr[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// ---------------------------------------------------------------- after the down-projection

struct PpMidArgs {
    const float* y;            // ksplit slots of (T, n1) fp32 products
    int ksplit;
    size_t slot_stride;        // T * n1
    int n1;                    // Hcq + Hckv + Dr
    int Hcq, Hckv, Dr;
    const int* bias0;          // (n1) or null
    const float* de0;          // (n1)
    const void* gamma1;        // (Hcq) F
    const void* beta1;         // (Hcq) F
    const void* qscale1;       // (1) F
    const int8_t* qoffset1;    // (1)
    __nv_bfloat16* codes1;     // (T, Hcq): codes as fp16 (exact), the A operand of gemm_w8
    const void* gamma2;        // (Hckv) F
    const void* cos;           // (T, Dr) F
    const void* sin;           // (T, Dr) F
    const int* slots;          // (T)
    long long nslots;
    void* kv;                  // (nslots, kv_ld) F
    int kv_ld;                 // Hckv + Dr (cacheMode 0) or Hckv (1)
    void* kr;                  // cacheMode 1: (nslots, Dr) F; cacheMode 0: null (k^R after k^N in kv)
    float eps_h, eps_l;        // epsilon as a float pair
    uint32_t* status;
};

// k ranges of the down-projection's partials that pp_mid_kernel requests at once (a round of
// 32 registers of loads at 1024 threads).
constexpr int kPpSlotRound = 8;

// One CTA per token; dynamic shared memory holds the token's n1 values as exact float pairs
// (y = (acc + bias) * deScale has at most 48 significant bits: acc + bias is an integer below
// 2^24 and deScale a float, so its product splits exactly into a float and the float error).
template <bool F16>
__global__ void __launch_bounds__(kPpRowThreads) pp_mid_kernel(const PpMidArgs a) {
    using H = Half16<F16>;
    extern __shared__ float2 ys[];
    __shared__ float2 red[kPpRowThreads / 32 + 1];
    pdl_launch_dependents();
    pdl_wait();
    const int t = blockIdx.x, tid = threadIdx.x;
    const float* y0 = a.y + (size_t)t * a.n1;
    float s1h = 0.f, s1l = 0.f, s2h = 0.f, s2l = 0.f;
    // four columns per thread and step (n1 % 4 == 0), the k-range loads unrolled so that they
    // are in flight together
    for (int j4 = tid; j4 < a.n1 / 4; j4 += kPpRowThreads) {
        // the k-range partials are integer-valued (int8 products), so their fp32 sum in k-range
        // order is the exact integer while it stays below 2^24; bias and scale then in double
        // kPpSlotRound k ranges' partials in flight at once (all of them at the decode plan's 8),
        // summed in k-range order
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s0 = 0; s0 < a.ksplit; s0 += kPpSlotRound) {
            float4 pk[kPpSlotRound];
#pragma unroll
            for (int i = 0; i < kPpSlotRound; ++i)
                pk[i] = s0 + i < a.ksplit
                            ? __ldcg(reinterpret_cast<const float4*>(y0 + (size_t)(s0 + i) * a.slot_stride) + j4)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int i = 0; i < kPpSlotRound; ++i)
                if (s0 + i < a.ksplit) acc.x += pk[i].x, acc.y += pk[i].y, acc.z += pk[i].z, acc.w += pk[i].w;
        }
        int4 b = make_int4(0, 0, 0, 0);
        if (a.bias0 != nullptr) b = reinterpret_cast<const int4*>(a.bias0)[j4];
        const float4 sc = reinterpret_cast<const float4*>(a.de0)[j4];
        const float av[4] = {acc.x, acc.y, acc.z, acc.w}, sv[4] = {sc.x, sc.y, sc.z, sc.w};
        const int bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int j = 4 * j4 + e;
            float yh, yl;
            two_prod(__fadd_rn(av[e], (float)bv[e]), sv[e], yh, yl);
            ys[j] = make_float2(yh, yl);
            // y^2 = yh^2 + 2 yh yl (+ yl^2, below the pair's precision)
            float ph, pl;
            two_prod(yh, yh, ph, pl);
            pl = fmaf(2.f * yh, yl, pl);
            if (j < a.Hcq)
                ff_add(s1h, s1l, ph, pl);
            else if (j < a.Hcq + a.Hckv)
                ff_add(s2h, s2l, ph, pl);
        }
    }
    const float2 ss1 = pp_block_sum<kPpRowThreads>(s1h, s1l, red);
    const float2 ss2 = pp_block_sum<kPpRowThreads>(s2h, s2l, red);   // its barriers also publish ys
    const PpNorm nr1 = pp_norm(ss1.x, ss1.y, a.Hcq, a.eps_h, a.eps_l);
    const float inv2 = pp_norm(ss2.x, ss2.y, a.Hckv, a.eps_h, a.eps_l).inv;
    // path 1: RmsNormQuant -> the up-projection's codes
    const float qs = H::load(a.qscale1, 0);
    const int qo = (int)a.qoffset1[0];
    for (int j8 = tid; j8 < a.Hcq / 8; j8 += kPpRowThreads) {   // eight columns per thread and step
        const uint4 g = reinterpret_cast<const uint4*>(a.gamma1)[j8];
        const uint4 b = reinterpret_cast<const uint4*>(a.beta1)[j8];
        const uint32_t gw[4] = {g.x, g.y, g.z, g.w}, bw[4] = {b.x, b.y, b.z, b.w};
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int j = 8 * j8 + 2 * e;
            o[e] = pack_f16(pp_code(ys[j].x, ys[j].y, H::lo(gw[e]), H::lo(bw[e]), true, nr1, qs, qo),
                            pp_code(ys[j + 1].x, ys[j + 1].y, H::hi(gw[e]), H::hi(bw[e]), true, nr1, qs, qo));
        }
        reinterpret_cast<uint4*>(a.codes1 + (size_t)t * a.Hcq)[j8] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    // paths 5 and 6: the cache row
    if (a.nslots <= 0) return;
    const long long slot = a.slots[t];
    if (slot < 0 || slot >= a.nslots) {
        if (tid == 0) atomicOr(a.status, kStatusCacheIndexRange);
        return;
    }
    for (int j4 = tid; j4 < a.Hckv / 4; j4 += kPpRowThreads) {   // Hckv % 4 == 0, kv rows 8-byte aligned
        const uint2 g = reinterpret_cast<const uint2*>(a.gamma2)[j4];
        const float2* yv = ys + a.Hcq + 4 * j4;
        *reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.kv) + (size_t)slot * a.kv_ld + 4 * j4) =
            pp_pack4<F16>(H::lo(g.x) * (yv[0].x * inv2), H::hi(g.x) * (yv[1].x * inv2),
                          H::lo(g.y) * (yv[2].x * inv2), H::hi(g.y) * (yv[3].x * inv2));
    }
    const int h = a.Dr / 2;
    const float2* yr = ys + a.Hcq + a.Hckv;
    for (int j = tid; j < h; j += kPpRowThreads) {
        const float v0 = yr[j].x, v1 = yr[j + h].x;
        const size_t tr = (size_t)t * a.Dr;
        const float o0 = v0 * H::load(a.cos, tr + j) - v1 * H::load(a.sin, tr + j);
        const float o1 = v1 * H::load(a.cos, tr + j + h) + v0 * H::load(a.sin, tr + j + h);
        if (a.kr != nullptr) {
            H::store(a.kr, (size_t)slot * a.Dr + j, o0);
            H::store(a.kr, (size_t)slot * a.Dr + j + h, o1);
        } else {
            H::store(a.kv, (size_t)slot * a.kv_ld + a.Hckv + j, o0);
            H::store(a.kv, (size_t)slot * a.kv_ld + a.Hckv + j + h, o1);
        }
    }
}

// ---------------------------------------------------------------- after the up-projection

struct PpUpArgs {
    const float* z;            // (T, n2) fp32 products, n2 = N * (D + Dr)
    int N, D, Dr;
    const int* bias1;          // (n2) or null
    const float* de1;          // (n2)
    const void* cos;           // (T, Dr) F
    const void* sin;           // (T, Dr) F
    void* qc;                  // (T, N, D) F: q^C, the A operand of the W^UK contraction
    void* qr;                  // q^R of (t, n) at qr + (t * N + n) * qr_ld
    int qr_ld;
};

// Heads per CTA of pp_up_kernel: the grid is T * ceil(N / kPpUpHeads).
constexpr int kPpUpHeads = 4;

// kPpUpHeads heads of one token per CTA; a thread takes four consecutive product columns
// (all its loads are independent 16-byte loads issued together).  D % 16 == 0, Dr % 8 == 0.
template <bool F16>
__global__ void __launch_bounds__(kPpThreads) pp_up_kernel(const PpUpArgs a) {
    using H = Half16<F16>;
    pdl_launch_dependents();
    pdl_wait();
    const int groups = (a.N + kPpUpHeads - 1) / kPpUpHeads;
    const int t = blockIdx.x / groups, n0 = (blockIdx.x % groups) * kPpUpHeads;
    const int nh = min(kPpUpHeads, a.N - n0);
    const int hd = a.D + a.Dr, h = a.Dr / 2;
    const int per_head = a.D / 4 + h / 4;
    const float* z = a.z + (size_t)t * a.N * hd;
    auto deq4 = [&](int c) {
        float4 v = __ldcg(reinterpret_cast<const float4*>(z + c));
        if (a.bias1 != nullptr) {
            const int4 b = *reinterpret_cast<const int4*>(a.bias1 + c);
            v.x += (float)b.x, v.y += (float)b.y, v.z += (float)b.z, v.w += (float)b.w;
        }
        const float4 s = *reinterpret_cast<const float4*>(a.de1 + c);
        return make_float4(v.x * s.x, v.y * s.y, v.z * s.z, v.w * s.w);
    };
    for (int task = threadIdx.x; task < nh * per_head; task += kPpThreads) {
        const int n = n0 + task / per_head, r = task % per_head;
        if (r < a.D / 4) {
            const float4 v = deq4(n * hd + 4 * r);
            *reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.qc) + ((size_t)t * a.N + n) * a.D + 4 * r) =
                pp_pack4<F16>(v.x, v.y, v.z, v.w);
        } else {
            const int j = 4 * (r - a.D / 4);
            const int c0 = n * hd + a.D + j;
            const float4 v0 = deq4(c0), v1 = deq4(c0 + h);
            const size_t tr = (size_t)t * a.Dr;
            const uint2 cl = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(a.cos) + tr + j);
            const uint2 ch = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(a.cos) + tr + j + h);
            const uint2 sl = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(a.sin) + tr + j);
            const uint2 sh = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(a.sin) + tr + j + h);
            const float x0[4] = {v0.x, v0.y, v0.z, v0.w}, x1[4] = {v1.x, v1.y, v1.z, v1.w};
            const float c_lo[4] = {H::lo(cl.x), H::hi(cl.x), H::lo(cl.y), H::hi(cl.y)};
            const float c_hi[4] = {H::lo(ch.x), H::hi(ch.x), H::lo(ch.y), H::hi(ch.y)};
            const float s_lo[4] = {H::lo(sl.x), H::hi(sl.x), H::lo(sl.y), H::hi(sl.y)};
            const float s_hi[4] = {H::lo(sh.x), H::hi(sh.x), H::lo(sh.y), H::hi(sh.y)};
            float o0[4], o1[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                o0[e] = x0[e] * c_lo[e] - x1[e] * s_lo[e];
                o1[e] = x1[e] * c_hi[e] + x0[e] * s_hi[e];
            }
            uint16_t* dst = static_cast<uint16_t*>(a.qr) + ((size_t)t * a.N + n) * a.qr_ld;
            *reinterpret_cast<uint2*>(dst + j) = pp_pack4<F16>(o0[0], o0[1], o0[2], o0[3]);
            *reinterpret_cast<uint2*>(dst + j + h) = pp_pack4<F16>(o1[0], o1[1], o1[2], o1[3]);
        }
    }
}

}  // namespace mla
