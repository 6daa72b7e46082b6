// Row kernels of the "aclnnMlaPreprocess" variant (the three contractions run on gemm_tc):
//   pp_widen_t_kernel   int8 weight stored one row per output column -> bf16 (k, n) for the
//                       GEMMs (exact: |v| <= 128 has at most 8 significant bits)
//   pp_quant_x_kernel   RmsNormQuant of the input (or the quantiser alone) -> int8 codes held
//                       as bf16, the A operand of the down-projection
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

// The int8 code of the page's static asymmetric quantiser,
//   code = clamp(round_half_away(v * qs) + qo, -128, 127),  v = (gamma * y) / r + beta  (norm)
//                                                            v = y                     (no norm)
// decided as in exact double arithmetic, in this operation order: the fp32 estimate decides
// unless it lies within its error bound of a rounding boundary (a half-integer), and then the
// double expression does.  The bound: four fp32 roundings of at most 2^-24 relative each, on
// terms no larger than (|gamma * y / r| + |beta|) * |qs|; 1e-5 of that is a 40x margin.
// r is sqrt(mean(y^2) + eps) in double; inv its fp32 reciprocal.
__device__ __forceinline__ float pp_code(double y, float g, float b, bool norm, double r, float inv, float qs,
                                         int qo) {
    const float yf = (float)y;
    const float a = norm ? g * yf * inv : yf;
    const float sf = (a + (norm ? b : 0.f)) * qs;
    const float margin = 1e-5f * (fabsf(a) + (norm ? fabsf(b) : 0.f)) * fabsf(qs) + 1e-30f;
    float q;
    if (fabsf(sf - floorf(sf) - 0.5f) <= margin) {
        const double v = norm ? __dadd_rn(__ddiv_rn(__dmul_rn((double)g, y), r), (double)b) : y;
        q = (float)round(__dmul_rn(v, (double)qs));   // round(): halves away from zero
    } else {
        q = roundf(sf);
    }
    return fminf(fmaxf(q + (float)qo, -128.f), 127.f);
}

// Deterministic double sum over the CTA (fixed shuffle tree, then the warps in order).
__device__ __forceinline__ double pp_block_sum(double v, double* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    if (warp == 0) {
        double r = lane < kPpThreads / 32 ? red[lane] : 0.0;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
        if (lane == 0) red[kPpThreads / 32] = r;
    }
    __syncthreads();
    return red[kPpThreads / 32];
}

// ---------------------------------------------------------------- weight widening

// src: int8 (R, C), one row per output column n (R = columns, C = k).  dst0: bf16 (C, rsplit)
// holding columns n < rsplit; dst1: bf16 (C, R - rsplit) holding the rest (may be null when
// rsplit == R).  64 x 64 tiles through shared memory, a 1D grid of ceil(C/64) * ceil(R/64).
// Requires C % 16 == 0, R % 8 == 0 and rsplit % 8 == 0 (16-byte loads and stores).
__global__ void __launch_bounds__(kPpThreads) pp_widen_t_kernel(const int8_t* __restrict__ src, int R, int C,
                                                                __nv_bfloat16* __restrict__ dst0,
                                                                __nv_bfloat16* __restrict__ dst1, int rsplit) {
    __shared__ __align__(16) int8_t tile[64][64 + 16];
    pdl_launch_dependents();
    pdl_wait();
    const int cb = (C + 63) / 64;   // one block per 64 x 64 tile, k-tile fastest
    const int c0 = (int)(blockIdx.x % cb) * 64, r0 = (int)(blockIdx.x / cb) * 64;
    const int tid = threadIdx.x;
    {
        const int rr = tid >> 2, cc = (tid & 3) * 16;
        const int r = r0 + rr, c = c0 + cc;
        int4 v = make_int4(0, 0, 0, 0);
        if (r < R && c < C) v = *reinterpret_cast<const int4*>(src + (size_t)r * C + c);
        *reinterpret_cast<int4*>(&tile[rr][cc]) = v;
    }
    __syncthreads();
#pragma unroll
    for (int it = 0; it < 2; ++it) {
        const int idx = tid + it * kPpThreads;
        const int kk = idx >> 3, nn = (idx & 7) * 8;
        const int k = c0 + kk, n = r0 + nn;
        if (k >= C || n >= R) continue;
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
            w[e] = pack_bf16((float)tile[nn + 2 * e][kk], (float)tile[nn + 2 * e + 1][kk]);
        const uint4 o = make_uint4(w[0], w[1], w[2], w[3]);
        if (n < rsplit)
            *reinterpret_cast<uint4*>(dst0 + (size_t)k * rsplit + n) = o;
        else
            *reinterpret_cast<uint4*>(dst1 + (size_t)k * (R - rsplit) + (n - rsplit)) = o;
    }
}

// ---------------------------------------------------------------- input quantisation

struct PpQuantArgs {
    const void* x;          // (T, He) F
    const void* gamma;      // (He) F
    const void* beta;       // (He) F
    const void* qscale;     // (1) F
    const int8_t* qoffset;  // (1)
    __nv_bfloat16* out;     // (T, He): codes as bf16
    int He;
    double eps;
    int do_norm;
};

// One CTA per token.  He % 8 == 0.
template <bool F16>
__global__ void __launch_bounds__(kPpThreads) pp_quant_x_kernel(const PpQuantArgs a) {
    using H = Half16<F16>;
    __shared__ double red[kPpThreads / 32 + 1];
    pdl_launch_dependents();
    pdl_wait();
    const int t = blockIdx.x, tid = threadIdx.x;
    const uint4* xr = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.x) + (size_t)t * a.He);
    const int n8 = a.He / 8;
    double r = 1.0;
    float inv = 1.f;
    if (a.do_norm) {
        // squares of 16-bit values are exact in double, and so is their sum for any order
        // (the terms span far fewer than 53 bits): r is the correctly rounded definition
        double ss = 0.0;
        for (int i = tid; i < n8; i += kPpThreads) {
            const uint4 v = xr[i];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const double lo = H::lo(w[e]), hi = H::hi(w[e]);
                ss += lo * lo + hi * hi;
            }
        }
        ss = pp_block_sum(ss, red);
        r = __dsqrt_rn(__dadd_rn(__ddiv_rn(ss, (double)a.He), a.eps));
        inv = (float)(1.0 / r);
    }
    const float qs = H::load(a.qscale, 0);
    const int qo = (int)a.qoffset[0];
    const uint4* gr = reinterpret_cast<const uint4*>(a.gamma);
    const uint4* br = reinterpret_cast<const uint4*>(a.beta);
    uint4* outr = reinterpret_cast<uint4*>(a.out + (size_t)t * a.He);
    for (int i = tid; i < n8; i += kPpThreads) {
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
            o[e] = pack_bf16(pp_code(H::lo(w[e]), H::lo(gw[e]), H::lo(bw[e]), nm, r, inv, qs, qo),
                             pp_code(H::hi(w[e]), H::hi(gw[e]), H::hi(bw[e]), nm, r, inv, qs, qo));
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
    __nv_bfloat16* codes1;     // (T, Hcq): codes as bf16
    const void* gamma2;        // (Hckv) F
    const void* cos;           // (T, Dr) F
    const void* sin;           // (T, Dr) F
    const int* slots;          // (T)
    long long nslots;
    void* kv;                  // (nslots, kv_ld) F
    int kv_ld;                 // Hckv + Dr (cacheMode 0) or Hckv (1)
    void* kr;                  // cacheMode 1: (nslots, Dr) F; cacheMode 0: null (k^R after k^N in kv)
    double eps;
    uint32_t* status;
};

// One CTA per token; dynamic shared memory holds the token's n1 values in double.
template <bool F16>
__global__ void __launch_bounds__(kPpThreads) pp_mid_kernel(const PpMidArgs a) {
    using H = Half16<F16>;
    extern __shared__ double ys[];
    __shared__ double red[kPpThreads / 32 + 1];
    pdl_launch_dependents();
    pdl_wait();
    const int t = blockIdx.x, tid = threadIdx.x;
    const float* y0 = a.y + (size_t)t * a.n1;
    double ss1 = 0.0, ss2 = 0.0;
    for (int j = tid; j < a.n1; j += kPpThreads) {
        // the k-range partials are integer-valued (int8 products), so their fp32 sum in k-range
        // order is the exact integer while it stays below 2^24; bias and scale then in double
        float acc = 0.f;
        for (int s = 0; s < a.ksplit; ++s) acc += __ldcg(y0 + (size_t)s * a.slot_stride + j);   // k-range order
        double v = (double)acc;
        if (a.bias0 != nullptr) v += (double)a.bias0[j];
        v = __dmul_rn(v, (double)a.de0[j]);
        ys[j] = v;
        if (j < a.Hcq)
            ss1 += v * v;
        else if (j < a.Hcq + a.Hckv)
            ss2 += v * v;
    }
    ss1 = pp_block_sum(ss1, red);
    ss2 = pp_block_sum(ss2, red);   // its barriers also publish ys
    const double r1 = __dsqrt_rn(__dadd_rn(__ddiv_rn(ss1, (double)a.Hcq), a.eps));
    const float inv1 = (float)(1.0 / r1);
    const float inv2 = (float)(1.0 / __dsqrt_rn(__dadd_rn(__ddiv_rn(ss2, (double)a.Hckv), a.eps)));
    // path 1: RmsNormQuant -> the up-projection's codes
    const float qs = H::load(a.qscale1, 0);
    const int qo = (int)a.qoffset1[0];
    for (int j = 2 * tid; j < a.Hcq; j += 2 * kPpThreads) {
        const float c0 = pp_code(ys[j], H::load(a.gamma1, j), H::load(a.beta1, j), true, r1, inv1, qs, qo);
        const float c1 = pp_code(ys[j + 1], H::load(a.gamma1, j + 1), H::load(a.beta1, j + 1), true, r1, inv1, qs, qo);
        *reinterpret_cast<uint32_t*>(a.codes1 + (size_t)t * a.Hcq + j) = pack_bf16(c0, c1);
    }
    // paths 5 and 6: the cache row
    if (a.nslots <= 0) return;
    const long long slot = a.slots[t];
    if (slot < 0 || slot >= a.nslots) {
        if (tid == 0) atomicOr(a.status, kStatusCacheIndexRange);
        return;
    }
    for (int j = tid; j < a.Hckv; j += kPpThreads)
        H::store(a.kv, (size_t)slot * a.kv_ld + j, H::load(a.gamma2, j) * ((float)ys[a.Hcq + j] * inv2));
    const int h = a.Dr / 2;
    const double* yr = ys + a.Hcq + a.Hckv;
    for (int j = tid; j < h; j += kPpThreads) {
        const float v0 = (float)yr[j], v1 = (float)yr[j + h];
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

// One CTA per token.
template <bool F16>
__global__ void __launch_bounds__(kPpThreads) pp_up_kernel(const PpUpArgs a) {
    using H = Half16<F16>;
    pdl_launch_dependents();
    pdl_wait();
    const int t = blockIdx.x, tid = threadIdx.x;
    const int hd = a.D + a.Dr;
    const size_t n2 = (size_t)a.N * hd;
    const float* z = a.z + (size_t)t * n2;
    auto deq = [&](int c) {
        float acc = __ldcg(z + c);
        if (a.bias1 != nullptr) acc += (float)a.bias1[c];
        return acc * a.de1[c];
    };
    for (int i = tid; i < a.N * a.D; i += kPpThreads) {
        const int n = i / a.D, d = i - n * a.D;
        H::store(a.qc, (size_t)t * a.N * a.D + i, deq(n * hd + d));
    }
    const int h = a.Dr / 2;
    const size_t tr = (size_t)t * a.Dr;
    for (int i = tid; i < a.N * h; i += kPpThreads) {
        const int n = i / h, j = i - n * h;
        const int c0 = n * hd + a.D + j;
        const float v0 = deq(c0), v1 = deq(c0 + h);
        const float o0 = v0 * H::load(a.cos, tr + j) - v1 * H::load(a.sin, tr + j);
        const float o1 = v1 * H::load(a.cos, tr + j + h) + v0 * H::load(a.sin, tr + j + h);
        const size_t base = ((size_t)t * a.N + n) * a.qr_ld;
        H::store(a.qr, base + j, o0);
        H::store(a.qr, base + j + h, o1);
    }
}

}  // namespace mla
