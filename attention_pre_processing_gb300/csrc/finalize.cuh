// Row-wise kernels around the GEMMs:
//   finalize_down: adds the down-projection's fp32 partials, then RmsNorm of c^Q and c^KV,
//                  "half" RoPE of k^R, the paged-cache writes of c^KV and k^R, and the bf16
//                  (or int8-coded) c^Q that feeds the up-projection.
//   finalize_up:   adds the up-projection's fp32 partials, applies RoPE to each head's rope
//                  columns (q^R) and writes q^C of every head for the W^UK contraction.
//   convert_i8_to_bf16: exact int8 -> bf16 widening of the int8 operands.
// One CTA handles one token at a time; every sum runs in a fixed order (deterministic).
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "gemm_tc.cuh"
#include "ptx.cuh"

namespace mla {

constexpr int kRowThreads = 256;

// Where the fp32 partial products of a GEMM live, and how to add them up.
struct PartialSrc {
    const float* p;
    int split;         // 1: stream-K slots (see gemm_tc.cuh); 0: one T x ncols matrix
    long long total;   // split: n_tiles * kblocks
    int grid;          // split: CTAs of the GEMM
    int kblocks;
    int bn;
    int T;
    int ncols;
};

// The CTA whose piece holds flattened k-block x.
__device__ __forceinline__ int piece_owner(long long x, long long total, int G) {
    long long c = ((x + 1) * G + total - 1) / total - 1;
    return (int)(c < G - 1 ? c : G - 1);
}

__device__ __forceinline__ float gather_sum(const PartialSrc& s, int t, int col) {
    if (!s.split) return s.p[(size_t)t * s.ncols + col];
    const int tile = col / s.bn;
    const int cin = col - tile * s.bn;
    const long long x0 = (long long)tile * s.kblocks;
    const int c0 = piece_owner(x0, s.total, s.grid);
    const int c1 = piece_owner(x0 + s.kblocks - 1, s.total, s.grid);
    float acc = 0.f;
    for (int c = c0; c <= c1; ++c) {
        const long long lo = (long long)c * s.total / s.grid;
        const int part = (lo / s.kblocks == tile) ? 0 : 1;
        acc += s.p[((size_t)(2 * c + part) * s.T + t) * s.bn + cin];
    }
    return acc;
}

// Deterministic block-wide sum / max (fixed shuffle tree, fixed warp order).
template <bool kMax>
__device__ __forceinline__ float block_reduce(float v, float* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float w = __shfl_xor_sync(0xffffffffu, v, o);
        v = kMax ? fmaxf(v, w) : v + w;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float r = kMax ? 0.f : 0.f;
    if (threadIdx.x < 32) {
        r = (lane < (int)(blockDim.x >> 5)) ? red[lane] : 0.f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float w = __shfl_xor_sync(0xffffffffu, r, o);
            r = kMax ? fmaxf(r, w) : r + w;
        }
        if (lane == 0) red[32] = r;
    }
    __syncthreads();
    return red[32];
}

struct DownArgs {
    int T, Hcq, Hckv, Dr;
    PartialSrc src;                     // ncols = Hcq + Hckv + Dr
    const float* scale_x;               // int8 tokenX: (T) per-token dequant, else null
    const float* scale_w_dq;            // (Hcq)
    const float* scale_w_dkvkr;         // (Hckv + Dr)
    const __nv_bfloat16* gamma_cq;
    const __nv_bfloat16* gamma_ckv;
    float eps_cq, eps_ckv;
    const __nv_bfloat16* rope_cos;      // (T, Dr)
    const __nv_bfloat16* rope_sin;
    const long long* cache_index;       // (T)
    long long nslots;                   // BlockNum * BlockSize
    void* kv_cache;                     // (nslots, Hckv) bf16 or int8
    int kv_int8;
    const float* quant_scale_ckv;       // (Hckv)
    void* kr_cache;                     // (nslots, Dr) bf16 or int8
    int kr_int8;
    const float* quant_scale_ckr;       // (Dr)
    __nv_bfloat16* c_q;                 // (T, Hcq): bf16 c^Q, or int8 codes held as bf16
    int cq_quant;                       // dynamic per-token int8 codes of c^Q
    const float* smooth_cq;             // (Hcq) or null
    float* c_q_scale;                   // (T)
    uint32_t* status;
};

__global__ void __launch_bounds__(kRowThreads) finalize_down_kernel(const DownArgs a) {
    extern __shared__ float ys[];   // Hcq + Hckv + Dr
    __shared__ float red[33];
    pdl_wait();
    const int ncols = a.Hcq + a.Hckv + a.Dr;
    const int h = a.Dr / 2;
    for (int t = blockIdx.x; t < a.T; t += gridDim.x) {
        const float sx = a.scale_x ? a.scale_x[t] : 1.f;
        for (int c = threadIdx.x; c < ncols; c += blockDim.x) {
            float v = gather_sum(a.src, t, c);
            if (a.scale_x) v *= sx * (c < a.Hcq ? a.scale_w_dq[c] : a.scale_w_dkvkr[c - a.Hcq]);
            ys[c] = v;
        }
        __syncthreads();
        float sq = 0.f, skv = 0.f;
        for (int j = threadIdx.x; j < a.Hcq; j += blockDim.x) sq += ys[j] * ys[j];
        for (int j = threadIdx.x; j < a.Hckv; j += blockDim.x) skv += ys[a.Hcq + j] * ys[a.Hcq + j];
        sq = block_reduce<false>(sq, red);
        skv = block_reduce<false>(skv, red);
        // RmsNorm: gamma * y / sqrt(mean(y^2) + eps), epsilon inside the root.
        const float inv_q = 1.f / sqrtf(sq / (float)a.Hcq + a.eps_cq);
        const float inv_kv = 1.f / sqrtf(skv / (float)a.Hckv + a.eps_ckv);

        if (!a.cq_quant) {
            for (int j = threadIdx.x; j < a.Hcq; j += blockDim.x)
                a.c_q[(size_t)t * a.Hcq + j] = __float2bfloat16_rn(__bfloat162float(a.gamma_cq[j]) * ys[j] * inv_q);
        } else {
            // Per-token dynamic int8 codes of c^Q (times the smooth scales when given).
            float m = 0.f;
            for (int j = threadIdx.x; j < a.Hcq; j += blockDim.x) {
                float u = __bfloat162float(a.gamma_cq[j]) * ys[j] * inv_q;
                if (a.smooth_cq) u *= a.smooth_cq[j];
                m = fmaxf(m, fabsf(u));
            }
            m = block_reduce<true>(m, red);
            const float scale = m / 127.f;
            for (int j = threadIdx.x; j < a.Hcq; j += blockDim.x) {
                float u = __bfloat162float(a.gamma_cq[j]) * ys[j] * inv_q;
                if (a.smooth_cq) u *= a.smooth_cq[j];
                const int q = scale > 0.f ? quant_i8(__fdiv_rn(u, scale)) : 0;
                a.c_q[(size_t)t * a.Hcq + j] = __int2bfloat16_rn(q);
            }
            if (threadIdx.x == 0) a.c_q_scale[t] = scale;
        }

        if (a.nslots > 0) {
            const long long slot = a.cache_index[t];
            if (slot < 0 || slot >= a.nslots) {
                if (threadIdx.x == 0) atomicOr(a.status, kStatusCacheIndexRange);
            } else {
                for (int j = threadIdx.x; j < a.Hckv; j += blockDim.x) {
                    const float v = __bfloat162float(a.gamma_ckv[j]) * ys[a.Hcq + j] * inv_kv;
                    if (a.kv_int8)
                        reinterpret_cast<int8_t*>(a.kv_cache)[slot * a.Hckv + j] =
                            (int8_t)quant_i8(v * a.quant_scale_ckv[j]);
                    else
                        reinterpret_cast<__nv_bfloat16*>(a.kv_cache)[slot * a.Hckv + j] = __float2bfloat16_rn(v);
                }
                const float* kr = ys + a.Hcq + a.Hckv;
                const __nv_bfloat16* cs = a.rope_cos + (size_t)t * a.Dr;
                const __nv_bfloat16* sn = a.rope_sin + (size_t)t * a.Dr;
                for (int j = threadIdx.x; j < h; j += blockDim.x) {
                    const float x0 = kr[j], x1 = kr[j + h];
                    const float o0 = x0 * __bfloat162float(cs[j]) - x1 * __bfloat162float(sn[j]);
                    const float o1 = x1 * __bfloat162float(cs[j + h]) + x0 * __bfloat162float(sn[j + h]);
                    if (a.kr_int8) {
                        int8_t* d = reinterpret_cast<int8_t*>(a.kr_cache) + slot * a.Dr;
                        d[j] = (int8_t)quant_i8(o0 * a.quant_scale_ckr[j]);
                        d[j + h] = (int8_t)quant_i8(o1 * a.quant_scale_ckr[j + h]);
                    } else {
                        __nv_bfloat16* d = reinterpret_cast<__nv_bfloat16*>(a.kr_cache) + slot * a.Dr;
                        d[j] = __float2bfloat16_rn(o0);
                        d[j + h] = __float2bfloat16_rn(o1);
                    }
                }
            }
        }
        __syncthreads();
    }
    pdl_launch_dependents();
}

struct UpArgs {
    int T, N, D, Dr;
    PartialSrc src;                     // ncols = N * (D + Dr)
    const float* row_scale;             // (T) dequant of int8 c^Q codes, or null
    const float* col_scale;             // (N*(D+Dr)) dequant of int8 weightUqQr, or null
    const __nv_bfloat16* rope_cos;
    const __nv_bfloat16* rope_sin;
    __nv_bfloat16* q_c;                 // (T, N, D)
    __nv_bfloat16* q_rope;              // (T, N, Dr)
};

__global__ void __launch_bounds__(kRowThreads) finalize_up_kernel(const UpArgs a) {
    pdl_wait();
    const int h = a.Dr / 2;
    const int per_head = a.D + h;       // work items per head: D nope columns + Dr/2 rope pairs
    const int W = a.D + a.Dr;
    for (int t = blockIdx.x; t < a.T; t += gridDim.x) {
        const float rs = a.row_scale ? a.row_scale[t] : 1.f;
        const __nv_bfloat16* cs = a.rope_cos + (size_t)t * a.Dr;
        const __nv_bfloat16* sn = a.rope_sin + (size_t)t * a.Dr;
        for (int p = threadIdx.x; p < a.N * per_head; p += blockDim.x) {
            const int n = p / per_head;
            const int r = p - n * per_head;
            const int base = n * W;
            if (r < a.D) {
                float v = gather_sum(a.src, t, base + r);
                if (a.col_scale) v *= rs * a.col_scale[base + r];
                a.q_c[((size_t)t * a.N + n) * a.D + r] = __float2bfloat16_rn(v);
            } else {
                const int j = r - a.D;
                float x0 = gather_sum(a.src, t, base + a.D + j);
                float x1 = gather_sum(a.src, t, base + a.D + j + h);
                if (a.col_scale) {
                    x0 *= rs * a.col_scale[base + a.D + j];
                    x1 *= rs * a.col_scale[base + a.D + j + h];
                }
                const float o0 = x0 * __bfloat162float(cs[j]) - x1 * __bfloat162float(sn[j]);
                const float o1 = x1 * __bfloat162float(cs[j + h]) + x0 * __bfloat162float(sn[j + h]);
                __nv_bfloat16* d = a.q_rope + ((size_t)t * a.N + n) * a.Dr;
                d[j] = __float2bfloat16_rn(o0);
                d[j + h] = __float2bfloat16_rn(o1);
            }
        }
    }
    pdl_launch_dependents();
}

// Exact int8 -> bf16 widening (|v| <= 128 has at most 8 significant bits).
__global__ void __launch_bounds__(256) convert_i8_to_bf16_kernel(const int8_t* __restrict__ src,
                                                                 __nv_bfloat16* __restrict__ dst, long long n) {
    pdl_wait();
    const long long n16 = n / 16;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += stride) {
        const int4 v = reinterpret_cast<const int4*>(src)[i];
        const int w[4] = {v.x, v.y, v.z, v.w};
        uint4 o[2];
        uint32_t* ow = reinterpret_cast<uint32_t*>(o);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int b0 = (int)(int8_t)((w[k] >> (16 * e)) & 0xFF);
                const int b1 = (int)(int8_t)((w[k] >> (16 * e + 8)) & 0xFF);
                ow[2 * k + e] = pack_bf16((float)b0, (float)b1);
            }
        }
        reinterpret_cast<uint4*>(dst)[2 * i] = o[0];
        reinterpret_cast<uint4*>(dst)[2 * i + 1] = o[1];
    }
    for (long long i = n16 * 16 + (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
        dst[i] = __int2bfloat16_rn((int)src[i]);
    pdl_launch_dependents();
}

}  // namespace mla
