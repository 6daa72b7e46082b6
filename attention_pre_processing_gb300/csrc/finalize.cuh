// Row-wise kernels around the GEMMs:
//   finalize_down: reads the down-projection's fp32 rows, then RmsNorm of c^Q and c^KV,
//                  "half" RoPE of k^R, the paged-cache writes of c^KV and k^R, and the bf16
//                  (or int8-coded) c^Q that feeds the up-projection.
//   finalize_up:   reads the up-projection's fp32 rows, applies RoPE to each head's rope
//                  columns (q^R) and writes q^C of every head for the W^UK contraction.
//   convert_i8_to_bf16: exact int8 -> bf16 widening of the int8 operands.
// Every sum runs in a fixed order (deterministic).
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "gemm_tc.cuh"
#include "ptx.cuh"

namespace mla {

constexpr int kRowThreads = 256;

// fp32 product rows written by a GEMM: `slots` k-range slots of T x ncols, row-major, added
// in slot order.
struct PartialSrc {
    const float* p;
    int ncols;
    int slots;
    size_t slot_stride;   // T * ncols
};

__device__ __forceinline__ float gather_sum(const PartialSrc& s, int t, int col) {
    const float* p = s.p + (size_t)t * s.ncols + col;
    float v = __ldcg(p);
    for (int k = 1; k < s.slots; ++k) v += __ldcg(p + k * s.slot_stride);
    return v;
}

struct DownArgs {
    int T, Hcq, Hckv, Dr;
    PartialSrc src;                     // T x (Hcq + Hckv + Dr)
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
    int cq_quant;                       // dynamic per-token int8 codes of c^Q, written as fp16
    const float* smooth_cq;             // (Hcq) or null
    float* c_q_scale;                   // (T)
    int cq_done;                        // c^Q was written by the down-projection (rows only need c^KV | k^R)
    uint32_t* status;
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Barrier over the threads that share one row (the whole CTA).
struct CtaSync {
    __device__ __forceinline__ void operator()() const { __syncthreads(); }
};

// Deterministic reduction over NT threads (tid in [0, NT)): fixed shuffle tree per warp, then
// the per-warp values in warp order.  `red` holds NT/32 + 1 floats.
template <int NT, bool kMax, class Sync>
__device__ __forceinline__ float group_reduce(float v, float* red, int tid, Sync sync) {
    v = kMax ? warp_max(v) : warp_sum(v);
    const int warp = tid >> 5, lane = tid & 31;
    sync();
    if (lane == 0) red[warp] = v;
    sync();
    if (warp == 0) {
        float r = lane < NT / 32 ? red[lane] : 0.f;
        r = kMax ? warp_max(r) : warp_sum(r);
        if (lane == 0) red[NT / 32] = r;
    }
    sync();
    return red[NT / 32];
}

// The row work after the down-projection, for token t, by NT threads (tid in [0, NT)):
// add the k-range slots of the fp32 row (fixed order), RmsNorm of c^Q and c^KV (epsilon inside
// the root), "half" RoPE of k^R, the cache writes at cacheIndex[t], and c^Q for the
// up-projection (bf16, or per-token int8 codes held as bf16 when weightUqQr is int8).
// ys: Hcq + Hckv + Dr floats of shared memory; red: NT/32 + 1 floats; gcq / gckv: the gammas,
// already staged in shared memory.  Every load that does not depend on the partial sums is
// issued before them, and a thread's partial loads for up to kRowCols columns are in flight
// together: with few rows (decode) the row then costs about one memory latency; with many rows a
// small kRowCols keeps the registers, and so the rows in flight per SM, up.  kSlots > 0: every
// k-range slot (up to kSlots) of those columns is requested at once, instead of four slots per
// round (each round waits for the previous one's loads).
template <int NT, int kRowCols, class Sync, int kSlots = 0>
__device__ __forceinline__ void down_row(const DownArgs& a, int t, int tid, float* ys, float* red,
                                         const __nv_bfloat16* gcq, const __nv_bfloat16* gckv, Sync sync) {
    const int ncols = a.Hcq + a.Hckv + a.Dr;
    const int h = a.Dr / 2;
    const long long slot = a.nslots > 0 ? a.cache_index[t] : -1;
    const float sx = a.scale_x ? a.scale_x[t] : 1.f;
    const __nv_bfloat16* rc = a.rope_cos + (size_t)t * a.Dr;
    const __nv_bfloat16* rs = a.rope_sin + (size_t)t * a.Dr;
    float cos0 = 0.f, cos1 = 0.f, sin0 = 0.f, sin1 = 0.f;
    if (tid < h) {
        cos0 = __bfloat162float(rc[tid]);
        cos1 = __bfloat162float(rc[tid + h]);
        sin0 = __bfloat162float(rs[tid]);
        sin1 = __bfloat162float(rs[tid + h]);
    }
    const float* src = a.src.p + (size_t)t * a.src.ncols;
    float sq = 0.f, skv = 0.f;
    for (int c0 = tid; c0 < ncols; c0 += kRowCols * NT) {
        float v[kRowCols];
        if constexpr (kSlots > 0) {
            float w[kSlots][kRowCols];
#pragma unroll
            for (int k = 0; k < kSlots; ++k)
#pragma unroll
                for (int u = 0; u < kRowCols; ++u) {
                    const int c = c0 + u * NT;
                    w[k][u] = (k < a.src.slots && c < ncols) ? __ldcg(src + k * a.src.slot_stride + c) : 0.f;
                }
#pragma unroll
            for (int u = 0; u < kRowCols; ++u) {
                v[u] = w[0][u];
#pragma unroll
                for (int k = 1; k < kSlots; ++k) v[u] += w[k][u];   // k-range order
            }
        } else {
#pragma unroll
        for (int u = 0; u < kRowCols; ++u) {
            const int c = c0 + u * NT;
            v[u] = c < ncols ? __ldcg(src + c) : 0.f;
        }
        for (int k0 = 1; k0 < a.src.slots; k0 += 4) {
            float w[4][kRowCols];
#pragma unroll
            for (int k = 0; k < 4; ++k)
#pragma unroll
                for (int u = 0; u < kRowCols; ++u) {
                    const int c = c0 + u * NT;
                    w[k][u] = (k0 + k < a.src.slots && c < ncols) ? __ldcg(src + (k0 + k) * a.src.slot_stride + c) : 0.f;
                }
#pragma unroll
            for (int k = 0; k < 4; ++k)
#pragma unroll
                for (int u = 0; u < kRowCols; ++u) v[u] += w[k][u];
        }
        }
#pragma unroll
        for (int u = 0; u < kRowCols; ++u) {
            const int c = c0 + u * NT;
            if (c >= ncols) continue;
            float y = v[u];
            if (a.scale_x) y *= sx * (c < a.Hcq ? a.scale_w_dq[c] : a.scale_w_dkvkr[c - a.Hcq]);
            ys[c] = y;
            if (c < a.Hcq) sq += y * y;
            else if (c < a.Hcq + a.Hckv) skv += y * y;
        }
    }
    sq = group_reduce<NT, false>(sq, red, tid, sync);
    skv = group_reduce<NT, false>(skv, red, tid, sync);   // its barriers also publish ys
    // RmsNorm: gamma * y / sqrt(mean(y^2) + eps), epsilon inside the root.
    const float inv_q = 1.f / sqrtf(sq / (float)a.Hcq + a.eps_cq);
    const float inv_kv = 1.f / sqrtf(skv / (float)a.Hckv + a.eps_ckv);

    __nv_bfloat16* cq = a.c_q + (size_t)t * a.Hcq;
    if (a.cq_done) {
    } else if (!a.cq_quant) {
        for (int j = 2 * tid; j < a.Hcq; j += 2 * NT) {
            const __nv_bfloat162 g2 = *reinterpret_cast<const __nv_bfloat162*>(gcq + j);
            *reinterpret_cast<__nv_bfloat162*>(cq + j) =
                __floats2bfloat162_rn(__low2float(g2) * ys[j] * inv_q, __high2float(g2) * ys[j + 1] * inv_q);
        }
    } else {
        // Per-token dynamic int8 codes of c^Q (times the smooth scales when given).
        float m = 0.f;
        for (int j = tid; j < a.Hcq; j += NT) {
            float u = __bfloat162float(gcq[j]) * ys[j] * inv_q;
            if (a.smooth_cq) u *= a.smooth_cq[j];
            m = fmaxf(m, fabsf(u));
        }
        m = group_reduce<NT, true>(m, red, tid, sync);
        const float scale = m / 127.f;
        for (int j = tid; j < a.Hcq; j += NT) {
            float u = __bfloat162float(gcq[j]) * ys[j] * inv_q;
            if (a.smooth_cq) u *= a.smooth_cq[j];
            const int q = scale > 0.f ? quant_i8(__fdiv_rn(u, scale)) : 0;
            reinterpret_cast<__half*>(cq)[j] = __int2half_rn(q);   // exact: the fp16 A operand of the int8 GEMM
        }
        if (tid == 0) a.c_q_scale[t] = scale;
    }

    if (a.nslots > 0) {
        if (slot < 0 || slot >= a.nslots) {
            if (tid == 0) atomicOr(a.status, kStatusCacheIndexRange);
        } else {
            const float* ykv = ys + a.Hcq;
            if (a.kv_int8) {
                int8_t* d = reinterpret_cast<int8_t*>(a.kv_cache) + slot * a.Hckv;
                for (int j = tid; j < a.Hckv; j += NT)
                    d[j] = (int8_t)quant_i8(__bfloat162float(gckv[j]) * ykv[j] * inv_kv * a.quant_scale_ckv[j]);
            } else {
                __nv_bfloat16* d = reinterpret_cast<__nv_bfloat16*>(a.kv_cache) + slot * a.Hckv;
                for (int j = 2 * tid; j < a.Hckv; j += 2 * NT) {
                    const __nv_bfloat162 g2 = *reinterpret_cast<const __nv_bfloat162*>(gckv + j);
                    *reinterpret_cast<__nv_bfloat162*>(d + j) =
                        __floats2bfloat162_rn(__low2float(g2) * ykv[j] * inv_kv, __high2float(g2) * ykv[j + 1] * inv_kv);
                }
            }
            const float* kr = ys + a.Hcq + a.Hckv;
            for (int j = tid; j < h; j += NT) {
                const bool pre = j < NT;   // this thread's first pair: tables already in registers
                const float cj = pre ? cos0 : __bfloat162float(rc[j]);
                const float ch = pre ? cos1 : __bfloat162float(rc[j + h]);
                const float sj = pre ? sin0 : __bfloat162float(rs[j]);
                const float sh = pre ? sin1 : __bfloat162float(rs[j + h]);
                const float x0 = kr[j], x1 = kr[j + h];
                const float o0 = x0 * cj - x1 * sj;
                const float o1 = x1 * ch + x0 * sh;
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
    sync();   // ys and red are reused by the next row
}

// L2 prefetch of everything the row work of this CTA's tokens reads besides the partials.
__device__ __forceinline__ void prefetch_down_inputs(const DownArgs& a, int tid, int nthr) {
    prefetch_l2_range(a.scale_w_dq, a.scale_w_dq ? (size_t)a.Hcq * 4 : 0, tid, nthr);
    prefetch_l2_range(a.scale_w_dkvkr, a.scale_w_dkvkr ? (size_t)(a.Hckv + a.Dr) * 4 : 0, tid, nthr);
    prefetch_l2_range(a.quant_scale_ckv, a.quant_scale_ckv ? (size_t)a.Hckv * 4 : 0, tid, nthr);
    prefetch_l2_range(a.smooth_cq, a.smooth_cq ? (size_t)a.Hcq * 4 : 0, tid, nthr);
    if (tid == 0) {
        for (int t = blockIdx.x; t < a.T; t += gridDim.x) {
            prefetch_l2(a.rope_cos + (size_t)t * a.Dr);
            prefetch_l2(a.rope_sin + (size_t)t * a.Dr);
            prefetch_l2(a.cache_index + t);
            if (a.scale_x) prefetch_l2(a.scale_x + t);
        }
    }
}

// Dynamic shared memory of finalize_down_kernel: the fp32 row, then the two gammas.
__host__ __device__ inline size_t down_smem_bytes(int Hcq, int Hckv, int Dr) {
    return (((size_t)(Hcq + Hckv + Dr) * 4 + 15) & ~(size_t)15) + (size_t)(Hcq + Hckv) * 2;
}

// One CTA of NT threads per token (grid-stride).  ROWCOLS: columns of partial sums a thread has
// in flight; KS > 0: all of their k-range slots (up to KS) at once.
template <int ROWCOLS, int NT = kRowThreads, int KS = 0>
__global__ void __launch_bounds__(NT) finalize_down_kernel(const DownArgs a) {
    extern __shared__ __align__(16) uint8_t fsm[];
    float* ys = reinterpret_cast<float*>(fsm);
    __nv_bfloat16* gcq = reinterpret_cast<__nv_bfloat16*>(fsm + (((size_t)(a.Hcq + a.Hckv + a.Dr) * 4 + 15) & ~(size_t)15));
    __nv_bfloat16* gckv = gcq + a.Hcq;
    __shared__ float red[NT / 32 + 1];
    // All CTAs of this grid are resident once every one has passed here: the next kernel may
    // start its prologue (and its first weight loads) now.
    pdl_launch_dependents();
    // The gammas and the other small inputs do not depend on the previous kernel: stage and
    // prefetch them while it finishes, so that the row work does not wait on cold lines.
    // (Hcq and Hckv are multiples of 8: 16-byte copies.)
    for (int i = threadIdx.x; i < a.Hcq / 8; i += NT)
        reinterpret_cast<uint4*>(gcq)[i] = reinterpret_cast<const uint4*>(a.gamma_cq)[i];
    for (int i = threadIdx.x; i < a.Hckv / 8; i += NT)
        reinterpret_cast<uint4*>(gckv)[i] = reinterpret_cast<const uint4*>(a.gamma_ckv)[i];
    prefetch_down_inputs(a, threadIdx.x, NT);
    pdl_wait();
    __syncthreads();
    for (int t = blockIdx.x; t < a.T; t += gridDim.x)
        down_row<NT, ROWCOLS, CtaSync, KS>(a, t, threadIdx.x, ys, red, gcq, gckv, CtaSync{});
}

// Warp-per-token variant of the row work for many tokens (one k-range slot): each lane keeps
// its columns of the fp32 row in registers (column pairs 2*lane + 64*k), the two sums of
// squares and the int8 absmax are warp reductions (fixed shuffle tree), and no block barrier is
// needed, so that every row of a large call can be in flight at once.  Limits: Hcq <= 64 *
// kWQ, Hckv <= 64 * kWKV, Hcq and Hckv multiples of 64, Dr = 64.
constexpr int kWQ = 32;    // column pairs per lane of c^Q: Hcq <= 2048
constexpr int kWKV = 8;    // column pairs per lane of c^KV: Hckv <= 512
constexpr int kWarpRowThreads = 128;

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__global__ void __launch_bounds__(kWarpRowThreads) finalize_down_warp_kernel(const DownArgs a) {
    pdl_launch_dependents();
    prefetch_down_inputs(a, threadIdx.x, kWarpRowThreads);
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (kWarpRowThreads / 32) + (threadIdx.x >> 5);
    if (t >= a.T) return;   // whole warp
    const int nq = a.cq_done ? 0 : a.Hcq / 64, nkv = a.Hckv / 64, h = a.Dr / 2;
    const float* src = a.src.p + (size_t)t * a.src.ncols;
    const long long slot = a.nslots > 0 ? a.cache_index[t] : -1;
    const float sx = a.scale_x ? a.scale_x[t] : 1.f;
    // loads: the whole row of this token, every load in flight together
    float2 yq[kWQ], ykv[kWKV];
#pragma unroll
    for (int k = 0; k < kWQ; ++k)
        if (k < nq) yq[k] = __ldcs(reinterpret_cast<const float2*>(src + 2 * lane + 64 * k));
#pragma unroll
    for (int k = 0; k < kWKV; ++k)
        if (k < nkv) ykv[k] = __ldcs(reinterpret_cast<const float2*>(src + a.Hcq + 2 * lane + 64 * k));
    float kr0 = __ldcs(src + a.Hcq + a.Hckv + lane), kr1 = __ldcs(src + a.Hcq + a.Hckv + lane + h);
    const float cos0 = __bfloat162float(a.rope_cos[(size_t)t * a.Dr + lane]);
    const float cos1 = __bfloat162float(a.rope_cos[(size_t)t * a.Dr + lane + h]);
    const float sin0 = __bfloat162float(a.rope_sin[(size_t)t * a.Dr + lane]);
    const float sin1 = __bfloat162float(a.rope_sin[(size_t)t * a.Dr + lane + h]);
    if (a.scale_x) {
#pragma unroll
        for (int k = 0; k < kWQ; ++k)
            if (k < nq) {
                const int c = 2 * lane + 64 * k;
                yq[k].x *= sx * a.scale_w_dq[c];
                yq[k].y *= sx * a.scale_w_dq[c + 1];
            }
#pragma unroll
        for (int k = 0; k < kWKV; ++k)
            if (k < nkv) {
                const int c = 2 * lane + 64 * k;
                ykv[k].x *= sx * a.scale_w_dkvkr[c];
                ykv[k].y *= sx * a.scale_w_dkvkr[c + 1];
            }
        kr0 *= sx * a.scale_w_dkvkr[a.Hckv + lane];
        kr1 *= sx * a.scale_w_dkvkr[a.Hckv + lane + h];
    }
    float sq = 0.f, skv = 0.f;
#pragma unroll
    for (int k = 0; k < kWQ; ++k)
        if (k < nq) sq += yq[k].x * yq[k].x + yq[k].y * yq[k].y;
#pragma unroll
    for (int k = 0; k < kWKV; ++k)
        if (k < nkv) skv += ykv[k].x * ykv[k].x + ykv[k].y * ykv[k].y;
    sq = warp_sum_f(sq);
    skv = warp_sum_f(skv);
    // RmsNorm: gamma * y / sqrt(mean(y^2) + eps), epsilon inside the root.
    const float inv_q = 1.f / sqrtf(sq / (float)a.Hcq + a.eps_cq);
    const float inv_kv = 1.f / sqrtf(skv / (float)a.Hckv + a.eps_ckv);

    __nv_bfloat16* cq = a.c_q + (size_t)t * a.Hcq;
    if (!a.cq_quant) {
#pragma unroll
        for (int k = 0; k < kWQ; ++k)
            if (k < nq) {
                const int c = 2 * lane + 64 * k;
                const __nv_bfloat162 g2 = *reinterpret_cast<const __nv_bfloat162*>(a.gamma_cq + c);
                *reinterpret_cast<__nv_bfloat162*>(cq + c) =
                    __floats2bfloat162_rn(__low2float(g2) * yq[k].x * inv_q, __high2float(g2) * yq[k].y * inv_q);
            }
    } else {
        // per-token dynamic int8 codes of c^Q (times the smooth scales when given)
        float m = 0.f;
#pragma unroll
        for (int k = 0; k < kWQ; ++k)
            if (k < nq) {
                const int c = 2 * lane + 64 * k;
                const __nv_bfloat162 g2 = *reinterpret_cast<const __nv_bfloat162*>(a.gamma_cq + c);
                float u0 = __low2float(g2) * yq[k].x * inv_q, u1 = __high2float(g2) * yq[k].y * inv_q;
                if (a.smooth_cq) {
                    u0 *= a.smooth_cq[c];
                    u1 *= a.smooth_cq[c + 1];
                }
                yq[k] = make_float2(u0, u1);
                m = fmaxf(m, fmaxf(fabsf(u0), fabsf(u1)));
            }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        const float scale = m / 127.f;
#pragma unroll
        for (int k = 0; k < kWQ; ++k)
            if (k < nq) {
                const int c = 2 * lane + 64 * k;
                const int q0 = scale > 0.f ? quant_i8(__fdiv_rn(yq[k].x, scale)) : 0;
                const int q1 = scale > 0.f ? quant_i8(__fdiv_rn(yq[k].y, scale)) : 0;
                // exact fp16 codes: the A operand of the int8-weight GEMM
                *reinterpret_cast<__half2*>(cq + c) = __halves2half2(__int2half_rn(q0), __int2half_rn(q1));
            }
        if (lane == 0) a.c_q_scale[t] = scale;
    }

    if (a.nslots <= 0) return;
    if (slot < 0 || slot >= a.nslots) {
        if (lane == 0) atomicOr(a.status, kStatusCacheIndexRange);
        return;
    }
    if (a.kv_int8) {
        int8_t* d = reinterpret_cast<int8_t*>(a.kv_cache) + slot * a.Hckv;
#pragma unroll
        for (int k = 0; k < kWKV; ++k)
            if (k < nkv) {
                const int c = 2 * lane + 64 * k;
                d[c] = (int8_t)quant_i8(__bfloat162float(a.gamma_ckv[c]) * ykv[k].x * inv_kv * a.quant_scale_ckv[c]);
                d[c + 1] = (int8_t)quant_i8(__bfloat162float(a.gamma_ckv[c + 1]) * ykv[k].y * inv_kv * a.quant_scale_ckv[c + 1]);
            }
    } else {
        __nv_bfloat16* d = reinterpret_cast<__nv_bfloat16*>(a.kv_cache) + slot * a.Hckv;
#pragma unroll
        for (int k = 0; k < kWKV; ++k)
            if (k < nkv) {
                const int c = 2 * lane + 64 * k;
                const __nv_bfloat162 g2 = *reinterpret_cast<const __nv_bfloat162*>(a.gamma_ckv + c);
                *reinterpret_cast<__nv_bfloat162*>(d + c) =
                    __floats2bfloat162_rn(__low2float(g2) * ykv[k].x * inv_kv, __high2float(g2) * ykv[k].y * inv_kv);
            }
    }
    // "half" RoPE of k^R: lane j holds the pair (j, j + Dr/2)
    const float o0 = kr0 * cos0 - kr1 * sin0;
    const float o1 = kr1 * cos1 + kr0 * sin1;
    if (a.kr_int8) {
        int8_t* d = reinterpret_cast<int8_t*>(a.kr_cache) + slot * a.Dr;
        d[lane] = (int8_t)quant_i8(o0 * a.quant_scale_ckr[lane]);
        d[lane + h] = (int8_t)quant_i8(o1 * a.quant_scale_ckr[lane + h]);
    } else {
        __nv_bfloat16* d = reinterpret_cast<__nv_bfloat16*>(a.kr_cache) + slot * a.Dr;
        d[lane] = __float2bfloat16_rn(o0);
        d[lane + h] = __float2bfloat16_rn(o1);
    }
}

struct UpArgs {
    int T, N, D, Dr;
    PartialSrc src;                     // T x N * (D + Dr)
    const float* row_scale;             // (T) dequant of int8 c^Q codes, or null
    const float* col_scale;             // (N*(D+Dr)) dequant of int8 weightUqQr, or null
    const __nv_bfloat16* rope_cos;
    const __nv_bfloat16* rope_sin;
    __nv_bfloat16* q_c;                 // (T, N, D)
    __nv_bfloat16* q_rope;              // (T, N, Dr)
};

__global__ void __launch_bounds__(kRowThreads) finalize_up_kernel(const UpArgs a) {
    pdl_launch_dependents();
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
}

// Exact int8 -> fp16 widening (|v| <= 128 has at most 8 significant bits), for the fp16 A operand
// of the int8-weight GEMM.
__global__ void __launch_bounds__(256) convert_i8_to_f16_kernel(const int8_t* __restrict__ src,
                                                                __half* __restrict__ dst, long long n) {
    pdl_launch_dependents();
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
                const __half2 h = __halves2half2(__int2half_rn(b0), __int2half_rn(b1));
                ow[2 * k + e] = *reinterpret_cast<const uint32_t*>(&h);
            }
        }
        reinterpret_cast<uint4*>(dst)[2 * i] = o[0];
        reinterpret_cast<uint4*>(dst)[2 * i + 1] = o[1];
    }
    for (long long i = n16 * 16 + (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
        dst[i] = __int2half_rn((int)src[i]);
}

}  // namespace mla
