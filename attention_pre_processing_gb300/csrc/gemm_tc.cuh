// Warp-specialised tcgen05 GEMM for the MLA prolog's three contractions.
//
//   D[rows, cols] = A[rows, K] . B[K, cols]
//   A: activations, K-major bf16 (x, c^Q, or q^C of one head), fetched by TMA, 128-byte swizzle.
//   B: weights in their (k, n) orientation (n contiguous), i.e. MN-major, fetched by TMA in
//      64-column boxes, 128-byte swizzle.
//   D: fp32 in tensor memory; MSUB sub-tiles of 128 rows, BN columns each.
//
// Roles (192 threads): warp 0 issues TMA loads into a STAGES-deep shared-memory ring, warp 1
// allocates tensor memory and issues tcgen05.mma, warps 2..5 drain the accumulator through
// tcgen05.ld and run the epilogue.  Every wait is bounded (kWaitLimitNs); a wait that gives up
// raises MLA_DEV_WAIT_TIMEOUT, the other roles stop at their next wait, tensor memory is freed
// and the kernel returns.
//
// Work: "tile" mode walks whole (row tile, column tile) pairs with the full K range.  "split"
// mode (few rows: decode) cuts the flattened (column tile, k-block) range into one contiguous
// piece per CTA, so that every SM streams the same number of weight bytes; a CTA's piece covers
// at most two column tiles and each part is written as an fp32 partial slot (2*cta + part).
// The finalize kernels add the slots of a tile in fixed CTA order (deterministic).
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"

namespace mla {

constexpr int kBK = 64;          // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr int kGemmThreads = 192;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

constexpr uint32_t kStatusCacheIndexRange = 0x1u;
constexpr uint32_t kStatusWaitTimeout = 0x2u;

enum Epi : int { EPI_F32 = 0, EPI_QROPE = 1, EPI_QN = 2 };

struct GemmArgs {
    int T;               // valid A rows
    int kblocks;         // ceil(K / 64)
    int ncols;           // valid product columns (EPI_QN: Hckv of one head)
    int n_tiles;         // column tiles (EPI_QN: N * tiles_per_head)
    int m_tiles;         // row tiles of MSUB*128 rows (tile mode)
    int split;           // 1: stream-K pieces with fp32 partial slots
    long long total;     // split: n_tiles * kblocks
    int b_split_col;     // B columns below this come from map b0, the rest from b1
    int head_mode;       // A and B are per-head 3D maps (W^UK contraction)
    int tiles_per_head;  // EPI_QN
    int clear_status;    // block 0 zeroes *status once earlier grids have finished
    // EPI_F32
    float* out_f32;      // split: slots of T x BN; tile: T x ncols
    // EPI_QROPE (one head of D=128 nope + Dr=64 rope columns per tile)
    int N;
    __nv_bfloat16* q_c;            // (T, N, 128)
    __nv_bfloat16* q_rope;         // (T, N, 64)
    const __nv_bfloat16* rope_cos; // (T, 64)
    const __nv_bfloat16* rope_sin; // (T, 64)
    const float* row_scale;        // optional (T): per-token dequant
    const float* col_scale;        // optional (ncols): per-column dequant
    // EPI_QN
    int Hckv;
    __nv_bfloat16* q_out_bf16;     // (T, N, Hckv)
    int8_t* q_out_i8;              // (T, N, Hckv)
    float* q_scale;                // (T, N)
    uint32_t* status;
};

template <int BN, int MSUB, int STAGES>
struct GemmCfg {
    static constexpr int kASub = 128 * kBK * 2;             // one 128-row A sub-tile: 16 KB
    static constexpr int kAStage = MSUB * kASub;
    static constexpr int kBStage = BN * kBK * 2;            // BN/64 boxes of 64 x 64
    static constexpr int kStageBytes = kAStage + kBStage;
    static constexpr int kAcc = MSUB * BN;                  // TMEM columns per accumulator set
    static constexpr int kNBuf = (2 * kAcc <= 512) ? 2 : 1;
    static constexpr int kTmemCols = (kNBuf * kAcc <= 32) ? 32 : (kNBuf * kAcc <= 64) ? 64
                                     : (kNBuf * kAcc <= 128) ? 128 : (kNBuf * kAcc <= 256) ? 256 : 512;
    static constexpr int kNParts = BN > 256 ? 2 : 1;        // MMA N <= 256
    static constexpr int kMmaN = BN / kNParts;
    static constexpr int kBarBytes = 8 * (2 * STAGES + 2 * 2 + 1) + 16;
    static constexpr size_t kSmem = 1024 + (size_t)STAGES * kStageBytes + kBarBytes;
    static_assert(BN % 64 == 0, "BN must be a multiple of 64");
    static_assert(kMmaN % 16 == 0 && kMmaN <= 256, "bad MMA N");
    static_assert(kAcc <= 512, "accumulator exceeds TMEM");
};

struct Unit {
    int m_tile, n_tile, kb0, kb1, slot;
};

// The idx-th unit of work of this CTA.
__device__ __forceinline__ bool get_unit(const GemmArgs& a, int idx, Unit& u) {
    if (a.split) {
        const long long G = gridDim.x;
        const long long lo = (long long)blockIdx.x * a.total / G;
        const long long hi = ((long long)blockIdx.x + 1) * a.total / G;
        if (lo >= hi || idx > 1) return false;
        const int KB = a.kblocks;
        const int t0 = (int)(lo / KB);
        if (idx == 0) {
            u.m_tile = 0;
            u.n_tile = t0;
            u.kb0 = (int)(lo - (long long)t0 * KB);
            long long e = hi - (long long)t0 * KB;
            u.kb1 = (int)(e < KB ? e : KB);
            u.slot = 2 * blockIdx.x;
            return true;
        }
        if (hi <= (long long)(t0 + 1) * KB) return false;
        u.m_tile = 0;
        u.n_tile = t0 + 1;
        u.kb0 = 0;
        u.kb1 = (int)(hi - (long long)(t0 + 1) * KB);
        u.slot = 2 * blockIdx.x + 1;
        return true;
    }
    const long long i = (long long)blockIdx.x + (long long)idx * gridDim.x;
    if (i >= (long long)a.m_tiles * a.n_tiles) return false;
    u.m_tile = (int)(i % a.m_tiles);   // row tiles fastest: neighbouring CTAs share a weight tile
    u.n_tile = (int)(i / a.m_tiles);
    u.kb0 = 0;
    u.kb1 = a.kblocks;
    u.slot = 0;
    return true;
}

__device__ __forceinline__ float bits_f(uint32_t u) { return __uint_as_float(u); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Round half away from zero, saturate to [-127, 127].
__device__ __forceinline__ int quant_i8(float v) {
    float r = roundf(v);
    r = fminf(fmaxf(r, -127.f), 127.f);
    return (int)r;
}

// ------------------------------------------------------------------ epilogues

// fp32 store of one 32-column chunk of one row.
__device__ __forceinline__ void store_f32_chunk(float* dst, const uint32_t (&r)[32], int nvalid) {
    if (nvalid >= 32 && ((reinterpret_cast<uintptr_t>(dst) & 15) == 0)) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            reinterpret_cast<uint4*>(dst)[i] = make_uint4(r[4 * i], r[4 * i + 1], r[4 * i + 2], r[4 * i + 3]);
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (i < nvalid) dst[i] = bits_f(r[i]);
    }
}

// bf16 store of one 32-column chunk (64 bytes) of one row.
__device__ __forceinline__ void store_bf16_chunk(__nv_bfloat16* dst, const float (&v)[32], int nvalid) {
    if (nvalid >= 32 && ((reinterpret_cast<uintptr_t>(dst) & 15) == 0)) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint4 w;
            w.x = pack_bf16(v[8 * i + 0], v[8 * i + 1]);
            w.y = pack_bf16(v[8 * i + 2], v[8 * i + 3]);
            w.z = pack_bf16(v[8 * i + 4], v[8 * i + 5]);
            w.w = pack_bf16(v[8 * i + 6], v[8 * i + 7]);
            reinterpret_cast<uint4*>(dst)[i] = w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (i < nvalid) dst[i] = __float2bfloat16_rn(v[i]);
    }
}

template <int BN, int MSUB>
__device__ __forceinline__ void epilogue_f32(const GemmArgs& a, const Unit& u, uint32_t tacc, int row_in) {
    float* base;
    long long ld;
    int col_limit;
    if (a.split) {
        base = a.out_f32 + (size_t)u.slot * (size_t)a.T * BN;
        ld = BN;
        col_limit = BN;
    } else {
        base = a.out_f32 + (size_t)u.n_tile * BN;
        ld = a.ncols;
        col_limit = a.ncols - u.n_tile * BN;
    }
#pragma unroll 1
    for (int ms = 0; ms < MSUB; ++ms) {
        const int row = (u.m_tile * MSUB + ms) * 128 + row_in;
#pragma unroll 1
        for (int ch = 0; ch < BN / 32; ++ch) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(tacc + ms * BN + ch * 32, r);
            tmem_ld_wait();
            if (row < a.T && ch * 32 < col_limit)
                store_f32_chunk(base + (size_t)row * ld + ch * 32, r, col_limit - ch * 32);
        }
    }
}

// One head per tile: columns [0,128) are q^C (nope), [128,192) the rope part of W^QR.
template <int MSUB>
__device__ __forceinline__ void epilogue_qrope(const GemmArgs& a, const Unit& u, uint32_t tacc, int row_in) {
    constexpr int D = 128, DR = 64, H = 32, BN = 192;
    const int head = u.n_tile;
#pragma unroll 1
    for (int ms = 0; ms < MSUB; ++ms) {
        const int row = (u.m_tile * MSUB + ms) * 128 + row_in;
        const bool valid = row < a.T;
        const float rs = (valid && a.row_scale) ? a.row_scale[row] : 1.f;
        const float* cs = a.col_scale ? a.col_scale + (size_t)head * BN : nullptr;
#pragma unroll 1
        for (int ch = 0; ch < D / 32; ++ch) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(tacc + ms * BN + ch * 32, r);
            tmem_ld_wait();
            if (valid) {
                float v[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    v[i] = bits_f(r[i]);
                    if (cs) v[i] *= rs * cs[ch * 32 + i];
                }
                store_bf16_chunk(a.q_c + ((size_t)row * a.N + head) * D + ch * 32, v, 32);
            }
        }
        uint32_t ra[32], rb[32];
        tmem_ld_32x32b_x32(tacc + ms * BN + D, ra);
        tmem_ld_32x32b_x32(tacc + ms * BN + D + H, rb);
        tmem_ld_wait();
        if (valid) {
            const uint4* cp = reinterpret_cast<const uint4*>(a.rope_cos + (size_t)row * DR);
            const uint4* sp = reinterpret_cast<const uint4*>(a.rope_sin + (size_t)row * DR);
            float o0[32], o1[32];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint4 c0 = cp[q], c1 = cp[q + 4], s0 = sp[q], s1 = sp[q + 4];
                const uint32_t cw0[4] = {c0.x, c0.y, c0.z, c0.w}, cw1[4] = {c1.x, c1.y, c1.z, c1.w};
                const uint32_t sw0[4] = {s0.x, s0.y, s0.z, s0.w}, sw1[4] = {s1.x, s1.y, s1.z, s1.w};
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int j = q * 8 + e;
                    const float cj = (e & 1) ? bf16_hi(cw0[e >> 1]) : bf16_lo(cw0[e >> 1]);
                    const float sj = (e & 1) ? bf16_hi(sw0[e >> 1]) : bf16_lo(sw0[e >> 1]);
                    const float ch = (e & 1) ? bf16_hi(cw1[e >> 1]) : bf16_lo(cw1[e >> 1]);
                    const float sh = (e & 1) ? bf16_hi(sw1[e >> 1]) : bf16_lo(sw1[e >> 1]);
                    float x0 = bits_f(ra[j]), x1 = bits_f(rb[j]);
                    if (cs) {
                        x0 *= rs * cs[D + j];
                        x1 *= rs * cs[D + H + j];
                    }
                    o0[j] = x0 * cj - x1 * sj;
                    o1[j] = x1 * ch + x0 * sh;
                }
            }
            __nv_bfloat16* dst = a.q_rope + ((size_t)row * a.N + head) * DR;
            store_bf16_chunk(dst, o0, 32);
            store_bf16_chunk(dst + H, o1, 32);
        }
    }
}

template <int BN>
__device__ __forceinline__ void epilogue_qn(const GemmArgs& a, const Unit& u, uint32_t tacc, int row_in) {
    const int head = u.n_tile / a.tiles_per_head;
    const int c0 = (u.n_tile % a.tiles_per_head) * BN;
    const int row = u.m_tile * 128 + row_in;
    const bool valid = row < a.T;
    const size_t rowoff = ((size_t)row * a.N + head) * a.Hckv;
    if (a.q_out_i8 == nullptr) {
#pragma unroll 1
        for (int ch = 0; ch < BN / 32; ++ch) {
            const int col = c0 + ch * 32;
            if (col >= a.Hckv) break;   // uniform across the warp
            uint32_t r[32];
            tmem_ld_32x32b_x32(tacc + ch * 32, r);
            tmem_ld_wait();
            if (valid) {
                float v[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = bits_f(r[i]);
                store_bf16_chunk(a.q_out_bf16 + rowoff + col, v, a.Hckv - col);
            }
        }
        return;
    }
    // Dynamic int8 quantisation of the whole (token, head) row: this thread owns the row.
    float m = 0.f;
#pragma unroll 1
    for (int ch = 0; ch < BN / 32; ++ch) {
        const int col = ch * 32;
        if (col >= a.Hckv) break;
        uint32_t r[32];
        tmem_ld_32x32b_x32(tacc + col, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (col + i < a.Hckv) m = fmaxf(m, fabsf(bits_f(r[i])));
    }
    const float scale = m / 127.f;
#pragma unroll 1
    for (int ch = 0; ch < BN / 32; ++ch) {
        const int col = ch * 32;
        if (col >= a.Hckv) break;
        uint32_t r[32];
        tmem_ld_32x32b_x32(tacc + col, r);
        tmem_ld_wait();
        if (valid) {
            uint32_t w[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                uint32_t packed = 0;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int q = (scale > 0.f) ? quant_i8(__fdiv_rn(bits_f(r[4 * i + e]), scale)) : 0;
                    packed |= ((uint32_t)(q & 0xFF)) << (8 * e);
                }
                w[i] = packed;
            }
            int8_t* dst = a.q_out_i8 + rowoff + col;
            const int nvalid = a.Hckv - col;
            if (nvalid >= 32 && ((reinterpret_cast<uintptr_t>(dst) & 15) == 0)) {
                reinterpret_cast<uint4*>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
                reinterpret_cast<uint4*>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
            } else {
                for (int i = 0; i < 32 && i < nvalid; ++i) dst[i] = (int8_t)((w[i >> 2] >> (8 * (i & 3))) & 0xFF);
            }
        }
    }
    if (valid) a.q_scale[(size_t)row * a.N + head] = scale;
}

// ---------------------------------------------------------------------- kernel

template <int BN, int MSUB, int STAGES, int EPI>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b0,
                   const __grid_constant__ CUtensorMap map_b1, const GemmArgs args) {
    using C = GemmCfg<BN, MSUB, STAGES>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + (size_t)STAGES * C::kAStage;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)STAGES * C::kStageBytes);
    uint64_t* full = bars;
    uint64_t* empty = bars + STAGES;
    uint64_t* tfull = bars + 2 * STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* done = tempty + 2;
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(done + 1);
    volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&map_a);
        tma_prefetch_map(&map_b0);
        tma_prefetch_map(&map_b1);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&tfull[b]), 1);
            mbar_init(smem_u32(&tempty[b]), 128);
        }
        mbar_init(smem_u32(done), 1);
        *s_abort = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(s_tmem), C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *s_tmem;

    // Everything above overlaps the previous grid; inputs are read only after it completes.
    pdl_wait();
    if (args.clear_status && blockIdx.x == 0 && threadIdx.x == 0) *args.status = 0u;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_a = policy_evict_last();
            uint32_t it = 0;
            Unit u;
            bool ok = true;
            for (int idx = 0; ok && get_unit(args, idx, u); ++idx) {
                int head = 0, c0 = 0;
                if (args.head_mode) {
                    head = u.n_tile / args.tiles_per_head;
                    c0 = (u.n_tile % args.tiles_per_head) * BN;
                } else {
                    c0 = u.n_tile * BN;
                }
                for (int kb = u.kb0; kb < u.kb1; ++kb, ++it) {
                    const int s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1;
                    if (!mbar_wait(smem_u32(&empty[s]), ph ^ 1, s_abort, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(&full[s]);
                    mbar_arrive_expect_tx(fb, C::kStageBytes);
                    const uint32_t a_dst = smem_u32(sA + (size_t)s * C::kAStage);
                    const uint32_t b_dst = smem_u32(sB + (size_t)s * C::kBStage);
#pragma unroll
                    for (int ms = 0; ms < MSUB; ++ms) {
                        const int r0 = (u.m_tile * MSUB + ms) * 128;
                        if (args.head_mode)
                            tma_load_3d(a_dst + ms * C::kASub, &map_a, fb, kb * kBK, head, r0, pol_a);
                        else
                            tma_load_2d(a_dst + ms * C::kASub, &map_a, fb, kb * kBK, r0, pol_a);
                    }
#pragma unroll
                    for (int j = 0; j < BN / 64; ++j) {
                        const int col = c0 + 64 * j;
                        const uint32_t dst = b_dst + j * (64 * kBK * 2);
                        if (args.head_mode)
                            tma_load_3d(dst, &map_b0, fb, col, kb * kBK, head, pol_w);
                        else if (col < args.b_split_col)
                            tma_load_2d(dst, &map_b0, fb, col, kb * kBK, pol_w);
                        else
                            tma_load_2d(dst, &map_b1, fb, col - args.b_split_col, kb * kBK, pol_w);
                    }
                }
            }
            if (!ok) {
                *s_abort = 1;
                atomicOr(args.status, kStatusWaitTimeout);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(128, C::kMmaN, false, true);
            uint32_t it = 0, ai = 0;
            Unit u;
            bool ok = true;
            for (int idx = 0; ok && get_unit(args, idx, u); ++idx, ++ai) {
                const int b = ai % C::kNBuf;
                const uint32_t aph = (ai / C::kNBuf) & 1;
                if (!mbar_wait(smem_u32(&tempty[b]), aph ^ 1, s_abort, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_base = tmem_base + b * C::kAcc;
                for (int kb = u.kb0; kb < u.kb1; ++kb, ++it) {
                    const int s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1;
                    if (!mbar_wait(smem_u32(&full[s]), ph, s_abort, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_base = smem_u32(sA + (size_t)s * C::kAStage);
                    const uint32_t b_base = smem_u32(sB + (size_t)s * C::kBStage);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
#pragma unroll
                        for (int ms = 0; ms < MSUB; ++ms) {
                            const uint64_t adesc = smem_desc_sw128(a_base + ms * C::kASub + kk * 32, 16, 1024);
#pragma unroll
                            for (int np = 0; np < C::kNParts; ++np) {
                                const uint64_t bdesc = smem_desc_sw128(
                                    b_base + np * (C::kMmaN / 64) * (64 * kBK * 2) + kk * 16 * 128, 64 * kBK * 2, 1024);
                                umma_bf16(d_base + ms * BN + np * C::kMmaN, adesc, bdesc, idesc,
                                          (kb > u.kb0 || kk > 0) ? 1u : 0u);
                            }
                        }
                    }
                    umma_commit(smem_u32(&empty[s]));
                }
                if (!ok) break;
                umma_commit(smem_u32(&tfull[b]));
            }
            if (!ok) {
                *s_abort = 1;
                atomicOr(args.status, kStatusWaitTimeout);
            }
            // Drain: every MMA issued above completes before tensor memory is freed.
            umma_commit(smem_u32(done));
            mbar_wait(smem_u32(done), 0, s_abort, kWaitLimitNs / 4);
        }
    } else {
        // ------------------------------------------------------------ epilogue warps
        const int q = warp & 3;   // TMEM lane quarter this warp may access
        const int row_in = q * 32 + lane;
        uint32_t ai = 0;
        Unit u;
        for (int idx = 0; get_unit(args, idx, u); ++idx, ++ai) {
            const int b = ai % C::kNBuf;
            const uint32_t aph = (ai / C::kNBuf) & 1;
            int ok = 1;
            if (lane == 0) ok = mbar_wait(smem_u32(&tfull[b]), aph, s_abort, kWaitLimitNs) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) {
                    *s_abort = 1;
                    atomicOr(args.status, kStatusWaitTimeout);
                }
                break;
            }
            __syncwarp();
            tc_fence_after();
            const uint32_t tacc = tmem_base + ((uint32_t)(q * 32) << 16) + b * C::kAcc;
            if constexpr (EPI == EPI_F32) {
                epilogue_f32<BN, MSUB>(args, u, tacc, row_in);
            } else if constexpr (EPI == EPI_QROPE) {
                epilogue_qrope<MSUB>(args, u, tacc, row_in);
            } else {
                epilogue_qn<BN>(args, u, tacc, row_in);
            }
            tc_fence_before();
            mbar_arrive(smem_u32(&tempty[b]));
        }
    }

    // Let the next grid start its prologue while this one tears down.
    pdl_launch_dependents();
    tc_fence_before();
    __syncthreads();
    if (*s_abort) {
        // A wait gave up: give copies that may still be in flight time to land.
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < 20000000ull) {
        }
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::kTmemCols);
    }
}

}  // namespace mla
