// Warp-specialised tcgen05 GEMM for the MLA prolog's three contractions.
//
//   D[rows, cols] = A[rows, K] . B[K, cols]
//   A: activations, K-major bf16 (x, c^Q, or q^C of one head), fetched by TMA, 128-byte swizzle.
//      The A box has a_box_rows rows (T rounded up to 8 when T <= 128): rows past it in the
//      128-row MMA operand hold stale shared memory and only feed accumulator rows >= T,
//      which are never stored.
//   B: weights in their (k, n) orientation (n contiguous), i.e. MN-major, fetched by TMA in
//      64-column boxes, 128-byte swizzle.
//   D: fp32 in tensor memory; MSUB sub-tiles of 128 rows, BN columns each.
//
// Roles (192 threads): warp 0 issues TMA loads into a `stages`-deep shared-memory ring, warp 1
// allocates tensor memory and issues tcgen05.mma, warps 2..5 drain the accumulator with
// tcgen05.ld and run the epilogue.  Every wait is bounded (kWaitLimitNs); a wait that gives up
// raises MLA_DEV_WAIT_TIMEOUT, the other roles stop at their next wait, tensor memory is freed
// and the kernel returns.
//
// Work: units are (row tile, column tile, k range).  With ksplit = S > 1 (decode-sized T) the
// K dimension is cut into S equal ranges and each unit's fp32 product goes to its own slot of a
// S x T x ncols buffer, which the row-wise finalize kernel adds in fixed order (deterministic).
// All CTAs start together and walk K in the same order, so CTAs of one k range read the same
// weight rows at the same time (DRAM page locality).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "ptx.cuh"

namespace mla {

constexpr int kBK = 64;          // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr int kGemmThreads = 192;   // with one epilogue warp per TMEM lane quarter
// Threads of a GEMM CTA with EPW epilogue warps per TMEM lane quarter.
__host__ __device__ constexpr int gemm_threads(int epw) { return 64 + 128 * epw; }
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr size_t kSmemLimit = 232448;             // 227 KB opt-in per CTA

constexpr uint32_t kStatusCacheIndexRange = 0x1u;
constexpr uint32_t kStatusWaitTimeout = 0x2u;

enum Epi : int { EPI_F32 = 0, EPI_QROPE = 1, EPI_QN = 2, EPI_DOWN = 3 };

struct GemmArgs {
    int T;               // valid A rows
    int kblocks;         // ceil(K / 64)
    int ncols;           // valid product columns (EPI_QN: Hckv of one head)
    int n_tiles;         // column tiles (EPI_QN: N * tiles_per_head)
    int m_tiles;         // row tiles of MSUB*128 rows
    int ksplit;          // k ranges (EPI_F32 only): unit products go to slot k_range
    int b_split_col;     // B columns below this come from map b0, the rest from b1
    int head_mode;       // A and B are per-head 3D maps (W^UK contraction)
    int tiles_per_head;  // EPI_QN
    int clear_status;    // block 0 zeroes *status once earlier grids have finished
    int a_ready;         // A is a caller input (not written by an earlier kernel of the call):
                         // its tiles may be requested before the grid dependency resolves
    int b_late;          // B is written by an earlier kernel of the call (a widened int8 weight):
                         // no weight tile is requested before the grid dependency resolves
    int a_box_rows;      // rows of one A TMA box (multiple of 8, <= 128)
    int stages;          // ring depth actually used (<= MAXST)
    // EPI_F32: ksplit slots of T x ncols row-major fp32
    float* out_f32;
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
    __nv_bfloat16* q_out_bf16;     // (T, N, q_ld), the first Hckv of each q_ld written (16-bit output)
    int q_ld;                      // elements from one head's row to the next (0: Hckv)
    int f16;                       // A, B and the 16-bit output are fp16 instead of bf16
    int8_t* q_out_i8;              // (T, N, Hckv)
    float* q_scale;                // (T, N)
    int tma_out;                   // store the output through shared memory with TMA (map_o, map_o2)
    int a_one_box;                 // one A box spans all MSUB x 128 rows (map_a box height MSUB*128)
    int b_blocks;                  // the B maps are 3D (64 columns, k, 64-column blocks): one box
                                   // brings all BN/64 column blocks of a k-block; in head_mode the
                                   // k rows of head n start at n * head_rows
    int head_rows;                 // head_mode with b_blocks: weight rows per head (D)
    int n_fastest;                 // pair tiles: column tile fastest (the row tiles of A then come
                                   // from HBM once, shared by the pairs of all column tiles)
    // EPI_DOWN (prefill down-projection): columns below cq_cols leave as bf16(gamma_cq * y)
    // through map_o2 with each row's sum of y^2 per (tile, epilogue part) in ss_out; the rest
    // as fp32 through map_o
    int cq_cols;
    const __nv_bfloat16* gamma_cq;
    float* ss_out;                 // T x nss
    int nss;                       // sums per row
    // EPI_QROPE with ss_in: the RmsNorm scale 1 / sqrt(sum(ss_in[row]) / hcq + eps_cq) of each
    // row multiplies the product (c^Q reaches the up-projection as bf16(gamma_cq * y))
    const float* ss_in;            // T x nss
    int hcq;
    float eps_cq;
    uint32_t* status;
};

// OUTB: 4 KB staging buffers per epilogue warp for TMA stores of the output (0 = none).
// KPS: k-blocks per pipeline stage.  With KPS = 2 a weight box spans 128 k rows (16 KB): the
// TMA engine moves far more bytes per box request from L2 than with 64-row boxes.
template <int BN, int MSUB, int MAXST, int OUTB = 0, int KPS = 1, int EPW = 1>
struct GemmCfg {
    static constexpr int kOutBytes = 4 * EPW * OUTB * 4096;
    // split epilogues that need a whole row (EPI_QN int8): two 128-row x EPW partial maxima
    static constexpr int kXBytes = EPW > 1 ? 2 * 128 * EPW * 4 : 0;
    static constexpr int kBStage = BN * kBK * 2 * KPS;      // BN/64 boxes of 64 cols x 64*KPS rows
    static constexpr int kAcc = MSUB * BN;                  // TMEM columns per accumulator set
    static constexpr int kNBuf = (2 * kAcc <= 512) ? 2 : 1;
    static constexpr int kTmemCols = (kNBuf * kAcc <= 32) ? 32 : (kNBuf * kAcc <= 64) ? 64
                                     : (kNBuf * kAcc <= 128) ? 128 : (kNBuf * kAcc <= 256) ? 256 : 512;
    static constexpr int kNParts = BN > 256 ? 2 : 1;        // MMA N <= 256
    static constexpr int kMmaN = BN / kNParts;
    static constexpr int kBarBytes = 1024;                  // mbarriers + flags, first in smem
    static_assert(8 * (2 * MAXST + 5) + 16 <= kBarBytes, "barrier area");
    static_assert(BN % 64 == 0, "BN must be a multiple of 64");
    static_assert(kMmaN % 16 == 0 && kMmaN <= 256, "bad MMA N");
    static_assert(kAcc <= 512, "accumulator exceeds TMEM");

    static __host__ __device__ int a_stage_bytes(int a_box_rows) { return KPS * MSUB * a_box_rows * 128; }
    static __host__ __device__ int stage_bytes(int a_box_rows) { return a_stage_bytes(a_box_rows) + kBStage; }
    // A region first: a 128-row MMA operand read from the last A stage with a short box runs
    // at most 16 KB past it, into the B ring (>= 2 stages of >= 8 KB), inside the block.
    static __host__ __device__ size_t smem_bytes(int stages, int a_box_rows) {
        return 1024 + kBarBytes + (size_t)stages * stage_bytes(a_box_rows) + kOutBytes + kXBytes;
    }
    static __host__ int max_stages(int a_box_rows) {
        int s = (int)((kSmemLimit - 1024 - kBarBytes - kOutBytes - kXBytes) / stage_bytes(a_box_rows));
        return s < MAXST ? s : MAXST;
    }
    static_assert(2 * kBStage >= 16384, "B ring must cover the A over-read");
};

struct Unit {
    int m_tile, n_tile, kb0, kb1, ks;
};

// The idx-th unit of work of this CTA: k range slowest, row tile fastest (neighbouring CTAs
// share a weight tile; CTAs of one k range stream the same weight rows).
__device__ __forceinline__ bool get_unit(const GemmArgs& a, int idx, Unit& u) {
    const long long i = (long long)blockIdx.x + (long long)idx * gridDim.x;
    const long long per_k = (long long)a.m_tiles * a.n_tiles;
    if (i >= per_k * a.ksplit) return false;
    u.ks = (int)(i / per_k);
    const long long r = i - (long long)u.ks * per_k;
    u.m_tile = (int)(r % a.m_tiles);
    u.n_tile = (int)(r / a.m_tiles);
    u.kb0 = (int)((long long)u.ks * a.kblocks / a.ksplit);
    u.kb1 = (int)((long long)(u.ks + 1) * a.kblocks / a.ksplit);
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

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
// The same over the NT epilogue threads of a CTA with more than four epilogue warps.
template <int NT>
__device__ __forceinline__ void epi_bar_n() { asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory"); }
template <int NT>
__device__ __forceinline__ bool epi_any_n(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(v ? 1u : 0u), "n"(NT)
        : "memory");
    return r != 0;
}

// Barrier over the 128 epilogue threads that also ORs a flag: every thread gets the same answer.
__device__ __forceinline__ bool epi_any(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(v ? 1u : 0u)
        : "memory");
    return r != 0;
}

// ----------------------------------------------------------- accumulator sources

// Rows of the accumulator, 32 columns at a time, straight from tensor memory (warp-collective).
struct TmemSrc {
    uint32_t tacc;
    __device__ __forceinline__ void load(int ms, int bn, int col, float (&v)[32]) const {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tacc + ms * bn + col, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = bits_f(r[i]);
    }
    // 128 consecutive columns: four loads in flight, one wait
    __device__ __forceinline__ void load128(int col, uint32_t (&r)[4][32]) const {
#pragma unroll
        for (int h = 0; h < 4; ++h) tmem_ld_32x32b_x32(tacc + col + 32 * h, r[h]);
        tmem_ld_wait();
    }
};

// ------------------------------------------------------------------ epilogues

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

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// 32 values -> fp16 (round to nearest even), as store_bf16_chunk.
__device__ __forceinline__ void store_f16_chunk(__nv_bfloat16* dst_bits, const float (&v)[32], int nvalid) {
    __half* dst = reinterpret_cast<__half*>(dst_bits);
    if (nvalid >= 32 && ((reinterpret_cast<uintptr_t>(dst) & 15) == 0)) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint4 w;
            w.x = pack_f16(v[8 * i + 0], v[8 * i + 1]);
            w.y = pack_f16(v[8 * i + 2], v[8 * i + 3]);
            w.z = pack_f16(v[8 * i + 4], v[8 * i + 5]);
            w.w = pack_f16(v[8 * i + 6], v[8 * i + 7]);
            reinterpret_cast<uint4*>(dst)[i] = w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (i < nvalid) dst[i] = __float2half_rn(v[i]);
    }
}

__device__ __forceinline__ void store_f32_chunk(float* dst, const float (&v)[32], int nvalid) {
    if (nvalid >= 32 && ((reinterpret_cast<uintptr_t>(dst) & 15) == 0)) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            reinterpret_cast<float4*>(dst)[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (i < nvalid) dst[i] = v[i];
    }
}

// fp32 rows of the product into slot ks of the ksplit x T x ncols buffer.
template <int BN, int MSUB, class Src>
__device__ __forceinline__ void epilogue_f32(const GemmArgs& a, int row0, int n_tile, int ks, const Src& src) {
    const int col_limit = a.ncols - n_tile * BN;
    float* out = a.out_f32 + (size_t)ks * a.T * a.ncols;
#pragma unroll 1
    for (int ms = 0; ms < MSUB; ++ms) {
        const int row = row0 + ms * 128;
#pragma unroll 1
        for (int ch = 0; ch < BN / 32; ++ch) {
            if (ch * 32 >= col_limit) break;   // uniform across the warp
            float v[32];
            src.load(ms, BN, ch * 32, v);
            if (row < a.T) store_f32_chunk(out + (size_t)row * a.ncols + n_tile * BN + ch * 32, v,
                                           col_limit - ch * 32);
        }
    }
}

// One head per tile: columns [0,128) are q^C (nope), [128,192) the rope part of W^QR.
template <int MSUB, class Src>
__device__ __forceinline__ void epilogue_qrope(const GemmArgs& a, int row0, int head, const Src& src) {
    constexpr int D = 128, DR = 64, H = 32, BN = 192;
#pragma unroll 1
    for (int ms = 0; ms < MSUB; ++ms) {
        const int row = row0 + ms * 128;
        const bool valid = row < a.T;
        const float rs = (valid && a.row_scale) ? a.row_scale[row] : 1.f;
        const float* cs = a.col_scale ? a.col_scale + (size_t)head * BN : nullptr;
#pragma unroll 1
        for (int ch = 0; ch < D / 32; ++ch) {
            float v[32];
            src.load(ms, BN, ch * 32, v);
            if (valid) {
                if (cs) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] *= rs * cs[ch * 32 + i];
                }
                store_bf16_chunk(a.q_c + ((size_t)row * a.N + head) * D + ch * 32, v, 32);
            }
        }
        float x0[32], x1[32];
        src.load(ms, BN, D, x0);
        src.load(ms, BN, D + H, x1);
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
                    float a0 = x0[j], a1 = x1[j];
                    if (cs) {
                        a0 *= rs * cs[D + j];
                        a1 *= rs * cs[D + H + j];
                    }
                    o0[j] = a0 * cj - a1 * sj;
                    o1[j] = a1 * ch + a0 * sh;
                }
            }
            __nv_bfloat16* dst = a.q_rope + ((size_t)row * a.N + head) * DR;
            store_bf16_chunk(dst, o0, 32);
            store_bf16_chunk(dst + H, o1, 32);
        }
    }
}

template <int BN>
__device__ __forceinline__ void epilogue_qn(const GemmArgs& a, const Unit& u, const TmemSrc& src, int row_in) {
    const int head = u.n_tile / a.tiles_per_head;
    const int c0 = (u.n_tile % a.tiles_per_head) * BN;
    const int row = u.m_tile * 128 + row_in;
    const bool valid = row < a.T;
    const size_t rowoff = ((size_t)row * a.N + head) * (a.q_ld > 0 ? a.q_ld : a.Hckv);
    if (a.q_out_i8 == nullptr) {
#pragma unroll 1
        for (int ch = 0; ch < BN / 32; ++ch) {
            const int col = c0 + ch * 32;
            if (col >= a.Hckv) break;   // uniform across the warp
            float v[32];
            src.load(0, BN, ch * 32, v);
            if (valid) {
                if (a.f16)
                    store_f16_chunk(a.q_out_bf16 + rowoff + col, v, a.Hckv - col);
                else
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
        float v[32];
        src.load(0, BN, col, v);
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (col + i < a.Hckv) m = fmaxf(m, fabsf(v[i]));
    }
    const float scale = m / 127.f;
#pragma unroll 1
    for (int ch = 0; ch < BN / 32; ++ch) {
        const int col = ch * 32;
        if (col >= a.Hckv) break;
        float v[32];
        src.load(0, BN, col, v);
        if (valid) {
            uint32_t w[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                uint32_t packed = 0;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int q = (scale > 0.f) ? quant_i8(__fdiv_rn(v[4 * i + e], scale)) : 0;
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

// q^N of one tile through shared memory and TMA stores.  Each epilogue warp turns its 32 rows,
// one 128-byte column chunk at a time, into a 32 x 128-byte box in the 128-byte-swizzled
// layout (16-byte chunk c of row r at (c ^ (r % 8)) * 16), then one lane stores the box with
// TMA; rows at or past T fall outside the tensor map and are not written.  `obuf` holds the
// warp's OUTB staging buffers, `ob` the next one to use.
template <int OUTB>
struct OutStage {
    uint8_t* obuf;
    int ob;
    const CUtensorMap* map;
    int lane;
    __device__ __forceinline__ void put(const uint32_t (&w)[32], int x, int y) { put(w, x, y, map); }
    __device__ __forceinline__ void put(const uint32_t (&w)[32], int x, int y, const CUtensorMap* m) {
        const uint32_t buf = smem_u32(obuf + ob * 4096);
        if (lane == 0) bulk_wait_read<OUTB - 1>();   // the store that last read this buffer
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 8; ++c)
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                             buf + (uint32_t)(lane * 128 + ((c ^ (lane & 7)) << 4))),
                         "r"(w[4 * c]), "r"(w[4 * c + 1]), "r"(w[4 * c + 2]), "r"(w[4 * c + 3])
                         : "memory");
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(m, buf, x, y);
            bulk_commit();
        }
        ob = (ob + 1 == OUTB) ? 0 : ob + 1;
    }
    // The last stores have read their shared memory (the CTA may exit: the grid completes only
    // once its bulk stores have landed, before any dependent grid reads them).
    __device__ __forceinline__ void drain() const {
        if (lane == 0) bulk_wait_read<0>();
        __syncwarp();
    }
};

// fp32 product rows (EPI_F32) through shared memory and TMA stores: 32-row x 32-column (128-byte)
// boxes of the T x ncols matrix; rows and columns past its extent are not written.  With k ranges
// the map spans the ksplit slots (ksplit * T rows) and slot ks starts at row ks * T: T must then be
// a multiple of 32, so that no box crosses into the next slot.
template <int BN, int MSUB, int OUTB, int EPW = 1>
__device__ __forceinline__ void epilogue_f32_tma(const GemmArgs& a, const Unit& u, const TmemSrc& src, int q,
                                                 OutStage<OUTB>& out, int part = 0) {
#pragma unroll 1
    for (int ms = 0; ms < MSUB; ++ms) {
        const int row0 = u.m_tile * MSUB * 128 + ms * 128 + q * 32;
        if (row0 >= a.T) continue;   // warp-uniform
#pragma unroll 1
        for (int ch = part; ch < BN / 32; ch += EPW) {   // this warp's share of the columns
            const int col = u.n_tile * BN + ch * 32;
            if (col >= a.ncols) break;
            uint32_t w[32];
            tmem_ld_32x32b_x32(src.tacc + ms * BN + ch * 32, w);
            tmem_ld_wait();
            out.put(w, col, u.ks * a.T + row0);
        }
    }
}

// Prefill down-projection (EPI_DOWN): a tile of c^Q columns leaves as bf16(gamma_cq * y)
// through map_c in 64-column blocks, and each row's sum of y^2 over this warp's blocks goes to
// ss_out[row][tile * EPW + part]; a tile of c^KV | k^R columns leaves as fp32 through map_f (the
// row pass reads those).  A tile never straddles cq_cols.
template <int BN, int OUTB, int EPW>
__device__ __forceinline__ void epilogue_down_tma(const GemmArgs& a, const Unit& u, const TmemSrc& src, int q,
                                                  OutStage<OUTB>& out, const CUtensorMap* map_f,
                                                  const CUtensorMap* map_c, int part) {
    const int row0 = u.m_tile * 128 + q * 32;
    if (row0 >= a.T) return;   // warp-uniform
    const int c0 = u.n_tile * BN;
    if (c0 >= a.cq_cols) {
        epilogue_f32_tma<BN, 1, OUTB, EPW>(a, u, src, q, out, part);
        return;
    }
    const int row = row0 + out.lane;
    float s2 = 0.f;
#pragma unroll 1
    for (int blk = part; blk < BN / 64; blk += EPW) {
        const int col = c0 + 64 * blk;
        float v0[32], v1[32];
        src.load(0, BN, 64 * blk, v0);
        src.load(0, BN, 64 * blk + 32, v1);
        uint32_t w[32];
        const uint4* gp = reinterpret_cast<const uint4*>(a.gamma_cq + col);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const float* v = h ? v1 : v0;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint4 g = __ldg(gp + 4 * h + k);
                const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float x0 = v[8 * k + 2 * e], x1 = v[8 * k + 2 * e + 1];
                    s2 += x0 * x0 + x1 * x1;
                    w[16 * h + 4 * k + e] = pack_bf16(bf16_lo(gw[e]) * x0, bf16_hi(gw[e]) * x1);
                }
            }
        }
        out.put(w, col, row0, map_c);
    }
    if (row < a.T) a.ss_out[(size_t)row * a.nss + u.n_tile * EPW + part] = s2;
}

// One head per tile (EPI_QROPE, no dequant scales): q^C (128 columns) and RoPE(q^R) (64
// columns) through shared memory and TMA stores into the (T, N*128) and (T, N*64) views.
template <int MSUB, int OUTB>
__device__ __forceinline__ void epilogue_qrope_tma(const GemmArgs& a, const Unit& u, const TmemSrc& src, int q,
                                                   OutStage<OUTB>& out, const CUtensorMap* map_c,
                                                   const CUtensorMap* map_r) {
    constexpr int BN = 192, D = 128, DR = 64, H = 32;
    const int head = u.n_tile;
#pragma unroll 1
    for (int ms = 0; ms < MSUB; ++ms) {
        const int row0 = u.m_tile * MSUB * 128 + ms * 128 + q * 32;
        if (row0 >= a.T) continue;   // warp-uniform
        const int row = row0 + out.lane;
        const bool valid = row < a.T;
        // this row's RoPE tables, requested before the tensor-memory reads
        uint4 c4[8], s4[8];
        const uint4* cp = reinterpret_cast<const uint4*>(a.rope_cos + (size_t)(valid ? row : 0) * DR);
        const uint4* sp = reinterpret_cast<const uint4*>(a.rope_sin + (size_t)(valid ? row : 0) * DR);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            c4[i] = __ldg(cp + i);
            s4[i] = __ldg(sp + i);
        }
#pragma unroll 1
        for (int j = 0; j < D / 64; ++j) {
            uint32_t w[32];
            float v[32];
            src.load(ms, BN, 64 * j, v);
#pragma unroll
            for (int i = 0; i < 16; ++i) w[i] = pack_bf16(v[2 * i], v[2 * i + 1]);
            src.load(ms, BN, 64 * j + 32, v);
#pragma unroll
            for (int i = 0; i < 16; ++i) w[16 + i] = pack_bf16(v[2 * i], v[2 * i + 1]);
            out.put(w, head * D + 64 * j, row0, map_c);
        }
        float x0[32], x1[32];
        src.load(ms, BN, D, x0);
        src.load(ms, BN, D + H, x1);
        uint32_t w[32];
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
            const uint32_t cw0[4] = {c4[qq].x, c4[qq].y, c4[qq].z, c4[qq].w};
            const uint32_t cw1[4] = {c4[qq + 4].x, c4[qq + 4].y, c4[qq + 4].z, c4[qq + 4].w};
            const uint32_t sw0[4] = {s4[qq].x, s4[qq].y, s4[qq].z, s4[qq].w};
            const uint32_t sw1[4] = {s4[qq + 4].x, s4[qq + 4].y, s4[qq + 4].z, s4[qq + 4].w};
            float o0[8], o1[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int jj = qq * 8 + e;
                const float cj = (e & 1) ? bf16_hi(cw0[e >> 1]) : bf16_lo(cw0[e >> 1]);
                const float sj = (e & 1) ? bf16_hi(sw0[e >> 1]) : bf16_lo(sw0[e >> 1]);
                const float ch = (e & 1) ? bf16_hi(cw1[e >> 1]) : bf16_lo(cw1[e >> 1]);
                const float sh = (e & 1) ? bf16_hi(sw1[e >> 1]) : bf16_lo(sw1[e >> 1]);
                o0[e] = x0[jj] * cj - x1[jj] * sj;
                o1[e] = x1[jj] * ch + x0[jj] * sh;
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                w[qq * 4 + e] = pack_bf16(o0[2 * e], o0[2 * e + 1]);
                w[16 + qq * 4 + e] = pack_bf16(o1[2 * e], o1[2 * e + 1]);
            }
        }
        out.put(w, head * DR, row0, map_r);
    }
}

// Up-projection tiles of BN columns that need not align with heads (D = 128, Dr = 64): the
// 192 columns of head h are three 64-column blocks, the first two q^C, the third W^QR, so every
// 64-column block of a tile is wholly q^C or wholly rope, and the RoPE pairs (j, j + 32) of a
// rope block lie in the same block.  Each block goes through shared memory and a TMA store into
// the (T, N*128) or (T, N*64) view.
template <int BN, int MSUB, int OUTB, int EPW = 1>
__device__ __forceinline__ void epilogue_qrope_blocks_tma(const GemmArgs& a, const Unit& u, const TmemSrc& src,
                                                          int q, OutStage<OUTB>& out, const CUtensorMap* map_c,
                                                          const CUtensorMap* map_r, int part = 0) {
    constexpr int DR = 64;
#pragma unroll 1
    for (int ms = 0; ms < MSUB; ++ms) {
        const int row0 = u.m_tile * MSUB * 128 + ms * 128 + q * 32;
        if (row0 >= a.T) continue;   // warp-uniform
        const int row = row0 + out.lane;
        const bool valid = row < a.T;
        float inv = 1.f;
        if (a.ss_in != nullptr && valid) {
            float s2 = 0.f;
            for (int k = 0; k < a.nss; ++k) s2 += a.ss_in[(size_t)row * a.nss + k];
            inv = 1.f / sqrtf(s2 / (float)a.hcq + a.eps_cq);
        }
#pragma unroll 1
        for (int blk = part; blk < BN / 64; blk += EPW) {   // this warp's share of the blocks
            const int b = (u.n_tile * BN) / 64 + blk;   // global 64-column block
            if (b * 64 >= a.ncols) break;               // uniform across the warp
            const int head = b / 3, part = b % 3;
            float v0[32], v1[32];
            src.load(ms, BN, 64 * blk, v0);
            src.load(ms, BN, 64 * blk + 32, v1);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                v0[i] *= inv;
                v1[i] *= inv;
            }
            uint32_t w[32];
            if (part < 2) {
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    w[i] = pack_bf16(v0[2 * i], v0[2 * i + 1]);
                    w[16 + i] = pack_bf16(v1[2 * i], v1[2 * i + 1]);
                }
                out.put(w, head * 128 + part * 64, row0, map_c);
            } else {
                const uint4* cp = reinterpret_cast<const uint4*>(a.rope_cos + (size_t)(valid ? row : 0) * DR);
                const uint4* sp = reinterpret_cast<const uint4*>(a.rope_sin + (size_t)(valid ? row : 0) * DR);
#pragma unroll
                for (int qq = 0; qq < 4; ++qq) {
                    const uint4 c0 = __ldg(cp + qq), c1 = __ldg(cp + qq + 4), s0 = __ldg(sp + qq), s1 = __ldg(sp + qq + 4);
                    const uint32_t cw0[4] = {c0.x, c0.y, c0.z, c0.w}, cw1[4] = {c1.x, c1.y, c1.z, c1.w};
                    const uint32_t sw0[4] = {s0.x, s0.y, s0.z, s0.w}, sw1[4] = {s1.x, s1.y, s1.z, s1.w};
                    float o0[8], o1[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int jj = qq * 8 + e;
                        const float cj = (e & 1) ? bf16_hi(cw0[e >> 1]) : bf16_lo(cw0[e >> 1]);
                        const float sj = (e & 1) ? bf16_hi(sw0[e >> 1]) : bf16_lo(sw0[e >> 1]);
                        const float ch = (e & 1) ? bf16_hi(cw1[e >> 1]) : bf16_lo(cw1[e >> 1]);
                        const float sh = (e & 1) ? bf16_hi(sw1[e >> 1]) : bf16_lo(sw1[e >> 1]);
                        o0[e] = v0[jj] * cj - v1[jj] * sj;
                        o1[e] = v1[jj] * ch + v0[jj] * sh;
                    }
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        w[qq * 4 + e] = pack_bf16(o0[2 * e], o0[2 * e + 1]);
                        w[16 + qq * 4 + e] = pack_bf16(o1[2 * e], o1[2 * e + 1]);
                    }
                }
                out.put(w, head * DR, row0, map_r);
            }
        }
    }
}

template <int BN, int OUTB>
__device__ __forceinline__ void epilogue_qn_tma(const GemmArgs& a, const Unit& u, const TmemSrc& src, int q,
                                                OutStage<OUTB>& out) {
    const int head = u.n_tile / a.tiles_per_head;
    const int c0 = (u.n_tile % a.tiles_per_head) * BN;
    const int row0 = u.m_tile * 128 + q * 32;   // this warp's first row
    const int row = row0 + out.lane;
    if (row0 >= a.T) return;                     // warp-uniform: no valid row here
    if (a.q_out_i8 == nullptr) {
#pragma unroll 1
        for (int j = 0; j < BN / 64; ++j) {
            const int col = c0 + 64 * j;
            if (col >= a.Hckv) break;   // uniform across the warp
            uint32_t w[32];
            float v[32];
            src.load(0, BN, 64 * j, v);
            if (a.f16) {
#pragma unroll
                for (int i = 0; i < 16; ++i) w[i] = pack_f16(v[2 * i], v[2 * i + 1]);
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) w[i] = pack_bf16(v[2 * i], v[2 * i + 1]);
            }
            src.load(0, BN, 64 * j + 32, v);
            if (a.f16) {
#pragma unroll
                for (int i = 0; i < 16; ++i) w[16 + i] = pack_f16(v[2 * i], v[2 * i + 1]);
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) w[16 + i] = pack_bf16(v[2 * i], v[2 * i + 1]);
            }
            out.put(w, head * (a.q_ld > 0 ? a.q_ld : a.Hckv) + col, row0);
        }
        return;
    }
    // Dynamic int8 quantisation of the whole (token, head) row (c0 = 0: one tile per head).
    float m = 0.f;
#pragma unroll 1
    for (int ch = 0; ch < BN / 32; ++ch) {
        const int col = ch * 32;
        if (col >= a.Hckv) break;
        float v[32];
        src.load(0, BN, col, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) m = fmaxf(m, fabsf(v[i]));
    }
    const float scale = m / 127.f;
#pragma unroll 1
    for (int j = 0; j < BN / 128; ++j) {
        const int col = 128 * j;
        if (col >= a.Hckv) break;
        uint32_t w[32];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            float v[32];
            src.load(0, BN, col + 32 * h, v);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                uint32_t packed = 0;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int qv = (scale > 0.f) ? quant_i8(__fdiv_rn(v[4 * i + e], scale)) : 0;
                    packed |= ((uint32_t)(qv & 0xFF)) << (8 * e);
                }
                w[8 * h + i] = packed;
            }
        }
        out.put(w, head * (a.q_ld > 0 ? a.q_ld : a.Hckv) + c0 + col, row0);
    }
    if (row < a.T) a.q_scale[(size_t)row * a.N + head] = scale;
}

// q^N of one whole-row tile (one head, BN >= Hckv) with EPW warps per TMEM lane quarter: the
// warp of share `part` owns 128-column chunks part, part + EPW, ...  For the int8 output each
// warp takes the absolute maximum over its columns of every row, the EPW partial maxima of a
// row meet in shared memory (`xbuf`, one of two buffers by tile parity, so that a fast warp's
// next tile never overwrites what a slow warp still reads), and every warp then quantises its
// own columns with the row's scale.  Rows at or past T take part in the exchange with a
// maximum of zero and store nothing.  Called by all 128 * EPW epilogue threads together.
template <int BN, int OUTB, int EPW>
__device__ __forceinline__ void epilogue_qn_split(const GemmArgs& a, const Unit& u, const TmemSrc& src, int q,
                                                  OutStage<OUTB>& out, int part, float* xbuf) {
    static_assert(BN % (128 * EPW) == 0 || BN == 128 * EPW, "whole 128-column chunks per warp");
    const int head = u.n_tile / a.tiles_per_head;
    const int c0 = (u.n_tile % a.tiles_per_head) * BN;
    const int row0 = u.m_tile * 128 + q * 32;   // this warp's first row
    const int row = row0 + out.lane;
    const bool any = row0 < a.T;                // warp-uniform
    const size_t ld = a.q_ld > 0 ? a.q_ld : a.Hckv;
    if (a.q_out_i8 == nullptr) {
        // 16-bit output: no row-wide step, each warp stores its own chunks
#pragma unroll 1
        for (int j = 2 * part; any && j < BN / 64; j += 2 * EPW) {
#pragma unroll 1
            for (int jj = j; jj < j + 2; ++jj) {
                const int col = c0 + 64 * jj;
                if (col >= a.Hckv) break;
                uint32_t w[32];
                float v[32];
                src.load(0, BN, 64 * jj, v);
#pragma unroll
                for (int i = 0; i < 16; ++i) w[i] = a.f16 ? pack_f16(v[2 * i], v[2 * i + 1]) : pack_bf16(v[2 * i], v[2 * i + 1]);
                src.load(0, BN, 64 * jj + 32, v);
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    w[16 + i] = a.f16 ? pack_f16(v[2 * i], v[2 * i + 1]) : pack_bf16(v[2 * i], v[2 * i + 1]);
                out.put(w, head * (int)ld + col, row0);
            }
        }
        return;
    }
    // int8: this warp's share of the row maximum
    float m = 0.f;
#pragma unroll 1
    for (int j = part; any && j < BN / 128; j += EPW) {
        if (c0 + 128 * j >= a.Hckv) break;
        uint32_t r[4][32];
        src.load128(128 * j, r);
#pragma unroll
        for (int h = 0; h < 4; ++h)
#pragma unroll
            for (int i = 0; i < 32; ++i) m = fmaxf(m, fabsf(bits_f(r[h][i])));
    }
    const int rin = q * 32 + out.lane;
    xbuf[part * 128 + rin] = m;
    epi_bar_n<128 * EPW>();
#pragma unroll
    for (int p = 0; p < EPW; ++p) m = fmaxf(m, xbuf[p * 128 + rin]);
    if (!any) return;
    const float scale = m / 127.f;
    // The codes round(v / scale) are taken as round(v * (127 / m)): the two differ only for
    // quotients within a few ulp of a half-integer, by one code at most.
    const float inv = m > 0.f ? __fdiv_rn(127.f, m) : 0.f;
#pragma unroll 1
    for (int j = part; j < BN / 128; j += EPW) {
        const int col = 128 * j;
        if (c0 + col >= a.Hckv) break;
        uint32_t w[32];
        uint32_t r[4][32];
        src.load128(col, r);
#pragma unroll
        for (int h = 0; h < 4; ++h) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                uint32_t packed = 0;
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    packed |= ((uint32_t)(quant_i8(bits_f(r[h][4 * i + e]) * inv) & 0xFF)) << (8 * e);
                w[8 * h + i] = packed;
            }
        }
        out.put(w, head * (int)ld + c0 + col, row0);
    }
    if (part == 0 && row < a.T) a.q_scale[(size_t)row * a.N + head] = scale;
}

// ---------------------------------------------------------------------- loads

// Weight tile of the stage starting at k-block kb: BN/64 boxes of 64 columns x (64 * KPS) rows
// (the tensor maps' box height).
template <int BN, int KPS = 1>
__device__ __forceinline__ void load_b(const GemmArgs& a, const Unit& u, int kb, uint32_t dst, uint32_t bar,
                                       const CUtensorMap* b0, const CUtensorMap* b1, uint64_t pol) {
    int head = 0, c0;
    if (a.head_mode) {
        head = u.n_tile / a.tiles_per_head;
        c0 = (u.n_tile % a.tiles_per_head) * BN;
    } else {
        c0 = u.n_tile * BN;
    }
    if (a.head_mode && a.b_blocks) {
        // one box: BN/64 column blocks of 64 x (64 * KPS) rows of head `head`
        tma_load_3d(dst, b0, bar, 0, head * a.head_rows + kb * kBK, c0 / 64, pol);
        return;
    }
    if (!a.head_mode && a.b_blocks) {
        // one box: BN/64 column blocks of 64 x (64 * KPS), laid out block after block (a tile
        // never straddles b_split_col)
        if (c0 < a.b_split_col)
            tma_load_3d(dst, b0, bar, 0, kb * kBK, c0 / 64, pol);
        else
            tma_load_3d(dst, b1, bar, 0, kb * kBK, (c0 - a.b_split_col) / 64, pol);
        return;
    }
#pragma unroll
    for (int j = 0; j < BN / 64; ++j) {
        const int col = c0 + 64 * j;
        const uint32_t d = dst + j * (64 * kBK * 2 * KPS);
        if (a.head_mode)
            tma_load_3d(d, b0, bar, col, kb * kBK, head, pol);
        else if (col < a.b_split_col)
            tma_load_2d(d, b0, bar, col, kb * kBK, pol);
        else
            tma_load_2d(d, b1, bar, col - a.b_split_col, kb * kBK, pol);
    }
}

// Activation tile of k-block kb: MSUB boxes of a_box_rows rows x 64 columns.
template <int MSUB>
__device__ __forceinline__ void load_a(const GemmArgs& a, const Unit& u, int kb, uint32_t dst, int a_box,
                                       uint32_t bar, const CUtensorMap* map, uint64_t pol) {
    const int head = a.head_mode ? u.n_tile / a.tiles_per_head : 0;
    if (!a.head_mode && a.a_one_box) {
        tma_load_2d(dst, map, bar, kb * kBK, u.m_tile * MSUB * 128, pol);
        return;
    }
#pragma unroll
    for (int ms = 0; ms < MSUB; ++ms) {
        const int r0 = (u.m_tile * MSUB + ms) * 128;
        if (a.head_mode)
            tma_load_3d(dst + ms * a_box, map, bar, kb * kBK, head, r0, pol);
        else
            tma_load_2d(dst + ms * a_box, map, bar, kb * kBK, r0, pol);
    }
}

// ---------------------------------------------------------------------- kernel

template <int BN, int MSUB, int MAXST, int EPI, int OUTB = 0, int KPS = 1, int EPW = 1>
__global__ void __launch_bounds__(gemm_threads(EPW), 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b0,
                   const __grid_constant__ CUtensorMap map_b1, const __grid_constant__ CUtensorMap map_o,
                   const __grid_constant__ CUtensorMap map_o2, const GemmArgs args) {
    using C = GemmCfg<BN, MSUB, MAXST, OUTB, KPS, EPW>;
    constexpr int kEpiThreads = 128 * EPW;
    static_assert(EPW == 1 || (OUTB > 0 && (EPI == EPI_F32 || EPI == EPI_QN || (EPI == EPI_QROPE && BN != 192))),
                  "split epilogues exist for TMA-stored fp32 rows, q^N tiles and head-unaligned RoPE tiles");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
    uint64_t* full = bars;
    uint64_t* empty = bars + MAXST;
    uint64_t* tfull = bars + 2 * MAXST;
    uint64_t* tempty = tfull + 2;
    uint64_t* done = tempty + 2;
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(done + 1);
    volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
    const int stages = args.stages;
    const int a_stage = C::a_stage_bytes(args.a_box_rows);
    const int a_box = args.a_box_rows * 128;
    uint8_t* sA = smem + C::kBarBytes;
    uint8_t* sB = sA + (size_t)stages * a_stage;
    uint8_t* sOut = sB + (size_t)stages * C::kBStage;   // OUTB x 4 KB per epilogue warp
    float* sX = reinterpret_cast<float*>(sOut + C::kOutBytes);   // C::kXBytes: split-epilogue exchange

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&map_a);
        tma_prefetch_map(&map_b0);
        tma_prefetch_map(&map_b1);
        if (OUTB > 0 && args.tma_out) {
            tma_prefetch_map(&map_o);
            if (EPI == EPI_QROPE) tma_prefetch_map(&map_o2);
        }
        for (int s = 0; s < stages; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&tfull[b]), 1);
            mbar_init(smem_u32(&tempty[b]), kEpiThreads);
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

    // Everything above overlaps the previous grid.  Once every CTA of this grid is resident the
    // next kernel may start its own prologue on free SMs.
    pdl_launch_dependents();
    if (warp != 0) pdl_wait();   // the producer waits inside its role, after the first weight loads
    if (args.clear_status && blockIdx.x == 0 && threadIdx.x == 64) *args.status = 0u;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_a = policy_evict_last();
            int s = 0;
            uint32_t ph = 0;
            Unit u;
            bool ok = true;
            // Weights do not depend on the previous kernel: the first ring of weight tiles is
            // requested before waiting for it; activation tiles follow once it has finished.
            int pre = 0;
            Unit u0;
            const bool have0 = get_unit(args, 0, u0);
            // The activation tiles of one stage: KPS k-blocks of MSUB boxes each.
            auto load_a_stage = [&](const Unit& uu, int kb, uint32_t dst, uint32_t fb) {
#pragma unroll
                for (int k = 0; k < KPS; ++k)
                    load_a<MSUB>(args, uu, kb + k, dst + k * MSUB * a_box, a_box, fb, &map_a, pol_a);
            };
            if (args.b_late) pdl_wait();   // the weights come from an earlier kernel of the call
            if (have0) {
                const int n0 = (u0.kb1 - u0.kb0) / KPS;
                pre = n0 < stages ? n0 : stages;
                for (int i = 0; i < pre; ++i) {
                    const uint32_t fb = smem_u32(&full[i]);
                    mbar_arrive_expect_tx(fb, (uint32_t)(a_stage + C::kBStage));
                    if (args.a_ready)   // stage i complete as early as possible
                        load_a_stage(u0, u0.kb0 + i * KPS, smem_u32(sA + (size_t)i * a_stage), fb);
                    load_b<BN, KPS>(args, u0, u0.kb0 + i * KPS, smem_u32(sB + (size_t)i * C::kBStage), fb, &map_b0,
                                    &map_b1, pol_w);
                }
            }
            pdl_wait();
            if (!args.a_ready)
                for (int i = 0; i < pre; ++i)
                    load_a_stage(u0, u0.kb0 + i * KPS, smem_u32(sA + (size_t)i * a_stage), smem_u32(&full[i]));
            s = pre % stages;
            ph = (pre == stages) ? 1u : 0u;
            for (int idx = 0; ok && get_unit(args, idx, u); ++idx) {
                for (int kb = u.kb0 + (idx == 0 ? pre * KPS : 0); kb < u.kb1; kb += KPS) {
                    if (!mbar_wait(smem_u32(&empty[s]), ph ^ 1, s_abort, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(&full[s]);
                    mbar_arrive_expect_tx(fb, (uint32_t)(a_stage + C::kBStage));
                    load_b<BN, KPS>(args, u, kb, smem_u32(sB + (size_t)s * C::kBStage), fb, &map_b0, &map_b1, pol_w);
                    load_a_stage(u, kb, smem_u32(sA + (size_t)s * a_stage), fb);
                    if (++s == stages) {
                        s = 0;
                        ph ^= 1;
                    }
                }
            }
            if (!ok) {
                *s_abort = 1;
                atomicOr(args.status, kStatusWaitTimeout);
            }
        } else {
            pdl_wait();
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = args.f16 ? idesc_f16_f32(128, C::kMmaN, false, true)
                                            : idesc_bf16_f32(128, C::kMmaN, false, true);
            const uint64_t a_desc0 = smem_desc_sw128(smem_u32(sA), 16, 1024);
            const uint64_t b_desc0 = smem_desc_sw128(smem_u32(sB), 64 * kBK * 2 * KPS, 1024);
            int s = 0;
            uint32_t ph = 0, ai = 0;
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
                for (int kb = u.kb0; kb < u.kb1; kb += KPS) {
                    if (!mbar_wait(smem_u32(&full[s]), ph, s_abort, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // Descriptors of this stage, advanced by constant offsets (the start-address
                    // field counts 16-byte units): cheap enough to keep the tensor core fed.
                    const uint64_t a_desc = a_desc0 + (uint64_t)s * (uint64_t)(a_stage >> 4);
                    const uint64_t b_desc = b_desc0 + (uint64_t)s * (uint64_t)(C::kBStage >> 4);
                    constexpr int kBox = 64 * kBK * 2 * KPS;   // one weight box (column stride of B)
#pragma unroll
                    for (int k = 0; k < KPS; ++k)
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
#pragma unroll
                        for (int ms = 0; ms < MSUB; ++ms) {
                            const uint64_t adesc = a_desc + (uint64_t)((((k * MSUB + ms) * a_box) >> 4) + 2 * kk);
#pragma unroll
                            for (int np = 0; np < C::kNParts; ++np) {
                                const uint64_t bdesc =
                                    b_desc + (uint64_t)(((np * (C::kMmaN / 64) * kBox + k * (64 * kBK * 2)) >> 4) + 128 * kk);
                                umma_bf16(d_base + ms * BN + np * C::kMmaN, adesc, bdesc, idesc,
                                          (kb > u.kb0 || k > 0 || kk > 0) ? 1u : 0u);
                            }
                        }
                    }
                    umma_commit(smem_u32(&empty[s]));
                    if (++s == stages) {
                        s = 0;
                        ph ^= 1;
                    }
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
        const int part = (warp - 2) >> 2;   // which share of the columns (EPW warps per quarter)
        const int row_in = q * 32 + lane;
        OutStage<OUTB> ostage{sOut + (size_t)(warp - 2) * OUTB * 4096, 0, &map_o, lane};
        if constexpr (EPI == EPI_QROPE) {
            // This thread's RoPE table rows of its first tile, into L2 during the main loop.
            Unit u0;
            if (get_unit(args, 0, u0)) {
                for (int ms = 0; ms < MSUB; ++ms) {
                    const int r = u0.m_tile * MSUB * 128 + ms * 128 + row_in;
                    if (r < args.T) {
                        prefetch_l2(args.rope_cos + (size_t)r * 64);
                        prefetch_l2(args.rope_sin + (size_t)r * 64);
                    }
                }
            }
        }
        uint32_t ai = 0;
        Unit u;
        for (int idx = 0; get_unit(args, idx, u); ++idx, ++ai) {
            const int b = ai % C::kNBuf;
            const uint32_t aph = (ai / C::kNBuf) & 1;
            int ok = 1;
            if (lane == 0) ok = mbar_wait(smem_u32(&tfull[b]), aph, s_abort, kWaitLimitNs) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok && lane == 0) {
                *s_abort = 1;
                atomicOr(args.status, kStatusWaitTimeout);
            }
            // The epilogue warps stop together or not at all.
            if (epi_any_n<kEpiThreads>(!ok)) break;
            __syncwarp();
            tc_fence_after();
            const TmemSrc tsrc{tmem_base + ((uint32_t)(q * 32) << 16) + b * C::kAcc};
            const int row0 = u.m_tile * MSUB * 128 + row_in;
            if constexpr (EPI == EPI_F32) {
                if constexpr (EPW > 1) {
                    epilogue_f32_tma<BN, MSUB, OUTB, EPW>(args, u, tsrc, q, ostage, part);
                } else if constexpr (OUTB > 0) {
                    if (args.tma_out)
                        epilogue_f32_tma<BN, MSUB, OUTB>(args, u, tsrc, q, ostage);
                    else
                        epilogue_f32<BN, MSUB>(args, row0, u.n_tile, u.ks, tsrc);
                } else {
                    epilogue_f32<BN, MSUB>(args, row0, u.n_tile, u.ks, tsrc);
                }
            } else if constexpr (EPI == EPI_QROPE) {
                if constexpr (BN != 192) {
                    static_assert(OUTB > 0, "head-unaligned tiles store through TMA");
                    epilogue_qrope_blocks_tma<BN, MSUB, OUTB, EPW>(args, u, tsrc, q, ostage, &map_o, &map_o2, part);
                } else if constexpr (OUTB > 0) {
                    if (args.tma_out)
                        epilogue_qrope_tma<MSUB, OUTB>(args, u, tsrc, q, ostage, &map_o, &map_o2);
                    else
                        epilogue_qrope<MSUB>(args, row0, u.n_tile, tsrc);
                } else {
                    epilogue_qrope<MSUB>(args, row0, u.n_tile, tsrc);
                }
            } else {
                if constexpr (EPW > 1) {
                    epilogue_qn_split<BN, OUTB, EPW>(args, u, tsrc, q, ostage, part, sX + (ai & 1) * 128 * EPW);
                } else if constexpr (OUTB > 0) {
                    if (args.tma_out)
                        epilogue_qn_tma<BN, OUTB>(args, u, tsrc, q, ostage);
                    else
                        epilogue_qn<BN>(args, u, tsrc, row_in);
                } else {
                    epilogue_qn<BN>(args, u, tsrc, row_in);
                }
            }
            tc_fence_before();
            mbar_arrive(smem_u32(&tempty[b]));
        }
        if constexpr (OUTB > 0) ostage.drain();   // the stores have read their shared memory
    }

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
