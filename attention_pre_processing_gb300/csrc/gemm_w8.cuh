// GEMM with int8 weights streamed as int8 and widened in shared memory: out = A . W with A fp16
// (T, K) row-major (int8 codes held as fp16, exact) and W int8 in one of two orientations:
//   MN = false: (ncols, K) row-major, one row per output column (the aclnnMlaPreprocess variant,
//               "transposeWdq/Wuq" true), widened into K-major B tiles;
//   MN = true:  (K, ncols) row-major, the (k, n) orientation of aclnnMlaPrologV2WeightNz's int8
//               weights, widened into MN-major B tiles (64-column blocks of 64 k rows); the
//               columns below b_split_col come from map_b8, the rest from map_b8b (two weights
//               side by side, as W^DQ | W^DkvKr).
//
// GB300's int8 tensor rate is far below its fp16 rate, so the contraction runs as fp16 MMAs with
// fp32 accumulation (exact for these integer products while the sums stay below 2^24).  fp16
// rather than bf16 because a byte fits its 10-bit mantissa: placing the biased byte under the
// exponent of 1024 (one byte permute) and subtracting 1152 (one paired half subtraction) widens
// two weights, where int-to-float conversions run at a quarter of the ALU rate and were the
// bottleneck (0.8 us per 12 KB stage, measured).  Widening the weights in global memory first
// would move three bytes per weight through HBM more than needed; here the int8 tile crosses HBM
// once:
//   warp 0      TMA producer: per stage, kW8Kb k-blocks of A tiles (128-byte swizzle) and one
//               int8 weight box (plain rows): BN rows x 64 * kW8Kb k, or 64 * kW8Kb k rows x BN;
//               with A8 the A tiles are one int8 box (int8 tokenX, rows x 64 * kW8Kb bytes),
//               requested with the weights before the grid dependency when A is a call input
//   warp 1      TMEM allocation and the tcgen05.mma issuer (B 128-byte swizzle)
//   warps 2-5   epilogue: TMEM -> fp32 k-range slots (split-K), as gemm_tc's EPI_F32, or (EPI_QROPE,
//               one 192-column head per tile) dequant scales, RoPE and q^C, as gemm_tc's
//   warps 6-13  converters: per stage, each 16-byte int8 chunk of its k-blocks -> two 16-byte fp16
//               chunks of the swizzled B slots (chunk c of 128-byte row r at (c ^ (r % 8)) * 16;
//               rows are output columns (K-major) or k (MN-major, one 8 KB block per 64 columns)),
//               then a wait for the stage's A tiles (A8: and their widening into the pair's fp16 A
//               slots, the same 128-byte-swizzled K-major layout), a proxy fence and one arrival
//               on the slots' "B full" barrier (so the MMA thread waits once per stage)
// The int8 and A tiles run in a deep ring of stages (the weight stream's latency hiding); the
// fp16 B tiles in a ring of kBSlots slots, as deep as the shared memory allows (8 slots of 8 KB at
// BN = 64, 4 at BN = 128 and 192, 2 with 256-row tiles), so that the converters run ahead of the
// MMAs.  The slots change hands a stage (kKb k-blocks) at a time: one "B full" wait and one
// "B empty" commit per stage, not per k-block.  At decode sizes each hand-over between the
// single-thread roles costs ~0.1 us (measured with cycle-counter stamps), so a CTA's time follows
// its number of hand-overs: per-stage hand-over took the variant's call 59.4 -> 57.3 us, and
// folding the A tiles' wait into "B full" a further ~1.5 us.
// Stage s is reused only after the MMAs that read it commit (empty[s]), which follows its
// conversion; a slot pair only after the MMAs that read it commit (bempty).  Every wait is
// bounded and sets kStatusWaitTimeout.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "gemm_tc.cuh"
#include "ptx.cuh"

namespace mla {

// Converter threads: eight warps, two per scheduler, so that one warp's shared-memory latency
// hides behind the other's arithmetic (with four, a 24 KB stage took ~1 us to convert, measured).
constexpr int kW8Conv = 256;
constexpr int kW8Threads = 64 + 128 + kW8Conv;

// k-blocks of 64 per int8 stage: one TMA box of 64 * kW8Kb bytes per weight row.  The TMA
// engine moves a box row by row, at a per-SM rate of rows, so longer rows move more bytes.
constexpr int kW8Kb = 2;
static_assert(kW8Kb >= 1 && kW8Kb <= 4, "a TMA box row holds at most 256 elements");

template <int BN, int MSUB, int MAXST, bool MN = false, bool A8 = false>
struct W8Cfg {
    static constexpr int kKb = kW8Kb;
    static constexpr int kB8Row = MN ? BN : kBK * kKb;   // bytes per int8 box row
    static constexpr int kB8Stage = BN * kBK * kKb;  // int8: BN columns x 64 * kKb k
    static constexpr int kBStage = BN * kBK * 2;     // fp16: BN rows x 128 bytes
    static constexpr int kBSlots = MSUB == 1 ? (BN <= 64 ? 8 : 4) : 2;   // fp16 B slots
    static constexpr int kBPairs = kBSlots / kKb;   // handed over per stage: kKb slots per barrier
    static_assert(kBSlots % kKb == 0, "whole stages of slots");
    static constexpr int kAcc = MSUB * BN;
    static constexpr int kNBuf = (2 * kAcc <= 512) ? 2 : 1;
    static constexpr int kTmemCols = (kNBuf * kAcc <= 32) ? 32 : (kNBuf * kAcc <= 64) ? 64
                                     : (kNBuf * kAcc <= 128) ? 128 : (kNBuf * kAcc <= 256) ? 256 : 512;
    static constexpr int kBarBytes = 1024;
    static_assert(8 * (3 * MAXST + 2 * kBSlots + 5) + 16 <= kBarBytes, "barrier area");
    static_assert(BN % 16 == 0 && BN <= 256, "MMA N");
    static_assert(!MN || BN % 64 == 0, "MN-major tiles are whole 64-column blocks");
    static_assert(kAcc <= 512, "accumulator exceeds TMEM");
    static_assert(!A8 || MSUB == 1, "int8 activations: one 128-row tile");
    // A per stage: fp16 boxes (128-byte swizzle), or with A8 one int8 box of 64 * kKb bytes per
    // row, widened by the converters into fp16 A slots (one per fp16 B slot, a_box_rows x 128 B)
    static __host__ __device__ int a_stage_bytes(int a_box_rows) {
        return A8 ? kKb * a_box_rows * 64 : kKb * MSUB * a_box_rows * 128;
    }
    static __host__ __device__ int a_slot_bytes(int a_box_rows) { return A8 ? a_box_rows * 128 : 0; }
    static __host__ __device__ int stage_bytes(int a_box_rows) { return a_stage_bytes(a_box_rows) + kB8Stage; }
    // Layout: barriers | A ring (A8: fp16 A slots) | fp16 B slots | int8 ring | (A8) int8 A
    // ring.  A 128-row MMA read of a short A box runs at most 16 KB past its stage or slot, into
    // the B slots (>= 16 KB), inside the block.
    static __host__ __device__ size_t smem_bytes(int stages, int a_box_rows) {
        return 1024 + kBarBytes + (size_t)kBSlots * (kBStage + a_slot_bytes(a_box_rows)) +
               (size_t)stages * stage_bytes(a_box_rows);
    }
    static __host__ int max_stages(int a_box_rows) {
        int s = (int)((kSmemLimit - 1024 - kBarBytes - kBSlots * (kBStage + a_slot_bytes(a_box_rows))) /
                      stage_bytes(a_box_rows));
        return s < MAXST ? s : MAXST;
    }
    static_assert(kBSlots * kBStage >= 16384, "the B slots must cover the A over-read");
};

// Sixteen int8 values (one 16-byte chunk) widened to fp16 and stored as the 16-byte chunks cc and
// cc + 1 of the 128-byte shared-memory row at `row`, 128-byte swizzled (chunk c at (c ^ sw) * 16).
// The biased byte b + 128 goes under the exponent of 1024 (one byte permute); subtracting 1152
// leaves b, exactly.
__device__ __forceinline__ void w8_widen_store(int4 v, uint32_t row, uint32_t cc, uint32_t sw) {
    const uint32_t w[4] = {(uint32_t)v.x, (uint32_t)v.y, (uint32_t)v.z, (uint32_t)v.w};
    uint32_t o[8];
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480u), __ushort_as_half(0x6480u));   // 1152
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const uint32_t ub = w[e] ^ 0x80808080u;   // bytes b + 128, in 0..255
        uint32_t lo = __byte_perm(ub, 0x64646464u, 0x4140u), hi = __byte_perm(ub, 0x64646464u, 0x4342u);
        __half2 hl = __hsub2(*reinterpret_cast<__half2*>(&lo), bias);
        __half2 hh = __hsub2(*reinterpret_cast<__half2*>(&hi), bias);
        o[2 * e] = *reinterpret_cast<uint32_t*>(&hl);
        o[2 * e + 1] = *reinterpret_cast<uint32_t*>(&hh);
    }
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(row + ((cc ^ sw) << 4)), "r"(o[0]), "r"(o[1]),
                 "r"(o[2]), "r"(o[3])
                 : "memory");
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(row + (((cc + 1) ^ sw) << 4)), "r"(o[4]),
                 "r"(o[5]), "r"(o[6]), "r"(o[7])
                 : "memory");
}

template <int BN, int MSUB, int MAXST, bool MN = false, int EPI = EPI_F32, bool A8 = false>
__global__ void __launch_bounds__(kW8Threads, 1)
    gemm_w8_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b8,
                   const __grid_constant__ CUtensorMap map_b8b, const GemmArgs args) {
    using C = W8Cfg<BN, MSUB, MAXST, MN, A8>;
    static_assert(EPI == EPI_F32 || (EPI == EPI_QROPE && BN == 192), "epilogues: fp32 slots, or one head per tile");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
    uint64_t* full = bars;                 // A tile landed (TMA)
    uint64_t* empty = bars + MAXST;        // the stage's MMAs completed
    uint64_t* full8 = bars + 2 * MAXST;    // int8 weight tile landed (TMA)
    uint64_t* bfull = bars + 3 * MAXST;    // fp16 slot written by the converters [kBSlots]
    uint64_t* bempty = bfull + C::kBSlots; // fp16 slot's MMAs completed [kBSlots]
    uint64_t* tfull = bempty + C::kBSlots;
    uint64_t* tempty = tfull + 2;
    uint64_t* done = tempty + 2;
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(done + 1);
    volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
    const int stages = args.stages;
    const int a_stage = C::a_stage_bytes(args.a_box_rows);
    const int a_box = args.a_box_rows * 128;
    const int a_slot = C::a_slot_bytes(args.a_box_rows);
    uint8_t* sA = smem + C::kBarBytes;   // fp16 A stages, or (A8) fp16 A slots
    uint8_t* sB = sA + (A8 ? (size_t)C::kBSlots * a_slot : (size_t)stages * a_stage);
    uint8_t* sB8 = sB + (size_t)C::kBSlots * C::kBStage;
    uint8_t* sA8 = sB8 + (size_t)stages * C::kB8Stage;   // A8: int8 activation stages

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&map_a);
        tma_prefetch_map(&map_b8);
        if (MN) tma_prefetch_map(&map_b8b);
        for (int s = 0; s < stages; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
            mbar_init(smem_u32(&full8[s]), 1);
        }
        for (int b = 0; b < C::kBPairs; ++b) {
            mbar_init(smem_u32(&bfull[b]), kW8Conv);
            mbar_init(smem_u32(&bempty[b]), 1);
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

    pdl_launch_dependents();
    // The weights are inputs of the call: the producer requests its first ring of int8 weight
    // tiles before waiting for the previous kernel (its activation tiles after), and the
    // converters, which touch shared memory only, widen them meanwhile.  The MMA and epilogue
    // warps wait here.
    if (warp >= 1 && warp < 6) pdl_wait();
    if (args.clear_status && blockIdx.x == 0 && threadIdx.x == 64) *args.status = 0u;

    auto fail = [&]() {
        *s_abort = 1;
        atomicOr(args.status, kStatusWaitTimeout);
    };

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_a = policy_evict_last();
            int s = 0;
            uint32_t ph = 0;
            Unit u;
            bool ok = true;
            // one stage: the int8 weight box (the whole box lands, zeros past K) ...
            auto issue_w = [&](int st, const Unit& uu, int kb) {
                const uint32_t f8 = smem_u32(&full8[st]);
                const uint32_t dst = smem_u32(sB8 + (size_t)st * C::kB8Stage);
                mbar_arrive_expect_tx(f8, (uint32_t)C::kB8Stage);
                if constexpr (MN) {
                    const int c0 = uu.n_tile * BN;   // a tile never straddles b_split_col
                    if (c0 < args.b_split_col)
                        tma_load_2d(dst, &map_b8, f8, c0, kb * kBK, pol_w);
                    else
                        tma_load_2d(dst, &map_b8b, f8, c0 - args.b_split_col, kb * kBK, pol_w);
                } else {
                    tma_load_2d(dst, &map_b8, f8, kb * kBK, uu.n_tile * BN, pol_w);
                }
            };
            // ... and its activation tiles (the unit's last stage may be short)
            auto issue_a = [&](int st, const Unit& uu, int kb) {
                const uint32_t fa = smem_u32(&full[st]);
                if constexpr (A8) {
                    // one int8 box: a_box_rows rows x 64 * kKb bytes (zeros past K and past T)
                    mbar_arrive_expect_tx(fa, (uint32_t)a_stage);
                    tma_load_2d(smem_u32(sA8 + (size_t)st * a_stage), &map_a, fa, kb * kBK, uu.m_tile * 128, pol_a);
                } else {
                    const int nkb = min(C::kKb, uu.kb1 - kb);
                    mbar_arrive_expect_tx(fa, (uint32_t)(nkb * MSUB * a_box));
                    for (int i = 0; i < nkb; ++i)
                        load_a<MSUB>(args, uu, kb + i, smem_u32(sA + (size_t)st * a_stage + i * MSUB * a_box), a_box,
                                     fa, &map_a, pol_a);
                }
            };
            if (args.b_late) pdl_wait();   // the weights come from an earlier kernel of the call
            int pre = 0;
            Unit u0;
            if (get_unit(args, 0, u0)) {
                const int n0 = (u0.kb1 - u0.kb0 + C::kKb - 1) / C::kKb;
                pre = n0 < stages ? n0 : stages;
                for (int i = 0; i < pre; ++i) {
                    issue_w(i, u0, u0.kb0 + i * C::kKb);
                    if (args.a_ready) issue_a(i, u0, u0.kb0 + i * C::kKb);   // A is an input of the call
                }
            }
            pdl_wait();
            if (!args.a_ready)
                for (int i = 0; i < pre; ++i) issue_a(i, u0, u0.kb0 + i * C::kKb);
            s = pre % stages;
            ph = (pre == stages) ? 1u : 0u;
            for (int idx = 0; ok && get_unit(args, idx, u); ++idx) {
                for (int kb = u.kb0 + (idx == 0 ? pre * C::kKb : 0); kb < u.kb1; kb += C::kKb) {
                    if (!mbar_wait(smem_u32(&empty[s]), ph ^ 1, s_abort, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    issue_w(s, u, kb);
                    issue_a(s, u, kb);
                    if (++s == stages) {
                        s = 0;
                        ph ^= 1;
                    }
                }
            }
            if (!ok) fail();
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            // fp16, A K-major; B K-major or MN-major (64-column blocks 8 KB apart)
            constexpr uint32_t idesc = idesc_f16_f32(128, BN, false, MN);
            constexpr uint64_t b_step = MN ? 128 : 2;   // one K = 16 step: 16 rows, or 32 bytes of a row
            const uint64_t a_desc0 = smem_desc_sw128(smem_u32(sA), 16, 1024);
            const uint64_t b_desc0 = smem_desc_sw128(smem_u32(sB), MN ? 64 * 128 : 16, 1024);
            int s = 0;
            uint32_t ph = 0, ai = 0, gs = 0;   // gs: stages so far (fp16 slot pair gs % kBPairs)
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
                for (int kb = u.kb0; ok && kb < u.kb1; kb += C::kKb) {
                    const int nkb = min(C::kKb, u.kb1 - kb);
                    // the stage's fp16 slots: pair gp (kKb slots from kKb * gp); "B full" also
                    // means the stage's A tiles have landed (the converters wait for them)
                    const int gp = (int)(gs % C::kBPairs);
                    if (!mbar_wait(smem_u32(&bfull[gp]), (gs / C::kBPairs) & 1u, s_abort, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    for (int i = 0; i < nkb; ++i) {
                        const int j = gp * C::kKb + i;
                        const uint64_t a_desc =
                            A8 ? a_desc0 + (uint64_t)(((size_t)j * a_slot) >> 4)
                               : a_desc0 + (uint64_t)(((size_t)s * a_stage + (size_t)i * MSUB * a_box) >> 4);
                        const uint64_t b_desc = b_desc0 + (uint64_t)j * (uint64_t)(C::kBStage >> 4);
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; ++kk)
#pragma unroll
                            for (int ms = 0; ms < MSUB; ++ms)
                                umma_bf16(d_base + ms * BN, a_desc + (uint64_t)(((ms * a_box) >> 4) + 2 * kk),
                                          b_desc + b_step * kk, idesc, (kb + i > u.kb0 || kk > 0) ? 1u : 0u);
                    }
                    umma_commit(smem_u32(&bempty[gp]));
                    ++gs;
                    if (!ok) break;
                    umma_commit(smem_u32(&empty[s]));
                    if (++s == stages) {
                        s = 0;
                        ph ^= 1;
                    }
                }
                if (!ok) break;
                umma_commit(smem_u32(&tfull[b]));
            }
            if (!ok) fail();
            umma_commit(smem_u32(done));
            mbar_wait(smem_u32(done), 0, s_abort, kWaitLimitNs / 4);
        }
    } else if (warp < 6) {
        // ------------------------------------------------------------ epilogue warps
        const int q = warp & 3;
        const int row_in = q * 32 + lane;
        uint32_t ai = 0;
        Unit u;
        for (int idx = 0; get_unit(args, idx, u); ++idx, ++ai) {
            const int b = ai % C::kNBuf;
            const uint32_t aph = (ai / C::kNBuf) & 1;
            int ok = 1;
            if (lane == 0) ok = mbar_wait(smem_u32(&tfull[b]), aph, s_abort, kWaitLimitNs) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok && lane == 0) fail();
            if (epi_any_n<128>(!ok)) break;
            __syncwarp();
            tc_fence_after();
            const TmemSrc tsrc{tmem_base + ((uint32_t)(q * 32) << 16) + b * C::kAcc};
            if constexpr (EPI == EPI_QROPE)
                epilogue_qrope<MSUB>(args, u.m_tile * MSUB * 128 + row_in, u.n_tile, tsrc);
            else
                epilogue_f32<BN, MSUB>(args, u.m_tile * MSUB * 128 + row_in, u.n_tile, u.ks, tsrc);
            tc_fence_before();
            mbar_arrive(smem_u32(&tempty[b]));
        }
    } else {
        // ------------------------------------------------------------ converters
        const int ct = threadIdx.x - 192;   // 0 .. kW8Conv - 1
        int s = 0;
        uint32_t ph = 0, gs = 0;
        Unit u;
        bool ok = true;
        for (int idx = 0; ok && get_unit(args, idx, u); ++idx) {
            for (int kb = u.kb0; ok && kb < u.kb1; kb += C::kKb) {
                const int nkb = min(C::kKb, u.kb1 - kb);
                if (!mbar_wait(smem_u32(&full8[s]), ph, s_abort, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                const int gp = (int)(gs % C::kBPairs);
                if (!mbar_wait(smem_u32(&bempty[gp]), ((gs / C::kBPairs) & 1u) ^ 1u, s_abort, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                for (int i = 0; i < nkb; ++i) {
                    const int j = gp * C::kKb + i;
                    // k-block i of the stage: 16 bytes of the int8 box's rows at i * kBK (K-major), or
                    // its 64 rows from 64 i on (MN-major)
                    const uint8_t* src = sB8 + (size_t)s * C::kB8Stage + (MN ? (size_t)i * kBK * BN : (size_t)i * kBK);
                    const uint32_t dst = smem_u32(sB + (size_t)j * C::kBStage);
#pragma unroll 2
                    for (int task = ct; task < BN * 4; task += kW8Conv) {
                        // K-major: row r = output column, chunk c = k 16c .. 16c+15 (4 per row);
                        // MN-major: row r = k, chunk c = columns 16c .. 16c+15 (BN / 16 per row)
                        const int r = MN ? task / (BN / 16) : task >> 2;
                        const int c = MN ? task % (BN / 16) : task & 3;
                        const int4 v = *reinterpret_cast<const int4*>(src + r * C::kB8Row + c * 16);
                        // the fp16 row (128 bytes) and its 16-byte chunk pair
                        const uint32_t row = MN ? dst + (uint32_t)((c >> 2) * (64 * 128) + r * 128) : dst + (uint32_t)(r * 128);
                        w8_widen_store(v, row, MN ? 2u * (uint32_t)(c & 3) : 2u * (uint32_t)c, (uint32_t)(r & 7));
                    }
                }
                // the stage's A tiles too: one wait for the MMA thread per stage
                if (!mbar_wait(smem_u32(&full[s]), ph, s_abort, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                if constexpr (A8) {
                    // the int8 activation box (row r = token, 64 * kKb bytes) into the pair's fp16
                    // A slots (K-major, 128-byte swizzle)
                    const uint8_t* srcA = sA8 + (size_t)s * a_stage;
                    for (int i = 0; i < nkb; ++i) {
                        const uint32_t dstA = smem_u32(sA + (size_t)(gp * C::kKb + i) * a_slot);
                        for (int task = ct; task < args.a_box_rows * 4; task += kW8Conv) {
                            const int r = task >> 2, c = task & 3;
                            const int4 v = *reinterpret_cast<const int4*>(srcA + r * (kBK * C::kKb) + i * kBK + c * 16);
                            w8_widen_store(v, dstA + (uint32_t)(r * 128), 2u * (uint32_t)c, (uint32_t)(r & 7));
                        }
                    }
                }
                fence_proxy_async_smem();   // the tensor core reads what these threads wrote
                mbar_arrive(smem_u32(&bfull[gp]));
                ++gs;
                if (!ok) break;
                if (++s == stages) {
                    s = 0;
                    ph ^= 1;
                }
            }
        }
        if (!ok) fail();
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
