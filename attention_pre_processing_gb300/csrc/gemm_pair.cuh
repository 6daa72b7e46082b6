// Pair-CTA tcgen05 GEMM for prefill-sized token counts: a cluster of two CTAs on two SMs
// computes one 256-row x BN-column tile with tcgen05.mma.cta_group::2 (M = 256).
//
//   D[rows, cols] = A[rows, K] . B[K, cols]    (A: activations, K-major; B: weights, N-major)
//
// CTA r of the pair loads A rows [256 m + 128 r, +128) and B columns [BN n + BN/2 r, +BN/2) of
// each k-block into its own shared memory; the even CTA issues the MMA, which reads both CTAs'
// operands at the same offsets and writes each CTA's 128 rows of D into that CTA's tensor
// memory.  Per k-block each SM therefore receives 128 x 64 activation and BN/2 x 64 weight
// elements instead of the 128 x 64 and BN x 64 of a one-SM 128 x BN tile: a third less
// shared-memory traffic for the same tensor-core work, and the weight stream is what bounds
// the one-SM tiles.
//
// Roles (64 + 128 EPW threads per CTA):
//   warp 0, lane 0     TMA producer (both CTAs): its own halves of A and B into a ring of stages
//   warp 1             allocates tensor memory for the pair (both CTAs together); lane 0 of the
//                      even CTA issues the MMAs, lane 0 of the odd CTA tells the even CTA that a
//                      stage of its operands has landed (a remote mbarrier arrival)
//   warps 2..          epilogue (both CTAs): each CTA drains its own 128 rows of the accumulator
// The even CTA's commits arrive on both CTAs' barriers (multicast), so each producer learns when
// its stage has been read, and each epilogue when its accumulator is complete.  Two accumulators
// of BN columns let one tile's epilogue overlap the next tile's main loop.  Every wait is
// bounded (kWaitLimitNs): a wait that gives up raises MLA_DEV_WAIT_TIMEOUT and the roles stop.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "gemm_tc.cuh"
#include "ptx.cuh"

namespace mla {

// KPS: k-blocks of 64 per stage.  The activation box is (64 k, 128 rows, KPS k-blocks) and the
// weight box (64 columns, 64 KPS k rows, BN/128 column blocks) of a 3D view of each matrix, so a
// stage is two TMA requests however large it is.
template <int BN, int MAXST, int OUTB, int EPW, int KPS>
struct PairCfg {
    static constexpr int kHalfN = BN / 2;                  // B columns held by each CTA
    static constexpr int kABlock = 128 * kBK * 2;          // 128 rows x 64 k
    static constexpr int kBBlock = 64 * kBK * KPS * 2;     // 64 columns x 64 KPS k rows
    static constexpr int kAStage = KPS * kABlock;
    static constexpr int kBStage = (kHalfN / 64) * kBBlock;
    static constexpr int kStage = kAStage + kBStage;
    static constexpr int kTmemCols = 512;                  // two accumulators of BN columns
    static constexpr int kOutBytes = 4 * EPW * OUTB * 4096;
    static constexpr int kBarBytes = 1024;
    static_assert(BN % 128 == 0 && BN <= 256, "pair tiles: BN in {128, 256}");
    static_assert(2 * BN <= kTmemCols, "two accumulators");
    static_assert(8 * (3 * MAXST + 5) + 16 <= kBarBytes, "barrier area");

    static __host__ int max_stages() {
        int s = (int)((kSmemLimit - 1024 - kBarBytes - kOutBytes) / kStage);
        return s < MAXST ? s : MAXST;
    }
    static __host__ __device__ size_t smem_bytes(int stages) {
        return 1024 + kBarBytes + (size_t)stages * kStage + kOutBytes;
    }
};

// The idx-th 256-row tile of this pair: row tile fastest, or column tile fastest (n_fastest).
__device__ __forceinline__ bool get_pair_unit(const GemmArgs& a, int idx, Unit& u) {
    const long long npairs = gridDim.x >> 1;
    const long long i = (long long)(blockIdx.x >> 1) + (long long)idx * npairs;
    if (i >= (long long)a.m_tiles * a.n_tiles) return false;
    if (a.n_fastest) {
        u.n_tile = (int)(i % a.n_tiles);
        u.m_tile = (int)(i / a.n_tiles);
    } else {
        u.m_tile = (int)(i % a.m_tiles);
        u.n_tile = (int)(i / a.m_tiles);
    }
    u.kb0 = 0;
    u.kb1 = a.kblocks;
    u.ks = 0;
    return true;
}

template <int BN, int MAXST, int EPI, int OUTB, int EPW, int KPS>
__global__ void __launch_bounds__(gemm_threads(EPW), 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b0,
                     const __grid_constant__ CUtensorMap map_b1, const __grid_constant__ CUtensorMap map_o,
                     const __grid_constant__ CUtensorMap map_o2, const GemmArgs args) {
    using C = PairCfg<BN, MAXST, OUTB, EPW, KPS>;
    constexpr int kEpiThreads = 128 * EPW;
    static_assert(OUTB > 0 && (EPI == EPI_F32 || EPI == EPI_QROPE || EPI == EPI_DOWN), "pair tiles store through TMA");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
    uint64_t* full = bars;                   // [MAXST] this CTA's operands of the stage landed
    uint64_t* empty = full + MAXST;          // [MAXST] the pair's MMAs have read the stage
    uint64_t* pfull = empty + MAXST;         // [MAXST] even CTA: the odd CTA's operands landed
    uint64_t* tfull = pfull + MAXST;         // [2] accumulator complete
    uint64_t* tempty = tfull + 2;            // [2] even CTA: both CTAs drained the accumulator
    uint64_t* done = tempty + 2;
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(done + 1);
    volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
    const int stages = args.stages;
    uint8_t* sA = smem + C::kBarBytes;
    uint8_t* sB = sA + (size_t)stages * C::kAStage;
    uint8_t* sOut = sB + (size_t)stages * C::kBStage;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;

    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&map_a);
        tma_prefetch_map(&map_b0);
        tma_prefetch_map(&map_b1);
        tma_prefetch_map(&map_o);
        if (EPI != EPI_F32) tma_prefetch_map(&map_o2);
        for (int s = 0; s < stages; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
            mbar_init(smem_u32(&pfull[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&tfull[b]), 1);
            mbar_init(smem_u32(&tempty[b]), kEpiThreads + 1);   // own epilogue + the odd CTA's
        }
        mbar_init(smem_u32(done), 1);
        *s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) tmem_alloc_pair(smem_u32(s_tmem), C::kTmemCols);
    tc_fence_before();
    __syncthreads();
    cluster_sync();   // both CTAs' barriers and tensor memory exist before either uses the other's
    tc_fence_after();
    const uint32_t tmem_base = *s_tmem;

    pdl_launch_dependents();
    if (warp != 0) pdl_wait();
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
            auto load_b_half = [&](const Unit& u, int kb, uint32_t dst, uint32_t fb) {
                const int c = u.n_tile * BN + (int)rank * C::kHalfN;   // never straddles b_split_col
                if (c < args.b_split_col)
                    tma_load_3d(dst, &map_b0, fb, 0, kb * kBK, c / 64, pol_w);
                else
                    tma_load_3d(dst, &map_b1, fb, 0, kb * kBK, (c - args.b_split_col) / 64, pol_w);
            };
            auto load_a_half = [&](const Unit& u, int kb, uint32_t dst, uint32_t fb) {
                tma_load_3d(dst, &map_a, fb, 0, u.m_tile * 256 + (int)rank * 128, kb, pol_a);
            };
            const int nst = args.kblocks / KPS;   // stages per tile
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            // The first ring of weight tiles goes out before the grid dependency resolves (unless
            // an earlier kernel of the call writes them).
            int pre = 0;
            Unit u0;
            if (args.b_late) pdl_wait();   // the weights come from an earlier kernel of the call
            if (get_pair_unit(args, 0, u0)) {
                pre = nst < stages ? nst : stages;
                for (int i = 0; i < pre; ++i) {
                    const uint32_t fb = smem_u32(&full[i]);
                    mbar_arrive_expect_tx(fb, (uint32_t)C::kStage);
                    load_b_half(u0, i * KPS, smem_u32(sB + (size_t)i * C::kBStage), fb);
                    if (args.a_ready) load_a_half(u0, i * KPS, smem_u32(sA + (size_t)i * C::kAStage), fb);
                }
            }
            pdl_wait();
            if (!args.a_ready)
                for (int i = 0; i < pre; ++i)
                    load_a_half(u0, i * KPS, smem_u32(sA + (size_t)i * C::kAStage), smem_u32(&full[i]));
            s = pre % stages;
            ph = (pre == stages) ? 1u : 0u;
            Unit u;
            for (int idx = 0; ok && get_pair_unit(args, idx, u); ++idx) {
                for (int i = (idx == 0 ? pre : 0); i < nst; ++i) {
                    if (!mbar_wait(smem_u32(&empty[s]), ph ^ 1, s_abort, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(&full[s]);
                    mbar_arrive_expect_tx(fb, (uint32_t)C::kStage);
                    load_b_half(u, i * KPS, smem_u32(sB + (size_t)s * C::kBStage), fb);
                    load_a_half(u, i * KPS, smem_u32(sA + (size_t)s * C::kAStage), fb);
                    if (++s == stages) {
                        s = 0;
                        ph ^= 1;
                    }
                }
            }
            if (!ok) fail();
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // -------------------------------------------------------- MMA issuer (even CTA)
            constexpr uint32_t idesc = idesc_bf16_f32(256, BN, false, true);
            const uint64_t a_desc0 = smem_desc_sw128(smem_u32(sA), 16, 1024);
            const uint64_t b_desc0 = smem_desc_sw128(smem_u32(sB), C::kBBlock, 1024);
            const int nst = args.kblocks / KPS;
            int s = 0;
            uint32_t ph = 0, ai = 0;
            bool ok = true;
            Unit u;
            for (int idx = 0; ok && get_pair_unit(args, idx, u); ++idx, ++ai) {
                const int b = ai & 1;
                const uint32_t aph = (ai >> 1) & 1;
                if (!mbar_wait(smem_u32(&tempty[b]), aph ^ 1, s_abort, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + b * BN;
                for (int i = 0; i < nst; ++i) {
                    if (!mbar_wait(smem_u32(&full[s]), ph, s_abort, kWaitLimitNs) ||
                        !mbar_wait(smem_u32(&pfull[s]), ph, s_abort, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t a_desc = a_desc0 + (uint64_t)s * (uint64_t)(C::kAStage >> 4);
                    const uint64_t b_desc = b_desc0 + (uint64_t)s * (uint64_t)(C::kBStage >> 4);
#pragma unroll
                    for (int k = 0; k < KPS; ++k)
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; ++kk)
                            umma_bf16_pair(d, a_desc + (uint64_t)((k * C::kABlock) >> 4) + 2 * kk,
                                           b_desc + (uint64_t)((k * kBK * 128) >> 4) + 128 * kk, idesc,
                                           (i > 0 || k > 0 || kk > 0) ? 1u : 0u);
                    umma_commit_pair(smem_u32(&empty[s]));
                    if (++s == stages) {
                        s = 0;
                        ph ^= 1;
                    }
                }
                if (!ok) break;
                umma_commit_pair(smem_u32(&tfull[b]));
            }
            if (!ok) fail();
            // Drain: every MMA issued above completes before tensor memory is freed.
            umma_commit_pair(smem_u32(done));
            mbar_wait(smem_u32(done), 0, s_abort, kWaitLimitNs / 4);
        } else if (lane == 0) {
            // -------------------------------------------------------- stage forwarder (odd CTA)
            const uint32_t peer_pfull = mapa_shared(smem_u32(pfull), 0);
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            Unit u;
            const int nst = args.kblocks / KPS;
            for (int idx = 0; ok && get_pair_unit(args, idx, u); ++idx) {
                for (int i = 0; i < nst; ++i) {
                    if (!mbar_wait(smem_u32(&full[s]), ph, s_abort, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_remote(peer_pfull + (uint32_t)(s * 8));
                    if (++s == stages) {
                        s = 0;
                        ph ^= 1;
                    }
                }
            }
            if (!ok) fail();
        }
    } else {
        // ------------------------------------------------------------ epilogue warps
        const int q = warp & 3;
        const int part = (warp - 2) >> 2;
        OutStage<OUTB> ostage{sOut + (size_t)(warp - 2) * OUTB * 4096, 0, &map_o, lane};
        const uint32_t peer_tempty = mapa_shared(smem_u32(tempty), 0);
        uint32_t ai = 0;
        Unit u;
        for (int idx = 0; get_pair_unit(args, idx, u); ++idx, ++ai) {
            const int b = ai & 1;
            const uint32_t aph = (ai >> 1) & 1;
            int ok = 1;
            if (lane == 0) ok = mbar_wait_sleep(smem_u32(&tfull[b]), aph, s_abort, kWaitLimitNs) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok && lane == 0) fail();
            if (epi_any_n<kEpiThreads>(!ok)) break;
            __syncwarp();
            tc_fence_after();
            const TmemSrc tsrc{tmem_base + ((uint32_t)(q * 32) << 16) + b * BN};
            Unit uh = u;                              // this CTA's 128 rows as a 128-row tile
            uh.m_tile = u.m_tile * 2 + (int)rank;
            if constexpr (EPI == EPI_F32)
                epilogue_f32_tma<BN, 1, OUTB, EPW>(args, uh, tsrc, q, ostage, part);
            else if constexpr (EPI == EPI_DOWN)
                epilogue_down_tma<BN, OUTB, EPW>(args, uh, tsrc, q, ostage, &map_o, &map_o2, part);
            else
                epilogue_qrope_blocks_tma<BN, 1, OUTB, EPW>(args, uh, tsrc, q, ostage, &map_o, &map_o2, part);
            tc_fence_before();
            if (leader) {
                mbar_arrive(smem_u32(&tempty[b]));
            } else {
                epi_bar_n<kEpiThreads>();   // every epilogue thread of this CTA has read the accumulator
                if (threadIdx.x == 64) mbar_arrive_remote(peer_tempty + (uint32_t)(b * 8));
            }
        }
        ostage.drain();
    }

    tc_fence_before();
    __syncthreads();
    if (*s_abort) {
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < 20000000ull) {
        }
    }
    cluster_sync();   // the even CTA's MMAs are complete and both CTAs have drained
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem_base, C::kTmemCols);
}

}  // namespace mla
