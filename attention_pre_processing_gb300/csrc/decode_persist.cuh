// The whole bf16 prolog for decode-sized token counts in ONE persistent kernel: one CTA per SM,
// all CTAs co-resident (cooperative launch).  Every CTA streams its weights through one ring of
// 24 KB stages (three 64 x 64 boxes) from the first to the last phase, so HBM never waits for a
// kernel boundary; only the tensor-core work waits for the data it depends on.
//
//   P1   x . [W^DQ | W^DkvKr]: 192-column tiles x s1 k ranges, one unit per CTA; each unit
//        stores its fp32 product into its k-range slot of y and counts itself in on its tile's
//        counter.  Once a c^Q tile's count is complete, its CTAs add the tile's slots in k-range
//        order, one 16-column chunk each, and write bf16(gamma * y) (P3's activation) and each
//        token's sum of y^2 over the chunk
//   P3   head n = CTA index: c^Q by TMA, each 64-column k-block as soon as its four chunks are
//        written;
//        (gamma * y) . W^UqQr[:, head n]; the epilogue multiplies by the token's 1 / RMS,
//        applies RoPE to the rope columns (queryRopeOut) and writes q^C straight into shared
//        memory as P4's A operand
//   P4   q^C . W^UK[n] (512 columns) -> queryOut through TMA stores
//   KV   CTAs without a head, once the c^KV / k^R tiles are complete: the slots added in
//        k-range order, RmsNorm of c^KV and RoPE of k^R, written to the caches at cacheIndex
//
// RmsNorm(y) . W = (1 / RMS(y)) * ((gamma * y) . W): the per-token scale moves behind the
// contraction, so no row pass sits between the reduction and P3.
//
// The MMAs are M = 64 (T <= 64 token rows) by N = the weight columns: an MMA costs the same for
// M = 64 and M = 128 (its time grows with N only), reads half the token rows from shared memory,
// and puts rows 16 q .. 16 q + 15 in TMEM lanes 32 q .. 32 q + 15, so that the epilogue warp of
// lane quarter q holds tokens 16 q ..: two warps share the P1 and P3 epilogues at T = 32.  P4's
// token rows are written by the P3 epilogue itself, spread so that all four warps share P4's
// epilogue: token t sits in row 16 (t / tpq) + t % tpq, tpq = ceil(T / 4) tokens per quarter.
//
// Every sum is taken in a fixed order, so calls are bit-reproducible.  Each tile's counter is
// reset at the start of the call by the tile's first k-range CTA, which then stores the call's
// tag in the tile's flag; readers wait for the flag and a complete counter.  Flags of another
// call hold another tag, so the workspace needs no initialisation.
//
// Roles (256 threads): warp 0 streams weight stages with TMA (one 3D box of three 64-column
// blocks per stage); warp 1 allocates tensor memory and issues tcgen05.mma; warp 2 loads the
// activation tiles with TMA (x for P1, then each c^Q k-block once its chunk flags hold the call's
// tag); warp 3 is idle; warps 4..7 run the zeroing, the epilogues and the cache rows.  Every wait is bounded: a wait that gives up sets
// MLA_DEV_WAIT_TIMEOUT, the other roles stop at their next wait, tensor memory is freed and the
// kernel returns.

#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "gemm_tc.cuh"
#include "ptx.cuh"

namespace mla {

constexpr int kPThreads = 256;
constexpr int kPBox = 8192;                  // one 64 x 64 bf16 weight box
constexpr int kPStage = 3 * kPBox;           // one weight stage: up to 192 columns
constexpr int kPMaxW = 12;                   // weight stages at most
constexpr int kPA = 4;                       // P1 activation slots (TMA)
constexpr int kPA3 = 24;                     // P3 activation (c^Q) slots at most
constexpr int kPTile = 192;                  // P1 columns per tile
constexpr int kPChunk = 16;                  // columns per c^Q reduction chunk
constexpr int kPMaxT = 64;                   // tokens at most
constexpr int kPMaxS = 16;                   // k ranges at most

struct PersistArgs {
    int T, a_rows, a_bytes, wst;        // tokens, A box rows, A slot bytes, weight stages
    int na3;                            // P3 activation (c^Q) slots, <= kPA3
    int pf;                             // P3 weight stages requested into L2 beyond the ring
    // P1
    int hcq, hckv, dr, ncols1, n1, s1, kb1;
    float* y;                           // s1 k-range slots of T x ncols1 fp32 products
    unsigned int* cnt;                  // n1: k ranges of the tile stored
    unsigned long long* zflags;         // n1: the tile's counter is reset (call tag)
    __nv_bfloat16* cq;                  // T x Hcq: bf16(gamma_cq * y), P3's activation
    float* ss;                          // (Hcq / 16) x T: each c^Q chunk's sum of y^2 per token
    unsigned long long* cqflags;        // Hcq / 16: the chunk's cq and ss are written (call tag)
    const __nv_bfloat16* gamma_cq;
    const __nv_bfloat16* gamma_ckv;
    float eps_cq, eps_ckv;
    // KV
    const long long* cache_index;
    long long nslots;
    __nv_bfloat16* kv_cache;
    __nv_bfloat16* kr_cache;
    const __nv_bfloat16* rope_cos;      // (T, Dr)
    const __nv_bfloat16* rope_sin;
    // P3 / P4
    int N, kb2;                         // heads, k-blocks of Hcq
    __nv_bfloat16* q_rope;              // T x N x 64
    __nv_bfloat16* q_out;               // T x N x 512
    unsigned long long tag;             // unique per call
    uint32_t* status;
};

// One weight stage of this CTA's sequence: P1 k-blocks, then P3 k-blocks, then P4 groups.
struct PStep {
    int phase;    // 1, 3, 4
    int kb;       // k-block
    int g;        // P4: column group (0: 0..191, 1: 192..383, 2: 384..511)
    bool first;   // overwrite the accumulator
    bool last;    // last stage of the phase: commit the accumulator
};

__device__ __forceinline__ int p1_range(const PersistArgs& a, int* tile, int* ks, int* kb0) {
    const int u = blockIdx.x;
    if (u >= a.n1 * a.s1) return 0;
    *tile = u % a.n1;
    *ks = u / a.n1;
    *kb0 = *ks * a.kb1 / a.s1;
    return (*ks + 1) * a.kb1 / a.s1 - *kb0;
}

__device__ __forceinline__ bool p_step(const PersistArgs& a, int i, int n1s, PStep& s) {
    if (i < n1s) {
        s = {1, i, 0, i == 0, i == n1s - 1};
        return true;
    }
    i -= n1s;
    if ((int)blockIdx.x >= a.N) return false;
    if (i < a.kb2) {
        s = {3, i, 0, i == 0, i == a.kb2 - 1};
        return true;
    }
    i -= a.kb2;
    if (i < 6) {   // D = 128: three column groups x two k-blocks, group by group
        const int g = i / 2, kb = i % 2;
        s = {4, kb, g, kb == 0, i == 5};
        return true;
    }
    return false;
}

// ------------------------------------------------------------------ dependency flags

__device__ __forceinline__ unsigned int ld_relaxed_u32(const unsigned int* p) {
    unsigned int v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// Polls (bounded) until every lane's entries t0 + lane + 32 k (< t1) satisfy `ready`: one
// round issues all four relaxed loads before it looks at any, so a round costs one trip to
// L2, not four; a short sleep between rounds keeps the lines from being hammered.
template <typename T, typename Ready>
__device__ __forceinline__ bool poll_lanes(const T* base, int t0, int t1, Ready ready, uint64_t start,
                                           const volatile int* abort) {
    const int lane = threadIdx.x & 31;
    while (true) {
        T v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int t = t0 + lane + 32 * k;
            if constexpr (sizeof(T) == 8) v[k] = t < t1 ? ld_relaxed_u64(base + t) : T(0);
            else v[k] = t < t1 ? ld_relaxed_u32(base + t) : T(0);
        }
        bool all = true;
#pragma unroll
        for (int k = 0; k < 4; ++k) all &= t0 + lane + 32 * k >= t1 || ready(v[k]);
        if (__all_sync(0xffffffffu, all)) return true;
        if (*abort || global_timer_ns() - start > kWaitLimitNs) return false;
        __nanosleep(64);
    }
}

// Waits (bounded) until tiles t0 .. t1 - 1 are ready: the tile's flag holds `tag` and, if
// `need` > 0, its counter holds `need` (every k range stored; at most 128 tiles).  Called by
// all 128 epilogue threads together; one warp polls.  Flags first, then an acquire fence, so
// the counters read after it are this call's (the flag says the counter was reset); then the
// counters.  The named barrier releases the other warps, and every thread then takes an
// acquire fence for what the flags and counters published (a relaxed read that saw a release
// write, followed by a fence, synchronises with it).  `flags_seen`: these threads already waited
// for the same flags in this call, so only the counters are polled (one L2 round trip fewer).
__device__ __forceinline__ bool wait_tiles(const unsigned long long* zf, const unsigned int* cnt, int t0, int t1,
                                           unsigned int need, unsigned long long tag, const volatile int* abort,
                                           int etid, bool flags_seen = false) {
    bool ok = true;
    if (etid < 32) {
        const uint64_t start = global_timer_ns();
        if (!flags_seen) ok = poll_lanes(zf, t0, t1, [tag](unsigned long long v) { return v == tag; }, start, abort);
        if (ok && need > 0) {
            asm volatile("fence.acq_rel.gpu;" ::: "memory");
            ok = poll_lanes(cnt, t0, t1, [need](unsigned int v) { return v == need; }, start, abort);
        }
    }
    const bool bad = epi_any(!ok);
    asm volatile("fence.acq_rel.gpu;" ::: "memory");   // acquire: what the flags and counters published
    return !bad;
}

// Diagnostic: two waits that nothing can satisfy, so that the time limit, the status bit and the
// clean return can be tested without a fault.  which == 0: the persistent kernel's flag wait
// (wait_tiles, limit kWaitLimitNs) on a flag that never holds the tag ~0; which == 1: an
// mbarrier wait (limit 10 ms) on a barrier nothing arrives on.  One CTA of 128 threads.
__global__ void __launch_bounds__(128) wait_probe_kernel(const unsigned long long* flag, uint32_t* status, int which) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int s_abort_v;
    const int etid = threadIdx.x;
    if (etid == 0) {
        mbar_init(smem_u32(&bar), 1);
        s_abort_v = 0;
        fence_barrier_init();
    }
    __syncthreads();
    bool ok = true;
    if (which == 0) {
        ok = wait_tiles(flag, nullptr, 0, 1, 0u, ~0ull, &s_abort_v, etid);
    } else {
        if (etid == 0) ok = mbar_wait(smem_u32(&bar), 0, &s_abort_v, 10000000ull);
        ok = !epi_any(!ok);
    }
    if (!ok && etid == 0) atomicOr(status, kStatusWaitTimeout);
}

// ------------------------------------------------------------------ helpers

// 32 values of row `row` (columns col0..col0+31 of a head's q^C) -> bf16 into the K-major,
// 128-byte-swizzled A operand of P4: k-block col/64 at slot base + kb * slot_bytes.
__device__ __forceinline__ void chain_store(uint32_t base, int slot_bytes, int row, int col0, const float (&v)[32]) {
#pragma unroll
    for (int c8 = 0; c8 < 4; ++c8) {
        const int d = col0 + c8 * 8;
        const uint32_t addr =
            base + (uint32_t)((d >> 6) * slot_bytes + row * 128 + ((((d & 63) >> 3) ^ (row & 7)) << 4));
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pack_bf16(v[8 * c8], v[8 * c8 + 1])),
                     "r"(pack_bf16(v[8 * c8 + 2], v[8 * c8 + 3])), "r"(pack_bf16(v[8 * c8 + 4], v[8 * c8 + 5])),
                     "r"(pack_bf16(v[8 * c8 + 6], v[8 * c8 + 7]))
                     : "memory");
    }
}

// The activation region: P1's TMA ring, later P3's ring of na3 c^Q slots, later P4's A operand
// (two k-blocks of 64 rows x 128 bytes, so at least 16 KB).
__host__ __device__ inline size_t persist_act_bytes(int a_bytes, int na3) {
    const size_t r = (size_t)na3 * a_bytes;
    return r < 16384 ? 16384 : r;
}
constexpr int kP4Blk = 64 * 128;   // one k-block of P4's A operand (64 rows)

// Shared memory split of the persistent kernel for a given activation slot size (T token rows
// of 128 bytes): the c^Q slots first, as many of the kb2 k-blocks as leave kPMinW weight stages
// (with every k-block resident, c^Q requests never wait for the MMAs to free a slot), then the
// weight ring with the rest, and kPPre P3 stages in flight before P3 starts (ring + L2).
constexpr int kPMinW = 6;    // weight stages at least (P4's six stages in distinct slots)
constexpr int kPPre = 16;    // P3 weight stages requested before the reduction completes
struct PersistSlots {
    int na3, wst, pf;
};
__host__ __device__ inline PersistSlots persist_slots(int a_bytes, int kb2, size_t smem_limit);

// Alignment slack, barriers and a 1 KB scratch, the activation region and the weight ring.
__host__ __device__ inline size_t persist_smem_bytes(int a_bytes, int na3, int wst) {
    return 1024 + 2048 + persist_act_bytes(a_bytes, na3) + (size_t)wst * kPStage;
}

__host__ __device__ inline PersistSlots persist_slots(int a_bytes, int kb2, size_t smem_limit) {
    PersistSlots r{0, 0, 0};
    const size_t fixed = 1024 + 2048 + (size_t)kPMinW * kPStage;
    if (smem_limit <= fixed) return r;
    int na3 = (int)((smem_limit - fixed) / (size_t)a_bytes);
    if (na3 > kb2) na3 = kb2;
    if (na3 > kPA3) na3 = kPA3;
    if (na3 < 2) return r;
    int wst = (int)((smem_limit - persist_smem_bytes(a_bytes, na3, 0)) / kPStage);
    if (wst > kPMaxW) wst = kPMaxW;
    r.na3 = na3;
    r.wst = wst;
    r.pf = kPPre > wst ? kPPre - wst : 0;
    return r;
}

// ------------------------------------------------------------------ kernel

static_assert(8 * (2 * kPMaxW + 2 * kPA + 2 * kPA3 + 3 + 3 + 4) + 16 <= 1024, "barrier area");

__global__ void __launch_bounds__(kPThreads, 1)
    decode_persist_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_wdq,
                          const __grid_constant__ CUtensorMap map_wdkvkr, const __grid_constant__ CUtensorMap map_cq,
                          const __grid_constant__ CUtensorMap map_wuqqr, const __grid_constant__ CUtensorMap map_wuk,
                          const __grid_constant__ CUtensorMap map_o, const PersistArgs args) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
    uint64_t* wfull = bars;                       // [kPMaxW]
    uint64_t* wempty = wfull + kPMaxW;            // [kPMaxW]
    uint64_t* afull = wempty + kPMaxW;            // [kPA]
    uint64_t* aempty = afull + kPA;               // [kPA]
    uint64_t* afull3 = aempty + kPA;              // [kPA3]
    uint64_t* aempty3 = afull3 + kPA3;            // [kPA3]
    uint64_t* tfull = aempty3 + kPA3;             // [3]: P1, P3 accumulators ([2] unused)
    uint64_t* tfull4 = tfull + 3;                 // [3]: P4 column groups
    uint64_t* chain_full = tfull4 + 3;
    uint64_t* p1_done = chain_full + 1;          // this CTA's P1 product and chunk reductions are stored
    uint64_t* cq_all = p1_done + 1;              // warp 2 saw every c^Q chunk flag hold the tag
    uint64_t* done = cq_all + 1;
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(done + 1);
    volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
    volatile int* s_last = s_abort + 1;   // this CTA stored the last k range of its P1 tile
    float* scratch = reinterpret_cast<float*>(smem + 1024);   // 1 KB: the KV rows' warp sums
    uint8_t* aring = smem + 2048;
    uint8_t* wring = aring + persist_act_bytes(args.a_bytes, args.na3);
    const int na3 = args.na3;
    const int wst = args.wst;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = gridDim.x;
    const bool head = (int)blockIdx.x < args.N;
    int tile = 0, ks = 0, kb0 = 0;
    const int n1s = p1_range(args, &tile, &ks, &kb0);

    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&map_x);
        tma_prefetch_map(&map_cq);
        tma_prefetch_map(&map_wdq);
        tma_prefetch_map(&map_wdkvkr);
        tma_prefetch_map(&map_wuqqr);
        tma_prefetch_map(&map_wuk);
        for (int s = 0; s < wst; ++s) {
            mbar_init(smem_u32(&wfull[s]), 1);
            mbar_init(smem_u32(&wempty[s]), 1);
        }
        for (int s = 0; s < kPA; ++s) {
            mbar_init(smem_u32(&afull[s]), 1);
            mbar_init(smem_u32(&aempty[s]), 1);
        }
        for (int s = 0; s < na3; ++s) {
            mbar_init(smem_u32(&afull3[s]), 1);
            mbar_init(smem_u32(&aempty3[s]), 1);
        }
        for (int p = 0; p < 3; ++p) {
            mbar_init(smem_u32(&tfull[p]), 1);
            mbar_init(smem_u32(&tfull4[p]), 1);
        }
        mbar_init(smem_u32(chain_full), 128);
        mbar_init(smem_u32(p1_done), 1);
        mbar_init(smem_u32(cq_all), 1);
        mbar_init(smem_u32(done), 1);
        *s_abort = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(s_tmem), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *s_tmem;
    if (blockIdx.x == 0 && threadIdx.x == 32) *args.status = 0u;

    auto fail = [&]() {
        *s_abort = 1;
        atomicOr(args.status, kStatusWaitTimeout);
    };

    if (warp == 0) {
        // ------------------------------------------------------------ weight stream
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            int s = 0;
            uint32_t ph = 0;
            PStep st;
            for (int i = 0; p_step(args, i, n1s, st); ++i) {
                // a spinning wait (try_wait suspends in hardware): the refill follows the
                // slot's release at once (with the spinning accumulator waits, ~0.4 us per call
                // less than polls that sleep)
                if (!mbar_wait(smem_u32(&wempty[s]), ph ^ 1, s_abort, kWaitLimitNs)) {
                    fail();
                    break;
                }
                const uint32_t fb = smem_u32(&wfull[s]);
                const uint32_t dst = smem_u32(wring + (size_t)s * kPStage);
                // One request per stage: three 64-column blocks of 64 k rows (a block past the
                // matrix, the fourth of W^UK's last group, is zero-filled and still counted).
                mbar_arrive_expect_tx(fb, (uint32_t)kPStage);
                if (st.phase == 1) {
                    const int col = tile * 192;   // a tile never straddles W^DQ | W^DkvKr
                    if (col < args.hcq)
                        tma_load_3d(dst, &map_wdq, fb, 0, (kb0 + st.kb) * 64, col / 64, pol);
                    else
                        tma_load_3d(dst, &map_wdkvkr, fb, 0, (kb0 + st.kb) * 64, (col - args.hcq) / 64, pol);
                } else if (st.phase == 3) {
                    tma_load_3d(dst, &map_wuqqr, fb, 0, st.kb * 64, (int)blockIdx.x * 3, pol);
                } else {
                    tma_load_3d(dst, &map_wuk, fb, 0, (int)blockIdx.x * 128 + st.kb * 64, st.g * 3, pol);
                }
                if (++s == wst) {
                    s = 0;
                    ph ^= 1;
                }
                // The ring now holds the first P3 stages, which wait for the reduction: while HBM
                // idles, the next pf P3 stages are requested into L2 (all of P3 / P4 would load L2
                // enough to stretch the reduction's dependency chain).
                if (head && i == n1s + wst - 1) {
                    const uint64_t keep = policy_evict_last();
                    PStep pf;
                    for (int k = i + 1; k <= i + args.pf && p_step(args, k, n1s, pf); ++k)
                        if (pf.phase == 3) tma_prefetch_l2_3d(&map_wuqqr, 0, pf.kb * 64, (int)blockIdx.x * 3, keep);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // One explicit loop per phase; the operand descriptors are built once and advanced by
        // constant offsets (their start-address field counts 16-byte units), so that a stage
        // costs little more than its four MMAs.
        if (lane == 0) {
            constexpr uint32_t id192 = idesc_bf16_f32(64, 192, false, true);
            constexpr uint32_t id128 = idesc_bf16_f32(64, 128, false, true);
            const uint64_t adesc0 = smem_desc_sw128(smem_u32(aring), 16, 1024);
            const uint64_t bdesc0 = smem_desc_sw128(smem_u32(wring), kPBox, 1024);
            const uint64_t a_unit = (uint64_t)(args.a_bytes >> 4);   // one activation slot
            constexpr uint64_t w_unit = kPStage >> 4;                 // one weight stage
            int sw = 0;
            uint32_t phw = 0;
            bool ok = true;
            // The next weight stage has landed.
            auto wait_w = [&]() -> bool { return mbar_wait(smem_u32(&wfull[sw]), phw, s_abort, kWaitLimitNs); };
            // One weight stage: K = 64 (four k16 MMAs) into accumulator columns d; returns the
            // ring slot to release once they complete.
            auto mma4 = [&](uint64_t adesc, uint32_t d, uint32_t idesc, bool first) -> int {
                tc_fence_after();
                const uint64_t bdesc = bdesc0 + (uint64_t)sw * w_unit;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    umma_bf16(d, adesc + 2 * kk, bdesc + 128 * kk, idesc, (first && kk == 0) ? 0u : 1u);
                const int used = sw;
                if (++sw == wst) {
                    sw = 0;
                    phw ^= 1;
                }
                return used;
            };
            // Each loop waits for the NEXT stage's operands while the tensor core runs this
            // stage's MMAs, and only then queues the commits that release this stage: the
            // tcgen05 queue is short, so a wait placed after the commits would leave the tensor
            // core idle for its duration every stage.
            // P1: activation slots filled by TMA
            {
                int sa = 0;
                uint32_t pha = 0;
                if (n1s > 0) ok = mbar_wait(smem_u32(&afull[0]), 0, s_abort, kWaitLimitNs) && wait_w();
                for (int i = 0; ok && i < n1s; ++i) {
                    const int used_w = mma4(adesc0 + (uint64_t)sa * a_unit, tmem_base + 256, id192, i == 0);
                    const int used_a = sa;
                    if (++sa == kPA) {
                        sa = 0;
                        pha ^= 1;
                    }
                    if (i + 1 < n1s) ok = mbar_wait(smem_u32(&afull[sa]), pha, s_abort, kWaitLimitNs) && wait_w();
                    umma_commit(smem_u32(&wempty[used_w]));
                    umma_commit(smem_u32(&aempty[used_a]));
                }
                if (ok && n1s > 0) umma_commit(smem_u32(&tfull[0]));
            }
            if (head) {
                // P3: activation slots filled by TMA (c^Q), two k-blocks per round: eight MMAs
                // between waits keep the tensor core's short queue from draining (kb2 is even)
                int sa = 0;
                uint32_t pha = 0;
                for (int kb = 0; ok && kb < args.kb2; kb += 2) {
                    const int sa1 = sa + 1 == na3 ? 0 : sa + 1;
                    const uint32_t pha1 = sa + 1 == na3 ? pha ^ 1 : pha;
                    const int sw1 = sw + 1 == wst ? 0 : sw + 1;
                    const uint32_t phw1 = sw + 1 == wst ? phw ^ 1 : phw;
                    ok = mbar_wait(smem_u32(&afull3[sa]), pha, s_abort, kWaitLimitNs) && wait_w() &&
                         mbar_wait(smem_u32(&afull3[sa1]), pha1, s_abort, kWaitLimitNs) &&
                         mbar_wait(smem_u32(&wfull[sw1]), phw1, s_abort, kWaitLimitNs);
                    if (!ok) break;
                    const int uw0 = mma4(adesc0 + (uint64_t)sa * a_unit, tmem_base, id192, kb == 0);
                    const int uw1 = mma4(adesc0 + (uint64_t)sa1 * a_unit, tmem_base, id192, false);
                    umma_commit(smem_u32(&wempty[uw0]));
                    umma_commit(smem_u32(&aempty3[sa]));
                    umma_commit(smem_u32(&wempty[uw1]));
                    umma_commit(smem_u32(&aempty3[sa1]));
                    sa = sa1 + 1 == na3 ? 0 : sa1 + 1;
                    pha = sa1 + 1 == na3 ? pha1 ^ 1 : pha1;
                }
                if (ok) umma_commit(smem_u32(&tfull[1]));
                // P4: A = q^C, two 64-row k-blocks at the start of the activation region; column
                // group by column group (both k-blocks), each group's accumulator committed on
                // its own so that its epilogue overlaps the next groups' MMAs
                ok = ok && mbar_wait(smem_u32(chain_full), 0, s_abort, kWaitLimitNs) && wait_w();
                for (int g = 0; ok && g < 3; ++g) {
                    const uint32_t id = g == 2 ? id128 : id192;
                    const int u0 = mma4(adesc0, tmem_base + 192 * g, id, true);
                    ok = wait_w();
                    int u1 = -1;
                    if (ok) u1 = mma4(adesc0 + (kP4Blk >> 4), tmem_base + 192 * g, id, false);
                    if (ok && g < 2) ok = wait_w();
                    umma_commit(smem_u32(&wempty[u0]));
                    if (u1 >= 0) umma_commit(smem_u32(&wempty[u1]));
                    if (ok) umma_commit(smem_u32(&tfull4[g]));
                }
            }
            if (!ok) fail();
            umma_commit(smem_u32(done));
            mbar_wait(smem_u32(done), 0, s_abort, kWaitLimitNs / 4);
        }
    } else if (warp == 2) {
        // ------------------------------------------------------------ activation tiles
        const uint64_t pol = policy_evict_last();
        bool ok = true;
        if (lane == 0) {
            int sa = 0;
            uint32_t ph = 0;
            for (int i = 0; ok && i < n1s; ++i) {
                if (!mbar_wait_sleep(smem_u32(&aempty[sa]), ph ^ 1, s_abort, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                const uint32_t fb = smem_u32(&afull[sa]);
                mbar_arrive_expect_tx(fb, (uint32_t)args.a_bytes);
                tma_load_2d(smem_u32(aring + (size_t)sa * args.a_bytes), &map_x, fb, (kb0 + i) * 64, 0, pol);
                if (++sa == kPA) {
                    sa = 0;
                    ph ^= 1;
                }
            }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (ok && head) {
            // P3's activation tiles: c^Q k-block kb is requested as soon as its four 16-column
            // chunk flags hold the call's tag (the chunks are reduced in parallel by other CTAs,
            // so early k-blocks need not wait for the last chunk).  Polling starts once this
            // CTA's own P1 work is stored (the other CTAs finish theirs at about the same time;
            // earlier polling only loads L2 while the reductions run).  One round loads every chunk
            // flag not yet seen (four per lane): one trip to L2; the longest prefix of set flags
            // gives the k-blocks that may be requested, in order.  c^Q was written by
            // other CTAs' ordinary stores and is read here by the TMA engine: a relaxed read that
            // saw the release, an acquire fence, then the proxy fence.  Once every flag is seen,
            // cq_all tells the epilogue warps (their 1 / RMS needs every chunk's sum of squares).
            if (lane == 0) ok = mbar_wait_sleep(smem_u32(p1_done), 0, s_abort, kWaitLimitNs);
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            const int nchunks = args.hcq / kPChunk;   // <= 128
            int seen = 0;     // chunk flags seen, in order
            int issued = 0;   // k-blocks requested
            const uint64_t t0 = global_timer_ns();
            while (ok && issued < args.kb2) {
                if (seen < nchunks) {
                    bool set[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int c = seen + lane + 32 * k;
                        set[k] = c >= nchunks || ld_relaxed_u64(args.cqflags + c) == args.tag;
                    }
                    int run = 0;   // consecutive set flags from `seen` on
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const unsigned m = __ballot_sync(0xffffffffu, set[k]);
                        if (run == 32 * k) run += m == 0xffffffffu ? 32 : __ffs(~m) - 1;
                    }
                    if (run > 0) {
                        seen = min(nchunks, seen + run);
                        asm volatile("fence.acq_rel.gpu;" ::: "memory");
                        if (seen == nchunks && lane == 0) mbar_arrive(smem_u32(cq_all));
                    }
                }
                const int ready = seen / 4;   // k-blocks whose four chunks are written
                if (ready > issued) {
                    if (lane == 0) {
                        asm volatile("fence.proxy.async;" ::: "memory");
                        for (; ok && issued < ready; ++issued) {
                            const int s3 = issued % na3;
                            if (issued >= na3 && !mbar_wait_sleep(smem_u32(&aempty3[s3]), ((issued / na3) & 1) ^ 1,
                                                                   s_abort, kWaitLimitNs)) {
                                ok = false;
                                break;
                            }
                            const uint32_t fb = smem_u32(&afull3[s3]);
                            mbar_arrive_expect_tx(fb, (uint32_t)args.a_bytes);
                            tma_load_2d(smem_u32(aring + (size_t)s3 * args.a_bytes), &map_cq, fb, issued * 64, 0, pol);
                        }
                    }
                    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                    issued = __shfl_sync(0xffffffffu, issued, 0);
                } else {
                    // nothing new: give up at the limit (lane 0 decides for the warp)
                    int stop = 0;
                    if (lane == 0) stop = (*s_abort || global_timer_ns() - t0 > kWaitLimitNs) ? 1 : 0;
                    if (__shfl_sync(0xffffffffu, stop, 0)) ok = false;
                    else __nanosleep(128);
                }
            }
        }
        if (!ok && lane == 0) fail();
    } else if (warp == 3) {
        // idle
    } else {
        // ------------------------------------------------------------ epilogue warps
        const int etid = threadIdx.x - 128;   // 0..127
        const int q = warp & 3;               // TMEM lane quarter
        const int row = q * 16 + lane;        // the token of this lane in P1 / P3 (M = 64 layout)
        const int T = args.T;
        const bool rowok = lane < 16 && row < T;
        const int tpq = (T + 3) / 4;          // P4: tokens per lane quarter
        bool ok = true;
        // Accumulator waits spin (they are on the dependency chain); the others sleep.
        auto acc_ready = [&](int p) -> bool {
            int r = 1;
            if (lane == 0) r = mbar_wait(smem_u32(&tfull[p]), 0, s_abort, kWaitLimitNs) ? 1 : 0;
            r = __shfl_sync(0xffffffffu, r, 0);
            __syncwarp();
            tc_fence_after();
            return r != 0;
        };
        const int ncq = args.hcq / kPTile;    // P1 tiles of c^Q columns; the rest are c^KV | k^R

        // ---- counter reset: the first k-range CTA of each P1 tile zeroes the tile's counter,
        // then stores the call's tag in the tile's flag (release: the named barrier orders the
        // reset before it)
        if ((int)blockIdx.x < args.n1) {
            const int zt = blockIdx.x;
            if (etid == 0) *reinterpret_cast<volatile unsigned int*>(args.cnt + zt) = 0u;
            epi_bar();
            if (etid == 0)
                asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(args.zflags + zt), "l"(args.tag) : "memory");
        }

        // ---- P1: this CTA's k-range product of one 192-column tile, into its k-range slot of y
        if (n1s > 0) {
            const size_t slot_stride = (size_t)T * args.ncols1;
            // the counter is reset (long before the product is ready: the wait overlaps P1)
            ok = wait_tiles(args.zflags, args.cnt, tile, tile + 1, 0u, args.tag, s_abort, etid);
            ok = acc_ready(0) && ok;
            ok = !epi_any(!ok);
            // The warps whose TMEM lanes hold rows < T stage the product in shared memory (P1's
            // activation slots: its MMAs have completed), then all 128 threads store it with
            // coalesced 16-byte stores (a row-per-thread pattern would send one L2 request per
            // 16 bytes).  The staging row stride (196 floats) spreads the row writes over banks.
            constexpr int kStg = kPTile + 4;
            float* stg = reinterpret_cast<float*>(aring);
            if (ok && q * 16 < T) {
#pragma unroll 1
                for (int ch = 0; ch < kPTile / 32; ++ch) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(q * 32) << 16) + 256 + ch * 32, r);
                    tmem_ld_wait();
                    if (rowok) {
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            *reinterpret_cast<uint4*>(stg + row * kStg + ch * 32 + 4 * i) =
                                make_uint4(r[4 * i], r[4 * i + 1], r[4 * i + 2], r[4 * i + 3]);
                    }
                }
            }
            epi_bar();
            if (ok) {
                float* dst = args.y + ks * slot_stride + tile * kPTile;
                for (int i = etid; i < T * (kPTile / 4); i += 128) {
                    const int r = i / (kPTile / 4), c4 = i % (kPTile / 4);
                    *reinterpret_cast<float4*>(dst + (size_t)r * args.ncols1 + 4 * c4) =
                        *reinterpret_cast<const float4*>(stg + r * kStg + 4 * c4);
                }
            }
            // Count this k range in: the named barrier orders every thread's stores before
            // thread 0's release.
            epi_bar();
            if (etid == 0) {
                unsigned int old = 0;
                if (ok) asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(args.cnt + tile) : "memory");
                *s_last = ok && old + 1 == (unsigned int)args.s1 ? 1 : 0;
            }
            epi_bar();
            constexpr int kChunks = kPTile / kPChunk;   // chunks per tile
            if (ok && tile < ncq && ks < kChunks) {
                // The tile's CTAs reduce it, chunk c by the CTAs with c = ks (mod s1): once every
                // k range is stored (the CTA that completed the count knows at once, the others
                // wait for the counter), the chunk's slots are added in k-range order,
                // bf16(gamma * y) goes to cq and each token's sum of y^2 over the chunk to ss;
                // then the chunk's flag.
                // (the tile's flag was seen before the slot was stored)
                if (!*s_last)
                    ok = wait_tiles(args.zflags, args.cnt, tile, tile + 1, (unsigned int)args.s1, args.tag, s_abort, etid, true);
                else asm volatile("fence.acq_rel.gpu;" ::: "memory");
                for (int c = ks; ok && c < kChunks; c += args.s1) {
                    const int col0 = tile * kPTile + c * kPChunk;
                    // four threads per row, one float4 each; 32 rows per round
                    const int f4 = etid & 3, rsub = etid >> 2;
                    const int col = col0 + 4 * f4;
                    const uint2 g = *reinterpret_cast<const uint2*>(args.gamma_cq + col);
                    for (int r0 = 0; r0 < T; r0 += 32) {
                        const int r = r0 + rsub;
                        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                        if (r < T) {
                            const float* src = args.y + (size_t)r * args.ncols1 + col;
                            float4 w[kPMaxS];
#pragma unroll
                            for (int j = 0; j < kPMaxS; ++j)
                                if (j < args.s1) w[j] = __ldcg(reinterpret_cast<const float4*>(src + j * slot_stride));
#pragma unroll
                            for (int j = 0; j < kPMaxS; ++j)   // k-range order
                                if (j < args.s1) {
                                    v.x += w[j].x;
                                    v.y += w[j].y;
                                    v.z += w[j].z;
                                    v.w += w[j].w;
                                }
                            uint2 o;
                            o.x = pack_bf16(bf16_lo(g.x) * v.x, bf16_hi(g.x) * v.y);
                            o.y = pack_bf16(bf16_lo(g.y) * v.z, bf16_hi(g.y) * v.w);
                            *reinterpret_cast<uint2*>(args.cq + (size_t)r * args.hcq + col) = o;
                        }
                        float s2 = v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
                        s2 += __shfl_xor_sync(0xffffffffu, s2, 1);
                        s2 += __shfl_xor_sync(0xffffffffu, s2, 2);
                        if (f4 == 0 && r < T) args.ss[(size_t)(col0 / kPChunk) * T + r] = s2;
                    }
                    epi_bar();
                    if (etid == 0)
                        asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(args.cqflags + col0 / kPChunk), "l"(args.tag)
                                     : "memory");
                }
            }
        }
        if (!ok) fail();
        ok = !epi_any(!ok);   // uniform over the 128 threads: the waits below are collective
        if (etid == 0) mbar_arrive(smem_u32(p1_done));   // warp 2 may start polling the chunk flags

        if (ok && head) {
            // Every c^Q chunk is written (warp 2 saw every flag; P3's MMAs wait for their own
            // k-blocks only), so each row's 1 / RMS from the chunks' sums of y^2 (in chunk order)
            {
                int r = 1;
                if (lane == 0) r = mbar_wait_sleep(smem_u32(cq_all), 0, s_abort, kWaitLimitNs) ? 1 : 0;
                ok = __shfl_sync(0xffffffffu, r, 0) != 0;
                ok = !epi_any(!ok);
            }
            // This row's RoPE tables, loaded before P3's product is ready
            uint4 rcs[16];
            if (ok && rowok) {
                const uint4* cp = reinterpret_cast<const uint4*>(args.rope_cos + (size_t)row * 64);
                const uint4* sp = reinterpret_cast<const uint4*>(args.rope_sin + (size_t)row * 64);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    rcs[i] = cp[i];
                    rcs[8 + i] = sp[i];
                }
            }
            float inv = 0.f;
            if (ok && rowok) {
                float s2 = 0.f;
                for (int c = 0; c < args.hcq / kPChunk; ++c) s2 += __ldcg(args.ss + (size_t)c * T + row);
                inv = 1.f / sqrtf(s2 / (float)args.hcq + args.eps_cq);
            }
            // ---- P3 epilogue: 1 / RMS per token, RoPE -> queryRopeOut, q^C -> P4's A operand
            // (token `row` in P4 row 16 (row / tpq) + row % tpq)
            // Every TMEM column of P3 (q^C and the rope part) is read before P4 may start (its
            // first group's accumulator reuses those columns); RoPE and the queryRopeOut stores
            // then run beside P4's MMAs.
            ok = acc_ready(1);
            const bool act = ok && q * 16 < T;   // warp-uniform
            float x0[32], x1[32];
            if (act) {
                const TmemSrc src{tmem_base + ((uint32_t)(q * 32) << 16)};
                const uint32_t chain = smem_u32(aring);
                const int prow = 16 * (row / tpq) + row % tpq;
#pragma unroll 1
                for (int ch = 0; ch < 4; ++ch) {
                    float v[32];
                    src.load(0, 0, ch * 32, v);
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] *= inv;
                    if (rowok) chain_store(chain, kP4Blk, prow, ch * 32, v);
                }
                src.load(0, 0, 128, x0);
                src.load(0, 0, 160, x1);
            }
            fence_proxy_async_smem();   // q^C written by threads, read by the tensor core
            tc_fence_before();
            mbar_arrive(smem_u32(chain_full));
            if (act) {
                if (rowok) {
                    float o0[32], o1[32];
#pragma unroll
                    for (int qq = 0; qq < 4; ++qq) {
                        const uint4 c0 = rcs[qq], c1 = rcs[qq + 4], s0 = rcs[8 + qq], s1 = rcs[8 + qq + 4];
                        const uint32_t cw0[4] = {c0.x, c0.y, c0.z, c0.w}, cw1[4] = {c1.x, c1.y, c1.z, c1.w};
                        const uint32_t sw0[4] = {s0.x, s0.y, s0.z, s0.w}, sw1[4] = {s1.x, s1.y, s1.z, s1.w};
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int j = qq * 8 + e;
                            const float cj = (e & 1) ? bf16_hi(cw0[e >> 1]) : bf16_lo(cw0[e >> 1]);
                            const float sj = (e & 1) ? bf16_hi(sw0[e >> 1]) : bf16_lo(sw0[e >> 1]);
                            const float ch = (e & 1) ? bf16_hi(cw1[e >> 1]) : bf16_lo(cw1[e >> 1]);
                            const float sh = (e & 1) ? bf16_hi(sw1[e >> 1]) : bf16_lo(sw1[e >> 1]);
                            const float a0 = x0[j] * inv, a1 = x1[j] * inv;
                            o0[j] = a0 * cj - a1 * sj;
                            o1[j] = a1 * ch + a0 * sh;
                        }
                    }
                    __nv_bfloat16* dst = args.q_rope + ((size_t)row * args.N + blockIdx.x) * 64;
                    store_bf16_chunk(dst, o0, 32);
                    store_bf16_chunk(dst + 32, o1, 32);
                }
            }

            // ---- P4 epilogue: queryOut through shared memory and TMA stores (boxes of the warp's
            // tpq tokens x 64 columns), group by group.  Staging: the ring slots of P4's first two
            // weight stages (the last phase: once group 0 is complete they are never loaded
            // again); 8 KB per warp, two warps per slot.
            {
                const int slot = (n1s + args.kb2 + (q >> 1)) % wst;
                OutStage<2> out{wring + (size_t)slot * kPStage + (size_t)(q & 1) * 2 * 4096, 0, &map_o, lane};
                const TmemSrc src{tmem_base + ((uint32_t)(q * 32) << 16)};
                for (int g = 0; ok && g < 3; ++g) {
                    int r = 1;
                    if (lane == 0) r = mbar_wait(smem_u32(&tfull4[g]), 0, s_abort, kWaitLimitNs) ? 1 : 0;
                    ok = __shfl_sync(0xffffffffu, r, 0) != 0;
                    __syncwarp();
                    tc_fence_after();
                    if (!ok || q * tpq >= T) continue;
#pragma unroll 1
                    for (int j = 3 * g; j < (g == 2 ? 8 : 3 * g + 3); ++j) {
                        uint32_t w[32];
                        float v[32];
                        src.load(0, 0, 64 * j, v);
#pragma unroll
                        for (int i = 0; i < 16; ++i) w[i] = pack_bf16(v[2 * i], v[2 * i + 1]);
                        src.load(0, 0, 64 * j + 32, v);
#pragma unroll
                        for (int i = 0; i < 16; ++i) w[16 + i] = pack_bf16(v[2 * i], v[2 * i + 1]);
                        out.put(w, (int)blockIdx.x * 512 + 64 * j, q * tpq);
                    }
                }
                if (q * tpq < T) out.drain();
            }
        }

        // ---- KV: the cache rows, by the CTAs without a head (or by every CTA if none is free),
        // once the c^KV | k^R tiles are complete
        ok = !epi_any(!ok);
        if (ok && args.nslots > 0) {
            const int spare = G - args.N;
            const int first = spare > 0 ? (int)blockIdx.x - args.N : (int)blockIdx.x;
            const int step = spare > 0 ? spare : G;
            const int h = args.dr / 2;
            if (first >= 0 && first < T)
                ok = wait_tiles(args.zflags, args.cnt, ncq, args.n1, (unsigned int)args.s1, args.tag, s_abort, etid);
            if (ok && first >= 0) {
                float* wsum = scratch;   // the four warps' sums of squares
                for (int t = first; t < T; t += step) {
                    const long long slot = args.cache_index[t];
                    if (slot < 0 || slot >= args.nslots) {   // the same for every thread
                        if (etid == 0) atomicOr(args.status, kStatusCacheIndexRange);
                        continue;
                    }
                    // y of this token's c^KV | k^R columns: the k-range slots added in order
                    const float* yr = args.y + (size_t)t * args.ncols1 + args.hcq;
                    const size_t slot_stride = (size_t)T * args.ncols1;
                    float4 v = __ldcg(reinterpret_cast<const float4*>(yr) + etid);
                    float kr0 = 0.f, kr1 = 0.f;
                    if (etid < h) {
                        kr0 = __ldcg(yr + args.hckv + etid);
                        kr1 = __ldcg(yr + args.hckv + etid + h);
                    }
                    for (int j = 1; j < args.s1; ++j) {
                        const float* yj = yr + j * slot_stride;
                        const float4 w = __ldcg(reinterpret_cast<const float4*>(yj) + etid);
                        v.x += w.x;
                        v.y += w.y;
                        v.z += w.z;
                        v.w += w.w;
                        if (etid < h) {
                            kr0 += __ldcg(yj + args.hckv + etid);
                            kr1 += __ldcg(yj + args.hckv + etid + h);
                        }
                    }
                    // RmsNorm of c^KV: four of the Hckv = 512 values per thread
                    float s2 = v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, o);
                    if (lane == 0) wsum[q] = s2;
                    epi_bar();
                    const float inv = 1.f / sqrtf(((wsum[0] + wsum[1]) + (wsum[2] + wsum[3])) / (float)args.hckv + args.eps_ckv);
                    const uint2 g = *reinterpret_cast<const uint2*>(args.gamma_ckv + 4 * etid);
                    uint2 o;
                    o.x = pack_bf16(bf16_lo(g.x) * v.x * inv, bf16_hi(g.x) * v.y * inv);
                    o.y = pack_bf16(bf16_lo(g.y) * v.z * inv, bf16_hi(g.y) * v.w * inv);
                    *reinterpret_cast<uint2*>(args.kv_cache + slot * args.hckv + 4 * etid) = o;
                    // RoPE of k^R
                    if (etid < h) {
                        const __nv_bfloat16* cs = args.rope_cos + (size_t)t * args.dr;
                        const __nv_bfloat16* sn = args.rope_sin + (size_t)t * args.dr;
                        __nv_bfloat16* dkr = args.kr_cache + slot * args.dr;
                        const float x0 = kr0, x1 = kr1;
                        dkr[etid] = __float2bfloat16_rn(x0 * __bfloat162float(cs[etid]) - x1 * __bfloat162float(sn[etid]));
                        dkr[etid + h] =
                            __float2bfloat16_rn(x1 * __bfloat162float(cs[etid + h]) + x0 * __bfloat162float(sn[etid + h]));
                    }
                    epi_bar();   // wsum is reused by the next token
                }
            }
        }
        if (!ok && etid == 0) fail();
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
        tmem_dealloc(tmem_base, 512);
    }
}

}  // namespace mla
