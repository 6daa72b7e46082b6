// The whole prolog for decode-sized token counts (T <= 128) in ONE persistent kernel: one CTA
// per SM, all CTAs co-resident (cooperative launch).  The weights (122.6 MB at DeepSeek-V3
// shapes) then stream from HBM as one continuous flow, without the launch latency, ramp-up and
// tail that every kernel boundary costs.
//
//   phase 1  down-projection x . [W^DQ | W^DKV | W^KR]: 64-column tiles x s1 k ranges, one unit
//            per CTA, fp32 products into s1 slots of T x ncols1
//   ---- grid barrier 0
//   phase 2  row work per token (CTA t < T): slot sums in fixed order, RmsNorm, RoPE(k^R), the
//            cache writes, c^Q (bf16 or int8 codes)
//   ---- grid barrier 1
//   phase 3  up-projection c^Q . W^UqQr, one head (192 columns) per CTA, full K; the epilogue
//            applies RoPE -> queryRopeOut and writes q^C (bf16) straight into shared memory as
//            the next contraction's A operand (no global round trip, no grid barrier)
//   phase 4  q^C . W^UK[n] for the same head, 512 columns -> queryOut (bf16, or int8 with the
//            row absmax scale)
//
// Shared memory holds two rings: 8 KB weight boxes (64 k-rows x 64 columns, 128-byte swizzle),
// ~20 deep in every phase, and a small ring of activation tiles.  Each MMA takes one activation
// tile and one weight box (N = 64), so a k-step's boxes may sit anywhere in the ring.
//
// Roles (224 threads): warp 0 streams the weight boxes with TMA, from phase 1 straight through
// phase 4 (weights never wait for a barrier); warp 1 issues tcgen05.mma; warps 2..5 load the
// activation tiles with ordinary 16-byte loads (so they never queue behind weight rows in the
// TMA engine), run the epilogues and the row work; warp 6 watches the grid barriers.
//
// Grid barriers: each CTA stores the call's 48-bit tag in its arrival flag; CTA 0 gathers all
// flags and stores the tag into one "done" line per CTA (128 bytes apart, so no line is polled
// by more than one CTA).  Flags from another call hold another tag, so the workspace needs no
// initialisation.  Every wait is bounded.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "finalize.cuh"
#include "gemm_tc.cuh"
#include "ptx.cuh"

namespace mla {

constexpr int kFusedThreads = 224;
constexpr int kBox = 8192;               // one weight box: 64 x 64 bf16
constexpr int kFusedMaxB = 28;           // weight-box slots
constexpr int kFusedMaxA = 8;            // activation slots
constexpr int kDoneStride = 16;          // u64 per done line (128 bytes)

struct FusedArgs {
    int T;
    int a_bytes;        // one activation tile: a_box_rows x 128 bytes
    int rb, ra;         // weight-box slots, activation slots
    // phase 1
    const __nv_bfloat16* x;  // tokenX (bf16), T x ncols_x
    int ncols_x;
    int nt1, s1, kb1, hcq;   // 64-column tiles, k ranges, k-blocks of He, W^DQ / W^DkvKr split column
    int ncols1;
    float* y1;               // s1 x T x ncols1
    // phase 2
    DownArgs down;
    // phase 3 / 4 epilogue fields (q_rope, rope tables, scales / q_out, q_scale, Hckv, N)
    GemmArgs ep;
    int N, kb2, kb4, nbox4;  // heads, k-blocks of Hcq and of D, 64-column boxes of Hckv
    // grid barriers
    unsigned long long* arrive_flags;   // 2 x G
    unsigned long long* done_flags;     // 2 x G x kDoneStride
    unsigned long long tag;
    uint32_t* status;
};

// One k-step: an activation tile and `nbox` weight boxes.
struct FStep {
    int phase;   // 1, 3, 4
    int tile;    // phase 1: 64-column tile; phases 3/4: head
    int kb;
    int nbox;
    int ks;      // phase 1: k range
    bool first;  // first k-step of the unit (the MMA overwrites the accumulator)
    bool last;   // last k-step of the unit (commit the accumulator)
};

__device__ __forceinline__ int f_steps1(const FusedArgs& a, int cta, int* kb0, int* tile, int* ks) {
    if (cta >= a.nt1 * a.s1) return 0;
    *tile = cta % a.nt1;
    *ks = cta / a.nt1;
    *kb0 = *ks * a.kb1 / a.s1;
    return (*ks + 1) * a.kb1 / a.s1 - *kb0;
}

// The i-th k-step of this CTA across phases 1, 3, 4.
__device__ __forceinline__ bool f_step(const FusedArgs& a, int i, FStep& s) {
    const int cta = blockIdx.x;
    int kb0 = 0, tile = 0, ks = 0;
    const int n1 = f_steps1(a, cta, &kb0, &tile, &ks);
    if (i < n1) {
        s = {1, tile, kb0 + i, 1, ks, i == 0, i == n1 - 1};
        return true;
    }
    i -= n1;
    if (cta >= a.N) return false;
    if (i < a.kb2) {
        s = {3, cta, i, 3, 0, i == 0, i == a.kb2 - 1};
        return true;
    }
    i -= a.kb2;
    if (i < a.kb4) {
        s = {4, cta, i, a.nbox4, 0, i == 0, i == a.kb4 - 1};
        return true;
    }
    return false;
}

// ------------------------------------------------------------------ grid barrier

// Flag accesses are relaxed; the writer fences once before its stores and the reader fences
// once after it has seen every flag (a release / acquire per access would each wait for all of
// the thread's outstanding memory operations).
__device__ __forceinline__ void flag_store(unsigned long long* f, unsigned long long tag) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(f), "l"(tag) : "memory");
}
__device__ __forceinline__ unsigned long long flag_load(const unsigned long long* f) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(f) : "memory");
    return v;
}

// After a barrier has been observed: later loads (generic or TMA) see the writes it published.
__device__ __forceinline__ void acquire_published() {
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// ------------------------------------------------------------------ loads

// Global coordinates of weight box j of step st (x = column, y = k row, z = head for W^UK).
struct BoxCoord {
    const CUtensorMap* map;
    int x, y, z;
    bool three_d;
};

__device__ __forceinline__ BoxCoord f_box(const FStep& st, int j, const FusedArgs& a, const CUtensorMap* wdq,
                                          const CUtensorMap* wdkvkr, const CUtensorMap* wuqqr,
                                          const CUtensorMap* wuk) {
    if (st.phase == 1) {
        const int col = st.tile * 64;
        return col < a.hcq ? BoxCoord{wdq, col, st.kb * kBK, 0, false}
                           : BoxCoord{wdkvkr, col - a.hcq, st.kb * kBK, 0, false};
    }
    if (st.phase == 3) return BoxCoord{wuqqr, st.tile * 192 + 64 * j, st.kb * kBK, 0, false};
    return BoxCoord{wuk, 64 * j, st.kb * kBK, st.tile, true};
}

__device__ __forceinline__ void f_load_box(const BoxCoord& b, uint32_t dst, uint32_t bar, uint64_t pol) {
    if (b.three_d)
        tma_load_3d(dst, b.map, bar, b.x, b.y, b.z, pol);
    else
        tma_load_2d(dst, b.map, bar, b.x, b.y, pol);
}

// 32 values of one row of q^C (columns col0..col0+31 of the head) -> bf16 into the K-major,
// 128-byte-swizzled shared-memory image of the next contraction's A operand: k-block col/64 at
// chain + kb * kb_bytes, row r at r * 128 bytes, 16-byte chunk c at (c ^ (r % 8)) * 16.
__device__ __forceinline__ void store_chain_chunk(uint32_t chain, int kb_bytes, int row, int col0,
                                                  const float (&v)[32]) {
#pragma unroll
    for (int c8 = 0; c8 < 4; ++c8) {
        const int d = col0 + c8 * 8;
        const uint32_t addr = chain + (uint32_t)((d >> 6) * kb_bytes + row * 128 + ((((d & 63) >> 3) ^ (row & 7)) << 4));
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr),
                     "r"(pack_bf16(v[8 * c8 + 0], v[8 * c8 + 1])), "r"(pack_bf16(v[8 * c8 + 2], v[8 * c8 + 3])),
                     "r"(pack_bf16(v[8 * c8 + 4], v[8 * c8 + 5])), "r"(pack_bf16(v[8 * c8 + 6], v[8 * c8 + 7]))
                     : "memory");
    }
}

// Phase-3 epilogue: one head (128 nope + 64 rope columns) of this thread's row.  q^R goes to
// queryRopeOut; q^C goes to the shared-memory A operand of phase 4.
template <class Src>
__device__ __forceinline__ void epilogue_qrope_chain(const GemmArgs& a, int row, int head, const Src& src,
                                                     uint32_t chain, int kb_bytes) {
    constexpr int D = 128, DR = 64, H = 32, BN = 192;
    const bool valid = row < a.T;
    const float rs = (valid && a.row_scale) ? a.row_scale[row] : 1.f;
    const float* cs = a.col_scale ? a.col_scale + (size_t)head * BN : nullptr;
#pragma unroll 1
    for (int ch = 0; ch < D / 32; ++ch) {
        float v[32];
        src.load(0, BN, ch * 32, v);
        if (valid) {
            if (cs) {
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] *= rs * cs[ch * 32 + i];
            }
            store_chain_chunk(chain, kb_bytes, row, ch * 32, v);
        }
    }
    float x0[32], x1[32];
    src.load(0, BN, D, x0);
    src.load(0, BN, D + H, x1);
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

// Shared-memory bytes of the fused kernel: alignment slack, header, one fp32 row, the phase-4
// A operand (two k-blocks), the activation ring and the weight-box ring.
__host__ __device__ inline size_t fused_smem_bytes(int ncols1, int a_bytes, int ra, int rb) {
    const size_t ys = ((size_t)ncols1 * 4 + 1023) & ~(size_t)1023;
    return 1024 + 1024 + ys + 2 * (size_t)a_bytes + (size_t)ra * a_bytes + (size_t)rb * kBox;
}

// ------------------------------------------------------------------ kernel

__global__ void __launch_bounds__(kFusedThreads, 1)
    decode_fused_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_wdq,
                        const __grid_constant__ CUtensorMap map_wdkvkr, const __grid_constant__ CUtensorMap map_cq,
                        const __grid_constant__ CUtensorMap map_wuqqr, const __grid_constant__ CUtensorMap map_wuk,
                        const FusedArgs args) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
    uint64_t* bfull = bars;                       // [kFusedMaxB]
    uint64_t* bempty = bfull + kFusedMaxB;        // [kFusedMaxB]
    uint64_t* afull = bempty + kFusedMaxB;        // [kFusedMaxA]
    uint64_t* aempty = afull + kFusedMaxA;        // [kFusedMaxA]
    uint64_t* tfull = aempty + kFusedMaxA;
    uint64_t* tempty = tfull + 1;
    uint64_t* done = tempty + 1;
    uint64_t* chain_full = done + 1;
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(chain_full + 1);
    volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
    volatile int* s_passed = reinterpret_cast<volatile int*>(s_tmem + 2);   // [2]
    float* red = reinterpret_cast<float*>(smem + 960);                      // 5 floats
    const int ys_bytes = ((args.ncols1 * 4) + 1023) & ~1023;
    float* ys = reinterpret_cast<float*>(smem + 1024);                      // one fp32 row
    const uint32_t chain = smem_u32(smem + 1024 + ys_bytes);                 // phase-4 A: 2 k-blocks
    uint8_t* aring = smem + 1024 + ys_bytes + 2 * args.a_bytes;
    uint8_t* bring = aring + (size_t)args.ra * args.a_bytes;
    const int rb = args.rb, ra = args.ra;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = gridDim.x;

    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&map_wdq);
        tma_prefetch_map(&map_wdkvkr);
        tma_prefetch_map(&map_wuqqr);
        tma_prefetch_map(&map_wuk);
        for (int s = 0; s < rb; ++s) {
            mbar_init(smem_u32(&bfull[s]), 1);
            mbar_init(smem_u32(&bempty[s]), 1);
        }
        for (int s = 0; s < ra; ++s) {
            mbar_init(smem_u32(&afull[s]), 128);   // the 128 loader threads
            mbar_init(smem_u32(&aempty[s]), 1);
        }
        mbar_init(smem_u32(tfull), 1);
        mbar_init(smem_u32(tempty), 128);
        mbar_init(smem_u32(done), 1);
        mbar_init(smem_u32(chain_full), 128);
        *s_abort = 0;
        s_passed[0] = s_passed[1] = 0;
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
    if (blockIdx.x == 0 && threadIdx.x == 64) *args.status = 0u;

    auto fail = [&]() {
        *s_abort = 1;
        atomicOr(args.status, kStatusWaitTimeout);
    };

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();
            int sb = 0;
            uint32_t phb = 0;
            bool ok = true;
            FStep st;
            for (int i = 0; ok && f_step(args, i, st); ++i) {
                for (int j = 0; j < st.nbox; ++j) {
                    if (!mbar_wait(smem_u32(&bempty[sb]), phb ^ 1, s_abort, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(&bfull[sb]);
                    mbar_arrive_expect_tx(fb, (uint32_t)kBox);
                    f_load_box(f_box(st, j, args, &map_wdq, &map_wdkvkr, &map_wuqqr, &map_wuk),
                               smem_u32(bring + (size_t)sb * kBox), fb, pol_w);
                    if (++sb == rb) {
                        sb = 0;
                        phb ^= 1;
                    }
                }
            }
            if (!ok) fail();
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(128, 64, false, true);
            int sb = 0, sa = 0;
            uint32_t phb = 0, pha = 0, acc_uses = 0;
            bool ok = true;
            FStep st;
            for (int i = 0; ok && f_step(args, i, st); ++i) {
                if (st.first) {
                    // the previous unit's epilogue has drained the accumulator
                    if (!mbar_wait(smem_u32(tempty), (acc_uses & 1) ^ 1, s_abort, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    if (st.phase == 4 && !mbar_wait(smem_u32(chain_full), 0, s_abort, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                }
                uint32_t a_base;
                if (st.phase == 4) {
                    a_base = chain + (uint32_t)(st.kb * args.a_bytes);
                } else {
                    if (!mbar_wait(smem_u32(&afull[sa]), pha, s_abort, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    a_base = smem_u32(aring + (size_t)sa * args.a_bytes);
                }
                for (int j = 0; j < st.nbox; ++j) {
                    if (!mbar_wait(smem_u32(&bfull[sb]), phb, s_abort, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t b_base = smem_u32(bring + (size_t)sb * kBox);
                    const uint32_t d = tmem_base + (uint32_t)(64 * j);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        umma_bf16(d, smem_desc_sw128(a_base + kk * 32, 16, 1024),
                                  smem_desc_sw128(b_base + kk * 16 * 128, kBox, 1024), idesc,
                                  (st.first && kk == 0) ? 0u : 1u);
                    umma_commit(smem_u32(&bempty[sb]));
                    if (++sb == rb) {
                        sb = 0;
                        phb ^= 1;
                    }
                }
                if (!ok) break;
                if (st.phase != 4) {
                    umma_commit(smem_u32(&aempty[sa]));
                    if (++sa == ra) {
                        sa = 0;
                        pha ^= 1;
                    }
                }
                if (st.last) {
                    umma_commit(smem_u32(tfull));
                    ++acc_uses;
                }
            }
            if (!ok) fail();
            umma_commit(smem_u32(done));
            mbar_wait(smem_u32(done), 0, s_abort, kWaitLimitNs / 4);
        }
    } else if (warp == 6) {
        // ------------------------------------------------------------ barrier watcher
        for (int b = 0; b < 2 && !*s_abort; ++b) {
            const uint64_t t0 = global_timer_ns();
            bool ok = true;
            if (blockIdx.x == 0) {
                // gather every CTA's arrival, then broadcast to one line per CTA
                const unsigned long long* f = args.arrive_flags + (size_t)b * G;
                while (true) {
                    bool all = true;
                    for (int c = lane; c < G; c += 32) all &= (flag_load(f + c) == args.tag);
                    if (__all_sync(0xffffffffu, all)) break;
                    if (*s_abort || global_timer_ns() - t0 > kWaitLimitNs) {
                        ok = false;
                        break;
                    }
                    __nanosleep(32);
                }
                if (ok) {
                    __threadfence();
                    for (int c = lane; c < G; c += 32)
                        flag_store(args.done_flags + ((size_t)b * G + c) * kDoneStride, args.tag);
                }
            } else {
                if (lane == 0) {
                    const unsigned long long* f = args.done_flags + ((size_t)b * G + blockIdx.x) * kDoneStride;
                    while (flag_load(f) != args.tag) {
                        if (*s_abort || global_timer_ns() - t0 > kWaitLimitNs) {
                            ok = false;
                            break;
                        }
                        __nanosleep(64);
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            }
            if (!ok) {
                if (lane == 0) fail();
                break;
            }
            __threadfence();
            if (lane == 0) s_passed[b] = 1;
            __syncwarp();
        }
    } else {
        // ------------------------------------------------------------ epilogue / row warps
        const int etid = threadIdx.x - 64;   // 0..127
        const int q = warp & 3;
        const int row_in = q * 32 + lane;
        const TmemSrc tsrc{tmem_base + ((uint32_t)(q * 32) << 16)};
        uint32_t uses = 0;
        bool ok = true;
        auto wait_acc = [&]() -> bool {
            int r = 1;
            if (lane == 0) r = mbar_wait(smem_u32(tfull), uses & 1, s_abort, kWaitLimitNs) ? 1 : 0;
            r = __shfl_sync(0xffffffffu, r, 0);
            if (!r && lane == 0) fail();
            const bool bad = epi_any(!r);
            __syncwarp();
            tc_fence_after();
            return !bad;
        };
        auto release_acc = [&]() {
            tc_fence_before();
            mbar_arrive(smem_u32(tempty));
            ++uses;
        };
        auto arrive = [&](int b) {
            __threadfence();
            epi_bar();
            if (etid == 0) flag_store(args.arrive_flags + (size_t)b * G + blockIdx.x, args.tag);
        };
        // Activation tiles of this CTA's k-steps in [first, first + n), row-major source with
        // leading dimension ld, loaded in batches so that several tiles' loads are in flight.
        int sa = 0;
        uint32_t pha = 0;
        const int rows = args.a_bytes / 128;
        const int per_thread = (rows * 8 + 127) / 128;      // 16-byte chunks per thread per tile
        const int batch = per_thread >= 8 ? 1 : 8 / per_thread;
        auto load_a = [&](const __nv_bfloat16* src, int ld, int kb0, int n) -> bool {
            for (int b0 = 0; b0 < n; b0 += batch) {
                const int nb = (n - b0) < batch ? (n - b0) : batch;
                int r = 1;
                if (etid == 0) {
                    int s2 = sa;
                    uint32_t p2 = pha;
                    for (int k = 0; k < nb && r; ++k) {
                        r = mbar_wait(smem_u32(&aempty[s2]), p2 ^ 1, s_abort, kWaitLimitNs) ? 1 : 0;
                        if (++s2 == ra) {
                            s2 = 0;
                            p2 ^= 1;
                        }
                    }
                    if (!r) fail();
                }
                if (epi_any(!r)) return false;
                uint4 v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int k = u / per_thread, c = etid + (u % per_thread) * 128;
                    const int row = c >> 3, ch = c & 7;
                    v[u] = make_uint4(0, 0, 0, 0);
                    const int col = (kb0 + b0 + k) * 64 + ch * 8;
                    if (u < nb * per_thread && row < args.T && col + 8 <= ld)
                        v[u] = __ldcg(reinterpret_cast<const uint4*>(src + (size_t)row * ld + col));
                }
                int s2 = sa;
                uint32_t p2 = pha;
                for (int k = 0; k < nb; ++k) {
                    const uint32_t slot = smem_u32(aring + (size_t)s2 * args.a_bytes);
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        if (u / per_thread != k || u >= nb * per_thread) continue;
                        const int c = etid + (u % per_thread) * 128;
                        const int row = c >> 3, ch = c & 7;
                        if (row < rows)
                            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                                             slot + (uint32_t)(row * 128 + ((ch ^ (row & 7)) << 4))),
                                         "r"(v[u].x), "r"(v[u].y), "r"(v[u].z), "r"(v[u].w)
                                         : "memory");
                    }
                    // generic-proxy shared-memory writes -> visible to the tensor core
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    mbar_arrive(smem_u32(&afull[s2]));
                    if (++s2 == ra) {
                        s2 = 0;
                        p2 ^= 1;
                    }
                }
                sa = s2;
                pha = p2;
            }
            return true;
        };
        auto wait_barrier = [&](int b) -> bool {
            const uint64_t t0 = global_timer_ns();
            int r = 1;
            while (!s_passed[b]) {
                if (*s_abort || global_timer_ns() - t0 > kWaitLimitNs) {
                    r = 0;
                    break;
                }
                __nanosleep(32);
            }
            if (!r && etid == 0) fail();
            acquire_published();
            return !epi_any(!r);
        };

        // phase 1: this CTA's k-range product of one 64-column tile
        int kb0, tile, ks;
        const int n1 = f_steps1(args, blockIdx.x, &kb0, &tile, &ks);
        if (n1 > 0) {
            ok = load_a(args.x, args.ncols_x, kb0, n1);
            if (ok) ok = wait_acc();
            if (ok) {
                GemmArgs e = args.ep;
                e.T = args.T;
                e.ncols = args.ncols1;
                e.out_f32 = args.y1;
                epilogue_f32<64, 1>(e, row_in, tile, ks, tsrc);
                release_acc();
            }
        }
        if (ok) {
            arrive(0);
            ok = wait_barrier(0);
        }
        // phase 2: row work of token t = CTA index
        if (ok) {
            for (int t = blockIdx.x; t < args.T; t += gridDim.x)
                down_row<128>(args.down, t, etid, ys, red, EpiSync{});
            arrive(1);
        }
        // phase 3: up-projection of head blockIdx.x; q^C into shared memory for phase 4
        if (ok && (int)blockIdx.x < args.N) {
            ok = wait_barrier(1);
            if (ok) ok = load_a(args.down.c_q, args.hcq, 0, args.kb2);
            if (ok) ok = wait_acc();
            if (ok) {
                epilogue_qrope_chain(args.ep, row_in, blockIdx.x, tsrc, chain, args.a_bytes);
                // generic-proxy shared-memory writes -> visible to the tensor core (async proxy)
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                mbar_arrive(smem_u32(chain_full));
                release_acc();
            }
        }
        // phase 4: W^UK contraction of head blockIdx.x
        if (ok && (int)blockIdx.x < args.N) {
            ok = wait_acc();
            if (ok) {
                Unit u{0, (int)blockIdx.x, 0, args.kb4, 0};
                epilogue_qn<512>(args.ep, u, tsrc, row_in);
                release_acc();
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (*s_abort) {
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
