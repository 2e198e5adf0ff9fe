// Tensor-core rate probe: back-to-back tcgen05.mma from shared memory (no loads,
// no epilogue), timed in SM clock cycles.  It pins the per-SM, per-clock dense
// bf16 rate of an MMA shape, from which the nominal peak of the GPU follows as
// SMs x clock x rate -- and, with the issue-path variants, what the issuing
// thread's own instructions between MMAs cost the tensor pipe.
#pragma once

#include <cuda.h>

#include <cstdint>

#include "ptx.cuh"

namespace gb {

// Per scheduling unit (CTA, or CTA pair): cycles from the first MMA issued to the
// completion of the last; 0 if its wait ran out.  kProbeMaxUnits entries.
constexpr int kProbeMaxUnits = 256;
__device__ unsigned long long g_probe_cycles[kProbeMaxUnits];

// What the issuing thread does around the MMAs (compile-time, so the plain loop has
// nothing else in it).  Every "per k-block" step happens once per four MMAs, as in
// the GEMM kernels' 64-wide k-blocks.
enum : int {
    kProbePlain = 0,         // MMAs only
    kProbeCommit = 1,        // + tcgen05.commit to an mbarrier per k-block (both CTAs of a pair)
    kProbeWait = 2,          // + an already-satisfied mbarrier try_wait per k-block
    kProbeFence = 3,         // + tcgen05.fence::after_thread_sync per k-block
    kProbeWaitFence = 4,     // + wait and fence per k-block
    kProbeGemmStep = 5,      // + wait, fence, descriptors from the stage index, commit: the GEMM issuer's step
    kProbeAlu = 6,           // + `alu` dependent integer operations between consecutive MMAs
    // MMAs alone while warps 1-3 of both CTAs read the other TMEM accumulator in a loop
    // (tcgen05.ld.32x32b of 16, 32 or 64 columns + wait::ld), as an epilogue does
    kProbeTmemLd16 = 7,
    kProbeTmemLd32 = 8,
    kProbeTmemLd64 = 9,
    // MMAs reading six distinct 32 KiB stages in turn (one 64-wide k-block each), as the
    // GEMM ring does, instead of one tile
    kProbeStages = 10,
    // four distinct stages, while warp 1 streams 16 KiB bulk copies from global memory
    // into a separate 32 KiB region of shared memory (the writes a TMA operand ring makes)
    kProbeStagesWrites = 11,
    // four distinct stages, while warps 1-3 write 16-byte vectors into a separate 64 KiB
    // region of shared memory as fast as they can (shared-memory bandwidth pressure)
    kProbeStagesStores = 12,
    // four distinct stages, while warp 1 (mode 13) or warps 1 and 2 (mode 14) keep
    // four 16 KiB 2-D TMA tile loads each (64 x 128 bf16 boxes, 128-byte swizzle, the
    // GEMM's operand boxes) in flight into other shared memory
    kProbeStagesTma = 13,
    kProbeStagesTma2 = 14,
    // MMAs on one tile while warps 1-3 repeat an epilogue's steps: 15 four 16-byte
    // shared-memory stores then fence.proxy.async.shared::cta and a warp sync; 16 polling
    // an mbarrier phase that never completes (mbarrier.try_wait); 17 (warp 1) 2-D TMA
    // stores of a 16 KiB shared-memory box with at most two groups pending
    kProbeFenceProxy = 15,
    kProbePoll = 16,
    kProbeTmaStore = 17,
    // MMAs on one tile with 256 threads: warps 4-7 -- one on each SMSP, warp 4 beside the
    // issuing thread's -- run 18 an FMA-heavy loop (an epilogue's activation math), 19 a
    // poll of an mbarrier that never completes (an idle epilogue's wait)
    kProbeSmspMath = 18,
    kProbeSmspPoll = 19,
    // a GEMM mainloop without an epilogue: a 6-stage ring of A and B boxes (128 rows x 64
    // each per CTA, 128-byte swizzle) filled by TMA from the probe source (L2-resident),
    // full/empty mbarriers, MMAs of each stage's four K slices, a commit per stage to the
    // empty barriers of both CTAs; producers are warp 0 (A, and the byte count) and warp 2
    // (B) of every CTA, the MMA issuer is warp 1 of the leader
    kProbePipeline = 20,
    // as kProbePlain with B MN-major (the layout of a row-major [K, N] operand: 64-column
    // blocks of 128-byte rows, one row per K index)
    kProbeMnMajor = 21,
    kProbeModes = 22,
};

// Source of the bulk copies of probe mode 11 (read only; its contents do not matter).
constexpr uint32_t kProbeSrcBytes = 1u << 20;
__device__ __align__(128) uint8_t g_probe_src[kProbeSrcBytes];

// TMEM loads completed by the leader CTA's loader warps during the run (probe modes 7-9).
__device__ unsigned long long g_probe_loads[kProbeMaxUnits];

template <int CG>
__device__ __forceinline__ void probe_commit(uint32_t bar) {
    if constexpr (CG == 2) mma_commit_multicast2(bar, 0x3);
    else mma_commit<1>(bar);
}

template <int CG, int N>
__device__ __forceinline__ void probe_pipeline(uint8_t* smem, int num_mma, uint64_t timeout_ns,
                                               const CUtensorMap& tmap) {
    constexpr uint32_t kStages = 6;
    constexpr uint32_t kABytes = 128 * 128;          // 128 rows x 64 bf16
    constexpr uint32_t kBBytes = (N / CG) * 128;
    constexpr uint32_t kStageBytes = kABytes + kBBytes;
    static_assert(1024 + kStages * kStageBytes + 32 * 8 <= 200 * 1024, "probe pipeline shared memory");
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
    uint64_t* empty = full + kStages;
    uint64_t* done_bar = empty + kStages;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = CG == 2 ? cluster_ctarank() : 0u;
    const int unit = CG == 2 ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
    const int kblocks = num_mma / 4;
    if (threadIdx.x == 0) {
        for (uint32_t i = 0; i < kStages; ++i) {
            mbar_init(smem_addr(&full[i]), 1);
            mbar_init(smem_addr(&empty[i]), 1);
        }
        mbar_init(smem_addr(done_bar), 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc<CG>(smem_addr(tmem_slot), 512);
        tmem_relinquish<CG>();
    }
    tc_fence_before_sync();
    if constexpr (CG == 2) cluster_sync(); else __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;
    if ((warp == 0 || warp == 2) && lane == 0) {
        // producers; the source rows walk the 1 MiB source in 128-row steps
        uint32_t s = 0, ph = 0;
        for (int kb = 0; kb < kblocks && ok; ++kb) {
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(smem_addr(&empty[s]), ph ^ 1u)) {
                if (global_timer_ns() - t0 > timeout_ns) { ok = false; break; }
            }
            if (!ok) break;
            const uint32_t own_full = smem_addr(&full[s]);
            const uint32_t fb = CG == 2 ? mapa_shared(own_full, 0) : own_full;
            const int32_t row = static_cast<int32_t>((static_cast<uint32_t>(kb) * 128u + rank * 256u) % 8192u);
            uint8_t* st = smem + s * kStageBytes;
            if (warp == 0) {
                if (rank == 0) mbar_arrive_expect_tx(own_full, CG * kStageBytes);
                if constexpr (CG == 2) tma_load_2d_pair(smem_addr(st), &tmap, fb, 0, row);
                else tma_load_2d(smem_addr(st), &tmap, fb, 0, row);
            } else {
                for (uint32_t h = 0; h < kBBytes / 16384u; ++h) {
                    const int32_t brow = static_cast<int32_t>((static_cast<uint32_t>(row) + 128u * (h + 1)) % 8192u);
                    if constexpr (CG == 2) tma_load_2d_pair(smem_addr(st + kABytes + h * 16384u), &tmap, fb, 0, brow);
                    else tma_load_2d(smem_addr(st + kABytes + h * 16384u), &tmap, fb, 0, brow);
                }
            }
            if (++s == kStages) { s = 0; ph ^= 1u; }
        }
        if (!ok && rank == 0) {  // drain (bounded): the last stages' loads land
            for (uint32_t i = 0; i < kStages; ++i) {
                const uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(smem_addr(&full[i]), 0) && !mbar_try_wait(smem_addr(&full[i]), 1)) {
                    if (global_timer_ns() - t0 > timeout_ns) break;
                }
            }
        }
    } else if (warp == 1 && lane == 0 && rank == 0) {
        constexpr uint32_t idesc = idesc_bf16_f32(128 * CG, N);
        uint32_t s = 0, ph = 0;
        const long long c0 = clock64();
        bool issued = false;
        for (int kb = 0; kb < kblocks; ++kb) {
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(smem_addr(&full[s]), ph)) {
                if (global_timer_ns() - t0 > timeout_ns) { ok = false; break; }
            }
            if (!ok) break;
            tc_fence_after_sync();
            const uint32_t a_addr = smem_addr(smem + s * kStageBytes);
            const uint64_t ad = sdesc_kmajor_sw128(a_addr);
            const uint64_t bd = sdesc_kmajor_sw128(a_addr + kABytes);
            mma_bf16_x4<CG>(tmem, ad, ad + 2, ad + 4, ad + 6, bd, bd + 2, bd + 4, bd + 6, idesc, kb > 0 ? 1u : 0u);
            issued = true;
            if constexpr (CG == 2) mma_commit_multicast2(smem_addr(&empty[s]), 0x3);
            else mma_commit<1>(smem_addr(&empty[s]));
            if (++s == kStages) { s = 0; ph ^= 1u; }
        }
        if (issued) {
            if constexpr (CG == 2) mma_commit_multicast2(smem_addr(done_bar), 0x3);
            else mma_commit<1>(smem_addr(done_bar));
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(smem_addr(done_bar), 0)) {
                if (global_timer_ns() - t0 > timeout_ns) { ok = false; break; }
            }
        }
        const long long c1 = clock64();
        if (unit < kProbeMaxUnits) g_probe_cycles[unit] = ok ? static_cast<unsigned long long>(c1 - c0) : 0ull;
    } else if (CG == 2 && rank == 1 && warp == 1 && lane == 0) {
        // the peer also receives the last commit: wait for it before its memory goes away
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(smem_addr(done_bar), 0)) {
            if (global_timer_ns() - t0 > timeout_ns) break;
        }
    }
    __syncwarp();
    tc_fence_before_sync();
    if constexpr (CG == 2) cluster_sync(); else __syncthreads();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc<CG>(tmem, 512);
    }
}

// One unit issues `num_mma` MMAs of M = 128 * CG rows, N columns and K = 16 into
// TMEM accumulator 0 (or, with `alternate`, into accumulators 0 and 1 in turn),
// reading a zeroed 128 x 64 A tile and an N/CG x 64 B tile per CTA (K-major,
// 128-byte swizzle), then commits once and waits for the commit (bounded by
// `timeout_ns`).  Launched with enough dynamic shared memory that one CTA holds an
// SM, so its 512 TMEM columns are free.
template <int CG, int N, int MODE>
__global__ void __launch_bounds__(256, 1) mma_rate_kernel(int num_mma, int alternate, uint64_t timeout_ns, int alu,
                                                          const __grid_constant__ CUtensorMap tmap) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    if constexpr (MODE == kProbePipeline) {
        probe_pipeline<CG, N>(smem, num_mma, timeout_ns, tmap);
        return;
    }
    constexpr int kARows = 128;
    constexpr int kBRows = N / CG;
    constexpr uint32_t kABytes = kARows * 128;
    constexpr uint32_t kBBytes = kBRows * 128;
    constexpr bool kTmaWriters = MODE == kProbeStagesTma || MODE == kProbeStagesTma2;
    constexpr bool kStaged = MODE == kProbeStages || MODE == kProbeStagesWrites || MODE == kProbeStagesStores ||
                             kTmaWriters;
    // operand stages read in turn (6 as in the GEMM ring; 4 beside the bulk-copy target)
    constexpr uint32_t kStages = MODE == kProbeStages ? 6 : (kStaged ? (MODE == kProbeStagesTma2 ? 2 : 4) : 1);
    constexpr uint32_t kStageBytes = kABytes + kBBytes;
    // bulk-copy (mode 11: four 16 KiB copies in flight), store (mode 12) or TMA (modes
    // 13, 14: four 16 KiB boxes in flight per writer warp) target
    constexpr uint32_t kWriteBytes = (MODE == kProbeStagesWrites || MODE == kProbeStagesStores || MODE == kProbeStagesTma ||
                                      MODE == kProbeFenceProxy || MODE == kProbeTmaStore)
                                         ? 65536u
                                         : MODE == kProbeStagesTma2 ? 131072u : 0u;
    // the whole layout (1 KiB alignment slack, stages, copy target, 7 barrier words) fits
    // the launch's 200 KiB of dynamic shared memory
    static_assert(1024 + kStages * kStageBytes + kWriteBytes + 16 * 8 <= 200 * 1024, "probe shared memory");
    uint8_t* a_tile = smem;
    uint8_t* b_tile = smem + kABytes;
    uint8_t* wregion = smem + kStages * kStageBytes;
    uint64_t* bar = reinterpret_cast<uint64_t*>(wregion + kWriteBytes);
    uint64_t* bar_step = bar + 1;  // per-k-block commits land here (nobody waits on it)
    uint64_t* bar_idle = bar + 2;  // never arrived: waiting on its previous phase returns at once
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 3);
    volatile int32_t* done = reinterpret_cast<volatile int32_t*>(bar + 4);    // set when the MMAs are done
    uint32_t* ld_count = reinterpret_cast<uint32_t*>(bar + 5);                // loads by warps 1-3
    uint64_t* bar_copy = bar + 6;  // 8 barriers: bulk copies (mode 11), TMA loads (4 per writer warp, modes 13-14)
    constexpr bool kLoaders = MODE >= kProbeTmemLd16 && MODE <= kProbeTmemLd64;
    constexpr int kLdCols = MODE == kProbeTmemLd16 ? 16 : MODE == kProbeTmemLd32 ? 32 : 64;

    // operands: zeros, or (bit 1 of `alternate`) bf16 values of a hash of the position,
    // exponents near 1 and both signs (the switching activity of real data)
    const bool noisy = (alternate & 2) != 0;
    for (uint32_t i = threadIdx.x * 16; i < kStages * kStageBytes; i += blockDim.x * 16) {
        uint32_t w[4] = {0u, 0u, 0u, 0u};
        if (noisy) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                uint32_t h = (i + 4u * k) * 2654435761u;
                h ^= h >> 15;
                h *= 2246822519u;
                h ^= h >> 13;
                // two bf16: sign bit, exponent 126..127, 7 random mantissa bits each
                const uint32_t lo = ((h & 1u) << 15) | ((126u + ((h >> 1) & 1u)) << 7) | ((h >> 2) & 0x7Fu);
                const uint32_t hi = (((h >> 9) & 1u) << 15) | ((126u + ((h >> 10) & 1u)) << 7) | ((h >> 11) & 0x7Fu);
                w[k] = lo | (hi << 16);
            }
        }
        st_shared_v4(smem_addr(smem + i), w[0], w[1], w[2], w[3]);
    }
    fence_proxy_async_smem();  // the zeros are visible to the tensor core (async proxy)
    if (threadIdx.x == 0) {
        mbar_init(smem_addr(bar), 1);
        mbar_init(smem_addr(bar_step), 1);
        mbar_init(smem_addr(bar_idle), 1);
        for (int i = 0; i < 8; ++i) mbar_init(smem_addr(bar_copy + i), 1);
        *done = 0;
        *ld_count = 0;
        fence_mbar_init();
    }
    const int warp = threadIdx.x >> 5;
    if (warp == 0) {
        tmem_alloc<CG>(smem_addr(tmem_slot), 512);
        tmem_relinquish<CG>();
    }
    tc_fence_before_sync();
    if constexpr (CG == 2) cluster_sync(); else __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const uint32_t rank = CG == 2 ? cluster_ctarank() : 0u;
    const int unit = CG == 2 ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);

    if (threadIdx.x == 0) {
        bool ok = true;
        if (rank == 0) {
            constexpr bool mn = MODE == kProbeMnMajor;
            constexpr uint32_t idesc = idesc_bf16_f32(128 * CG, N) | (mn ? kIdescBMnMajor : 0u);
            const uint64_t adesc = sdesc_kmajor_sw128(smem_addr(a_tile));
            // MN-major: 64-column blocks 8 KiB apart, a 16-row K slice is 2 KiB (>> 4: 128)
            const uint64_t bdesc = mn ? sdesc_mnmajor_sw128(smem_addr(b_tile), 64 * 64 * 2) : sdesc_kmajor_sw128(smem_addr(b_tile));
            constexpr uint64_t bstep = mn ? 128u : 2u;
            uint32_t x = static_cast<uint32_t>(num_mma);  // the ALU chain's value (kept live)
            const long long c0 = clock64();
            if constexpr (MODE == kProbePlain || MODE == kProbeAlu || MODE == kProbeMnMajor) {
                for (int i = 0; i < num_mma; ++i) {
                    const uint32_t acc_col = (alternate & 1) ? static_cast<uint32_t>(i & 1) * 256u : 0u;
                    const int j = i & 3;  // walk the four 16-wide K slices of the tile
                    mma_bf16<CG>(tmem + acc_col, adesc + 2 * j, bdesc + bstep * j, idesc, i >= 2 ? 1u : 0u);
                    if constexpr (MODE == kProbeAlu) {
                        for (int a = 0; a < alu; ++a) asm volatile("mad.lo.u32 %0, %0, 3, 1;" : "+r"(x));
                    }
                }
            } else {
                // four MMAs per k-block, with the per-k-block steps of MODE
                for (int kb = 0; kb < num_mma / 4; ++kb) {
                    uint64_t ad = adesc, bd = bdesc;
                    if constexpr (MODE == kProbeWait || MODE == kProbeWaitFence || MODE == kProbeGemmStep) {
                        // the phase before the first one counts as complete, so this returns at
                        // once; the bound only guards the loop
                        for (int spin = 0; spin < 1000000 && !mbar_try_wait(smem_addr(bar_idle), 1); ++spin) {
                        }
                    }
                    if constexpr (MODE == kProbeFence || MODE == kProbeWaitFence || MODE == kProbeGemmStep)
                        tc_fence_after_sync();
                    if constexpr (MODE == kProbeGemmStep) {
                        // descriptors rebuilt from a stage index every k-block, as the GEMM
                        // issuer builds them (every stage index maps to the one zeroed tile)
                        const uint32_t s = static_cast<uint32_t>(kb) % 6u;
                        const uint32_t base = smem_addr(a_tile) + (s & 0u) * 32768u;
                        ad = sdesc_kmajor_sw128(base);
                        bd = sdesc_kmajor_sw128(base + kABytes);
                    }
                    if constexpr (kStaged) {  // this k-block's own stage
                        const uint32_t base = smem_addr(a_tile) + (static_cast<uint32_t>(kb) % kStages) * kStageBytes;
                        ad = sdesc_kmajor_sw128(base);
                        bd = sdesc_kmajor_sw128(base + kABytes);
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int i = kb * 4 + j;
                        const uint32_t acc_col = (alternate & 1) ? static_cast<uint32_t>(i & 1) * 256u : 0u;
                        mma_bf16<CG>(tmem + acc_col, ad + 2 * j, bd + 2 * j, idesc, i >= 2 ? 1u : 0u);
                    }
                    if constexpr (MODE == kProbeCommit || MODE == kProbeGemmStep) probe_commit<CG>(smem_addr(bar_step));
                }
            }
            probe_commit<CG>(smem_addr(bar));
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(smem_addr(bar), 0)) {
                if (global_timer_ns() - t0 > timeout_ns) {
                    ok = false;
                    break;
                }
            }
            const long long c1 = clock64();
            *done = 1;
            if (x == 0xdeadbeefu) ok = false;  // keeps the ALU chain from being dropped
            if (unit < kProbeMaxUnits) g_probe_cycles[unit] = ok ? static_cast<unsigned long long>(c1 - c0) : 0ull;
        } else {
            // the peer CTA of a pair also receives the commits' arrivals: wait for the last
            // before its shared memory can go away
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(smem_addr(bar), 0)) {
                if (global_timer_ns() - t0 > timeout_ns) break;
            }
            *done = 1;
        }
    } else if (MODE == kProbeStagesWrites && warp == 1) {
        // writer: 16 KiB bulk copies into four slots of the write region, four in flight;
        // a slot is refilled once its previous copy has landed; stops when the MMAs are
        // done (bounded by an iteration count), after its copies in flight have landed
        if ((threadIdx.x & 31) == 0) {
            uint32_t phases = 0, n = 0;
            uint32_t pending = 0;  // one bit per slot: a copy into it is in flight
            auto land = [&](uint32_t slot) {  // wait (bounded) for the slot's copy to land
                const uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(smem_addr(bar_copy + slot), (phases >> slot) & 1u)) {
                    if (global_timer_ns() - t0 > timeout_ns) break;
                }
                phases ^= 1u << slot;
                pending &= ~(1u << slot);
            };
            for (int it = 0; it < 400000 && !*done; ++it) {
                const uint32_t slot = static_cast<uint32_t>(it & 3);
                if (pending & (1u << slot)) {
                    land(slot);
                    ++n;
                }
                mbar_arrive_expect_tx(smem_addr(bar_copy + slot), 16384u);
                bulk_load(smem_addr(wregion + slot * 16384u),
                          g_probe_src + (static_cast<uint32_t>(it) * 16384u) % kProbeSrcBytes, 16384u,
                          smem_addr(bar_copy + slot));
                pending |= 1u << slot;
            }
            for (uint32_t slot = 0; slot < 4; ++slot)  // nothing stays in flight
                if (pending & (1u << slot)) land(slot);
            if (rank == 0 && unit < kProbeMaxUnits) atomicAdd(ld_count, n);
        }
    } else if (kTmaWriters && (warp == 1 || (MODE == kProbeStagesTma2 && warp == 2))) {
        // TMA writer(s): 16 KiB 2-D boxes of the probe source (its rows at 128-row steps)
        // into four 16 KiB slots of this warp's 64 KiB part of the write region, four in
        // flight; stops when the MMAs are done, after its loads in flight have landed
        if ((threadIdx.x & 31) == 0) {
            const uint32_t wbase = static_cast<uint32_t>(warp - 1) * 65536u;
            uint64_t* bars = bar_copy + 4 * (warp - 1);
            uint32_t phases = 0, n = 0;
            uint32_t pending = 0;
            auto land = [&](uint32_t slot) {
                const uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(smem_addr(bars + slot), (phases >> slot) & 1u)) {
                    if (global_timer_ns() - t0 > timeout_ns) break;
                }
                phases ^= 1u << slot;
                pending &= ~(1u << slot);
            };
            for (int it = 0; it < 400000 && !*done; ++it) {
                const uint32_t slot = static_cast<uint32_t>(it & 3);
                if (pending & (1u << slot)) {
                    land(slot);
                    ++n;
                }
                mbar_arrive_expect_tx(smem_addr(bars + slot), 16384u);
                tma_load_2d(smem_addr(wregion + wbase + slot * 16384u), &tmap, smem_addr(bars + slot), 0,
                            static_cast<int32_t>((static_cast<uint32_t>(it) * 128u) % (kProbeSrcBytes / 128u)));
                pending |= 1u << slot;
            }
            for (uint32_t slot = 0; slot < 4; ++slot)
                if (pending & (1u << slot)) land(slot);
            if (rank == 0 && unit < kProbeMaxUnits) atomicAdd(ld_count, n);
        }
    } else if (MODE == kProbeSmspMath && warp >= 4) {
        uint32_t n = 0;
        float x = static_cast<float>(threadIdx.x) * 1e-3f, y = 0.5f;
        for (int it = 0; it < 2000000 && !*done; ++it) {
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                x = fmaf(x, 0.999f, 1e-4f);
                y = fmaf(y, x, 0.25f) * 0.5f;
            }
            ++n;
        }
        if ((threadIdx.x & 31) == 0 && rank == 0) atomicAdd(ld_count, n + (y == 12345.0f ? 1u : 0u));
    } else if (MODE == kProbeSmspPoll && warp >= 4) {
        uint32_t n = 0;
        if ((threadIdx.x & 31) == 0) {
            for (int it = 0; it < 20000000 && !*done; ++it) {
                if (mbar_try_wait(smem_addr(bar_idle), 0)) break;
                ++n;
            }
            if (rank == 0) atomicAdd(ld_count, n);
        }
        __syncwarp();
    } else if (MODE == kProbeFenceProxy && warp >= 1) {
        uint32_t n = 0;
        const uint32_t base = smem_addr(wregion) + static_cast<uint32_t>(warp - 1) * 16384u + (threadIdx.x & 31) * 64u;
        for (int it = 0; it < 2000000 && !*done; ++it) {
#pragma unroll
            for (int u = 0; u < 4; ++u) st_shared_v4(base + ((u ^ ((threadIdx.x >> 1) & 3)) << 4), it, u, n, 3u);
            fence_proxy_async_smem();
            __syncwarp();
            ++n;
        }
        if ((threadIdx.x & 31) == 0 && rank == 0) atomicAdd(ld_count, n);
    } else if (MODE == kProbePoll && warp >= 1) {
        uint32_t n = 0;
        if ((threadIdx.x & 31) == 0) {
            // phase 0 of bar_idle never completes (nothing arrives on it)
            for (int it = 0; it < 20000000 && !*done; ++it) {
                if (mbar_try_wait(smem_addr(bar_idle), 0)) break;
                ++n;
            }
            if (rank == 0) atomicAdd(ld_count, n);
        }
        __syncwarp();
    } else if (MODE == kProbeTmaStore && warp == 1) {
        // TMA stores of a 16 KiB box of shared memory into the probe source buffer, at
        // most two store groups pending
        if ((threadIdx.x & 31) == 0) {
            uint32_t n = 0;
            for (int it = 0; it < 400000 && !*done; ++it) {
                const uint32_t slot = static_cast<uint32_t>(it & 1);
                bulk_wait_group_read<1>();
                tma_store_2d(&tmap, smem_addr(wregion + slot * 16384u), 0,
                             static_cast<int32_t>((static_cast<uint32_t>(it) * 128u) % (kProbeSrcBytes / 128u)));
                bulk_commit_group();
                ++n;
            }
            bulk_wait_group<0>();
            if (rank == 0 && unit < kProbeMaxUnits) atomicAdd(ld_count, n);
        }
    } else if (MODE == kProbeStagesStores && warp >= 1) {
        // 16-byte shared-memory stores into the store region until the MMAs are done
        uint32_t n = 0;
        const uint32_t base = smem_addr(wregion) + static_cast<uint32_t>(warp - 1) * 16384u + (threadIdx.x & 31) * 16u;
        for (int it = 0; it < 4000000 && !*done; ++it) {
#pragma unroll
            for (int u = 0; u < 8; ++u)
                st_shared_v4(base + ((static_cast<uint32_t>(it) * 8u + u) & 31u) * 512u, it, u, n, 7u);
            n += 8;
        }
        if ((threadIdx.x & 31) == 0 && rank == 0) atomicAdd(ld_count, n);
    } else if (kLoaders && warp >= 1) {
        // loader warps: read accumulator 1 (columns 256..511) of this warp's lane quadrant
        // until the MMAs are done (bounded by an iteration count)
        const uint32_t base = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + 256u;
        uint32_t n = 0;
        uint32_t sink = 0;
        for (int it = 0; it < 400000 && !*done; ++it) {
            const uint32_t col = static_cast<uint32_t>(it % (256 / kLdCols)) * kLdCols;
            if constexpr (kLdCols == 16) {
                uint32_t r[16];
                tmem_ld_32x32b_x16(base + col, r);
                tmem_wait_ld();
                sink ^= r[0] ^ r[15];
            } else if constexpr (kLdCols == 32) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(base + col, r);
                tmem_wait_ld();
                sink ^= r[0] ^ r[31];
            } else {
                uint32_t r[64];
                tmem_ld_32x32b_x64(base + col, r);
                tmem_wait_ld();
                sink ^= r[0] ^ r[63];
            }
            ++n;
        }
        if ((threadIdx.x & 31) == 0) atomicAdd(ld_count, n + (sink == 0x12345678u ? 1u : 0u));
    }
    __syncthreads();
    if ((kLoaders || MODE == kProbeStagesWrites || MODE == kProbeStagesStores || kTmaWriters || MODE >= kProbeFenceProxy) &&
        threadIdx.x == 0 && rank == 0 && unit < kProbeMaxUnits)
        g_probe_loads[unit] = *ld_count;
    tc_fence_before_sync();
    if constexpr (CG == 2) cluster_sync(); else __syncthreads();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc<CG>(tmem, 512);
    }
}

}  // namespace gb
