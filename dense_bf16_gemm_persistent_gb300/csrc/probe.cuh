// Tensor-core rate probe: back-to-back tcgen05.mma from shared memory (no loads,
// no epilogue), timed in SM clock cycles.  It pins the per-SM, per-clock dense
// bf16 rate of an MMA shape, from which the nominal peak of the GPU follows as
// SMs x clock x rate.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace gb {

// Per scheduling unit (CTA, or CTA pair): cycles from the first MMA issued to the
// completion of the last; 0 if its wait ran out.  kProbeMaxUnits entries.
constexpr int kProbeMaxUnits = 256;
__device__ unsigned long long g_probe_cycles[kProbeMaxUnits];

// One unit issues `num_mma` MMAs of M = 128 * CG rows, N columns and K = 16 into
// TMEM accumulator 0 (or, with `alternate`, into accumulators 0 and 1 in turn),
// reading a zeroed 128 x 64 A tile and an N/CG x 64 B tile per CTA (K-major,
// 128-byte swizzle), then commits once and waits for the commit (bounded by
// `timeout_ns`).  Launched with enough dynamic shared memory that one CTA holds
// an SM, so its 512 TMEM columns are free.
template <int CG, int N>
__global__ void __launch_bounds__(128, 1) mma_rate_kernel(int num_mma, int alternate, uint64_t timeout_ns) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    constexpr int kARows = 128;
    constexpr int kBRows = N / CG;
    constexpr uint32_t kABytes = kARows * 128;
    constexpr uint32_t kBBytes = kBRows * 128;
    uint8_t* a_tile = smem;
    uint8_t* b_tile = smem + kABytes;
    uint64_t* bar = reinterpret_cast<uint64_t*>(b_tile + kBBytes);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 1);

    for (uint32_t i = threadIdx.x * 16; i < kABytes + kBBytes; i += blockDim.x * 16)
        st_shared_v4(smem_addr(smem + i), 0u, 0u, 0u, 0u);
    fence_proxy_async_smem();  // the zeros are visible to the tensor core (async proxy)
    if (threadIdx.x == 0) {
        mbar_init(smem_addr(bar), 1);
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
            constexpr uint32_t idesc = idesc_bf16_f32(128 * CG, N);
            const uint64_t adesc = sdesc_kmajor_sw128(smem_addr(a_tile));
            const uint64_t bdesc = sdesc_kmajor_sw128(smem_addr(b_tile));
            const long long c0 = clock64();
            for (int i = 0; i < num_mma; ++i) {
                const uint32_t acc_col = alternate ? static_cast<uint32_t>(i & 1) * 256u : 0u;
                const int j = i & 3;  // walk the four 16-wide K slices of the tile
                mma_bf16<CG>(tmem + acc_col, adesc + 2 * j, bdesc + 2 * j, idesc, i >= 2 ? 1u : 0u);
            }
            if constexpr (CG == 2) mma_commit_multicast2(smem_addr(bar), 0x3);
            else mma_commit<1>(smem_addr(bar));
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(smem_addr(bar), 0)) {
                if (global_timer_ns() - t0 > timeout_ns) {
                    ok = false;
                    break;
                }
            }
            const long long c1 = clock64();
            if (unit < kProbeMaxUnits) g_probe_cycles[unit] = ok ? static_cast<unsigned long long>(c1 - c0) : 0ull;
        } else {
            // the peer CTA of a pair also receives the commit's arrival: wait for it
            // before its shared memory can go away
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(smem_addr(bar), 0)) {
                if (global_timer_ns() - t0 > timeout_ns) break;
            }
        }
    }
    tc_fence_before_sync();
    if constexpr (CG == 2) cluster_sync(); else __syncthreads();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc<CG>(tmem, 512);
    }
}

}  // namespace gb
