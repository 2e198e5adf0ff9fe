// Persistent, warp-specialised bf16 GEMM with a fused epilogue for sm_103a.
//
//   D[m,n] = bf16( epi( sum_k A[m,k] B[n,k] ) )        (one B operand: linear)
//   D[m,n] = bf16( silu(sum_k A B1) * sum_k A B2 )      (two B operands: Llama FFN)
//
// Design (the techniques are the ones "Automate performant Hopper matmul",
// NVIDIA/Fuser issue #3819, lists for its Hopper kernel; here they are mapped
// to tcgen05/TMEM):
//   * warp 0 lane 0  -- producer: TMA loads of A and B tiles into an S-stage
//                       shared-memory ring (section "K loop efficiency":
//                       pipelining with several stages in flight).
//   * warp 1         -- allocates TMEM; lane 0 issues tcgen05.mma into a
//                       double-buffered fp32 accumulator and tcgen05.commit
//                       to release each stage once (section "Syncing issues":
//                       one commit per stage, one per tile).
//   * warps 4..7     -- epilogue: tcgen05.ld of 32-column chunks, bias,
//                       activation, epilogue input, bf16 rounding, and a
//                       chunked TMA store whose shared-memory wait is delayed
//                       until the buffer is reused (sections "Epilogue inputs"
//                       and "TMA store and stmatrix").
//   * all barriers are initialised once, outside the persistent tile loop, and
//     the ring position comes from a k-block counter that runs on across
//     tiles (section "Syncing persistent matmuls").
//   * the persistent tile loop walks tiles in groups of `group_m` tile-rows
//     with a serpentine over tile-columns, and reverses the K direction on
//     every other tile of a CTA when `zigzag` is set (section "Operand load
//     efficiency/L2 locality/grid swizzling").
// Every wait is bounded in time; a wait that runs out records an error code in
// the device status word, raises a CTA-wide abort flag, and the kernel drains
// its in-flight copies and MMAs, frees TMEM and returns.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include <cstdint>

#include "ptx.cuh"

namespace gb {

constexpr int kBM = 128;          // tile rows (TMEM lanes)
constexpr int kBK = 64;           // k-block: 64 bf16 = one 128-byte swizzle row
constexpr int kThreads = 256;     // 8 warps: producer, MMA, 2 spare, 4 epilogue
constexpr int kEpiWarp0 = 4;
constexpr int kTmemCols = 512;    // two accumulator buffers of 256 columns
constexpr int kAccStride = 256;
constexpr int kDChunk = 32;       // epilogue chunk: 32 columns
constexpr int kDStageBytes = 32 * kDChunk * 2;  // one warp's 32x32 bf16 staging box

enum : uint32_t {
    kFlagBias = 1u,
    kFlagResidual = 2u,
    kFlagDTma = 4u,      // D stored by TMA (16-byte aligned rows)
    kFlagRVec = 8u,      // R rows 16-byte aligned: vector loads
    kFlagBiasVec = 16u,  // bias 16-byte aligned: vector loads
};

// Codes written to the device status word (low byte = gb_status_t).
enum : uint32_t { kStatusTimeout = 4u };
enum : uint32_t { kRoleProducer = 1u, kRoleMma = 2u, kRoleEpilogue = 3u };

enum : int { kInjectNone = 0, kInjectSkipFirstStage = 1 };

struct GemmParams {  // the CUtensorMap members give it their 64-byte alignment
    CUtensorMap tm_a;   // A [M, K], box {64, 128}, 128B swizzle
    CUtensorMap tm_b0;  // B (or W1) [N, K], box {64, BN}, 128B swizzle
    CUtensorMap tm_b1;  // W3 [N, K] (FFN only)
    CUtensorMap tm_d;   // D [M, N], box {32, 32}, 64B swizzle (TMA store path)
    const uint16_t* bias;
    const uint16_t* r;
    uint16_t* d;
    int64_t ldr;
    int64_t ldd;
    int32_t m, n, k;
    int32_t num_m_blocks, num_n_blocks, num_tiles, num_k_blocks;
    int32_t group_m;
    int32_t zigzag;
    int32_t act;
    uint32_t flags;
    uint64_t timeout_ns;
    int32_t inject;
    // split-K: each tile's k-blocks are cut into `splits` ranges of `kb_per_split`;
    // work item w = tile * splits + split.  With splits > 1 every epilogue warp
    // writes its fp32 partial slab to `ws` and the last of the splits (counted in
    // `ws_cnt`, one counter per 32-row slab, zero on entry) reduces them in split
    // order and runs the epilogue.
    int32_t splits;
    int32_t kb_per_split;
    float* ws;
    uint32_t* ws_cnt;
};

struct SharedCtl {
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    volatile int32_t abort;
};

// The device status word of this translation unit (see gb_get_device_status).
__device__ uint32_t g_gb_status;

__device__ __forceinline__ void record_timeout(uint32_t role, uint32_t where, volatile int32_t* abort) {
    atomicCAS(&g_gb_status, 0u, kStatusTimeout | (role << 8) | ((where & 0xffffu) << 16));
    *abort = 1;
}

// Bounded wait for the phase of `bar` with the given parity.  Returns false if
// the CTA is aborting or the time limit ran out (then it records the timeout).
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int32_t* abort,
                                         uint64_t timeout_ns, uint32_t role, uint32_t where) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (global_timer_ns() - t0 > timeout_ns) {
            record_timeout(role, where, abort);
            return false;
        }
    }
}

// Bounded wait that ignores the abort flag: used while draining after an abort.
__device__ __forceinline__ bool drain_bar(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > timeout_ns) return false;
    }
    return true;
}

// Persistent tile order: groups of `group_m` tile-rows; inside a group the
// tile-row index runs fastest; odd groups walk the tile-columns backwards.
__device__ __forceinline__ void tile_coords(int32_t tile, const GemmParams& p, int32_t& mb, int32_t& nb) {
    const int32_t per_group = p.group_m * p.num_n_blocks;
    const int32_t group = tile / per_group;
    const int32_t first_m = group * p.group_m;
    const int32_t rows = min(p.num_m_blocks - first_m, p.group_m);
    const int32_t local = tile - group * per_group;
    mb = first_m + local % rows;
    nb = local / rows;
    if (group & 1) nb = p.num_n_blocks - 1 - nb;
}

// ---------------------------------------------------------------- epilogue math

__device__ __forceinline__ float act_apply(int act, float x) {
    // GELU (tanh form): 0.5 x (1 + tanh(u)) = x / (1 + e^{-2u}), u = sqrt(2/pi)(x + 0.044715 x^3),
    // evaluated as x / (1 + 2^{x (c0 + c1 x^2)}) with c0 = -2 log2(e) sqrt(2/pi), c1 = 0.044715 c0.
    // SiLU: x / (1 + e^{-x}) = x / (1 + 2^{-x log2(e)}).
    constexpr double kLog2e = 1.4426950408889634;
    constexpr double kSqrt2OverPi = 0.7978845608028654;
    constexpr float c0 = static_cast<float>(-2.0 * kLog2e * kSqrt2OverPi);
    constexpr float c1 = static_cast<float>(-2.0 * kLog2e * kSqrt2OverPi * 0.044715);
    switch (act) {
        case 1: {
            const float z = x * fmaf(c1, x * x, c0);
            return x * rcp_approx(1.0f + ex2_approx(z));
        }
        case 2:
            return x * rcp_approx(1.0f + ex2_approx(x * static_cast<float>(-kLog2e)));
        case 3:
            return fmaxf(x, 0.0f);
        default:
            return x;
    }
}

__device__ __forceinline__ float silu(float x) {
    constexpr float kNegLog2e = -1.4426950408889634f;
    return x * rcp_approx(1.0f + ex2_approx(x * kNegLog2e));
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// Add 32 consecutive bf16 values (a row segment of length `valid` <= 32) to v.
__device__ __forceinline__ void add_bf16_row(float (&v)[32], const uint16_t* src, int valid, bool vec_ok) {
    if (vec_ok && valid == 32) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 w = ld_global_nc_v4(src + 8 * i);
            v[8 * i + 0] += bf16_lo(w.x);
            v[8 * i + 1] += bf16_hi(w.x);
            v[8 * i + 2] += bf16_lo(w.y);
            v[8 * i + 3] += bf16_hi(w.y);
            v[8 * i + 4] += bf16_lo(w.z);
            v[8 * i + 5] += bf16_hi(w.z);
            v[8 * i + 6] += bf16_lo(w.w);
            v[8 * i + 7] += bf16_hi(w.w);
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            if (j < valid) v[j] += __uint_as_float(static_cast<uint32_t>(__ldg(src + j)) << 16);
        }
    }
}

// Bias, activation and epilogue input (linear), bf16 rounding, and the store of
// one 32-column chunk of row m (this lane) of the warp's 32-row slab at row0.
template <int NUM_B>
__device__ __forceinline__ void finish_chunk(const GemmParams& p, float (&v)[32], int32_t m, int32_t row0,
                                             int32_t n0, int lane, int q, uint8_t* dstage, uint32_t& dcount) {
    const int valid = min(32, p.n - n0);
    if (NUM_B == 1) {
        if (p.flags & kFlagBias) add_bf16_row(v, p.bias + n0, valid, p.flags & kFlagBiasVec);
        switch (p.act) {
            case 1:
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = act_apply(1, v[j]);
                break;
            case 2:
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = act_apply(2, v[j]);
                break;
            case 3:
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = act_apply(3, v[j]);
                break;
            default:
                break;
        }
        if ((p.flags & kFlagResidual) && m < p.m)
            add_bf16_row(v, p.r + static_cast<int64_t>(m) * p.ldr + n0, valid, p.flags & kFlagRVec);
    }

    uint32_t packed[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) packed[j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);

    if (p.flags & kFlagDTma) {
        uint8_t* buf = dstage + (q * 2 + (dcount & 1u)) * kDStageBytes;
        if (lane == 0) bulk_wait_group_read<1>();  // the store that last used this buffer has read it
        __syncwarp();
        // 64-byte rows, 16-byte units XOR-swizzled with (row / 2) % 4 (TMA 64B swizzle).
        const uint32_t row_addr = smem_addr(buf) + lane * 64;
        const uint32_t sw = (lane >> 1) & 3u;
#pragma unroll
        for (int u = 0; u < 4; ++u)
            st_shared_v4(row_addr + ((u ^ sw) << 4), packed[4 * u], packed[4 * u + 1], packed[4 * u + 2],
                         packed[4 * u + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(&p.tm_d, smem_addr(buf), n0, row0);
            bulk_commit_group();
        }
        ++dcount;
    } else if (m < p.m) {
        uint16_t* dst = p.d + static_cast<int64_t>(m) * p.ldd + n0;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            if (j < valid)
                dst[j] = static_cast<uint16_t>((j & 1) ? (packed[j >> 1] >> 16) : (packed[j >> 1] & 0xffffu));
        }
    }
}

__device__ __forceinline__ void st_global_f32x32(float* dst, const uint32_t (&r)[32]) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
        asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(dst + 4 * i), "r"(r[4 * i]), "r"(r[4 * i + 1]),
                     "r"(r[4 * i + 2]), "r"(r[4 * i + 3])
                     : "memory");
}

// v += 32 floats at src (bypassing L1: written by other CTAs of this launch).
__device__ __forceinline__ void add_f32x32_cg(float (&v)[32], const float* src) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float4 x = __ldcg(reinterpret_cast<const float4*>(src) + i);
        v[4 * i] += x.x;
        v[4 * i + 1] += x.y;
        v[4 * i + 2] += x.z;
        v[4 * i + 3] += x.w;
    }
}

// ---------------------------------------------------------------- the kernel

// Compile-time shape of one kernel variant.
//   BN    : output tile width (columns of D per tile)
//   NUM_B : 1 (linear) or 2 (FFN: W1 and W3 share the A tile)
//   PAIR  : CTA pair with cta_group::2 (256-row tiles, each CTA holds 128 rows
//           of A) or a single CTA (128-row tiles)
// Every variant issues ONE MMA per 16-wide K slice with N = NUM_B * BN: for the
// FFN the B operand is [W1 tile ; W3 tile], so the accumulator holds
// [X.W1^T | X.W3^T] and the A tile is read once for both products.  In a pair
// the B operand is split along N between the two CTAs, so the even CTA loads
// the W1 tile and the odd CTA the W3 tile.
template <int BN, int NUM_B, int STAGES, bool PAIR>
struct KernelShape {
    static constexpr int kCG = PAIR ? 2 : 1;
    static constexpr int kTileM = kBM * kCG;
    static constexpr int kMmaN = NUM_B * BN;
    static constexpr int kBRows = kMmaN / kCG;  // rows of the B operand this CTA holds
    static constexpr int kBBox = NUM_B == 1 ? kBRows : BN;  // rows per B TMA box
    static constexpr uint32_t kABytes = kBM * kBK * 2;
    static constexpr uint32_t kBBytes = kBRows * kBK * 2;
    static constexpr uint32_t kStageBytes = kABytes + kBBytes;
    static constexpr uint32_t kTxBytes = kCG * kStageBytes;  // bytes the leader's full barrier waits for
    static constexpr uint32_t kRingBytes = STAGES * kStageBytes;
    static constexpr uint32_t kDStageTotal = 4 * 2 * kDStageBytes;
    static constexpr uint32_t kBarBytes = 2 * STAGES * 8;
    static constexpr uint32_t kSmemBytes =
        1024 /* alignment slack */ + kRingBytes + kDStageTotal + kBarBytes + sizeof(SharedCtl);
    static constexpr uint32_t kIdesc = idesc_bf16_f32(kTileM, kMmaN);
    static constexpr uint32_t kAccEmptyArrivals = 4 * kCG;  // epilogue warps of every CTA in the pair
    static_assert(kMmaN <= kAccStride, "accumulator buffer holds at most 256 columns");
    static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "tile width");
    static_assert(kBRows % 8 == 0 && kBRows <= 256 && kMmaN % 16 == 0, "B operand rows");
    static_assert(NUM_B == 1 || BN == kBRows || 2 * BN == kBRows, "FFN: one product per CTA or both stacked");
    static_assert(kSmemBytes <= 232448, "shared memory per CTA");
};

template <int BN, int NUM_B, int STAGES, bool PAIR>
__global__ void __launch_bounds__(kThreads, 1) gemm_persistent_kernel(const __grid_constant__ GemmParams p) {
    using S = KernelShape<BN, NUM_B, STAGES, PAIR>;
    constexpr int CG = S::kCG;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* ring = smem;
    uint8_t* dstage = smem + S::kRingBytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(dstage + S::kDStageTotal);
    uint64_t* empty = full + STAGES;
    SharedCtl* ctl = reinterpret_cast<SharedCtl*>(empty + STAGES);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint64_t tmo = p.timeout_ns;
    const uint32_t rank = PAIR ? cluster_ctarank() : 0u;  // position in the CTA pair
    const bool leader = rank == 0;
    const int32_t unit = PAIR ? static_cast<int32_t>(blockIdx.x >> 1) : static_cast<int32_t>(blockIdx.x);
    const int32_t units = PAIR ? static_cast<int32_t>(gridDim.x >> 1) : static_cast<int32_t>(gridDim.x);
    const int32_t num_work = p.num_tiles * p.splits;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_addr(&full[s]), 1);
            mbar_init(smem_addr(&empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_addr(&ctl->acc_full[b]), 1);
            mbar_init(smem_addr(&ctl->acc_empty[b]), S::kAccEmptyArrivals);
        }
        mbar_init(smem_addr(&ctl->drain), 1);
        ctl->abort = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        if (p.num_k_blocks > 0) {
            tma_prefetch_desc(&p.tm_a);
            tma_prefetch_desc(&p.tm_b0);
            if (NUM_B == 2) tma_prefetch_desc(&p.tm_b1);
        }
        if (p.flags & kFlagDTma) tma_prefetch_desc(&p.tm_d);
    }
    if (warp == 1) {
        tmem_alloc<CG>(smem_addr(&ctl->tmem_base), kTmemCols);
        tmem_relinquish<CG>();
    }
    tc_fence_before_sync();
    if constexpr (PAIR) cluster_sync(); else __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = ctl->tmem_base;
    volatile int32_t* abort_flag = &ctl->abort;

    if (warp == 0) {
        // ------------------------------------------------------------ producer (every CTA)
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            int32_t local = 0;
            for (int32_t w = unit; ok && w < num_work; w += units, ++local) {
                const int32_t tile = w / p.splits;
                const int32_t kb0 = (w - tile * p.splits) * p.kb_per_split;
                const int32_t nkb = min(p.num_k_blocks - kb0, p.kb_per_split);
                int32_t mb, nb;
                tile_coords(tile, p, mb, nb);
                const bool reverse = p.zigzag && (local & 1);
                const int32_t a_row = mb * S::kTileM + static_cast<int32_t>(rank) * kBM;
                const int32_t b_row = nb * BN + static_cast<int32_t>(rank) * S::kBRows;
                for (int32_t kk = 0; kk < nkb; ++kk, ++it) {
                    const int32_t kb = kb0 + (reverse ? nkb - 1 - kk : kk);
                    const uint32_t s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1u;
                    if (!wait_bar(smem_addr(&empty[s]), ph ^ 1u, abort_flag, tmo, kRoleProducer, s)) {
                        ok = false;
                        break;
                    }
                    if (p.inject == kInjectSkipFirstStage && it == 0 && leader) continue;  // test hook
                    uint8_t* st = ring + s * S::kStageBytes;
                    const uint32_t own_full = smem_addr(&full[s]);
                    if (leader) mbar_arrive_expect_tx(own_full, S::kTxBytes);
                    uint8_t* sb = st + S::kABytes;
                    if constexpr (PAIR) {
                        const uint32_t fb = mapa_shared(own_full, 0);  // the leader's full barrier
                        tma_load_2d_pair(smem_addr(st), &p.tm_a, fb, kb * kBK, a_row);
                        if (NUM_B == 1)
                            tma_load_2d_pair(smem_addr(sb), &p.tm_b0, fb, kb * kBK, b_row);
                        else  // this CTA's half of the N = 2 BN operand is one whole product
                            tma_load_2d_pair(smem_addr(sb), leader ? &p.tm_b0 : &p.tm_b1, fb, kb * kBK, nb * BN);
                    } else {
                        tma_load_2d(smem_addr(st), &p.tm_a, own_full, kb * kBK, a_row);
                        tma_load_2d(smem_addr(sb), &p.tm_b0, own_full, kb * kBK, NUM_B == 1 ? b_row : nb * BN);
                        if (NUM_B == 2)
                            tma_load_2d(smem_addr(sb + BN * kBK * 2), &p.tm_b1, own_full, kb * kBK, nb * BN);
                    }
                }
            }
            if (!ok && leader) {
                // Drain: the leader's full barriers count the bytes of both CTAs; wait
                // (bounded) for the loads of the last STAGES k-blocks to land.
                const uint32_t first = it > STAGES ? it - STAGES : 0u;
                for (uint32_t i = first; i < it; ++i) {
                    if (p.inject == kInjectSkipFirstStage && i == 0) continue;
                    drain_bar(smem_addr(&full[i % STAGES]), (i / STAGES) & 1u, tmo);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (leader CTA)
        if (lane == 0 && leader) {
            uint32_t it = 0;
            bool ok = true;
            bool issued = false;
            int32_t local = 0;
            for (int32_t w = unit; ok && w < num_work; w += units, ++local) {
                const int32_t tile = w / p.splits;
                const int32_t kb0 = (w - tile * p.splits) * p.kb_per_split;
                const int32_t nkb = min(p.num_k_blocks - kb0, p.kb_per_split);
                const uint32_t b = local & 1;
                const uint32_t aph = (local >> 1) & 1u;
                if (!wait_bar(smem_addr(&ctl->acc_empty[b]), aph ^ 1u, abort_flag, tmo, kRoleMma, 0x100u | b)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + b * kAccStride;
                for (int32_t kk = 0; kk < nkb; ++kk, ++it) {
                    const uint32_t s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1u;
                    if (!wait_bar(smem_addr(&full[s]), ph, abort_flag, tmo, kRoleMma, s)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t a_addr = smem_addr(ring + s * S::kStageBytes);
                    const uint64_t adesc = sdesc_kmajor_sw128(a_addr);
                    const uint64_t bdesc = sdesc_kmajor_sw128(a_addr + S::kABytes);
#pragma unroll
                    for (int j = 0; j < kBK / 16; ++j) {
                        // +32 bytes along K per 16-element slice: +2 in the >>4-encoded address
                        const uint32_t acc = (kk > 0 || j > 0) ? 1u : 0u;
                        mma_bf16<CG>(d_tmem, adesc + 2 * j, bdesc + 2 * j, S::kIdesc, acc);
                    }
                    issued = true;
                    if constexpr (PAIR) mma_commit_multicast2(smem_addr(&empty[s]), 0x3);
                    else mma_commit<1>(smem_addr(&empty[s]));
                }
                if (!ok) break;
                if constexpr (PAIR) mma_commit_multicast2(smem_addr(&ctl->acc_full[b]), 0x3);
                else mma_commit<1>(smem_addr(&ctl->acc_full[b]));
            }
            if (!ok && issued) {
                // Drain: every MMA issued so far must finish before TMEM is freed.
                mma_commit<CG>(smem_addr(&ctl->drain));
                drain_bar(smem_addr(&ctl->drain), 0, tmo);
            }
        }
        __syncwarp();
    } else if (warp >= kEpiWarp0) {
        // ------------------------------------------------------------ epilogue (every CTA)
        const int q = warp - kEpiWarp0;  // == warp % 4: this warp's TMEM lane quadrant
        const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
        const int32_t slab_row = static_cast<int32_t>(rank) * kBM + q * 32 + lane;  // row within the tile
        constexpr int64_t kPartFloats = static_cast<int64_t>(S::kTileM) * BN;       // one partial accumulator
        uint32_t dcount = 0;
        int32_t local = 0;
        for (int32_t w = unit; w < num_work; w += units, ++local) {
            const uint32_t b = local & 1;
            const uint32_t aph = (local >> 1) & 1u;
            bool ok = true;
            if (lane == 0)
                ok = wait_bar(smem_addr(&ctl->acc_full[b]), aph, abort_flag, tmo, kRoleEpilogue, b);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after_sync();

            const int32_t tile = w / p.splits;
            int32_t mb, nb;
            tile_coords(tile, p, mb, nb);
            const int32_t row0 = mb * S::kTileM + static_cast<int32_t>(rank) * kBM + q * 32;  // this warp's slab
            const int32_t m = row0 + lane;
            const bool warp_rows = row0 < p.m;
            const uint32_t tcol = tmem_base + lane_base + b * kAccStride;
            const bool split_mode = p.splits > 1;
            float* part = p.ws + static_cast<int64_t>(w) * NUM_B * kPartFloats + static_cast<int64_t>(slab_row) * BN;

#pragma unroll 1
            for (int c = 0; c < BN / kDChunk; ++c) {
                const int32_t n0 = nb * BN + c * kDChunk;
                const bool chunk_on = warp_rows && n0 < p.n;
                float v[32];
                if (chunk_on && p.num_k_blocks > 0) {
                    uint32_t r0[32];
                    tmem_ld_32x32b_x32(tcol + c * kDChunk, r0);
                    if (NUM_B == 2) {
                        uint32_t r1[32];
                        tmem_ld_32x32b_x32(tcol + BN + c * kDChunk, r1);
                        tmem_wait_ld();
                        if (split_mode) {
                            st_global_f32x32(part + c * kDChunk, r0);
                            st_global_f32x32(part + kPartFloats + c * kDChunk, r1);
                        } else {
#pragma unroll
                            for (int j = 0; j < 32; ++j) v[j] = silu(__uint_as_float(r0[j])) * __uint_as_float(r1[j]);
                        }
                    } else {
                        tmem_wait_ld();
                        if (split_mode) {
                            st_global_f32x32(part + c * kDChunk, r0);
                        } else {
#pragma unroll
                            for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r0[j]);
                        }
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = 0.0f;
                }
                if (c == BN / kDChunk - 1) {
                    // All TMEM reads of this buffer are done: hand it back to the MMA issuer.
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) {
                        if constexpr (PAIR) mbar_arrive_cluster(mapa_shared(smem_addr(&ctl->acc_empty[b]), 0));
                        else mbar_arrive(smem_addr(&ctl->acc_empty[b]));
                    }
                }
                if (!chunk_on || split_mode) continue;
                finish_chunk<NUM_B>(p, v, m, row0, n0, lane, q, dstage, dcount);
            }
            if (!split_mode || !warp_rows) continue;

            // split-K: publish this partial; the last split of this slab reduces all of them.
            __threadfence();
            __syncwarp();
            uint32_t* cnt = p.ws_cnt + tile * (4 * S::kCG) + static_cast<int32_t>(rank) * 4 + q;
            uint32_t arrived = 0;
            if (lane == 0) arrived = atomicAdd(cnt, 1u);
            arrived = __shfl_sync(0xffffffffu, arrived, 0);
            if (arrived != static_cast<uint32_t>(p.splits - 1)) continue;
            __threadfence();
            const float* base = p.ws + static_cast<int64_t>(tile) * p.splits * NUM_B * kPartFloats +
                                static_cast<int64_t>(slab_row) * BN;
#pragma unroll 1
            for (int c = 0; c < BN / kDChunk; ++c) {
                const int32_t n0 = nb * BN + c * kDChunk;
                if (n0 >= p.n) break;
                float v[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = 0.0f;
                if (NUM_B == 2) {
                    float v3[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) v3[j] = 0.0f;
                    for (int32_t sp = 0; sp < p.splits; ++sp) {
                        const float* src = base + static_cast<int64_t>(sp) * NUM_B * kPartFloats + c * kDChunk;
                        add_f32x32_cg(v, src);
                        add_f32x32_cg(v3, src + kPartFloats);
                    }
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = silu(v[j]) * v3[j];
                } else {
                    for (int32_t sp = 0; sp < p.splits; ++sp)
                        add_f32x32_cg(v, base + static_cast<int64_t>(sp) * kPartFloats + c * kDChunk);
                }
                finish_chunk<NUM_B>(p, v, m, row0, n0, lane, q, dstage, dcount);
            }
            if (lane == 0) atomicExch(cnt, 0u);  // ready for the next launch
        }
        if (lane == 0) bulk_wait_group<0>();
        __syncwarp();
    }

    // ---------------------------------------------------------------- teardown
    // (for a pair, the cluster barrier also keeps each CTA's shared memory alive
    // until the peer has stopped signalling its barriers)
    tc_fence_before_sync();
    if constexpr (PAIR) cluster_sync(); else __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc<CG>(tmem_base, kTmemCols);
    }
}

}  // namespace gb
