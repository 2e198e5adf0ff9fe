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
//   * warps 4..7 or 4..11 -- epilogue, one or two warpgroups (template EPI):
//                       tcgen05.ld of 32-column chunks, bias, activation,
//                       epilogue input (prefetched by TMA into a per-warp box
//                       queue), bf16 rounding, and chunked TMA stores from a
//                       per-warp queue of staging boxes, each reused only after
//                       its store has read it (sections "Epilogue inputs" and
//                       "TMA store and stmatrix").  Two warpgroups either share
//                       every tile's chunks or alternate tiles (ping-pong, one
//                       TMEM buffer each; section "ping-pong").
//   * with two epilogue warpgroups, registers move from the control warpgroup
//     to them with setmaxnreg after the role split (section "Register
//     usage/spilling").
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
// Warpgroup 0: producer (warp 0), TMEM allocator + MMA issuer (warp 1), two
// spare warps.  Warpgroups 1..EPI: epilogue; epilogue warp e = warp - 4 reads
// TMEM lane quadrant e % 4 (= warp % 4) and takes every EPI-th 32-column chunk
// starting at e / 4.  One epilogue warpgroup suits long-K tiles (the epilogue
// hides under the MMAs); two suit epilogue-bound shapes (short K, epilogue
// input, unaligned rows).
constexpr int kEpiWarp0 = 4;
template <int EPI>
struct WarpLayout {
    static constexpr int kGroups = EPI;
    static constexpr int kEpiWarps = 4 * EPI;
    static constexpr int kThreads = 128 * (1 + EPI);
    // With two epilogue warpgroups, registers move to them after the role split
    // (setmaxnreg).  The launch gives every thread 65536 / kThreads registers
    // (rounded down to 8); the budgets must fit in that pool.
    static constexpr bool kRealloc = EPI == 2;
    static constexpr int kRegsLaunch = (65536 / kThreads) / 8 * 8;
    static constexpr int kRegsControl = 80;
    static constexpr int kRegsEpilogue = 208;
    static_assert(!kRealloc || 128 * kRegsControl + 128 * EPI * kRegsEpilogue <= kThreads * kRegsLaunch,
                  "register budgets exceed the launch pool");
    static_assert(EPI == 1 || EPI == 2 || EPI == 4, "one, two or four epilogue warpgroups");
    // Four epilogue warpgroups (lean variant, short-K residual work): only the paired
    // epilogue path is compiled in, so the whole kernel fits the 96 registers a thread
    // of a 640-thread block gets.  Warpgroups 2h and 2h + 1 serve the tiles of parity h
    // (TMEM buffer h), each taking every other 64-column step.
    static constexpr bool kLean = EPI == 4;
};
constexpr int kTmemCols = 512;    // two accumulator buffers of 256 columns
constexpr int kAccStride = 256;
constexpr int kDChunk = 32;       // epilogue chunk: 32 columns
constexpr int kDStageBytes = 32 * kDChunk * 2;  // one warp's 32x32 bf16 staging box
// Each epilogue warp owns a queue of D staging boxes (stores in flight) and, with
// an epilogue input, a queue of R boxes (loads in flight); the depths are chosen
// at launch, from 2 up to this.
constexpr int kMaxBoxes = 8;

enum : uint32_t {
    kFlagBias = 1u,
    kFlagResidual = 2u,
    kFlagDTma = 4u,      // D stored by TMA (16-byte aligned rows)
    kFlagRVec = 8u,      // R rows 16-byte aligned: vector loads
    kFlagBiasVec = 16u,  // bias 16-byte aligned: vector loads
    kFlagRTma = 32u,     // R loaded by TMA into shared memory, prefetched ahead of use
    kFlagZ = 64u,        // also store the pre-activation Z = bf16(acc + bias)
    kFlagZTma = 128u,    // Z stored by TMA (16-byte aligned rows)
    kFlagBMn = 256u,     // B is MN-major: a row-major [K, N] matrix (contraction over its rows)
    kFlagDact = 512u,    // the epilogue input multiplies: v *= act'(R) (activation gradient), no act
    kFlagRAsync = 1024u, // R rows not 16-byte aligned (4-byte aligned base): cp.async word copies into
                         // shared-memory slots, prefetched ahead of use like the TMA boxes
    kFlagWide = 2048u,   // paired path with 32x64 R and D boxes (128-byte swizzle): one TMA load, one
                         // TMA store, one barrier wait and one fence per 64 columns
    kFlagWideD = 4096u,  // paired path with 32x64 D boxes and 32x32 R boxes (the two chunks of a
                         // step adjacent; one TMA store and one fence per 64 columns)
};
constexpr uint32_t kWideBoxBytes = 32 * 2 * kDChunk * 2;  // one warp's 32x64 bf16 box
// One R slot of the cp.async queue: 32 rows x 17 words (a 32-column row segment that
// starts on a 2-byte boundary spans up to 17 aligned 4-byte words).  The 68-byte row
// stride also makes a lane's reads of its own row conflict-free (17 is odd).
constexpr uint32_t kRSlotWords = 17;
constexpr uint32_t kRSlotAsyncBytes = 32 * kRSlotWords * 4;
constexpr uint32_t kMnBoxBytes = 64 * kBK * 2;  // one MN-major B box: 64 columns x 64 contraction rows

// Codes written to the device status word (low byte = gb_status_t).
enum : uint32_t { kStatusTimeout = 4u };
enum : uint32_t { kRoleProducer = 1u, kRoleMma = 2u, kRoleEpilogue = 3u };

enum : int { kInjectNone = 0, kInjectSkipFirstStage = 1 };

struct GemmParams {  // the CUtensorMap members give it their 64-byte alignment
    CUtensorMap tm_a;   // A [M, K], box {64, 128}, 128B swizzle
    CUtensorMap tm_b0;  // B (or W1) [N, K], box {64, BN}, 128B swizzle
    CUtensorMap tm_b1;  // W3 [N, K] (FFN only)
    CUtensorMap tm_d;   // D [M, N], box {32, 32}, 64B swizzle (TMA store path)
    CUtensorMap tm_r;   // R [M, N], box {32, 32}, 64B swizzle (TMA load path)
    CUtensorMap tm_z;   // Z [M, N], box {32, 32}, 64B swizzle (TMA store path)
    const uint16_t* bias;
    const uint16_t* r;
    uint16_t* d;
    uint16_t* z;
    int64_t ldz;
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
    // adds its fp32 partial slab into the tile's accumulator in `ws` (fp32
    // reductions in L2; zero on entry), and the last split to finish a 32-row
    // slab (counted in `ws_cnt`, zero on entry) reads the sum and runs the
    // epilogue.
    int32_t splits;
    int32_t kb_per_split;
    float* ws;
    uint32_t* ws_cnt;
    int32_t stages;   // depth of the operand ring (<= the variant's maximum)
    // D staging boxes per epilogue warp, 2..kMaxBoxes, counted in 32x32 boxes (a wide
    // 32x64 box takes two)
    int32_t d_boxes;
    int32_t r_boxes;  // R queue entries per epilogue warp: 2..kMaxBoxes with an epilogue input (linear), else 0
    uint32_t r_warp_bytes;  // bytes of one epilogue warp's R queue: r_boxes x r_slot_bytes
    // Ping-pong (two epilogue warpgroups, no split): warpgroup g takes every work item
    // of local parity g -- always TMEM buffer g -- and all of its chunks, instead of
    // both warpgroups sharing every tile's chunks.
    int32_t pingpong;
    // L2 eviction hints (l2_policy codes: 0 none, 1 evict first, 2 evict last) for the
    // TMA loads of A, of B (W1/W3), of R, and the TMA stores of D and Z.
    uint32_t hint_a, hint_b, hint_r, hint_d;
    // A multicast between two CTA pairs (4-CTA clusters, CTA-pair variants only): a work
    // item is one tile-row x 2 tile-columns; pair q of the cluster computes tile-column
    // 2 * item + q, and each CTA loads half of its A tile and multicasts it to the CTA
    // of the other pair that needs the same rows (tm_a_half: box {64, 64}).
    int32_t mc;
    int32_t sched_n_blocks;  // tile-columns of the work-item grid (num_n_blocks, or half of it with mc)
    // MMA issue loop: 0 descriptors rebuilt per k-block; 1 lean (descriptors advanced
    // per stage); 2 lean, and the next stage's wait and fence done while the k-block's
    // third MMA runs, before its fourth is issued
    int32_t issue;
    // TMEM columns per tcgen05.ld on the express path (32, or 64: two chunks per load)
    // producer threads: 1 (warp 0 issues the A and B loads of every stage) or 2 (warp 0
    // the A loads and the expected byte count, warp 2 the B loads)
    int32_t prod;
    CUtensorMap tm_a_half;
    // Timing trace (libraries built with GB_TRACE only): kTraceWords words per CTA.
    unsigned long long* trace;
};

// Bytes of one D / R queue entry of a launch: a 32x32 box, a 32x64 box (wide), or a
// cp.async slot (unaligned R rows).
__host__ __device__ __forceinline__ uint32_t d_slot_bytes(const GemmParams& p) {
    return (p.flags & (kFlagWide | kFlagWideD)) ? kWideBoxBytes : kDStageBytes;
}
__host__ __device__ __forceinline__ uint32_t r_slot_bytes(const GemmParams& p) {
    return (p.flags & kFlagRAsync) ? kRSlotAsyncBytes : (p.flags & kFlagWide) ? kWideBoxBytes : kDStageBytes;
}

// Trace record of one CTA (GB_TRACE builds): where each role waited, in SM clock
// cycles, and when the CTA started and finished, in %globaltimer nanoseconds.
constexpr int kTraceWords = 32;
enum : int {
    kTrStartNs = 0,        // kernel entry
    kTrSetupNs = 1,        // barriers initialised, TMEM allocated
    kTrMmaFullCyc = 2,     // MMA issuer: cycles blocked on operand stages (full)
    kTrMmaFullN = 3,
    kTrMmaAccCyc = 4,      // MMA issuer: cycles blocked on a free accumulator (acc_empty)
    kTrMmaAccN = 5,
    kTrProdEmptyCyc = 6,   // producer: cycles blocked on a free stage (empty)
    kTrProdEmptyN = 7,
    kTrEpiFullCyc = 8,     // epilogue warp 0: cycles blocked on a finished accumulator
    kTrEpiFullN = 9,
    kTrEpiBodyCyc = 10,    // epilogue warp 0: cycles spent on its tiles after the wait
    kTrMmaFirstNs = 11,    // MMA issuer: first MMA issued
    kTrMmaLastNs = 12,     // MMA issuer: last accumulator committed
    kTrEndNs = 13,         // epilogue warp 0 done
    kTrMmaItems = 14,      // work items this CTA's MMA issuer ran
    kTrMmaCyc = 15,        // MMA issuer: cycles from its first wait to its last commit
    // epilogue warp 0, cycles per phase of its chunk loop (express and paired paths)
    kTrEpDBox = 16,        // waiting for free D staging boxes
    kTrEpTmemLd = 17,      // tcgen05.ld + wait::ld
    kTrEpRWait = 18,       // waiting for the chunk's R box
    kTrEpMath = 19,        // bias, activation, epilogue input, bf16 packing, staging stores
    kTrEpStore = 20,       // proxy fence, warp sync, TMA store issue
    kTrEpRIssue = 21,      // issuing the next R box loads
    kTrEpSteps = 22,       // chunk steps
    // MMA issuer: k-block-to-k-block intervals (cycles between the first MMAs of
    // consecutive k-blocks of a tile) whose wait did not block, by length:
    // < 560, 560-700, 700-1000, >= 1000; and their total cycles
    kTrKbFast = 23,
    kTrKbMid = 24,
    kTrKbSlow = 25,
    kTrKbVerySlow = 26,
    kTrKbCycUnblocked = 27,
    kTrKbCycBlocked = 28,  // the same intervals' total where the wait did block
    kTrMmaWaitCyc = 29,    // MMA issuer: cycles inside every operand wait (try_wait can suspend inside)
};

// Per-phase cycle counters of the first epilogue warp (GB_TRACE builds).
#ifdef GB_TRACE
#define GB_TR_T0(name) long long name = clock64()
#define GB_TR_ADD(arr, idx, t0)                                        \
    do {                                                               \
        const long long _t1 = clock64();                               \
        if (arr) arr[(idx) - kTrEpDBox] += static_cast<uint32_t>(_t1 - (t0)); \
        t0 = _t1;                                                      \
    } while (0)
#else
#define GB_TR_T0(name)
#define GB_TR_ADD(arr, idx, t0)
#endif

struct TraceAcc {  // blocked cycles and blocked waits of one thread
    unsigned long long cyc = 0, n = 0;
};

struct SharedCtl {
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    volatile int32_t abort;
    uint32_t trace_ep[8];  // GB_TRACE builds: the first epilogue warp's per-phase cycle counters
};

// The device status word of this translation unit (see gb_get_device_status).
__device__ uint32_t g_gb_status;

__device__ __forceinline__ void record_timeout(uint32_t role, uint32_t where, volatile int32_t* abort) {
    atomicCAS(&g_gb_status, 0u, kStatusTimeout | (role << 8) | ((where & 0xffffu) << 16));
    *abort = 1;
}

// Suspend-time bound (ns) of the pipeline's ring and accumulator waits (see mbar_try_wait_for).
constexpr uint32_t kRingSuspendNs = 64;

// One try of a wait: with a suspend-time bound when kSuspendNs > 0.
template <uint32_t kSuspendNs>
__device__ __forceinline__ bool try_bar(uint32_t bar, uint32_t parity) {
    if constexpr (kSuspendNs > 0) return mbar_try_wait_for<kSuspendNs>(bar, parity);
    else return mbar_try_wait(bar, parity);
}

// Bounded wait for the phase of `bar` with the given parity.  Returns false if
// the CTA is aborting or the time limit ran out (then it records the timeout).
template <uint32_t kSuspendNs = 0>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int32_t* abort,
                                         uint64_t timeout_ns, uint32_t role, uint32_t where,
                                         TraceAcc* acc = nullptr) {
    if (try_bar<kSuspendNs>(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
#ifdef GB_TRACE
    const long long c0 = clock64();
#endif
    while (true) {
        if (try_bar<kSuspendNs>(bar, parity)) {
#ifdef GB_TRACE
            if (acc) {
                acc->cyc += static_cast<unsigned long long>(clock64() - c0);
                acc->n += 1;
            }
#endif
            return true;
        }
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
    const int32_t per_group = p.group_m * p.sched_n_blocks;
    const int32_t group = tile / per_group;
    const int32_t first_m = group * p.group_m;
    const int32_t rows = min(p.num_m_blocks - first_m, p.group_m);
    const int32_t local = tile - group * per_group;
    mb = first_m + local % rows;
    nb = local / rows;
    if (group & 1) nb = p.sched_n_blocks - 1 - nb;
}

// The tile this CTA computes for work-item tile index `tile`: with A multicast, pair
// `pairi` of the cluster takes tile-column 2 * item-column + pairi.
__device__ __forceinline__ void work_tile(int32_t tile, const GemmParams& p, uint32_t pairi, int32_t& mb,
                                          int32_t& nb) {
    tile_coords(tile, p, mb, nb);
    if (p.mc) nb = 2 * nb + static_cast<int32_t>(pairi);
}

// TMA operand loads and output stores, with an L2 policy when one is set.
template <bool PAIR>
__device__ __forceinline__ void tma_load_op(uint32_t dst, const void* tm, uint32_t bar, int32_t c0, int32_t c1,
                                            uint64_t pol) {
    if constexpr (PAIR) {
        if (pol) tma_load_2d_pair_hint(dst, tm, bar, c0, c1, pol);
        else tma_load_2d_pair(dst, tm, bar, c0, c1);
    } else {
        if (pol) tma_load_2d_hint(dst, tm, bar, c0, c1, pol);
        else tma_load_2d(dst, tm, bar, c0, c1);
    }
}

// `hint` is an l2_policy code; the policy is made at the store, so the epilogue keeps
// no 64-bit policy register live across its loops.
__device__ __forceinline__ void tma_store_op(const void* tm, uint32_t src, int32_t c0, int32_t c1, uint32_t hint) {
    if (hint) tma_store_2d_hint(tm, src, c0, c1, l2_policy(hint));
    else tma_store_2d(tm, src, c0, c1);
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

// Derivatives of act_apply's activations, for the activation-gradient epilogue:
// GELU (tanh form) x s(x) with s = 1 / (1 + e^{-2u}):  s (1 + x (1 - s) 2 sqrt(2/pi) (1 + 3 0.044715 x^2));
// SiLU x s(x) with s = 1 / (1 + e^{-x}):              s (1 + x (1 - s));  ReLU: 1 for x > 0, else 0.
__device__ __forceinline__ float dact_apply(int act, float x) {
    constexpr double kLog2e = 1.4426950408889634;
    constexpr double kSqrt2OverPi = 0.7978845608028654;
    constexpr float c0 = static_cast<float>(-2.0 * kLog2e * kSqrt2OverPi);
    constexpr float c1 = static_cast<float>(-2.0 * kLog2e * kSqrt2OverPi * 0.044715);
    constexpr float k0 = static_cast<float>(2.0 * kSqrt2OverPi);
    constexpr float k1 = static_cast<float>(2.0 * kSqrt2OverPi * 3.0 * 0.044715);
    switch (act) {
        case 1: {
            const float x2 = x * x;
            const float sg = rcp_approx(1.0f + ex2_approx(x * fmaf(c1, x2, c0)));
            return sg * fmaf(x * (1.0f - sg), fmaf(k1, x2, k0), 1.0f);
        }
        case 2: {
            const float sg = rcp_approx(1.0f + ex2_approx(x * static_cast<float>(-kLog2e)));
            return sg * fmaf(x, 1.0f - sg, 1.0f);
        }
        case 3:
            return x > 0.0f ? 1.0f : 0.0f;
        default:
            return 1.0f;
    }
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// How an epilogue input value r combines with the accumulator value v: OP 0 adds
// (v + r), OP 1..3 multiplies by the derivative of activation OP at r (v * act'(r),
// the activation gradient), OP 4 leaves v (the identity's derivative is 1).
template <int OP>
__device__ __forceinline__ void combine2(float& a, float& b, uint32_t w) {
    if constexpr (OP == 0) {
        a += bf16_lo(w);
        b += bf16_hi(w);
    } else if constexpr (OP <= 3) {
        a *= dact_apply(OP, bf16_lo(w));
        b *= dact_apply(OP, bf16_hi(w));
    }
}

// The combine OP of this launch's epilogue input.
__device__ __forceinline__ int input_op(uint32_t flags, int act) {
    return (flags & 512u /* kFlagDact */) ? (act >= 1 && act <= 3 ? act : 4) : 0;
}

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

// Add this lane's row of a 32x32 bf16 box staged by TMA with 64-byte swizzling.
__device__ __forceinline__ void add_bf16_box_row(float (&v)[32], uint32_t box, int lane) {
    const uint32_t row = box + lane * 64;
    const uint32_t sw = (lane >> 1) & 3u;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        uint32_t w0, w1, w2, w3;
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(w0), "=r"(w1), "=r"(w2), "=r"(w3)
                     : "r"(row + ((u ^ sw) << 4)));
        v[8 * u + 0] += bf16_lo(w0);
        v[8 * u + 1] += bf16_hi(w0);
        v[8 * u + 2] += bf16_lo(w1);
        v[8 * u + 3] += bf16_hi(w1);
        v[8 * u + 4] += bf16_lo(w2);
        v[8 * u + 5] += bf16_hi(w2);
        v[8 * u + 6] += bf16_lo(w3);
        v[8 * u + 7] += bf16_hi(w3);
    }
}

// Combine this lane's row of a 32x32 bf16 box staged by TMA (64-byte swizzle) into v.
template <int OP>
__device__ __forceinline__ void combine_box_row(float (&v)[32], uint32_t box, int lane) {
    const uint32_t row = box + lane * 64;
    const uint32_t sw = (lane >> 1) & 3u;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        uint32_t w0, w1, w2, w3;
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(w0), "=r"(w1), "=r"(w2), "=r"(w3)
                     : "r"(row + ((u ^ sw) << 4)));
        combine2<OP>(v[8 * u + 0], v[8 * u + 1], w0);
        combine2<OP>(v[8 * u + 2], v[8 * u + 3], w1);
        combine2<OP>(v[8 * u + 4], v[8 * u + 5], w2);
        combine2<OP>(v[8 * u + 6], v[8 * u + 7], w3);
    }
}

// The epilogue input of one chunk from its TMA box: added (linear), or the
// activation gradient's multiplier act'(r) (kFlagDact).
__device__ __forceinline__ void apply_input_box(const GemmParams& p, float (&v)[32], uint32_t box, int lane) {
    switch (input_op(p.flags, p.act)) {
        case 0: combine_box_row<0>(v, box, lane); break;
        case 1: combine_box_row<1>(v, box, lane); break;
        case 2: combine_box_row<2>(v, box, lane); break;
        case 3: combine_box_row<3>(v, box, lane); break;
        default: break;
    }
}

// Write chunk `half` (0: columns 0-31, 1: 32-63) of this lane's row of a 32x64 bf16
// box, 128-byte swizzled for the TMA store (16-byte unit u of row r at u ^ (r % 8)).
__device__ __forceinline__ void stage_wide_half(uint32_t box, const float (&v)[32], int half, int lane) {
    const uint32_t row_addr = box + lane * 128;
    const uint32_t sw = lane & 7u;
#pragma unroll
    for (int u = 0; u < 4; ++u)
        st_shared_v4(row_addr + (((4 * half + u) ^ sw) << 4), pack_bf16x2(v[8 * u], v[8 * u + 1]),
                     pack_bf16x2(v[8 * u + 2], v[8 * u + 3]), pack_bf16x2(v[8 * u + 4], v[8 * u + 5]),
                     pack_bf16x2(v[8 * u + 6], v[8 * u + 7]));
}

// Combine chunk `half` of this lane's row of a 32x64 bf16 box staged by TMA (128-byte
// swizzle) into v.
template <int OP>
__device__ __forceinline__ void combine_wide_half(float (&v)[32], uint32_t box, int half, int lane) {
    const uint32_t row = box + lane * 128;
    const uint32_t sw = lane & 7u;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        uint32_t w0, w1, w2, w3;
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(w0), "=r"(w1), "=r"(w2), "=r"(w3)
                     : "r"(row + (((4 * half + u) ^ sw) << 4)));
        combine2<OP>(v[8 * u + 0], v[8 * u + 1], w0);
        combine2<OP>(v[8 * u + 2], v[8 * u + 3], w1);
        combine2<OP>(v[8 * u + 4], v[8 * u + 5], w2);
        combine2<OP>(v[8 * u + 6], v[8 * u + 7], w3);
    }
}

__device__ __forceinline__ void apply_input_wide(const GemmParams& p, float (&v)[32], uint32_t box, int half,
                                                 int lane) {
    switch (input_op(p.flags, p.act)) {
        case 0: combine_wide_half<0>(v, box, half, lane); break;
        case 1: combine_wide_half<1>(v, box, half, lane); break;
        case 2: combine_wide_half<2>(v, box, half, lane); break;
        case 3: combine_wide_half<3>(v, box, half, lane); break;
        default: break;
    }
}

// Combine this lane's row of a cp.async R slot (17 words per row, 68-byte stride) into v.
// The row segment starts `sh` bits (0 or 16) into the row's first word.
template <int OP>
__device__ __forceinline__ void combine_slot_row(float (&v)[32], uint32_t slot, uint32_t sh, int lane) {
    const uint32_t row = slot + static_cast<uint32_t>(lane) * (kRSlotWords * 4);
    uint32_t w[kRSlotWords];
#pragma unroll
    for (uint32_t k = 0; k < kRSlotWords; ++k)
        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(w[k]) : "r"(row + 4 * k));
#pragma unroll
    for (int k = 0; k < 16; ++k) combine2<OP>(v[2 * k], v[2 * k + 1], __funnelshift_r(w[k], w[k + 1], sh));
}

// The epilogue input of one chunk from its cp.async slot; `m` is this lane's row.  The
// base is 4-byte aligned, so the segment starts mid-word exactly when its element
// index m * ldr + n0 is odd.
__device__ __forceinline__ void apply_input_slot(const GemmParams& p, float (&v)[32], uint32_t slot, int32_t m,
                                                 int32_t n0, int lane) {
    const uint32_t sh = ((static_cast<uint32_t>(m) & static_cast<uint32_t>(p.ldr)) ^ static_cast<uint32_t>(n0)) & 1u
                            ? 16u : 0u;
    switch (input_op(p.flags, p.act)) {
        case 0: combine_slot_row<0>(v, slot, sh, lane); break;
        case 1: combine_slot_row<1>(v, slot, sh, lane); break;
        case 2: combine_slot_row<2>(v, slot, sh, lane); break;
        case 3: combine_slot_row<3>(v, slot, sh, lane); break;
        default: break;
    }
}

// The same from global memory: a 16-byte aligned row segment of 32 values (rows past M skipped).
template <int OP>
__device__ __forceinline__ void combine_row_vec(float (&v)[32], const uint16_t* src) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint4 w = ld_global_nc_v4(src + 8 * i);
        combine2<OP>(v[8 * i + 0], v[8 * i + 1], w.x);
        combine2<OP>(v[8 * i + 2], v[8 * i + 3], w.y);
        combine2<OP>(v[8 * i + 4], v[8 * i + 5], w.z);
        combine2<OP>(v[8 * i + 6], v[8 * i + 7], w.w);
    }
}

// Write this lane's row of a 32x32 bf16 box, 64-byte swizzled for the TMA store.
__device__ __forceinline__ void stage_box_row(uint32_t box, const float (&v)[32], int lane) {
    const uint32_t row_addr = box + lane * 64;
    const uint32_t sw = (lane >> 1) & 3u;
#pragma unroll
    for (int u = 0; u < 4; ++u)
        st_shared_v4(row_addr + ((u ^ sw) << 4), pack_bf16x2(v[8 * u], v[8 * u + 1]),
                     pack_bf16x2(v[8 * u + 2], v[8 * u + 3]), pack_bf16x2(v[8 * u + 4], v[8 * u + 5]),
                     pack_bf16x2(v[8 * u + 6], v[8 * u + 7]));
}

// Rows of D or R that are not 16-byte aligned (e.g. N = 4099): go through a
// per-warp shared-memory transpose, so every global access instruction covers one
// contiguous 64-byte row segment instead of 32 scattered 2-byte ones.  The buffer is
// one 32x32 staging box in the TMA 64-byte swizzle (16-byte unit u of row r at
// u ^ ((r / 2) % 4)): a lane's own row moves as four conflict-free 16-byte accesses,
// and column r (element `lane` of row r) is 64 contiguous bytes of the box.
// Warp-collective.
struct TransposeCols {  // this lane's element of a row, for the four swizzle phases of a row
    uint32_t at[4];
    __device__ __forceinline__ TransposeCols(uint32_t buf, int lane) {
#pragma unroll
        for (uint32_t k = 0; k < 4; ++k)
            at[k] = buf + ((((static_cast<uint32_t>(lane) >> 3) ^ k) << 4) | ((static_cast<uint32_t>(lane) & 7u) << 1));
    }
    // shared address of element `lane` of row r (r a compile-time constant after unrolling)
    __device__ __forceinline__ uint32_t row(int r) const { return at[(r >> 1) & 3] + static_cast<uint32_t>(r) * 64u; }
};

__device__ __forceinline__ void store_rows_transposed(const GemmParams& p, uint16_t* out, int64_t ld,
                                                      const uint32_t (&packed)[16], int32_t row0, int32_t n0,
                                                      int valid, int lane, uint32_t tbuf) {
    if (lane == 0) bulk_wait_group_read<0>();  // TMA stores of this warp no longer read the buffer
    __syncwarp();
    const uint32_t row_addr = tbuf + lane * 64;
    const uint32_t sw = (lane >> 1) & 3u;
#pragma unroll
    for (int u = 0; u < 4; ++u)
        st_shared_v4(row_addr + ((u ^ sw) << 4), packed[4 * u], packed[4 * u + 1], packed[4 * u + 2], packed[4 * u + 3]);
    __syncwarp();
    const int rows = min(32, p.m - row0);
    const TransposeCols col(tbuf, lane);
    uint16_t h[32];
#pragma unroll
    for (int r = 0; r < 32; ++r)  // all reads first...
        asm volatile("ld.shared.u16 %0, [%1];" : "=h"(h[r]) : "r"(col.row(r)));
    uint16_t* dst = out + static_cast<int64_t>(row0) * ld + n0 + lane;
    if (lane < valid) {
#pragma unroll
        for (int r = 0; r < 32; ++r)  // ...then one coalesced 64-byte row segment per store
            if (r < rows) dst[static_cast<int64_t>(r) * ld] = h[r];
    }
    __syncwarp();
}

__device__ __forceinline__ void add_rows_transposed(const GemmParams& p, float (&v)[32], int32_t row0, int32_t n0,
                                                    int valid, int lane, uint32_t tbuf) {
    const int rows = min(32, p.m - row0);
    const uint16_t* src = p.r + static_cast<int64_t>(row0) * p.ldr + n0 + lane;
    uint16_t h[32];
#pragma unroll
    for (int r = 0; r < 32; ++r)  // all 32 coalesced row-segment loads in flight together
        h[r] = (r < rows && lane < valid) ? __ldg(src + static_cast<int64_t>(r) * p.ldr) : uint16_t(0);
    const TransposeCols col(tbuf, lane);
#pragma unroll
    for (int r = 0; r < 32; ++r) asm volatile("st.shared.u16 [%0], %1;" ::"r"(col.row(r)), "h"(h[r]) : "memory");
    __syncwarp();
    apply_input_box(p, v, tbuf, lane);  // this lane's row, as from a TMA box
    __syncwarp();
}

// Store one 32x32 bf16 chunk of an output: by TMA from the next box of this
// warp's queue of d_boxes staging boxes (a box is rewritten only after the store
// that used it has read it -- so several outputs share the queue), or through
// the shared-memory transpose when the output's rows are not 16-byte aligned.
// `dbox` is this warp's first box, `dslot` the queue position (wraps).
__device__ __forceinline__ void store_chunk(const GemmParams& p, const CUtensorMap* tm, uint16_t* out, int64_t ld,
                                            bool by_tma, const uint32_t (&packed)[16], int32_t row0, int32_t n0,
                                            int valid, int lane, uint32_t dbox, int32_t& dslot) {
    if (by_tma) {
        const uint32_t buf = dbox + dslot * kDStageBytes;
        if (lane == 0) bulk_wait_group_read_at_most(p.d_boxes - 1);  // the store that last used this box has read it
        __syncwarp();
        // 64-byte rows, 16-byte units XOR-swizzled with (row / 2) % 4 (TMA 64B swizzle).
        const uint32_t row_addr = buf + lane * 64;
        const uint32_t sw = (lane >> 1) & 3u;
#pragma unroll
        for (int u = 0; u < 4; ++u)
            st_shared_v4(row_addr + ((u ^ sw) << 4), packed[4 * u], packed[4 * u + 1], packed[4 * u + 2],
                         packed[4 * u + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_op(tm, buf, n0, row0, p.hint_d);
            bulk_commit_group();
        }
        if (++dslot == p.d_boxes) dslot = 0;
    } else {
        store_rows_transposed(p, out, ld, packed, row0, n0, valid, lane, dbox);
    }
}

// Bias, activation and epilogue input (linear), bf16 rounding, and the store of
// one 32-column chunk of row m (this lane) of the warp's 32-row slab at row0.
template <int NUM_B>
// `rbox` is the shared-memory address of this chunk's R box when R came by TMA
// (0: read R from global memory); `tbuf_r` is this warp's transpose buffer for an
// R whose rows are not 16-byte aligned; `dbox`/`dslot` are this warp's D staging
// queue and its position.  Warp-collective.
__device__ __forceinline__ void finish_chunk(const GemmParams& p, float (&v)[32], int32_t m, int32_t row0,
                                             int32_t n0, int lane, uint32_t dbox, int32_t& dslot,
                                             uint32_t rbox, uint32_t tbuf_r,
                                             uint32_t* tr_ep = nullptr) {
    GB_TR_T0(tx);
    const int valid = min(32, p.n - n0);
    if (NUM_B == 1) {
        if (p.flags & kFlagBias) add_bf16_row(v, p.bias + n0, valid, p.flags & kFlagBiasVec);
        if (p.flags & kFlagZ) {  // second output: the pre-activation
            uint32_t zp[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) zp[j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);
            store_chunk(p, &p.tm_z, p.z, p.ldz, p.flags & kFlagZTma, zp, row0, n0, valid, lane, dbox, dslot);
        }
        const bool dact = p.flags & kFlagDact;
        if (!dact) {
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
        }
        if (rbox) {
            if (p.flags & kFlagRAsync) apply_input_slot(p, v, rbox, m, n0, lane);
            else apply_input_box(p, v, rbox, lane);
        } else if (p.flags & kFlagResidual) {
            if (p.flags & kFlagRVec) {
                // R (Z) rows are 16-byte aligned and ldr is a multiple of 8, so a row's
                // segment is readable to 32 columns whenever the row exists (a partial
                // segment's tail columns are not stored).  The scalar path covers the
                // segment past the row's end.
                if (m < p.m) {
                    const uint16_t* src = p.r + static_cast<int64_t>(m) * p.ldr + n0;
                    if (valid == 32) {
                        switch (input_op(p.flags, p.act)) {
                            case 0: combine_row_vec<0>(v, src); break;
                            case 1: combine_row_vec<1>(v, src); break;
                            case 2: combine_row_vec<2>(v, src); break;
                            case 3: combine_row_vec<3>(v, src); break;
                            default: break;
                        }
                    } else if (!dact) {
                        add_bf16_row(v, src, valid, false);
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (j < valid)
                                v[j] *= dact_apply(p.act, __uint_as_float(static_cast<uint32_t>(__ldg(src + j)) << 16));
                    }
                }
            } else {
                GB_TR_ADD(tr_ep, kTrEpMath, tx);
                add_rows_transposed(p, v, row0, n0, valid, lane, tbuf_r);
                GB_TR_ADD(tr_ep, kTrEpRWait, tx);
            }
        }
    }

    uint32_t packed[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) packed[j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);
    GB_TR_ADD(tr_ep, kTrEpMath, tx);
    store_chunk(p, &p.tm_d, p.d, p.ldd, p.flags & kFlagDTma, packed, row0, n0, valid, lane, dbox, dslot);
    GB_TR_ADD(tr_ep, kTrEpStore, tx);
}

// 32 floats added into global memory with vector fp32 reductions (performed in L2).
__device__ __forceinline__ void red_add_f32x32(float* dst, const uint32_t (&r)[32]) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
        asm volatile("red.relaxed.gpu.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst + 4 * i),
                     "f"(__uint_as_float(r[4 * i])), "f"(__uint_as_float(r[4 * i + 1])),
                     "f"(__uint_as_float(r[4 * i + 2])), "f"(__uint_as_float(r[4 * i + 3]))
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

// ---------------------------------------------------------------- lean MMA issue

// The stage descriptors of ring slot `slot`: the slot's A tile and, kABytes further,
// its B tile (K-major, or MN-major boxes of 64 columns).
__device__ __forceinline__ void stage_descs(uint32_t ring0, uint32_t slot, uint32_t stage_bytes, uint32_t a_bytes,
                                            bool b_mn, uint64_t& ad, uint64_t& bd) {
    const uint32_t a_addr = ring0 + slot * stage_bytes;
    ad = sdesc_kmajor_sw128(a_addr);
    bd = b_mn ? sdesc_mnmajor_sw128(a_addr + a_bytes, kMnBoxBytes) : sdesc_kmajor_sw128(a_addr + a_bytes);
}

// The MMA issuer's loop over one item's k-blocks for the common operand forms: the
// descriptor steps, the instruction descriptor and the commit mask are compile-time
// constants, and nothing but the stage wait runs between k-blocks.  `s`, `ph` and `it`
// carry the ring position across items (it == 0: nothing consumed yet).  Without A
// multicast the cluster is the CTA pair itself, so the stage is freed in ranks 0 and 1
// (kMask 0x3); with A multicast between two pairs, in all four CTAs (0xF).
// Returns false if a wait gave up.
template <int CG, uint32_t kStageBytes, uint32_t kABytes, uint32_t kIdescK, bool BMN, uint16_t kMask = 0x3>
__device__ __forceinline__ bool issue_kblocks(uint32_t d_tmem, int32_t nkb, uint64_t* full, uint64_t* empty,
                                              uint8_t* ring, uint32_t stages, uint32_t& s, uint32_t& ph,
                                              uint32_t& it, volatile int32_t* abort_flag, uint64_t tmo,
                                              TraceAcc& tr_full, bool& issued) {
    constexpr uint32_t kIdesc = kIdescK | (BMN ? kIdescBMnMajor : 0u);
    // per 16-element K slice: +32 bytes in a K-major tile (+2 encoded), +16 rows of 128 bytes
    // in an MN-major one (+128 encoded)
    constexpr uint64_t kBStep = BMN ? (16u * 128u) >> 4 : 2u;
    for (int32_t kk = 0; kk < nkb; ++kk, ++it) {
        if (it > 0 && ++s == stages) {
            s = 0;
            ph ^= 1u;
        }
        if (!wait_bar<kRingSuspendNs>(smem_addr(&full[s]), ph, abort_flag, tmo, kRoleMma, s, &tr_full)) return false;
        tc_fence_after_sync();
        const uint32_t a_addr = smem_addr(ring + s * kStageBytes);
        const uint64_t ad = sdesc_kmajor_sw128(a_addr);
        const uint64_t bd = BMN ? sdesc_mnmajor_sw128(a_addr + kABytes, kMnBoxBytes) : sdesc_kmajor_sw128(a_addr + kABytes);
        mma_bf16_x4<CG>(d_tmem, ad, ad + 2, ad + 4, ad + 6, bd, bd + kBStep, bd + 2 * kBStep, bd + 3 * kBStep, kIdesc,
                        kk > 0 ? 1u : 0u);
        issued = true;
        if constexpr (CG == 2) mma_commit_multicast2(smem_addr(&empty[s]), kMask);
        else mma_commit<1>(smem_addr(&empty[s]));
    }
    return true;
}

// One work item's k-blocks on the lean issue path.  The ring position (s, ph) and the
// k-block counter `it` describe the k-block consumed last (it == 0: none yet), as in
// the rebuild path, so both paths can follow each other.  Returns false if a wait gave up.
template <int CG, uint32_t kStageBytes, uint32_t kABytes>
__device__ __forceinline__ bool issue_tile_lean(const GemmParams& p, uint32_t d_tmem, int32_t nkb, uint64_t* full,
                                                uint64_t* empty, uint8_t* ring, uint32_t stages, uint32_t& s,
                                                uint32_t& ph, uint32_t& it, bool b_mn, uint32_t idesc, uint32_t bstep,
                                                uint16_t empty_mask, volatile int32_t* abort_flag, uint64_t tmo,
                                                TraceAcc& tr_full, bool& issued) {
    if (nkb <= 0) return true;
    const uint32_t ring0 = smem_addr(ring);
    const uint32_t full0 = smem_addr(full), empty0 = smem_addr(empty);
    // position of the first k-block of this item
    uint32_t cs = s, cph = ph;
    if (it > 0 && ++cs == stages) {
        cs = 0;
        cph ^= 1u;
    }
    uint64_t ad, bd;
    stage_descs(ring0, cs, kStageBytes, kABytes, b_mn, ad, bd);
    if (!wait_bar<kRingSuspendNs>(full0 + 8 * cs, cph, abort_flag, tmo, kRoleMma, cs, &tr_full)) return false;
    tc_fence_after_sync();
    const bool lookahead = p.issue == 2;
    for (int32_t kk = 0; kk < nkb; ++kk) {
        mma_bf16<CG>(d_tmem, ad, bd, idesc, kk > 0 ? 1u : 0u);
        mma_bf16<CG>(d_tmem, ad + 2, bd + bstep, idesc, 1u);
        mma_bf16<CG>(d_tmem, ad + 4, bd + 2 * bstep, idesc, 1u);
        issued = true;
        const uint32_t done = cs;
        const uint64_t ad3 = ad + 6, bd3 = bd + 3 * bstep;
        const bool more = kk + 1 < nkb;
        if (more) {  // the next k-block's stage
            if (++cs == stages) {
                cs = 0;
                cph ^= 1u;
                ad -= static_cast<uint64_t>((stages - 1) * (kStageBytes >> 4));
                bd -= static_cast<uint64_t>((stages - 1) * (kStageBytes >> 4));
            } else {
                ad += kStageBytes >> 4;
                bd += kStageBytes >> 4;
            }
            if (lookahead) {
                if (!wait_bar<kRingSuspendNs>(full0 + 8 * cs, cph, abort_flag, tmo, kRoleMma, cs, &tr_full)) return false;
                tc_fence_after_sync();
            }
        }
        mma_bf16<CG>(d_tmem, ad3, bd3, idesc, 1u);
        if constexpr (CG == 2) mma_commit_multicast2(empty0 + 8 * done, empty_mask);
        else mma_commit<1>(empty0 + 8 * done);
        if (more && !lookahead) {
            if (!wait_bar<kRingSuspendNs>(full0 + 8 * cs, cph, abort_flag, tmo, kRoleMma, cs, &tr_full)) return false;
            tc_fence_after_sync();
        }
    }
    s = cs;
    ph = cph;
    it += static_cast<uint32_t>(nkb);
    return true;
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
template <int BN, int NUM_B, int STAGES, bool PAIR, int EPI>
struct KernelShape {
    using W = WarpLayout<EPI>;
    static constexpr int kEpiWarps = W::kEpiWarps;
    static constexpr int kThreads = W::kThreads;
    static constexpr int kCG = PAIR ? 2 : 1;
    static constexpr int kMaxStages = STAGES;  // the ring depth is chosen at launch, up to this
    static constexpr int kTileM = kBM * kCG;
    static constexpr int kMmaN = NUM_B * BN;
    static constexpr int kBRows = kMmaN / kCG;  // rows of the B operand this CTA holds
    static constexpr int kBBox = NUM_B == 1 ? kBRows : BN;  // rows per B TMA box
    static constexpr uint32_t kABytes = kBM * kBK * 2;
    static constexpr uint32_t kBBytes = kBRows * kBK * 2;
    static constexpr uint32_t kStageBytes = kABytes + kBBytes;
    static constexpr uint32_t kTxBytes = kCG * kStageBytes;  // bytes the leader's full barrier waits for
    static constexpr uint32_t kBarBytes = 2 * STAGES * 8 + kMaxBoxes * kEpiWarps * 8;  // ring + R barriers
    // Layout: [barriers][control] in the first 1 KiB or 2 (fixed offsets, whatever the
    // queue sizes), then [ring: stages x stage][D boxes: warps x d_boxes][R boxes: warps x r_boxes].
    // `r_slot`, `d_slot`: bytes of one R / D queue entry (a 32x32 or 32x64 TMA box, or a
    // cp.async slot).
    static constexpr uint32_t kCtlBytes = (kBarBytes + sizeof(SharedCtl) + 1023) / 1024 * 1024;
    static constexpr uint32_t smem_bytes(int stages, int d_boxes, int r_boxes, uint32_t r_slot = kDStageBytes,
                                         uint32_t d_slot = kDStageBytes) {
        return 1024 /* alignment slack */ + kCtlBytes + stages * kStageBytes +
               static_cast<uint32_t>(kEpiWarps * d_boxes) * d_slot + static_cast<uint32_t>(kEpiWarps * r_boxes) * r_slot;
    }
    static_assert(kBarBytes + sizeof(SharedCtl) <= kCtlBytes, "barriers and control block fit in their block");
    static constexpr uint32_t kIdesc = idesc_bf16_f32(kTileM, kMmaN);
    static constexpr uint32_t kAccEmptyArrivals = kEpiWarps * kCG;  // epilogue warps of every CTA in the pair
    // split-K counters per tile: one per epilogue warp of every CTA of the tile, laid out
    // for the most epilogue warps any variant of this tile shape has (two warpgroups), so
    // the workspace size does not depend on which epilogue layout a call picks
    static constexpr int kSlabs = 8 * kCG;
    static_assert(kEpiWarps <= 8 || W::kLean, "split-K counter layout (the lean variant has no split-K path)");
    static_assert(kMmaN <= kAccStride, "accumulator buffer holds at most 256 columns");
    static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "tile width");
    static_assert(kBRows % 8 == 0 && kBRows <= 256 && kMmaN % 16 == 0, "B operand rows");
    static_assert(NUM_B == 1 || BN == kBRows || 2 * BN == kBRows, "FFN: one product per CTA or both stacked");
    static_assert(smem_bytes(STAGES, 2, 0) <= 232448, "the deepest ring fits with two D boxes per warp");
    static_assert(smem_bytes(2, 2, NUM_B == 1 ? 2 : 0) <= 232448, "a two-stage ring fits with two D and R boxes");
};

template <int BN, int NUM_B, int STAGES, bool PAIR, int EPI>
__global__ void __launch_bounds__(128 * (1 + EPI), 1) gemm_persistent_kernel(const __grid_constant__ GemmParams p) {
    using S = KernelShape<BN, NUM_B, STAGES, PAIR, EPI>;
    using W = WarpLayout<EPI>;
    constexpr int kEpiWarps = W::kEpiWarps;
    constexpr int kEpiGroups = W::kGroups;
    constexpr int CG = S::kCG;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t stages = static_cast<uint32_t>(p.stages);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + STAGES;
    uint64_t* rbar = empty + STAGES;  // kMaxBoxes per epilogue warp
    SharedCtl* ctl = reinterpret_cast<SharedCtl*>(rbar + kMaxBoxes * kEpiWarps);
    uint8_t* ring = smem + S::kCtlBytes;
    uint8_t* dstage = ring + stages * S::kStageBytes;
    const bool r_async = (NUM_B == 1) && (p.flags & kFlagRAsync);
    uint8_t* rstage = dstage + kEpiWarps * p.d_boxes * kDStageBytes;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // (the wait limit p.timeout_ns is read from the parameter space where used: no register held)
#ifdef GB_TRACE
    unsigned long long* trace = p.trace ? p.trace + static_cast<size_t>(blockIdx.x) * kTraceWords : nullptr;
    if (trace && threadIdx.x == 0) trace[kTrStartNs] = global_timer_ns();
#endif
    const uint32_t crank = PAIR ? cluster_ctarank() : 0u;  // position in the cluster (pair, or two pairs)
    const uint32_t rank = crank & 1u;                      // position in the CTA pair
    const uint32_t pairi = crank >> 1;                     // which pair of the cluster (A multicast)
    const uint32_t lead = crank & ~1u;                     // cluster rank of this pair's leader
    const bool leader = rank == 0;
    const bool mc = PAIR && p.mc != 0;
    const int32_t cta_per_unit = PAIR ? (mc ? 4 : 2) : 1;
    const int32_t unit = static_cast<int32_t>(blockIdx.x) / cta_per_unit;
    const int32_t units = static_cast<int32_t>(gridDim.x) / cta_per_unit;
    const uint16_t pair_mask = static_cast<uint16_t>(0x3u << lead);  // both CTAs of this pair
    const int32_t num_work = p.num_tiles * p.splits;
    // ping-pong takes effect with two epilogue warpgroups and no split only
    const bool pingpong = W::kLean || (kEpiGroups == 2 && p.pingpong != 0 && p.splits == 1);
    constexpr int kGroupsPerBuffer = W::kLean ? 2 : 1;  // with ping-pong: warpgroups serving one TMEM buffer

    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < stages; ++s) {
            mbar_init(smem_addr(&full[s]), 1);
            // with A multicast a stage is free once both pairs' MMAs have read it
            mbar_init(smem_addr(&empty[s]), mc ? 2 : 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_addr(&ctl->acc_full[b]), 1);
            // every epilogue warp of the pair frees a buffer; with ping-pong only the
            // warpgroup that owns it
            mbar_init(smem_addr(&ctl->acc_empty[b]), pingpong ? S::kAccEmptyArrivals / kEpiGroups * kGroupsPerBuffer
                                                              : S::kAccEmptyArrivals);
        }
        mbar_init(smem_addr(&ctl->drain), 1);
        // an R box lands on one arrival with its byte count (TMA); a cp.async slot on the
        // 32 lanes' arrivals as their copies land
        for (int i = 0; i < kMaxBoxes * kEpiWarps; ++i) mbar_init(smem_addr(&rbar[i]), r_async ? 32 : 1);
        ctl->abort = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        if (p.num_k_blocks > 0) {
            tma_prefetch_desc(mc ? &p.tm_a_half : &p.tm_a);
            tma_prefetch_desc(&p.tm_b0);
            if (NUM_B == 2) tma_prefetch_desc(&p.tm_b1);
        }
        if (p.flags & kFlagDTma) tma_prefetch_desc(&p.tm_d);
        if (p.flags & kFlagRTma) tma_prefetch_desc(&p.tm_r);
        if (p.flags & kFlagZTma) tma_prefetch_desc(&p.tm_z);
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
#ifdef GB_TRACE
    if (trace && threadIdx.x == 0) trace[kTrSetupNs] = global_timer_ns();
#endif

    // Role split.  Each warpgroup sets its register budget inside its own branch, so
    // the compiler holds the control roles to the small budget and gives the
    // epilogue the large one; only the short teardown after the branches is shared.
    if (warp < kEpiWarp0) {
        if constexpr (W::kRealloc) setmaxnreg_dec<W::kRegsControl>();
        // An MN-major B tile is two TMA boxes per stage: with two producer threads, warps 2
        // and 3 take the B loads of alternate stages, so no thread issues more than one
        // stage's worth of boxes per stage time (one thread issuing two boxes per stage
        // falls behind the MMAs: measured on GB300, the MatmulOp MLP 0.731 -> 0.663 ms with
        // the split; the same split costs the one-box K-major B 4 %, so it is MN-major only)
        const bool b_par = (p.flags & kFlagBMn) && p.prod == 2;
        if (warp == 0 || (warp == 2 && p.prod >= 2) || (warp == 3 && (p.prod == 3 || b_par))) {
            // ------------------------------------------------------------ producer (every CTA)
            // One thread issues every stage's loads, or two split them: warp 0 the A tile (and
            // the leader's expected byte count), warp 2 the B tile.  Both wait for the stage
            // to be free; the full barrier completes when all of the stage's bytes have landed.
            // prod == 3: warps 0 and 2 load the upper and lower halves of the A tile, warp 3 B
            const bool split_a = p.prod == 3 && !mc;
            const bool do_a = warp == 0 || (split_a && warp == 2);
            const bool do_b = p.prod == 1 || (p.prod == 2 && (warp == 2 || (b_par && warp == 3))) ||
                              (p.prod == 3 && warp == 3);
            if (lane == 0) {
                uint32_t it = 0;
                uint32_t s = 0, ph = 0;  // ring slot and phase of k-block `it`
                bool ok = true;
                int32_t local = 0;
                const uint64_t pol_a = l2_policy(p.hint_a);
                const uint64_t pol_b = l2_policy(p.hint_b);
                TraceAcc tr_empty;
                // Lean loop for the common form (K-major B, A by warp 0 and B by warp 2, no A
                // multicast, no test hook): per k-block only the stage wait, the byte count and
                // this thread's one box, with the box's map, rows and offset fixed per tile.
                // Measured on GB300: the same loads issued from the general loop below, which
                // branches per k-block on those options, leave the tensor pipe idle longer (MLP
                // launch 0.678 -> 0.601 ms with this loop alone, one CTA pair 1.69 -> 1.44 ms).
                const bool lean_loads = !mc && !(p.flags & kFlagBMn) && p.prod == 2 && p.inject == 0;
                // the same for an MN-major B (two boxes per stage; warps 2 and 3 take the B
                // boxes of alternate stages)
                const bool lean_mn = !mc && b_par && NUM_B == 1 && p.inject == 0;
                // and with A multicast between two pairs (4-CTA clusters): warp 0 loads its
                // 64-row half of the A tile into its own and the other pair's same-rank CTA
                const bool lean_mc = mc && !(p.flags & kFlagBMn) && p.prod == 2 && p.inject == 0;
                const bool is_a = warp == 0;
                for (int32_t w = unit; lean_loads && ok && w < num_work; w += units, ++local) {
                    const int32_t tile = w / p.splits;
                    const int32_t kb0 = (w - tile * p.splits) * p.kb_per_split;
                    const int32_t nkb = min(p.num_k_blocks - kb0, p.kb_per_split);
                    int32_t mb, nb;
                    work_tile(tile, p, pairi, mb, nb);
                    const bool reverse = p.zigzag && (local & 1);
                    // this thread's box: A rows of this CTA; B rows of this CTA's half of the pair
                    // tile, or (two B operands in a pair) the whole BN rows of this CTA's operand
                    const CUtensorMap* map = is_a ? &p.tm_a : (NUM_B == 2 && PAIR && !leader) ? &p.tm_b1 : &p.tm_b0;
                    const int32_t row = is_a ? mb * S::kTileM + static_cast<int32_t>(rank) * kBM
                                             : nb * BN + (NUM_B == 1 ? static_cast<int32_t>(rank) * S::kBRows : 0);
                    const uint32_t off = is_a ? 0u : static_cast<uint32_t>(S::kABytes);
                    const uint64_t pol = is_a ? pol_a : pol_b;
                    for (int32_t kk = 0; kk < nkb; ++kk, ++it) {
                        const int32_t kb = kb0 + (reverse ? nkb - 1 - kk : kk);
                        if (it > 0 && ++s == stages) {
                            s = 0;
                            ph ^= 1u;
                        }
                        if (!wait_bar<kRingSuspendNs>(smem_addr(&empty[s]), ph ^ 1u, abort_flag, p.timeout_ns, kRoleProducer, s, &tr_empty)) {
                            ok = false;
                            break;
                        }
                        const uint32_t own_full = smem_addr(&full[s]);
                        if (leader && is_a) mbar_arrive_expect_tx(own_full, S::kTxBytes);
                        const uint32_t dst = smem_addr(ring + s * S::kStageBytes) + off;
                        if constexpr (PAIR) {
                            tma_load_op<true>(dst, map, mapa_shared(own_full, lead), kb * kBK, row, pol);
                        } else {
                            tma_load_op<false>(dst, map, own_full, kb * kBK, row, pol);
                            if (NUM_B == 2 && !is_a)
                                tma_load_op<false>(dst + BN * kBK * 2, &p.tm_b1, own_full, kb * kBK, row, pol);
                        }
                    }
                }
                for (int32_t w = unit; lean_mn && ok && w < num_work; w += units, ++local) {
                    const int32_t tile = w / p.splits;
                    const int32_t kb0 = (w - tile * p.splits) * p.kb_per_split;
                    const int32_t nkb = min(p.num_k_blocks - kb0, p.kb_per_split);
                    int32_t mb, nb;
                    work_tile(tile, p, pairi, mb, nb);
                    const bool reverse = p.zigzag && (local & 1);
                    const int32_t a_row = mb * S::kTileM + static_cast<int32_t>(rank) * kBM;
                    const int32_t b_row = nb * BN + static_cast<int32_t>(rank) * S::kBRows;
                    const uint32_t my_parity = warp == 3 ? 1u : 0u;
                    for (int32_t kk = 0; kk < nkb; ++kk, ++it) {
                        const int32_t kb = kb0 + (reverse ? nkb - 1 - kk : kk);
                        if (it > 0 && ++s == stages) {
                            s = 0;
                            ph ^= 1u;
                        }
                        if (!is_a && (it & 1u) != my_parity) continue;  // the other B thread's stage
                        if (!wait_bar<kRingSuspendNs>(smem_addr(&empty[s]), ph ^ 1u, abort_flag, p.timeout_ns, kRoleProducer, s, &tr_empty)) {
                            ok = false;
                            break;
                        }
                        const uint32_t own_full = smem_addr(&full[s]);
                        if (leader && is_a) mbar_arrive_expect_tx(own_full, S::kTxBytes);
                        const uint32_t fb = PAIR ? mapa_shared(own_full, lead) : own_full;
                        const uint32_t dst = smem_addr(ring + s * S::kStageBytes);
                        if (is_a) {
                            tma_load_op<PAIR>(dst, &p.tm_a, fb, kb * kBK, a_row, pol_a);
                        } else {
#pragma unroll
                            for (int h = 0; h < S::kBRows / 64; ++h)
                                tma_load_op<PAIR>(dst + S::kABytes + h * kMnBoxBytes, &p.tm_b0, fb, b_row + h * 64, kb * kBK,
                                                  pol_b);
                        }
                    }
                }
                if constexpr (PAIR) {
                    const uint16_t mc_mask = static_cast<uint16_t>((1u << rank) | (1u << (2 + rank)));
                    for (int32_t w = unit; lean_mc && ok && w < num_work; w += units, ++local) {
                        const int32_t tile = w / p.splits;
                        const int32_t kb0 = (w - tile * p.splits) * p.kb_per_split;
                        const int32_t nkb = min(p.num_k_blocks - kb0, p.kb_per_split);
                        int32_t mb, nb;
                        work_tile(tile, p, pairi, mb, nb);
                        const bool reverse = p.zigzag && (local & 1);
                        const CUtensorMap* map = is_a ? &p.tm_a_half : (NUM_B == 2 && !leader) ? &p.tm_b1 : &p.tm_b0;
                        const int32_t row = is_a ? mb * S::kTileM + static_cast<int32_t>(rank) * kBM +
                                                       static_cast<int32_t>(pairi) * (kBM / 2)
                                                 : nb * BN + (NUM_B == 1 ? static_cast<int32_t>(rank) * S::kBRows : 0);
                        const uint32_t off = is_a ? pairi * (S::kABytes / 2) : static_cast<uint32_t>(S::kABytes);
                        for (int32_t kk = 0; kk < nkb; ++kk, ++it) {
                            const int32_t kb = kb0 + (reverse ? nkb - 1 - kk : kk);
                            if (it > 0 && ++s == stages) {
                                s = 0;
                                ph ^= 1u;
                            }
                            if (!wait_bar<kRingSuspendNs>(smem_addr(&empty[s]), ph ^ 1u, abort_flag, p.timeout_ns, kRoleProducer, s,
                                                          &tr_empty)) {
                                ok = false;
                                break;
                            }
                            const uint32_t own_full = smem_addr(&full[s]);
                            if (leader && is_a) mbar_arrive_expect_tx(own_full, S::kTxBytes);
                            const uint32_t dst = smem_addr(ring + s * S::kStageBytes) + off;
                            const uint32_t fb = mapa_shared(own_full, lead);
                            if (is_a) tma_load_2d_pair_multicast(dst, map, fb, kb * kBK, row, mc_mask);
                            else tma_load_op<true>(dst, map, fb, kb * kBK, row, pol_b);
                        }
                    }
                }
                for (int32_t w = unit; !lean_loads && !lean_mn && !lean_mc && ok && w < num_work; w += units, ++local) {
                    const int32_t tile = w / p.splits;
                    const int32_t kb0 = (w - tile * p.splits) * p.kb_per_split;
                    const int32_t nkb = min(p.num_k_blocks - kb0, p.kb_per_split);
                    int32_t mb, nb;
                    work_tile(tile, p, pairi, mb, nb);
                    const bool reverse = p.zigzag && (local & 1);
                    const int32_t a_row = mb * S::kTileM + static_cast<int32_t>(rank) * kBM;
                    const int32_t b_row = nb * BN + static_cast<int32_t>(rank) * S::kBRows;
                    for (int32_t kk = 0; kk < nkb; ++kk, ++it) {
                        const int32_t kb = kb0 + (reverse ? nkb - 1 - kk : kk);
                        if (kk > 0 || it > 0) {
                            if (++s == stages) {
                                s = 0;
                                ph ^= 1u;
                            }
                        }
                        // the other B thread's stage (MN-major B with two producer threads)
                        if (b_par && warp != 0 && (it & 1u) != (warp == 3 ? 1u : 0u)) continue;
                        if (!wait_bar<kRingSuspendNs>(smem_addr(&empty[s]), ph ^ 1u, abort_flag, p.timeout_ns, kRoleProducer, s, &tr_empty)) {
                            ok = false;
                            break;
                        }
                        if (p.inject == kInjectSkipFirstStage && it == 0 && leader && warp == 0) continue;  // test hook
                        uint8_t* st = ring + s * S::kStageBytes;
                        const uint32_t own_full = smem_addr(&full[s]);
                        if (leader && warp == 0) mbar_arrive_expect_tx(own_full, S::kTxBytes);
                        uint8_t* sb = st + S::kABytes;
                        if (mc && do_a) {
                            // A multicast: this CTA loads rows [pairi * 64, +64) of its 128-row A
                            // tile into that offset of its own and the other pair's same-rank CTA
                            const uint32_t fb = mapa_shared(own_full, lead);
                            tma_load_2d_pair_multicast(smem_addr(st + pairi * (S::kABytes / 2)), &p.tm_a_half, fb,
                                                       kb * kBK, a_row + static_cast<int32_t>(pairi) * (kBM / 2),
                                                       static_cast<uint16_t>((1u << rank) | (1u << (2 + rank))));
                        }
                        if (NUM_B == 1 && (p.flags & kFlagBMn)) {
                            // MN-major B (a row-major [K, N] matrix): boxes of 64 output columns
                            // x 64 contraction rows, one after the other along N
                            const uint32_t fb = PAIR ? mapa_shared(own_full, lead) : own_full;
                            if (split_a && do_a) {
                                const int32_t half = warp == 0 ? 0 : 1;
                                tma_load_op<PAIR>(smem_addr(st + half * (S::kABytes / 2)), &p.tm_a_half, fb, kb * kBK,
                                                  a_row + half * (kBM / 2), pol_a);
                            } else if (!mc && do_a) {
                                tma_load_op<PAIR>(smem_addr(st), &p.tm_a, fb, kb * kBK, a_row, pol_a);
                            }
                            if (do_b) {
#pragma unroll
                                for (int h = 0; h < S::kBRows / 64; ++h)
                                    tma_load_op<PAIR>(smem_addr(sb + h * kMnBoxBytes), &p.tm_b0, fb, b_row + h * 64,
                                                      kb * kBK, pol_b);
                            }
                        } else if constexpr (PAIR) {
                            const uint32_t fb = mapa_shared(own_full, lead);  // the pair leader's full barrier
                            if (split_a && do_a) {  // this warp's 64-row half of the A tile
                                const int32_t half = warp == 0 ? 0 : 1;
                                tma_load_op<true>(smem_addr(st + half * (S::kABytes / 2)), &p.tm_a_half, fb, kb * kBK,
                                                  a_row + half * (kBM / 2), pol_a);
                            } else if (!mc && do_a) {
                                tma_load_op<true>(smem_addr(st), &p.tm_a, fb, kb * kBK, a_row, pol_a);
                            }
                            if (do_b) {
                                if (NUM_B == 1)
                                    tma_load_op<true>(smem_addr(sb), &p.tm_b0, fb, kb * kBK, b_row, pol_b);
                                else  // this CTA's half of the N = 2 BN operand is one whole product
                                    tma_load_op<true>(smem_addr(sb), leader ? &p.tm_b0 : &p.tm_b1, fb, kb * kBK,
                                                      nb * BN, pol_b);
                            }
                        } else {
                            if (split_a && do_a) {
                                const int32_t half = warp == 0 ? 0 : 1;
                                tma_load_op<false>(smem_addr(st + half * (S::kABytes / 2)), &p.tm_a_half, own_full,
                                                   kb * kBK, a_row + half * (kBM / 2), pol_a);
                            } else if (do_a) {
                                tma_load_op<false>(smem_addr(st), &p.tm_a, own_full, kb * kBK, a_row, pol_a);
                            }
                            if (do_b) {
                                tma_load_op<false>(smem_addr(sb), &p.tm_b0, own_full, kb * kBK,
                                                   NUM_B == 1 ? b_row : nb * BN, pol_b);
                                if (NUM_B == 2)
                                    tma_load_op<false>(smem_addr(sb + BN * kBK * 2), &p.tm_b1, own_full, kb * kBK,
                                                       nb * BN, pol_b);
                            }
                        }
                    }
                }
#ifdef GB_TRACE
                if (trace && warp == 0) {
                    trace[kTrProdEmptyCyc] = tr_empty.cyc;
                    trace[kTrProdEmptyN] = tr_empty.n;
                }
#endif
                if (!ok && leader) {
                    // Drain: the leader's full barriers count the bytes of both CTAs (and of
                    // both producer threads); wait (bounded) for the k-blocks this thread
                    // issued among the last `stages` to land.
                    const uint32_t first = it > stages ? it - stages : 0u;
                    for (uint32_t i = first; i < it; ++i) {
                        if (p.inject == kInjectSkipFirstStage && i == 0) continue;
                        drain_bar(smem_addr(&full[i % stages]), (i / stages) & 1u, p.timeout_ns);
                    }
                }
            }
            __syncwarp();
        } else if (warp == 1) {
            // ------------------------------------------------------------ MMA issuer (leader CTA)
            if (lane == 0 && leader) {
                uint32_t it = 0;
                uint32_t s = 0, ph = 0;  // ring slot and phase of k-block `it`
                bool ok = true;
                bool issued = false;
                int32_t local = 0;
                TraceAcc tr_full, tr_acc;
#ifdef GB_TRACE
                unsigned long long kb_hist[7] = {0, 0, 0, 0, 0, 0, 0};  // [6]: cycles inside every full wait
                long long kb_prev = 0;
#endif
                const bool b_mn = NUM_B == 1 && (p.flags & kFlagBMn);
                const uint32_t idesc = S::kIdesc | (b_mn ? kIdescBMnMajor : 0u);
                const uint32_t bstep = b_mn ? (16u * 128u) >> 4 : 2u;
                // the common forms' loop (measured on GB300 with the lean load loop: MLP launch
                // 0.601 -> 0.590 ms, one CTA pair 1.44 -> 1.31 ms)
                const bool lean_issue = p.issue == 0 && !(mc && b_mn);
#ifdef GB_TRACE
                const long long mma_c0 = clock64();
                if (trace) trace[kTrMmaFirstNs] = 0;
#endif
                for (int32_t w = unit; ok && w < num_work; w += units, ++local) {
                    const int32_t tile = w / p.splits;
                    const int32_t kb0 = (w - tile * p.splits) * p.kb_per_split;
                    const int32_t nkb = min(p.num_k_blocks - kb0, p.kb_per_split);
                    const uint32_t b = local & 1;
                    const uint32_t aph = (local >> 1) & 1u;
                    if (!wait_bar<kRingSuspendNs>(smem_addr(&ctl->acc_empty[b]), aph ^ 1u, abort_flag, p.timeout_ns, kRoleMma, 0x100u | b,
                                  &tr_acc)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t d_tmem = tmem_base + b * kAccStride;
                    if (lean_issue) {
#ifdef GB_TRACE
                        if (trace && !issued) trace[kTrMmaFirstNs] = global_timer_ns();
#endif
                        const bool kb_ok =
                            b_mn ? issue_kblocks<CG, S::kStageBytes, S::kABytes, S::kIdesc, true>(
                                       d_tmem, nkb, full, empty, ring, stages, s, ph, it, abort_flag, p.timeout_ns, tr_full, issued)
                            : mc ? issue_kblocks<CG, S::kStageBytes, S::kABytes, S::kIdesc, false, 0xF>(
                                       d_tmem, nkb, full, empty, ring, stages, s, ph, it, abort_flag, p.timeout_ns, tr_full, issued)
                                 : issue_kblocks<CG, S::kStageBytes, S::kABytes, S::kIdesc, false>(
                                       d_tmem, nkb, full, empty, ring, stages, s, ph, it, abort_flag, p.timeout_ns, tr_full, issued);
                        if (!kb_ok) {
                            ok = false;
                            break;
                        }
                        if constexpr (PAIR) mma_commit_multicast2(smem_addr(&ctl->acc_full[b]), pair_mask);
                        else mma_commit<1>(smem_addr(&ctl->acc_full[b]));
                        continue;
                    }
                    if (p.issue == 1 || p.issue == 2) {
                        // Lean issue: the stage's descriptors advance with the ring position
                        // (no per-k-block rebuild), and with issue == 2 the next stage's wait and
                        // fence run while this k-block's third MMA executes.
                        if (!issue_tile_lean<CG, S::kStageBytes, S::kABytes>(
                                p, d_tmem, nkb, full, empty, ring, stages, s, ph, it, b_mn, idesc, bstep,
                                mc ? static_cast<uint16_t>(0xF) : pair_mask, abort_flag, p.timeout_ns, tr_full, issued)) {
                            ok = false;
                            break;
                        }
                        if constexpr (PAIR) mma_commit_multicast2(smem_addr(&ctl->acc_full[b]), pair_mask);
                        else mma_commit<1>(smem_addr(&ctl->acc_full[b]));
                        continue;
                    }
                    for (int32_t kk = 0; kk < nkb; ++kk, ++it) {
                        if (it > 0 && ++s == stages) {
                            s = 0;
                            ph ^= 1u;
                        }
#ifdef GB_TRACE
                        const unsigned long long blocked_before = tr_full.n;
                        const long long wait_c0 = clock64();
#endif
                        if (!wait_bar<kRingSuspendNs>(smem_addr(&full[s]), ph, abort_flag, p.timeout_ns, kRoleMma, s, &tr_full)) {
                            ok = false;
                            break;
                        }
#ifdef GB_TRACE
                        kb_hist[6] += static_cast<unsigned long long>(clock64() - wait_c0);
#endif
                        tc_fence_after_sync();
#ifdef GB_TRACE
                        if (trace && !issued) trace[kTrMmaFirstNs] = global_timer_ns();
                        {
                            const long long now = clock64();
                            if (kk > 0) {
                                const long long d = now - kb_prev;
                                if (tr_full.n != blocked_before) {
                                    kb_hist[5] += static_cast<unsigned long long>(d);
                                } else {
                                    kb_hist[d < 560 ? 0 : d < 700 ? 1 : d < 1000 ? 2 : 3] += 1;
                                    kb_hist[4] += static_cast<unsigned long long>(d);
                                }
                            }
                            kb_prev = now;
                        }
#endif
                        const uint32_t a_addr = smem_addr(ring + s * S::kStageBytes);
                        const uint64_t adesc = sdesc_kmajor_sw128(a_addr);
                        const uint64_t bdesc = b_mn ? sdesc_mnmajor_sw128(a_addr + S::kABytes, kMnBoxBytes)
                                                    : sdesc_kmajor_sw128(a_addr + S::kABytes);
                        // per 16-element K slice: +32 bytes in a K-major tile, +16 rows of 128 bytes
                        // in an MN-major one (+2 / +128 in the >>4-encoded address); the four MMAs
                        // leave one asm block back to back
                        if (p.issue == 3) {  // the MMAs as four separate statements (comparison)
#pragma unroll
                            for (int j = 0; j < kBK / 16; ++j)
                                mma_bf16<CG>(d_tmem, adesc + 2 * j, bdesc + bstep * j, idesc, (kk > 0 || j > 0) ? 1u : 0u);
                        } else {
                            const uint64_t bdesc1 = bdesc + bstep, bdesc2 = bdesc1 + bstep, bdesc3 = bdesc2 + bstep;
                            mma_bf16_x4<CG>(d_tmem, adesc, adesc + 2, adesc + 4, adesc + 6, bdesc, bdesc1, bdesc2,
                                            bdesc3, idesc, kk > 0 ? 1u : 0u);
                        }
                        issued = true;
                        // the stage is free in this pair (and, with A multicast, in the other pair's
                        // view too: its producers write A halves into this pair's stage)
                        if constexpr (PAIR) mma_commit_multicast2(smem_addr(&empty[s]), mc ? 0xF : pair_mask);
                        else mma_commit<1>(smem_addr(&empty[s]));
                    }
                    if (!ok) break;
                    if constexpr (PAIR) mma_commit_multicast2(smem_addr(&ctl->acc_full[b]), pair_mask);
                    else mma_commit<1>(smem_addr(&ctl->acc_full[b]));
                }
#ifdef GB_TRACE
                if (trace) {
                    trace[kTrMmaLastNs] = global_timer_ns();
                    trace[kTrMmaCyc] = static_cast<unsigned long long>(clock64() - mma_c0);
                    trace[kTrMmaFullCyc] = tr_full.cyc;
                    trace[kTrMmaFullN] = tr_full.n;
                    trace[kTrMmaAccCyc] = tr_acc.cyc;
                    trace[kTrMmaAccN] = tr_acc.n;
                    trace[kTrMmaItems] = static_cast<unsigned long long>(local);
                    for (int i = 0; i < 7; ++i) trace[kTrKbFast + i] = kb_hist[i];
                }
#endif
                if (!ok && issued) {
                    // Drain: every MMA issued so far must finish before TMEM is freed.
                    mma_commit<CG>(smem_addr(&ctl->drain));
                    drain_bar(smem_addr(&ctl->drain), 0, p.timeout_ns);
                }
            }
            __syncwarp();
        }
    } else {
        if constexpr (W::kRealloc) setmaxnreg_inc<W::kRegsEpilogue>();
        // ------------------------------------------------------------ epilogue (every CTA)
        const int e = warp - kEpiWarp0;  // epilogue warp index: staging buffers, counters
        const int q = e & 3;              // == warp % 4: this warp's TMEM lane quadrant
        const int g = e >> 2;             // this warp's warpgroup among the epilogue warpgroups
        // Chunks of a tile this warp stores: g, g + kEpiGroups, ... when the warpgroups
        // share every tile; all of them, on every other tile, with ping-pong (lean variant:
        // g % 2, g % 2 + 2, ... on the tiles of parity g / 2).
        const bool pp = pingpong;
        const int owner = W::kLean ? g >> 1 : g;  // with ping-pong: the tile parity this warp serves
        const int c0 = pp ? (W::kLean ? (g & 1) : 0) : g;
        const int cstep = pp ? kGroupsPerBuffer : kEpiGroups;
        constexpr int kChunks = BN / kDChunk;
        const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
        const int32_t slab_row = static_cast<int32_t>(rank) * kBM + q * 32 + lane;  // row within the tile
        constexpr int64_t kPartFloats = static_cast<int64_t>(S::kTileM) * BN;       // one partial accumulator
        const uint32_t dbox = smem_addr(dstage) + e * p.d_boxes * kDStageBytes;  // this warp's D staging queue
        int32_t dslot = 0;
        int32_t local = 0;
        TraceAcc tr_accfull;
#ifdef GB_TRACE
        unsigned long long tr_body = 0;
        // per-phase counters in shared memory (no registers held across the loops); only the
        // first epilogue warp's lane 0 counts
        uint32_t* tr_ep = (e == 0 && lane == 0) ? ctl->trace_ep : nullptr;
        if (tr_ep)
            for (int i = 0; i < 8; ++i) tr_ep[i] = 0;
#endif

        // R by TMA (linear, no split): a cursor over this warp's future (tile, chunk)
        // pairs keeps up to r_boxes 32x32 R boxes in flight ahead of their use, so
        // the loads for the next tile overlap the current tile's MMAs.
        const bool r_tma = (NUM_B == 1) && (p.flags & kFlagRTma);
        // R rows not 16-byte aligned: the same queue, filled by per-lane cp.async word copies
        // (general path; the host sets this only without split-K)
        const bool r_queue = r_tma || r_async;
        const bool express = p.splits == 1 && p.num_k_blocks > 0 && (p.flags & kFlagDTma) &&
                             !(p.flags & (kFlagResidual | kFlagZ));
        // Paired path (R by TMA, D by TMA, no second output, no split): two chunks per
        // step, so the fixed cost of a step (waits, fence, warp syncs, branches) is
        // paid once per 64 columns and the two chunks' chains overlap.
        const bool paired = r_tma && p.splits == 1 && p.num_k_blocks > 0 && (p.flags & kFlagDTma) &&
                            !(p.flags & kFlagZ);
        // this warp's R boxes; also the transpose buffer for unaligned R rows (the
        // boxes are unused then)
        const uint32_t r_slot = r_slot_bytes(p);  // bytes per R queue entry
        const uint32_t rbox0 = smem_addr(rstage) + e * p.r_warp_bytes;
        const uint32_t tbuf_r = rbox0;
        // Wide boxes (paired path only): a step covers chunks (c, c + 1); warpgroup g takes
        // the steps starting at chunk 2g, 2g + 2 * groups, ... (all of them with ping-pong),
        // i.e. first chunk 2 * c0 and stride 2 * cstep.  The R cursor walks this warp's R
        // boxes: chunks, or the first chunks of wide steps.
        // With 32x64 D boxes only (kFlagWideD) the steps are the same adjacent pairs but R
        // still comes in 32x32 boxes: the cursor walks 2c0, 2c0 + 1, 2c0 + 2 cstep, ...
        const bool wide = (NUM_B == 1) && (p.flags & kFlagWide);
        const bool adj = (NUM_B == 1) && (p.flags & (kFlagWide | kFlagWideD));  // steps of adjacent chunks
        int32_t rc_w = unit, rc_local = 0, rc_c = adj ? 2 * c0 : c0, rc_mb = -1, rc_nb = -1;
        // the cursor's next R box after rc_c within a tile
        auto rc_next = [&](int32_t c) { return wide ? c + 2 * cstep : adj ? ((c & 1) ? c + 2 * cstep - 1 : c + 1) : c + cstep; };
        uint32_t r_pending = 0, r_phase = 0;  // R boxes issued and not yet used; one parity bit per box
        int32_t r_islot = 0, r_uslot = 0;                 // queue positions of the next load and the next use
        auto r_find = [&]() -> bool {  // move the cursor to the next chunk this warp will store
            while (rc_w < num_work) {
                if (pp && (rc_local & 1) != owner) {  // the other warpgroup's work item
                    rc_w += units;
                    ++rc_local;
                    continue;
                }
                if (rc_mb < 0) work_tile(rc_w, p, pairi, rc_mb, rc_nb);
                const int32_t r0 = rc_mb * S::kTileM + static_cast<int32_t>(rank) * kBM + q * 32;
                if (rc_c < kChunks && r0 < p.m && rc_nb * BN + rc_c * kDChunk < p.n) return true;
                rc_c = rc_next(rc_c);
                if (rc_c >= kChunks) {
                    rc_c = adj ? 2 * c0 : c0;
                    rc_w += units;
                    ++rc_local;
                    rc_mb = -1;
                }
            }
            return false;
        };
        auto r_issue = [&]() {
            if (!r_queue || !r_find()) return;
            if (r_async) {
                // 32 rows x 17 words, row-major over the warp: copy t = 32 i + lane is word
                // t % 17 of row t / 17, so each instruction reads consecutive words of two or three rows
                // and writes 128 contiguous bytes of the slot.  A word reads only the bytes
                // of its row segment [n0, n0 + valid) (src-size), except that a segment
                // starting on a 2-byte boundary also reads the element just before it (in
                // the tensor: the base is 4-byte aligned, so that element index is >= 0).
                const int32_t rbase = rc_mb * S::kTileM + static_cast<int32_t>(rank) * kBM + q * 32;
                const int32_t n0 = rc_nb * BN + rc_c * kDChunk;
                const int32_t valid = min(kDChunk, p.n - n0);
                const uint32_t dst0 = rbox0 + r_islot * kRSlotAsyncBytes;
                const uint32_t bar = smem_addr(&rbar[e * kMaxBoxes + r_islot]);
                const uintptr_t base = reinterpret_cast<uintptr_t>(p.r);
#pragma unroll 1
                for (uint32_t i = 0; i < kRSlotWords; ++i) {
                    const uint32_t t = i * 32u + static_cast<uint32_t>(lane);
                    const uint32_t rr = t / kRSlotWords;
                    const uint32_t j = t - rr * kRSlotWords;
                    const int32_t row = rbase + static_cast<int32_t>(rr);
                    const void* src = p.r;
                    uint32_t bytes = 0;
                    if (row < p.m) {
                        const uintptr_t a = base + 2u * static_cast<uintptr_t>(static_cast<int64_t>(row) * p.ldr + n0);
                        const uintptr_t w = (a & ~static_cast<uintptr_t>(3)) + 4u * j;
                        const uintptr_t end = a + 2u * static_cast<uintptr_t>(valid);
                        if (w < end) {
                            bytes = static_cast<uint32_t>(min(static_cast<uintptr_t>(4), end - w));
                            src = reinterpret_cast<const void*>(w);
                        }
                    }
                    cp_async_4(dst0 + 4u * t, src, bytes);
                }
                cp_async_mbar_arrive_noinc(bar);
            } else if (lane == 0) {
                const uint32_t bar = smem_addr(&rbar[e * kMaxBoxes + r_islot]);
                mbar_arrive_expect_tx(bar, r_slot);
                tma_load_op<false>(rbox0 + r_islot * r_slot, &p.tm_r, bar, rc_nb * BN + rc_c * kDChunk,
                                   rc_mb * S::kTileM + static_cast<int32_t>(rank) * kBM + q * 32, l2_policy(p.hint_r));
            }
            ++r_pending;
            if (++r_islot == p.r_boxes) r_islot = 0;
            rc_c = rc_next(rc_c);
            if (rc_c >= kChunks) {
                rc_c = adj ? 2 * c0 : c0;
                rc_w += units;
                ++rc_local;
                rc_mb = -1;
            }
        };
        if (r_queue)
            for (int i = 0; i < p.r_boxes; ++i) r_issue();

        for (int32_t w = unit; w < num_work; w += units, ++local) {
            if (pp && (local & 1) != owner) continue;  // the other warpgroups' tile
            const uint32_t b = local & 1;
            const uint32_t aph = (local >> 1) & 1u;
            bool ok = true;
            if (lane == 0)
                ok = wait_bar<kRingSuspendNs>(smem_addr(&ctl->acc_full[b]), aph, abort_flag, p.timeout_ns, kRoleEpilogue, b, &tr_accfull);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after_sync();
#ifdef GB_TRACE
            const long long body_c0 = clock64();
            struct BodyTimer {  // adds the cycles of this iteration, however it ends
                unsigned long long& sum;
                long long c0;
                __device__ ~BodyTimer() { sum += static_cast<unsigned long long>(clock64() - c0); }
            } body_timer{tr_body, body_c0};
#endif

            const int32_t tile = w / p.splits;
            int32_t mb, nb;
            work_tile(tile, p, pairi, mb, nb);
            const int32_t row0 = mb * S::kTileM + static_cast<int32_t>(rank) * kBM + q * 32;  // this warp's slab
            const int32_t m = row0 + lane;
            const bool warp_rows = row0 < p.m;
            const uint32_t tcol = tmem_base + lane_base + b * kAccStride;
            if constexpr (!W::kLean) {
                if (express) {
                    // Express path (no epilogue input, no second output, TMA-stored D, no
                    // split): a compact loop, so the hot epilogue code next to the MMA
                    // issuer stays small.  With 32x64 D boxes (kFlagWideD) a step is two
                    // adjacent chunks (2 c0 + 2 i cstep and the next) staged into one box:
                    // one box wait, one proxy fence and one TMA store per 64 columns; a box
                    // half past N is clipped by the store.
                    if constexpr (EPI == 1) {
                        const bool wide_e = p.flags & kFlagWideD;
                        const int halves = wide_e ? 2 : 1;
                        const int adv = wide_e ? 2 * cstep : cstep;
                        const int nbox = wide_e ? p.d_boxes >> 1 : p.d_boxes;
#pragma unroll 1
                        for (int c = wide_e ? 2 * c0 : c0; c < kChunks; c += adv) {
                            const bool last_step = c + adv >= kChunks;
                            uint32_t buf = 0;
                            bool staged = false;
#pragma unroll 1
                            for (int i = 0; i < halves; ++i) {
                                const int ci = c + i;
                                const int32_t n0 = nb * BN + ci * kDChunk;
                                const bool chunk_on = warp_rows && n0 < p.n;
                                float v[32];
                                GB_TR_T0(tx);
                                if (chunk_on) {
                                    uint32_t r0[32];
                                    tmem_ld_32x32b_x32(tcol + ci * kDChunk, r0);
                                    if (NUM_B == 2) {
                                        uint32_t r1[32];
                                        tmem_ld_32x32b_x32(tcol + BN + ci * kDChunk, r1);
                                        tmem_wait_ld();
#pragma unroll
                                        for (int j = 0; j < 32; ++j) v[j] = silu(__uint_as_float(r0[j])) * __uint_as_float(r1[j]);
                                    } else {
                                        tmem_wait_ld();
#pragma unroll
                                        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r0[j]);
                                    }
                                }
                                if (last_step && i == halves - 1) {  // this warp's last TMEM reads of the buffer
                                    tc_fence_before_sync();
                                    __syncwarp();
                                    if (lane == 0) {
                                        if constexpr (PAIR) mbar_arrive_cluster(mapa_shared(smem_addr(&ctl->acc_empty[b]), lead));
                                        else mbar_arrive(smem_addr(&ctl->acc_empty[b]));
                                    }
                                }
                                GB_TR_ADD(tr_ep, kTrEpTmemLd, tx);
                                if (!chunk_on) continue;
                                if (NUM_B == 1) {
                                    if (p.flags & kFlagBias) add_bf16_row(v, p.bias + n0, min(32, p.n - n0), p.flags & kFlagBiasVec);
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
                                }
                                uint32_t packed[16];  // (packed before the box wait: v's registers are free by then)
#pragma unroll
                                for (int j = 0; j < 16; ++j) packed[j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);
                                GB_TR_ADD(tr_ep, kTrEpMath, tx);
                                if (!staged) {
                                    buf = dbox + dslot * d_slot_bytes(p);
                                    // the store that last used this box has read it
                                    if (lane == 0) bulk_wait_group_read_at_most(nbox - 1);
                                    __syncwarp();
                                    if (++dslot == nbox) dslot = 0;
                                    staged = true;
                                }
                                GB_TR_ADD(tr_ep, kTrEpDBox, tx);
                                {
                                    // 32x64 box, 128-byte swizzle: unit u of row r at u ^ (r % 8); 32x32
                                    // box, 64-byte swizzle: unit u at u ^ ((r / 2) % 4)
                                    const uint32_t row_addr = buf + lane * (wide_e ? 128 : 64);
                                    const uint32_t sw = wide_e ? (lane & 7u) : ((lane >> 1) & 3u);
                                    const uint32_t u0 = wide_e ? 4u * static_cast<uint32_t>(i) : 0u;
#pragma unroll
                                    for (uint32_t u = 0; u < 4; ++u)
                                        st_shared_v4(row_addr + (((u0 + u) ^ sw) << 4), packed[4 * u], packed[4 * u + 1],
                                                     packed[4 * u + 2], packed[4 * u + 3]);
                                }
                                GB_TR_ADD(tr_ep, kTrEpMath, tx);
                            }
                            if (!staged) continue;
                            GB_TR_T0(ts);
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                tma_store_op(&p.tm_d, buf, nb * BN + c * kDChunk, row0, p.hint_d);
                                bulk_commit_group();
                            }
                            GB_TR_ADD(tr_ep, kTrEpStore, ts);
#ifdef GB_TRACE
                            if (tr_ep) tr_ep[kTrEpSteps - kTrEpDBox] += 1;
#endif
                        }
                    } else {
                        // (two epilogue warpgroups: 32x32 boxes only -- the 32x64 step's extra live
                        // state does not fit the 168 registers of the 384-thread launch)
#pragma unroll 1
                        for (int c = c0; c < kChunks; c += cstep) {
                            const int32_t n0 = nb * BN + c * kDChunk;
                            const bool chunk_on = warp_rows && n0 < p.n;
                            float v[32];
                            GB_TR_T0(tx);
                            if (chunk_on) {
                                uint32_t r0[32];
                                tmem_ld_32x32b_x32(tcol + c * kDChunk, r0);
                                if (NUM_B == 2) {
                                    uint32_t r1[32];
                                    tmem_ld_32x32b_x32(tcol + BN + c * kDChunk, r1);
                                    tmem_wait_ld();
#pragma unroll
                                    for (int j = 0; j < 32; ++j) v[j] = silu(__uint_as_float(r0[j])) * __uint_as_float(r1[j]);
                                } else {
                                    tmem_wait_ld();
#pragma unroll
                                    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r0[j]);
                                }
                            }
                            if (c + cstep >= kChunks) {
                                tc_fence_before_sync();
                                __syncwarp();
                                if (lane == 0) {
                                    if constexpr (PAIR) mbar_arrive_cluster(mapa_shared(smem_addr(&ctl->acc_empty[b]), lead));
                                    else mbar_arrive(smem_addr(&ctl->acc_empty[b]));
                                }
                            }
                            GB_TR_ADD(tr_ep, kTrEpTmemLd, tx);
                            if (!chunk_on) continue;
                            if (NUM_B == 1) {
                                if (p.flags & kFlagBias) add_bf16_row(v, p.bias + n0, min(32, p.n - n0), p.flags & kFlagBiasVec);
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
                            }
                            uint32_t packed[16];
#pragma unroll
                            for (int j = 0; j < 16; ++j) packed[j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);
                            GB_TR_ADD(tr_ep, kTrEpMath, tx);
                            const uint32_t buf = dbox + dslot * kDStageBytes;
                            if (lane == 0) bulk_wait_group_read_at_most(p.d_boxes - 1);  // the store that last used this box has read it
                            __syncwarp();
                            GB_TR_ADD(tr_ep, kTrEpDBox, tx);
                            const uint32_t row_addr = buf + lane * 64;
                            const uint32_t sw = (lane >> 1) & 3u;
#pragma unroll
                            for (int u = 0; u < 4; ++u)
                                st_shared_v4(row_addr + ((u ^ sw) << 4), packed[4 * u], packed[4 * u + 1], packed[4 * u + 2],
                                             packed[4 * u + 3]);
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                tma_store_op(&p.tm_d, buf, n0, row0, p.hint_d);
                                bulk_commit_group();
                            }
                            if (++dslot == p.d_boxes) dslot = 0;
                            GB_TR_ADD(tr_ep, kTrEpStore, tx);
#ifdef GB_TRACE
                            if (tr_ep) tr_ep[kTrEpSteps - kTrEpDBox] += 1;
#endif
                        }
                    }
                    continue;
                }
            }
            if constexpr (NUM_B == 1) {
                if (paired) {
                    // This warp's chunks of the tile come in pairs (c, c + cs): kChunks /
                    // cstep is even for every variant.  The two chunks are computed one after
                    // the other (one chunk's registers), but share one wait for free D boxes,
                    // one proxy fence and one warp sync before their stores.  Chunk b is on
                    // only if chunk a is.  With wide boxes the pair is two adjacent chunks
                    // (cs = 1; pairs start at 2 * c0, 2 * c0 + 2 * cstep, ...) that share one
                    // 32x64 R box and one 32x64 D box (one TMA load, one store, one R wait);
                    // a box half past N is loaded as zeros and clipped by the store.
                    const bool wide_d = adj;  // 32x64 D boxes (with or without 32x64 R boxes)
                    const int cs = adj ? 1 : cstep;
                    bool rok = true;
#pragma unroll 1
                    for (int c = adj ? 2 * c0 : c0; c < kChunks; c += 2 * cstep) {
                        const bool last = c + 2 * cstep >= kChunks;
                        const int nchunks = !(warp_rows && nb * BN + c * kDChunk < p.n) ? 0
                                            : (nb * BN + (c + cs) * kDChunk < p.n ? 2 : 1);
                        GB_TR_T0(tx);
                        if (nchunks > 0) {
                            // D boxes free (two, or one wide): the stores that last used them
                            // have read them
                            if (lane == 0) bulk_wait_group_read_at_most(wide_d ? (p.d_boxes >> 1) - 1 : p.d_boxes - 2);
                            __syncwarp();
                        }
                        GB_TR_ADD(tr_ep, kTrEpDBox, tx);
#ifdef GB_TRACE
                        if (tr_ep) tr_ep[kTrEpSteps - kTrEpDBox] += 1;
#endif
                        uint32_t box_a = 0, rcur = 0;
#pragma unroll 1
                        for (int i = 0; i < 2; ++i) {
                            const int ci = c + i * cs;
                            const int32_t n0 = nb * BN + ci * kDChunk;
                            float v[32];
                            if (i < nchunks) {
                                uint32_t r0[32];
                                tmem_ld_32x32b_x32(tcol + ci * kDChunk, r0);
                                tmem_wait_ld();
#pragma unroll
                                for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r0[j]);
                            }
                            GB_TR_ADD(tr_ep, kTrEpTmemLd, tx);
                            if (last && i == 1) {  // this warp's last TMEM reads of the buffer are done
                                tc_fence_before_sync();
                                __syncwarp();
                                if (lane == 0) {
                                    if constexpr (PAIR) mbar_arrive_cluster(mapa_shared(smem_addr(&ctl->acc_empty[b]), lead));
                                    else mbar_arrive(smem_addr(&ctl->acc_empty[b]));
                                }
                            }
                            if (i >= nchunks) continue;
                            if (p.flags & kFlagBias) add_bf16_row(v, p.bias + n0, min(32, p.n - n0), p.flags & kFlagBiasVec);
                            switch ((p.flags & kFlagDact) ? 0 : p.act) {
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
                            GB_TR_ADD(tr_ep, kTrEpMath, tx);
                            if (!wide || i == 0) {
                                // this chunk's (step's) R box: the one at the use position of the queue
                                const uint32_t bar = smem_addr(&rbar[e * kMaxBoxes + r_uslot]);
                                const uint32_t par = (r_phase >> r_uslot) & 1u;
                                // every lane waits (and so acquires the TMA data) itself: no lane-0
                                // branch and broadcast on the per-step path
                                rok = __all_sync(0xffffffffu,
                                                 wait_bar(bar, par, abort_flag, p.timeout_ns, kRoleEpilogue, 0x200u | r_uslot));
                                if (!rok) break;
                                r_phase ^= 1u << r_uslot;
                                rcur = rbox0 + r_uslot * r_slot;
                                --r_pending;
                                if (++r_uslot == p.r_boxes) r_uslot = 0;
                            }
                            GB_TR_ADD(tr_ep, kTrEpRWait, tx);
                            uint32_t box = box_a;
                            if (!wide_d || i == 0) {
                                box = dbox + dslot * d_slot_bytes(p);
                                if (++dslot == (wide_d ? p.d_boxes >> 1 : p.d_boxes)) dslot = 0;
                            }
                            if (wide) apply_input_wide(p, v, rcur, i, lane);
                            else apply_input_box(p, v, rcur, lane);
                            if (wide_d) stage_wide_half(box, v, i, lane);
                            else stage_box_row(box, v, lane);
                            GB_TR_ADD(tr_ep, kTrEpMath, tx);
                            if (i == 0) {
                                box_a = box;
                                continue;
                            }
                            // both chunks staged: one proxy fence orders this lane's staging writes
                            // and R box reads before the TMA stores and the refills of the boxes
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                tma_store_op(&p.tm_d, box_a, n0 - cs * kDChunk, row0, p.hint_d);
                                bulk_commit_group();
                                if (!wide_d) {
                                    tma_store_op(&p.tm_d, box, n0, row0, p.hint_d);
                                    bulk_commit_group();
                                }
                            }
                            GB_TR_ADD(tr_ep, kTrEpStore, tx);
                        }
                        if (!rok) break;
                        if (nchunks == 1) {  // chunk a alone (b is past N)
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                tma_store_op(&p.tm_d, box_a, nb * BN + c * kDChunk, row0, p.hint_d);
                                bulk_commit_group();
                            }
                        }
                        GB_TR_T0(ti);
                        const int n_issue = wide ? (nchunks > 0 ? 1 : 0) : nchunks;
#pragma unroll 1
                        for (int i = 0; i < n_issue; ++i) r_issue();
                        GB_TR_ADD(tr_ep, kTrEpRIssue, ti);
                    }
                    if (!rok) break;
                    continue;
                }
            }

            if constexpr (!W::kLean) {
                const bool split_mode = p.splits > 1;
                // this slab's rows of the tile's fp32 accumulator (split-K only)
                float* acc_ws = p.ws + static_cast<int64_t>(tile) * NUM_B * kPartFloats + static_cast<int64_t>(slab_row) * BN;

#pragma unroll 1
                for (int c = c0; c < kChunks; c += cstep) {
                    const int32_t n0 = nb * BN + c * kDChunk;
                    const bool chunk_on = warp_rows && n0 < p.n;
                    float v[32];
                    GB_TR_T0(tg);
#ifdef GB_TRACE
                    if (tr_ep) tr_ep[kTrEpSteps - kTrEpDBox] += 1;
#endif
                    if (chunk_on && p.num_k_blocks > 0) {
                        uint32_t r0[32];
                        tmem_ld_32x32b_x32(tcol + c * kDChunk, r0);
                        if (NUM_B == 2) {
                            uint32_t r1[32];
                            tmem_ld_32x32b_x32(tcol + BN + c * kDChunk, r1);
                            tmem_wait_ld();
                            if (split_mode) {
                                if (m < p.m) {
                                    red_add_f32x32(acc_ws + c * kDChunk, r0);
                                    red_add_f32x32(acc_ws + kPartFloats + c * kDChunk, r1);
                                }
                            } else {
#pragma unroll
                                for (int j = 0; j < 32; ++j) v[j] = silu(__uint_as_float(r0[j])) * __uint_as_float(r1[j]);
                            }
                        } else {
                            tmem_wait_ld();
                            if (split_mode) {
                                if (m < p.m) red_add_f32x32(acc_ws + c * kDChunk, r0);
                            } else {
#pragma unroll
                                for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r0[j]);
                            }
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] = 0.0f;
                    }
                    if (c + cstep >= kChunks) {
                        // This warp's TMEM reads of this buffer are done: hand it back to the MMA issuer.
                        tc_fence_before_sync();
                        __syncwarp();
                        if (lane == 0) {
                            if constexpr (PAIR) mbar_arrive_cluster(mapa_shared(smem_addr(&ctl->acc_empty[b]), lead));
                            else mbar_arrive(smem_addr(&ctl->acc_empty[b]));
                        }
                    }
                    GB_TR_ADD(tr_ep, kTrEpTmemLd, tg);
                    if (!chunk_on || split_mode) continue;
                    uint32_t rbox = 0;
                    if (r_queue) {
                        const uint32_t bar = smem_addr(&rbar[e * kMaxBoxes + r_uslot]);
                        const uint32_t par = (r_phase >> r_uslot) & 1u;
                        bool rok = true;
                        // every lane waits (and so acquires the slot's data) itself
                        rok = __all_sync(0xffffffffu,
                                         wait_bar(bar, par, abort_flag, p.timeout_ns, kRoleEpilogue, 0x200u | r_uslot));
                        if (!rok) break;
                        r_phase ^= 1u << r_uslot;
                        rbox = rbox0 + r_uslot * r_slot;
                    }
                    GB_TR_ADD(tr_ep, kTrEpRWait, tg);
#ifdef GB_TRACE
                    finish_chunk<NUM_B>(p, v, m, row0, n0, lane, dbox, dslot, rbox, tbuf_r, tr_ep);
#else
                    finish_chunk<NUM_B>(p, v, m, row0, n0, lane, dbox, dslot, rbox, tbuf_r);
#endif
                    if (r_queue) {
                        __syncwarp();  // every lane has read the box: refill it
                        if (r_tma) fence_proxy_async_smem();
                        --r_pending;
                        if (++r_uslot == p.r_boxes) r_uslot = 0;
                        r_issue();
                    }
                }
                if (*abort_flag) break;
                if (!split_mode || !warp_rows) continue;

                // split-K: this partial is in the accumulator; the last split of the slab finishes it.
                __threadfence();
                __syncwarp();
                uint32_t* cnt = p.ws_cnt + tile * S::kSlabs + static_cast<int32_t>(rank) * kEpiWarps + e;
                uint32_t arrived = 0;
                if (lane == 0) arrived = atomicAdd(cnt, 1u);
                arrived = __shfl_sync(0xffffffffu, arrived, 0);
                if (arrived != static_cast<uint32_t>(p.splits - 1)) continue;
                __threadfence();
#pragma unroll 1
                for (int c = c0; c < kChunks; c += cstep) {
                    const int32_t n0 = nb * BN + c * kDChunk;
                    if (n0 >= p.n) break;
                    float v[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = 0.0f;
                    add_f32x32_cg(v, acc_ws + c * kDChunk);
                    if (NUM_B == 2) {
                        float v3[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j) v3[j] = 0.0f;
                        add_f32x32_cg(v3, acc_ws + kPartFloats + c * kDChunk);
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] = silu(v[j]) * v3[j];
                    }
                    finish_chunk<NUM_B>(p, v, m, row0, n0, lane, dbox, dslot, 0u, tbuf_r);
                }
            }
        }
#ifdef GB_TRACE
        if (trace && e == 0 && lane == 0) {
            trace[kTrEpiFullCyc] = tr_accfull.cyc;
            trace[kTrEpiFullN] = tr_accfull.n;
            trace[kTrEpiBodyCyc] = tr_body;
            trace[kTrEndNs] = global_timer_ns();
            for (int i = 0; i < 7; ++i) trace[kTrEpDBox + i] = tr_ep[i];
        }
#endif
        if (lane == 0) {
            // R boxes still in flight after an early stop (at most r_boxes, from the use
            // position on): wait (bounded) for them to land.
            int32_t slot = r_uslot;
            for (uint32_t i = 0; i < r_pending; ++i) {
                drain_bar(smem_addr(&rbar[e * kMaxBoxes + slot]), (r_phase >> slot) & 1u, p.timeout_ns);
                if (++slot == p.r_boxes) slot = 0;
            }
            // the staging boxes must outlive the TMA stores' reads of them; the stores'
            // global writes complete with the grid
            bulk_wait_group_read<0>();
        }
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
