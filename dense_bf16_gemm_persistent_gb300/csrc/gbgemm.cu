// C ABI of the library: argument validation, tile planning, TMA descriptor
// cache and kernel launch.  The device code lives in gemm_kernel.cuh.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cinttypes>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <algorithm>
#include <list>
#include <mutex>
#include <string>

#include "../../include/gbgemm.h"
#include "gemm_kernel.cuh"
#include "probe.cuh"

namespace {

using gb::GemmParams;

constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;  // TMA coordinates are signed 32-bit
constexpr int64_t kMaxLd = (int64_t(1) << 39) - 1;   // TMA strides are below 2^40 bytes
constexpr uint64_t kDefaultTimeoutNs = 4000000000ull;

thread_local std::string t_error;
thread_local std::string t_plan;  // a plan without a launch ("empty (no launch)")

// The last launch's plan, kept as values and formatted only when gb_last_plan asks
// (formatting it on every call cost host time on latency-bound launches).
struct PlanRec {
    bool valid = false;
    const char* kernel = "";
    int pair = 0, mc = 0, epi = 0, pingpong = 0, tile_m = 0, bn = 0, stages = 0, d_boxes = 0, r_boxes = 0;
    long long grid = 0;
    int tiles = 0, k_blocks = 0, splits = 0, group = 0, zigzag = 0, prod = 0;
    unsigned hint_a = 0, hint_b = 0, hint_r = 0, hint_d = 0;
    const char* d_store = "";
    const char* r_load = "";
    const char* z_store = "";
};
thread_local PlanRec t_plan_rec;

gb_status_t fail(gb_status_t s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_error = buf;
    return s;
}

gb_status_t cuda_fail(cudaError_t e, const char* what) {
    return fail(GB_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

// ---------------------------------------------------------------- configuration override

struct Config {
    int bn = 0;          // 0 = heuristic
    int grid = 0;        // 0 = one CTA per SM
    int persistent = 1;  // 0 = one tile per CTA
    int group = 0;       // 0 = heuristic
    int zigzag = -1;     // -1 = heuristic
    int pair = -1;       // -1 = heuristic, 0 = single CTAs, 1 = CTA pairs
    int stages = 0;      // 0 = the deepest ring that fits
    int epi = 0;         // epilogue warpgroups: 0 = heuristic, 1 or 2
    int boxes = 0;       // staging boxes per epilogue warp (D, and R by TMA): 0 = heuristic, 2..8
    int pingpong = -1;   // 1: the two epilogue warpgroups alternate tiles (implies epi=2; no effect with
                         // split-K); 0: they share every tile; -1 = auto (alternate on short-K work items)
    // L2 eviction hints for the TMA traffic of A, B, R and D (and Z): -1 = default,
    // 0 = none, 1 = evict first, 2 = evict last
    int hint_a = -1, hint_b = -1, hint_r = -1, hint_d = -1;
    int mc = -1;         // A multicast between two CTA pairs (4-CTA clusters): -1 auto, 0 off, 1 on
    int issue = -1;      // MMA issue loop: -1 auto, 0 rebuild, 1 lean, 2 lean with look-ahead wait
    int prod = 0;        // producer threads: 0 auto, 1 or 2 (A and B loads issued by different warps)
    int r_async = -1;    // unaligned R rows (no split): -1 auto, 0 synchronous loads at use, 1 cp.async queue
    int r_boxes = 0;     // R queue depth per epilogue warp: 0 = heuristic, 2..8
    int wide = -1;       // 32x64 boxes on the paired epilogue path: -1 auto, 0 off, 1 R and D, 2 D only
};

std::mutex g_cfg_mu;
Config g_cfg;
uint64_t g_timeout_ns = kDefaultTimeoutNs;
int g_inject = 0;
// Trace buffer (libraries built with GB_TRACE): device memory of the caller.
unsigned long long* g_trace = nullptr;
size_t g_trace_bytes = 0;

Config current_config(uint64_t* timeout, int* inject) {
    std::lock_guard<std::mutex> lk(g_cfg_mu);
    *timeout = g_timeout_ns;
    *inject = g_inject;
    return g_cfg;
}

// ---------------------------------------------------------------- device properties

struct DeviceInfo {
    bool ready = false;
    int sms = 0;
    int major = 0, minor = 0;
    size_t smem_optin = 0;
};
std::mutex g_dev_mu;
DeviceInfo g_dev[64];

gb_status_t device_info(int* dev_out, DeviceInfo* info) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(GB_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.ready) {
        int v = 0;
        if ((e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
        if ((e = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute(major)");
        if ((e = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute(minor)");
        if ((e = cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute(smem)");
        d.smem_optin = static_cast<size_t>(v);
        d.ready = true;
    }
    if (d.major != 10 || d.minor != 3)
        return fail(GB_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a only", dev, d.major,
                    d.minor);
    *dev_out = dev;
    *info = d;
    return GB_OK;
}

// ---------------------------------------------------------------- TMA descriptors

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

struct TmapKey {
    const void* base;
    uint64_t inner, outer, stride_bytes;
    uint32_t box_inner, box_outer;
    int swizzle;
    bool operator==(const TmapKey& o) const {
        return base == o.base && inner == o.inner && outer == o.outer && stride_bytes == o.stride_bytes &&
               box_inner == o.box_inner && box_outer == o.box_outer && swizzle == o.swizzle;
    }
};

std::mutex g_tmap_mu;
std::list<std::pair<TmapKey, CUtensorMap>> g_tmap_cache;  // most recent first
constexpr size_t kTmapCacheSize = 128;

// A 2-D bf16 tensor map: `outer` rows of `inner` elements, rows `stride_bytes` apart.
gb_status_t make_tmap(CUtensorMap* out, const void* base, uint64_t inner, uint64_t outer, uint64_t stride_bytes,
                      uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle) {
    const TmapKey key{base, inner, outer, stride_bytes, box_inner, box_outer, static_cast<int>(swizzle)};
    {
        std::lock_guard<std::mutex> lk(g_tmap_mu);
        for (auto it = g_tmap_cache.begin(); it != g_tmap_cache.end(); ++it) {
            if (it->first == key) {
                *out = it->second;
                if (it != g_tmap_cache.begin()) g_tmap_cache.splice(g_tmap_cache.begin(), g_tmap_cache, it);
                return GB_OK;
            }
        }
    }
    auto fn = encode_fn();
    if (!fn) return fail(GB_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {stride_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    CUtensorMap m;
    CUresult r = fn(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(GB_ERR_CUDA,
                    "cuTensorMapEncodeTiled failed (%d) for base=%p dims=(%" PRIu64 ",%" PRIu64 ") stride=%" PRIu64
                    " box=(%u,%u)",
                    static_cast<int>(r), base, inner, outer, stride_bytes, box_inner, box_outer);
    std::lock_guard<std::mutex> lk(g_tmap_mu);
    g_tmap_cache.emplace_front(key, m);
    if (g_tmap_cache.size() > kTmapCacheSize) g_tmap_cache.pop_back();
    *out = m;
    return GB_OK;
}

// ---------------------------------------------------------------- kernels and launch

// One kernel variant: its launch attributes are set once per device, and for CTA
// pairs the number of co-resident clusters is queried once per device.
template <int BN, int NUM_B, int STAGES, bool PAIR, int EPI>
struct Variant {
    using S = gb::KernelShape<BN, NUM_B, STAGES, PAIR, EPI>;
    static constexpr int kEpi = EPI;
    static constexpr int kBN = BN;
    static constexpr int kStages = STAGES;
    static constexpr bool kPair = PAIR;
    static constexpr int kTileM = S::kTileM;

    static gb_status_t prepare(int dev, const DeviceInfo& info, int* max_units, int* max_units_mc) {
        static std::mutex mu;
        static bool ready[64] = {};
        static int units[64] = {};
        static int units_mc[64] = {};
        auto kern = gb::gemm_persistent_kernel<BN, NUM_B, STAGES, PAIR, EPI>;
        const uint32_t smem_max = S::smem_bytes(STAGES, 2, 0);
        const uint32_t smem_min = S::smem_bytes(2, 2, NUM_B == 1 ? 2 : 0);
        if (smem_min > info.smem_optin)
            return fail(GB_ERR_UNSUPPORTED, "kernel needs %u bytes of shared memory, device allows %zu", smem_min,
                        info.smem_optin);
        std::lock_guard<std::mutex> lk(mu);
        if (!ready[dev]) {
            const int attr_bytes = static_cast<int>(info.smem_optin);
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, attr_bytes);
            if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
            if (PAIR) {
                cudaLaunchConfig_t cfg = {};
                cudaLaunchAttribute attr[1];
                attr[0].id = cudaLaunchAttributeClusterDimension;
                attr[0].val.clusterDim.x = 2;
                attr[0].val.clusterDim.y = 1;
                attr[0].val.clusterDim.z = 1;
                cfg.gridDim = dim3(2 * (info.sms / 2), 1, 1);
                cfg.blockDim = dim3(S::kThreads, 1, 1);
                cfg.dynamicSmemBytes = smem_max;
                cfg.attrs = attr;
                cfg.numAttrs = 1;
                int n = 0;
                e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
                if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveClusters");
                if (n < 1) return fail(GB_ERR_UNSUPPORTED, "no CTA pair fits on this device");
                units[dev] = n;
                // clusters of two CTA pairs (A multicast); 0 if none fits
                attr[0].val.clusterDim.x = 4;
                cfg.gridDim = dim3(4 * (info.sms / 4), 1, 1);
                int n4 = 0;
                e = cudaOccupancyMaxActiveClusters(&n4, kern, &cfg);
                units_mc[dev] = e == cudaSuccess ? n4 : 0;
                (void)cudaGetLastError();
            } else {
                units[dev] = info.sms;
                units_mc[dev] = 0;
            }
            ready[dev] = true;
        }
        *max_units = units[dev];
        if (max_units_mc) *max_units_mc = units_mc[dev];
        return GB_OK;
    }

    // Shared memory of one launch: the operand ring and the epilogue warps' box
    // queues.  Long-K work items want the deepest ring (the MMAs must never wait
    // for operands) and two boxes per warp; work items of at most 4 k-blocks are
    // bound by the epilogue's global traffic, so they take a 3-stage ring and spend
    // the rest on deeper D/R queues (more bytes in flight per SM).  `r_mode`: 0 no
    // R boxes, 1 one box as the transpose buffer of unaligned R rows, 2 a queue
    // of R boxes loaded by TMA, 3 a queue of cp.async slots for unaligned R rows
    // (3 deep by default: a long-K tile's next chunks all land during its MMAs).
    // Unaligned D rows without a TMA-stored second output need one D box (the
    // transpose buffer), so such launches keep room for a deeper ring.
    // Boxes shrink first, then the ring, down to 2 each.
    struct Layout {
        int stages, d_boxes, r_boxes;
    };
    // Bytes of one R / D queue entry for a launch's flags.
    static uint32_t r_slot_bytes(uint32_t flags) {
        return (flags & gb::kFlagRAsync) ? gb::kRSlotAsyncBytes : (flags & gb::kFlagWide) ? gb::kWideBoxBytes
                                                                                          : gb::kDStageBytes;
    }
    static uint32_t d_slot_bytes(uint32_t flags) {
        return (flags & (gb::kFlagWide | gb::kFlagWideD)) ? gb::kWideBoxBytes : gb::kDStageBytes;
    }
    static Layout choose_layout(int kb_per_item, int r_mode, uint32_t flags, const Config& cfg, size_t smem_optin) {
        const bool short_k = kb_per_item <= 4;
        int st = cfg.stages > 0 ? std::min(cfg.stages, STAGES) : (short_k ? std::min(3, STAGES) : STAGES);
        st = std::max(2, st);
        int boxes = cfg.boxes > 0 ? cfg.boxes : (short_k ? gb::kMaxBoxes : 2);
        int rq = cfg.r_boxes > 0 ? cfg.r_boxes : (short_k ? gb::kMaxBoxes : 3);
        auto r_of = [&](int b) { return r_mode == 2 ? (cfg.r_boxes > 0 ? rq : b) : r_mode == 3 ? rq : (r_mode == 1 ? 1 : 0); };
        // D rows not 16-byte aligned and no TMA-stored second output: the D queue is only
        // the transpose buffer, one box
        const bool d_transpose_only = !(flags & gb::kFlagDTma) && !((flags & gb::kFlagZ) && (flags & gb::kFlagZTma));
        auto d_of = [&](int b) { return d_transpose_only && cfg.boxes <= 0 ? 1 : b; };
        const uint32_t rs = r_slot_bytes(flags), ds = d_slot_bytes(flags);
        if (kEpi == 4) {
            // Sixteen epilogue warps: per-warp queues must be short to fit.  32x64 D and R
            // boxes: one of each per warp (the other warps of the SM hide each one's waits);
            // 32x64 D and 32x32 R boxes: one D and three R; 32x32 boxes: two D and three R.
            // A 2-stage ring unless asked.
            const bool wide_d = flags & (gb::kFlagWide | gb::kFlagWideD), wide_r = flags & gb::kFlagWide;
            const int lst = cfg.stages > 0 ? std::min(cfg.stages, STAGES) : 2;
            int ld = cfg.boxes > 0 ? cfg.boxes : (wide_d ? 1 : 2);
            int lr = cfg.r_boxes > 0 ? cfg.r_boxes : (wide_r ? 1 : 3);
            const int dmin = wide_d ? 1 : 2, rmin = wide_r ? 1 : 2;
            while (lr > rmin && S::smem_bytes(lst, ld, lr, rs, ds) > smem_optin) --lr;
            while (ld > dmin && S::smem_bytes(lst, ld, lr, rs, ds) > smem_optin) --ld;
            int ls = lst;
            while (ls > 1 && S::smem_bytes(ls, ld, lr, rs, ds) > smem_optin) --ls;
            return Layout{ls, ld, lr};
        }
        if (short_k && (flags & gb::kFlagWide) && cfg.stages <= 0 && cfg.boxes <= 0 && cfg.r_boxes <= 0) {
            // Wide boxes on items of 1-4 k-blocks: a 2-stage ring is enough (the MMAs are a
            // few percent of the time) and the room goes to R boxes in flight, whose loads
            // gate every step (measured on GB300, K = 64 residual: 2 stages + 2 D + 3 R
            // boxes 3 % faster than 3 stages + 2 + 2).
            int r = gb::kMaxBoxes;
            while (r > 2 && S::smem_bytes(2, 2, r, rs, ds) > smem_optin) --r;
            return Layout{2, 2, r};
        }
        // (a cp.async queue gives up depth, down to 2, before the ring gives up a stage)
        while (r_mode == 3 && rq > 2 && S::smem_bytes(st, d_of(boxes), rq, rs, ds) > smem_optin) --rq;
        while (boxes > 2 && S::smem_bytes(st, d_of(boxes), r_of(boxes), rs, ds) > smem_optin) --boxes;
        while (st > 2 && S::smem_bytes(st, d_of(boxes), r_of(boxes), rs, ds) > smem_optin) --st;
        while (rq > 2 && S::smem_bytes(st, d_of(boxes), r_of(boxes), rs, ds) > smem_optin) --rq;
        return Layout{st, d_of(boxes), r_of(boxes)};
    }

    static gb_status_t launch(const GemmParams& p, int units, cudaStream_t stream) {
        auto kern = gb::gemm_persistent_kernel<BN, NUM_B, STAGES, PAIR, EPI>;
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        cfg.gridDim = dim3(units * S::kCG * (p.mc ? 2 : 1), 1, 1);
        cfg.blockDim = dim3(S::kThreads, 1, 1);
        cfg.dynamicSmemBytes = S::smem_bytes(p.stages, p.d_boxes, p.r_boxes, r_slot_bytes(p.flags));
        cfg.stream = stream;
        if (PAIR) {
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = p.mc ? 4 : 2;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
        }
        cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p);
        if (e != cudaSuccess) return cuda_fail(e, "cudaLaunchKernelEx");
        e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
        return GB_OK;
    }
};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned2(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 1u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

struct Problem {
    const void* a;
    int64_t lda;
    const void* b0;
    int64_t ldb0;
    const void* b1;
    int64_t ldb1;
    const void* bias;
    const void* r;
    int64_t ldr;
    int act;
    void* d;
    int64_t ldd;
    int64_t m, n, k;
    bool ffn;
    void* z = nullptr;  // optional second output (linear): the pre-activation
    int64_t ldz = 0;
    // B is a row-major [k, n] matrix (MN-major operand): the matmul form, and the
    // activation gradient
    bool b_mn = false;
    // activation gradient: the epilogue input r (the stored pre-activation) multiplies
    // by act'(r)
    bool dact = false;
};

gb_status_t validate(const Problem& pr) {
    const char* an = pr.ffn ? "X" : pr.dact ? "dY" : "A";
    const char* bn = pr.ffn ? "W1" : pr.dact ? "W" : "B";
    if (pr.m < 0 || pr.n < 0 || pr.k < 0)
        return fail(GB_ERR_INVALID_ARG, "negative size M=%" PRId64 " N=%" PRId64 " K=%" PRId64, pr.m, pr.n, pr.k);
    if (pr.act < GB_ACT_NONE || pr.act > GB_ACT_RELU) return fail(GB_ERR_INVALID_ARG, "unknown activation %d", pr.act);
    if (pr.m > kMaxDim || pr.n > kMaxDim || pr.k > kMaxDim)
        return fail(GB_ERR_UNSUPPORTED, "sizes must be below 2^31 (M=%" PRId64 " N=%" PRId64 " K=%" PRId64 ")", pr.m,
                    pr.n, pr.k);
    if (pr.m == 0 || pr.n == 0) return GB_OK;
    if (!pr.d) return fail(GB_ERR_INVALID_ARG, "D is null");
    // dims named as the caller sees them: for the activation gradient the output is
    // [M, K] and the contraction runs over N
    const char* nn = pr.dact ? "K" : "N";
    const char* kn = pr.dact ? "N" : "K";
    if (pr.dact && !pr.r) return fail(GB_ERR_INVALID_ARG, "Z is null");
    if (pr.ldd < pr.n) return fail(GB_ERR_INVALID_ARG, "ldd=%" PRId64 " < %s=%" PRId64, pr.ldd, nn, pr.n);
    if (pr.r && pr.ldr < pr.n)
        return fail(GB_ERR_INVALID_ARG, "ld%s=%" PRId64 " < %s=%" PRId64, pr.dact ? "z" : "r", pr.ldr, nn, pr.n);
    if (pr.k > 0) {
        if (!pr.a) return fail(GB_ERR_INVALID_ARG, "%s is null", an);
        if (!pr.b0) return fail(GB_ERR_INVALID_ARG, "%s is null", bn);
        if (pr.ffn && !pr.b1) return fail(GB_ERR_INVALID_ARG, "W3 is null");
        if (pr.lda < pr.k)
            return fail(GB_ERR_INVALID_ARG, "ld%s=%" PRId64 " < %s=%" PRId64, pr.ffn ? "x" : pr.dact ? "dy" : "a",
                        pr.lda, kn, pr.k);
        if (pr.b_mn && pr.ldb0 < pr.n)
            return fail(GB_ERR_INVALID_ARG, "ld%s=%" PRId64 " < %s=%" PRId64, pr.dact ? "w" : "b", pr.ldb0, nn, pr.n);
        if (!pr.b_mn && pr.ldb0 < pr.k)
            return fail(GB_ERR_INVALID_ARG, "ld%s=%" PRId64 " < K=%" PRId64, pr.ffn ? "w1" : "b", pr.ldb0, pr.k);
        if (pr.ffn && pr.ldb1 < pr.k) return fail(GB_ERR_INVALID_ARG, "ldw3=%" PRId64 " < K=%" PRId64, pr.ldb1, pr.k);
        if (!aligned16(pr.a) || !aligned16(pr.b0) || (pr.ffn && !aligned16(pr.b1)))
            return fail(GB_ERR_UNSUPPORTED, "operand base addresses must be 16-byte aligned for TMA");
        if (pr.lda % 8 || pr.ldb0 % 8 || (pr.ffn && pr.ldb1 % 8))
            return fail(GB_ERR_UNSUPPORTED, "operand leading dimensions must be multiples of 8 elements for TMA");
        if (pr.lda > kMaxLd || pr.ldb0 > kMaxLd || (pr.ffn && pr.ldb1 > kMaxLd))
            return fail(GB_ERR_UNSUPPORTED, "operand leading dimension too large for TMA");
    }
    if (pr.z && pr.ldz < pr.n) return fail(GB_ERR_INVALID_ARG, "ldz=%" PRId64 " < N=%" PRId64, pr.ldz, pr.n);
    if (!aligned2(pr.d) || (pr.r && !aligned2(pr.r)) || (pr.bias && !aligned2(pr.bias)) || (pr.z && !aligned2(pr.z)))
        return fail(GB_ERR_UNSUPPORTED, "D, R, Z and bias must be 2-byte aligned");
    if (pr.z && pr.ldz > kMaxLd) return fail(GB_ERR_UNSUPPORTED, "leading dimension too large");
    if (pr.ldd > kMaxLd || (pr.r && pr.ldr > kMaxLd)) return fail(GB_ERR_UNSUPPORTED, "leading dimension too large");
    return GB_OK;
}

struct SplitReq {
    bool allowed = false;    // the caller supplied a workspace (or asked for its size)
    int splits = 1;          // <= 0: choose automatically
    void* ws = nullptr;
    size_t ws_bytes = 0;
    bool query_only = false;  // compute the workspace size, launch nothing
    size_t* ws_needed = nullptr;
};

constexpr size_t kWsAlign = 256;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

template <class V>
gb_status_t plan_and_launch(const Problem& pr, const Config& cfg, int bn, int dev, const DeviceInfo& info,
                            uint64_t timeout_ns, int inject, cudaStream_t stream, const SplitReq& sr) {
    gb_status_t st;
    int max_units = 0, max_units_mc = 0;
    if ((st = V::prepare(dev, info, &max_units, &max_units_mc)) != GB_OK) return st;

    GemmParams prm;
    memset(&prm, 0, sizeof prm);
    prm.m = static_cast<int32_t>(pr.m);
    prm.n = static_cast<int32_t>(pr.n);
    prm.k = static_cast<int32_t>(pr.k);
    prm.num_m_blocks = static_cast<int32_t>(cdiv(pr.m, V::kTileM));
    prm.num_n_blocks = static_cast<int32_t>(cdiv(pr.n, bn));
    prm.num_k_blocks = static_cast<int32_t>(cdiv(pr.k, gb::kBK));
    // A multicast between two CTA pairs: on request, for CTA-pair variants without a
    // split, when 4-CTA clusters fit; a work item is then one tile-row x two tile-columns.
    const bool mc = V::kPair && V::kEpi != 4 && cfg.mc == 1 && max_units_mc > 0 && !(sr.allowed) && pr.k > 0;
    prm.mc = mc ? 1 : 0;
    prm.sched_n_blocks = mc ? static_cast<int32_t>(cdiv(prm.num_n_blocks, 2)) : prm.num_n_blocks;
    const int64_t tiles = static_cast<int64_t>(prm.num_m_blocks) * prm.sched_n_blocks;
    if (tiles > kMaxDim) return fail(GB_ERR_UNSUPPORTED, "too many tiles");
    prm.num_tiles = static_cast<int32_t>(tiles);

    // Split-K: only with a workspace.  Auto: when the tiles would leave more than
    // half of the scheduling units idle (and, unless K has at least 256 k-blocks,
    // more than three quarters), cut K so that tiles x splits fills them, keeping at
    // least 4 k-blocks per split and at most 64 splits.
    int splits = 1;
    if (sr.allowed && prm.num_k_blocks > 1) {
        if (sr.splits > 0) {
            splits = sr.splits;
        } else if (prm.num_k_blocks >= 8 && 2 * tiles <= max_units &&
                   (4 * tiles <= max_units || prm.num_k_blocks >= 256)) {
            // The fp32 partial sums cost about as much as a short K range saves: measured on
            // GB300, a tile set that already fills a quarter of the units runs faster unsplit
            // at K = 4096 (8191x96: 32.8 against 36.9 us) but split at K = 65536 (204 against
            // 323 us); beyond 64 splits the reductions outweigh the shorter K ranges.
            splits = static_cast<int>(std::min<int64_t>({max_units / tiles, prm.num_k_blocks / 4, 64}));
        }
        splits = std::max(1, std::min(splits, prm.num_k_blocks));
    }
    prm.kb_per_split = static_cast<int32_t>(cdiv(prm.num_k_blocks, splits));
    if (prm.kb_per_split > 0) splits = static_cast<int>(cdiv(prm.num_k_blocks, prm.kb_per_split));
    prm.splits = splits;
    // The lean variant (four epilogue warpgroups) has only the paired epilogue path: a
    // split plan runs on the two-warpgroup kernel instead.
    if constexpr (V::kEpi == 4) {
        if (splits != 1)
            return plan_and_launch<Variant<V::kBN, 1, 6, true, 2>>(pr, cfg, bn, dev, info, timeout_ns, inject, stream,
                                                                   sr);
    }
    const int64_t work = tiles * splits;
    if (work > kMaxDim) return fail(GB_ERR_UNSUPPORTED, "too many work items");

    const int num_b = pr.ffn ? 2 : 1;
    const size_t cnt_bytes = splits > 1 ? align_up(static_cast<size_t>(tiles) * V::S::kSlabs * 4, kWsAlign) : 0;
    // one fp32 accumulator tile per output tile (per product for the FFN)
    const size_t part_bytes =
        splits > 1 ? static_cast<size_t>(tiles) * num_b * V::kTileM * static_cast<size_t>(bn) * sizeof(float) : 0;
    const size_t ws_needed = cnt_bytes + part_bytes;
    if (sr.query_only) {
        *sr.ws_needed = ws_needed;
        return GB_OK;
    }
    if (ws_needed > 0) {
        if (!sr.ws) return fail(GB_ERR_INVALID_ARG, "split-K needs a workspace of %zu bytes", ws_needed);
        if (sr.ws_bytes < ws_needed)
            return fail(GB_ERR_INVALID_ARG, "workspace of %zu bytes is smaller than the %zu bytes needed", sr.ws_bytes,
                        ws_needed);
        if (reinterpret_cast<uintptr_t>(sr.ws) % kWsAlign)
            return fail(GB_ERR_INVALID_ARG, "workspace must be %zu-byte aligned", kWsAlign);
        prm.ws_cnt = static_cast<uint32_t*>(sr.ws);
        prm.ws = reinterpret_cast<float*>(static_cast<uint8_t*>(sr.ws) + cnt_bytes);
    }

    // 16 tile-rows per group (4096 rows of A for CTA pairs): measured on GB300 under the
    // power cap, 1.6-1.7 % faster than 8 or 24 on the 8192x14336x4096 MLP and FFN shapes
    // (fewer DRAM re-reads of B, so more power for the SMs).
    int group = cfg.group ? cfg.group : 16;
    if (group > prm.num_m_blocks) group = prm.num_m_blocks;
    prm.group_m = group < 1 ? 1 : group;
    prm.zigzag = cfg.zigzag >= 0 ? cfg.zigzag : (prm.kb_per_split >= 256 ? 1 : 0);
    prm.act = pr.ffn ? GB_ACT_NONE : pr.act;
    prm.bias = static_cast<const uint16_t*>(pr.bias);
    prm.r = static_cast<const uint16_t*>(pr.r);
    prm.d = static_cast<uint16_t*>(pr.d);
    prm.ldr = pr.ldr;
    prm.ldd = pr.ldd;
    prm.timeout_ns = timeout_ns;
    prm.inject = inject;
    // L2 policies: for long-K work items, A (re-read by every tile-column of its tile-row
    // group) is kept (evict last) and D, written once, goes first (evict first): measured on
    // the MLP shape, DRAM reads 376 -> 349 MB per launch and 1-3 % faster.  Short-K work
    // (bound by the epilogue's streams) measured no better with hints, so it takes none.
    auto hint = [](int cfg_value, int dflt) { return static_cast<uint32_t>(cfg_value >= 0 ? cfg_value : dflt); };
    const bool long_k = prm.kb_per_split >= 16;
    prm.hint_a = hint(cfg.hint_a, long_k ? 2 : 0);
    prm.hint_b = hint(cfg.hint_b, 0);
    prm.hint_r = hint(cfg.hint_r, 0);
    prm.hint_d = hint(cfg.hint_d, long_k ? 1 : 0);
    prm.issue = cfg.issue >= 0 ? cfg.issue : 0;
    // two producer threads by default: measured 7-12 % faster than one on the MLP, FFN,
    // activation-gradient, 64-bit and unaligned shapes (one thread issuing both loads of
    // every stage falls behind the MMAs)
    prm.prod = cfg.prod > 0 ? cfg.prod : 2;
    uint32_t flags = 0;
    if (!pr.ffn && pr.bias) flags |= gb::kFlagBias | (aligned16(pr.bias) ? gb::kFlagBiasVec : 0u);
    if (!pr.ffn && pr.r) flags |= gb::kFlagResidual | ((aligned16(pr.r) && pr.ldr % 8 == 0) ? gb::kFlagRVec : 0u);
    if (pr.b_mn) flags |= gb::kFlagBMn;
    if (pr.dact) flags |= gb::kFlagDact;
    const bool d_tma = aligned16(pr.d) && pr.ldd % 8 == 0;
    if (d_tma) flags |= gb::kFlagDTma;
    const bool r_tma = !pr.ffn && pr.r && aligned16(pr.r) && pr.ldr % 8 == 0 && splits == 1;
    if (r_tma) flags |= gb::kFlagRTma;
    // Unaligned R rows: cp.async word copies need a 4-byte aligned base (a segment's
    // first word may then start one element early, still inside the tensor).  Off by
    // default: measured on GB300 (N = 4099 residual shapes) the prefetch queue hides the
    // R loads, but the shared memory it takes costs one operand stage, and the launches
    // came out 0.5-2.5 % slower than synchronous loads at use.
    const bool r_async = !pr.ffn && pr.r && !(flags & gb::kFlagRVec) && splits == 1 && aligned4(pr.r) &&
                         cfg.r_async == 1;
    if (r_async) flags |= gb::kFlagRAsync;
    // Wide 32x64 boxes on the paired path (R and D by TMA, no Z, no split): one TMA load,
    // one TMA store, one R wait and one fence per 64 columns instead of per 32.  Measured
    // on GB300: +11 % on the K = 64 residual shape, +3 % on the activation-gradient shape;
    // on by default.  A wide step spans two chunks, so every warpgroup's share of a tile
    // must be whole steps.
    const bool paired = r_tma && pr.k > 0 && d_tma && !pr.z;
    const int groups = V::kEpi;
    const bool wide_fits = (V::kBN / gb::kDChunk) % (2 * groups) == 0;
    // The four-warpgroup kernel defaults to 32x64 D boxes with 32x32 R boxes (`wide=2`):
    // sixteen warps' queues of 32x64 R boxes leave room for one R box each (measured 7 %
    // slower than three 32x32 R boxes).
    const int wide_mode = cfg.wide >= 0 ? cfg.wide : (V::kEpi == 4 ? 2 : 1);
    if (paired && wide_fits && wide_mode == 1) flags |= gb::kFlagWide;
    if (paired && wide_fits && wide_mode == 2) flags |= gb::kFlagWideD;
    // The express path (no epilogue input, no second output, TMA-stored D, no split) of the
    // one-warpgroup kernel stages two adjacent chunks into one 32x64 D box per step as well.
    const bool express = splits == 1 && pr.k > 0 && d_tma && !pr.r && !pr.z;
    if (express && V::kEpi == 1 && wide_fits && wide_mode >= 1) flags |= gb::kFlagWideD;
    const bool z_tma = pr.z && aligned16(pr.z) && pr.ldz % 8 == 0;
    if (!pr.ffn && pr.z) flags |= gb::kFlagZ | (z_tma ? gb::kFlagZTma : 0u);
    prm.z = static_cast<uint16_t*>(pr.z);
    prm.ldz = pr.ldz;
    prm.flags = flags;
    {
        const int r_mode = r_tma ? 2 : r_async ? 3 : (!pr.ffn && pr.r && !(flags & gb::kFlagRVec)) ? 1 : 0;
        const auto lay = V::choose_layout(prm.kb_per_split, r_mode, flags, cfg, info.smem_optin);
        prm.stages = lay.stages;
        prm.d_boxes = lay.d_boxes;
        prm.r_boxes = lay.r_boxes;
        if (flags & (gb::kFlagWide | gb::kFlagWideD)) prm.d_boxes *= 2;  // counted in 32x32 boxes
        prm.r_warp_bytes = static_cast<uint32_t>(lay.r_boxes) * V::r_slot_bytes(flags);
        const uint32_t smem = V::S::smem_bytes(prm.stages, prm.d_boxes, prm.r_boxes, V::r_slot_bytes(flags));
        if (smem > info.smem_optin)
            return fail(GB_ERR_UNSUPPORTED, "shared memory layout (%d stages, %d/%d boxes) needs %u bytes, device allows %zu",
                        prm.stages, lay.d_boxes, lay.r_boxes, smem, info.smem_optin);
    }

    const uint32_t b_rows = static_cast<uint32_t>(V::S::kBBox);
    if (pr.k > 0) {
        if ((st = make_tmap(&prm.tm_a, pr.a, pr.k, pr.m, pr.lda * 2, gb::kBK, gb::kBM, CU_TENSOR_MAP_SWIZZLE_128B)) !=
            GB_OK)
            return st;
        if ((mc || prm.prod == 3) && (st = make_tmap(&prm.tm_a_half, pr.a, pr.k, pr.m, pr.lda * 2, gb::kBK, gb::kBM / 2,
                                                    CU_TENSOR_MAP_SWIZZLE_128B)) != GB_OK)
            return st;
        if (pr.b_mn) {
            // B [k rows (contraction), n columns]: boxes of 64 columns x 64 rows
            if ((st = make_tmap(&prm.tm_b0, pr.b0, pr.n, pr.k, pr.ldb0 * 2, 64, gb::kBK,
                                CU_TENSOR_MAP_SWIZZLE_128B)) != GB_OK)
                return st;
        } else if ((st = make_tmap(&prm.tm_b0, pr.b0, pr.k, pr.n, pr.ldb0 * 2, gb::kBK, b_rows,
                                   CU_TENSOR_MAP_SWIZZLE_128B)) != GB_OK) {
            return st;
        }
        if (pr.ffn && (st = make_tmap(&prm.tm_b1, pr.b1, pr.k, pr.n, pr.ldb1 * 2, gb::kBK, b_rows,
                                      CU_TENSOR_MAP_SWIZZLE_128B)) != GB_OK)
            return st;
    }
    const bool wide = flags & gb::kFlagWide, wide_d = flags & (gb::kFlagWide | gb::kFlagWideD);
    auto box_n = [](bool w) { return w ? 2 * gb::kDChunk : gb::kDChunk; };
    auto box_sw = [](bool w) { return w ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B; };
    if (d_tma && (st = make_tmap(&prm.tm_d, pr.d, pr.n, pr.m, pr.ldd * 2, box_n(wide_d), 32, box_sw(wide_d))) != GB_OK)
        return st;
    if (r_tma && (st = make_tmap(&prm.tm_r, pr.r, pr.n, pr.m, pr.ldr * 2, box_n(wide), 32, box_sw(wide))) != GB_OK)
        return st;
    if (z_tma &&
        (st = make_tmap(&prm.tm_z, pr.z, pr.n, pr.m, pr.ldz * 2, gb::kDChunk, 32, CU_TENSOR_MAP_SWIZZLE_64B)) != GB_OK)
        return st;

    // Scheduling units: CTAs, or CTA pairs.  Persistent: at most one per SM (pair
    // of SMs); one work item per unit otherwise.
    int64_t units = cfg.persistent ? (mc ? max_units_mc : max_units) : work;
    if (cfg.grid > 0) {
        const int64_t per_unit = V::kPair ? (mc ? 4 : 2) : 1;
        const int64_t cap = (cfg.grid + per_unit - 1) / per_unit;
        if (cap < units) units = cap;
    }
    if (units > work) units = work;
    if (units < 1) units = 1;

    // Ping-pong (two epilogue warpgroups alternating tiles): on by default for work
    // items of at most 4 k-blocks, where the epilogue is the whole cost (measured on
    // GB300: +9-13 % on the K = 64 residual shapes), if every unit gets at least 4 of
    // them (with fewer, one warpgroup would idle); off for long K, where sharing
    // every tile's chunks is 2.5-7.5 % faster.
    const bool pp_auto = prm.kb_per_split <= 4 && work >= 4 * units;
    prm.pingpong = (V::kEpi == 4 || (V::kEpi == 2 && splits == 1 && (cfg.pingpong == 1 || (cfg.pingpong < 0 && pp_auto))))
                       ? 1 : 0;

    PlanRec& rec = t_plan_rec;
    rec.valid = true;
    rec.kernel = pr.ffn ? "ffn_gated" : pr.dact ? "linear_dact" : pr.b_mn ? "matmul" : "linear";
    rec.pair = V::kPair ? 1 : 0;
    rec.mc = prm.mc;
    rec.epi = V::kEpi;
    rec.pingpong = prm.pingpong;
    rec.tile_m = V::kTileM;
    rec.bn = bn;
    rec.stages = prm.stages;
    rec.d_boxes = wide_d ? prm.d_boxes / 2 : prm.d_boxes;
    rec.r_boxes = prm.r_boxes;
    rec.grid = static_cast<long long>(units * (V::kPair ? (mc ? 4 : 2) : 1));
    rec.tiles = prm.num_tiles;
    rec.k_blocks = prm.num_k_blocks;
    rec.splits = splits;
    rec.group = prm.group_m;
    rec.zigzag = prm.zigzag;
    rec.prod = prm.prod;
    rec.hint_a = prm.hint_a;
    rec.hint_b = prm.hint_b;
    rec.hint_r = prm.hint_r;
    rec.hint_d = prm.hint_d;
    rec.d_store = d_tma ? (wide_d ? "tma.64x32" : "tma") : "st.transposed";
    rec.r_load = pr.r ? (r_tma ? (wide ? "tma.64x32" : "tma") : r_async ? "cp.async" : (flags & gb::kFlagRVec) ? "ld.v4"
                                                                                                      : "ld.transposed")
                      : "none";
    rec.z_store = pr.z ? (z_tma ? "tma" : "st.transposed") : "none";
    {
        std::lock_guard<std::mutex> lk(g_cfg_mu);
        const size_t need = static_cast<size_t>(units) * (V::kPair ? (mc ? 4 : 2) : 1) * gb::kTraceWords * 8;
        prm.trace = (g_trace && g_trace_bytes >= need) ? g_trace : nullptr;
    }
    if (ws_needed) {  // counters and accumulators start at zero
        cudaError_t e = cudaMemsetAsync(prm.ws_cnt, 0, ws_needed, stream);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(split-K workspace)");
    }
    return V::launch(prm, static_cast<int>(units), stream);
}

template <int EPI>
gb_status_t dispatch(const Problem& pr, const Config& cfg, int bn, bool pair, int dev, const DeviceInfo& info,
                     uint64_t timeout_ns, int inject, cudaStream_t stream, const SplitReq& sr) {
    using LinPair = Variant<256, 1, 6, true, EPI>;
    using LinSingle = Variant<256, 1, 4, false, EPI>;
    using LinNarrow = Variant<128, 1, 6, false, EPI>;
    using FfnPair = Variant<128, 2, 6, true, EPI>;
    using FfnSingle = Variant<128, 2, 4, false, EPI>;
    if (pr.ffn)
        return pair ? plan_and_launch<FfnPair>(pr, cfg, bn, dev, info, timeout_ns, inject, stream, sr)
                    : plan_and_launch<FfnSingle>(pr, cfg, bn, dev, info, timeout_ns, inject, stream, sr);
    if (bn == 256)
        return pair ? plan_and_launch<LinPair>(pr, cfg, bn, dev, info, timeout_ns, inject, stream, sr)
                    : plan_and_launch<LinSingle>(pr, cfg, bn, dev, info, timeout_ns, inject, stream, sr);
    return plan_and_launch<LinNarrow>(pr, cfg, bn, dev, info, timeout_ns, inject, stream, sr);
}

gb_status_t run(const Problem& pr, void* stream_ptr, const SplitReq& sr = SplitReq()) {
    gb_status_t st = validate(pr);
    if (st != GB_OK) return st;
    if (pr.m == 0 || pr.n == 0) {
        t_plan = "empty (no launch)";
        t_plan_rec.valid = false;
        if (sr.query_only) *sr.ws_needed = 0;
        return GB_OK;
    }
    int dev = 0;
    DeviceInfo info;
    if ((st = device_info(&dev, &info)) != GB_OK) return st;
    uint64_t timeout_ns;
    int inject;
    const Config cfg = current_config(&timeout_ns, &inject);
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);

    // Tile width: the FFN kernel holds two 128-column accumulators per buffer;
    // the linear kernel uses 256 columns unless N fits in 128.  CTA pairs
    // (256-row tiles) unless M fits in one 128-row tile.
    // Tiny outputs (256x256 pair tiles would use at most an eighth of the SMs): 128x128
    // tiles on single CTAs spread the work over more SMs and halve each tile's MMA chain
    // (measured on GB300, 256x384x512: 14.8 -> 12.3 us; the event-timing floor is 6.6 us).
    const int64_t pair_tiles = cdiv(pr.m, 2 * gb::kBM) * cdiv(pr.n, 256);
    const bool tiny = !pr.ffn && cfg.bn == 0 && cfg.pair < 0 && cfg.mc != 1 && cfg.epi != 4 &&
                      8 * 2 * pair_tiles <= info.sms;  // (not when the config asks for a CTA-pair feature)
    const int bn = pr.ffn ? 128 : (cfg.bn ? cfg.bn : (pr.n <= 128 || tiny ? 128 : 256));
    if (pr.ffn && cfg.bn && cfg.bn != 128) return fail(GB_ERR_UNSUPPORTED, "the FFN kernel supports bn=128 only");
    bool pair = cfg.pair >= 0 ? cfg.pair == 1 : pr.m > gb::kBM;
    if (!pr.ffn && bn == 128) pair = false;  // the 128-wide linear tile runs on single CTAs

    // Epilogue warpgroups: two when the epilogue carries more than the tile's MMAs
    // hide, one otherwise.  Measured on GB300 (interleaved A/B): one is 1-3 % faster on
    // long-K shapes, with or without an aligned epilogue input (K >= 4096); two are up
    // to 1.4x faster on short K (<= 16 k-blocks), on split-K plans over few tiles, and
    // with rows that go through the shared-memory transposes (N = 4099: two win by 12 %
    // at K = 4096; at K = 65536 the two were within run-to-run noise).  An epilogue input
    // or a second output needs two below 64 k-blocks; above, one was faster (MLP with its
    // pre-activation stored, 8192x14336x4096: 1538 against 1515 TFLOP/s).
    const int64_t kb = cdiv(pr.k, gb::kBK);
    const bool d_rows_aligned = aligned16(pr.d) && pr.ldd % 8 == 0;
    const bool r_rows_aligned = !pr.r || (aligned16(pr.r) && pr.ldr % 8 == 0);
    const bool z_rows_aligned = !pr.z || (aligned16(pr.z) && pr.ldz % 8 == 0);
    const int64_t tiles_est = cdiv(pr.m, pair ? 2 * gb::kBM : gb::kBM) * cdiv(pr.n, bn);
    const bool few_tiles_split = sr.allowed && 2 * tiles_est <= info.sms;
    const bool heavy_epilogue = kb <= 16 || few_tiles_split || !d_rows_aligned || !r_rows_aligned ||
                                !z_rows_aligned || ((pr.r || pr.z) && kb < 64);
    if (cfg.pingpong == 1 && cfg.epi == 1)
        return fail(GB_ERR_INVALID_ARG, "pingpong=1 needs two epilogue warpgroups (epi=2)");
    // Four epilogue warpgroups (lean kernel: paired path only): linear with an aligned
    // epilogue input, an aligned D, no second output, 256-wide tiles on CTA pairs.
    const bool lean_ok = !pr.ffn && !pr.b_mn && pr.r && !pr.z && r_rows_aligned && d_rows_aligned && kb > 0 &&
                         pair && bn == 256;
    // By default for work items of at most 4 k-blocks (the epilogue is the whole cost) over
    // at least two tiles per CTA pair: measured on GB300, K = 64 residual 8191x12288,
    // 0.121 -> 0.100 ms against two warpgroups.  Longer K wants the deeper operand ring
    // that sixteen warps' queues leave no room for (K = 1024: 0.080 against 0.102 ms).
    const bool lean_auto = lean_ok && kb <= 4 && tiles_est >= info.sms && cfg.pingpong != 0;
    int epi = cfg.pingpong == 1 ? 2 : cfg.epi > 0 ? cfg.epi : lean_auto ? 4 : (heavy_epilogue ? 2 : 1);
    if (epi == 4 && !lean_ok) epi = 2;
    if (epi == 4)
        return plan_and_launch<Variant<256, 1, 4, true, 4>>(pr, cfg, bn, dev, info, timeout_ns, inject, stream, sr);
    return epi == 2 ? dispatch<2>(pr, cfg, bn, pair, dev, info, timeout_ns, inject, stream, sr)
                    : dispatch<1>(pr, cfg, bn, pair, dev, info, timeout_ns, inject, stream, sr);
}

bool parse_int(const char* s, size_t n, long* out) {
    std::string t(s, n);
    char* end = nullptr;
    long v = strtol(t.c_str(), &end, 10);
    if (t.empty() || *end) return false;
    *out = v;
    return true;
}

// ---------------------------------------------------------------- static split-K scratch

// Scratch for gb_gemm_linear_splitk_noalloc: a fixed array in this library's own
// device memory, so that callers who may not allocate device memory can still
// run the split-K schedule.  Every GPU that loads the library holds these bytes
// until the process exits.  All calls share it.
constexpr size_t kStaticScratchBytes = size_t(32) << 20;  // 32 MiB
static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[64] = {};

// The device address of g_static_scratch on the current device `dev`.  In host
// code the array's name is only a host-side stand-in, so the address is looked
// up once per device (with that device current) and cached.
gb_status_t static_scratch_address(int dev, void** out) {
    if (dev < 0 || dev >= 64) return fail(GB_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* ptr = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&ptr, g_static_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static split-K scratch)");
        g_scratch_addr[dev] = ptr;
    }
    *out = g_scratch_addr[dev];
    return GB_OK;
}

// Workspace bytes the existing split-K plan needs for this problem and split count.
gb_status_t splitk_bytes_for(const Problem& pr, int splits, size_t* bytes) {
    SplitReq sr;
    sr.allowed = true;
    sr.splits = splits;
    sr.query_only = true;
    sr.ws_needed = bytes;
    *bytes = 0;
    return run(pr, nullptr, sr);
}

// ---------------------------------------------------------------- tensor-core rate probe

// The probe's TMA-writer modes read g_probe_src as bf16 [8192 rows][64 columns] in
// 128-row boxes (128-byte swizzle); other modes get an unused, zeroed map.
gb_status_t probe_source_map(CUtensorMap* out) {
    void* src = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&src, gb::g_probe_src);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(probe source)");
    return make_tmap(out, src, 64, gb::kProbeSrcBytes / 128, 128, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B);
}

template <int CG, int N, int MODE>
gb_status_t probe_launch(int units, int num_mma, int alternate, int alu, cudaStream_t stream) {
    CUtensorMap tmap;
    memset(&tmap, 0, sizeof tmap);
    if (MODE == gb::kProbeStagesTma || MODE == gb::kProbeStagesTma2 || MODE == gb::kProbeTmaStore ||
        MODE == gb::kProbePipeline) {
        gb_status_t st = probe_source_map(&tmap);
        if (st != GB_OK) return st;
    }
    auto kern = gb::mma_rate_kernel<CG, N, MODE>;
    const int smem = 200 * 1024;  // one CTA per SM: its 512 TMEM columns are free
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(probe)");
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(units * CG, 1, 1);
    cfg.blockDim = dim3(MODE == gb::kProbeSmspMath || MODE == gb::kProbeSmspPoll ? 256 : 128, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    if (CG == 2) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    e = cudaLaunchKernelEx(&cfg, kern, num_mma, alternate, static_cast<uint64_t>(1000000000ull), alu, tmap);
    if (e != cudaSuccess) return cuda_fail(e, "cudaLaunchKernelEx(probe)");
    return GB_OK;
}

template <int CG, int N>
gb_status_t probe_run(int mode, int units, int num_mma, int alternate, int alu, cudaStream_t stream) {
    if constexpr (CG != 2 || N != 256) {  // the issue-path variants exist for the GEMMs' pair shape only
        if (mode != gb::kProbePlain) return fail(GB_ERR_INVALID_ARG, "probe modes other than 0 need cta_group 2, n 256");
        return probe_launch<CG, N, gb::kProbePlain>(units, num_mma, alternate, alu, stream);
    } else {
    switch (mode) {
        case gb::kProbePlain: return probe_launch<CG, N, gb::kProbePlain>(units, num_mma, alternate, alu, stream);
        case gb::kProbeCommit: return probe_launch<CG, N, gb::kProbeCommit>(units, num_mma, alternate, alu, stream);
        case gb::kProbeWait: return probe_launch<CG, N, gb::kProbeWait>(units, num_mma, alternate, alu, stream);
        case gb::kProbeFence: return probe_launch<CG, N, gb::kProbeFence>(units, num_mma, alternate, alu, stream);
        case gb::kProbeWaitFence:
            return probe_launch<CG, N, gb::kProbeWaitFence>(units, num_mma, alternate, alu, stream);
        case gb::kProbeGemmStep: return probe_launch<CG, N, gb::kProbeGemmStep>(units, num_mma, alternate, alu, stream);
        case gb::kProbeAlu: return probe_launch<CG, N, gb::kProbeAlu>(units, num_mma, alternate, alu, stream);
        case gb::kProbeTmemLd16: return probe_launch<CG, N, gb::kProbeTmemLd16>(units, num_mma, alternate, alu, stream);
        case gb::kProbeTmemLd32: return probe_launch<CG, N, gb::kProbeTmemLd32>(units, num_mma, alternate, alu, stream);
        case gb::kProbeTmemLd64: return probe_launch<CG, N, gb::kProbeTmemLd64>(units, num_mma, alternate, alu, stream);
        case gb::kProbeStages: return probe_launch<CG, N, gb::kProbeStages>(units, num_mma, alternate, alu, stream);
        case gb::kProbeStagesWrites:
            return probe_launch<CG, N, gb::kProbeStagesWrites>(units, num_mma, alternate, alu, stream);
        case gb::kProbeStagesStores:
            return probe_launch<CG, N, gb::kProbeStagesStores>(units, num_mma, alternate, alu, stream);
        case gb::kProbeStagesTma: return probe_launch<CG, N, gb::kProbeStagesTma>(units, num_mma, alternate, alu, stream);
        case gb::kProbeStagesTma2: return probe_launch<CG, N, gb::kProbeStagesTma2>(units, num_mma, alternate, alu, stream);
        case gb::kProbeFenceProxy: return probe_launch<CG, N, gb::kProbeFenceProxy>(units, num_mma, alternate, alu, stream);
        case gb::kProbePoll: return probe_launch<CG, N, gb::kProbePoll>(units, num_mma, alternate, alu, stream);
        case gb::kProbeTmaStore: return probe_launch<CG, N, gb::kProbeTmaStore>(units, num_mma, alternate, alu, stream);
        case gb::kProbeSmspMath: return probe_launch<CG, N, gb::kProbeSmspMath>(units, num_mma, alternate, alu, stream);
        case gb::kProbeSmspPoll: return probe_launch<CG, N, gb::kProbeSmspPoll>(units, num_mma, alternate, alu, stream);
        case gb::kProbeMnMajor: return probe_launch<CG, N, gb::kProbeMnMajor>(units, num_mma, alternate, alu, stream);
        default: return probe_launch<CG, N, gb::kProbePipeline>(units, num_mma, alternate, alu, stream);
    }
    }
}

// Shared by the two probe entry points: launch, synchronise, median cycles per MMA.
gb_status_t probe_measure(int cta_group, int n, int mode, int alternate, int alu, int num_mma, int units,
                          double* cycles_per_mma, double* loads_per_mma = nullptr) {
    if (cta_group != 1 && cta_group != 2) return fail(GB_ERR_INVALID_ARG, "cta_group must be 1 or 2");
    if (n != 128 && n != 256) return fail(GB_ERR_INVALID_ARG, "n must be 128 or 256");
    if (num_mma < 8 || num_mma > 65536 || num_mma % 4) return fail(GB_ERR_INVALID_ARG, "num_mma must be a multiple of 4 in [8, 65536]");
    if (mode < 0 || mode >= gb::kProbeModes) return fail(GB_ERR_INVALID_ARG, "unknown probe mode %d", mode);
    if (alu < 0 || alu > 1024) return fail(GB_ERR_INVALID_ARG, "alu must be in [0, 1024]");
    int dev = 0;
    DeviceInfo info;
    gb_status_t st = device_info(&dev, &info);
    if (st != GB_OK) return st;
    const int max_units = std::min(gb::kProbeMaxUnits, info.sms / cta_group);
    if (units < 1 || units > max_units)
        return fail(GB_ERR_INVALID_ARG, "units must be in [1, %d] (one CTA per SM)", max_units);
    static const unsigned long long zeros[gb::kProbeMaxUnits] = {};
    cudaError_t e = cudaMemcpyToSymbol(gb::g_probe_cycles, zeros, sizeof zeros);
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(gb::g_probe_loads, zeros, sizeof zeros);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the probe results");
    cudaStream_t stream = nullptr;
    if (cta_group == 1)
        st = n == 128 ? probe_run<1, 128>(mode, units, num_mma, alternate, alu, stream)
                      : probe_run<1, 256>(mode, units, num_mma, alternate, alu, stream);
    else
        st = n == 128 ? probe_run<2, 128>(mode, units, num_mma, alternate, alu, stream)
                      : probe_run<2, 256>(mode, units, num_mma, alternate, alu, stream);
    if (st != GB_OK) return st;
    if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize(probe)");
    unsigned long long cyc[gb::kProbeMaxUnits];
    if ((e = cudaMemcpyFromSymbol(cyc, gb::g_probe_cycles, sizeof cyc)) != cudaSuccess)
        return cuda_fail(e, "reading the probe results");
    std::sort(cyc, cyc + units);
    if (cyc[0] == 0) return fail(GB_ERR_TIMEOUT, "a probe unit's wait for its MMAs ran out");
    *cycles_per_mma = static_cast<double>(cyc[units / 2]) / num_mma;
    if (loads_per_mma) {
        unsigned long long ld[gb::kProbeMaxUnits];
        if ((e = cudaMemcpyFromSymbol(ld, gb::g_probe_loads, sizeof ld)) != cudaSuccess)
            return cuda_fail(e, "reading the probe load counts");
        std::sort(ld, ld + units);
        *loads_per_mma = static_cast<double>(ld[units / 2]) / num_mma;
    }
    return GB_OK;
}

}  // namespace

extern "C" {

gb_status_t gb_measure_mma_rate(int cta_group, int n, int alternate, int num_mma, int units,
                                double* flops_per_clk_per_sm, double* cycles_per_mma) {
    t_error.clear();
    if (!flops_per_clk_per_sm || !cycles_per_mma) return fail(GB_ERR_INVALID_ARG, "output pointer is null");
    double per_mma = 0;
    gb_status_t st = probe_measure(cta_group, n, gb::kProbePlain, alternate ? 1 : 0, 0, num_mma, units, &per_mma);
    if (st != GB_OK) return st;
    *cycles_per_mma = per_mma;
    *flops_per_clk_per_sm = 2.0 * 128.0 * cta_group * n * 16.0 / per_mma / cta_group;
    return GB_OK;
}

gb_status_t gb_probe_mma_issue(int cta_group, int n, int mode, int alu, int num_mma, int units,
                               double* cycles_per_mma, double* tmem_loads_per_mma) {
    t_error.clear();
    if (!cycles_per_mma) return fail(GB_ERR_INVALID_ARG, "output pointer is null");
    // mode bit 8: operands of random bf16 values instead of zeros
    const int noisy = (mode >> 8) & 1;
    return probe_measure(cta_group, n, mode & 0xff, noisy ? 2 : 0, alu, num_mma, units, cycles_per_mma,
                         tmem_loads_per_mma);
}

gb_status_t gb_gemm_linear(const void* A, int64_t lda, const void* B, int64_t ldb, const void* bias, const void* R,
                           int64_t ldr, int act, void* D, int64_t ldd, int64_t M, int64_t N, int64_t K, void* stream) {
    t_error.clear();
    Problem pr{A, lda, B, ldb, nullptr, 0, bias, R, ldr, act, D, ldd, M, N, K, false};
    return run(pr, stream);
}

gb_status_t gb_gemm_linear_preact(const void* A, int64_t lda, const void* B, int64_t ldb, const void* bias,
                                  const void* R, int64_t ldr, int act, void* D, int64_t ldd, void* Z, int64_t ldz,
                                  int64_t M, int64_t N, int64_t K, void* stream) {
    t_error.clear();
    if (!Z && M > 0 && N > 0) return fail(GB_ERR_INVALID_ARG, "Z is null");
    Problem pr{A, lda, B, ldb, nullptr, 0, bias, R, ldr, act, D, ldd, M, N, K, false, Z, ldz};
    return run(pr, stream);
}

gb_status_t gb_gemm_linear_dact(const void* dY, int64_t lddy, const void* W, int64_t ldw, const void* Z,
                                int64_t ldz, int act, void* D, int64_t ldd, int64_t M, int64_t N, int64_t K,
                                void* stream) {
    t_error.clear();
    // output [M, K], contraction over N: in the plan's terms n = K and k = N
    Problem pr{dY, lddy, W, ldw, nullptr, 0, nullptr, Z, ldz, act, D, ldd, M, K, N, false};
    pr.b_mn = true;
    pr.dact = true;
    return run(pr, stream);
}

gb_status_t gb_gemm_matmul(const void* A, int64_t lda, const void* B, int64_t ldb, const void* bias, const void* R,
                           int64_t ldr, int act, void* D, int64_t ldd, int64_t M, int64_t N, int64_t K,
                           void* stream) {
    t_error.clear();
    Problem pr{A, lda, B, ldb, nullptr, 0, bias, R, ldr, act, D, ldd, M, N, K, false};
    pr.b_mn = true;
    return run(pr, stream);
}

gb_status_t gb_gemm_ffn_gated(const void* X, int64_t ldx, const void* W1, int64_t ldw1, const void* W3, int64_t ldw3,
                              void* D, int64_t ldd, int64_t M, int64_t N, int64_t K, void* stream) {
    t_error.clear();
    Problem pr{X, ldx, W1, ldw1, W3, ldw3, nullptr, nullptr, 0, GB_ACT_NONE, D, ldd, M, N, K, true};
    return run(pr, stream);
}

gb_status_t gb_gemm_linear_splitk(const void* A, int64_t lda, const void* B, int64_t ldb, const void* bias,
                                  const void* R, int64_t ldr, int act, void* D, int64_t ldd, int64_t M, int64_t N,
                                  int64_t K, int splits, void* workspace, size_t workspace_bytes, void* stream) {
    t_error.clear();
    Problem pr{A, lda, B, ldb, nullptr, 0, bias, R, ldr, act, D, ldd, M, N, K, false};
    SplitReq sr;
    sr.allowed = true;
    sr.splits = splits;
    sr.ws = workspace;
    sr.ws_bytes = workspace_bytes;
    return run(pr, stream, sr);
}

gb_status_t gb_gemm_ffn_gated_splitk(const void* X, int64_t ldx, const void* W1, int64_t ldw1, const void* W3,
                                     int64_t ldw3, void* D, int64_t ldd, int64_t M, int64_t N, int64_t K, int splits,
                                     void* workspace, size_t workspace_bytes, void* stream) {
    t_error.clear();
    Problem pr{X, ldx, W1, ldw1, W3, ldw3, nullptr, nullptr, 0, GB_ACT_NONE, D, ldd, M, N, K, true};
    SplitReq sr;
    sr.allowed = true;
    sr.splits = splits;
    sr.ws = workspace;
    sr.ws_bytes = workspace_bytes;
    return run(pr, stream, sr);
}

gb_status_t gb_splitk_workspace_bytes(int ffn, int64_t M, int64_t N, int64_t K, int splits, size_t* bytes) {
    t_error.clear();
    if (!bytes) return fail(GB_ERR_INVALID_ARG, "bytes is null");
    if (M < 0 || N < 0 || K < 0) return fail(GB_ERR_INVALID_ARG, "negative size");
    // Sizes only: fake, never-dereferenced operand addresses that pass validation.
    static const uint16_t dummy[8] __attribute__((aligned(16))) = {};
    const int64_t kk = K > 0 ? ((K + 7) / 8) * 8 : 0;
    Problem pr{dummy, kk, dummy, kk, ffn ? dummy : nullptr, kk, nullptr, nullptr, 0, GB_ACT_NONE,
               const_cast<uint16_t*>(dummy), N, M, N, K, ffn != 0};
    SplitReq sr;
    sr.allowed = true;
    sr.splits = splits;
    sr.query_only = true;
    sr.ws_needed = bytes;
    *bytes = 0;
    return run(pr, nullptr, sr);
}

gb_status_t gb_gemm_linear_splitk_noalloc(const void* A, int64_t lda, const void* B, int64_t ldb, const void* bias,
                                          const void* R, int64_t ldr, int act, void* D, int64_t ldd, int64_t M,
                                          int64_t N, int64_t K, int splits, void* stream) {
    t_error.clear();
    Problem pr{A, lda, B, ldb, nullptr, 0, bias, R, ldr, act, D, ldd, M, N, K, false};
    gb_status_t st = validate(pr);
    if (st != GB_OK) return st;
    if (pr.m == 0 || pr.n == 0) {
        t_plan = "empty (no launch)";
        t_plan_rec.valid = false;
        return GB_OK;
    }
    int dev = 0;
    DeviceInfo info;
    if ((st = device_info(&dev, &info)) != GB_OK) return st;
    void* scratch = nullptr;
    if ((st = static_scratch_address(dev, &scratch)) != GB_OK) return st;

    // Every split count above 1 needs the same scratch (one fp32 accumulator tile per
    // output tile, plus counters), so a plan that does not fit can only run unsplit.
    size_t need = 0;
    if ((st = splitk_bytes_for(pr, splits, &need)) != GB_OK) return st;
    if (need > kStaticScratchBytes) {
        if (splits > 1)
            return fail(GB_ERR_UNSUPPORTED,
                        "split-K of this problem needs %zu bytes of scratch, more than the %zu-byte static scratch "
                        "of gb_gemm_linear_splitk_noalloc, for any split count above 1; use splits=1 or "
                        "gb_gemm_linear_splitk with a workspace",
                        need, kStaticScratchBytes);
        splits = 1;  // automatic: the partials do not fit, so the call runs unsplit
    }
    SplitReq sr;
    sr.allowed = true;
    sr.splits = splits;
    sr.ws = scratch;
    sr.ws_bytes = kStaticScratchBytes;
    return run(pr, stream, sr);
}

gb_status_t gb_static_scratch_bytes(size_t* bytes) {
    if (!bytes) return fail(GB_ERR_INVALID_ARG, "bytes is null");
    *bytes = kStaticScratchBytes;
    return GB_OK;
}

gb_status_t gb_get_device_status(void* stream) {
    t_error.clear();
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    uint32_t v = 0;
    if ((e = cudaMemcpyFromSymbol(&v, gb::g_gb_status, sizeof v)) != cudaSuccess)
        return cuda_fail(e, "reading the device status word");
    if (v == 0) return GB_OK;
    const uint32_t zero = 0;
    if ((e = cudaMemcpyToSymbol(gb::g_gb_status, &zero, sizeof zero)) != cudaSuccess)
        return cuda_fail(e, "clearing the device status word");
    const uint32_t code = v & 0xffu, role = (v >> 8) & 0xffu, where = v >> 16;
    static const char* roles[] = {"?", "producer", "mma", "epilogue"};
    return fail(static_cast<gb_status_t>(code), "device pipeline wait timed out (role=%s, where=0x%x)",
                roles[role < 4 ? role : 0], where);
}

const char* gb_last_error(void) { return t_error.c_str(); }

gb_status_t gb_set_config(const char* spec) {
    Config c;
    if (spec && *spec) {
        const char* s = spec;
        while (*s) {
            const char* comma = strchr(s, ',');
            size_t len = comma ? static_cast<size_t>(comma - s) : strlen(s);
            const char* eq = static_cast<const char*>(memchr(s, '=', len));
            if (!eq) return fail(GB_ERR_INVALID_ARG, "config item without '=': %.*s", static_cast<int>(len), s);
            std::string key(s, static_cast<size_t>(eq - s));
            long v = 0;
            if (!parse_int(eq + 1, len - static_cast<size_t>(eq + 1 - s), &v))
                return fail(GB_ERR_INVALID_ARG, "bad value for %s", key.c_str());
            if (key == "bn" && (v == 128 || v == 256)) c.bn = static_cast<int>(v);
            else if (key == "grid" && v >= 0 && v <= 1000000) c.grid = static_cast<int>(v);
            else if (key == "persistent" && (v == 0 || v == 1)) c.persistent = static_cast<int>(v);
            else if (key == "group" && v >= 1 && v <= 1000000) c.group = static_cast<int>(v);
            else if (key == "zigzag" && v >= -1 && v <= 1) c.zigzag = static_cast<int>(v);
            else if (key == "pair" && v >= -1 && v <= 1) c.pair = static_cast<int>(v);
            else if (key == "stages" && v >= 0 && v <= 16) c.stages = static_cast<int>(v);
            else if (key == "epi" && (v == 0 || v == 1 || v == 2 || v == 4)) c.epi = static_cast<int>(v);
            else if (key == "boxes" && (v == 0 || (v >= 2 && v <= gb::kMaxBoxes))) c.boxes = static_cast<int>(v);
            else if (key == "pingpong" && v >= -1 && v <= 1) c.pingpong = static_cast<int>(v);
            else if (key == "hint_a" && v >= -1 && v <= 2) c.hint_a = static_cast<int>(v);
            else if (key == "hint_b" && v >= -1 && v <= 2) c.hint_b = static_cast<int>(v);
            else if (key == "hint_r" && v >= -1 && v <= 2) c.hint_r = static_cast<int>(v);
            else if (key == "hint_d" && v >= -1 && v <= 2) c.hint_d = static_cast<int>(v);
            else if (key == "mc" && v >= -1 && v <= 1) c.mc = static_cast<int>(v);
            else if (key == "issue" && v >= -1 && v <= 3) c.issue = static_cast<int>(v);
            else if (key == "prod" && v >= 0 && v <= 3) c.prod = static_cast<int>(v);
            else if (key == "r_async" && v >= -1 && v <= 1) c.r_async = static_cast<int>(v);
            else if (key == "r_boxes" && (v == 0 || (v >= 2 && v <= gb::kMaxBoxes))) c.r_boxes = static_cast<int>(v);
            else if (key == "wide" && v >= -1 && v <= 2) c.wide = static_cast<int>(v);
            else return fail(GB_ERR_INVALID_ARG, "unknown config key or value: %s=%ld", key.c_str(), v);
            s += len;
            if (*s == ',') ++s;
        }
    }
    std::lock_guard<std::mutex> lk(g_cfg_mu);
    g_cfg = c;
    return GB_OK;
}

gb_status_t gb_set_wait_timeout_ns(uint64_t ns) {
    std::lock_guard<std::mutex> lk(g_cfg_mu);
    g_timeout_ns = ns ? ns : kDefaultTimeoutNs;
    return GB_OK;
}

gb_status_t gb_last_plan(char* buf, size_t len) {
    if (!buf) return fail(GB_ERR_INVALID_ARG, "buf is null");
    if (len == 0) return GB_OK;
    const PlanRec& r = t_plan_rec;
    if (!r.valid) {
        snprintf(buf, len, "%s", t_plan.c_str());
        return GB_OK;
    }
    snprintf(buf, len,
             "kernel=%s pair=%d mc=%d epi=%d pingpong=%d tile=%dx%dx%d stages=%d boxes=%d/%d grid=%lld tiles=%d "
             "k_blocks=%d splits=%d group=%d zigzag=%d prod=%d hints=%u%u%u%u "
             "d_store=%s r_load=%s z_store=%s",
             r.kernel, r.pair, r.mc, r.epi, r.pingpong, r.tile_m, r.bn, gb::kBK, r.stages, r.d_boxes, r.r_boxes, r.grid,
             r.tiles, r.k_blocks, r.splits, r.group, r.zigzag, r.prod, r.hint_a, r.hint_b, r.hint_r, r.hint_d, r.d_store,
             r.r_load, r.z_store);
    return GB_OK;
}

gb_status_t gb_set_fault_injection(int mode) {
    if (mode != gb::kInjectNone && mode != gb::kInjectSkipFirstStage)
        return fail(GB_ERR_INVALID_ARG, "unknown fault-injection mode %d", mode);
    std::lock_guard<std::mutex> lk(g_cfg_mu);
    g_inject = mode;
    return GB_OK;
}

gb_status_t gb_set_trace_buffer(void* buf, size_t bytes) {
#ifdef GB_TRACE
    std::lock_guard<std::mutex> lk(g_cfg_mu);
    g_trace = static_cast<unsigned long long*>(buf);
    g_trace_bytes = buf ? bytes : 0;
    return GB_OK;
#else
    (void)buf;
    (void)bytes;
    return fail(GB_ERR_UNSUPPORTED, "this library was built without GB_TRACE");
#endif
}

const char* gb_version(void) { return "0.1.0"; }

}  // extern "C"
