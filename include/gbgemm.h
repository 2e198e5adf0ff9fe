/*
 * gbgemm -- persistent, warp-specialised bf16 GEMM with a fused epilogue for
 * GB300 (sm_103a): TMA -> shared-memory ring -> tcgen05.mma into TMEM ->
 * epilogue -> TMA store.  C ABI; plain pointers and sizes only.
 *
 * Operations (the problem statement of "Implement persistent matmul
 * scheduling", NVIDIA/Fuser PR #3812, and "Translate MmaOp patterns properly
 * on Hopper", NVIDIA/Fuser PR #4072: MatmulOp = A.B, LinearOp = linear layer
 * with bias, tensors in the EPILOGUE_INPUT role, the Llama-FFN horizontal
 * fusion; "Automate performant Hopper matmul", NVIDIA/Fuser issue #3819,
 * section "Epilogue"):
 *
 *   gb_gemm_linear    D[m,n] = bf16( act( sum_k A[m,k] B[n,k] + bias[n] ) + R[m,n] )
 *   gb_gemm_ffn_gated D[m,n] = bf16( silu( sum_k X[m,k] W1[n,k] ) * sum_k X[m,k] W3[n,k] )
 *
 * Arithmetic: bf16 operands, fp32 accumulation in tensor memory, fp32
 * epilogue, one round-to-nearest-even to bf16.  The accumulation order inside
 * the tensor core is not the sequential k order, so results agree with a
 * sequential fp32 sum up to rounding.
 *
 * Layouts.  Every matrix is row-major bf16 (passed as raw 16-bit storage) with
 * a leading dimension given in ELEMENTS.  A is [M,K] and B is [N,K]: both
 * operands are K-major ("TN"), as a linear layer stores its weight.  bias is a
 * contiguous [N] vector.  R and D are [M,N].
 *
 * Ownership.  All pointers are DEVICE pointers owned by the caller and must
 * stay valid until the work queued on `stream` has finished.  The library
 * allocates no device memory at run time: it keeps a host-side cache of TMA
 * descriptors, and its own static device memory holds only a 32-bit status
 * word and the scratch array of gb_gemm_linear_splitk_noalloc (both part of
 * the loaded module).
 *
 * Synchronisation.  Calls only validate, plan and enqueue on `stream` (a
 * cudaStream_t; NULL means the legacy default stream) and return at once.
 *
 * Aliasing.  D must not overlap A, B, X, W1, W3 or bias.  D == R (same pointer
 * and leading dimension) is allowed: every element of R is read before the same
 * element of D is written, by the same thread.
 *
 * Errors.  Every call returns a gb_status_t; nothing aborts or throws.
 * gb_last_error() gives a message for the last non-OK status on the calling
 * thread.  Faults that can only be seen on the device (a pipeline wait that
 * ran out of time) are recorded in the device status word and reported by
 * gb_get_device_status().
 *
 * Limits.  0 <= M, N, K < 2^31; leading dimensions >= the row length.
 * A, B, X, W1, W3: base address 16-byte aligned and leading dimension a
 * multiple of 8 elements (TMA requires 16-byte aligned rows), else
 * GB_ERR_UNSUPPORTED.  D, R, bias: any 2-byte aligned address and leading
 * dimension; when D (or R) is 16-byte aligned with a leading dimension that is
 * a multiple of 8, it moves by TMA, otherwise by predicated plain loads and
 * stores.  M == 0 or N == 0 is a no-op.  K == 0 gives D = act(bias) + R.
 */
#ifndef GBGEMM_H
#define GBGEMM_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define GB_API __attribute__((visibility("default")))
#else
#define GB_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GB_OK = 0,
    GB_ERR_INVALID_ARG = 1,  /* a null pointer, a negative size, a too-small leading dimension */
    GB_ERR_UNSUPPORTED = 2,  /* valid but outside what the kernels handle (alignment, size) */
    GB_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed (message in gb_last_error) */
    GB_ERR_TIMEOUT = 4       /* a device pipeline wait ran out of time (gb_get_device_status) */
} gb_status_t;

typedef enum {
    GB_ACT_NONE = 0,
    GB_ACT_GELU_TANH = 1,    /* 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))) */
    GB_ACT_SILU = 2,         /* x / (1 + exp(-x)) */
    GB_ACT_RELU = 3          /* max(x, 0) */
} gb_act_t;

/*
 * D = bf16( act(A . B^T + bias) + R ).
 * Matmul / linear layer with its fused epilogue ("Automate performant Hopper
 * matmul", sections "Persistent matmul" and "Epilogue"; the EPILOGUE_INPUT
 * role in "Translate MmaOp patterns properly on Hopper").
 *   A    [M,K], leading dimension lda (elements)        required if M,K > 0
 *   B    [N,K], leading dimension ldb                   required if N,K > 0
 *   bias [N] or NULL (no bias)
 *   R    [M,N] with leading dimension ldr, or NULL (no epilogue input)
 *   act  a gb_act_t value
 *   D    [M,N] with leading dimension ldd               required if M,N > 0
 *   stream  cudaStream_t to enqueue on
 * Returns GB_OK once the work is enqueued.
 */
GB_API gb_status_t gb_gemm_linear(const void* A, int64_t lda, const void* B, int64_t ldb,
                           const void* bias, const void* R, int64_t ldr, int act,
                           void* D, int64_t ldd, int64_t M, int64_t N, int64_t K,
                           void* stream);

/*
 * gb_gemm_linear with a second output: Z = bf16(A . B^T + bias), the
 * pre-activation a backward pass of the activation needs, stored from the
 * same epilogue pass; D as in gb_gemm_linear.  Both outputs leave through the
 * same per-warp staging boxes, each box rewritten only after the store that
 * used it has read it ("Automate performant Hopper matmul", section "TMA store
 * and stmatrix": reuse shared memory for TMA stores of several outputs by
 * waiting for the earlier stores).
 *   Z  [M,N] with leading dimension ldz (elements); required if M,N > 0; any
 *      2-byte alignment (TMA when 16-byte aligned rows, else the transpose
 *      path); must not overlap A, B, bias, R or D.
 * Errors and limits as gb_gemm_linear.
 */
GB_API gb_status_t gb_gemm_linear_preact(const void* A, int64_t lda, const void* B, int64_t ldb,
                                         const void* bias, const void* R, int64_t ldr, int act,
                                         void* D, int64_t ldd, void* Z, int64_t ldz,
                                         int64_t M, int64_t N, int64_t K, void* stream);

/*
 * D = bf16( silu(X . W1^T) * (X . W3^T) ): the Llama-FFN horizontal fusion,
 * two products sharing the X operand, both fp32-accumulated before the
 * epilogue ("Translate MmaOp patterns properly on Hopper", commit "Fix llama
 * ffn horizontal fusion on Ampere").
 *   X  [M,K] (ldx), W1 [N,K] (ldw1), W3 [N,K] (ldw3), D [M,N] (ldd).
 */
GB_API gb_status_t gb_gemm_ffn_gated(const void* X, int64_t ldx, const void* W1, int64_t ldw1,
                              const void* W3, int64_t ldw3, void* D, int64_t ldd,
                              int64_t M, int64_t N, int64_t K, void* stream);

/*
 * Split-K variants, for problems with too few output tiles to fill the GPU
 * (the skinny shapes: M or N of one tile, long K).  Split-K and stream-K are the
 * two schedules "Implement persistent matmul scheduling" (NVIDIA/Fuser PR #3812,
 * reviewer guide) records as unsupported by its persistent Hopper scheduler.
 *
 * The k-blocks of every output tile are cut into `splits` contiguous ranges;
 * each (tile, range) is one work item of the persistent kernel.  Every range
 * adds its fp32 partial accumulator into the tile's fp32 accumulator in the
 * workspace (fp32 reductions performed in L2); the last range to finish a
 * 32-row slab of a tile (a per-slab counter in the workspace) reads the sum
 * and applies the same epilogue as the non-split call.  The order of the fp32
 * additions across ranges is not fixed, so two calls may differ by rounding;
 * results equal a sequential fp32 sum up to rounding, like every other call
 * (inputs whose partial sums are exact give identical bits).
 *   splits     <= 0: chosen automatically (1 when the tiles fill half of the
 *              GPU, or a quarter of it with fewer than 256 64-wide k-blocks; at
 *              most 64); otherwise clamped to [1, number of 64-wide k-blocks].
 *   workspace  device memory owned by the caller, 256-byte aligned, at least
 *              gb_splitk_workspace_bytes() bytes (may be NULL when that is 0):
 *              one fp32 accumulator tile per output tile plus the counters.
 *              Each call clears it on `stream` first, so calls that share one
 *              workspace must be ordered on the GPU (same stream or events);
 *              overlapping calls on one workspace race.
 * Other arguments, errors and limits as gb_gemm_linear / gb_gemm_ffn_gated.
 * GB_ERR_INVALID_ARG if the workspace is missing, too small or misaligned.
 */
GB_API gb_status_t gb_gemm_linear_splitk(const void* A, int64_t lda, const void* B, int64_t ldb,
                                         const void* bias, const void* R, int64_t ldr, int act,
                                         void* D, int64_t ldd, int64_t M, int64_t N, int64_t K,
                                         int splits, void* workspace, size_t workspace_bytes,
                                         void* stream);

GB_API gb_status_t gb_gemm_ffn_gated_splitk(const void* X, int64_t ldx, const void* W1, int64_t ldw1,
                                            const void* W3, int64_t ldw3, void* D, int64_t ldd,
                                            int64_t M, int64_t N, int64_t K, int splits,
                                            void* workspace, size_t workspace_bytes, void* stream);

/*
 * Matrix product with B in its natural [K, N] layout (the MatmulOp form, A.B,
 * beside the LinearOp form A.B^T of gb_gemm_linear):
 *
 *   D[m,n] = bf16( act( sum_k A[m,k] B[k,n] + bias[n] ) + R[m,n] )
 *
 * B is a row-major [K, N] matrix (ldb >= N): the contraction runs over its rows,
 * so the tensor cores read it as an MN-major operand straight from its layout
 * (TMA boxes of 64 columns x 64 rows), with no transposed copy.  "Translate MmaOp
 * patterns properly on Hopper" (NVIDIA/Fuser PR #4072, description: MatmulOp and
 * LinearOp) names both forms.  A and B: base 16-byte aligned, lda and ldb
 * multiples of 8 (TMA), lda >= K, ldb >= N.  bias, R, D, act, the epilogue
 * order, the store and load paths, errors and limits as gb_gemm_linear.
 */
GB_API gb_status_t gb_gemm_matmul(const void* A, int64_t lda, const void* B, int64_t ldb, const void* bias,
                                  const void* R, int64_t ldr, int act, void* D, int64_t ldd, int64_t M, int64_t N,
                                  int64_t K, void* stream);

/*
 * Activation gradient of a linear layer's input (the backward-pass consumer of
 * the pre-activation that gb_gemm_linear_preact stores):
 *
 *   D[m,k] = bf16( sum_n dY[m,n] W[n,k] * act'(Z[m,k]) )
 *
 * dY [M,N] is the gradient of the layer's output, W [N,K] the layer's weight in
 * the same row-major layout gb_gemm_linear takes as B (so the contraction runs
 * over the rows of W: an MN-major tensor-core operand, read by TMA as it is, with
 * no transposed copy), and Z [M,K] the pre-activation whose activation `act`
 * produced the layer's input.  act' is the derivative of the tanh-form GELU, of
 * SiLU, of ReLU (1 for z > 0, else 0) or of the identity (1).  "Implement
 * persistent matmul scheduling" (NVIDIA/Fuser PR #3812, description: MLP
 * benchmark tests with epilogue fusions) and "Automate performant Hopper matmul"
 * (NVIDIA/Fuser issue #3819, section "Epilogue": epilogue inputs) name the
 * fusion pattern; the formula is its plain reading (chain rule).
 * dY and W: base 16-byte aligned, lddy and ldw multiples of 8 (TMA), lddy >= N,
 * ldw >= K.  Z and D: 2-byte aligned, ldz >= K, ldd >= K; TMA when 16-byte
 * aligned rows, else plain loads and stores.  Z is required (GB_ERR_INVALID_ARG
 * if NULL).  N == 0 gives D = 0 * act'(Z) (signed zeros).  D must not overlap dY
 * or W; D == Z (same pointer and leading dimension) is allowed.  Other arguments,
 * errors and limits as gb_gemm_linear.
 */
GB_API gb_status_t gb_gemm_linear_dact(const void* dY, int64_t lddy, const void* W, int64_t ldw,
                                       const void* Z, int64_t ldz, int act, void* D, int64_t ldd,
                                       int64_t M, int64_t N, int64_t K, void* stream);

/*
 * Workspace bytes the split-K call needs for this problem on the current
 * device under the current configuration (ffn: 0 = linear, 1 = FFN fusion;
 * splits as above).  Writes 0 when the plan does not split.  Needs a CUDA
 * device (the plan depends on the SM count); launches nothing.
 */
GB_API gb_status_t gb_splitk_workspace_bytes(int ffn, int64_t M, int64_t N, int64_t K, int splits,
                                             size_t* bytes);

/*
 * gb_gemm_linear_splitk without a workspace argument: the split-K partials and
 * counters live in a fixed 32 MiB array in this library's own device memory
 * (gb_static_scratch_bytes), so the call allocates no device memory at all.
 * The source pages have no counterpart to this entry point; it exists for
 * callers that may not allocate device memory themselves and cannot lend one --
 * for example a framework whose own caching allocator must own every device
 * allocation, or a serving runtime that reserves all memory at start-up and may
 * not allocate while it handles requests.
 *   splits  > 0: used as given (clamped as in gb_gemm_linear_splitk).  Every
 *           split count above 1 needs the same scratch (one fp32 tile per
 *           output tile plus counters); if that does not fit the static
 *           scratch the call returns GB_ERR_UNSUPPORTED with the bytes needed
 *           and allowed (splits = 1 always fits: it needs none).
 *           <= 0: automatic; when the automatic plan's partials do not fit,
 *           the call runs unsplit (splits = 1) instead.
 * Set-up: the first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current and caches it; make that first
 * call before any stream capture.  Every call on a device shares the one array,
 * which keeps the previous call's contents: each call clears the part it uses on
 * `stream` first, and calls that overlap on the GPU (different streams without
 * ordering) race on the array.  Other arguments, errors and limits as
 * gb_gemm_linear_splitk.
 */
GB_API gb_status_t gb_gemm_linear_splitk_noalloc(const void* A, int64_t lda, const void* B, int64_t ldb,
                                                 const void* bias, const void* R, int64_t ldr, int act,
                                                 void* D, int64_t ldd, int64_t M, int64_t N, int64_t K,
                                                 int splits, void* stream);

/* Size in bytes of the static scratch gb_gemm_linear_splitk_noalloc uses
 * (GB_ERR_INVALID_ARG for a null pointer). */
GB_API gb_status_t gb_static_scratch_bytes(size_t* bytes);

/*
 * Synchronise `stream`, then read and clear the current device's status word.
 * GB_OK if no kernel recorded a fault since the last call; GB_ERR_TIMEOUT if a
 * pipeline wait ran out of time (the kernel then stopped early and its output
 * is undefined); GB_ERR_CUDA if the synchronisation itself failed.
 * gb_last_error() then names the role and stage that gave up.
 */
GB_API gb_status_t gb_get_device_status(void* stream);

/* Message for the last non-OK status returned on the calling thread ("" if none).
 * The pointer stays valid until the next gbgemm call on the same thread. */
GB_API const char* gb_last_error(void);

/*
 * Tile-configuration override, the analogue of a heuristic plugin.  `spec` is
 * a comma-separated list of key=value pairs, or NULL / "" to restore the
 * built-in heuristic.  Keys: bn (linear tile width: 128 or 256), grid (maximum
 * number of CTAs; 0 = one per SM), persistent (0 = one tile per CTA),
 * group (tile-swizzle group size along M, >= 1), zigzag (0, 1, or -1 = auto),
 * pair (1 = CTA pairs with 256-row tiles, 0 = single CTAs with 128-row tiles,
 * -1 = auto; the 128-wide linear tile always runs on single CTAs), stages
 * (depth of the operand ring, >= 2, or 1 on the lean kernel; 0 = auto: the deepest that fits for
 * long K, 2-3 for work items of at most 4 k-blocks), boxes (D staging boxes
 * and TMA-loaded R boxes per epilogue warp, 2..8; 0 = auto: 2 for long K, the
 * deepest that fits for short K; boxes shrink before the ring does), r_boxes
 * (the R queue's depth alone, 2..8; 0 = auto), epi (epilogue warpgroups: 1, 2
 * or 4; 0 = auto: four for short-K residual work on CTA pairs with aligned
 * rows, two for other epilogue-bound shapes, else one; 4 runs the lean kernel,
 * which has only the paired epilogue path: other plans fall back to 2),
 * pingpong (1 = the two epilogue warpgroups alternate whole tiles, each owning
 * one TMEM accumulator buffer, instead of sharing every tile's chunks; implies
 * epi=2, GB_ERR_INVALID_ARG with epi=1 at the call, no effect with split-K;
 * 0 = never; -1 = auto: on for work items of at most 4 k-blocks), wide (the
 * paired epilogue path's boxes: 0 = 32x32 R and D boxes, 1 = 32x64 R and D
 * boxes, 2 = 32x64 D and 32x32 R boxes; -1 = auto: 1, or 2 on the lean
 * kernel), r_async (R rows that are not 16-byte aligned, without split: 1 =
 * per-lane cp.async word copies into a prefetch queue, 0 or -1 = synchronous
 * loads at use), mc (1 = A multicast between two CTA pairs in 4-CTA clusters,
 * without split), issue (MMA issue loop variant 0..3), prod (producer threads:
 * 1, 2 or 3; the lean loads need 2),
 * hint_a, hint_b, hint_r, hint_d (L2 eviction policy of the TMA loads of A,
 * of B / W1 / W3, of R, and of the TMA stores of D and Z: 0 = none, 1 = evict
 * first, 2 = evict last, -1 = the built-in choice).
 * Process-wide; returns GB_ERR_INVALID_ARG on an unknown key or value.
 */
GB_API gb_status_t gb_set_config(const char* spec);

/*
 * Upper bound, in nanoseconds, on every pipeline wait inside the kernels
 * (default 4e9, i.e. 4 s; 0 restores the default).  A wait that runs out
 * records GB_ERR_TIMEOUT in the device status word and the kernel returns.
 */
GB_API gb_status_t gb_set_wait_timeout_ns(uint64_t ns);

/*
 * Test hook for the failure path (process-wide).  mode 0: off (default).
 * mode 1: the producer never issues its first pipeline stage, so the MMA
 * role's wait on that stage runs out after the wait limit; every role then
 * stops, drains what it has in flight, frees TMEM and returns, and
 * gb_get_device_status() reports GB_ERR_TIMEOUT.  The output is undefined.
 * Nothing faults or hangs.  Returns GB_ERR_INVALID_ARG for other modes.
 */
GB_API gb_status_t gb_set_fault_injection(int mode);

/* Writes a one-line description of the last plan chosen on this thread
 * (tile shape, stages, grid, swizzle, store path) into buf (NUL-terminated,
 * truncated to len). Returns GB_OK, or GB_ERR_INVALID_ARG for a null buf. */
GB_API gb_status_t gb_last_plan(char* buf, size_t len);

/*
 * Timing trace, for a library built with -DGB_TRACE (the normal build returns
 * GB_ERR_UNSUPPORTED).  `buf` is device memory of the caller (NULL turns the
 * trace off).  Every later launch whose grid fits (32 unsigned 64-bit words per
 * CTA) writes one record per CTA: %globaltimer at entry, after set-up, at the
 * first MMA, at the last accumulator commit and at the end of the epilogue; the
 * SM clock cycles the producer, the MMA issuer and the first epilogue warp spent
 * blocked on their barriers (with the number of blocked waits); the first
 * epilogue warp's cycles per phase of its chunk loop (free D boxes, TMEM loads, R
 * waits, math, stores, R issue) and its step count; and a histogram of the MMA
 * issuer's k-block-to-k-block intervals.  The layout is kTrace* in gemm_kernel.cuh.
 */
GB_API gb_status_t gb_set_trace_buffer(void* buf, size_t bytes);

/*
 * Tensor-core rate probe (a measurement, not part of the GEMM path): `units`
 * CTAs (cta_group 1) or CTA pairs (cta_group 2), one per SM (pair of SMs), each
 * issue `num_mma` back-to-back tcgen05.mma.kind::f16 instructions of
 * M = 128 * cta_group, N = n (128 or 256), K = 16 from zeroed shared memory into
 * TMEM (alternate != 0: two accumulators in turn), with no loads and no
 * epilogue, and time them in SM clock cycles.  Writes the median over units of
 * the cycles per MMA and the dense bf16 rate per SM and clock it implies
 * (2 M N 16 / cycles / cta_group).  The nominal peak of the GPU is then
 * SMs x clock x that rate.  Runs on the legacy default stream and synchronises
 * the device.  num_mma a multiple of 4 in [8, 65536]; units in [1, SMs / cta_group].
 */
GB_API gb_status_t gb_measure_mma_rate(int cta_group, int n, int alternate, int num_mma, int units,
                                       double* flops_per_clk_per_sm, double* cycles_per_mma);

/*
 * The same probe with the issuing thread's steps around the MMAs (what those steps
 * cost the tensor pipe): mode 0 the MMAs alone; per four MMAs (one 64-wide
 * k-block) 1 a tcgen05.commit, 2 an already-satisfied mbarrier wait, 3 a
 * tcgen05.fence::after_thread_sync, 4 wait and fence, 5 wait, fence, descriptors
 * rebuilt from a stage index and a commit (the GEMM issuer's step); 6 `alu`
 * dependent integer operations after every MMA; 7, 8, 9 the MMAs alone while
 * warps 1-3 of every CTA read the other TMEM accumulator in a loop with
 * tcgen05.ld.32x32b of 16, 32 or 64 columns (an epilogue's TMEM reads); 10 the
 * MMAs reading six distinct 32 KiB operand stages in turn (an operand ring); 11
 * four stages while warp 1 keeps four 16 KiB bulk copies from global into other
 * shared memory in flight (a ring's fills); 12 four stages while warps 1-3 store
 * 16-byte vectors to other shared memory as fast as they can; 13 four stages
 * while warp 1 keeps four 16 KiB 2-D TMA tile loads (128-byte swizzle) into other
 * shared memory in flight, 14 the same from warps 1 and 2; 15-17 an epilogue's
 * steps in warps 1-3 beside the MMAs: 15 shared-memory stores then
 * fence.proxy.async and a warp sync, 16 polling an mbarrier that never completes,
 * 17 (warp 1) 2-D TMA stores of shared memory; 18, 19 with 256 threads, warps 4-7
 * (one on each SM sub-partition, warp 4 beside the issuing thread) running FMA
 * math (18) or polling an mbarrier that never completes (19); 20 a GEMM mainloop
 * without epilogue (TMA into a 6-stage ring, full/empty barriers, two producer
 * threads, the MMAs of each stage, a commit per stage); 21 as 0 with the B operand
 * MN-major (a row-major [K, N] matrix's layout, as gb_gemm_matmul and
 * gb_gemm_linear_dact read it).  Writes the median
 * cycles per MMA and, when tmem_loads_per_mma is not NULL, the TMEM loads (modes
 * 7-9), 16 KiB copies (modes 11, 13, 14) or warp-wide 16-byte stores (mode 12) the leader
 * CTA completed per MMA (0 otherwise).  mode | 256: the operand tiles hold random
 * bf16 values instead of zeros.
 */
GB_API gb_status_t gb_probe_mma_issue(int cta_group, int n, int mode, int alu, int num_mma, int units,
                                      double* cycles_per_mma, double* tmem_loads_per_mma);

/* Library version as "major.minor.patch". */
GB_API const char* gb_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GBGEMM_H */
