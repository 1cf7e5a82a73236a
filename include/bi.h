/*
 * bi.h - C ABI of the deterministic, batch-invariant training matmul (GB300, sm_103a).
 *
 * The three matmuls of a linear layer and a grouped per-row-expert variant:
 *
 *   forward   Y  = X * W (+ b)       X [M,K], W [K,N] ("[in, out]"), b [N], Y [M,N]
 *   dX        dX = dY * W^T          dY [M,N], dX [M,K]
 *   dW        dW = X^T * dY          dW [K,N]
 *   grouped   Y[m,:] = X[m,:] * W[e(m)]^T        W [E,N,K], row_experts [M] (u32)
 *             dX[m,:] = dY[m,:] * W[e(m)]        dW[e] = sum over rows of expert e
 *                                                 of dY[m,:]^T X[m,:] (always f32)
 *
 * Sources: sgemm-bi 0.1.1.post2 (PyPI page), sections "Use" (weight stored
 * [in, out]; the raw-pointer Engine.forward call with m, k, n, a dtype string,
 * a stream and a tensor-core flag) and "Determinism contracts" (the two tiers);
 * ViperLLM ffma.py, _FFMAAddmm (bias added in f32 before the single downcast;
 * gx = gy W^T, gW = x^T gy); rublas 0.1.45 src/tensor_grouped/mod.rs
 * (fn grouped_matmul_nt, struct GroupedBackward, GroupedMatmulError).
 *
 * ------------------------------------------------------------------------
 * Arithmetic contract
 * ------------------------------------------------------------------------
 * Scalar tier (tensor_cores = 0, a grouped f32 call, or a shape below the
 * tensor-core threshold): every output is one chain
 *      acc = +0.0f;  for i ascending: acc = fmaf(up(a_i), up(b_i), acc)
 * over the contracted index, where up() is the exact widening to f32.  The
 * forward adds up(b[n]) to acc in f32, then rounds once (round to nearest
 * even) to the operand type.  dW cuts the rows into chunks of BI_DW_CHUNK rows
 * counted from row 0, runs a chain per chunk, and adds the chunk partials by a
 * fixed pairwise tree over adjacent partials (an odd last partial is carried up
 * unchanged); then one rounding (or none, with dw_f32 = 1).  Grouped dweights
 * do the same per expert over that expert's rows in ascending row index.
 * Results are bit-identical to the reference CPU definition above, across
 * runs, and row m of Y / dX does not depend on M.
 *
 * Tensor-core tier (tensor_cores = 1, bf16/f16, non-M output dims >= 64, K and
 * N multiples of 8, 16-byte aligned pointers): tcgen05 MMA, f32 accumulation
 * in tensor memory, contracted index processed in fixed 64-wide blocks in
 * ascending order, no atomics.  Y and dX never split their contraction and
 * make no tile, order or instruction choice that depends on M, so each of
 * their rows is bit-identical for any M.  dW and the grouped dweights chain
 * the row blocks in ascending order inside the accumulator; an f32 result
 * over more than 8192 rows is taken in pieces of 8192 rows counted from row 0,
 * each added to the sum of the pieces before it.  A dense dW whose K x N
 * output tiles leave a partial last wave on 76 CTA pairs contracts each of
 * those tiles as up to 16 chunks of consecutive 64-row blocks, added by the
 * dW reduction's fixed pairwise tree (the choice depends on M, K and N only).
 * Results are bit-identical across runs and within the published tolerance
 * of the scalar tier (they are not bit-equal to it).
 *
 * f32 operands on the tensor-core tier (dense passes, K and N multiples of 4)
 * run as 3xTF32: each operand x is split into hi = tf32(x) and
 * lo = tf32(x - hi) (round to nearest, ties away), and each product is taken
 * as hi*hi + (lo*hi + hi*lo), the two sums in separate f32 accumulators added
 * once at the end.  The contraction is cut into fixed pieces of 4096 elements
 * counted from 0 (a length independent of M); each piece's f32 result is added
 * to the sum of the pieces before it, in piece order, then the bias.  Same
 * guarantees as above: run-to-run identical, M-invariant rows, within the
 * published f32 tolerance of the scalar tier.  Scratch for the parts comes
 * from the engine's stream-ordered pool.
 *
 * Dispatch looks only at (pass, dtype, tensor_cores, K, N): never at M.
 *
 * ------------------------------------------------------------------------
 * Conventions
 * ------------------------------------------------------------------------
 * - Every tensor is dense, row-major, contiguous, on the engine's device, and
 *   owned by the caller.  Pointers are device pointers.  bf16/f16 data are
 *   the IEEE encodings; f32 is binary32.
 * - No output of a call may overlap any of its inputs: the kernels read the
 *   inputs through the read-only data path while they write the outputs.
 * - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls only
 *   enqueue work; none of them synchronises with the host.
 * - Calls return a status and never throw or abort.  Arguments are checked on
 *   the host before anything is enqueued.  On error nothing is enqueued and
 *   bi_last_error() describes the cause.
 * - M = 0 is a successful no-op (the grouped backward still zeroes dW).
 * - Row ids >= E are padding: they give +0 rows in Y and dX and add nothing
 *   to dW.  They are not an error.
 * - Scratch memory is taken from an engine-owned, stream-ordered memory pool
 *   and returned in stream order, so calls on different streams do not share
 *   scratch.
 * - A device-side wait that does not finish within the engine's limit stops
 *   the kernel, which records BI_ERR_TIMEOUT in the engine's status word;
 *   bi_engine_check() reports it.
 */
#ifndef BI_H
#define BI_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct bi_engine_s* bi_engine;

typedef enum { BI_F32 = 0, BI_BF16 = 1, BI_F16 = 2 } bi_dtype;

typedef enum {
    BI_OK = 0,
    BI_ERR_INVALID_ARG = 1, /* null pointer, K/N/E = 0, bad dtype, negative size */
    BI_ERR_MISALIGNED = 2,  /* tensor-core tier chosen but a pointer is not 16-byte aligned */
    BI_ERR_UNSUPPORTED = 3, /* sizes beyond the library's indexing limits */
    BI_ERR_CUDA = 4,        /* a CUDA runtime or launch error (never turned into a fallback) */
    BI_ERR_OOM = 5,         /* scratch allocation failed */
    BI_ERR_TIMEOUT = 6      /* a device-side pipeline wait ran out (see bi_engine_check) */
} bi_status;

/* Passes, as seen by the dispatcher. */
typedef enum {
    BI_PASS_FORWARD = 0, BI_PASS_DX = 1, BI_PASS_DW = 2,
    BI_PASS_GROUPED_FORWARD = 3, BI_PASS_GROUPED_DINPUT = 4, BI_PASS_GROUPED_DWEIGHTS = 5
} bi_pass;

/* Tier request of the segmented grouped calls.  Source: rublas 0.1.45
 * src/tensor_grouped/mod.rs, enum GroupedStrategy and fn
 * grouped_matmul_nt_backward_segmented_with_strategy: the scalar tier is the
 * default, Auto takes the tensor cores only where they are supported, and an
 * explicit tensor-core request that cannot be met is an error, not a fallback. */
typedef enum { BI_STRATEGY_SCALAR = 0, BI_STRATEGY_TENSOR_CORE = 1, BI_STRATEGY_AUTO = 2 } bi_strategy;

/* Rows per chunk of the dW reduction tree (scalar tier). */
#define BI_DW_CHUNK 256

/* Create an engine bound to CUDA device `device`.  Source: sgemm-bi 0.1.1.post2,
 * "Use" (Engine(0) is created once and owns the compiled kernels).  The engine
 * owns a memory pool for scratch, a device status word and an error string.
 * Errors: BI_ERR_INVALID_ARG (out == NULL), BI_ERR_CUDA (no such device). */
bi_status bi_engine_create(int device, bi_engine* out);

/* Destroy an engine.  The caller must make sure no work enqueued through it is
 * still running (synchronise its streams first).  NULL is a no-op. */
void bi_engine_destroy(bi_engine engine);

/* Text of the last error on this engine (engine != NULL) or of the last error
 * on this thread for calls made with engine == NULL.  Owned by the library,
 * valid until the next call on the same engine / thread. */
const char* bi_last_error(bi_engine engine);

/* Wait for `stream`, then read and clear the engine's device status word.
 * Returns BI_ERR_TIMEOUT if a kernel gave up a pipeline wait since the last
 * check, BI_ERR_CUDA on a CUDA error, BI_OK otherwise. */
bi_status bi_engine_check(bi_engine engine, void* stream);

/* Forward: y[M,N] = round( X[M,K] * W[K,N] + bias[N] ), bias nullable.
 * Source: sgemm-bi 0.1.1.post2, "Use" (Engine.forward(y, x, w, bias|None, m, k,
 * n, dtype, stream, tensor_cores)); ViperLLM ffma.py, _FFMAAddmm.forward (bias in
 * f32, then one cast).  y must not overlap x, w or bias. */
bi_status bi_forward(bi_engine engine, void* y, const void* x, const void* w, const void* bias,
                     int64_t m, int64_t k, int64_t n, bi_dtype dtype, void* stream, int tensor_cores);

/* Input gradient: dx[M,K] = round( dY[M,N] * W[K,N]^T ).
 * Source: ViperLLM ffma.py, _FFMAAddmm.backward (gx = gy W^T); sgemm-bi
 * 0.1.1.post2 intro (deterministic dX). */
bi_status bi_backward_dx(bi_engine engine, void* dx, const void* dy, const void* w,
                         int64_t m, int64_t k, int64_t n, bi_dtype dtype, void* stream, int tensor_cores);

/* Weight gradient: dw[K,N] = X[M,K]^T * dY[M,N], reduced over M by the fixed
 * chunk tree.  dw_f32 = 1 writes f32 (no rounding), 0 writes the operand type.
 * Source: ViperLLM ffma.py, _FFMAAddmm.backward (gW = x^T gy, cast back);
 * sgemm-bi 0.1.1.post2 "Use" (the weight gradient is accumulated in f32). */
bi_status bi_backward_dw(bi_engine engine, void* dw, int dw_f32, const void* x, const void* dy,
                         int64_t m, int64_t k, int64_t n, bi_dtype dtype, void* stream, int tensor_cores);

/* Bias gradient: db[N] = sum over rows of dY[M,N], in a fixed order: chunks of
 * BI_DW_CHUNK rows from row 0, f32 additions from +0 in row order inside a
 * chunk, the dW tree over chunk sums; db_f32 = 1 writes f32, 0 rounds once to
 * the operand type.  Bit-identical across runs.  Source: sgemm-bi 0.1.1.post2,
 * "Determinism contracts" (the page computes the bias gradient as an f32
 * column sum in torch, outside its engine; this is that sum in fixed order);
 * ViperLLM ffma.py, _FFMAAddmm.backward (gb = gy.sum(0)). */
bi_status bi_bias_grad(bi_engine engine, void* db, int db_f32, const void* dy, int64_t m, int64_t n,
                       bi_dtype dtype, void* stream);

/* ---- FP8 e4m3 per-tensor-scaled linear (tensor-core tier only) ---------
 * Source: AstrAI csrc/kernels/fp8_mm.cu (quantize_kernel; fp8_linear_forward_scaled
 * and fp8_linear_backward_scaled: operands quantized with 1/scale, the GEMM's
 * f32 product multiplied by the two scales).  e4m3 here is the "fn" format: no
 * infinities, largest finite 448, NaN 0x7F/0xFF. */

/* q[i] = e4m3( up(src[i]) * (*scale_inv) ): one f32 multiply, then round to
 * nearest even with saturation to +-448.  *amax = max |up(src[i])| over the
 * unscaled values (NaN ignored; +0 for count = 0); it is zeroed first, then
 * reduced with an exact, order-independent maximum, so it is bit-identical
 * run to run.  src has src_dtype; q, amax, scale_inv are device pointers. */
bi_status bi_fp8_quantize(bi_engine engine, uint8_t* q, float* amax, const void* src, const float* scale_inv,
                          int64_t count, bi_dtype src_dtype, void* stream);

/* y[M,N] = round( (chain_k xq[m,k] * wq[k,n]) * (*scale_x * *scale_w) + bias[n] ),
 * xq [M,K] and wq [K,N] e4m3 codes, f32 accumulation, the scale product and
 * the scaling each one f32 rounding, bias (nullable; out_dtype, bf16/f16 only)
 * added in f32, one rounding to out_dtype (bf16, f16 or f32).  tcgen05
 * kind::f8f6f4 on CTA pairs, fixed K order, no split: run-to-run and batch
 * invariant like the bf16 tensor-core tier.  k and n multiples of 16;
 * 16-byte aligned pointers. */
bi_status bi_fp8_forward(bi_engine engine, void* y, const uint8_t* xq, const uint8_t* wq, const void* bias,
                         const float* scale_x, const float* scale_w, int64_t m, int64_t k, int64_t n,
                         bi_dtype out_dtype, void* stream);

/* dx[M,K] = round( (chain_n gq[m,n] * wq[k,n]) * (*scale_g * *scale_w) ). */
bi_status bi_fp8_backward_dx(bi_engine engine, void* dx, const uint8_t* gq, const uint8_t* wq,
                             const float* scale_g, const float* scale_w, int64_t m, int64_t k, int64_t n,
                             bi_dtype out_dtype, void* stream);

/* dw[K,N] = round( (sum over m of xq[m,k] * gq[m,n]) * (*scale_x * *scale_g) ),
 * the rows chained in ascending order in the tensor-memory accumulator; m = 0
 * writes +0. */
bi_status bi_fp8_backward_dw(bi_engine engine, void* dw, const uint8_t* xq, const uint8_t* gq,
                             const float* scale_x, const float* scale_g, int64_t m, int64_t k, int64_t n,
                             bi_dtype out_dtype, void* stream);

/* Grouped forward: y[m,:] = round( X[m,:] * W[e(m)]^T ) with W [E,N,K] and
 * e(m) = row_experts[m]; rows with e(m) >= E are +0.  Rows need not be sorted.
 * Source: rublas 0.1.45 src/tensor_grouped/mod.rs, fn grouped_matmul_nt
 * (an id outside [0,E) marks a padding row whose output is all zeros;
 * f32 accumulation with a single rounding of the output). */
bi_status bi_grouped_forward(bi_engine engine, void* y, const void* x, const void* w,
                             const uint32_t* row_experts, int64_t m, int64_t k, int64_t n, int64_t e,
                             bi_dtype dtype, void* stream, int tensor_cores);

/* Grouped backward: dx[m,:] = round( dY[m,:] * W[e(m)] ) (+0 for padding rows)
 * and dw[e] (f32, [E,N,K]) = sum over the rows of expert e, in ascending row
 * index, of dY[m,:]^T X[m,:]; an expert with no rows gets +0.  dx may be NULL
 * to compute dw only.  Source: rublas 0.1.45 src/tensor_grouped/mod.rs,
 * struct GroupedBackward (the weight gradient is kept in f32) and fn
 * grouped_matmul_nt_backward_segmented_with_strategy (the segment offsets are
 * built inside the library here, from row_experts). */
bi_status bi_grouped_backward(bi_engine engine, void* dx, float* dw, const void* x, const void* w,
                              const void* dy, const uint32_t* row_experts,
                              int64_t m, int64_t k, int64_t n, int64_t e,
                              bi_dtype dtype, void* stream, int tensor_cores);

/* Segmented grouped forward: the caller's rows are already grouped by expert.
 * offsets [E+1] (u32, device) gives expert g the rows [offsets[g],
 * offsets[g+1]); rows from offsets[E] to m are padding (+0 output rows).  The
 * result equals bi_grouped_forward on row ids listing that grouping, bit for
 * bit on either tier.  strategy: see bi_strategy; BI_ERR_UNSUPPORTED when the
 * tensor cores are requested for a dtype or shape they cannot take.  The
 * offsets are read on the device and not validated on the host: a sequence
 * that does not start at 0, decreases or exceeds m is clamped into range
 * (no out-of-bounds access) and bi_engine_check() then reports
 * BI_ERR_INVALID_ARG.  Source: rublas 0.1.45 src/tensor_grouped/mod.rs, fn
 * grouped_matmul_nt_segmented and its offsets invariant. */
bi_status bi_grouped_forward_segmented(bi_engine engine, void* y, const void* x, const void* w,
                                       const uint32_t* offsets, int64_t m, int64_t k, int64_t n,
                                       int64_t e, bi_dtype dtype, void* stream, bi_strategy strategy);

/* Segmented grouped backward: dx (nullable) and dw [E,N,K] f32 for rows
 * grouped by offsets as in bi_grouped_forward_segmented.  With
 * BI_STRATEGY_TENSOR_CORE both passes must be able to use the tensor cores.
 * Source: rublas 0.1.45 src/tensor_grouped/mod.rs, fn
 * grouped_matmul_nt_backward_segmented_with_strategy. */
bi_status bi_grouped_backward_segmented(bi_engine engine, void* dx, float* dw, const void* x,
                                        const void* w, const void* dy, const uint32_t* offsets,
                                        int64_t m, int64_t k, int64_t n, int64_t e, bi_dtype dtype,
                                        void* stream, bi_strategy strategy);

/* Grouped forward that allocates nothing.  No counterpart on the pages: this
 * entry point exists for callers that cannot allocate GPU memory when they run
 * it (a memory-budgeted runtime whose allocator must not be bypassed, a plug-in
 * handed buffers but no allocation rights, a path that must never block on the
 * device heap).  It computes exactly what bi_grouped_forward computes with
 * tensor_cores = 0 (the scalar tier, bit for bit), on the current CUDA device,
 * without an engine, and calls no cudaMalloc, cudaFree or other allocating
 * routine.  Its grouping scratch lives in one fixed 4 MiB device array inside
 * the library, reserved on every GPU that loads the library until the process
 * exits; calls needing more than that (4*(2E+4) + 4*M + 4*(E+1)*ceil(M/256)
 * bytes, each part rounded up to 256) return BI_ERR_UNSUPPORTED.  All calls on a
 * device share the array: calls whose GPU work overlaps (unordered streams or
 * threads) race and give wrong results.  The first call on a device resolves
 * the array's address on that device; make it before any stream capture.  If
 * the device's context is destroyed and recreated (cudaDeviceReset), the next
 * call resolves the address again in the new context before launching.
 * Errors are reported through bi_last_error(NULL). */
bi_status bi_grouped_forward_noalloc(void* y, const void* x, const void* w,
                                     const uint32_t* row_experts, int64_t m, int64_t k, int64_t n,
                                     int64_t e, bi_dtype dtype, void* stream);

/* ---- introspection ---------------------------------------------------- */

/* The dispatcher's choice for a call: 0 = scalar tier, 1 = tensor-core tier.
 * A pure function of its arguments (M is not one of them).  Source:
 * sgemm-bi 0.1.1.post2, "Determinism contracts" (shapes with an output
 * dimension below 64 go to the scalar tier, decided from the shape alone).
 * Tensor cores take bf16/f16 with K, N multiples of 8, and f32 (3xTF32, the
 * dense passes only) with K, N multiples of 4; everything else is scalar. */
int bi_dispatch_tier(int pass, bi_dtype dtype, int tensor_cores, int64_t k, int64_t n);

/* Number of kernels this engine has launched since it was created. */
uint64_t bi_launch_count(bi_engine engine);

/* Force the column width of the tensor-core tier's output tiles (0 restores
 * the automatic choice, which depends on the pass, K and N only).  Source:
 * sgemm-bi 0.1.1.post2, "Determinism contracts" (the tensor-core tier has two
 * tile families that give bit-identical results).  Here the families are the
 * widths 256 and 128 for every 16-bit dense and grouped pass, plus 176 and 192
 * for the grouped forward; a width a pass cannot take is ignored for that
 * pass.  The width only decides how output elements are grouped into work
 * units: each element is the same ascending chain of 64-wide contraction blocks
 * in one f32 accumulator, so every result is bit-identical for every setting
 * (the tests compare them).  Meant for tests and tuning; cols outside
 * {0, 128, 176, 192, 256} is BI_ERR_INVALID_ARG. */
bi_status bi_engine_set_tile_cols(bi_engine engine, int cols);

/* Host-side fault injection for allocation failure (no counterpart on the
 * pages).  The next `count` scratch allocations of this engine fail as if its
 * memory pool were exhausted (count < 0: every allocation until the setting is
 * changed; 0: none).  A call whose scratch allocation fails returns BI_ERR_OOM
 * with nothing enqueued and its outputs untouched; the engine stays usable.
 * Calls that need no scratch are unaffected.  It lets callers and tests
 * exercise their out-of-memory handling without exhausting a GPU. */
bi_status bi_engine_fail_allocations(bi_engine engine, int64_t count);

/* Set the limit (nanoseconds) after which a device-side pipeline wait gives up
 * and records BI_ERR_TIMEOUT.  Default 2e9 (2 s); 0 restores the default. */
bi_status bi_engine_set_wait_limit(bi_engine engine, uint64_t nanoseconds);

/* Self-test of the timeout path: launches one kernel that waits on a barrier
 * nothing completes, bounded by the engine's wait limit.  Afterwards
 * bi_engine_check() must report BI_ERR_TIMEOUT.  Faults nothing. */
bi_status bi_selftest_wait_timeout(bi_engine engine, void* stream);

/* Library version string. */
const char* bi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* BI_H */
