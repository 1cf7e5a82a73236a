// Internal declarations shared by the translation units of libbi (not installed).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>
#include <string>

#include "bi.h"

struct bi_engine_s {
    int device = 0;
    int sm_count = 0;
    cudaMemPool_t pool = nullptr;
    int* d_status = nullptr;               // device status word (0 = fine)
    uint64_t wait_limit_ns = 2000000000ull; // bounded device-side waits
    cudaStream_t side = nullptr;            // engine-owned stream for independent work within a call
    std::atomic<uint64_t> launches{0};
    std::atomic<int64_t> failing_allocs{0}; // injected scratch-allocation failures still to give (-1 = all)
    int tile_cols = 0;                      // forced tensor-core column tile (0 = chosen from the shape)
    std::mutex mu;                          // guards last_error
    std::string last_error;
};

namespace bi {

// Status codes written by kernels into the engine's status word.
enum DeviceStatus : int { DEV_OK = 0, DEV_TIMEOUT_PRODUCER = 1, DEV_TIMEOUT_MMA = 2,
                          DEV_TIMEOUT_EPILOGUE = 3, DEV_TIMEOUT_SELFTEST = 4,
                          DEV_BAD_OFFSETS = 5 };

// One-time setup per device (kernel attributes and occupancy queries belong to
// a device): value and status of the first call on each device, kept per
// instantiation of the caller's static.
constexpr int MAX_DEVICES = 64;
struct PerDeviceOnce {
    std::once_flag once[MAX_DEVICES];
    cudaError_t err[MAX_DEVICES] = {};
    int value[MAX_DEVICES] = {};
    template <typename F>  // F(int& value) -> cudaError_t
    cudaError_t run(int device, F&& f) {
        if (device < 0 || device >= MAX_DEVICES) return cudaErrorInvalidDevice;
        std::call_once(once[device], [&] { err[device] = f(value[device]); });
        return err[device];
    }
};

// Programmatic dependent launch: a kernel launched with launch_pdl may be
// scheduled while the previous kernel in its stream is still finishing.  It
// must call grid_dep_wait() before touching global memory (that waits for the
// previous kernel to complete and its writes to be visible); grid_dep_launch()
// lets the kernel after it be scheduled early in turn.  Both are no-ops for a
// kernel launched the ordinary way.
#ifdef __CUDACC__
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
#endif
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Everything a kernel launcher needs from the engine.
struct LaunchCtx {
    bi_engine eng;
    cudaStream_t stream;
    int sm_count;
    int* status;
    uint64_t wait_limit_ns;
    void count(uint64_t n = 1) const { eng->launches.fetch_add(n, std::memory_order_relaxed); }
};

// ---- scalar tier (scalar.cu) ---------------------------------------------
// "rows" kernels: out[r, c] = down( chain_l A[r, l] * B(l, c) (+ bias[c]) ), A
// contraction-contiguous [R, L]; B is [L, C] (b_contr_contig = 0) or [C, L] (1).
// Grouped: rows come from expert segments (seg/perm), B advanced by expert.
cudaError_t scalar_rows(const LaunchCtx& c, bi_dtype dt, void* out, const void* a, const void* b,
                        const void* bias, int64_t R, int64_t L, int64_t C, int b_contr_contig);
cudaError_t scalar_rows_grouped(const LaunchCtx& c, bi_dtype dt, void* out, const void* a,
                                const void* b, int64_t M, int64_t L, int64_t C, int64_t E,
                                int b_contr_contig, const uint32_t* seg, const uint32_t* perm);
// dW kernels: out[r, c] = tree over chunks of chain over rows m of A[m, r] * B[m, c].
// partials: workspace of J*R*C floats (may be null when J == 1).
cudaError_t scalar_dw(const LaunchCtx& c, bi_dtype dt, void* out, int out_f32, const void* a,
                      const void* b, int64_t M, int64_t R, int64_t C, float* partials);
cudaError_t scalar_dw_grouped(const LaunchCtx& c, bi_dtype dt, float* out, const void* a,
                              const void* b, int64_t M, int64_t R, int64_t C, int64_t E,
                              const uint32_t* seg, const uint32_t* perm, float* partials,
                              int64_t max_chunks);

// Bias gradient: out[N] = column sums of dY [M, N] in the dW chunk/tree order.
// partials: J*N floats (J = ceil(M/256)); may be null when J == 1.
cudaError_t bias_grad(const LaunchCtx& c, bi_dtype dt, void* out, int out_f32, const void* dy,
                      int64_t M, int64_t N, float* partials);

// ---- grouping (grouped.cu) ------------------------------------------------
// The tensor-core grouped passes cut each expert's sorted rows into tiles of
// GROUPED_TILE_ROWS rows, and read the expert's partial last block of
// GROUPED_TAIL_ROWS rows (dweights) from a zero-padded tail buffer.
constexpr int GROUPED_TILE_ROWS = 256;
constexpr int GROUPED_TAIL_ROWS = 64;
// Segment table layout (u32): [0, E+2) sorted offsets of groups 0..E (group E
// = padding) plus M; [E+2, 2E+3) first tile of experts 0..E, a prefix sum of
// ceil(count / GROUPED_TILE_ROWS) (entry E = all tiles); then the same total
// once more.
inline int64_t seg_table_len(int64_t E) { return 2 * E + 4; }
int64_t segment_scratch_bytes(int64_t M, int64_t E);
cudaError_t segment(const LaunchCtx& c, const uint32_t* ids, int64_t M, int64_t E, uint32_t* seg,
                    uint32_t* perm, void* scratch);
// The same table from caller offsets [E+1] (rows already grouped); the
// permutation is the identity.  Offsets are clamped into a nondecreasing
// sequence from 0 to at most M; a clamp records DEV_BAD_OFFSETS.
cudaError_t segment_from_offsets(const LaunchCtx& c, const uint32_t* offsets, int64_t M, int64_t E,
                                 uint32_t* seg, uint32_t* perm);
// 16-bit rows of length L (a multiple of 8).  gather_sorted: dst[s] = src[perm[s]]
// for the sorted rows of experts 0..E-1 (s < offsets[E]).  build_tails: for each
// expert g, rows [g*64, g*64+64) of dst hold its sorted rows from the last
// multiple of 64 on, then zeros.
// zero_out (nullable): an output [M, zero_C] (16-bit, zero_C a multiple of 8)
// whose padding rows are zeroed in the same launch.
cudaError_t gather_sorted(const LaunchCtx& c, const void* src, int64_t M, int64_t L, int64_t E,
                          const uint32_t* seg, const uint32_t* perm, void* dst, void* zero_out = nullptr,
                          int64_t zero_C = 0);
cudaError_t build_tails(const LaunchCtx& c, const void* src, int64_t L, int64_t E, const uint32_t* seg,
                        const uint32_t* perm, void* dst);
// Zero the rows of out [M, C] (element size esize) whose ids are padding.
cudaError_t zero_padding_rows(const LaunchCtx& c, void* out, int64_t C, int esize, int64_t E,
                              const uint32_t* seg, const uint32_t* perm);
cudaError_t selftest_wait(const LaunchCtx& c);

// ---- tensor-core tier (tc.cu) ----------------------------------------------
cudaError_t tc_forward(const LaunchCtx& c, bi_dtype dt, void* y, const void* x, const void* w,
                       const void* bias, int64_t M, int64_t K, int64_t N);
cudaError_t tc_dx(const LaunchCtx& c, bi_dtype dt, void* dx, const void* dy, const void* w,
                  int64_t M, int64_t K, int64_t N);
// dW: the output tiles of the last, partial wave run their contraction in
// chunks added by the dW tree; ws holds their f32 results (tc_dw_workspace_bytes,
// 0 = no split for this shape, ws may be null).
int64_t tc_dw_workspace_bytes(const LaunchCtx& c, int dw_f32, int64_t M, int64_t K, int64_t N);
cudaError_t tc_dw(const LaunchCtx& c, bi_dtype dt, void* dw, int dw_f32, const void* x,
                  const void* dy, int64_t M, int64_t K, int64_t N, float* ws);
// Grouped forward / dinput on a row-sorted operand a_sorted [M, K or N] (row
// s = original row perm[s]); output row perm[s] for every sorted row of an expert.
cudaError_t tc_grouped_rows(const LaunchCtx& c, bi_dtype dt, int pass_dinput, void* out, const void* a_sorted,
                            const void* w, int64_t M, int64_t K, int64_t N, int64_t E, const uint32_t* seg,
                            const uint32_t* perm);
// Grouped dweights [E,N,K] f32 from row-sorted dY and X plus their tail buffers.
// The units of the last partial wave contract in chunks summed by the dW tree;
// ws holds their f32 results (tc_grouped_dw_workspace_bytes; 0 = no split).
int64_t tc_grouped_dw_workspace_bytes(int64_t M, int64_t K, int64_t N, int64_t E);
cudaError_t tc_grouped_dw(const LaunchCtx& c, bi_dtype dt, float* dw, const void* dy_sorted, const void* x_sorted,
                          const void* dy_tail, const void* x_tail, int64_t M, int64_t K, int64_t N, int64_t E,
                          const uint32_t* seg, float* ws);
// FP8 e4m3 scaled matmuls on the CTA pair (pass 0 forward, 1 dX, 2 dW): the
// f32 product is multiplied by *sa * *sb, then (+ bias), then rounded to out_dt.
// The dW splits its last wave of tiles as tc_dw does (ws: tc_fp8_dw_workspace_bytes).
int64_t tc_fp8_dw_workspace_bytes(int out_f32, int64_t M, int64_t K, int64_t N);
cudaError_t tc_fp8_pass(const LaunchCtx& c, int pass, bi_dtype out_dt, void* out, const uint8_t* a,
                        const uint8_t* b, const void* bias, const float* sa, const float* sb, int64_t M,
                        int64_t K, int64_t N, float* ws);
// 3xTF32 (f32 operands on the tensor cores, tf32.cu and tc.cu).
// tf32_split: x [rows][cols] row-major into TF32 parts hi, lo.  Without transpose
// they keep x's layout; with transpose they are [cols][ld] (ld >= rows, a
// multiple of 4; the columns past rows are not written).
cudaError_t tf32_split(const LaunchCtx& c, const float* x, float* hi, float* lo, int64_t rows, int64_t cols,
                       bool transpose, int64_t ld);
// Contractions longer than this many elements run as pieces of this length, one
// launch each, every launch after the first adding its result to the output in
// piece order: the tensor core's accumulation error grows with the contraction
// length, and a fixed piece length (independent of the batch) bounds it.
constexpr int64_t TF32X3_PIECE = 4096;
// The same for the 16-bit and FP8 tensor-core passes whose result stays f32
// (dW with dw_f32, the FP8 dW in f32, the grouped dweights): contractions over
// more rows than this run in pieces of this many rows, summed in order in dW.
constexpr int64_t TC_PIECE_ROWS = 8192;
// out[r][c] = sum over pieces (in order) of the piece's sum over d of
// a[r][d] * b[c][d], + bias[c]; both operands K-major (a: rows x depth, leading
// dim lda; b: cols x depth, ldb); f32 out, leading dim ldo.
cudaError_t tc_tf32x3_pass(const LaunchCtx& c, const float* a_hi, const float* a_lo, int64_t lda,
                           const float* b_hi, const float* b_lo, int64_t ldb, float* out, int64_t ldo,
                           const float* bias, int64_t rows, int64_t cols, int64_t depth);
// FP8 quantize (fp8.cu): q = e4m3(up(src) * *scale_inv), amax = max |up(src)|.
cudaError_t fp8_quantize(const LaunchCtx& c, bi_dtype dt, uint8_t* q, float* amax, const void* src,
                         const float* scale_inv, int64_t count);

}  // namespace bi

namespace bi {
// Size limits every matmul entry point applies before it enqueues anything:
// BI_ERR_INVALID_ARG for a bad dtype, m < 0 or k, n <= 0 (e <= 0 for the
// grouped calls, e < 0 means "not grouped"), BI_ERR_UNSUPPORTED for sizes
// beyond the kernels' indexing (2^31 - 1 per dimension, k and n at most
// 8388480, e at most 65535, the grouped calls' U32 element counts).  Returns
// BI_OK or the status, with the reason in *why.
bi_status check_sizes(bi_dtype dt, int64_t m, int64_t k, int64_t n, int64_t e, const char** why);
// Records `msg` as this thread's last error (bi_last_error(NULL)) and returns st.
bi_status set_thread_error(bi_status st, const std::string& msg);
__host__ __device__ __forceinline__ int64_t lmin(int64_t a, int64_t b) { return a < b ? a : b; }
__host__ __device__ __forceinline__ int64_t lmax(int64_t a, int64_t b) { return a > b ? a : b; }
}  // namespace bi
