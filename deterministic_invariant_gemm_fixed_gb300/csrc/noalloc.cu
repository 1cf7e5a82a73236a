// Grouped forward that allocates nothing, for callers that cannot allocate GPU memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine) at the point
// where they need the grouped forward: code running inside a memory-budgeted
// runtime whose allocator must not be bypassed, plug-ins that are handed
// buffers but no allocation rights, or paths that must never block on or
// fragment the device heap.  bi_grouped_forward (tensor_cores = 0) needs a
// little scratch for grouping rows by expert (the segment table, the row
// permutation and a per-block histogram) and takes it from the engine's memory
// pool.  bi_grouped_forward_noalloc computes the same result, bit for bit, with
// that scratch placed in one fixed device array that is part of the library's
// image: it is reserved on every GPU that loads the library and held until the
// process exits.  The caller still passes every input and output buffer.
//
// Limits: the scratch the call needs -- 4*(2E+4) + 4*M + 4*(E+1)*ceil(M/256)
// bytes, each part rounded up to 256 bytes -- must fit in 4 MiB (for example
// M up to 262,144 rows with E up to 510 experts).  Larger calls are rejected
// with BI_ERR_UNSUPPORTED before anything is enqueued.
//
// Sharing: every call on a device uses the same array, which keeps whatever
// the last call left in it.  Calls whose work overlaps on the GPU (different
// streams, or different host threads, without ordering between them) race on
// the array and give wrong results; order them on one stream.  The kernels
// rebuild every part of the scratch they read (the histogram is cleared by its
// own kernel), so nothing carries over from one ordered call to the next.
//
// Set-up: the first call on a device looks up the array's device address with
// cudaGetSymbolAddress (the host-side name of the array is only a stand-in and
// must never be passed to a kernel) while that device is current, and caches
// it.  Make that first call before any stream capture begins.
#include <mutex>

#include "bi_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;  // 4 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

struct DeviceSlot {
    std::once_flag once;
    void* scratch = nullptr;        // device address of g_noalloc_scratch on this device
    int sm_count = 0;
    cudaError_t err = cudaSuccess;
    bi_engine_s counters;           // launch counter only; owns no device memory
};

constexpr int kMaxDevices = 64;
DeviceSlot g_slots[kMaxDevices];

int64_t round256(int64_t b) { return (b + 255) / 256 * 256; }

}  // namespace

extern "C" bi_status bi_grouped_forward_noalloc(void* y, const void* x, const void* w,
                                                const uint32_t* row_experts, int64_t m, int64_t k,
                                                int64_t n, int64_t e, bi_dtype dtype, void* stream) {
    if (dtype != BI_F32 && dtype != BI_BF16 && dtype != BI_F16)
        return bi::set_thread_error(BI_ERR_INVALID_ARG, "dtype must be BI_F32, BI_BF16 or BI_F16");
    if (m < 0 || k <= 0 || n <= 0 || e <= 0)
        return bi::set_thread_error(BI_ERR_INVALID_ARG, "need m >= 0 and k, n, e > 0");
    const uint64_t lim = 0xffffffffull;
    if (uint64_t(m) * uint64_t(k) > lim || uint64_t(m) * uint64_t(n) > lim ||
        uint64_t(e) * uint64_t(n) * uint64_t(k) > lim || e > 65535 || n > int64_t(65535) * 128)
        return bi::set_thread_error(BI_ERR_UNSUPPORTED, "grouped matmul exceeds U32 indexing");
    if (m == 0) return BI_OK;
    if (!y || !x || !w || !row_experts)
        return bi::set_thread_error(BI_ERR_INVALID_ARG, "y, x, w and row_experts must not be NULL");
    const int64_t seg_b = round256(bi::seg_table_len(e) * 4);
    const int64_t perm_b = round256(m * 4);
    const int64_t hist_b = round256(bi::segment_scratch_bytes(m, e));
    const int64_t need = seg_b + perm_b + hist_b;
    if (need > int64_t(kNoAllocScratchBytes))
        return bi::set_thread_error(
            BI_ERR_UNSUPPORTED,
            "bi_grouped_forward_noalloc: this call needs " + std::to_string(need) +
                " bytes of scratch; the fixed array holds 4194304 (use bi_grouped_forward)");

    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return bi::set_thread_error(BI_ERR_CUDA, "cudaGetDevice failed");
    if (dev < 0 || dev >= kMaxDevices)
        return bi::set_thread_error(BI_ERR_UNSUPPORTED, "device ordinal beyond 63");
    DeviceSlot& slot = g_slots[dev];
    std::call_once(slot.once, [&slot, dev] {
        // the current device is `dev`: resolve the array's address on it
        slot.counters.device = dev;  // per-device kernel set-up is keyed on it
        slot.err = cudaGetSymbolAddress(&slot.scratch, g_noalloc_scratch);
        if (slot.err == cudaSuccess)
            slot.err = cudaDeviceGetAttribute(&slot.sm_count, cudaDevAttrMultiProcessorCount, dev);
    });
    if (slot.err != cudaSuccess || !slot.scratch)
        return bi::set_thread_error(BI_ERR_CUDA, std::string("scratch set-up failed: ") +
                                                     cudaGetErrorName(slot.err));

    const bi::LaunchCtx c{&slot.counters, static_cast<cudaStream_t>(stream), slot.sm_count, nullptr,
                          slot.counters.wait_limit_ns};
    unsigned char* base = static_cast<unsigned char*>(slot.scratch);
    uint32_t* seg = reinterpret_cast<uint32_t*>(base);
    uint32_t* perm = reinterpret_cast<uint32_t*>(base + seg_b);
    void* hist = base + seg_b + perm_b;
    err = bi::segment(c, row_experts, m, e, seg, perm, hist);
    if (err == cudaSuccess) err = bi::scalar_rows_grouped(c, dtype, y, x, w, m, k, n, e, 1, seg, perm);
    if (err == cudaSuccess)
        err = bi::zero_padding_rows(c, y, n, dtype == BI_F32 ? 4 : 2, e, seg, perm);
    if (err != cudaSuccess)
        return bi::set_thread_error(BI_ERR_CUDA, std::string("bi_grouped_forward_noalloc: ") +
                                                     cudaGetErrorName(err));
    return BI_OK;
}
