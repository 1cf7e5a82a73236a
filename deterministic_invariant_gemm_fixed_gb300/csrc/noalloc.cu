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
// it together with the context it belongs to.  Make that first call before any
// stream capture begins.  If the device's context is later destroyed and
// recreated (cudaDeviceReset), the next call finds a different current context
// and looks the address up again before launching anything.
#include <cuda.h>

#include <mutex>

#include "bi_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;  // 4 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];
// Status word for the launchers (they may record a device-side condition);
// nothing in this entry point's kernels writes it today.
static __device__ __align__(16) int g_noalloc_status[4];

struct DeviceSlot {
    std::mutex mu;
    CUcontext ctx = nullptr;        // context the addresses below belong to
    void* scratch = nullptr;        // device address of g_noalloc_scratch on this device
    int* status = nullptr;          // device address of g_noalloc_status
    int sm_count = 0;
    bi_engine_s counters;           // launch counter only; owns no device memory
};

constexpr int kMaxDevices = 64;
DeviceSlot g_slots[kMaxDevices];

int64_t round256(int64_t b) { return (b + 255) / 256 * 256; }

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

CtxGetCurrentFn ctx_get_current() {
    static CtxGetCurrentFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(p);
    });
    return fn;
}

// Resolves (or re-resolves, after a context change) the device addresses of
// the fixed arrays for device `dev`, which is current.  Called with slot.mu held.
cudaError_t resolve(DeviceSlot& slot, int dev) {
    cudaError_t err = cudaSetDevice(dev);  // initialises the device's primary context if it has none yet
    if (err != cudaSuccess) return err;
    CtxGetCurrentFn get = ctx_get_current();
    if (!get) return cudaErrorNotSupported;
    CUcontext cur = nullptr;
    if (get(&cur) != CUDA_SUCCESS || cur == nullptr) return cudaErrorDeviceUninitialized;
    if (cur == slot.ctx && slot.scratch && slot.status) return cudaSuccess;
    slot.counters.device = dev;  // per-device kernel set-up is keyed on it
    void* sc = nullptr;
    void* st = nullptr;
    if ((err = cudaGetSymbolAddress(&sc, g_noalloc_scratch)) != cudaSuccess) return err;
    if ((err = cudaGetSymbolAddress(&st, g_noalloc_status)) != cudaSuccess) return err;
    if ((err = cudaDeviceGetAttribute(&slot.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return err;
    slot.scratch = sc;
    slot.status = static_cast<int*>(st);
    slot.ctx = cur;
    return cudaSuccess;
}

}  // namespace

extern "C" bi_status bi_grouped_forward_noalloc(void* y, const void* x, const void* w,
                                                const uint32_t* row_experts, int64_t m, int64_t k,
                                                int64_t n, int64_t e, bi_dtype dtype, void* stream) {
    // the same size limits as bi_grouped_forward
    const char* why = "";
    const bi_status size_st = bi::check_sizes(dtype, m, k, n, e < 0 ? 0 : e, &why);
    if (size_st != BI_OK) return bi::set_thread_error(size_st, std::string("bi_grouped_forward_noalloc: ") + why);
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
    void* scratch = nullptr;
    int* status = nullptr;
    {
        std::lock_guard<std::mutex> g(slot.mu);
        err = resolve(slot, dev);
        scratch = slot.scratch;
        status = slot.status;
    }
    if (err != cudaSuccess || !scratch)
        return bi::set_thread_error(BI_ERR_CUDA, std::string("scratch set-up failed: ") + cudaGetErrorName(err));

    const bi::LaunchCtx c{&slot.counters, static_cast<cudaStream_t>(stream), slot.sm_count, status,
                          slot.counters.wait_limit_ns};
    unsigned char* base = static_cast<unsigned char*>(scratch);
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
