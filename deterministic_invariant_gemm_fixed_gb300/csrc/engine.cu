// C ABI of libbi: argument validation, shape-only dispatch, scratch memory and
// kernel orchestration.  See include/bi.h for the contract of every entry point.
#include <cstdio>
#include <cstring>
#include <new>
#include <string>

#include "bi_internal.h"

namespace {

thread_local std::string tl_error;

// Record an error on the engine (or on the calling thread) and return `st`.
bi_status fail(bi_engine eng, bi_status st, const std::string& msg) {
    if (eng) {
        std::lock_guard<std::mutex> g(eng->mu);
        eng->last_error = msg;
    } else {
        tl_error = msg;
    }
    return st;
}

bi_status cuda_fail(bi_engine eng, cudaError_t e, const char* where) {
    return fail(eng, e == cudaErrorMemoryAllocation ? BI_ERR_OOM : BI_ERR_CUDA,
                std::string(where) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")");
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t dsize(bi_dtype dt) { return dt == BI_F32 ? 4 : 2; }

// Makes the engine's device current for the duration of a call, then restores.
struct DeviceGuard {
    int prev = -1;
    bool ok = true;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
        if (prev != dev) ok = cudaSetDevice(dev) == cudaSuccess;
    }
    ~DeviceGuard() {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

// Stream-ordered scratch from the engine's pool, released in stream order.
struct Scratch {
    bi_engine eng;
    cudaStream_t stream;
    void* ptr = nullptr;
    cudaError_t err = cudaSuccess;
    Scratch(bi_engine e, cudaStream_t s, size_t bytes) : eng(e), stream(s) {
        if (!bytes) return;
        if (take_injected_failure(e)) {  // bi_engine_fail_allocations: fail as an exhausted pool would
            err = cudaErrorMemoryAllocation;
            return;
        }
        err = cudaMallocFromPoolAsync(&ptr, bytes, e->pool, s);
    }
    static bool take_injected_failure(bi_engine e) {
        int64_t v = e->failing_allocs.load();
        while (v != 0) {
            if (v < 0) return true;
            if (e->failing_allocs.compare_exchange_weak(v, v - 1)) return true;
        }
        return false;
    }
    ~Scratch() {
        if (ptr) cudaFreeAsync(ptr, stream);
    }
};

const int64_t kMaxDim = (int64_t(1) << 31) - 1;

bi_status check_common(bi_engine eng, bi_dtype dt, int64_t m, int64_t k, int64_t n) {
    if (!eng) return fail(nullptr, BI_ERR_INVALID_ARG, "engine is NULL");
    const char* why = "";
    const bi_status st = bi::check_sizes(dt, m, k, n, -1, &why);
    return st == BI_OK ? BI_OK : fail(eng, st, why);
}

bi::LaunchCtx ctx(bi_engine eng, void* stream) {
    return bi::LaunchCtx{eng, static_cast<cudaStream_t>(stream), eng->sm_count, eng->d_status,
                         eng->wait_limit_ns};
}

// f32 operands on the tensor cores (3xTF32).  Each operand is a row-major
// [rows][cols] f32 matrix; `transpose` says its contraction index runs down the
// columns, so the split writes its TF32 parts transposed, rows padded to a
// multiple of 4 (16-byte TMA strides at any batch size).  The pair kernel then
// reads both operands K-major from stream-ordered scratch.
struct Tf32Operand {
    const void* src;
    int64_t rows, cols;
    bool transpose;
    int64_t ld() const { return transpose ? (rows + 3) / 4 * 4 : cols; }
    int64_t bytes() const { return ((transpose ? cols : rows) * ld() * 4 + 255) / 256 * 256; }
};

bi_status tf32x3(bi_engine eng, const bi::LaunchCtx& c, const Tf32Operand& a, const Tf32Operand& b, void* out,
                 int64_t ldo, const void* bias, int64_t rows, int64_t cols, int64_t depth, const char* name) {
    const int64_t a_b = a.bytes(), b_b = b.bytes();
    Scratch sc(eng, c.stream, static_cast<size_t>(2 * (a_b + b_b)));
    if (sc.err != cudaSuccess) return cuda_fail(eng, sc.err, "3xTF32 scratch");
    uint8_t* base = static_cast<uint8_t*>(sc.ptr);
    float* ah = reinterpret_cast<float*>(base);
    float* al = reinterpret_cast<float*>(base + a_b);
    float* bh = reinterpret_cast<float*>(base + 2 * a_b);
    float* bl = reinterpret_cast<float*>(base + 2 * a_b + b_b);
    cudaError_t e = bi::tf32_split(c, static_cast<const float*>(a.src), ah, al, a.rows, a.cols, a.transpose, a.ld());
    if (e == cudaSuccess)
        e = bi::tf32_split(c, static_cast<const float*>(b.src), bh, bl, b.rows, b.cols, b.transpose, b.ld());
    if (e == cudaSuccess)
        e = bi::tc_tf32x3_pass(c, ah, al, a.ld(), bh, bl, b.ld(), static_cast<float*>(out), ldo,
                               static_cast<const float*>(bias), rows, cols, depth);
    return e == cudaSuccess ? BI_OK : cuda_fail(eng, e, name);
}

}  // namespace

namespace bi {
bi_status set_thread_error(bi_status st, const std::string& msg) { return fail(nullptr, st, msg); }

bi_status check_sizes(bi_dtype dt, int64_t m, int64_t k, int64_t n, int64_t e, const char** why) {
    if (dt != BI_F32 && dt != BI_BF16 && dt != BI_F16) {
        *why = "dtype must be BI_F32, BI_BF16 or BI_F16";
        return BI_ERR_INVALID_ARG;
    }
    if (m < 0) { *why = "m must be >= 0"; return BI_ERR_INVALID_ARG; }
    if (k <= 0 || n <= 0) { *why = "k and n must be > 0"; return BI_ERR_INVALID_ARG; }
    if (m > kMaxDim || k > kMaxDim || n > kMaxDim) { *why = "a dimension exceeds 2^31 - 1"; return BI_ERR_UNSUPPORTED; }
    if (n > int64_t(65535) * 128 || k > int64_t(65535) * 128) {
        *why = "k and n are limited to 8388480";
        return BI_ERR_UNSUPPORTED;
    }
    if (e < 0) return BI_OK;  // not a grouped call
    if (e == 0) { *why = "e must be > 0"; return BI_ERR_INVALID_ARG; }
    if (e > 65535) { *why = "e is limited to 65535 experts"; return BI_ERR_UNSUPPORTED; }
    // the same U32 indexing limits as the grouped matmul of rublas (GroupedMatmulError)
    const uint64_t lim = 0xffffffffull;
    if (uint64_t(m) * uint64_t(k) > lim || uint64_t(m) * uint64_t(n) > lim ||
        uint64_t(e) * uint64_t(n) * uint64_t(k) > lim) {
        *why = "grouped matmul exceeds U32 indexing";
        return BI_ERR_UNSUPPORTED;
    }
    return BI_OK;
}
}  // namespace bi

extern "C" {

const char* bi_version(void) { return "bi 0.1.0 (sm_103a)"; }

int bi_dispatch_tier(int pass, bi_dtype dtype, int tensor_cores, int64_t k, int64_t n) {
    if (!tensor_cores) return 0;
    if (dtype != BI_BF16 && dtype != BI_F16 && dtype != BI_F32) return 0;
    // f32 operands reach the tensor cores through the 3xTF32 split, dense passes only
    const bool f32 = dtype == BI_F32;
    if (f32 && pass > BI_PASS_DW) return 0;
    const int64_t unit = f32 ? 4 : 8;  // elements per 16-byte row unit, for TMA
    if (k <= 0 || n <= 0 || k % unit != 0 || n % unit != 0) return 0;
    switch (pass) {
        case BI_PASS_FORWARD:
        case BI_PASS_GROUPED_FORWARD: return n >= 64 ? 1 : 0;
        case BI_PASS_DX:
        case BI_PASS_GROUPED_DINPUT: return k >= 64 ? 1 : 0;
        case BI_PASS_DW:
        case BI_PASS_GROUPED_DWEIGHTS: return (k >= 64 && n >= 64) ? 1 : 0;
        default: return 0;
    }
}

bi_status bi_engine_create(int device, bi_engine* out) {
    if (!out) return fail(nullptr, BI_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    int count = 0;
    cudaError_t e = cudaGetDeviceCount(&count);
    if (e != cudaSuccess) return cuda_fail(nullptr, e, "cudaGetDeviceCount");
    if (device < 0 || device >= count) return fail(nullptr, BI_ERR_CUDA, "no such CUDA device");
    bi_engine eng = new (std::nothrow) bi_engine_s();
    if (!eng) return fail(nullptr, BI_ERR_OOM, "engine allocation failed");
    eng->device = device;
    DeviceGuard g(device);
    if (!g.ok) { delete eng; return fail(nullptr, BI_ERR_CUDA, "cudaSetDevice failed"); }
    if ((e = cudaDeviceGetAttribute(&eng->sm_count, cudaDevAttrMultiProcessorCount, device)) != cudaSuccess) {
        delete eng;
        return cuda_fail(nullptr, e, "cudaDeviceGetAttribute");
    }
    cudaMemPoolProps props{};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = device;
    if ((e = cudaMemPoolCreate(&eng->pool, &props)) != cudaSuccess) {
        delete eng;
        return cuda_fail(nullptr, e, "cudaMemPoolCreate");
    }
    uint64_t keep = ~uint64_t(0);  // keep freed scratch cached in the pool
    cudaMemPoolSetAttribute(eng->pool, cudaMemPoolAttrReleaseThreshold, &keep);
    if ((e = cudaStreamCreateWithFlags(&eng->side, cudaStreamNonBlocking)) != cudaSuccess) {
        cudaMemPoolDestroy(eng->pool);
        delete eng;
        return cuda_fail(nullptr, e, "cudaStreamCreateWithFlags");
    }
    if ((e = cudaMalloc(&eng->d_status, 16)) != cudaSuccess ||
        (e = cudaMemset(eng->d_status, 0, 16)) != cudaSuccess) {
        cudaMemPoolDestroy(eng->pool);
        delete eng;
        return cuda_fail(nullptr, e, "status word");
    }
    *out = eng;
    return BI_OK;
}

void bi_engine_destroy(bi_engine eng) {
    if (!eng) return;
    {
        DeviceGuard g(eng->device);
        if (eng->side) cudaStreamDestroy(eng->side);
        cudaFree(eng->d_status);
        cudaMemPoolDestroy(eng->pool);
    }
    delete eng;
}

const char* bi_last_error(bi_engine eng) {
    if (!eng) return tl_error.c_str();
    std::lock_guard<std::mutex> g(eng->mu);
    return eng->last_error.c_str();
}

uint64_t bi_launch_count(bi_engine eng) { return eng ? eng->launches.load() : 0; }

bi_status bi_engine_fail_allocations(bi_engine eng, int64_t count) {
    if (!eng) return fail(nullptr, BI_ERR_INVALID_ARG, "engine is NULL");
    eng->failing_allocs.store(count < 0 ? -1 : count);
    return BI_OK;
}

bi_status bi_engine_set_tile_cols(bi_engine eng, int cols) {
    if (!eng) return fail(nullptr, BI_ERR_INVALID_ARG, "engine is NULL");
    if (cols != 0 && cols != 128 && cols != 176 && cols != 192 && cols != 256)
        return fail(eng, BI_ERR_INVALID_ARG, "tile columns must be 0 (automatic), 128, 176, 192 or 256");
    eng->tile_cols = cols;
    return BI_OK;
}

bi_status bi_engine_set_wait_limit(bi_engine eng, uint64_t ns) {
    if (!eng) return fail(nullptr, BI_ERR_INVALID_ARG, "engine is NULL");
    eng->wait_limit_ns = ns ? ns : 2000000000ull;
    return BI_OK;
}

bi_status bi_engine_check(bi_engine eng, void* stream) {
    if (!eng) return fail(nullptr, BI_ERR_INVALID_ARG, "engine is NULL");
    DeviceGuard g(eng->device);
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(eng, e, "cudaStreamSynchronize");
    int v = 0;
    if ((e = cudaMemcpy(&v, eng->d_status, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess)
        return cuda_fail(eng, e, "reading the status word");
    if (v != 0) {
        cudaMemset(eng->d_status, 0, sizeof(int));
        if (v == bi::DEV_BAD_OFFSETS)
            return fail(eng, BI_ERR_INVALID_ARG,
                        "segment offsets were not nondecreasing from 0 to at most m; they were clamped");
        static const char* who[] = {"", "TMA producer", "MMA issuer", "epilogue", "self-test"};
        return fail(eng, BI_ERR_TIMEOUT,
                    std::string("a device pipeline wait ran out (") + (v > 0 && v < 5 ? who[v] : "unknown") + ")");
    }
    return BI_OK;
}

bi_status bi_selftest_wait_timeout(bi_engine eng, void* stream) {
    if (!eng) return fail(nullptr, BI_ERR_INVALID_ARG, "engine is NULL");
    DeviceGuard g(eng->device);
    cudaError_t e = bi::selftest_wait(ctx(eng, stream));
    return e == cudaSuccess ? BI_OK : cuda_fail(eng, e, "self-test launch");
}

bi_status bi_forward(bi_engine eng, void* y, const void* x, const void* w, const void* bias,
                     int64_t m, int64_t k, int64_t n, bi_dtype dtype, void* stream, int tensor_cores) {
    bi_status st = check_common(eng, dtype, m, k, n);
    if (st != BI_OK) return st;
    if (m == 0) return BI_OK;
    if (!y || !x || !w) return fail(eng, BI_ERR_INVALID_ARG, "y, x and w must not be NULL");
    const int tier = bi_dispatch_tier(BI_PASS_FORWARD, dtype, tensor_cores, k, n);
    if (tier && (!aligned16(y) || !aligned16(x) || !aligned16(w)))
        return fail(eng, BI_ERR_MISALIGNED, "tensor-core tier needs 16-byte aligned y, x, w");
    DeviceGuard g(eng->device);
    if (!g.ok) return fail(eng, BI_ERR_CUDA, "cudaSetDevice failed");
    const bi::LaunchCtx c = ctx(eng, stream);
    if (tier && dtype == BI_F32)  // y = x w: x K-major as stored, w transposed
        return tf32x3(eng, c, {x, m, k, false}, {w, k, n, true}, y, n, bias, m, n, k, "bi_forward");
    cudaError_t e = tier ? bi::tc_forward(c, dtype, y, x, w, bias, m, k, n)
                         : bi::scalar_rows(c, dtype, y, x, w, bias, m, k, n, 0);
    return e == cudaSuccess ? BI_OK : cuda_fail(eng, e, "bi_forward");
}

bi_status bi_backward_dx(bi_engine eng, void* dx, const void* dy, const void* w, int64_t m,
                         int64_t k, int64_t n, bi_dtype dtype, void* stream, int tensor_cores) {
    bi_status st = check_common(eng, dtype, m, k, n);
    if (st != BI_OK) return st;
    if (m == 0) return BI_OK;
    if (!dx || !dy || !w) return fail(eng, BI_ERR_INVALID_ARG, "dx, dy and w must not be NULL");
    const int tier = bi_dispatch_tier(BI_PASS_DX, dtype, tensor_cores, k, n);
    if (tier && (!aligned16(dx) || !aligned16(dy) || !aligned16(w)))
        return fail(eng, BI_ERR_MISALIGNED, "tensor-core tier needs 16-byte aligned dx, dy, w");
    DeviceGuard g(eng->device);
    if (!g.ok) return fail(eng, BI_ERR_CUDA, "cudaSetDevice failed");
    const bi::LaunchCtx c = ctx(eng, stream);
    if (tier && dtype == BI_F32)  // dx = dy w^T: both K-major as stored
        return tf32x3(eng, c, {dy, m, n, false}, {w, k, n, false}, dx, k, nullptr, m, k, n, "bi_backward_dx");
    cudaError_t e = tier ? bi::tc_dx(c, dtype, dx, dy, w, m, k, n)
                         : bi::scalar_rows(c, dtype, dx, dy, w, nullptr, m, n, k, 1);
    return e == cudaSuccess ? BI_OK : cuda_fail(eng, e, "bi_backward_dx");
}

bi_status bi_backward_dw(bi_engine eng, void* dw, int dw_f32, const void* x, const void* dy,
                         int64_t m, int64_t k, int64_t n, bi_dtype dtype, void* stream, int tensor_cores) {
    bi_status st = check_common(eng, dtype, m, k, n);
    if (st != BI_OK) return st;
    if (!dw) return fail(eng, BI_ERR_INVALID_ARG, "dw must not be NULL");
    if (m > 0 && (!x || !dy)) return fail(eng, BI_ERR_INVALID_ARG, "x and dy must not be NULL");
    const int64_t J = (m + BI_DW_CHUNK - 1) / BI_DW_CHUNK;
    const int out_f32 = dw_f32 || dtype == BI_F32;
    const int tier = bi_dispatch_tier(BI_PASS_DW, dtype, tensor_cores, k, n);
    if (tier && m > 0 && (!aligned16(dw) || !aligned16(x) || !aligned16(dy)))
        return fail(eng, BI_ERR_MISALIGNED, "tensor-core tier needs 16-byte aligned dw, x, dy");
    DeviceGuard g(eng->device);
    if (!g.ok) return fail(eng, BI_ERR_CUDA, "cudaSetDevice failed");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (m == 0) {  // empty sum: +0
        cudaError_t e = cudaMemsetAsync(dw, 0, static_cast<size_t>(k * n * (out_f32 ? 4 : dsize(dtype))), s);
        return e == cudaSuccess ? BI_OK : cuda_fail(eng, e, "bi_backward_dw");
    }
    const bi::LaunchCtx c = ctx(eng, stream);
    if (tier && dtype == BI_F32)  // dw = x^T dy: both transposed (contraction over m)
        return tf32x3(eng, c, {x, m, k, true}, {dy, m, n, true}, dw, n, nullptr, k, n, m, "bi_backward_dw");
    if (tier) {
        Scratch ws(eng, s, static_cast<size_t>(bi::tc_dw_workspace_bytes(c, out_f32, m, k, n)));
        if (ws.err != cudaSuccess) return cuda_fail(eng, ws.err, "dW chunk scratch");
        cudaError_t e = bi::tc_dw(c, dtype, dw, out_f32, x, dy, m, k, n, static_cast<float*>(ws.ptr));
        return e == cudaSuccess ? BI_OK : cuda_fail(eng, e, "bi_backward_dw");
    }
    Scratch part(eng, s, J > 1 ? static_cast<size_t>(J * k * n * 4) : 0);
    if (part.err != cudaSuccess) return cuda_fail(eng, part.err, "dW scratch");
    cudaError_t e = bi::scalar_dw(c, dtype, dw, out_f32, x, dy, m, k, n, static_cast<float*>(part.ptr));
    return e == cudaSuccess ? BI_OK : cuda_fail(eng, e, "bi_backward_dw");
}

bi_status bi_bias_grad(bi_engine eng, void* db, int db_f32, const void* dy, int64_t m, int64_t n,
                       bi_dtype dtype, void* stream) {
    bi_status st = check_common(eng, dtype, m, 1, n);
    if (st != BI_OK) return st;
    if (!db) return fail(eng, BI_ERR_INVALID_ARG, "db must not be NULL");
    if (m > 0 && !dy) return fail(eng, BI_ERR_INVALID_ARG, "dy must not be NULL");
    const int64_t J = (m + BI_DW_CHUNK - 1) / BI_DW_CHUNK;
    const int out_f32 = db_f32 || dtype == BI_F32;
    DeviceGuard g(eng->device);
    if (!g.ok) return fail(eng, BI_ERR_CUDA, "cudaSetDevice failed");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (m == 0) {
        cudaError_t e = cudaMemsetAsync(db, 0, static_cast<size_t>(n * (out_f32 ? 4 : dsize(dtype))), s);
        return e == cudaSuccess ? BI_OK : cuda_fail(eng, e, "bi_bias_grad");
    }
    Scratch part(eng, s, J > 1 ? static_cast<size_t>(J * n * 4) : 0);
    if (part.err != cudaSuccess) return cuda_fail(eng, part.err, "bias-gradient scratch");
    cudaError_t e = bi::bias_grad(ctx(eng, stream), dtype, db, out_f32, dy, m, n, static_cast<float*>(part.ptr));
    return e == cudaSuccess ? BI_OK : cuda_fail(eng, e, "bi_bias_grad");
}

bi_status bi_fp8_quantize(bi_engine eng, uint8_t* q, float* amax, const void* src, const float* scale_inv,
                          int64_t count, bi_dtype src_dtype, void* stream) {
    if (!eng) return fail(nullptr, BI_ERR_INVALID_ARG, "engine is NULL");
    if (src_dtype != BI_F32 && src_dtype != BI_BF16 && src_dtype != BI_F16)
        return fail(eng, BI_ERR_INVALID_ARG, "dtype must be BI_F32, BI_BF16 or BI_F16");
    if (count < 0) return fail(eng, BI_ERR_INVALID_ARG, "count must be >= 0");
    if (!amax || !scale_inv || (count > 0 && (!q || !src)))
        return fail(eng, BI_ERR_INVALID_ARG, "q, amax, src and scale_inv must not be NULL");
    DeviceGuard g(eng->device);
    if (!g.ok) return fail(eng, BI_ERR_CUDA, "cudaSetDevice failed");
    cudaError_t e = bi::fp8_quantize(ctx(eng, stream), src_dtype, q, amax, src, scale_inv, count);
    return e == cudaSuccess ? BI_OK : cuda_fail(eng, e, "bi_fp8_quantize");
}

namespace {

bi_status fp8_pass(bi_engine eng, int pass, void* out, const uint8_t* a, const uint8_t* b, const void* bias,
                   const float* sa, const float* sb, int64_t m, int64_t k, int64_t n, bi_dtype out_dtype,
                   void* stream, const char* name) {
    bi_status st = check_common(eng, out_dtype, m, k, n);
    if (st != BI_OK) return st;
    if (k % 16 != 0 || n % 16 != 0)
        return fail(eng, BI_ERR_UNSUPPORTED, "FP8 operands need k and n multiples of 16 (16-byte rows)");
    if (bias && out_dtype == BI_F32)
        return fail(eng, BI_ERR_UNSUPPORTED, "a bias is supported with bf16 or f16 output");
    if (!out || !sa || !sb || (m > 0 && (!a || !b)))
        return fail(eng, BI_ERR_INVALID_ARG, "outputs, operands and scales must not be NULL");
    if (m == 0 && pass != 2) return BI_OK;
    if (!aligned16(out) || (m > 0 && (!aligned16(a) || !aligned16(b))))
        return fail(eng, BI_ERR_MISALIGNED, "FP8 operands and outputs need 16-byte alignment");
    DeviceGuard g(eng->device);
    if (!g.ok) return fail(eng, BI_ERR_CUDA, "cudaSetDevice failed");
    if (m == 0) {
        cudaError_t e = cudaMemsetAsync(out, 0, static_cast<size_t>(k * n * (out_dtype == BI_F32 ? 4 : 2)),
                                        static_cast<cudaStream_t>(stream));
        return e == cudaSuccess ? BI_OK : cuda_fail(eng, e, name);
    }
    Scratch ws(eng, static_cast<cudaStream_t>(stream),
               pass == 2 ? static_cast<size_t>(bi::tc_fp8_dw_workspace_bytes(out_dtype == BI_F32, m, k, n)) : 0);
    if (ws.err != cudaSuccess) return cuda_fail(eng, ws.err, "FP8 dW chunk scratch");
    cudaError_t e = bi::tc_fp8_pass(ctx(eng, stream), pass, out_dtype, out, a, b, bias, sa, sb, m, k, n,
                                    static_cast<float*>(ws.ptr));
    return e == cudaSuccess ? BI_OK : cuda_fail(eng, e, name);
}

}  // namespace

bi_status bi_fp8_forward(bi_engine eng, void* y, const uint8_t* xq, const uint8_t* wq, const void* bias,
                         const float* scale_x, const float* scale_w, int64_t m, int64_t k, int64_t n,
                         bi_dtype out_dtype, void* stream) {
    return fp8_pass(eng, 0, y, xq, wq, bias, scale_x, scale_w, m, k, n, out_dtype, stream, "bi_fp8_forward");
}

bi_status bi_fp8_backward_dx(bi_engine eng, void* dx, const uint8_t* gq, const uint8_t* wq,
                             const float* scale_g, const float* scale_w, int64_t m, int64_t k, int64_t n,
                             bi_dtype out_dtype, void* stream) {
    return fp8_pass(eng, 1, dx, gq, wq, nullptr, scale_g, scale_w, m, k, n, out_dtype, stream,
                    "bi_fp8_backward_dx");
}

bi_status bi_fp8_backward_dw(bi_engine eng, void* dw, const uint8_t* xq, const uint8_t* gq,
                             const float* scale_x, const float* scale_g, int64_t m, int64_t k, int64_t n,
                             bi_dtype out_dtype, void* stream) {
    return fp8_pass(eng, 2, dw, xq, gq, nullptr, scale_x, scale_g, m, k, n, out_dtype, stream,
                    "bi_fp8_backward_dw");
}

namespace {

bi_status check_grouped(bi_engine eng, bi_dtype dt, int64_t m, int64_t k, int64_t n, int64_t e) {
    if (!eng) return fail(nullptr, BI_ERR_INVALID_ARG, "engine is NULL");
    const char* why = "";
    const bi_status st = bi::check_sizes(dt, m, k, n, e < 0 ? 0 : e, &why);
    return st == BI_OK ? BI_OK : fail(eng, st, why);
}

}  // namespace

}  // extern "C"

namespace {

// Where the grouping of rows by expert comes from: expert ids (stable counting
// sort on the device) or caller offsets (rows already grouped).
struct Grouping {
    const uint32_t* ids;
    const uint32_t* offsets;
};

cudaError_t build_grouping(const bi::LaunchCtx& c, const Grouping& src, int64_t m, int64_t e,
                           uint32_t* seg, uint32_t* perm, void* hist) {
    if (src.ids) return bi::segment(c, src.ids, m, e, seg, perm, hist);
    return bi::segment_from_offsets(c, src.offsets, m, e, seg, perm);
}

int64_t round256(int64_t b) { return (b + 255) / 256 * 256; }

bi_status grouped_forward_impl(bi_engine eng, void* y, const void* x, const void* w, const Grouping& src,
                               int64_t m, int64_t k, int64_t n, int64_t e, bi_dtype dtype,
                               void* stream, int tier, const char* name) {
    if (tier && (!aligned16(y) || !aligned16(x) || !aligned16(w)))
        return fail(eng, BI_ERR_MISALIGNED, "tensor-core tier needs 16-byte aligned y, x, w");
    DeviceGuard g(eng->device);
    if (!g.ok) return fail(eng, BI_ERR_CUDA, "cudaSetDevice failed");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bi::LaunchCtx c = ctx(eng, stream);
    // scratch: seg table | perm | histogram | (row-sorted X).  Caller-grouped rows
    // (offsets) are already sorted: the tensor cores read X in place.
    const bool sorted_in_place = src.ids == nullptr;
    const int64_t seg_b = round256(bi::seg_table_len(e) * 4);
    const int64_t perm_b = round256(m * 4);
    const int64_t hist_b = src.ids ? round256(bi::segment_scratch_bytes(m, e)) : 0;
    const int64_t xs_b = tier && !sorted_in_place ? round256(m * k * 2) : 0;
    Scratch sc(eng, s, static_cast<size_t>(seg_b + perm_b + hist_b + xs_b));
    if (sc.err != cudaSuccess) return cuda_fail(eng, sc.err, "grouped scratch");
    uint8_t* base = static_cast<uint8_t*>(sc.ptr);
    uint32_t* seg = reinterpret_cast<uint32_t*>(base);
    uint32_t* perm = reinterpret_cast<uint32_t*>(base + seg_b);
    void* hist = base + seg_b + perm_b;
    void* xs = base + seg_b + perm_b + hist_b;
    cudaError_t err = build_grouping(c, src, m, e, seg, perm, hist);
    if (err == cudaSuccess) {
        if (tier) {
            const void* a = x;
            if (!sorted_in_place) {  // the gather also zeroes the padding rows of y
                err = bi::gather_sorted(c, x, m, k, e, seg, perm, xs, y, n);
                a = xs;
            }
            if (err == cudaSuccess) err = bi::tc_grouped_rows(c, dtype, 0, y, a, w, m, k, n, e, seg, perm);
        } else {
            err = bi::scalar_rows_grouped(c, dtype, y, x, w, m, k, n, e, 1, seg, perm);
        }
    }
    if (err == cudaSuccess && !(tier && !sorted_in_place))
        err = bi::zero_padding_rows(c, y, n, static_cast<int>(dsize(dtype)), e, seg, perm);
    return err == cudaSuccess ? BI_OK : cuda_fail(eng, err, name);
}

bi_status grouped_backward_impl(bi_engine eng, void* dx, float* dw, const void* x, const void* w,
                                const void* dy, const Grouping& src, int64_t m, int64_t k, int64_t n,
                                int64_t e, bi_dtype dtype, void* stream, int tier_dx, int tier_dw,
                                const char* name) {
    DeviceGuard g(eng->device);
    if (!g.ok) return fail(eng, BI_ERR_CUDA, "cudaSetDevice failed");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (m == 0) {
        cudaError_t err = cudaMemsetAsync(dw, 0, static_cast<size_t>(e * n * k * 4), s);
        return err == cudaSuccess ? BI_OK : cuda_fail(eng, err, name);
    }
    if ((tier_dx || tier_dw) &&
        (!aligned16(x) || !aligned16(w) || !aligned16(dy) || !aligned16(dw) || (dx && !aligned16(dx))))
        return fail(eng, BI_ERR_MISALIGNED, "tensor-core tier needs 16-byte aligned operands");
    const bi::LaunchCtx c = ctx(eng, stream);
    // scratch: seg table | perm | histogram | row-sorted dY, X (unless the caller
    // grouped the rows) | dY, X tail blocks (tensor-core dweights) | chunk partials
    // (scalar dweights)
    const bool sorted_in_place = src.ids == nullptr;
    const int64_t seg_b = round256(bi::seg_table_len(e) * 4);
    const int64_t perm_b = round256(m * 4);
    const int64_t hist_b = src.ids ? round256(bi::segment_scratch_bytes(m, e)) : 0;
    const bool need_dys = (tier_dx || tier_dw) && !sorted_in_place;
    const int64_t dys_b = need_dys ? round256(m * n * 2) : 0;
    const int64_t xs_b = tier_dw && !sorted_in_place ? round256(m * k * 2) : 0;
    const int64_t tails_b = tier_dw ? round256(e * bi::GROUPED_TAIL_ROWS * n * 2) +
                                          round256(e * bi::GROUPED_TAIL_ROWS * k * 2)
                                    : 0;
    const int64_t max_chunks = (m + BI_DW_CHUNK - 1) / BI_DW_CHUNK + e;
    const int64_t part_b = tier_dw ? round256(bi::tc_grouped_dw_workspace_bytes(m, k, n, e)) : max_chunks * n * k * 4;
    Scratch sc(eng, s, static_cast<size_t>(seg_b + perm_b + hist_b + dys_b + xs_b + tails_b + part_b));
    if (sc.err != cudaSuccess) return cuda_fail(eng, sc.err, "grouped scratch");
    uint8_t* base = static_cast<uint8_t*>(sc.ptr);
    uint32_t* seg = reinterpret_cast<uint32_t*>(base);
    uint32_t* perm = reinterpret_cast<uint32_t*>(base + seg_b);
    uint8_t* q = base + seg_b + perm_b;
    void* hist = q;
    q += hist_b;
    void* dys = q;
    q += dys_b;
    void* xs = q;
    q += xs_b;
    void* dyt = q;
    void* xt = q + (tier_dw ? round256(e * bi::GROUPED_TAIL_ROWS * n * 2) : 0);
    q += tails_b;
    float* part = reinterpret_cast<float*>(q);
    cudaError_t err = build_grouping(c, src, m, e, seg, perm, hist);
    const void* dy_sorted = dy;
    const void* x_sorted = sorted_in_place ? x : xs;
    // The dweights operands that dinput does not use (sorted X, both tail
    // buffers) are prepared on the engine's side stream while dinput runs;
    // the caller's stream waits for them before dweights (and before the
    // scratch is released).  The arithmetic is the same either way.
    const bool overlap = err == cudaSuccess && tier_dw && dx != nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
    if (overlap) {
        err = cudaEventCreateWithFlags(&fork, cudaEventDisableTiming);
        if (err == cudaSuccess) err = cudaEventCreateWithFlags(&join, cudaEventDisableTiming);
        if (err == cudaSuccess) err = cudaEventRecord(fork, s);
        if (err == cudaSuccess) err = cudaStreamWaitEvent(eng->side, fork, 0);
    }
    auto prepare_dw = [&](const bi::LaunchCtx& cc) {
        cudaError_t r = cudaSuccess;
        if (!sorted_in_place) r = bi::gather_sorted(cc, x, m, k, e, seg, perm, xs);
        if (r == cudaSuccess) r = bi::build_tails(cc, dy, n, e, seg, perm, dyt);
        if (r == cudaSuccess) r = bi::build_tails(cc, x, k, e, seg, perm, xt);
        return r;
    };
    cudaError_t side_err = cudaSuccess;
    if (overlap && err == cudaSuccess) {
        side_err = prepare_dw(ctx(eng, eng->side));
        const cudaError_t rj = cudaEventRecord(join, eng->side);  // recorded whatever happened above
        if (side_err == cudaSuccess) side_err = rj;
    }
    // the dY gather also zeroes the padding rows of dx when the tensor cores write dx
    const bool fused_zero = need_dys && dx && tier_dx;
    if (err == cudaSuccess && need_dys) {
        err = bi::gather_sorted(c, dy, m, n, e, seg, perm, dys, fused_zero ? dx : nullptr, k);
        dy_sorted = dys;
    }
    if (err == cudaSuccess && dx) {
        err = tier_dx ? bi::tc_grouped_rows(c, dtype, 1, dx, dy_sorted, w, m, k, n, e, seg, perm)
                      : bi::scalar_rows_grouped(c, dtype, dx, dy, w, m, n, k, e, 0, seg, perm);
        if (err == cudaSuccess && !fused_zero)
            err = bi::zero_padding_rows(c, dx, k, static_cast<int>(dsize(dtype)), e, seg, perm);
    }
    if (join) {  // always joined before anything below and before the scratch is freed
        const cudaError_t rw = cudaStreamWaitEvent(s, join, 0);
        if (err == cudaSuccess) err = side_err != cudaSuccess ? side_err : rw;
    }
    if (fork) cudaEventDestroy(fork);
    if (join) cudaEventDestroy(join);
    if (err == cudaSuccess) {
        if (tier_dw) {
            if (!overlap) err = prepare_dw(c);
            if (err == cudaSuccess)
                err = bi::tc_grouped_dw(c, dtype, dw, dy_sorted, x_sorted, dyt, xt, m, k, n, e, seg, part);
        } else {
            err = bi::scalar_dw_grouped(c, dtype, dw, dy, x, m, n, k, e, seg, perm, part, max_chunks);
        }
    }
    return err == cudaSuccess ? BI_OK : cuda_fail(eng, err, name);
}

// Strategy -> tier for one pass: -1 when the tensor cores were requested and
// the pass cannot use them.
int resolve_strategy(bi_strategy st, int pass, bi_dtype dt, int64_t k, int64_t n) {
    const int avail = bi_dispatch_tier(pass, dt, 1, k, n);
    switch (st) {
        case BI_STRATEGY_SCALAR: return 0;
        case BI_STRATEGY_TENSOR_CORE: return avail ? 1 : -1;
        case BI_STRATEGY_AUTO: return avail;
        default: return -2;
    }
}

}  // namespace

extern "C" {

bi_status bi_grouped_forward(bi_engine eng, void* y, const void* x, const void* w,
                             const uint32_t* row_experts, int64_t m, int64_t k, int64_t n, int64_t e,
                             bi_dtype dtype, void* stream, int tensor_cores) {
    bi_status st = check_grouped(eng, dtype, m, k, n, e);
    if (st != BI_OK) return st;
    if (m == 0) return BI_OK;
    if (!y || !x || !w || !row_experts)
        return fail(eng, BI_ERR_INVALID_ARG, "y, x, w and row_experts must not be NULL");
    const int tier = bi_dispatch_tier(BI_PASS_GROUPED_FORWARD, dtype, tensor_cores, k, n);
    return grouped_forward_impl(eng, y, x, w, Grouping{row_experts, nullptr}, m, k, n, e, dtype, stream,
                                tier, "bi_grouped_forward");
}

bi_status bi_grouped_backward(bi_engine eng, void* dx, float* dw, const void* x, const void* w,
                              const void* dy, const uint32_t* row_experts, int64_t m, int64_t k,
                              int64_t n, int64_t e, bi_dtype dtype, void* stream, int tensor_cores) {
    bi_status st = check_grouped(eng, dtype, m, k, n, e);
    if (st != BI_OK) return st;
    if (!dw) return fail(eng, BI_ERR_INVALID_ARG, "dw must not be NULL");
    if (m > 0 && (!x || !w || !dy || !row_experts))
        return fail(eng, BI_ERR_INVALID_ARG, "x, w, dy and row_experts must not be NULL");
    const int tier_dx = dx ? bi_dispatch_tier(BI_PASS_GROUPED_DINPUT, dtype, tensor_cores, k, n) : 0;
    const int tier_dw = bi_dispatch_tier(BI_PASS_GROUPED_DWEIGHTS, dtype, tensor_cores, k, n);
    return grouped_backward_impl(eng, dx, dw, x, w, dy, Grouping{row_experts, nullptr}, m, k, n, e, dtype,
                                 stream, tier_dx, tier_dw, "bi_grouped_backward");
}

bi_status bi_grouped_forward_segmented(bi_engine eng, void* y, const void* x, const void* w,
                                       const uint32_t* offsets, int64_t m, int64_t k, int64_t n,
                                       int64_t e, bi_dtype dtype, void* stream, bi_strategy strategy) {
    bi_status st = check_grouped(eng, dtype, m, k, n, e);
    if (st != BI_OK) return st;
    const int tier = resolve_strategy(strategy, BI_PASS_GROUPED_FORWARD, dtype, k, n);
    if (tier == -2) return fail(eng, BI_ERR_INVALID_ARG, "unknown strategy");
    if (tier < 0)
        return fail(eng, BI_ERR_UNSUPPORTED,
                    "the tensor-core tier was requested but is unavailable for this dtype and shape");
    if (m == 0) return BI_OK;
    if (!y || !x || !w || !offsets) return fail(eng, BI_ERR_INVALID_ARG, "y, x, w and offsets must not be NULL");
    return grouped_forward_impl(eng, y, x, w, Grouping{nullptr, offsets}, m, k, n, e, dtype, stream, tier,
                                "bi_grouped_forward_segmented");
}

bi_status bi_grouped_backward_segmented(bi_engine eng, void* dx, float* dw, const void* x, const void* w,
                                        const void* dy, const uint32_t* offsets, int64_t m, int64_t k,
                                        int64_t n, int64_t e, bi_dtype dtype, void* stream,
                                        bi_strategy strategy) {
    bi_status st = check_grouped(eng, dtype, m, k, n, e);
    if (st != BI_OK) return st;
    if (!dw) return fail(eng, BI_ERR_INVALID_ARG, "dw must not be NULL");
    int tier_dx = dx ? resolve_strategy(strategy, BI_PASS_GROUPED_DINPUT, dtype, k, n) : 0;
    int tier_dw = resolve_strategy(strategy, BI_PASS_GROUPED_DWEIGHTS, dtype, k, n);
    if (tier_dx == -2 || tier_dw == -2) return fail(eng, BI_ERR_INVALID_ARG, "unknown strategy");
    if (tier_dx < 0 || tier_dw < 0)
        return fail(eng, BI_ERR_UNSUPPORTED,
                    "the tensor-core tier was requested but is unavailable for this dtype and shape");
    if (m > 0 && (!x || !w || !dy || !offsets))
        return fail(eng, BI_ERR_INVALID_ARG, "x, w, dy and offsets must not be NULL");
    return grouped_backward_impl(eng, dx, dw, x, w, dy, Grouping{nullptr, offsets}, m, k, n, e, dtype,
                                 stream, tier_dx, tier_dw, "bi_grouped_backward_segmented");
}

}  // extern "C"
