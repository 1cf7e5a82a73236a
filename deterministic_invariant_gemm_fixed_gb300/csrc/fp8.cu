// FP8 e4m3 quantization with a deterministic amax.
//
// Source: AstrAI csrc/kernels/fp8_mm.cu, quantize_kernel -- dst = e4m3(src *
// scale_inv) with the saturating cast, and the largest |src| recorded with one
// atomic max on the float's bit pattern per block (valid because the bit
// patterns of non-negative floats are ordered like their values).  A maximum is
// exact and does not depend on the order in which blocks contribute, so the
// amax is bit-identical run to run.  The scale multiply is one f32 rounding,
// the cast one round-to-nearest-even step (CUDA's conversion intrinsic).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "bi_internal.h"

namespace bi {
namespace {

template <typename T> __device__ __forceinline__ float widen(T v);
template <> __device__ __forceinline__ float widen<float>(float v) { return v; }
template <> __device__ __forceinline__ float widen<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }
template <> __device__ __forceinline__ float widen<__half>(__half v) { return __half2float(v); }

__device__ __forceinline__ float amax_step(float mx, float v) {
    return fmaxf(mx, fabsf(v));  // a NaN input leaves the maximum unchanged
}

__device__ __forceinline__ uint8_t to_e4m3(float v, float si) {
    return static_cast<uint8_t>(__nv_cvt_float_to_fp8(__fmul_rn(v, si), __NV_SATFINITE, __NV_E4M3));
}

// Two codes at once (the packed conversion; same rounding and saturation as
// to_e4m3), the first value in the low byte.
__device__ __forceinline__ uint16_t to_e4m3x2(float a, float b, float si) {
    return static_cast<uint16_t>(
        __nv_cvt_float2_to_fp8x2(make_float2(__fmul_rn(a, si), __fmul_rn(b, si)), __NV_SATFINITE, __NV_E4M3));
}

// With vec != 0 (src 16-byte and q (16 / sizeof(T))-byte aligned), each step of
// a thread reads 16 bytes of source and writes 16 / sizeof(T) codes; the tail
// and unaligned buffers go element by element.
template <typename T>
__global__ void __launch_bounds__(256) fp8_quantize_kernel(const T* src, const float* scale_inv, uint8_t* q,
                                                          unsigned int* amax_bits, int64_t count, int vec) {
    grid_dep_wait();
    grid_dep_launch();
    constexpr int V = 16 / sizeof(T);
    const float si = __ldg(scale_inv);
    float mx = 0.0f;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t tid = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
    const int64_t nvec = vec ? count / V : 0;
    for (int64_t i = tid; i < nvec; i += stride) {
        const uint4 raw = __ldcs(reinterpret_cast<const uint4*>(src) + i);  // read once: streaming
        const T* e = reinterpret_cast<const T*>(&raw);
        float f[V];
#pragma unroll
        for (int j = 0; j < V; ++j) {
            f[j] = widen<T>(e[j]);
            mx = amax_step(mx, f[j]);
        }
        if (V == 8) {
            uint2 o;
            o.x = to_e4m3x2(f[0], f[1], si) | (static_cast<uint32_t>(to_e4m3x2(f[2], f[3], si)) << 16);
            o.y = to_e4m3x2(f[4 % V], f[5 % V], si) | (static_cast<uint32_t>(to_e4m3x2(f[6 % V], f[7 % V], si)) << 16);
            reinterpret_cast<uint2*>(q)[i] = o;
        } else {
            reinterpret_cast<uint32_t*>(q)[i] =
                to_e4m3x2(f[0], f[1], si) | (static_cast<uint32_t>(to_e4m3x2(f[2 % V], f[3 % V], si)) << 16);
        }
    }
    for (int64_t i = nvec * V + tid; i < count; i += stride) {
        const float v = widen<T>(src[i]);
        q[i] = to_e4m3(v, si);
        mx = amax_step(mx, v);
    }
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    __shared__ float wmax[8];
    if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = mx;
    __syncthreads();
    if (threadIdx.x == 0) {
        float b = 0.0f;
        for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) b = fmaxf(b, wmax[w]);
        atomicMax(amax_bits, __float_as_uint(b));
    }
}

}  // namespace

cudaError_t fp8_quantize(const LaunchCtx& c, bi_dtype dt, uint8_t* q, float* amax, const void* src,
                         const float* scale_inv, int64_t count) {
    cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(float), c.stream);
    if (e != cudaSuccess || count == 0) return e;
    const int64_t esize = dt == BI_F32 ? 4 : 2;
    const int64_t per = 16 / esize;  // elements per 16-byte step
    const int vec = (reinterpret_cast<uintptr_t>(src) % 16 == 0 && reinterpret_cast<uintptr_t>(q) % per == 0) ? 1 : 0;
    int64_t blocks = ((vec ? count / per : count) + 255) / 256;
    const int64_t cap = static_cast<int64_t>(c.sm_count) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    unsigned int* ab = reinterpret_cast<unsigned int*>(amax);
    const dim3 grid(static_cast<unsigned>(blocks)), block(256);
    switch (dt) {
        case BI_F32:
            e = launch_pdl(fp8_quantize_kernel<float>, grid, block, 0, c.stream, static_cast<const float*>(src),
                           scale_inv, q, ab, count, vec);
            break;
        case BI_BF16:
            e = launch_pdl(fp8_quantize_kernel<__nv_bfloat16>, grid, block, 0, c.stream,
                           static_cast<const __nv_bfloat16*>(src), scale_inv, q, ab, count, vec);
            break;
        default:
            e = launch_pdl(fp8_quantize_kernel<__half>, grid, block, 0, c.stream, static_cast<const __half*>(src),
                           scale_inv, q, ab, count, vec);
            break;
    }
    if (e != cudaSuccess) return e;
    c.count();
    return cudaGetLastError();
}

}  // namespace bi
