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

template <typename T>
__global__ void __launch_bounds__(256) fp8_quantize_kernel(const T* src, const float* scale_inv, uint8_t* q,
                                                          unsigned int* amax_bits, int64_t count) {
    const float si = __ldg(scale_inv);
    float mx = 0.0f;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < count; i += stride) {
        const float v = widen<T>(src[i]);
        q[i] = static_cast<uint8_t>(__nv_cvt_float_to_fp8(__fmul_rn(v, si), __NV_SATFINITE, __NV_E4M3));
        mx = fmaxf(mx, fabsf(v));  // a NaN input leaves the maximum unchanged
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
    int64_t blocks = (count + 255) / 256;
    const int64_t cap = static_cast<int64_t>(c.sm_count) * 8;
    if (blocks > cap) blocks = cap;
    unsigned int* ab = reinterpret_cast<unsigned int*>(amax);
    switch (dt) {
        case BI_F32: fp8_quantize_kernel<float><<<static_cast<unsigned>(blocks), 256, 0, c.stream>>>(static_cast<const float*>(src), scale_inv, q, ab, count); break;
        case BI_BF16: fp8_quantize_kernel<__nv_bfloat16><<<static_cast<unsigned>(blocks), 256, 0, c.stream>>>(static_cast<const __nv_bfloat16*>(src), scale_inv, q, ab, count); break;
        default: fp8_quantize_kernel<__half><<<static_cast<unsigned>(blocks), 256, 0, c.stream>>>(static_cast<const __half*>(src), scale_inv, q, ab, count); break;
    }
    c.count();
    return cudaGetLastError();
}

}  // namespace bi
