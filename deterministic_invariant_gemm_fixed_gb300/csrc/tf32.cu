// Split of f32 operands into two TF32 parts for the 3xTF32 tensor-core mode.
//
// hi = x rounded to TF32 (10 fraction bits; round to nearest, ties away, the
// PTX cvt.rna.tf32.f32 conversion); lo = (x - hi) rounded the same way (the
// subtraction is exact in f32).  Both parts are TF32 values stored as f32, so
// the tensor core reads them without further loss, and x*y is taken as
// hi_x*hi_y + hi_x*lo_y + lo_x*hi_y: the dropped lo*lo term and the rounding
// of lo are each below 2^-21 of |x*y|.  For x = +-Inf, hi = x and lo = NaN
// (Inf - Inf); the pair kernel's epilogue then keeps the infinite hi*hi sum
// and drops the cross terms, so infinities and NaN come out as the plain f32
// contraction gives them.
//
// The tensor cores read the parts K-major (the contraction index contiguous).
// Operands whose contraction runs down the columns (w in the forward pass, x
// and dy in dW) are transposed by the split itself: it reads every element
// once and writes both parts once either way, so the transpose costs no extra
// HBM traffic.
#include "bi_internal.h"

namespace bi {
namespace {

__device__ __forceinline__ float to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

__global__ void tf32_split_kernel(const float* x, float* hi, float* lo, int64_t count) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < count; i += stride) {
        const float v = x[i];
        const float h = to_tf32(v);
        hi[i] = h;
        lo[i] = to_tf32(__fsub_rn(v, h));
    }
}

// 32 x 32 tiles through shared memory (one padding column: the column-wise
// reads hit 32 different banks); 32 x 8 threads, each moving 4 elements.
constexpr int TT = 32;

__global__ void __launch_bounds__(256) tf32_split_t_kernel(const float* __restrict__ x, float* __restrict__ hi,
                                                           float* __restrict__ lo, int64_t rows, int64_t cols,
                                                           int64_t ld) {
    __shared__ float th[TT][TT + 1];
    __shared__ float tl[TT][TT + 1];
    const int64_t tiles_c = (cols + TT - 1) / TT;
    const int64_t tiles = ((rows + TT - 1) / TT) * tiles_c;
    const int tx = threadIdx.x, ty = threadIdx.y;
    for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
        const int64_t r0 = (t / tiles_c) * TT, c0 = (t % tiles_c) * TT;
        for (int i = ty; i < TT; i += 8) {
            const int64_t r = r0 + i, col = c0 + tx;
            if (r < rows && col < cols) {
                const float v = x[r * cols + col];
                const float h = to_tf32(v);
                th[i][tx] = h;
                tl[i][tx] = to_tf32(__fsub_rn(v, h));
            }
        }
        __syncthreads();
        for (int i = ty; i < TT; i += 8) {
            const int64_t col = c0 + i, r = r0 + tx;  // output row col, column r
            if (r < rows && col < cols) {
                hi[col * ld + r] = th[tx][i];
                lo[col * ld + r] = tl[tx][i];
            }
        }
        __syncthreads();
    }
}

}  // namespace

cudaError_t tf32_split(const LaunchCtx& c, const float* x, float* hi, float* lo, int64_t rows, int64_t cols,
                       bool transpose, int64_t ld) {
    const int64_t count = rows * cols;
    if (count == 0) return cudaSuccess;
    const int64_t cap = static_cast<int64_t>(c.sm_count) * 16;
    if (!transpose) {
        int64_t blocks = (count + 255) / 256;
        if (blocks > cap) blocks = cap;
        tf32_split_kernel<<<static_cast<unsigned>(blocks), 256, 0, c.stream>>>(x, hi, lo, count);
    } else {
        if (ld < rows) return cudaErrorInvalidValue;
        int64_t blocks = ((rows + TT - 1) / TT) * ((cols + TT - 1) / TT);
        if (blocks > cap) blocks = cap;
        tf32_split_t_kernel<<<static_cast<unsigned>(blocks), dim3(TT, 8), 0, c.stream>>>(x, hi, lo, rows, cols, ld);
    }
    c.count();
    return cudaGetLastError();
}

}  // namespace bi
