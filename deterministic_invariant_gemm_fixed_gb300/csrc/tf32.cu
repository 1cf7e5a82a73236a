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
// HBM traffic.  The transposing split needs rows of x whose length is a
// multiple of 4 floats and 16-byte aligned buffers (the tensor-core tier's
// shapes and pointers always are).
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

// The same, four elements per step with 16-byte loads and stores (all three
// pointers 16-byte aligned, count a multiple of 4).
__global__ void tf32_split4_kernel(const float4* x, float4* hi, float4* lo, int64_t count4) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < count4; i += stride) {
        const float4 v = x[i];
        const float4 h = make_float4(to_tf32(v.x), to_tf32(v.y), to_tf32(v.z), to_tf32(v.w));
        hi[i] = h;
        lo[i] = make_float4(to_tf32(__fsub_rn(v.x, h.x)), to_tf32(__fsub_rn(v.y, h.y)), to_tf32(__fsub_rn(v.z, h.z)),
                            to_tf32(__fsub_rn(v.w, h.w)));
    }
}

// Transposing split: 64 x 64 tiles through shared memory (one padding column),
// 256 threads, each reading four float4 along rows of x and writing four
// float4 of the parts (four consecutive rows of x for one column).  cols is a
// multiple of 4; ld (>= rows) a multiple of 4; the bases 16-byte aligned.
constexpr int TT = 64;

__global__ void __launch_bounds__(256) tf32_split_t_kernel(const float* __restrict__ x, float* __restrict__ hi,
                                                           float* __restrict__ lo, int64_t rows, int64_t cols,
                                                           int64_t ld) {
    __shared__ float th[TT][TT + 1];
    __shared__ float tl[TT][TT + 1];
    const int64_t tiles_c = (cols + TT - 1) / TT;
    const int64_t tiles = ((rows + TT - 1) / TT) * tiles_c;
    const int t16 = threadIdx.x & 15, t_hi = threadIdx.x >> 4;  // 16 float4 per 64-element row
    for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
        const int64_t r0 = (t / tiles_c) * TT, c0 = (t % tiles_c) * TT;
#pragma unroll
        for (int i = 0; i < 4; ++i) {  // x rows r0 + t_hi + 16i, columns c0 + 4 t16 .. +3
            const int r = t_hi + 16 * i, c = 4 * t16;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (r0 + r < rows && c0 + c < cols) v = *reinterpret_cast<const float4*>(x + (r0 + r) * cols + c0 + c);
            const float e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float h = to_tf32(e[j]);
                th[r][c + j] = h;
                tl[r][c + j] = to_tf32(__fsub_rn(e[j], h));
            }
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 4; ++i) {  // output row = x column c0 + oc; x rows r0 + 4 t16 .. +3
            const int oc = t_hi + 16 * i, r = 4 * t16;
            const int64_t col = c0 + oc, row = r0 + r;
            if (col < cols && row < rows) {
                const float4 h = make_float4(th[r][oc], th[r + 1][oc], th[r + 2][oc], th[r + 3][oc]);
                const float4 l = make_float4(tl[r][oc], tl[r + 1][oc], tl[r + 2][oc], tl[r + 3][oc]);
                if (row + 4 <= rows) {
                    *reinterpret_cast<float4*>(hi + col * ld + row) = h;
                    *reinterpret_cast<float4*>(lo + col * ld + row) = l;
                } else {  // the last rows of x: the rest of the padded row is never read
                    const float hv[4] = {h.x, h.y, h.z, h.w}, lv[4] = {l.x, l.y, l.z, l.w};
                    for (int j = 0; j < 4 && row + j < rows; ++j) {
                        hi[col * ld + row + j] = hv[j];
                        lo[col * ld + row + j] = lv[j];
                    }
                }
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
    const bool a16 = ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(hi) |
                       reinterpret_cast<uintptr_t>(lo)) & 15u) == 0;
    if (!transpose) {
        if (a16 && count % 4 == 0) {
            int64_t blocks = (count / 4 + 255) / 256;
            if (blocks > cap) blocks = cap;
            tf32_split4_kernel<<<static_cast<unsigned>(blocks), 256, 0, c.stream>>>(
                reinterpret_cast<const float4*>(x), reinterpret_cast<float4*>(hi), reinterpret_cast<float4*>(lo),
                count / 4);
        } else {
            int64_t blocks = (count + 255) / 256;
            if (blocks > cap) blocks = cap;
            tf32_split_kernel<<<static_cast<unsigned>(blocks), 256, 0, c.stream>>>(x, hi, lo, count);
        }
    } else {
        if (ld < rows || ld % 4 != 0 || cols % 4 != 0 || !a16) return cudaErrorInvalidValue;
        int64_t blocks = ((rows + TT - 1) / TT) * ((cols + TT - 1) / TT);
        if (blocks > cap) blocks = cap;
        tf32_split_t_kernel<<<static_cast<unsigned>(blocks), 256, 0, c.stream>>>(x, hi, lo, rows, cols, ld);
    }
    c.count();
    return cudaGetLastError();
}

}  // namespace bi
