/*
 * CPU oracle for the deterministic, batch-invariant training matmul.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or constant with
 * the CUDA library; the two meet only in the seeded host buffers that both are
 * given.
 *
 * What it computes is the scalar-tier contract of "sgemm-bi 0.1.1.post2"
 * (PyPI page, "Determinism contracts" table, row "f32 / typed scalar"):
 * bf16/f16 operands are widened exactly to f32, the product is formed by an
 * f32 kernel, and the result is rounded once, to nearest-even, to the operand
 * type.  The three matmuls of a linear layer follow the same page's "Use"
 * section (weight stored [in, out]) and the autograd function of
 * "ViperLLM ffma.py" (_FFMAAddmm.forward adds the bias in f32 before the one
 * downcast; _FFMAAddmm.backward forms gx = gy * W^T and gW = x^T * gy).  The
 * grouped per-row-expert variant follows "rublas 0.1.45
 * src/tensor_grouped/mod.rs" (fn grouped_matmul_nt: Y = X * W[e(m)]^T with
 * W shaped [E,N,K], ids outside [0,E) give zero rows, f32 accumulation and one
 * output rounding; struct GroupedBackward: dweights always f32).
 *
 * Where the pages leave the arithmetic open, the oracle takes these readings
 * (each is part of the library's published contract as well):
 *   - a dot product is a chain: acc = +0.0f, then acc = fmaf(a_i, b_i, acc)
 *     for i ascending over the contracted index;
 *   - the bias enters after the chain as one f32 add, then one rounding;
 *   - the dW reduction over rows is split into chunks of `chunk` consecutive
 *     rows counted from the first row; each chunk is a chain, and the chunk
 *     partials are summed by a pairwise tree over adjacent entries in which an
 *     odd last entry is carried up unchanged;
 *   - grouped rows are taken per expert in ascending original row index.
 *
 * Plain C, no blocking, no reassociation inside a chain.  Loops over
 * independent outputs may run in parallel (OpenMP) or be interleaved; that
 * cannot change a bit of any output because every output's chain is computed
 * in its own order.  Build with -ffp-contract=off and without -ffast-math.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_F32 = 0, OR_BF16 = 1, OR_F16 = 2 };

/* ------------------------------------------------------------------------ */
/* IEEE-754 format helpers, written from the binary16 / bfloat16 / binary32  */
/* encodings: sign bit, biased exponent, trailing significand.              */
/* ------------------------------------------------------------------------ */

static uint32_t f32_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float bits_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/* bfloat16 is the upper half of a binary32: widening appends 16 zero bits. */
static float up_bf16(uint16_t h) { return bits_f32((uint32_t)h << 16); }

/* binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
static float up_f16(uint16_t h)
{
    uint32_t sign = (uint32_t)(h >> 15) << 31;
    uint32_t e = (h >> 10) & 0x1fu;
    uint32_t frac = h & 0x3ffu;
    if (e == 0x1fu) /* inf or NaN: keep the fraction, left-aligned */
        return bits_f32(sign | 0x7f800000u | (frac << 13));
    if (e == 0) {   /* zero or subnormal: value = frac * 2^-24, exact */
        float mag = ldexpf((float)frac, -24);
        return sign ? -mag : mag;
    }
    /* normal: rebias the exponent from 15 to 127 */
    return bits_f32(sign | ((e - 15u + 127u) << 23) | (frac << 13));
}

/* Round `keep` (the retained high part) to nearest, ties to even, given the
 * discarded low part `rem` and the weight `half` of half a unit in the last
 * retained place.  Returns the increment (0 or 1). */
static uint32_t rne_increment(uint32_t keep, uint32_t rem, uint32_t half)
{
    if (rem > half) return 1;
    if (rem < half) return 0;
    return keep & 1u; /* exact tie: round to the even neighbour */
}

/* binary32 -> bfloat16, round to nearest even.  A NaN becomes the quiet NaN
 * 0x7FC0; overflow carries into the exponent and lands on infinity. */
static uint16_t rne_bf16(float f)
{
    uint32_t u = f32_bits(f);
    if ((u & 0x7fffffffu) > 0x7f800000u) return 0x7fc0u;
    uint32_t keep = u >> 16, rem = u & 0xffffu;
    return (uint16_t)(keep + rne_increment(keep, rem, 0x8000u));
}

/* binary32 -> binary16, round to nearest even, with gradual underflow.  A NaN
 * becomes the quiet NaN 0x7E00 with the input's sign. */
static uint16_t rne_f16(float f)
{
    uint32_t u = f32_bits(f);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    uint32_t ef = (u >> 23) & 0xffu;
    uint32_t frac = u & 0x7fffffu;
    if (ef == 0xffu) return frac ? (uint16_t)(sign | 0x7e00u) : (uint16_t)(sign | 0x7c00u);
    if (ef == 0) return sign; /* binary32 zero/subnormal: far below 2^-25 */
    int32_t e = (int32_t)ef - 127;   /* unbiased exponent */
    uint32_t sig = frac | 0x800000u;  /* 24-bit significand, value sig * 2^(e-23) */
    if (e > 15) return (uint16_t)(sign | 0x7c00u);
    if (e >= -14) {
        /* normal range: keep 11 significant bits (implicit one included) */
        uint32_t keep = sig >> 13, rem = sig & 0x1fffu;
        uint32_t mag = ((uint32_t)(e + 15) << 10) + (keep - 0x400u);
        mag += rne_increment(keep, rem, 0x1000u); /* a carry may reach 0x7c00 = inf */
        return (uint16_t)(sign | mag);
    }
    /* subnormal range: the unit is 2^-24, so keep sig >> (13 + (-14 - e)) */
    int32_t shift = 13 + (-14 - e);
    if (shift > 24) return sign; /* below 2^-25 in magnitude: rounds to zero */
    uint32_t keep = sig >> shift;
    uint32_t rem = sig & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1);
    return (uint16_t)(sign | (keep + rne_increment(keep, rem, half)));
}

/* Widen element i of a typed buffer. */
static float load_up(const void* p, int dtype, int64_t i)
{
    if (dtype == OR_F32) return ((const float*)p)[i];
    uint16_t h = ((const uint16_t*)p)[i];
    return dtype == OR_BF16 ? up_bf16(h) : up_f16(h);
}

/* Round an f32 result to the output type (identity for f32) and store it. */
static void store_down(void* p, int dtype, int64_t i, float v)
{
    if (dtype == OR_F32) { ((float*)p)[i] = v; return; }
    ((uint16_t*)p)[i] = dtype == OR_BF16 ? rne_bf16(v) : rne_f16(v);
}

/* Widen a whole typed buffer into a fresh f32 array (exact; caller frees). */
static float* widen(const void* p, int dtype, int64_t count)
{
    float* out = (float*)malloc((size_t)(count > 0 ? count : 1) * sizeof(float));
    if (!out) return NULL;
    for (int64_t i = 0; i < count; ++i) out[i] = load_up(p, dtype, i);
    return out;
}

/* The fixed dW tree: pairwise sums of adjacent entries, level by level; an odd
 * last entry is carried to the next level unchanged.  Works in place on v[0..J)
 * and returns the root (+0.0f when J == 0). */
static float tree_sum(float* v, int64_t J)
{
    if (J == 0) return 0.0f;
    while (J > 1) {
        int64_t pairs = J / 2;
        for (int64_t i = 0; i < pairs; ++i) v[i] = v[2 * i] + v[2 * i + 1];
        if (J & 1) v[pairs] = v[J - 1];
        J = pairs + (J & 1);
    }
    return v[0];
}

/* ------------------------------------------------------------------------ */
/* Exported scalar helpers (used by the tests to pin the format code).       */
/* ------------------------------------------------------------------------ */

void or_rne_array(uint16_t* out, const float* in, int64_t count, int dtype)
{
    for (int64_t i = 0; i < count; ++i) out[i] = dtype == OR_BF16 ? rne_bf16(in[i]) : rne_f16(in[i]);
}

void or_rne_bits_range(uint16_t* out, uint64_t first_bits, int64_t count, int dtype)
{
    /* out[i] = rne(float with bit pattern first_bits + i): exhaustive sweeps */
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < count; ++i) {
        float f = bits_f32((uint32_t)(first_bits + (uint64_t)i));
        out[i] = dtype == OR_BF16 ? rne_bf16(f) : rne_f16(f);
    }
}

void or_up_array(float* out, const uint16_t* in, int64_t count, int dtype)
{
    for (int64_t i = 0; i < count; ++i) out[i] = dtype == OR_BF16 ? up_bf16(in[i]) : up_f16(in[i]);
}

float or_fmaf(float a, float b, float c) { return fmaf(a, b, c); }

float or_tree_sum(float* v, int64_t J) { return tree_sum(v, J); }

int or_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void or_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ------------------------------------------------------------------------ */
/* Dense passes.  Row-major contiguous: X[M,K], W[K,N] ([in,out]), b[N],      */
/* Y[M,N], dY[M,N], dX[M,K], dW[K,N].                                        */
/* out_f32 != 0 writes the f32 value that would have been rounded.           */
/* ------------------------------------------------------------------------ */

/* Forward on a list of rows: Y_rows[i,n] = rne( chain_k X[rows[i],k]*W[k,n] (+ b[n]) ).
 * The whole forward is the case rows = 0..M-1; rows are independent, so any
 * subset is the same definition restricted. */
int or_forward_rows(void* y_rows, const void* x, const void* w, const void* bias,
                    const int64_t* rows, int64_t nrows, int64_t m, int64_t k, int64_t n,
                    int dtype, int out_f32)
{
    float* wf = widen(w, dtype, k * n);
    float* bf = bias ? widen(bias, dtype, n) : NULL;
    if (!wf || (bias && !bf)) { free(wf); free(bf); return -1; }
    int out_t = out_f32 ? OR_F32 : dtype;
    int failed = 0;
    #pragma omp parallel
    {
        float* acc = (float*)malloc((size_t)(n > 0 ? n : 1) * sizeof(float));
        if (!acc) failed = 1;
        #pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < nrows; ++i) {
            if (!acc) continue;
            int64_t r = rows ? rows[i] : i;
            if (r < 0 || r >= m) continue;
            for (int64_t j = 0; j < n; ++j) acc[j] = 0.0f;
            /* each acc[j] runs its own chain over k = 0, 1, ..., K-1 */
            for (int64_t kk = 0; kk < k; ++kk) {
                float a = load_up(x, dtype, r * k + kk);
                const float* wrow = wf + kk * n;
                for (int64_t j = 0; j < n; ++j) acc[j] = fmaf(a, wrow[j], acc[j]);
            }
            for (int64_t j = 0; j < n; ++j) {
                float v = bf ? acc[j] + bf[j] : acc[j];
                store_down(y_rows, out_t, i * n + j, v);
            }
        }
        free(acc);
    }
    free(wf); free(bf);
    return failed ? -1 : 0;
}

int or_forward(void* y, const void* x, const void* w, const void* bias,
               int64_t m, int64_t k, int64_t n, int dtype, int out_f32)
{
    return or_forward_rows(y, x, w, bias, NULL, m, m, k, n, dtype, out_f32);
}

/* dX on a list of rows: dX_rows[i,kk] = rne( chain_n dY[rows[i],n]*W[kk,n] ). */
int or_backward_dx_rows(void* dx_rows, const void* dy, const void* w,
                        const int64_t* rows, int64_t nrows, int64_t m, int64_t k, int64_t n,
                        int dtype, int out_f32)
{
    float* wf = widen(w, dtype, k * n);
    if (!wf) return -1;
    int out_t = out_f32 ? OR_F32 : dtype;
    int failed = 0;
    #pragma omp parallel
    {
        float* g = (float*)malloc((size_t)(n > 0 ? n : 1) * sizeof(float));
        if (!g) failed = 1;
        #pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < nrows; ++i) {
            if (!g) continue;
            int64_t r = rows ? rows[i] : i;
            if (r < 0 || r >= m) continue;
            for (int64_t j = 0; j < n; ++j) g[j] = load_up(dy, dtype, r * n + j);
            for (int64_t kk = 0; kk < k; ++kk) {
                const float* wrow = wf + kk * n;
                float acc = 0.0f;
                for (int64_t j = 0; j < n; ++j) acc = fmaf(g[j], wrow[j], acc);
                store_down(dx_rows, out_t, i * k + kk, acc);
            }
        }
        free(g);
    }
    free(wf);
    return failed ? -1 : 0;
}

int or_backward_dx(void* dx, const void* dy, const void* w,
                   int64_t m, int64_t k, int64_t n, int dtype, int out_f32)
{
    return or_backward_dx_rows(dx, dy, w, NULL, m, m, k, n, dtype, out_f32);
}

/* dW on a list of columns: dW_cols[kk, c] = down( tree_j p_j(kk, cols[c]) ) with
 * p_j = chain over rows r in [j*chunk, min(M,(j+1)*chunk)) of X[r,kk]*dY[r,col].
 * out_f32 != 0 keeps the f32 tree root (the dw_f32 flag of the library). */
int or_backward_dw_cols(void* dw_cols, const void* x, const void* dy,
                        const int64_t* cols, int64_t ncols, int64_t m, int64_t k, int64_t n,
                        int dtype, int64_t chunk, int out_f32)
{
    if (chunk <= 0) return -2;
    int64_t J = (m + chunk - 1) / chunk;
    int out_t = out_f32 ? OR_F32 : dtype;
    float* g = (float*)malloc((size_t)((m * ncols) > 0 ? m * ncols : 1) * sizeof(float));
    if (!g) return -1;
    for (int64_t r = 0; r < m; ++r)
        for (int64_t c = 0; c < ncols; ++c) {
            int64_t col = cols ? cols[c] : c;
            g[r * ncols + c] = (col >= 0 && col < n) ? load_up(dy, dtype, r * n + col) : 0.0f;
        }
    int failed = 0;
    #pragma omp parallel
    {
        float* part = (float*)malloc((size_t)((J * ncols) > 0 ? J * ncols : 1) * sizeof(float));
        float* col_parts = (float*)malloc((size_t)(J > 0 ? J : 1) * sizeof(float));
        if (!part || !col_parts) failed = 1;
        #pragma omp for schedule(dynamic, 1)
        for (int64_t kk = 0; kk < k; ++kk) {
            if (!part || !col_parts) continue;
            for (int64_t j = 0; j < J; ++j) {
                float* p = part + j * ncols;
                for (int64_t c = 0; c < ncols; ++c) p[c] = 0.0f;
                int64_t r_end = (j + 1) * chunk < m ? (j + 1) * chunk : m;
                for (int64_t r = j * chunk; r < r_end; ++r) {
                    float a = load_up(x, dtype, r * k + kk);
                    const float* grow = g + r * ncols;
                    for (int64_t c = 0; c < ncols; ++c) p[c] = fmaf(a, grow[c], p[c]);
                }
            }
            for (int64_t c = 0; c < ncols; ++c) {
                for (int64_t j = 0; j < J; ++j) col_parts[j] = part[j * ncols + c];
                store_down(dw_cols, out_t, kk * ncols + c, tree_sum(col_parts, J));
            }
        }
        free(part); free(col_parts);
    }
    free(g);
    return failed ? -1 : 0;
}

int or_backward_dw(void* dw, int dw_f32, const void* x, const void* dy,
                   int64_t m, int64_t k, int64_t n, int dtype, int64_t chunk)
{
    return or_backward_dw_cols(dw, x, dy, NULL, n, m, k, n, dtype, chunk, dw_f32);
}

/* Bias gradient: db[j] = down( tree_c p_c ) with p_c = sum over the rows r of
 * chunk c (rows [c*chunk, min(M,(c+1)*chunk)), ascending) of dY[r, j], each
 * step one f32 addition starting from +0.0f: the column sum that the bias's
 * gradient is, reduced with the same chunks and tree as dW.  The sgemm-bi page
 * leaves the bias gradient to a plain f32 column sum outside its engine; this
 * is the fixed-order version of that sum.  out_f32 != 0 keeps the f32 root. */
int or_bias_grad(void* db, const void* dy, int64_t m, int64_t n, int dtype, int64_t chunk, int out_f32)
{
    if (chunk <= 0) return -2;
    int64_t J = (m + chunk - 1) / chunk;
    int out_t = out_f32 ? OR_F32 : dtype;
    float* parts = (float*)malloc((size_t)(J > 0 ? J : 1) * sizeof(float));
    if (!parts) return -1;
    for (int64_t j = 0; j < n; ++j) {
        for (int64_t c = 0; c < J; ++c) {
            float acc = 0.0f;
            int64_t r_end = (c + 1) * chunk < m ? (c + 1) * chunk : m;
            for (int64_t r = c * chunk; r < r_end; ++r) acc = acc + load_up(dy, dtype, r * n + j);
            parts[c] = acc;
        }
        store_down(db, out_t, j, tree_sum(parts, J));
    }
    free(parts);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* FP8 e4m3 per-tensor-scaled linear (AstrAI csrc/kernels/fp8_mm.cu:         */
/* quantize_kernel, fp8_linear_forward_scaled, fp8_linear_backward_scaled).  */
/* e4m3 ("fn" flavour): 1 sign, 4 exponent bits (bias 7), 3 fraction bits,  */
/* no infinities, 0x7F/0xFF are NaN, largest finite 448.                     */
/* ------------------------------------------------------------------------ */

/* f32 -> e4m3, round to nearest even, saturating: anything whose rounding
 * would exceed 448 (and +-inf) becomes +-448; NaN becomes 0x7F. */
static uint8_t rne_e4m3(float f)
{
    uint32_t u = f32_bits(f);
    uint8_t sign = (uint8_t)((u >> 24) & 0x80u);
    uint32_t ef = (u >> 23) & 0xffu;
    uint32_t frac = u & 0x7fffffu;
    if (ef == 0xffu && frac) return 0x7fu;        /* NaN */
    if (ef == 0xffu) return (uint8_t)(sign | 0x7eu); /* inf saturates */
    if (ef == 0) return sign;                     /* f32 zero/subnormal: below 2^-10 */
    int32_t e = (int32_t)ef - 127;
    uint32_t sig = frac | 0x800000u;
    if (e > 8) return (uint8_t)(sign | 0x7eu);
    if (e >= -6) {
        /* normal: keep 4 significant bits (implicit one + 3) */
        uint32_t keep = sig >> 20, rem = sig & 0xfffffu;
        uint32_t mag = ((uint32_t)(e + 7) << 3) + (keep - 8u);
        mag += rne_increment(keep, rem, 0x80000u);
        if (mag > 0x7eu) mag = 0x7eu;             /* 480 and above is out of range */
        return (uint8_t)(sign | mag);
    }
    /* subnormal: the unit is 2^-9, keep sig >> (20 + (-6 - e)) */
    int32_t shift = 20 + (-6 - e);
    if (shift > 24) return sign;
    uint32_t keep = sig >> shift;
    uint32_t rem = sig & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1);
    return (uint8_t)(sign | (keep + rne_increment(keep, rem, half)));
}

static float up_e4m3(uint8_t q)
{
    uint32_t sign = (uint32_t)(q >> 7) << 31;
    uint32_t e = (q >> 3) & 0xfu, m = q & 7u;
    if (e == 0xfu && m == 7u) return bits_f32(sign | 0x7fc00000u);
    if (e == 0) { float mag = ldexpf((float)m, -9); return sign ? -mag : mag; }
    return bits_f32(sign | ((e - 7u + 127u) << 23) | (m << 20));
}

void or_e4m3_bits_range(uint8_t* out, uint64_t first_bits, int64_t count)
{
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < count; ++i) out[i] = rne_e4m3(bits_f32((uint32_t)(first_bits + (uint64_t)i)));
}

void or_up_e4m3_array(float* out, const uint8_t* in, int64_t count)
{
    for (int64_t i = 0; i < count; ++i) out[i] = up_e4m3(in[i]);
}

/* q[i] = e4m3(up(src[i]) * scale_inv), one f32 multiply then one rounding;
 * *amax = max |up(src[i])| over the unscaled values (+0 when count == 0). */
void or_fp8_quantize(uint8_t* q, float* amax, const void* src, int dtype, float scale_inv, int64_t count)
{
    float mx = 0.0f;
    for (int64_t i = 0; i < count; ++i) {
        float v = load_up(src, dtype, i);
        q[i] = rne_e4m3(v * scale_inv);
        float a = fabsf(v);
        if (a > mx) mx = a;
    }
    *amax = mx;
}

/* The scaled matmuls.  acc = chain over the contracted index of
 * up(a_i) * up(b_i) (exact products of e4m3 values), then
 * v = acc * (scale_a * scale_b) in f32, then (+ bias in f32), then one
 * rounding to out_dtype.  Forward y[m,n] (xq [M,K], wq [K,N]); dX[m,k] from
 * gq [M,N] and wq; dW[k,n] from xq and gq with the dW chunk tree over rows. */
int or_fp8_forward_rows(void* y_rows, const uint8_t* xq, const uint8_t* wq, const void* bias,
                        float sx, float sw, const int64_t* rows, int64_t nrows, int64_t m, int64_t k,
                        int64_t n, int out_dtype)
{
    const float s = sx * sw;
    #pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t r = rows ? rows[i] : i;
        if (r < 0 || r >= m) continue;
        for (int64_t j = 0; j < n; ++j) {
            float acc = 0.0f;
            for (int64_t kk = 0; kk < k; ++kk)
                acc = fmaf(up_e4m3(xq[r * k + kk]), up_e4m3(wq[kk * n + j]), acc);
            float v = acc * s;
            if (bias) v = v + load_up(bias, out_dtype, j);
            store_down(y_rows, out_dtype, i * n + j, v);
        }
    }
    return 0;
}

int or_fp8_backward_dx_rows(void* dx_rows, const uint8_t* gq, const uint8_t* wq, float sg, float sw,
                            const int64_t* rows, int64_t nrows, int64_t m, int64_t k, int64_t n, int out_dtype)
{
    const float s = sg * sw;
    #pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t r = rows ? rows[i] : i;
        if (r < 0 || r >= m) continue;
        for (int64_t kk = 0; kk < k; ++kk) {
            float acc = 0.0f;
            for (int64_t j = 0; j < n; ++j)
                acc = fmaf(up_e4m3(gq[r * n + j]), up_e4m3(wq[kk * n + j]), acc);
            store_down(dx_rows, out_dtype, i * k + kk, acc * s);
        }
    }
    return 0;
}

int or_fp8_backward_dw(void* dw, const uint8_t* xq, const uint8_t* gq, float sx, float sg,
                       int64_t m, int64_t k, int64_t n, int out_dtype, int64_t chunk)
{
    if (chunk <= 0) return -2;
    const float s = sx * sg;
    int64_t J = (m + chunk - 1) / chunk;
    int failed = 0;
    #pragma omp parallel
    {
        float* parts = (float*)malloc((size_t)(J > 0 ? J : 1) * sizeof(float));
        if (!parts) failed = 1;
        #pragma omp for collapse(2) schedule(dynamic, 16)
        for (int64_t kk = 0; kk < k; ++kk)
            for (int64_t j = 0; j < n; ++j) {
                if (!parts) continue;
                for (int64_t c = 0; c < J; ++c) {
                    float acc = 0.0f;
                    int64_t r_end = (c + 1) * chunk < m ? (c + 1) * chunk : m;
                    for (int64_t r = c * chunk; r < r_end; ++r)
                        acc = fmaf(up_e4m3(xq[r * k + kk]), up_e4m3(gq[r * n + j]), acc);
                    parts[c] = acc;
                }
                store_down(dw, out_dtype, kk * n + j, tree_sum(parts, J) * s);
            }
        free(parts);
    }
    return failed ? -1 : 0;
}

/* ------------------------------------------------------------------------ */
/* Grouped per-row-expert passes.  X[M,K], W[E,N,K], row_experts[M] (U32),   */
/* Y[M,N], dY[M,N], dX[M,K], dW[E,N,K] (always f32).                         */
/* ------------------------------------------------------------------------ */

/* Stable segmentation: perm lists the rows of expert 0, then expert 1, ...,
 * then every padding row (id >= E), each group in ascending row index;
 * offsets[g] is where group g starts (g = 0..E, group E = padding) and
 * offsets[E+1] = M. */
int or_grouped_segment(const uint32_t* ids, int64_t m, int64_t e, uint32_t* perm, uint32_t* offsets)
{
    int64_t pos = 0;
    for (int64_t g = 0; g <= e; ++g) {
        offsets[g] = (uint32_t)pos;
        for (int64_t r = 0; r < m; ++r) {
            int64_t id = ids[r] < (uint64_t)e ? (int64_t)ids[r] : e;
            if (id == g) perm[pos++] = (uint32_t)r;
        }
    }
    offsets[e + 1] = (uint32_t)pos;
    return pos == m ? 0 : -1;
}

/* Y[r,j] = rne( chain_k X[r,k] * W[e(r), j, k] ) for e(r) < E, else +0. */
int or_grouped_forward_rows(void* y_rows, const void* x, const void* w, const uint32_t* ids,
                            const int64_t* rows, int64_t nrows, int64_t m, int64_t k, int64_t n,
                            int64_t e, int dtype, int out_f32)
{
    int out_t = out_f32 ? OR_F32 : dtype;
    #pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t r = rows ? rows[i] : i;
        if (r < 0 || r >= m) continue;
        uint32_t id = ids[r];
        for (int64_t j = 0; j < n; ++j) {
            float acc = 0.0f;
            if (id < (uint64_t)e) {
                const int64_t wbase = ((int64_t)id * n + j) * k;
                for (int64_t kk = 0; kk < k; ++kk)
                    acc = fmaf(load_up(x, dtype, r * k + kk), load_up(w, dtype, wbase + kk), acc);
            }
            store_down(y_rows, out_t, i * n + j, acc); /* padding rows: +0 */
        }
    }
    return 0;
}

int or_grouped_forward(void* y, const void* x, const void* w, const uint32_t* ids,
                       int64_t m, int64_t k, int64_t n, int64_t e, int dtype, int out_f32)
{
    return or_grouped_forward_rows(y, x, w, ids, NULL, m, m, k, n, e, dtype, out_f32);
}

/* dinput: dX[r,kk] = rne( chain_n dY[r,n] * W[e(r), n, kk] ), +0 for padding. */
int or_grouped_dinput_rows(void* dx_rows, const void* w, const void* dy, const uint32_t* ids,
                           const int64_t* rows, int64_t nrows, int64_t m, int64_t k, int64_t n,
                           int64_t e, int dtype, int out_f32)
{
    int out_t = out_f32 ? OR_F32 : dtype;
    #pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t r = rows ? rows[i] : i;
        if (r < 0 || r >= m) continue;
        uint32_t id = ids[r];
        for (int64_t kk = 0; kk < k; ++kk) {
            float acc = 0.0f;
            if (id < (uint64_t)e) {
                for (int64_t j = 0; j < n; ++j)
                    acc = fmaf(load_up(dy, dtype, r * n + j),
                               load_up(w, dtype, ((int64_t)id * n + j) * k + kk), acc);
            }
            store_down(dx_rows, out_t, i * k + kk, acc);
        }
    }
    return 0;
}

/* dweights on a list of (expert, n) pairs: dW_sel[i, kk] = tree_c p_c with p_c
 * the chain, over the rows of expert g = sel_e[i] taken in ascending row index
 * and cut into chunks of `chunk` rows counted from the expert's first row, of
 * dY[r, j] * X[r, kk] (j = sel_n[i]).  f32 result.  An expert with no rows gets
 * +0.  Padding rows contribute nothing.  Passing sel_e = sel_n = NULL and
 * nsel = E*N computes the whole dW[E,N,K]. */
int or_grouped_dweights_sel(float* dw_sel, const void* x, const void* dy, const uint32_t* ids,
                            const int64_t* sel_e, const int64_t* sel_n, int64_t nsel,
                            int64_t m, int64_t k, int64_t n, int64_t e, int dtype, int64_t chunk)
{
    if (chunk <= 0) return -2;
    uint32_t* perm = (uint32_t*)malloc((size_t)(m > 0 ? m : 1) * sizeof(uint32_t));
    uint32_t* offs = (uint32_t*)malloc((size_t)(e + 2) * sizeof(uint32_t));
    float* xf = widen(x, dtype, m * k);
    if (!perm || !offs || !xf) { free(perm); free(offs); free(xf); return -1; }
    or_grouped_segment(ids, m, e, perm, offs);
    int failed = 0;
    #pragma omp parallel
    {
        int64_t jmax = m / chunk + 2;
        float* parts = (float*)malloc((size_t)jmax * k * sizeof(float));
        float* col = (float*)malloc((size_t)jmax * sizeof(float));
        if (!parts || !col) failed = 1;
        #pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < nsel; ++i) {
            if (!parts || !col) continue;
            int64_t g = sel_e ? sel_e[i] : i / n;
            int64_t j = sel_n ? sel_n[i] : i % n;
            if (g < 0 || g >= e || j < 0 || j >= n) continue;
            int64_t s = offs[g], cnt = (int64_t)offs[g + 1] - s;
            int64_t J = (cnt + chunk - 1) / chunk;
            /* parts[c*K + kk] runs the chain of chunk c for output (g, j, kk) */
            for (int64_t c = 0; c < J; ++c) {
                float* p = parts + c * k;
                for (int64_t kk = 0; kk < k; ++kk) p[kk] = 0.0f;
                int64_t l_end = (c + 1) * chunk < cnt ? (c + 1) * chunk : cnt;
                for (int64_t l = c * chunk; l < l_end; ++l) {
                    int64_t r = perm[s + l];
                    float gy = load_up(dy, dtype, r * n + j);
                    const float* xrow = xf + r * k;
                    for (int64_t kk = 0; kk < k; ++kk) p[kk] = fmaf(gy, xrow[kk], p[kk]);
                }
            }
            for (int64_t kk = 0; kk < k; ++kk) {
                for (int64_t c = 0; c < J; ++c) col[c] = parts[c * k + kk];
                dw_sel[i * k + kk] = tree_sum(col, J);
            }
        }
        free(parts); free(col);
    }
    free(perm); free(offs); free(xf);
    return failed ? -1 : 0;
}

int or_grouped_dweights(float* dw, const void* x, const void* dy, const uint32_t* ids,
                        int64_t m, int64_t k, int64_t n, int64_t e, int dtype, int64_t chunk)
{
    return or_grouped_dweights_sel(dw, x, dy, ids, NULL, NULL, e * n, m, k, n, e, dtype, chunk);
}
