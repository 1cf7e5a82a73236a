// Scalar tier: fixed-order f32 fmaf chains, one output element per accumulator.
//
// Contract (sgemm-bi 0.1.1.post2, "Determinism contracts", row "f32 / typed
// scalar"): bf16/f16 operands are widened exactly to f32, the f32 kernel runs,
// and the result is rounded once to nearest-even.  Each output's chain is
//     acc = +0.0f;  for l = 0, 1, ..., L-1:  acc = fmaf(a_l, b_l, acc)
// and the forward adds the bias to acc in f32 before the single rounding
// (ViperLLM ffma.py, _FFMAAddmm.forward).  Elements past the end of the
// contraction are staged as zeros on both operands; fmaf(0, 0, acc) returns acc
// exactly because acc is never -0 (it starts at +0 and a rounded sum is -0 only
// when both addends are -0), so padding does not change a bit.
//
// Tiling: a 256-thread CTA computes a 128 x 128 output tile; each thread owns
// 8 x 8 outputs (rows {4ty..4ty+3, 64+4ty..}, cols {4tx.., 64+4tx..}) and keeps
// their accumulators in registers, as pairs of adjacent columns: the paired
// FP32 FMA (fma.rn.f32x2) performs two independent round-to-nearest fmaf on
// the two lanes, so each accumulator still follows its own chain while the
// instruction count halves.  Operands are loaded with 16-byte vector loads
// (when sizes and alignment allow), widened, and staged through a double
// buffer in shared memory, 16 contraction steps at a time; every A value is
// stored twice, so one 16-byte shared load gives two (a, a) lane pairs.
//
// dW reduction over rows (the weight gradient): rows are cut into chunks of
// BI_DW_CHUNK rows from row 0 (per expert, from the expert's first row, for the
// grouped dweights).  One CTA computes one chunk's chain for its tile; a second
// kernel adds the chunk partials with the fixed pairwise tree (adjacent pairs,
// odd last partial carried), evaluated as a binary counter, which performs the
// same additions on the same operands.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "bi_internal.h"

namespace bi {
namespace {

constexpr int TM = 128, TN = 128, TK = 16, NT = 256, PAD = 4;

template <typename T> struct Elem;
template <> struct Elem<float> {
    static __device__ __forceinline__ float up(float v) { return v; }
    static __device__ __forceinline__ float down(float v) { return v; }
};
template <> struct Elem<__nv_bfloat16> {
    static __device__ __forceinline__ float up(__nv_bfloat16 v) { return __bfloat162float(v); }
    static __device__ __forceinline__ __nv_bfloat16 down(float v) { return __float2bfloat16_rn(v); }
};
template <> struct Elem<__half> {
    static __device__ __forceinline__ float up(__half v) { return __half2float(v); }
    static __device__ __forceinline__ __half down(float v) { return __float2half_rn(v); }
};

// Load 8 consecutive elements starting at p (widened to f32).  VEC: p is
// 16-byte aligned and all 8 are in range; otherwise `avail` of them are valid.
template <typename T, bool VEC>
__device__ __forceinline__ void load8(const T* p, int avail, float (&v)[8]) {
    if (VEC && avail >= 8) {
        if (sizeof(T) == 4) {
            const float4 a = __ldg(reinterpret_cast<const float4*>(p));
            const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
            v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
            v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
        } else {
            const uint4 a = __ldg(reinterpret_cast<const uint4*>(p));
            const T* h = reinterpret_cast<const T*>(&a);
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = Elem<T>::up(h[i]);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = i < avail ? Elem<T>::up(p[i]) : 0.0f;
    }
}

// Shared tile: s[l][i] with l the contraction step, i the row or column; A
// holds each value twice (a[l][2r] = a[l][2r+1] = A value of tile row r).
template <int TMV>
struct SmemT {
    float a[2][TK][2 * TMV + PAD];
    float b[2][TK][TN + PAD];
};
using Smem = SmemT<TM>;

// acc = (fmaf(a.lo, b.lo, acc.lo), fmaf(a.hi, b.hi, acc.hi)), each rounded to nearest.
__device__ __forceinline__ void fma2(uint64_t& acc, uint64_t a, uint64_t b) {
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b));
}
// Accumulator (i, j) of a thread: lane j % 2 of pair acc[i][j / 2].
__device__ __forceinline__ float acc_lane(const uint64_t (&acc)[8][4], int i, int j) {
    const uint64_t v = acc[i][j >> 1];
    return __uint_as_float(static_cast<uint32_t>((j & 1) ? (v >> 32) : v));
}

// ------------------------------------------------------------------ cp.async staging

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// 16-byte global -> shared copy; src_bytes = 0 writes zeros (src is not read).
__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// One block of the operands as they lie in global memory (raw element type),
// filled by cp.async: A rows of TK elements, B as TK rows of TN columns, or
// (BT) TN columns of TK elements; every row padded by 16 bytes, which keeps
// the widening reads conflict-free.
template <typename T, int TMV, bool BT>
struct RawT {
    static constexpr int PADE = 16 / sizeof(T);
    T a[TMV][TK + PADE];
    T b[BT ? TN : TK][(BT ? TK : TN) + PADE];
};
constexpr int RAW_STAGES = 3;
// dW: both operands are [rows][out] with out contiguous: TK rows of TM / TN outs.
template <typename T>
struct RawDwT {
    static constexpr int PADE = 16 / sizeof(T);
    T a[TK][TM + PADE];
    T b[TK][TN + PADE];
};

// 8 consecutive raw elements from shared memory, widened (p 16-byte aligned).
template <typename T>
__device__ __forceinline__ void smem_load8(const T* p, float (&v)[8]) {
    if (sizeof(T) == 4) {
        const float4 a = reinterpret_cast<const float4*>(p)[0];
        const float4 b = reinterpret_cast<const float4*>(p)[1];
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
        const uint4 a = *reinterpret_cast<const uint4*>(p);
        const T* h = reinterpret_cast<const T*>(&a);
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = Elem<T>::up(h[i]);
    }
}

// 8x8 micro-tile product over one staged block: each accumulator (i, j)
// chains over l ascending; pair q of row i holds columns 2q and 2q+1.
template <int TMV = TM>
__device__ __forceinline__ void mma_block(const float (*as)[2 * TMV + PAD], const float (*bs)[TN + PAD],
                                          int ty, int tx, uint64_t (&acc)[8][4]) {
#pragma unroll
    for (int l = 0; l < TK; ++l) {
        const ulonglong2 a0 = *reinterpret_cast<const ulonglong2*>(&as[l][ty * 8]);
        const ulonglong2 a1 = *reinterpret_cast<const ulonglong2*>(&as[l][ty * 8 + 4]);
        const ulonglong2 a2 = *reinterpret_cast<const ulonglong2*>(&as[l][TMV + ty * 8]);
        const ulonglong2 a3 = *reinterpret_cast<const ulonglong2*>(&as[l][TMV + ty * 8 + 4]);
        const ulonglong2 b0 = *reinterpret_cast<const ulonglong2*>(&bs[l][tx * 4]);
        const ulonglong2 b1 = *reinterpret_cast<const ulonglong2*>(&bs[l][64 + tx * 4]);
        const uint64_t a[8] = {a0.x, a0.y, a1.x, a1.y, a2.x, a2.y, a3.x, a3.y};
        const uint64_t b[4] = {b0.x, b0.y, b1.x, b1.y};
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int q = 0; q < 4; ++q) fma2(acc[i][q], a[i], b[q]);
    }
}

// Thread (ty, tx) owns rows {4ty..4ty+3, TMV/2+4ty..} and columns {4tx..4tx+3, 64+4tx..}.
template <int TMV = TM>
__device__ __forceinline__ int mrow(int ty, int i) { return i < 4 ? ty * 4 + i : TMV / 2 + ty * 4 + (i - 4); }

// ------------------------------------------------------------------ rows kernels

struct RowsArgs {
    void* out;
    const void* a;      // [R or M, L], contraction contiguous
    const void* b;      // [L, C] or [C, L] (per expert when grouped)
    const void* bias;   // [C] or null
    int64_t R, L, C;
    int64_t E;
    const uint32_t* seg;
    const uint32_t* perm;
};

// out[r, c] = down( chain_l a[r, l] * b(l, c) (+ bias[c]) )
// TMV = tile height (128 or 64); 2*TMV threads, each owning 8 x 8 outputs.
template <typename T, bool BT, bool GROUPED, bool VEC, int TMV>
__global__ void __launch_bounds__(2 * TMV, TMV == 128 ? 1 : (VEC ? 4 : 3)) scalar_rows_kernel(const RowsArgs p) {
    constexpr int NTV = 2 * TMV;
    constexpr int SL = (TK * TN) / (NTV * 8);  // 8-element B slots per thread
    extern __shared__ __align__(16) uint8_t smem_rows[];
    SmemT<TMV>& sm = *reinterpret_cast<SmemT<TMV>*>(smem_rows);
    const int tid = threadIdx.x, ty = tid / 16, tx = tid % 16;
    const T* A = static_cast<const T*>(p.a);
    const T* B = static_cast<const T*>(p.b);
    const int64_t L = p.L, C = p.C;
    const int64_t c0 = static_cast<int64_t>(blockIdx.y) * TN;

    // rows of this tile: r0 + i (dense) or sorted positions of one expert
    int64_t r0 = static_cast<int64_t>(blockIdx.x) * TMV;
    int64_t rvalid = p.R - r0;
    uint32_t sbase = 0;
    if (GROUPED) {
        int64_t t = blockIdx.x;
        int g = 0;
        bool found = false;
        for (; g < p.E; ++g) {
            const int64_t cnt = p.seg[g + 1] - p.seg[g];
            const int64_t tiles = (cnt + TMV - 1) / TMV;
            if (t < tiles) { found = true; break; }
            t -= tiles;
        }
        if (!found) return;
        const int64_t cnt = p.seg[g + 1] - p.seg[g];
        sbase = p.seg[g] + static_cast<uint32_t>(t * TMV);
        rvalid = cnt - t * TMV;
        B += static_cast<int64_t>(g) * C * L;
    }
    if (rvalid > TMV) rvalid = TMV;

    // global -> register staging of one TK block
    // A: TMV rows x 16 steps; a warp covers 32 different rows with the same
    // 8-step half, so its transposing stores hit 32 different banks
    const int a_row = tid % TMV, a_seg = (tid / TMV) * 8;
    int64_t a_src_row = -1;
    if (a_row < rvalid) a_src_row = GROUPED ? static_cast<int64_t>(p.perm[sbase + a_row]) : r0 + a_row;
    float ra[8], rb[SL][8];
    auto load_a = [&](int64_t l0) {
        const int64_t l = l0 + a_seg;
        const int avail = a_src_row < 0 ? 0 : static_cast<int>(lmin(8, lmax(0, L - l)));
        load8<T, VEC>(A + (a_src_row < 0 ? 0 : a_src_row * L + l), avail, ra);
    };
    auto load_b = [&](int64_t l0) {
#pragma unroll
        for (int q = 0; q < SL; ++q) {
            const int e = tid + q * NTV;  // 0..255
            if (BT) {  // b(l, c) = B[c * L + l]: 128 cols x 16 steps
                const int c = e % TN, s = (e / TN) * 8;
                const int64_t gc = c0 + c, l = l0 + s;
                const int avail = gc < C ? static_cast<int>(lmin(8, lmax(0, L - l))) : 0;
                load8<T, VEC>(B + (avail ? gc * L + l : 0), avail, rb[q]);
            } else {   // b(l, c) = B[l * C + c]: 16 steps x 128 cols
                const int l = e / 16, s = (e % 16) * 8;
                const int64_t gl = l0 + l, gc = c0 + s;
                const int avail = gl < L ? static_cast<int>(lmin(8, lmax(0, C - gc))) : 0;
                load8<T, VEC>(B + (avail ? gl * C + gc : 0), avail, rb[q]);
            }
        }
    };
    auto store = [&](int buf) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            *reinterpret_cast<float2*>(&sm.a[buf][a_seg + i][2 * a_row]) = make_float2(ra[i], ra[i]);
#pragma unroll
        for (int q = 0; q < SL; ++q) {
            const int e = tid + q * NTV;
            if (BT) {
                const int c = e % TN, s = (e / TN) * 8;
#pragma unroll
                for (int i = 0; i < 8; ++i) sm.b[buf][s + i][c] = rb[q][i];
            } else {
                const int l = e / 16, s = (e % 16) * 8;
                *reinterpret_cast<float4*>(&sm.b[buf][l][s]) = make_float4(rb[q][0], rb[q][1], rb[q][2], rb[q][3]);
                *reinterpret_cast<float4*>(&sm.b[buf][l][s + 4]) = make_float4(rb[q][4], rb[q][5], rb[q][6], rb[q][7]);
            }
        }
    };

    uint64_t acc[8][4];  // +0.0f in both lanes
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[i][q] = 0;

    const int64_t nkb = (L + TK - 1) / TK;
    if constexpr (VEC) {
        // cp.async ring of RAW_STAGES raw blocks; block kb+1 is widened into the
        // f32 tiles while block kb is multiplied (one barrier per block)
        using Raw = RawT<T, TMV, BT>;
        Raw* raw = reinterpret_cast<Raw*>(smem_rows + sizeof(SmemT<TMV>));
        constexpr int EPC = 16 / static_cast<int>(sizeof(T));  // elements per 16-byte chunk
        constexpr int ACPR = TK / EPC;                         // A chunks per row
        constexpr int ACH = TMV * ACPR;
        constexpr int AQ = (ACH + NTV - 1) / NTV;
        constexpr int BCH = TK * TN / EPC;
        constexpr int BQ = BCH / NTV;
        int64_t a_src[AQ];  // source row of this thread's A chunks, or -1
#pragma unroll
        for (int q = 0; q < AQ; ++q) {
            const int e = tid + q * NTV, row = e / ACPR;
            a_src[q] = -1;
            if (e < ACH && row < rvalid) a_src[q] = GROUPED ? static_cast<int64_t>(p.perm[sbase + row]) : r0 + row;
        }
        auto issue = [&](int64_t kb, int slot) {
            if (kb < nkb) {
                const int64_t l0 = kb * TK;
                Raw& r = raw[slot];
#pragma unroll
                for (int q = 0; q < AQ; ++q) {
                    const int e = tid + q * NTV;
                    if (e < ACH) {
                        const int row = e / ACPR, ch = e % ACPR;
                        const int64_t l = l0 + ch * EPC;
                        const bool ok = a_src[q] >= 0 && l < L;
                        cp_async16(&r.a[row][ch * EPC], ok ? static_cast<const void*>(A + a_src[q] * L + l) : A,
                                   ok ? 16u : 0u);
                    }
                }
#pragma unroll
                for (int q = 0; q < BQ; ++q) {
                    const int e = tid + q * NTV;
                    if (BT) {  // column c: TK elements of B[c * L + l]
                        const int c = e / ACPR, ch = e % ACPR;
                        const int64_t gc = c0 + c, l = l0 + ch * EPC;
                        const bool ok = gc < C && l < L;
                        cp_async16(&r.b[c][ch * EPC], ok ? static_cast<const void*>(B + gc * L + l) : B, ok ? 16u : 0u);
                    } else {   // step l: TN elements of B[l * C + c]
                        constexpr int CPR = TN / EPC;
                        const int l = e / CPR, ch = e % CPR;
                        const int64_t gl = l0 + l, gc = c0 + ch * EPC;
                        const bool ok = gl < L && gc < C;
                        cp_async16(&r.b[l][ch * EPC], ok ? static_cast<const void*>(B + gl * C + gc) : B, ok ? 16u : 0u);
                    }
                }
            }
            cp_async_commit();  // an empty group past the end keeps the count uniform
        };
        auto widen = [&](int slot, int buf) {
            const Raw& r = raw[slot];
            {   // A: row a_row, steps a_seg..a_seg+7, each value stored twice
                float v[8];
                smem_load8<T>(&r.a[a_row][a_seg], v);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    *reinterpret_cast<float2*>(&sm.a[buf][a_seg + i][2 * a_row]) = make_float2(v[i], v[i]);
            }
            constexpr int EB = TK * TN / NTV;  // B elements per thread (8 or 16)
            if (BT) {  // column c, steps lseg..lseg+EB-1, transposed into sm.b[l][c]
                const int c = tid % TN, lseg = (tid / TN) * EB;
#pragma unroll
                for (int h = 0; h < EB; h += 8) {
                    float v[8];
                    smem_load8<T>(&r.b[c][lseg + h], v);
#pragma unroll
                    for (int i = 0; i < 8; ++i) sm.b[buf][lseg + h + i][c] = v[i];
                }
            } else {   // step l, columns cseg..cseg+EB-1
                const int l = tid / (TN / EB), cseg = (tid % (TN / EB)) * EB;
#pragma unroll
                for (int h = 0; h < EB; h += 8) {
                    float v[8];
                    smem_load8<T>(&r.b[l][cseg + h], v);
                    *reinterpret_cast<float4*>(&sm.b[buf][l][cseg + h]) = make_float4(v[0], v[1], v[2], v[3]);
                    *reinterpret_cast<float4*>(&sm.b[buf][l][cseg + h + 4]) = make_float4(v[4], v[5], v[6], v[7]);
                }
            }
        };
        static_assert(RAW_STAGES == 3, "the waits below assume three raw stages");
        issue(0, 0);
        issue(1, 1);
        cp_async_wait<1>();
        __syncthreads();
        widen(0, 0);
        issue(2, 2);
        for (int64_t kb = 0; kb < nkb; ++kb) {
            cp_async_wait<1>();  // block kb+1 has landed (this thread's copies)
            __syncthreads();     // ... everyone's; block kb widened; tiles of kb-1 no longer read
            if (kb + 1 < nkb) widen(static_cast<int>((kb + 1) % RAW_STAGES), static_cast<int>((kb + 1) & 1));
            issue(kb + RAW_STAGES, static_cast<int>(kb % RAW_STAGES));  // block kb's slot, already widened
            mma_block<TMV>(sm.a[kb & 1], sm.b[kb & 1], ty, tx, acc);
        }
        cp_async_wait<0>();
    } else {
        load_a(0); load_b(0); store(0);
        __syncthreads();
        int buf = 0;
        for (int64_t kb = 0; kb < nkb; ++kb) {
            const bool more = kb + 1 < nkb;
            if (more) { load_a((kb + 1) * TK); load_b((kb + 1) * TK); }
            mma_block<TMV>(sm.a[buf], sm.b[buf], ty, tx, acc);
            if (more) store(buf ^ 1);
            __syncthreads();
            buf ^= 1;
        }
    }

    // epilogue: (+ bias), one rounding, store
    T* out = static_cast<T*>(p.out);
    const T* bias = static_cast<const T*>(p.bias);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int lr = mrow<TMV>(ty, i);
        if (lr >= rvalid) continue;
        const int64_t orow = GROUPED ? static_cast<int64_t>(p.perm[sbase + lr]) : r0 + lr;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int64_t c = c0 + mrow(tx, j);
            if (c >= C) continue;
            float v = acc_lane(acc, i, j);
            if (bias) v = v + Elem<T>::up(bias[c]);
            out[orow * C + c] = Elem<T>::down(v);
        }
    }
}

// ------------------------------------------------------------------ narrow rows kernel

// Outputs at most 64 columns wide (an output dimension below the tensor-core
// threshold), and small outputs that the 128-column tiles would spread over
// fewer CTAs than the GPU has SMs: 16 x 64 tiles on 256 threads (column tile
// blockIdx.y), 2 x 2 outputs per thread, so a small output still spreads over
// many CTAs.  Same chains as above: each output is fmaf over l ascending from
// +0 (paired FMA lanes), then (+ bias) and one rounding.  Dense only.
constexpr int NW_TM = 16, NW_TN = 64, NW_TK = 32;

template <typename T, bool BT>
__global__ void __launch_bounds__(256) scalar_rows_narrow_kernel(const RowsArgs p) {
    __shared__ __align__(16) float as[2][NW_TK][2 * NW_TM + 4];  // A doubled: [l][2r], [l][2r+1]
    __shared__ __align__(16) float bs[2][NW_TK][NW_TN + 4];
    const int tid = threadIdx.x, ty = tid >> 5, tx = tid & 31;  // rows 2ty, 2ty+1; cols 2tx, 2tx+1
    const T* A = static_cast<const T*>(p.a);
    const T* B = static_cast<const T*>(p.b);
    const int64_t L = p.L, C = p.C;
    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * NW_TM;
    const int64_t c0 = static_cast<int64_t>(blockIdx.y) * NW_TN;
    const int64_t rvalid = lmin(NW_TM, p.R - r0);
    // staging: A 16 rows x 32 steps (2 per thread), B 32 steps x 64 cols (8 per thread)
    const int a_row = tid >> 4, a_l = (tid & 15) * 2;
    const int b_i = BT ? (tid >> 2) : (tid >> 3);              // BT: column; else step
    const int b_j = BT ? (tid & 3) * 8 : (tid & 7) * 8;        // BT: first step; else first column
    float ra[2], rb[8];
    auto load = [&](int64_t l0) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int64_t l = l0 + a_l + i;
            ra[i] = (a_row < rvalid && l < L) ? Elem<T>::up(A[(r0 + a_row) * L + l]) : 0.0f;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (BT) {  // b(l, c) = B[c * L + l]
                const int64_t c = c0 + b_i, l = l0 + b_j + i;
                rb[i] = (c < C && l < L) ? Elem<T>::up(B[c * L + l]) : 0.0f;
            } else {   // b(l, c) = B[l * C + c]
                const int64_t l = l0 + b_i, c = c0 + b_j + i;
                rb[i] = (l < L && c < C) ? Elem<T>::up(B[l * C + c]) : 0.0f;
            }
        }
    };
    auto store = [&](int buf) {
#pragma unroll
        for (int i = 0; i < 2; ++i)
            *reinterpret_cast<float2*>(&as[buf][a_l + i][2 * a_row]) = make_float2(ra[i], ra[i]);
        if (BT) {
#pragma unroll
            for (int i = 0; i < 8; ++i) bs[buf][b_j + i][b_i] = rb[i];
        } else {
            *reinterpret_cast<float4*>(&bs[buf][b_i][b_j]) = make_float4(rb[0], rb[1], rb[2], rb[3]);
            *reinterpret_cast<float4*>(&bs[buf][b_i][b_j + 4]) = make_float4(rb[4], rb[5], rb[6], rb[7]);
        }
    };
    uint64_t acc[2] = {0, 0};  // rows 2ty, 2ty+1; lanes = cols 2tx, 2tx+1
    const int64_t nkb = (L + NW_TK - 1) / NW_TK;
    load(0);
    store(0);
    __syncthreads();
    for (int64_t kb = 0; kb < nkb; ++kb) {
        const int buf = static_cast<int>(kb & 1);
        const bool more = kb + 1 < nkb;
        if (more) load((kb + 1) * NW_TK);
#pragma unroll
        for (int l = 0; l < NW_TK; ++l) {
            const ulonglong2 a = *reinterpret_cast<const ulonglong2*>(&as[buf][l][4 * ty]);
            const uint64_t b = *reinterpret_cast<const uint64_t*>(&bs[buf][l][2 * tx]);
            fma2(acc[0], a.x, b);
            fma2(acc[1], a.y, b);
        }
        if (more) store(buf ^ 1);
        __syncthreads();
    }
    T* out = static_cast<T*>(p.out);
    const T* bias = static_cast<const T*>(p.bias);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int lr = 2 * ty + i;
        if (lr >= rvalid) continue;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int64_t c = c0 + 2 * tx + j;
            if (c >= C) continue;
            float v = __uint_as_float(static_cast<uint32_t>(j ? (acc[i] >> 32) : acc[i]));
            if (bias) v = v + Elem<T>::up(bias[c]);
            out[(r0 + lr) * C + c] = Elem<T>::down(v);
        }
    }
}

// ------------------------------------------------------------------ dW kernels

struct DwArgs {
    void* out;          // final output (direct mode) [R, C]
    int out_f32;
    float* partials;    // [chunks, R, C] or null for direct mode
    const void* a;      // [M, R] (row-major over m, r contiguous)
    const void* b;      // [M, C]
    int64_t M, R, C;
    int64_t E;
    const uint32_t* seg;
    const uint32_t* perm;
};

// partial[z][r][c] = chain over the rows of chunk z of a[m, r] * b[m, c]
template <typename T, bool GROUPED, bool VEC>
__global__ void __launch_bounds__(NT, 2) scalar_dw_chunk_kernel(const DwArgs p) {
    extern __shared__ __align__(16) uint8_t smem_dw[];
    Smem& sm = *reinterpret_cast<Smem*>(smem_dw);
    const int tid = threadIdx.x, ty = tid / 16, tx = tid % 16;
    const T* A = static_cast<const T*>(p.a);
    const T* Bm = static_cast<const T*>(p.b);
    const int64_t R = p.R, C = p.C;
    const int64_t r0 = static_cast<int64_t>(blockIdx.y) * TM;
    const int64_t c0 = static_cast<int64_t>(blockIdx.x) * TN;
    const int64_t z = blockIdx.z;

    // rows of this chunk: positions [pos0, pos0 + cnt) (dense: rows; grouped: sorted positions)
    int64_t pos0, cnt;
    if (GROUPED) {
        int64_t t = z;
        int g = 0;
        bool found = false;
        for (; g < p.E; ++g) {
            const int64_t n_g = p.seg[g + 1] - p.seg[g];
            const int64_t j_g = (n_g + BI_DW_CHUNK - 1) / BI_DW_CHUNK;
            if (t < j_g) { found = true; break; }
            t -= j_g;
        }
        if (!found) return;
        const int64_t n_g = p.seg[g + 1] - p.seg[g];
        pos0 = p.seg[g] + t * BI_DW_CHUNK;
        cnt = lmin(BI_DW_CHUNK, n_g - t * BI_DW_CHUNK);
    } else {
        pos0 = z * BI_DW_CHUNK;
        cnt = lmin(BI_DW_CHUNK, p.M - pos0);
    }

    // both operands are [rows, out] with out contiguous: 16 rows x 128 outs each
    const int l_ld = tid / 16, s_ld = (tid % 16) * 8;
    float ra[8], rb[8];
    auto load = [&](int64_t l0) {
        const int64_t l = l0 + l_ld;
        int64_t row = -1;
        if (l < cnt) row = GROUPED ? static_cast<int64_t>(p.perm[pos0 + l]) : pos0 + l;
        const int av_a = row < 0 ? 0 : static_cast<int>(lmin(8, lmax(0, R - (r0 + s_ld))));
        const int av_b = row < 0 ? 0 : static_cast<int>(lmin(8, lmax(0, C - (c0 + s_ld))));
        load8<T, VEC>(A + (av_a ? row * R + r0 + s_ld : 0), av_a, ra);
        load8<T, VEC>(Bm + (av_b ? row * C + c0 + s_ld : 0), av_b, rb);
    };
    // A doubled: this thread's 64 contiguous bytes as four 16-byte pieces,
    // written in an order rotated by the thread index so the 16 threads of a
    // row hit different banks in each store instruction
    const int rot = tid & 3;
    auto store = [&](int buf) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int c = (q + rot) & 3;
            const float v0 = c == 0 ? ra[0] : c == 1 ? ra[2] : c == 2 ? ra[4] : ra[6];
            const float v1 = c == 0 ? ra[1] : c == 1 ? ra[3] : c == 2 ? ra[5] : ra[7];
            *reinterpret_cast<float4*>(&sm.a[buf][l_ld][2 * s_ld + 4 * c]) = make_float4(v0, v0, v1, v1);
        }
        *reinterpret_cast<float4*>(&sm.b[buf][l_ld][s_ld]) = make_float4(rb[0], rb[1], rb[2], rb[3]);
        *reinterpret_cast<float4*>(&sm.b[buf][l_ld][s_ld + 4]) = make_float4(rb[4], rb[5], rb[6], rb[7]);
    };

    uint64_t acc[8][4];  // +0.0f in both lanes
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[i][q] = 0;

    const int64_t nkb = (cnt + TK - 1) / TK;
    if (VEC && nkb > 0) {
        // cp.async ring of RAW_STAGES raw blocks, as in the rows kernel
        using Raw = RawDwT<T>;
        Raw* raw = reinterpret_cast<Raw*>(smem_dw + sizeof(Smem));
        constexpr int EPC = 16 / static_cast<int>(sizeof(T));
        constexpr int CPR = TM / EPC;            // chunks per row (TM == TN)
        constexpr int Q = TK * CPR / NT;         // chunks per thread and operand (1 or 2)
        auto issue = [&](int64_t kb, int slot) {
            if (kb < nkb) {
                Raw& r = raw[slot];
#pragma unroll
                for (int q = 0; q < Q; ++q) {
                    const int e = tid + q * NT, l = e / CPR, ch = e % CPR;
                    const int64_t lr = kb * TK + l;
                    int64_t row = -1;
                    if (lr < cnt) row = GROUPED ? static_cast<int64_t>(p.perm[pos0 + lr]) : pos0 + lr;
                    const int64_t ca = r0 + ch * EPC, cb = c0 + ch * EPC;
                    const bool oka = row >= 0 && ca < R, okb = row >= 0 && cb < C;
                    cp_async16(&r.a[l][ch * EPC], oka ? static_cast<const void*>(A + row * R + ca) : A, oka ? 16u : 0u);
                    cp_async16(&r.b[l][ch * EPC], okb ? static_cast<const void*>(Bm + row * C + cb) : Bm, okb ? 16u : 0u);
                }
            }
            cp_async_commit();
        };
        const int rot = tid & 3;  // rotated piece order of the doubled A stores (conflict-free)
        auto widen = [&](int slot, int buf) {
            const Raw& r = raw[slot];
            float va[8], vb[8];
            smem_load8<T>(&r.a[l_ld][s_ld], va);
            smem_load8<T>(&r.b[l_ld][s_ld], vb);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int c = (q + rot) & 3;
                const float v0 = c == 0 ? va[0] : c == 1 ? va[2] : c == 2 ? va[4] : va[6];
                const float v1 = c == 0 ? va[1] : c == 1 ? va[3] : c == 2 ? va[5] : va[7];
                *reinterpret_cast<float4*>(&sm.a[buf][l_ld][2 * s_ld + 4 * c]) = make_float4(v0, v0, v1, v1);
            }
            *reinterpret_cast<float4*>(&sm.b[buf][l_ld][s_ld]) = make_float4(vb[0], vb[1], vb[2], vb[3]);
            *reinterpret_cast<float4*>(&sm.b[buf][l_ld][s_ld + 4]) = make_float4(vb[4], vb[5], vb[6], vb[7]);
        };
        issue(0, 0);
        issue(1, 1);
        cp_async_wait<1>();
        __syncthreads();
        widen(0, 0);
        issue(2, 2);
        for (int64_t kb = 0; kb < nkb; ++kb) {
            cp_async_wait<1>();
            __syncthreads();
            if (kb + 1 < nkb) widen(static_cast<int>((kb + 1) % RAW_STAGES), static_cast<int>((kb + 1) & 1));
            issue(kb + RAW_STAGES, static_cast<int>(kb % RAW_STAGES));
            mma_block(sm.a[kb & 1], sm.b[kb & 1], ty, tx, acc);
        }
        cp_async_wait<0>();
    } else if (nkb > 0) {
        load(0); store(0);
        __syncthreads();
        int buf = 0;
        for (int64_t kb = 0; kb < nkb; ++kb) {
            const bool more = kb + 1 < nkb;
            if (more) load((kb + 1) * TK);
            mma_block(sm.a[buf], sm.b[buf], ty, tx, acc);
            if (more) store(buf ^ 1);
            __syncthreads();
            buf ^= 1;
        }
    }

#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t r = r0 + mrow(ty, i);
        if (r >= R) continue;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int64_t c = c0 + mrow(tx, j);
            if (c >= C) continue;
            const float v = acc_lane(acc, i, j);
            if (p.partials) {
                p.partials[(z * R + r) * C + c] = v;
            } else if (p.out_f32) {
                static_cast<float*>(p.out)[r * C + c] = v;
            } else {
                static_cast<T*>(p.out)[r * C + c] = Elem<T>::down(v);
            }
        }
    }
}

constexpr int SK_R = 4;  // most output rows of the matrix-vector kernel

// ------------------------------------------------------------------ matrix-vector kernel

// Batches of at most 4 rows (a matrix-vector product): one warp per 32 output
// columns, one column per lane, so every output column is a chain of its own
// lane: acc = fmaf(up(a[r, l]), up(b(l, c)), acc) for l ascending from +0, one
// plain fmaf per step (RR rows = RR independent chains per lane), then (+ bias)
// and one rounding -- the chain of every other kernel of this tier.  The
// operands stream through a 16-stage (f32: 10) cp.async ring of 64-step blocks: B as
// [step][32 columns] (one 2- or 4-byte shared load per step and lane) or, when
// B is contraction-contiguous, [column][64 steps] (one 16-byte load per 8
// steps); the rows of A are widened once per block into shared memory and read
// as broadcasts.  Each group of 8 steps loads its operands into registers
// while the previous group's FMAs run, so the dependent fmaf chain, not the
// loads, sets the pace.  Requires 16-byte aligned rows of whole 16-byte units.
constexpr int GV_STEPS = 64;   // contraction steps per stage
// ring depth: enough 64-step blocks in flight to cover the DRAM latency at the
// chain's pace (16-bit stages are 4.5-5 KB, f32 stages 9-9.5 KB)
template <typename T>
__host__ __device__ constexpr int gv_stages() { return sizeof(T) == 4 ? 10 : 16; }
template <typename T, bool BT>
struct GemvStage {
    static constexpr int PADE = BT ? 16 / sizeof(T) : 0;
    T b[BT ? 32 : GV_STEPS][(BT ? GV_STEPS : 32) + PADE];
    T a[SK_R][GV_STEPS];
};

template <typename T, bool BT, int RR>  // RR: rows computed (R <= RR <= 4)
__global__ void __launch_bounds__(32) scalar_rows_gemv_kernel(const RowsArgs p) {
    using Stage = GemvStage<T, BT>;
    constexpr int GV_STAGES = gv_stages<T>();
    extern __shared__ __align__(16) uint8_t smem_gv[];
    Stage* ring = reinterpret_cast<Stage*>(smem_gv);
    float(*aw)[GV_STEPS] = reinterpret_cast<float(*)[GV_STEPS]>(smem_gv + GV_STAGES * sizeof(Stage));  // [RR][steps]
    const int lane = threadIdx.x;
    const T* A = static_cast<const T*>(p.a);
    const T* B = static_cast<const T*>(p.b);
    const int64_t R = p.R, L = p.L, C = p.C;
    const int64_t c0 = static_cast<int64_t>(blockIdx.x) * 32;
    constexpr int U = 16 / sizeof(T);               // elements per 16-byte unit
    // B units of one stage: [step][32 columns] = 64 rows of 32/U units, or
    // [32 columns][64 steps] = 32 rows of 64/U units; 32 lanes take them in turn
    constexpr int B_UPR = BT ? GV_STEPS / U : 32 / U;
    constexpr int B_ROWS = BT ? 32 : GV_STEPS;
    constexpr int B_UNITS = B_UPR * B_ROWS;
    static_assert(B_UNITS % 32 == 0, "whole passes of the warp");
    constexpr int A_UPR = GV_STEPS / U;
    const int64_t nkb = (L + GV_STEPS - 1) / GV_STEPS;
    auto issue = [&](int64_t kb) {
        Stage& st = ring[kb % GV_STAGES];
        const int64_t l0 = kb * GV_STEPS;
#pragma unroll
        for (int i = 0; i < B_UNITS / 32; ++i) {
            const int u = lane + 32 * i;
            const int row = u / B_UPR, seg = (u % B_UPR) * U;
            bool ok;
            const T* src;
            if (BT) {  // column c0 + row, steps l0 + seg ..
                ok = c0 + row < C && l0 + seg < L;
                src = B + (c0 + row) * L + l0 + seg;
            } else {   // step l0 + row, columns c0 + seg ..
                ok = l0 + row < L && c0 + seg < C;
                src = B + (l0 + row) * C + c0 + seg;
            }
            cp_async16(&st.b[row][seg], ok ? src : B, ok ? 16u : 0u);
        }
        for (int u = lane; u < RR * A_UPR; u += 32) {
            const int r = u / A_UPR, seg = (u % A_UPR) * U;
            const bool ok = r < R && l0 + seg < L;
            cp_async16(&st.a[r][seg], ok ? A + r * L + l0 + seg : A, ok ? 16u : 0u);
        }
    };
    for (int64_t kb = 0; kb < GV_STAGES - 1; ++kb) {
        if (kb < nkb) issue(kb);
        cp_async_commit();
    }
    float acc[RR];
#pragma unroll
    for (int r = 0; r < RR; ++r) acc[r] = 0.0f;
    for (int64_t kb = 0; kb < nkb; ++kb) {
        cp_async_wait<GV_STAGES - 2>();
        __syncwarp();  // block kb has landed for every lane; block kb - 1 is no longer read
        if (kb + GV_STAGES - 1 < nkb) issue(kb + GV_STAGES - 1);
        cp_async_commit();
        const Stage& st = ring[kb % GV_STAGES];
        for (int u = lane; u < RR * GV_STEPS; u += 32) aw[u / GV_STEPS][u % GV_STEPS] = Elem<T>::up(st.a[u / GV_STEPS][u % GV_STEPS]);
        __syncwarp();
        // group g of 8 steps: operands in registers one group ahead of the FMAs
        float bc[8], ac[RR][8];
        auto fetch = [&](int j0, float (&bv)[8], float (&av)[RR][8]) {
            if (BT) {
                smem_load8<T>(&st.b[lane][j0], bv);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) bv[i] = Elem<T>::up(st.b[j0 + i][lane]);
            }
#pragma unroll
            for (int r = 0; r < RR; ++r) {
                const float4 x0 = *reinterpret_cast<const float4*>(&aw[r][j0]);
                const float4 x1 = *reinterpret_cast<const float4*>(&aw[r][j0 + 4]);
                av[r][0] = x0.x; av[r][1] = x0.y; av[r][2] = x0.z; av[r][3] = x0.w;
                av[r][4] = x1.x; av[r][5] = x1.y; av[r][6] = x1.z; av[r][7] = x1.w;
            }
        };
        fetch(0, bc, ac);
#pragma unroll
        for (int j0 = 0; j0 < GV_STEPS; j0 += 8) {
            float bn[8], an[RR][8];
            if (j0 + 8 < GV_STEPS) fetch(j0 + 8, bn, an);
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int r = 0; r < RR; ++r) acc[r] = fmaf(ac[r][i], bc[i], acc[r]);
            if (j0 + 8 < GV_STEPS) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    bc[i] = bn[i];
#pragma unroll
                    for (int r = 0; r < RR; ++r) ac[r][i] = an[r][i];
                }
            }
        }
        __syncwarp();  // aw is rewritten for the next block
    }
    cp_async_wait<0>();
    const int64_t c = c0 + lane;
    if (c >= C) return;
    T* out = static_cast<T*>(p.out);
    const T* bias = static_cast<const T*>(p.bias);
    const float bc = bias != nullptr ? Elem<T>::up(bias[c]) : 0.0f;
#pragma unroll
    for (int r = 0; r < RR; ++r) {
        if (r >= R) break;
        out[r * C + c] = Elem<T>::down(bias != nullptr ? __fadd_rn(acc[r], bc) : acc[r]);
    }
}

// Chunk chains for outputs at most 64 columns wide, and for small outputs that
// the 128 x 128 tiles would spread over fewer CTAs than the GPU has SMs: 16 x 64
// tiles on 256 threads (column tile blockIdx.z), 2 x 2 outputs per thread, one
// CTA per (tile, chunk).  Same chains as scalar_dw_chunk_kernel (rows of the
// chunk ascending from +0).  Dense only.
template <typename T>
__global__ void __launch_bounds__(256) scalar_dw_narrow_kernel(const DwArgs p) {
    __shared__ __align__(16) float as[2][NW_TK][2 * NW_TM + 4];  // A doubled: [l][2r], [l][2r+1]
    __shared__ __align__(16) float bs[2][NW_TK][NW_TN + 4];
    const int tid = threadIdx.x, ty = tid >> 5, tx = tid & 31;  // rows 2ty, 2ty+1; cols 2tx, 2tx+1
    const T* A = static_cast<const T*>(p.a);
    const T* Bm = static_cast<const T*>(p.b);
    const int64_t R = p.R, C = p.C;
    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * NW_TM;
    const int64_t c0 = static_cast<int64_t>(blockIdx.z) * NW_TN;
    const int64_t z = blockIdx.y;
    const int64_t pos0 = z * BI_DW_CHUNK;
    const int64_t cnt = lmin(BI_DW_CHUNK, p.M - pos0);
    // staging of a 32-row block: A [l][16 r] (2 per thread), B [l][64 c] (8 per thread)
    const int sl = tid >> 3, sa = (tid & 7) * 2, sb = (tid & 7) * 8;
    float ra[2], rb[8];
    auto load = [&](int64_t l0) {
        const bool ok = l0 + sl < cnt;
        const int64_t row = pos0 + l0 + sl;
#pragma unroll
        for (int i = 0; i < 2; ++i)
            ra[i] = (ok && r0 + sa + i < R) ? Elem<T>::up(A[row * R + r0 + sa + i]) : 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) rb[i] = (ok && c0 + sb + i < C) ? Elem<T>::up(Bm[row * C + c0 + sb + i]) : 0.0f;
    };
    auto store = [&](int buf) {
        *reinterpret_cast<float4*>(&as[buf][sl][2 * sa]) = make_float4(ra[0], ra[0], ra[1], ra[1]);
        *reinterpret_cast<float4*>(&bs[buf][sl][sb]) = make_float4(rb[0], rb[1], rb[2], rb[3]);
        *reinterpret_cast<float4*>(&bs[buf][sl][sb + 4]) = make_float4(rb[4], rb[5], rb[6], rb[7]);
    };
    uint64_t acc[2] = {0, 0};
    const int64_t nkb = (cnt + NW_TK - 1) / NW_TK;
    if (nkb > 0) {
        load(0);
        store(0);
        __syncthreads();
        for (int64_t kb = 0; kb < nkb; ++kb) {
            const int buf = static_cast<int>(kb & 1);
            const bool more = kb + 1 < nkb;
            if (more) load((kb + 1) * NW_TK);
#pragma unroll
            for (int l = 0; l < NW_TK; ++l) {
                const ulonglong2 a = *reinterpret_cast<const ulonglong2*>(&as[buf][l][4 * ty]);
                const uint64_t b = *reinterpret_cast<const uint64_t*>(&bs[buf][l][2 * tx]);
                fma2(acc[0], a.x, b);
                fma2(acc[1], a.y, b);
            }
            if (more) store(buf ^ 1);
            __syncthreads();
        }
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int64_t r = r0 + 2 * ty + i;
        if (r >= R) continue;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int64_t c = c0 + 2 * tx + j;
            if (c >= C) continue;
            const float v = __uint_as_float(static_cast<uint32_t>(j ? (acc[i] >> 32) : acc[i]));
            if (p.partials) p.partials[(z * R + r) * C + c] = v;
            else if (p.out_f32) static_cast<float*>(p.out)[r * C + c] = v;
            else static_cast<T*>(p.out)[r * C + c] = Elem<T>::down(v);
        }
    }
}

// The fixed tree over J chunk partials of one output, as a binary counter:
// after chunk j the counter merges the two newest entries once per trailing
// zero bit of j+1 (pairs of equal, aligned blocks), and at the end folds the
// remaining entries from the newest down.  Same pairs, same operands as the
// level-by-level pairwise tree with the odd last entry carried.
__device__ __forceinline__ float tree_counter(const float* part, int64_t stride, int64_t J) {
    float st[32];
    int sp = 0;
    for (int64_t j = 0; j < J; ++j) {
        st[sp++] = part[j * stride];
        for (uint64_t c = static_cast<uint64_t>(j) + 1; (c & 1u) == 0; c >>= 1) {
            st[sp - 2] = st[sp - 2] + st[sp - 1];
            --sp;
        }
    }
    float v = sp ? st[sp - 1] : 0.0f;
    for (int i = sp - 2; i >= 0; --i) v = st[i] + v;
    return v;
}

// The same tree for J <= 32, level by level as defined (adjacent pairs, an odd
// last entry carried up), with all J partials loaded first and every index
// fixed at compile time, so the partials stay in registers.
__device__ __forceinline__ float tree_levels32(const float* part, int64_t stride, int J) {
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = j < J ? part[j * stride] : 0.0f;
    int n = J;
#pragma unroll
    for (int lvl = 0; lvl < 5; ++lvl) {
#pragma unroll
        for (int i = 0; i < (16 >> lvl); ++i) v[i] = (2 * i + 1 < n) ? v[2 * i] + v[2 * i + 1] : v[2 * i];
        n = (n + 1) / 2;
    }
    return v[0];
}

__device__ __forceinline__ float tree_from(const float* part, int64_t stride, int64_t J) {
    return J <= 32 ? tree_levels32(part, stride, static_cast<int>(J)) : tree_counter(part, stride, J);
}

template <typename T>
__global__ void dw_tree_kernel(const float* partials, int64_t RC, int64_t J, void* out, int out_f32) {
    for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < RC;
         e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const float v = tree_from(partials + e, RC, J);
        if (out_f32) static_cast<float*>(out)[e] = v;
        else static_cast<T*>(out)[e] = Elem<T>::down(v);
    }
}

// grouped: blockIdx.y = expert; chunk range of expert g follows experts 0..g-1
__global__ void dw_tree_grouped_kernel(const float* partials, int64_t RC, const uint32_t* seg,
                                       float* out) {
    const int g = blockIdx.y;
    int64_t cstart = 0;
    for (int q = 0; q < g; ++q) cstart += (static_cast<int64_t>(seg[q + 1] - seg[q]) + BI_DW_CHUNK - 1) / BI_DW_CHUNK;
    const int64_t J = (static_cast<int64_t>(seg[g + 1] - seg[g]) + BI_DW_CHUNK - 1) / BI_DW_CHUNK;
    for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < RC;
         e += static_cast<int64_t>(gridDim.x) * blockDim.x)
        out[g * RC + e] = tree_from(partials + cstart * RC + e, RC, J);
}

// ------------------------------------------------------------------ bias gradient

// Column sums of dY in the fixed order of the dW reduction: chunk c (blockIdx.y)
// of BI_DW_CHUNK rows, f32 additions from +0.0f in row order; one thread per
// column, so a warp reads consecutive columns of one row.  Sixteen rows' loads
// are issued before their additions, which keeps enough bytes in flight for
// HBM while the additions stay in row order.  With `partials` the chunk sums go
// to the workspace for the tree; without it (one chunk) the result is rounded
// and stored directly.
template <typename T>
__global__ void __launch_bounds__(256) bias_chunk_kernel(const T* dy, int64_t M, int64_t N, float* partials,
                                                        void* out, int out_f32) {
    const int64_t j = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
    const int64_t c = blockIdx.y;
    if (j >= N) return;
    const int64_t r0 = c * BI_DW_CHUNK;
    const int64_t r1 = lmin(M, r0 + BI_DW_CHUNK);
    const T* col = dy + j;
    float acc = 0.0f;
    int64_t r = r0;
    for (; r + 16 <= r1; r += 16) {
        T v[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) v[u] = col[(r + u) * N];
#pragma unroll
        for (int u = 0; u < 16; ++u) acc = __fadd_rn(acc, Elem<T>::up(v[u]));
    }
    for (; r < r1; ++r) acc = __fadd_rn(acc, Elem<T>::up(col[r * N]));
    if (partials) partials[c * N + j] = acc;
    else if (out_f32) static_cast<float*>(out)[j] = acc;
    else static_cast<T*>(out)[j] = Elem<T>::down(acc);
}

// ------------------------------------------------------------------ host helpers

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Row tiles for R rows at tile height tm (grouped: an upper bound over experts).
int64_t row_tiles_for(int64_t R, int64_t E, bool grouped, int tm) {
    return (R + tm - 1) / tm + (grouped ? E : 0);
}

// Dynamic shared memory above the 48 KB default needs each kernel's opt-in,
// once per kernel (the template argument is the kernel itself) and device.
template <auto KERN>
cudaError_t allow_smem(const LaunchCtx& c, size_t bytes) {
    static PerDeviceOnce setup;
    return setup.run(c.eng->device, [&](int&) {
        return cudaFuncSetAttribute(KERN, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
    });
}

template <typename T, bool BT, bool G, bool V, int TMV>
cudaError_t launch_rows(const LaunchCtx& c, dim3 grid, const RowsArgs& a) {
    const size_t bytes = sizeof(SmemT<TMV>) + (V ? RAW_STAGES * sizeof(RawT<T, TMV, BT>) : 0);
    const cudaError_t e = allow_smem<scalar_rows_kernel<T, BT, G, V, TMV>>(c, bytes);
    if (e != cudaSuccess) return e;
    scalar_rows_kernel<T, BT, G, V, TMV><<<grid, 2 * TMV, bytes, c.stream>>>(a);
    return cudaSuccess;
}

template <typename T, bool BT, bool G>
cudaError_t rows_t(const LaunchCtx& c, const RowsArgs& a) {
    // 8-element loads need rows of whole 16-byte units and aligned bases
    const int64_t unit = 16 / sizeof(T);
    bool vec = aligned16(a.a) && aligned16(a.b) && a.L % unit == 0 && (BT || a.C % unit == 0);
    if (sizeof(T) == 4) vec = vec && a.L % 4 == 0 && (BT || a.C % 4 == 0);
    // The tile shape does not touch any output's chain, so it may follow the
    // shape: 64-row tiles when 128-row tiles would leave the SMs under-filled.
    const int64_t col_tiles = (a.C + TN - 1) / TN;
    const bool small = row_tiles_for(a.R, a.E, G, 128) * col_tiles < int64_t(c.sm_count) * 6;
    cudaError_t e;
    if (small) {
        dim3 grid(static_cast<unsigned>(row_tiles_for(a.R, a.E, G, 64)), static_cast<unsigned>(col_tiles));
        e = vec ? launch_rows<T, BT, G, true, 64>(c, grid, a) : launch_rows<T, BT, G, false, 64>(c, grid, a);
    } else {
        dim3 grid(static_cast<unsigned>(row_tiles_for(a.R, a.E, G, 128)), static_cast<unsigned>(col_tiles));
        e = vec ? launch_rows<T, BT, G, true, 128>(c, grid, a) : launch_rows<T, BT, G, false, 128>(c, grid, a);
    }
    if (e != cudaSuccess) return e;
    c.count();
    return cudaGetLastError();
}

template <typename T>
cudaError_t rows_dispatch(const LaunchCtx& c, const RowsArgs& a, int bt, bool grouped) {
    if (grouped) return bt ? rows_t<T, true, true>(c, a) : rows_t<T, false, true>(c, a);
    return bt ? rows_t<T, true, false>(c, a) : rows_t<T, false, false>(c, a);
}

template <typename T, bool G>
cudaError_t dw_chunks_t(const LaunchCtx& c, const DwArgs& a, int64_t chunks) {
    const int64_t unit = 16 / sizeof(T);
    const bool vec = aligned16(a.a) && aligned16(a.b) && a.R % unit == 0 && a.C % unit == 0;
    dim3 grid(static_cast<unsigned>((a.C + TN - 1) / TN), static_cast<unsigned>((a.R + TM - 1) / TM),
              static_cast<unsigned>(chunks));
    const size_t vbytes = sizeof(Smem) + RAW_STAGES * sizeof(RawDwT<T>);
    const cudaError_t e = vec ? allow_smem<scalar_dw_chunk_kernel<T, G, true>>(c, vbytes)
                              : allow_smem<scalar_dw_chunk_kernel<T, G, false>>(c, sizeof(Smem));
    if (e != cudaSuccess) return e;
    if (vec) scalar_dw_chunk_kernel<T, G, true><<<grid, NT, vbytes, c.stream>>>(a);
    else scalar_dw_chunk_kernel<T, G, false><<<grid, NT, sizeof(Smem), c.stream>>>(a);
    c.count();
    return cudaGetLastError();
}

unsigned tree_grid(int64_t n, int sm) {
    int64_t b = (n + 255) / 256;
    const int64_t cap = static_cast<int64_t>(sm) * 8;
    return static_cast<unsigned>(b < cap ? (b > 0 ? b : 1) : cap);
}

}  // namespace

template <typename T>
bool gemv_ok(const RowsArgs& a) {
    const int64_t unit = 16 / sizeof(T);
    return aligned16(a.a) && aligned16(a.b) && a.L % unit == 0 && a.C % unit == 0;
}

template <typename T, bool BT, int RR>
cudaError_t launch_gemv(const LaunchCtx& c, const RowsArgs& a) {
    const size_t bytes = gv_stages<T>() * sizeof(GemvStage<T, BT>) + RR * GV_STEPS * sizeof(float);
    const cudaError_t e = allow_smem<scalar_rows_gemv_kernel<T, BT, RR>>(c, bytes);
    if (e != cudaSuccess) return e;
    scalar_rows_gemv_kernel<T, BT, RR><<<static_cast<unsigned>((a.C + 31) / 32), 32, bytes, c.stream>>>(a);
    return cudaSuccess;
}

template <typename T>
cudaError_t rows_gemv_t(const LaunchCtx& c, const RowsArgs& a, int bt) {
    cudaError_t e;
    if (bt) e = a.R <= 1 ? launch_gemv<T, true, 1>(c, a) : a.R <= 2 ? launch_gemv<T, true, 2>(c, a)
                                                                   : launch_gemv<T, true, 4>(c, a);
    else e = a.R <= 1 ? launch_gemv<T, false, 1>(c, a) : a.R <= 2 ? launch_gemv<T, false, 2>(c, a)
                                                                  : launch_gemv<T, false, 4>(c, a);
    if (e != cudaSuccess) return e;
    c.count();
    return cudaGetLastError();
}

// The narrow kernels take an output when it is at most 64 columns wide, or when
// it is small: the 128-column tiles would give fewer CTAs than the GPU has SMs
// while the 16 x 64 tiles give more, and its column tiles fit a grid dimension.
// (Any tiling gives every output the same chain.)
bool narrow_rows(const LaunchCtx& c, int64_t R, int64_t C) {
    if (C <= NW_TN) return true;
    const int64_t col_tiles = (C + NW_TN - 1) / NW_TN;
    return col_tiles <= 65535 && ((R + 63) / 64) * ((C + TN - 1) / TN) < c.sm_count &&
           ((R + NW_TM - 1) / NW_TM) * col_tiles > ((R + 63) / 64) * ((C + TN - 1) / TN);
}
bool narrow_dw(const LaunchCtx& c, int64_t R, int64_t C, int64_t J) {
    if (C <= NW_TN) return true;
    const int64_t col_tiles = (C + NW_TN - 1) / NW_TN;
    return col_tiles <= 65535 && J <= 65535 && ((R + TM - 1) / TM) * ((C + TN - 1) / TN) * J < c.sm_count;
}

template <typename T>
cudaError_t rows_narrow_t(const LaunchCtx& c, const RowsArgs& a, int bt) {
    const dim3 grid(static_cast<unsigned>((a.R + NW_TM - 1) / NW_TM), static_cast<unsigned>((a.C + NW_TN - 1) / NW_TN));
    if (bt) scalar_rows_narrow_kernel<T, true><<<grid, 256, 0, c.stream>>>(a);
    else scalar_rows_narrow_kernel<T, false><<<grid, 256, 0, c.stream>>>(a);
    c.count();
    return cudaGetLastError();
}

cudaError_t scalar_rows(const LaunchCtx& c, bi_dtype dt, void* out, const void* a, const void* b,
                        const void* bias, int64_t R, int64_t L, int64_t C, int b_contr_contig) {
    RowsArgs args{out, a, b, bias, R, L, C, 0, nullptr, nullptr};
    if (C > NW_TN && R <= SK_R) {  // a few rows: one lane per output column (the kernel changes no chain)
        switch (dt) {
            case BI_F32: if (gemv_ok<float>(args)) return rows_gemv_t<float>(c, args, b_contr_contig); break;
            case BI_BF16: if (gemv_ok<__nv_bfloat16>(args)) return rows_gemv_t<__nv_bfloat16>(c, args, b_contr_contig); break;
            default: if (gemv_ok<__half>(args)) return rows_gemv_t<__half>(c, args, b_contr_contig); break;
        }
    }
    if (narrow_rows(c, R, C)) {  // narrow or small output: the tile shape changes no chain
        switch (dt) {
            case BI_F32: return rows_narrow_t<float>(c, args, b_contr_contig);
            case BI_BF16: return rows_narrow_t<__nv_bfloat16>(c, args, b_contr_contig);
            default: return rows_narrow_t<__half>(c, args, b_contr_contig);
        }
    }
    switch (dt) {
        case BI_F32: return rows_dispatch<float>(c, args, b_contr_contig, false);
        case BI_BF16: return rows_dispatch<__nv_bfloat16>(c, args, b_contr_contig, false);
        default: return rows_dispatch<__half>(c, args, b_contr_contig, false);
    }
}

cudaError_t scalar_rows_grouped(const LaunchCtx& c, bi_dtype dt, void* out, const void* a,
                                const void* b, int64_t M, int64_t L, int64_t C, int64_t E,
                                int b_contr_contig, const uint32_t* seg, const uint32_t* perm) {
    RowsArgs args{out, a, b, nullptr, M, L, C, E, seg, perm};
    switch (dt) {
        case BI_F32: return rows_dispatch<float>(c, args, b_contr_contig, true);
        case BI_BF16: return rows_dispatch<__nv_bfloat16>(c, args, b_contr_contig, true);
        default: return rows_dispatch<__half>(c, args, b_contr_contig, true);
    }
}

cudaError_t scalar_dw(const LaunchCtx& c, bi_dtype dt, void* out, int out_f32, const void* a,
                      const void* b, int64_t M, int64_t R, int64_t C, float* partials) {
    const int64_t J = (M + BI_DW_CHUNK - 1) / BI_DW_CHUNK;
    DwArgs args{out, out_f32, J > 1 ? partials : nullptr, a, b, M, R, C, 0, nullptr, nullptr};
    cudaError_t e;
    if (narrow_dw(c, R, C, J)) {  // narrow or small output: the tile shape changes no chain
        const dim3 grid(static_cast<unsigned>((R + NW_TM - 1) / NW_TM), static_cast<unsigned>(J),
                        static_cast<unsigned>((C + NW_TN - 1) / NW_TN));
        switch (dt) {
            case BI_F32: scalar_dw_narrow_kernel<float><<<grid, 256, 0, c.stream>>>(args); break;
            case BI_BF16: scalar_dw_narrow_kernel<__nv_bfloat16><<<grid, 256, 0, c.stream>>>(args); break;
            default: scalar_dw_narrow_kernel<__half><<<grid, 256, 0, c.stream>>>(args); break;
        }
        c.count();
        e = cudaGetLastError();
    } else {
        switch (dt) {
            case BI_F32: e = dw_chunks_t<float, false>(c, args, J); break;
            case BI_BF16: e = dw_chunks_t<__nv_bfloat16, false>(c, args, J); break;
            default: e = dw_chunks_t<__half, false>(c, args, J); break;
        }
    }
    if (e != cudaSuccess || J <= 1) return e;
    const int64_t RC = R * C;
    const unsigned grid = tree_grid(RC, c.sm_count);
    switch (dt) {
        case BI_F32: dw_tree_kernel<float><<<grid, 256, 0, c.stream>>>(partials, RC, J, out, out_f32); break;
        case BI_BF16: dw_tree_kernel<__nv_bfloat16><<<grid, 256, 0, c.stream>>>(partials, RC, J, out, out_f32); break;
        default: dw_tree_kernel<__half><<<grid, 256, 0, c.stream>>>(partials, RC, J, out, out_f32); break;
    }
    c.count();
    return cudaGetLastError();
}

template <typename T>
void launch_bias_chunks(const LaunchCtx& c, const void* dy, int64_t M, int64_t N, int64_t J, float* part,
                        void* out, int out_f32) {
    dim3 grid(static_cast<unsigned>((N + 255) / 256), static_cast<unsigned>(J));
    bias_chunk_kernel<T><<<grid, 256, 0, c.stream>>>(static_cast<const T*>(dy), M, N, part, out, out_f32);
}

cudaError_t bias_grad(const LaunchCtx& c, bi_dtype dt, void* out, int out_f32, const void* dy,
                      int64_t M, int64_t N, float* partials) {
    const int64_t J = (M + BI_DW_CHUNK - 1) / BI_DW_CHUNK;
    float* part = J > 1 ? partials : nullptr;
    switch (dt) {
        case BI_F32: launch_bias_chunks<float>(c, dy, M, N, J, part, out, out_f32); break;
        case BI_BF16: launch_bias_chunks<__nv_bfloat16>(c, dy, M, N, J, part, out, out_f32); break;
        default: launch_bias_chunks<__half>(c, dy, M, N, J, part, out, out_f32); break;
    }
    c.count();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || J <= 1) return e;
    const unsigned tg = tree_grid(N, c.sm_count);
    switch (dt) {
        case BI_F32: dw_tree_kernel<float><<<tg, 256, 0, c.stream>>>(partials, N, J, out, out_f32); break;
        case BI_BF16: dw_tree_kernel<__nv_bfloat16><<<tg, 256, 0, c.stream>>>(partials, N, J, out, out_f32); break;
        default: dw_tree_kernel<__half><<<tg, 256, 0, c.stream>>>(partials, N, J, out, out_f32); break;
    }
    c.count();
    return cudaGetLastError();
}

cudaError_t scalar_dw_grouped(const LaunchCtx& c, bi_dtype dt, float* out, const void* a,
                              const void* b, int64_t M, int64_t R, int64_t C, int64_t E,
                              const uint32_t* seg, const uint32_t* perm, float* partials,
                              int64_t max_chunks) {
    DwArgs args{out, 1, partials, a, b, M, R, C, E, seg, perm};
    cudaError_t e;
    if (max_chunks > 0) {
        switch (dt) {
            case BI_F32: e = dw_chunks_t<float, true>(c, args, max_chunks); break;
            case BI_BF16: e = dw_chunks_t<__nv_bfloat16, true>(c, args, max_chunks); break;
            default: e = dw_chunks_t<__half, true>(c, args, max_chunks); break;
        }
        if (e != cudaSuccess) return e;
    }
    const int64_t RC = R * C;
    dim3 grid(tree_grid(RC, c.sm_count) / (E > 8 ? 8 : 1) + 1, static_cast<unsigned>(E));
    dw_tree_grouped_kernel<<<grid, 256, 0, c.stream>>>(partials, RC, seg, out);
    c.count();
    return cudaGetLastError();
}

}  // namespace bi
