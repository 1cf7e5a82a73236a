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
constexpr int64_t kMaxGridYZ = 65535;  // largest grid.y / grid.z

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

// Loads that stay where they are written.  A block's staging loads are issued
// before the previous block's FMAs and used after them; as plain loads the
// compiler may move them down to their use, past the FMA loop, and each block
// then waits the whole memory latency.  As volatile instructions they are
// issued in place.
__device__ __forceinline__ uint4 ldg_keep16(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}
// One element's bits (a 16-bit value in the low half).
template <typename T>
__device__ __forceinline__ uint32_t ldg_keep_bits(const T* p) {
    uint32_t v;
    if constexpr (sizeof(T) == 4) {
        asm volatile("ld.global.nc.b32 %0, [%1];" : "=r"(v) : "l"(p));
    } else {
        uint16_t h;
        asm volatile("ld.global.nc.b16 %0, [%1];" : "=h"(h) : "l"(p));
        v = h;
    }
    return v;
}
// 8 consecutive elements as loaded (their bits).  They are widened to f32 only
// when stored to shared memory, after the FMAs the load overlaps: a widening
// right after the load would make the thread wait for the load there.
template <typename T>
struct Raw8 {
    uint32_t w[2 * sizeof(T)];  // 4 words of two 16-bit elements, or 8 f32 words
};
// Load 8 consecutive elements starting at p.  VEC: p is 16-byte aligned and
// all 8 are in range; otherwise `avail` of them are loaded, the rest are +0.
template <typename T, bool VEC>
__device__ __forceinline__ void load8(const T* p, int avail, Raw8<T>& r) {
    if (VEC && avail >= 8) {
        const uint4 a = ldg_keep16(p);
        r.w[0] = a.x; r.w[1] = a.y; r.w[2] = a.z; r.w[3] = a.w;
        if constexpr (sizeof(T) == 4) {
            const uint4 b = ldg_keep16(reinterpret_cast<const uint4*>(p) + 1);
            r.w[4] = b.x; r.w[5] = b.y; r.w[6] = b.z; r.w[7] = b.w;
        }
    } else if constexpr (sizeof(T) == 4) {
#pragma unroll
        for (int i = 0; i < 8; ++i) r.w[i] = i < avail ? ldg_keep_bits(p + i) : 0u;
    } else {
#pragma unroll
        for (int i = 0; i < 8; i += 2)
            r.w[i / 2] = (i < avail ? ldg_keep_bits(p + i) : 0u) | ((i + 1 < avail ? ldg_keep_bits(p + i + 1) : 0u) << 16);
    }
}
template <typename T>
__device__ __forceinline__ void widen8(const Raw8<T>& r, float (&v)[8]) {
    if constexpr (sizeof(T) == 4) {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r.w[i]);
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint16_t b = static_cast<uint16_t>(r.w[i / 2] >> (16 * (i & 1)));
            v[i] = Elem<T>::up(*reinterpret_cast<const T*>(&b));
        }
    }
}

// Contraction padding.  Steps past the end of a contraction are staged as
// A = -0 and B = +0: their product is -0, and x + (-0) = x for every x, signed
// zeros included (+0 + -0 = +0, -0 + -0 = -0), so a padded step leaves the
// chain exactly where the last real step put it.  (+0 for both would turn a
// chain at -0 into +0.)  v[i] for i >= avail becomes -0.
__device__ __forceinline__ void pad_neg_zero(float (&v)[8], int avail) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
        if (i >= avail) v[i] = -0.0f;
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
    Raw8<T> ra, rb[SL];
    int ra_n = 0;  // valid steps of ra (the rest is contraction padding)
    auto load_a = [&](int64_t l0) {
        const int64_t l = l0 + a_seg;
        ra_n = a_src_row < 0 ? 0 : static_cast<int>(lmin(8, lmax(0, L - l)));
        load8<T, VEC>(A + (a_src_row < 0 ? 0 : a_src_row * L + l), ra_n, ra);
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
        float va[8];
        widen8<T>(ra, va);
        pad_neg_zero(va, ra_n);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            *reinterpret_cast<float2*>(&sm.a[buf][a_seg + i][2 * a_row]) = make_float2(va[i], va[i]);
#pragma unroll
        for (int q = 0; q < SL; ++q) {
            const int e = tid + q * NTV;
            float vb[8];
            widen8<T>(rb[q], vb);
            if (BT) {
                const int c = e % TN, s = (e / TN) * 8;
#pragma unroll
                for (int i = 0; i < 8; ++i) sm.b[buf][s + i][c] = vb[i];
            } else {
                const int l = e / 16, s = (e % 16) * 8;
                *reinterpret_cast<float4*>(&sm.b[buf][l][s]) = make_float4(vb[0], vb[1], vb[2], vb[3]);
                *reinterpret_cast<float4*>(&sm.b[buf][l][s + 4]) = make_float4(vb[4], vb[5], vb[6], vb[7]);
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
        auto widen = [&](int slot, int buf, int64_t l0) {
            const Raw& r = raw[slot];
            {   // A: row a_row, steps a_seg..a_seg+7, each value stored twice
                float v[8];
                smem_load8<T>(&r.a[a_row][a_seg], v);
                pad_neg_zero(v, static_cast<int>(lmin(8, lmax(0, L - (l0 + a_seg)))));
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
        widen(0, 0, 0);
        issue(2, 2);
        for (int64_t kb = 0; kb < nkb; ++kb) {
            cp_async_wait<1>();  // block kb+1 has landed (this thread's copies)
            __syncthreads();     // ... everyone's; block kb widened; tiles of kb-1 no longer read
            if (kb + 1 < nkb)
                widen(static_cast<int>((kb + 1) % RAW_STAGES), static_cast<int>((kb + 1) & 1), (kb + 1) * TK);
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
// fewer CTAs than the GPU has SMs.  Such outputs are few and their chains long,
// so the kernel is built for independent chains per thread: one output row per
// lane and 8 columns per warp (32 x 32 tiles on 4 warps), each thread holding
// 8 chains as 4 paired-FMA accumulators.  A step of a thread is one 8-byte
// load of its row's A value (stored twice, f32), two 16-byte broadcast loads
// of the warp's 8 B values and 4 paired FMAs.  Same chains as above: each
// output is fmaf over l ascending from +0, then (+ bias) and one rounding.
// The contraction is staged in double-buffered blocks of 64 steps, the next
// block's global loads issued before the current block's FMAs.  Steps past the
// end of the contraction hold A = -0 and B = +0: their product, -0, added to
// any value leaves it unchanged (signed zeros included), so the padding adds
// nothing to a chain.  Dense only.
constexpr int NW_TM = 32, NW_TN = 32, NW_TK = 64, NW_THREADS = 128;
struct NarrowSmem {
    float2 a[2][NW_TK][NW_TM];           // (a, a) for row r at step l
    float b[2][NW_TK][NW_TN + 4];
};
// With 16-byte aligned operands the rows kernel's raw blocks come through a
// cp.async ring of NW_RAW blocks (five in flight while one is multiplied: a
// block's FMAs take a fraction of the memory latency) and are widened one
// block ahead into the f32 tiles, as in the tiled kernels.  Rows padded by 16
// bytes.  (The dW kernel's chunks are at most 4 blocks long; there the ring's
// shared memory costs more resident CTAs than it saves.)
constexpr int NW_RAW = 6;
template <typename T, bool BT>
struct NarrowRaw {  // rows kernel: A [32 rows][64 steps]; B [64 steps][32 cols] or (BT) [32 cols][64 steps]
    static constexpr int PADE = 16 / sizeof(T);
    T a[NW_TM][NW_TK + PADE];
    T b[BT ? NW_TN : NW_TK][(BT ? NW_TK : NW_TN) + PADE];
};

// The compute of one staged block, 8 steps at a time: the operands of 8 steps
// are loaded first, then their 32 paired FMAs run (step order kept within each
// accumulator), so one shared-memory latency covers 8 steps.
__device__ __forceinline__ void narrow_block(const NarrowSmem& sm, int buf, int lane, int w, uint64_t (&acc)[4]) {
    const float2 (*a)[NW_TM] = sm.a[buf];
    const float (*b)[NW_TN + 4] = sm.b[buf];
#pragma unroll
    for (int l0 = 0; l0 < NW_TK; l0 += 8) {
        uint64_t av[8];
        ulonglong2 b0[8], b1[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            av[i] = *reinterpret_cast<const uint64_t*>(&a[l0 + i][lane]);
            b0[i] = *reinterpret_cast<const ulonglong2*>(&b[l0 + i][8 * w]);
            b1[i] = *reinterpret_cast<const ulonglong2*>(&b[l0 + i][8 * w + 4]);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            fma2(acc[0], av[i], b0[i].x);
            fma2(acc[1], av[i], b0[i].y);
            fma2(acc[2], av[i], b1[i].x);
            fma2(acc[3], av[i], b1[i].y);
        }
    }
}

template <typename T, bool BT, bool VEC>
__global__ void __launch_bounds__(NW_THREADS) scalar_rows_narrow_kernel(const RowsArgs p) {
    extern __shared__ __align__(16) uint8_t smem_nw[];
    NarrowSmem& sm = *reinterpret_cast<NarrowSmem*>(smem_nw);
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const T* A = static_cast<const T*>(p.a);
    const T* B = static_cast<const T*>(p.b);
    const int64_t R = p.R, L = p.L, C = p.C;
    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * NW_TM;
    const int64_t c0 = static_cast<int64_t>(blockIdx.y) * NW_TN;
    // staging of a block: A 32 rows x 64 steps (16 consecutive steps of one
    // row per thread, the rows across the lanes); B 64 steps x 32 columns, 16
    // values per thread: 16 consecutive columns of one step, or (BT) 16
    // consecutive steps of one column (the columns across the lanes)
    const int a_l = w * 16;
    const bool a_ok = r0 + lane < R;
    const int b_i = BT ? lane : (tid >> 1);             // BT: column; else step
    const int b_j = BT ? w * 16 : (tid & 1) * 16;       // BT: first step; else first column
    Raw8<T> ra[2], rb[2];
    int ra_n[2] = {0, 0};
    auto avail = [](int64_t lim, int64_t at) { return static_cast<int>(lmax(0, lmin(8, lim - at))); };
    auto load = [&](int64_t l0) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t l = l0 + a_l + 8 * h;
            ra_n[h] = a_ok ? avail(L, l) : 0;
            load8<T, VEC>(A + (a_ok ? (r0 + lane) * L + l : 0), ra_n[h], ra[h]);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            if (BT) {  // b(l, c) = B[c * L + l]
                const int64_t c = c0 + b_i, l = l0 + b_j + 8 * h;
                const int n = c < C ? avail(L, l) : 0;
                load8<T, VEC>(B + (n ? c * L + l : 0), n, rb[h]);
            } else {   // b(l, c) = B[l * C + c]
                const int64_t l = l0 + b_i, c = c0 + b_j + 8 * h;
                const int n = l < L ? avail(C, c) : 0;
                load8<T, VEC>(B + (n ? l * C + c : 0), n, rb[h]);
            }
        }
    };
    auto store = [&](int buf) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float v[8];
            widen8<T>(ra[h], v);
            pad_neg_zero(v, ra_n[h]);
#pragma unroll
            for (int i = 0; i < 8; ++i) sm.a[buf][a_l + 8 * h + i][lane] = make_float2(v[i], v[i]);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float v[8];
            widen8<T>(rb[h], v);
            if (BT) {
#pragma unroll
                for (int i = 0; i < 8; ++i) sm.b[buf][b_j + 8 * h + i][b_i] = v[i];
            } else {
                *reinterpret_cast<float4*>(&sm.b[buf][b_i][b_j + 8 * h]) = make_float4(v[0], v[1], v[2], v[3]);
                *reinterpret_cast<float4*>(&sm.b[buf][b_i][b_j + 8 * h + 4]) = make_float4(v[4], v[5], v[6], v[7]);
            }
        }
    };
    const bool active = c0 + 8 * w < C;  // a warp whose 8 columns all lie past C only stages
    uint64_t acc[4] = {0, 0, 0, 0};
    const int64_t nkb = (L + NW_TK - 1) / NW_TK;
    if constexpr (VEC) {
        using Raw = NarrowRaw<T, BT>;
        Raw* raw = reinterpret_cast<Raw*>(smem_nw + sizeof(NarrowSmem));
        constexpr int EPC = 16 / static_cast<int>(sizeof(T));  // elements per 16-byte chunk
        constexpr int CPR_L = NW_TK / EPC, CPR_C = NW_TN / EPC;
        auto issue = [&](int64_t kb, int slot) {
            if (kb < nkb) {
                Raw& rw = raw[slot];
                const int64_t l0 = kb * NW_TK;
#pragma unroll
                for (int e = tid; e < NW_TM * CPR_L; e += NW_THREADS) {  // A: row, chunk of steps
                    const int row = e / CPR_L, ch = e % CPR_L;
                    const int64_t l = l0 + ch * EPC;
                    const bool ok = r0 + row < R && l < L;
                    cp_async16(&rw.a[row][ch * EPC], ok ? static_cast<const void*>(A + (r0 + row) * L + l) : A,
                               ok ? 16u : 0u);
                }
#pragma unroll
                for (int e = tid; e < NW_TK * CPR_C; e += NW_THREADS) {
                    if (BT) {  // column c, chunk of steps
                        const int c = e / CPR_L, ch = e % CPR_L;
                        const int64_t gc = c0 + c, l = l0 + ch * EPC;
                        const bool ok = gc < C && l < L;
                        cp_async16(&rw.b[c][ch * EPC], ok ? static_cast<const void*>(B + gc * L + l) : B, ok ? 16u : 0u);
                    } else {   // step l, chunk of columns
                        const int l = e / CPR_C, ch = e % CPR_C;
                        const int64_t gl = l0 + l, gc = c0 + ch * EPC;
                        const bool ok = gl < L && gc < C;
                        cp_async16(&rw.b[l][ch * EPC], ok ? static_cast<const void*>(B + gl * C + gc) : B, ok ? 16u : 0u);
                    }
                }
            }
            cp_async_commit();  // an empty group past the end keeps the count uniform
        };
        auto widen = [&](int slot, int buf, int64_t l0) {
            const Raw& rw = raw[slot];
#pragma unroll
            for (int h = 0; h < 2; ++h) {  // A: row `lane`, steps a_l + 8h ..
                float v[8];
                smem_load8<T>(&rw.a[lane][a_l + 8 * h], v);
                pad_neg_zero(v, static_cast<int>(lmin(8, lmax(0, L - (l0 + a_l + 8 * h)))));
#pragma unroll
                for (int i = 0; i < 8; ++i) sm.a[buf][a_l + 8 * h + i][lane] = make_float2(v[i], v[i]);
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float v[8];
                if (BT) {
                    smem_load8<T>(&rw.b[b_i][b_j + 8 * h], v);
#pragma unroll
                    for (int i = 0; i < 8; ++i) sm.b[buf][b_j + 8 * h + i][b_i] = v[i];
                } else {
                    smem_load8<T>(&rw.b[b_i][b_j + 8 * h], v);
                    *reinterpret_cast<float4*>(&sm.b[buf][b_i][b_j + 8 * h]) = make_float4(v[0], v[1], v[2], v[3]);
                    *reinterpret_cast<float4*>(&sm.b[buf][b_i][b_j + 8 * h + 4]) = make_float4(v[4], v[5], v[6], v[7]);
                }
            }
        };
        for (int s = 0; s < NW_RAW - 1; ++s) issue(s, s);
        cp_async_wait<NW_RAW - 2>();  // block 0 has landed (this thread's copies)
        __syncthreads();
        widen(0, 0, 0);
        issue(NW_RAW - 1, NW_RAW - 1);
        for (int64_t kb = 0; kb < nkb; ++kb) {
            cp_async_wait<NW_RAW - 2>();  // block kb+1 has landed
            __syncthreads();              // ... everyone's; block kb widened; tiles of kb-1 free
            if (kb + 1 < nkb)
                widen(static_cast<int>((kb + 1) % NW_RAW), static_cast<int>((kb + 1) & 1), (kb + 1) * NW_TK);
            issue(kb + NW_RAW, static_cast<int>(kb % NW_RAW));  // block kb's slot, already widened
            if (active) narrow_block(sm, static_cast<int>(kb & 1), lane, w, acc);
        }
        cp_async_wait<0>();
    } else {
        load(0);
        store(0);
        __syncthreads();
        for (int64_t kb = 0; kb < nkb; ++kb) {
            const int buf = static_cast<int>(kb & 1);
            const bool more = kb + 1 < nkb;
            if (more) load((kb + 1) * NW_TK);
            if (active) narrow_block(sm, buf, lane, w, acc);
            if (more) store(buf ^ 1);
            __syncthreads();
        }
    }
    const int64_t r = r0 + lane;
    if (!active || r >= R) return;
    T* out = static_cast<T*>(p.out);
    const T* bias = static_cast<const T*>(p.bias);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int64_t c = c0 + 8 * w + j;
        if (c >= C) break;
        float v = __uint_as_float(static_cast<uint32_t>((j & 1) ? (acc[j >> 1] >> 32) : acc[j >> 1]));
        if (bias) v = v + Elem<T>::up(bias[c]);
        out[r * C + c] = Elem<T>::down(v);
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
    int64_t z0;         // first chunk of this launch (a grid dimension holds at most 65535)
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
    const int64_t z = blockIdx.z + p.z0;

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
    Raw8<T> ra_raw, rb_raw;
    int ra_n = 0;
    auto load = [&](int64_t l0) {
        const int64_t l = l0 + l_ld;
        int64_t row = -1;
        if (l < cnt) row = GROUPED ? static_cast<int64_t>(p.perm[pos0 + l]) : pos0 + l;
        const int av_a = row < 0 ? 0 : static_cast<int>(lmin(8, lmax(0, R - (r0 + s_ld))));
        const int av_b = row < 0 ? 0 : static_cast<int>(lmin(8, lmax(0, C - (c0 + s_ld))));
        load8<T, VEC>(A + (av_a ? row * R + r0 + s_ld : 0), av_a, ra_raw);
        load8<T, VEC>(Bm + (av_b ? row * C + c0 + s_ld : 0), av_b, rb_raw);
        ra_n = av_a;  // rows past the chunk (and outputs past R, which are not stored) pad with -0
    };
    // A doubled: this thread's 64 contiguous bytes as four 16-byte pieces,
    // written in an order rotated by the thread index so the 16 threads of a
    // row hit different banks in each store instruction
    const int rot = tid & 3;
    auto store = [&](int buf) {
        float ra[8], rb[8];
        widen8<T>(ra_raw, ra);
        widen8<T>(rb_raw, rb);
        pad_neg_zero(ra, ra_n);
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
        auto widen = [&](int slot, int buf, int64_t kb) {
            const Raw& r = raw[slot];
            float va[8], vb[8];
            smem_load8<T>(&r.a[l_ld][s_ld], va);
            smem_load8<T>(&r.b[l_ld][s_ld], vb);
            if (kb * TK + l_ld >= cnt) pad_neg_zero(va, 0);  // a row past the chunk
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
        widen(0, 0, 0);
        issue(2, 2);
        for (int64_t kb = 0; kb < nkb; ++kb) {
            cp_async_wait<1>();
            __syncthreads();
            if (kb + 1 < nkb) widen(static_cast<int>((kb + 1) % RAW_STAGES), static_cast<int>((kb + 1) & 1), kb + 1);
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
// fused multiply-add per step (RR rows = RR independent chains per lane), then
// (+ bias) and one rounding -- the chain of every other kernel of this tier.
// The operands stream through a 16-stage (f32: 10) cp.async ring of 64-step
// blocks: B as [step][32 columns] (one 2- or 4-byte shared load per step and
// lane) or, when B is contraction-contiguous, [column][64 steps] (one 16-byte
// load per 8 or 4 steps); the rows of A are read from the ring as broadcasts.
// 16-bit operands go into the multiply-add as they are (fma_up), so a step is
// one shared load (or less) and one FMA.  Steps past L (L is a multiple of 8)
// hold A = -0 and B = +0, which leave every chain unchanged (see
// pad_neg_zero).  Each group of 8 steps loads its
// operands into registers while the previous group's FMAs run, so the
// dependent chain, not the loads, sets the pace.  Requires 16-byte aligned
// rows of whole 16-byte units.
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

// acc + a * b for 16-bit a and b, rounded once to f32.  Widening an f16 or
// bf16 value to f32 is exact, so this equals fmaf(up(a), up(b), acc) bit for
// bit; the mixed-precision form takes the 16-bit operands directly.
template <typename T> __device__ __forceinline__ float fma_up(uint16_t a, uint16_t b, float acc);
template <> __device__ __forceinline__ float fma_up<__half>(uint16_t a, uint16_t b, float acc) {
    float d;
    asm("fma.rn.f32.f16 %0, %1, %2, %3;" : "=f"(d) : "h"(a), "h"(b), "f"(acc));
    return d;
}
template <> __device__ __forceinline__ float fma_up<__nv_bfloat16>(uint16_t a, uint16_t b, float acc) {
    float d;
    asm("fma.rn.f32.bf16 %0, %1, %2, %3;" : "=f"(d) : "h"(a), "h"(b), "f"(acc));
    return d;
}
// element i of 8 consecutive T held as raw 32-bit words
template <typename T> __device__ __forceinline__ uint32_t raw_elem(const uint32_t (&w)[8 * sizeof(T) / 4], int i) {
    if (sizeof(T) == 4) return w[i];
    return (w[i >> 1] >> (16 * (i & 1))) & 0xffffu;
}
template <typename T> __device__ __forceinline__ float step_fma(uint32_t a, uint32_t b, float acc) {
    if constexpr (sizeof(T) == 4) return fmaf(__uint_as_float(a), __uint_as_float(b), acc);
    else return fma_up<T>(static_cast<uint16_t>(a), static_cast<uint16_t>(b), acc);
}

template <typename T, bool BT, int RR>  // RR: rows computed (R <= RR <= 4)
__global__ void __launch_bounds__(32) scalar_rows_gemv_kernel(const RowsArgs p) {
    using Stage = GemvStage<T, BT>;
    constexpr int GV_STAGES = gv_stages<T>();
    constexpr int WD = 8 * sizeof(T) / 4;           // 32-bit words of 8 elements
    extern __shared__ __align__(16) uint8_t smem_gv[];
    Stage* ring = reinterpret_cast<Stage*>(smem_gv);
    const int lane = threadIdx.x;
    const T* __restrict__ A = static_cast<const T*>(p.a);
    const T* __restrict__ B = static_cast<const T*>(p.b);
    const int64_t R = p.R, C = p.C;
    const int L = static_cast<int>(p.L);  // a contraction is at most 8388480 long
    const int64_t c0 = static_cast<int64_t>(blockIdx.x) * 32;
    constexpr int U = 16 / sizeof(T);               // elements per 16-byte unit
    // B units of one stage: [step][32 columns] = 64 rows of 32/U units, or
    // [32 columns][64 steps] = 32 rows of 64/U units; 32 lanes take them in turn
    constexpr int B_UPR = BT ? GV_STEPS / U : 32 / U;
    constexpr int B_ROWS = BT ? 32 : GV_STEPS;
    constexpr int B_PER = B_UPR * B_ROWS / 32;      // units per lane and stage
    static_assert(B_UPR * B_ROWS % 32 == 0, "whole passes of the warp");
    constexpr int A_UPR = GV_STEPS / U;
    constexpr int A_PER = (RR * A_UPR + 31) / 32;
    const int nkb = (L + GV_STEPS - 1) / GV_STEPS;
    // Each lane's units keep their place in every stage: source pointers that
    // advance one block per issued stage, and the step bound of each unit.
    const T* bsrc[B_PER];
    int blim[B_PER];
#pragma unroll
    for (int i = 0; i < B_PER; ++i) {
        const int u = lane + 32 * i, row = u / B_UPR, seg = (u % B_UPR) * U;
        if (BT) {  // column c0 + row, steps seg ..
            const bool cok = c0 + row < C;
            bsrc[i] = cok ? B + (c0 + row) * L + seg : B;
            blim[i] = cok ? L - seg : 0;
        } else {   // step row, columns c0 + seg ..
            const bool cok = c0 + seg < C;
            bsrc[i] = cok ? B + static_cast<int64_t>(row) * C + c0 + seg : B;
            blim[i] = cok ? L - row : 0;
        }
    }
    const T* asrc[A_PER];
    int alim[A_PER];
#pragma unroll
    for (int i = 0; i < A_PER; ++i) {
        const int u = lane + 32 * i, r = u / A_UPR, seg = (u % A_UPR) * U;
        const bool ok = u < RR * A_UPR && r < R;
        asrc[i] = ok ? A + r * L + seg : A;
        alim[i] = ok ? L - seg : 0;
    }
    const int64_t bstep = BT ? GV_STEPS : GV_STEPS * C;
    int l_issue = 0;
    int slot_issue = 0;
    auto issue = [&]() {
        Stage& st = ring[slot_issue];
#pragma unroll
        for (int i = 0; i < B_PER; ++i) {
            const int u = lane + 32 * i, row = u / B_UPR, seg = (u % B_UPR) * U;
            const bool ok = l_issue < blim[i];
            cp_async16(&st.b[row][seg], ok ? bsrc[i] : B, ok ? 16u : 0u);
            bsrc[i] += bstep;
        }
#pragma unroll
        for (int i = 0; i < A_PER; ++i) {
            const int u = lane + 32 * i, r = u / A_UPR, seg = (u % A_UPR) * U;
            if (u < RR * A_UPR) {
                if (l_issue < alim[i]) {
                    cp_async16(&st.a[r][seg], asrc[i], 16u);
                } else {  // past the contraction (or R): -0, so that a padded step adds -0 * +0
                    const uint32_t nz = sizeof(T) == 4 ? 0x80000000u : 0x80008000u;
                    *reinterpret_cast<uint4*>(&st.a[r][seg]) = make_uint4(nz, nz, nz, nz);
                }
            }
            asrc[i] += GV_STEPS;
        }
        l_issue += GV_STEPS;
        slot_issue = slot_issue + 1 == GV_STAGES ? 0 : slot_issue + 1;
    };
    for (int kb = 0; kb < GV_STAGES - 1; ++kb) {
        if (kb < nkb) issue();
        cp_async_commit();
    }
    float acc[RR];
#pragma unroll
    for (int r = 0; r < RR; ++r) acc[r] = 0.0f;
    int slot = 0;
    for (int kb = 0; kb < nkb; ++kb) {
        cp_async_wait<GV_STAGES - 2>();
        __syncwarp();  // block kb has landed for every lane; block kb - 1 is no longer read
        if (kb + GV_STAGES - 1 < nkb) issue();
        cp_async_commit();
        const Stage& st = ring[slot];
        slot = slot + 1 == GV_STAGES ? 0 : slot + 1;
        // group of 8 steps: raw operands in registers one group ahead of the FMAs
        // B of 8 steps: 16-byte loads when B is contraction-contiguous (elements
        // packed in words, like A); otherwise one load per step, one element per
        // register (BW words)
        constexpr int BW = BT ? WD : 8;
        uint32_t bw[BW], aw[RR][WD];
        auto b_elem = [](const uint32_t (&bv)[BW], int i) -> uint32_t {
            if constexpr (BT) return raw_elem<T>(bv, i);
            else return bv[i];
        };
        auto fetch = [&](int j0, uint32_t (&bv)[BW], uint32_t (&av)[RR][WD]) {
            if constexpr (BT) {
#pragma unroll
                for (int q = 0; q < WD; q += 4) {
                    const uint4 v = *reinterpret_cast<const uint4*>(&st.b[lane][j0 + q * 4 / sizeof(T)]);
                    bv[q] = v.x; bv[q + 1] = v.y; bv[q + 2] = v.z; bv[q + 3] = v.w;
                }
            } else if constexpr (sizeof(T) == 4) {
#pragma unroll
                for (int i = 0; i < 8; ++i) bv[i] = *reinterpret_cast<const uint32_t*>(&st.b[j0 + i][lane]);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) bv[i] = *reinterpret_cast<const uint16_t*>(&st.b[j0 + i][lane]);
            }
#pragma unroll
            for (int r = 0; r < RR; ++r)
#pragma unroll
                for (int q = 0; q < WD; q += 4) {
                    const uint4 v = *reinterpret_cast<const uint4*>(&st.a[r][j0 + q * 4 / sizeof(T)]);
                    av[r][q] = v.x; av[r][q + 1] = v.y; av[r][q + 2] = v.z; av[r][q + 3] = v.w;
                }
        };
        fetch(0, bw, aw);
#pragma unroll
        for (int j0 = 0; j0 < GV_STEPS; j0 += 8) {
            uint32_t bn[BW], an[RR][WD];
            if (j0 + 8 < GV_STEPS) fetch(j0 + 8, bn, an);
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int r = 0; r < RR; ++r)
                    acc[r] = step_fma<T>(raw_elem<T>(aw[r], i), b_elem(bw, i), acc[r]);
            if (j0 + 8 < GV_STEPS) {
#pragma unroll
                for (int q = 0; q < BW; ++q) bw[q] = bn[q];
#pragma unroll
                for (int q = 0; q < WD; ++q)
#pragma unroll
                    for (int r = 0; r < RR; ++r) aw[r][q] = an[r][q];
            }
        }
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
// the 128 x 128 tiles would spread over fewer CTAs than the GPU has SMs: the
// narrow rows kernel's layout (one output row r per lane, 8 columns per warp,
// 32 x 32 tiles, column tile blockIdx.z) with the chunk's rows as the
// contraction, one CTA per (tile, chunk).  Same chains as
// scalar_dw_chunk_kernel (rows of the chunk ascending from +0); padded steps
// hold A = -0, B = +0 and change no chain.  Dense only.
template <typename T, bool VEC>
__global__ void __launch_bounds__(NW_THREADS) scalar_dw_narrow_kernel(const DwArgs p) {
    extern __shared__ __align__(16) uint8_t smem_nw[];
    NarrowSmem& sm = *reinterpret_cast<NarrowSmem*>(smem_nw);
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const T* A = static_cast<const T*>(p.a);
    const T* Bm = static_cast<const T*>(p.b);
    const int64_t R = p.R, C = p.C;
    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * NW_TM;
    const int64_t c0 = static_cast<int64_t>(blockIdx.z) * NW_TN;
    const int64_t z = blockIdx.y + p.z0;
    const int64_t pos0 = z * BI_DW_CHUNK;
    const int64_t cnt = lmin(BI_DW_CHUNK, p.M - pos0);
    // staging of a block of 64 chunk rows: A[m, r0 + lane] for 16 rows m per
    // thread (a warp reads 32 consecutive r of one row: coalesced); B[m, c0 ..]
    // as 16 consecutive columns of one row m per thread
    const int a_m = w * 16;
    const bool a_ok = r0 + lane < R;
    const int b_m = tid >> 1, b_c = (tid & 1) * 16;
    uint32_t ra[16];  // bits of A[m, r]; past the chunk: -0
    Raw8<T> rb[2];
    constexpr uint32_t NEG_ZERO = sizeof(T) == 4 ? 0x80000000u : 0x8000u;
    auto avail = [](int64_t lim, int64_t at) { return static_cast<int>(lmax(0, lmin(8, lim - at))); };
    auto load = [&](int64_t l0) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int64_t m = l0 + a_m + i;
            ra[i] = a_ok && m < cnt ? ldg_keep_bits(A + (pos0 + m) * R + r0 + lane) : NEG_ZERO;
        }
        const int64_t m = l0 + b_m;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int n = m < cnt ? avail(C, c0 + b_c + 8 * h) : 0;
            load8<T, VEC>(Bm + (n ? (pos0 + m) * C + c0 + b_c + 8 * h : 0), n, rb[h]);
        }
    };
    auto store = [&](int buf) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float v;
            if constexpr (sizeof(T) == 4) {
                v = __uint_as_float(ra[i]);
            } else {
                const uint16_t b = static_cast<uint16_t>(ra[i]);
                v = Elem<T>::up(*reinterpret_cast<const T*>(&b));
            }
            sm.a[buf][a_m + i][lane] = make_float2(v, v);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float v[8];
            widen8<T>(rb[h], v);
            *reinterpret_cast<float4*>(&sm.b[buf][b_m][b_c + 8 * h]) = make_float4(v[0], v[1], v[2], v[3]);
            *reinterpret_cast<float4*>(&sm.b[buf][b_m][b_c + 8 * h + 4]) = make_float4(v[4], v[5], v[6], v[7]);
        }
    };
    const bool active = c0 + 8 * w < C;
    uint64_t acc[4] = {0, 0, 0, 0};
    const int64_t nkb = (cnt + NW_TK - 1) / NW_TK;
    if (nkb > 0) {
        load(0);
        store(0);
        __syncthreads();
        for (int64_t kb = 0; kb < nkb; ++kb) {
            const int buf = static_cast<int>(kb & 1);
            const bool more = kb + 1 < nkb;
            if (more) load((kb + 1) * NW_TK);
            if (active) narrow_block(sm, buf, lane, w, acc);
            if (more) store(buf ^ 1);
            __syncthreads();
        }
    }
    const int64_t r = r0 + lane;
    if (!active || r >= R) return;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int64_t c = c0 + 8 * w + j;
        if (c >= C) break;
        const float v = __uint_as_float(static_cast<uint32_t>((j & 1) ? (acc[j >> 1] >> 32) : acc[j >> 1]));
        if (p.partials) p.partials[(z * R + r) * C + c] = v;
        else if (p.out_f32) static_cast<float*>(p.out)[r * C + c] = v;
        else static_cast<T*>(p.out)[r * C + c] = Elem<T>::down(v);
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
                                                        void* out, int out_f32, int64_t c0) {
    const int64_t j = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
    const int64_t c = blockIdx.y + c0;
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
    const size_t vbytes = sizeof(Smem) + RAW_STAGES * sizeof(RawDwT<T>);
    cudaError_t e = vec ? allow_smem<scalar_dw_chunk_kernel<T, G, true>>(c, vbytes)
                        : allow_smem<scalar_dw_chunk_kernel<T, G, false>>(c, sizeof(Smem));
    if (e != cudaSuccess) return e;
    for (int64_t z0 = 0; z0 < chunks; z0 += kMaxGridYZ) {  // chunks in grid.z, sliced
        DwArgs s = a;
        s.z0 = z0;
        const dim3 grid(static_cast<unsigned>((a.C + TN - 1) / TN), static_cast<unsigned>((a.R + TM - 1) / TM),
                        static_cast<unsigned>(lmin(kMaxGridYZ, chunks - z0)));
        if (vec) scalar_dw_chunk_kernel<T, G, true><<<grid, NT, vbytes, c.stream>>>(s);
        else scalar_dw_chunk_kernel<T, G, false><<<grid, NT, sizeof(Smem), c.stream>>>(s);
        c.count();
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
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
    const size_t bytes = gv_stages<T>() * sizeof(GemvStage<T, BT>);
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
// while the 32 x 32 tiles give more, and its column tiles fit a grid dimension.
// (Any tiling gives every output the same chain.)
constexpr int64_t NARROW_COLS = 64;  // outputs this wide or less always take the narrow kernels
bool narrow_rows(const LaunchCtx& c, int64_t R, int64_t C) {
    if (C <= NARROW_COLS) return true;
    const int64_t col_tiles = (C + NW_TN - 1) / NW_TN;
    return col_tiles <= 65535 && ((R + 63) / 64) * ((C + TN - 1) / TN) < c.sm_count &&
           ((R + NW_TM - 1) / NW_TM) * col_tiles > ((R + 63) / 64) * ((C + TN - 1) / TN);
}
bool narrow_dw(const LaunchCtx& c, int64_t R, int64_t C, int64_t J) {
    if (C <= NARROW_COLS) return true;
    const int64_t col_tiles = (C + NW_TN - 1) / NW_TN;
    return col_tiles <= 65535 && ((R + TM - 1) / TM) * ((C + TN - 1) / TN) * J < c.sm_count;
}

template <typename T, bool BT, bool V>
cudaError_t launch_rows_narrow(const LaunchCtx& c, dim3 grid, const RowsArgs& a) {
    const size_t bytes = sizeof(NarrowSmem) + (V ? NW_RAW * sizeof(NarrowRaw<T, BT>) : 0);
    const cudaError_t e = allow_smem<scalar_rows_narrow_kernel<T, BT, V>>(c, bytes);
    if (e != cudaSuccess) return e;
    scalar_rows_narrow_kernel<T, BT, V><<<grid, NW_THREADS, bytes, c.stream>>>(a);
    return cudaSuccess;
}

template <typename T>
cudaError_t rows_narrow_t(const LaunchCtx& c, const RowsArgs& a, int bt) {
    const dim3 grid(static_cast<unsigned>((a.R + NW_TM - 1) / NW_TM), static_cast<unsigned>((a.C + NW_TN - 1) / NW_TN));
    // 16-byte loads need aligned bases and rows of whole 16-byte units
    const int64_t unit = 16 / sizeof(T);
    const bool vec = aligned16(a.a) && aligned16(a.b) && a.L % unit == 0 && (bt || a.C % unit == 0);
    cudaError_t e;
    if (bt) e = vec ? launch_rows_narrow<T, true, true>(c, grid, a) : launch_rows_narrow<T, true, false>(c, grid, a);
    else e = vec ? launch_rows_narrow<T, false, true>(c, grid, a) : launch_rows_narrow<T, false, false>(c, grid, a);
    if (e != cudaSuccess) return e;
    c.count();
    return cudaGetLastError();
}

template <typename T>
cudaError_t dw_narrow_t(const LaunchCtx& c, const DwArgs& a, int64_t chunks) {
    const int64_t unit = 16 / sizeof(T);  // A is read element by element; B in 16-byte vectors
    const bool vec = aligned16(a.b) && a.C % unit == 0;
    const size_t bytes = sizeof(NarrowSmem);
    cudaError_t e = vec ? allow_smem<scalar_dw_narrow_kernel<T, true>>(c, bytes)
                        : allow_smem<scalar_dw_narrow_kernel<T, false>>(c, bytes);
    if (e != cudaSuccess) return e;
    for (int64_t z0 = 0; z0 < chunks; z0 += kMaxGridYZ) {  // chunks in grid.y, sliced
        DwArgs s = a;
        s.z0 = z0;
        const dim3 grid(static_cast<unsigned>((a.R + NW_TM - 1) / NW_TM),
                        static_cast<unsigned>(lmin(kMaxGridYZ, chunks - z0)),
                        static_cast<unsigned>((a.C + NW_TN - 1) / NW_TN));
        if (vec) scalar_dw_narrow_kernel<T, true><<<grid, NW_THREADS, bytes, c.stream>>>(s);
        else scalar_dw_narrow_kernel<T, false><<<grid, NW_THREADS, bytes, c.stream>>>(s);
        c.count();
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t scalar_rows(const LaunchCtx& c, bi_dtype dt, void* out, const void* a, const void* b,
                        const void* bias, int64_t R, int64_t L, int64_t C, int b_contr_contig) {
    RowsArgs args{out, a, b, bias, R, L, C, 0, nullptr, nullptr};
    if (C > NARROW_COLS && R <= SK_R) {  // a few rows: one lane per output column (the kernel changes no chain)
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
        switch (dt) {
            case BI_F32: e = dw_narrow_t<float>(c, args, J); break;
            case BI_BF16: e = dw_narrow_t<__nv_bfloat16>(c, args, J); break;
            default: e = dw_narrow_t<__half>(c, args, J); break;
        }
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
cudaError_t launch_bias_chunks(const LaunchCtx& c, const void* dy, int64_t M, int64_t N, int64_t J, float* part,
                               void* out, int out_f32) {
    for (int64_t c0 = 0; c0 < J; c0 += kMaxGridYZ) {  // chunks in grid.y, sliced
        const dim3 grid(static_cast<unsigned>((N + 255) / 256), static_cast<unsigned>(lmin(kMaxGridYZ, J - c0)));
        bias_chunk_kernel<T><<<grid, 256, 0, c.stream>>>(static_cast<const T*>(dy), M, N, part, out, out_f32, c0);
        c.count();
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t bias_grad(const LaunchCtx& c, bi_dtype dt, void* out, int out_f32, const void* dy,
                      int64_t M, int64_t N, float* partials) {
    const int64_t J = (M + BI_DW_CHUNK - 1) / BI_DW_CHUNK;
    float* part = J > 1 ? partials : nullptr;
    cudaError_t e;
    switch (dt) {
        case BI_F32: e = launch_bias_chunks<float>(c, dy, M, N, J, part, out, out_f32); break;
        case BI_BF16: e = launch_bias_chunks<__nv_bfloat16>(c, dy, M, N, J, part, out, out_f32); break;
        default: e = launch_bias_chunks<__half>(c, dy, M, N, J, part, out, out_f32); break;
    }
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
