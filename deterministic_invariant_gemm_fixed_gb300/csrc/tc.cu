// Tensor-core tier: persistent, warp-specialised tcgen05 GEMM kernels for sm_103a.
//
// Contract (sgemm-bi 0.1.1.post2, "Determinism contracts", row "tensor cores"):
// f32 accumulation, bit-identical across runs, each output row of Y and dX
// independent of M.  Every arithmetic choice for Y and dX is fixed by
// (pass, dtype, K, N):
//   - every pass, dense and grouped, runs tcgen05.mma.cta_group::2 M256 x N256
//     on a CTA pair (tc_gemm_pair_kernel; K16 per instruction for bf16/f16),
//     except a 16-bit dW whose 256-column tiling gives few work units, which
//     runs M256 x N128 (the tile width never enters an element's chain); f32
//     accumulators live in tensor memory;
//   - the contracted index is walked in 64-wide blocks in ascending order, four
//     K16 instructions per block, accumulating into the same TMEM tile;
//   - Y and dX never split their contraction; no atomics, no stream-K;
//   - M only decides how many tiles of Y and dX exist and which CTA runs which
//     tile, which cannot change the arithmetic of any output element.
// dW contracts over M itself: a result kept in f32 takes pieces of 8192 rows,
// and the tiles of its last, partial wave contract in chunks added by the dW
// reduction's fixed pairwise tree (chosen from M, K and N; dw_split).
//
// Roles (192 threads per CTA):
//   warp 0 lane 0  TMA producer: cp.async.bulk.tensor loads into a ring of stages
//   warp 1 lane 0  MMA issuer (warp 1 also owns the TMEM allocation)
//   warps 2..5     epilogue: tcgen05.ld -> (+bias) -> one rounding -> st.global
// The accumulator is double-buffered (2 x N TMEM columns) so the epilogue of
// one tile overlaps the main loop of the next.  Every mbarrier wait is bounded
// by a %globaltimer limit; on expiry the kernel records a status code, stops all
// roles, drains its own copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "bi_internal.h"

namespace bi {
namespace {

constexpr int BM = 128;        // tile rows = MMA M
constexpr int BN = 256;        // tile cols = MMA N (the 16-bit passes also have a 128-column tile)
constexpr int BK = 64;         // contraction block = one 128-byte swizzle row of 16-bit data
constexpr int THREADS = 192;
constexpr int BAR_BYTES = 256;
constexpr int GROUP_M = 16;    // raster: 16 row-tiles share the column sweep (L2 reuse)
static_assert(GROUPED_TILE_ROWS == 256 && GROUPED_TAIL_ROWS == BK,
              "the grouping's tile and tail sizes are the pair kernel's");

enum Mode { DENSE = 0, GROUPED_ROWS = 1, GROUPED_DW = 2 };

struct Params {
    void* out;
    int64_t ldo;             // row stride of out, elements
    int64_t rows, cols;      // output extent of one problem (for masking)
    const void* bias;        // dense forward only (nullable)
    int num_m, num_n, num_kb;
    const uint32_t* seg;     // grouped: segment table
    const uint32_t* perm;    // grouped rows: sorted position -> original row
    int E;
    const float* scale_a;    // FP8: per-tensor scales applied to the f32 product
    const float* scale_b;
    int accum_out;           // f32 out, a contraction piece after the first: out += result
    int split_from, split_s; // dense: tiles from split_from on run their contraction as split_s chunks
    float* partials;         // ... whose f32 results go here, 256 x BN per (tile, chunk)
    int* status;
    unsigned long long wait_limit;
};

// ---------------------------------------------------------------- PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.b32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait.  Returns false if this CTA is aborting or the limit ran out
// (then the status word is written and the CTA-wide abort flag raised).
__device__ __noinline__ bool mbar_wait_impl(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                            int* status, unsigned long long limit, int code) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 15u) == 0) {
            if (*abort_flag) return false;
            if (globaltimer() - t0 > limit) {
                *abort_flag = 1;
                if (status) *reinterpret_cast<volatile int*>(status) = code;
                return false;
            }
        }
    }
}
#define mbar_wait(bar, parity, abort_flag, p, code) \
    mbar_wait_impl((bar), (parity), (abort_flag), (p).status, (p).wait_limit, (code))

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05 format): start address, leading and
// stride byte offsets (>> 4), version 1 at bit 46, 128-byte swizzle (2) at bit 61.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;
    d |= 2ull << 61;
    return d;
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32"
        " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
          "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- output types

template <int FMT> struct OutT;
template <> struct OutT<0> {
    using T = __half;
    static __device__ __forceinline__ uint32_t pack(float a, float b) {
        __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    }
    static __device__ __forceinline__ float load(const void* p, int64_t i) {
        return __half2float(reinterpret_cast<const __half*>(p)[i]);
    }
    static __device__ __forceinline__ void store1(void* p, int64_t i, float v) {
        reinterpret_cast<__half*>(p)[i] = __float2half_rn(v);
    }
};
template <> struct OutT<1> {
    using T = __nv_bfloat16;
    static __device__ __forceinline__ uint32_t pack(float a, float b) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    }
    static __device__ __forceinline__ float load(const void* p, int64_t i) {
        return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i]);
    }
    static __device__ __forceinline__ void store1(void* p, int64_t i, float v) {
        reinterpret_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
    }
};

// ---------------------------------------------------------------- CTA-pair kernel
//
// Every pass runs on a pair of CTAs (a 2-CTA cluster) that run one
// tcgen05.mma.cta_group::2 of shape M256 x BN x K16 (BN = 256, or 128 for the
// few-tile dW): CTA r of the pair holds rows [128r, 128r+128) of the A tile and
// columns [r BN/2, (r+1) BN/2) of the B tile in its own shared memory, and
// receives rows [128r, 128r+128) of the 256 x BN accumulator in its own tensor
// memory.  Only CTA 0 issues MMAs.  Per CTA a 64-wide contraction block is
// 32 KB (A 16 KB + B 16 KB), so a 7-stage ring fits (24 KB and 9 stages at
// BN = 128).  Each output element is one ascending chain of K16 blocks
// in its accumulator; the instruction shape and the CTA mapping are fixed by
// the pass, never by M.
//
// Work units (256 x BN output tiles), by mode:
//   DENSE         a grouped raster over (row pair-tile, column tile);
//   GROUPED_ROWS  forward / dinput: 256 consecutive rows of one expert in the
//                 row-sorted operand, starting at any row (rows past the
//                 expert's end are computed and discarded); the epilogue writes
//                 row perm[s] of the output;
//   GROUPED_DW    dweights: (expert, n tile, k tile), contraction over the
//                 expert's rows in 64-row blocks read in place, the partial
//                 last block read from a zero-padded tail buffer (tmA2/tmB2).
//
// Barriers: full[s] (CTA 0, count 1, 64 KB expected from both CTAs' copies),
// empty[s] (each CTA, released by CTA 0's commit multicast to both), tfull[b]
// (each CTA, commit multicast), tempty[b] (CTA 0, 8 arrivals: the 4 epilogue
// warps of each CTA).
constexpr int P_A_BYTES = 128 * BK * 2;  // one 128 x 128-byte tile
constexpr int SMEM_LIMIT = 227 * 1024;
// B holds bnt / 2 rows of 128 bytes per CTA (bnt = the tile's columns).
__host__ __device__ constexpr int p_b_bytes(int bnt) { return (bnt / 2) * BK * 2; }
// Stage layout per operand type: one A and one B tile, or for the 3xTF32 mode
// (IN = 3) the high and low parts of both (A_hi, B_hi, A_lo, B_lo).
__host__ __device__ constexpr int p_tiles(int in) { return in == 3 ? 2 : 1; }
// bytes the copies of one stage deliver to one CTA
__host__ __device__ constexpr int p_load_bytes(int in, int bnt) { return p_tiles(in) * (P_A_BYTES + p_b_bytes(bnt)); }
// a stage starts on a 1024-byte boundary (the 128-byte swizzle's atom)
__host__ __device__ constexpr int p_stage_bytes(int in, int bnt) { return (p_load_bytes(in, bnt) + 1023) / 1024 * 1024; }
// Output staging of the TMA-store epilogue: per epilogue warp two slices of
// 32 rows x 128 bytes (double-buffered), 32 KB per CTA.
constexpr int OUT_STAGE_BYTES = 4 * 2 * 32 * 128;
// as many stages as fit beside the output staging (3 for the 3xTF32 mode's
// 64 KB stages)
__host__ __device__ constexpr int p_stages(int in, int bnt, bool tma_out) {
    return (SMEM_LIMIT - 1024 - BAR_BYTES - (tma_out ? OUT_STAGE_BYTES : 0)) / p_stage_bytes(in, bnt);
}
__host__ __device__ constexpr int p_smem_bytes(int in, int bnt, bool tma_out) {
    return 1024 + p_stages(in, bnt, tma_out) * p_stage_bytes(in, bnt) + (tma_out ? OUT_STAGE_BYTES : 0) + BAR_BYTES;
}
static_assert(p_stages(0, 256, false) == 7 && p_stages(0, 256, true) == 6 && p_stages(0, 128, true) == 8 &&
              p_stages(3, 256, true) == 3 && p_stages(0, 176, false) == 8, "ring depths");
static_assert(p_smem_bytes(0, 256, true) <= SMEM_LIMIT && p_smem_bytes(0, 128, true) <= SMEM_LIMIT &&
              p_smem_bytes(3, 256, true) <= SMEM_LIMIT && p_smem_bytes(0, 256, false) <= SMEM_LIMIT,
              "stages fit the shared memory of one CTA");
// TMEM columns: the power of two that holds two accumulators of bnt columns;
// accumulator b starts at column b * (allocation / 2).
__host__ __device__ constexpr int p_tmem_cols(int bnt) { return 2 * bnt <= 256 ? 256 : 512; }

__device__ __forceinline__ uint32_t mapa_rank(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int x, int y,
                                                 uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                                 uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar_cluster)
        : "memory");
}

// TMA store of a staged 32-row slice (2-D, or 3-D with the expert as z), in a
// bulk async-group of the issuing thread; the group's smem reads finish before
// cp.async.bulk.wait_group.read returns, its global writes before wait_group.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(x), "r"(y)
                 : "memory");
}
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int x, int y, int z) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(x), "r"(y), "r"(z)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory"); }
template <int N>
__device__ __forceinline__ void bulk_wait() { asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Raster of the dense tiles: GROUP_M row pairs share a sweep over the column
// tiles (L2 reuse of the B columns).
__host__ __device__ __forceinline__ void dense_raster(int t, int units_m, int num_n, int& mpair, int& nb) {
    const int span = GROUP_M * num_n;
    const int grp = t / span;
    const int first = grp * GROUP_M;
    const int gsize = min(units_m - first, GROUP_M);
    const int r = t - grp * span;
    mpair = first + r % gsize;
    nb = r / gsize;
}

// One work unit of the pair kernel.
struct PairTile {
    int g;        // expert (grouped modes)
    int mpair;    // 256-row output tile (dense, dweights); tile within the expert (rows)
    int nb;       // BN-column output tile
    int nkb;      // contraction blocks
    int row0;     // grouped: first sorted row of the unit (rows) / of the expert (dweights)
    int row_end;  // grouped: end of the expert's sorted rows
    int full_kb;  // dweights: blocks read in place; block full_kb is the tail block
    int kb0;      // first contraction block of this unit (dweights chunks, dense chunks)
    int part;     // chunk unit: its slot in p.partials; -1 = the unit writes the output
    int npiece;   // contraction pieces (grouped dweights: runs of at most DW_PIECE_KB blocks)
};

// Contraction pieces of a unit: a grouped dweights unit walks its blocks
// [kb0, kb0 + nkb) in pieces cut at multiples of DW_PIECE_KB blocks counted
// from the expert's first row, each piece one run of the accumulator, the
// pieces' f32 results added in order by the epilogue; every other unit is one
// piece (a dense f32 dW takes its pieces as separate launches).
constexpr int DW_PIECE_KB = static_cast<int>(TC_PIECE_ROWS / BK);
template <int MODE>
__device__ __forceinline__ void unit_piece(const PairTile& u, int pc, int& kb0, int& nkb) {
    if (MODE != GROUPED_DW || u.nkb == 0) {
        kb0 = u.kb0;
        nkb = u.nkb;
        return;
    }
    const int first = u.kb0 / DW_PIECE_KB;
    const int lo = max(u.kb0, (first + pc) * DW_PIECE_KB);
    const int hi = min(u.kb0 + u.nkb, (first + pc + 1) * DW_PIECE_KB);
    kb0 = lo;
    nkb = hi - lo;
}

template <int MODE>
__device__ __forceinline__ bool pair_tile(const Params& p, int t, PairTile& u) {
    const int units_m = (p.num_m + 1) / 2;
    u.part = -1;
    u.npiece = 1;
    if (MODE == DENSE) {
        // tiles [0, split_from) whole; each later tile as split_s consecutive
        // units, chunk j contracting blocks [j nkb / s, (j + 1) nkb / s)
        int tile = t, chunk = -1;
        if (p.split_s > 1 && t >= p.split_from) {
            const int q = t - p.split_from;
            tile = p.split_from + q / p.split_s;
            chunk = q - (q / p.split_s) * p.split_s;
            u.part = q;
        }
        if (tile >= units_m * p.num_n) return false;
        dense_raster(tile, units_m, p.num_n, u.mpair, u.nb);
        u.g = 0;
        u.row0 = 0;
        u.row_end = 0;
        u.full_kb = p.num_kb;
        if (chunk < 0) {
            u.kb0 = 0;
            u.nkb = p.num_kb;
        } else {
            u.kb0 = chunk * p.num_kb / p.split_s;
            u.nkb = (chunk + 1) * p.num_kb / p.split_s - u.kb0;
        }
        return true;
    }
    const uint32_t* off = p.seg;            // sorted offsets of buckets 0..E, then m
    const uint32_t* tst = p.seg + p.E + 2;  // first 256-row tile of each expert; tst[E] = all
    if (MODE == GROUPED_ROWS) {
        const int rt = t / p.num_n;
        if (rt >= static_cast<int>(tst[p.E])) return false;
        int lo = 0, hi = p.E - 1;  // the largest g < E with tst[g] <= rt
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (static_cast<int>(tst[mid]) <= rt) lo = mid; else hi = mid - 1;
        }
        u.g = lo;
        u.nb = t - rt * p.num_n;
        u.mpair = rt - static_cast<int>(tst[lo]);
        u.row0 = static_cast<int>(off[lo]) + u.mpair * 256;
        u.row_end = static_cast<int>(off[lo + 1]);
        u.nkb = p.num_kb;
        u.full_kb = p.num_kb;
        u.kb0 = 0;
        return true;
    }
    // units [0, split_from) whole; each later unit as split_s consecutive chunk
    // units, chunk j contracting blocks [j nkb / s, (j + 1) nkb / s) of the
    // unit's blocks in this piece (possibly none: an empty chunk)
    int tile = t, chunk = -1;
    if (p.split_s > 1 && t >= p.split_from) {
        const int q = t - p.split_from;
        tile = p.split_from + q / p.split_s;
        chunk = q - (q / p.split_s) * p.split_s;
        u.part = q;
    }
    const int per = units_m * p.num_n;
    const int g = tile / per;
    if (g >= p.E) return false;
    const int r = tile - g * per;
    const int cnt = static_cast<int>(off[g + 1] - off[g]);
    u.g = g;
    u.mpair = r / p.num_n;
    u.nb = r - u.mpair * p.num_n;
    u.row0 = static_cast<int>(off[g]);
    u.row_end = u.row0 + cnt;
    u.full_kb = cnt / BK;
    u.kb0 = 0;  // all of the expert's blocks, or this chunk's share of them
    u.nkb = (cnt + BK - 1) / BK;
    if (chunk >= 0) {
        const int c0 = chunk * u.nkb / p.split_s;
        u.nkb = (chunk + 1) * u.nkb / p.split_s - c0;
        u.kb0 = c0;
    }
    u.npiece = u.nkb == 0 ? 1 : (u.kb0 + u.nkb - 1) / DW_PIECE_KB - u.kb0 / DW_PIECE_KB + 1;
    return true;
}

template <int IN>
__device__ __forceinline__ void mma_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
    if (IN == 3) {  // tf32 x tf32 -> f32
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
            : "memory");
    } else if (IN == 2) {  // e4m3 x e4m3 -> f32
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
            : "memory");
    } else {        // f16 x f16 or bf16 x bf16 -> f32
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
            : "memory");
    }
}

__device__ __forceinline__ void mma_commit_pair_mc(uint32_t bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(bar), "h"(mask)
        : "memory");
}

__device__ __forceinline__ void mma_commit_pair(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster)
                 : "memory");
}

// kind::f16: format 0 = f16, 1 = bf16; kind::f8f6f4: 0 = e4m3; kind::tf32: 2 = tf32.
template <int IN, bool A_MN, bool B_MN, int BNT>
__device__ __forceinline__ constexpr uint32_t instr_desc_pair() {
    constexpr uint32_t FMT = IN == 1 ? 1u : (IN == 3 ? 2u : 0u);
    return (1u << 4) | (FMT << 7) | (FMT << 10) |
           (static_cast<uint32_t>(A_MN) << 15) | (static_cast<uint32_t>(B_MN) << 16) |
           (static_cast<uint32_t>(BNT >> 3) << 17) | (static_cast<uint32_t>(256 >> 4) << 24);
}

// IN: 0 f16, 1 bf16, 2 e4m3 (scaled by *scale_a * *scale_b), 3 f32 as a
// 3xTF32 split (tmA/tmB hold the high parts, tmA2/tmB2 the low parts).  OUT:
// 0 f16, 1 bf16, 2 f32.  A contraction block is one 128-byte swizzle row per
// tile row (64, 128 or 32 elements); four MMAs of K = 16 / 32 / 8 cover it
// (three per K step in the 3xTF32 mode).
//
// Accumulators: two BN-column TMEM buffers, so the epilogue of one tile
// overlaps the MMAs of the next.  The 3xTF32 mode uses both halves of TMEM for
// one tile instead: hi*hi accumulates in columns 0-255, lo*hi + hi*lo in
// columns 256-511, and the epilogue adds the two (one rounding) unless the
// hi*hi sum is infinite, which then is the result.  The tensor
// core's accumulation rounding then hits the large sum once per K step rather
// than three times, and the small sum's rounding is 2^-11 smaller.
template <int IN, int OUT, bool A_MN, bool B_MN, int MODE, int BNT>
__global__ void __launch_bounds__(THREADS, 1)
    tc_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmB2,
                        const __grid_constant__ CUtensorMap tmO, const __grid_constant__ CUtensorMap tmP,
                        const Params p) {
    constexpr int ES = IN == 2 ? 1 : (IN == 3 ? 4 : 2);  // operand element size, bytes
    // the tf32 operands are always staged K-major (the split kernel transposes)
    static_assert(IN != 3 || (!A_MN && !B_MN), "3xTF32 takes K-major operands only");
    static_assert(MODE == DENSE || IN <= 1, "grouped passes take bf16 / f16 operands");
    // tile widths: 256, or for 16-bit operands any multiple of 16 from 128 up;
    // an MN-major B tile is whole 64-column swizzle atoms per CTA (128 or 256)
    static_assert(BNT == 256 || (IN <= 1 && BNT % 16 == 0 && BNT >= 128 && BNT < 256 && MODE != GROUPED_DW &&
                                 (!B_MN || BNT == 128)),
                  "tile width");
    constexpr int BN = BNT;                 // tile columns = MMA N
    constexpr int TMEM_COLS = p_tmem_cols(BN);
    constexpr int ACC_STRIDE = TMEM_COLS / 2;  // TMEM columns from one accumulator to the next
    constexpr int P_B_BYTES = p_b_bytes(BN);
    // the TMA-store epilogue writes every output laid out as rows of the tile
    // (not the grouped rows, which go to rows perm[s])
    constexpr bool TMAO = MODE != GROUPED_ROWS;
    constexpr int P_STAGES = p_stages(IN, BN, TMAO);
    constexpr int P_STAGE_BYTES = p_stage_bytes(IN, BN);
    constexpr int P_LOAD_BYTES = p_load_bytes(IN, BN);
    constexpr int BKE = 128 / ES;           // contraction elements per block
    constexpr int NACC = IN == 3 ? 1 : 2;   // accumulator buffers in flight
    constexpr int MN_ATOMS = ES;            // 128-byte atoms across a 128-wide MN-major tile
    constexpr int B_ATOMS = (BN / 2) * ES / 128;  // the same across this CTA's B columns
    constexpr uint32_t MN_STEP = (32 / ES) * 128;  // one MMA's rows of an MN-major tile, bytes
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const uint32_t sbase = smem_u32(smem);
    uint8_t* out_stage = smem + P_STAGES * P_STAGE_BYTES;  // 1024-aligned; used when TMAO
    uint64_t* bars = reinterpret_cast<uint64_t*>(out_stage + (TMAO ? OUT_STAGE_BYTES : 0));
    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (P_STAGES + s); };
    auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * P_STAGES + b); };
    auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * P_STAGES + 2 + b); };
    const uint32_t drain_bar = bar0 + 8u * (2 * P_STAGES + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * P_STAGES + 5);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t crank = blockIdx.x & 1u;
    const int cidx = static_cast<int>(blockIdx.x >> 1);
    const int ncl = static_cast<int>(gridDim.x >> 1);

    if (threadIdx.x == 0) {
        for (int s = 0; s < P_STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull_bar(b), 1);
            mbar_init(tempty_bar(b), 8);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {  // one warp of each CTA of the pair allocates together
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
    // set-up above touches no global memory; everything below may read what
    // the previous kernel in the stream wrote
    grid_dep_wait();
    grid_dep_launch();

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------------------ producer (both CTAs)
        int s = 0;
        uint32_t ph = 0;
        PairTile u;
        for (int t = cidx; pair_tile<MODE>(p, t, u); t += ncl) {
            // A rows (MN-major: A columns) and B columns of this CTA
            const int arow = (MODE == GROUPED_ROWS ? u.row0 : u.mpair * 256) + static_cast<int>(crank) * 128;
            const int bcol = u.nb * BN + static_cast<int>(crank) * (BN / 2);
            for (int pc = 0; pc < u.npiece; ++pc) {
            int pkb0, pnkb;
            unit_piece<MODE>(u, pc, pkb0, pnkb);
            for (int kb = 0; kb < pnkb; ++kb) {
                if (!mbar_wait(empty_bar(s), ph ^ 1u, abort_flag, p, DEV_TIMEOUT_PRODUCER)) goto done_p;
                const uint32_t fb_leader = mapa_rank(full_bar(s), 0);
                if (crank == 0) mbar_expect_tx(full_bar(s), 2 * P_LOAD_BYTES);
                int kofs = (pkb0 + kb) * BKE;  // contraction coordinate
                bool tail = false;
                if (MODE == GROUPED_DW) {  // the expert's rows in place, or its tail block
                    const int kba = pkb0 + kb;
                    tail = kba == u.full_kb;
                    kofs = tail ? u.g * BKE : u.row0 + kba * BKE;
                }
#pragma unroll
                for (int part = 0; part < p_tiles(IN); ++part) {
                    const uint32_t a_dst = sbase + s * P_STAGE_BYTES + part * (P_A_BYTES + P_B_BYTES);
                    const uint32_t b_dst = a_dst + P_A_BYTES;
                    const CUtensorMap* ma = (part || tail) ? &tmA2 : &tmA;
                    const CUtensorMap* mb = (part || tail) ? &tmB2 : &tmB;
                    if (A_MN) {
                        for (int a = 0; a < MN_ATOMS; ++a)
                            tma_load_2d_pair(a_dst + a * (BKE * 128), ma, arow + a * (128 / ES), kofs, fb_leader);
                    } else {
                        tma_load_2d_pair(a_dst, ma, kofs, arow, fb_leader);
                    }
                    if (MODE == GROUPED_ROWS) {  // W[g] through a 3-D map
                        if (B_MN) {
                            for (int b = 0; b < B_ATOMS; ++b)
                                tma_load_3d_pair(b_dst + b * (BKE * 128), mb, bcol + b * (128 / ES), kofs, u.g,
                                                 fb_leader);
                        } else {
                            tma_load_3d_pair(b_dst, mb, kofs, bcol, u.g, fb_leader);
                        }
                    } else if (B_MN) {
                        for (int b = 0; b < B_ATOMS; ++b)
                            tma_load_2d_pair(b_dst + b * (BKE * 128), mb, bcol + b * (128 / ES), kofs, fb_leader);
                    } else {
                        tma_load_2d_pair(b_dst, mb, kofs, bcol, fb_leader);
                    }
                }
                if (++s == P_STAGES) { s = 0; ph ^= 1u; }
            }
            }
        }
    done_p:;
        // Copies of this CTA complete on CTA 0's barriers; CTA 0's MMA thread
        // consumes them before it finishes, and the pair meets at the cluster
        // barrier below before either CTA releases its shared memory.
    } else if (warp == 1 && lane == 0 && crank == 0) {
        // ------------------------------------------------------------ MMA issuer (CTA 0)
        constexpr uint32_t idesc = instr_desc_pair<IN, A_MN, B_MN, BN>();
        int s = 0;
        uint32_t ph = 0;
        int ab = 0;
        uint32_t aph = 0;
        PairTile u;
        for (int t = cidx; pair_tile<MODE>(p, t, u); t += ncl) {
          for (int pc = 0; pc < u.npiece; ++pc) {
            int pkb0, pnkb;
            unit_piece<MODE>(u, pc, pkb0, pnkb);
            if (pnkb == 0) continue;  // empty expert or chunk: the epilogue writes +0 (-0 for a chunk)
            if (!mbar_wait(tempty_bar(ab), aph ^ 1u, abort_flag, p, DEV_TIMEOUT_MMA)) goto done_m;
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(ab * ACC_STRIDE);
            for (int kb = 0; kb < pnkb; ++kb) {
                if (!mbar_wait(full_bar(s), ph, abort_flag, p, DEV_TIMEOUT_MMA)) goto done_m;
                tc_fence_after();
                const uint32_t a_s = sbase + s * P_STAGE_BYTES;
                const uint32_t b_s = a_s + P_A_BYTES;
                auto desc_a = [&](uint32_t base, int kk) {
                    // K-major: 32 bytes along the swizzled row per MMA;
                    // MN-major: one MMA's worth of 128-byte rows
                    return A_MN ? smem_desc(base + kk * MN_STEP, BKE * 128, 1024) : smem_desc(base + kk * 32, 16, 1024);
                };
                auto desc_b = [&](uint32_t base, int kk) {
                    return B_MN ? smem_desc(base + kk * MN_STEP, BKE * 128, 1024) : smem_desc(base + kk * 32, 16, 1024);
                };
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    if (IN == 3) {
                        const uint32_t a_lo = a_s + (P_A_BYTES + P_B_BYTES), b_lo = a_lo + P_A_BYTES;
                        const uint32_t acc = (kb | kk) != 0 ? 1u : 0u;
                        mma_pair<IN>(d_tmem + BN, desc_a(a_lo, kk), desc_b(b_s, kk), idesc, acc);
                        mma_pair<IN>(d_tmem + BN, desc_a(a_s, kk), desc_b(b_lo, kk), idesc, 1u);
                        mma_pair<IN>(d_tmem, desc_a(a_s, kk), desc_b(b_s, kk), idesc, acc);
                    } else {
                        mma_pair<IN>(d_tmem, desc_a(a_s, kk), desc_b(b_s, kk), idesc, (kb | kk) != 0 ? 1u : 0u);
                    }
                }
                mma_commit_pair_mc(empty_bar(s), 0x3);
                if (++s == P_STAGES) { s = 0; ph ^= 1u; }
            }
            mma_commit_pair_mc(tfull_bar(ab), 0x3);
            if (++ab == NACC) { ab = 0; aph ^= 1u; }
          }
        }
    done_m:
        mma_commit_pair(drain_bar);
        mbar_wait(drain_bar, 0, abort_flag, p, DEV_TIMEOUT_MMA);
    } else if (warp >= 2) {
        // ------------------------------------------------------------ epilogue (both CTAs)
        const int q = warp & 3;
        const int r = q * 32 + lane;
        const uint32_t tempty_leader0 = mapa_rank(tempty_bar(0), 0);
        const uint32_t tempty_leader1 = mapa_rank(tempty_bar(1), 0);
        int ab = 0;
        uint32_t aph = 0;
        const float scale = IN == 2 ? __fmul_rn(__ldg(p.scale_a), __ldg(p.scale_b)) : 1.0f;
        int oslot = 0;  // output slices this warp has staged (TMA-store epilogue)
        PairTile u;
        for (int t = cidx; pair_tile<MODE>(p, t, u); t += ncl) {
            int64_t orow = -1;  // output row of this thread, or -1
            void* out = p.out;
            if (MODE == GROUPED_ROWS) {
                const int srow = u.row0 + static_cast<int>(crank) * 128 + r;  // sorted row
                if (srow < u.row_end) orow = p.perm[srow];
            } else {
                const int64_t gr = static_cast<int64_t>(u.mpair) * 256 + crank * 128 + r;
                if (gr < p.rows) orow = gr;
                if (MODE == GROUPED_DW) out = static_cast<float*>(p.out) + static_cast<int64_t>(u.g) * p.rows * p.ldo;
            }
            const int64_t col0 = static_cast<int64_t>(u.nb) * BN;
            // the tile's bias, read before its accumulator is ready: lane l holds
            // columns col0 + 8l .. col0 + 8l + 7, handed out by shuffles below
            float bv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int64_t c = col0 + 8 * lane + i;
                bv[i] = (p.bias != nullptr && c < p.cols)
                            ? (OUT == 2 ? static_cast<const float*>(p.bias)[c] : OutT<OUT == 1 ? 1 : 0>::load(p.bias, c))
                            : 0.0f;
            }
            static_assert(BN <= 8 * 32, "one 8-column bias slice per lane");
          for (int pc = 0; pc < u.npiece; ++pc) {
            int pkb0, pnkb;
            unit_piece<MODE>(u, pc, pkb0, pnkb);
            // the result is added to the sum so far: a grouped dweights piece after
            // the first, or a dense f32 dW launch after the first
            const bool add_prev = MODE == GROUPED_DW ? pc > 0 : p.accum_out != 0;
            if (pnkb == 0) {
                if (MODE == GROUPED_DW && u.part >= 0) {
                    // an empty chunk: -0, the exact identity of the chunk sum's additions
                    float* dst = p.partials + static_cast<int64_t>(u.part) * (256 * BN) +
                                 static_cast<int64_t>(crank * 128 + r) * BN;
                    for (int c = 0; c < BN; ++c) dst[c] = -0.0f;
                } else if (orow >= 0 && !add_prev) {  // an expert with no rows: +0
                    for (int64_t c = col0; c < col0 + BN && c < p.cols; ++c)
                        static_cast<float*>(out)[orow * p.ldo + c] = 0.0f;
                }
                continue;
            }
            bool ok = mbar_wait(tfull_bar(ab), aph, abort_flag, p, DEV_TIMEOUT_EPILOGUE);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) goto done_e;
            tc_fence_after();
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                   static_cast<uint32_t>(ab * ACC_STRIDE);
            // f = the finished f32 results of columns col0 + c0 .. c0 + 15 of this
            // thread's row: the accumulator (+ the 3xTF32 cross terms, x the FP8
            // scales), + the earlier pieces' sum, + the bias.  All lanes take part.
            auto values16 = [&](int c0, float (&f)[16]) {
                __syncwarp();  // lanes past the output rows rejoin before the aligned load
                uint32_t v[16];
                tmem_ld16(tbase + c0, v);
                uint32_t v2[16];
                if (IN == 3) tmem_ld16(tbase + BN + c0, v2);
                float bias16[16];  // every lane takes part in the shuffles
                if (p.bias != nullptr) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) bias16[i] = __shfl_sync(0xffffffffu, bv[i & 7], (c0 >> 3) + (i >> 3));
                }
#pragma unroll
                for (int i = 0; i < 16; ++i) f[i] = __uint_as_float(v[i]);
                if (IN == 3) {
                    // an infinite hi*hi sum is the result: the cross terms of an
                    // infinite operand (Inf * lo, with lo = 0 or NaN) carry no value
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        if (!isinf(f[i])) f[i] = __fadd_rn(f[i], __uint_as_float(v2[i]));
                }
                if (IN == 2) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) f[i] = __fmul_rn(f[i], scale);
                }
                const int64_t cb = col0 + c0;
                if (OUT == 2 && add_prev && orow >= 0) {  // the earlier pieces' sum, left in the output
                    const float* prev = static_cast<const float*>(out) + orow * p.ldo + cb;
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        if (cb + i < p.cols) f[i] = __fadd_rn(prev[i], f[i]);
                }
                if (p.bias != nullptr) {  // the bias has the output's type
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        if (cb + i < p.cols) f[i] = __fadd_rn(f[i], bias16[i]);
                }
            };
            const bool to_partials = IN <= 2 && MODE != GROUPED_ROWS && u.part >= 0;
            if (TMAO && to_partials && u.npiece == 1) {
                // a chunk unit's raw f32 sum goes to its 256 x BN slot of the
                // partials through the same staging, a 2-D map over the slots
                // (tmP, 32 columns per slice)
                const int rowbase = u.part * 256 + static_cast<int>(crank) * 128 + q * 32;
                for (int cs = 0; cs < BN; cs += 32) {
                    if (col0 + cs >= p.cols) break;
                    if (lane == 0) bulk_wait_read<1>();
                    __syncwarp();
                    const uint32_t buf = smem_u32(out_stage) + static_cast<uint32_t>(q * 8192 + (oslot & 1) * 4096);
                    const uint32_t rowaddr = buf + static_cast<uint32_t>(lane * 128);
#pragma unroll
                    for (int c16 = 0; c16 < 32; c16 += 16) {
                        __syncwarp();
                        uint32_t v[16];
                        tmem_ld16(tbase + cs + c16, v);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                                             rowaddr + static_cast<uint32_t>(((c16 / 4 + i) ^ (lane & 7)) * 16)),
                                         "r"(v[4 * i]), "r"(v[4 * i + 1]), "r"(v[4 * i + 2]), "r"(v[4 * i + 3])
                                         : "memory");
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmP, buf, cs, rowbase);
                        bulk_commit();
                    }
                    ++oslot;
                }
            } else if (TMAO && !to_partials && !(MODE == GROUPED_DW && u.npiece > 1)) {
                // TMA-store epilogue: this warp's 32 rows go out in slices of 128
                // bytes per row, staged in shared memory with the 128-byte swizzle
                // (16-byte chunk c of row r at chunk c ^ (r % 8)), two slices in
                // flight per warp
                constexpr int OES = OUT == 2 ? 4 : 2;  // output element size
                constexpr int CPS = 128 / OES;         // columns per slice
                const int rowbase = u.mpair * 256 + static_cast<int>(crank) * 128 + q * 32;
                for (int cs = 0; cs < BN; cs += CPS) {
                    if (col0 + cs >= p.cols) break;
                    if (lane == 0) bulk_wait_read<1>();  // the slice stored two slices ago has been read
                    __syncwarp();
                    const uint32_t buf = smem_u32(out_stage) + static_cast<uint32_t>(q * 8192 + (oslot & 1) * 4096);
                    const uint32_t rowaddr = buf + static_cast<uint32_t>(lane * 128);
#pragma unroll
                    for (int c16 = 0; c16 < CPS; c16 += 16) {
                        float f[16];
                        values16(cs + c16, f);
                        const int cc0 = c16 * OES / 16;  // first 16-byte chunk of these columns
                        if (OUT == 2) {
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(
                                                 rowaddr + static_cast<uint32_t>(((cc0 + i) ^ (lane & 7)) * 16)),
                                             "f"(f[4 * i]), "f"(f[4 * i + 1]), "f"(f[4 * i + 2]), "f"(f[4 * i + 3])
                                             : "memory");
                        } else {
                            using O = OutT<OUT == 1 ? 1 : 0>;
#pragma unroll
                            for (int i = 0; i < 2; ++i)
                                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                                                 rowaddr + static_cast<uint32_t>(((cc0 + i) ^ (lane & 7)) * 16)),
                                             "r"(O::pack(f[8 * i], f[8 * i + 1])), "r"(O::pack(f[8 * i + 2], f[8 * i + 3])),
                                             "r"(O::pack(f[8 * i + 4], f[8 * i + 5])), "r"(O::pack(f[8 * i + 6], f[8 * i + 7]))
                                             : "memory");
                        }
                    }
                    fence_proxy_async_smem();  // this lane's rows are visible to the store
                    __syncwarp();
                    if (lane == 0) {
                        if (MODE == GROUPED_DW) tma_store_3d(&tmO, buf, static_cast<int>(col0) + cs, rowbase, u.g);
                        else tma_store_2d(&tmO, buf, static_cast<int>(col0) + cs, rowbase);
                        bulk_commit();
                    }
                    ++oslot;
                }
            } else {
            for (int c0 = 0; c0 < BN; c0 += 16) {
                if (col0 + c0 >= p.cols) break;
                if (to_partials) {  // a chunk's raw f32 sum (unscaled)
                    __syncwarp();
                    uint32_t v[16];
                    tmem_ld16(tbase + c0, v);
                    float* dst = p.partials + static_cast<int64_t>(u.part) * (256 * BN) +
                                 static_cast<int64_t>(crank * 128 + r) * BN + c0;
#pragma unroll
                    for (int i = 0; i < 16; i += 4) {
                        float4 w4 = make_float4(__uint_as_float(v[i]), __uint_as_float(v[i + 1]),
                                                __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]));
                        if (MODE == GROUPED_DW && add_prev) {  // the chunk's earlier pieces, left here
                            const float4 pv = *reinterpret_cast<const float4*>(dst + i);
                            w4 = make_float4(__fadd_rn(pv.x, w4.x), __fadd_rn(pv.y, w4.y), __fadd_rn(pv.z, w4.z),
                                             __fadd_rn(pv.w, w4.w));
                        }
                        *reinterpret_cast<float4*>(dst + i) = w4;
                    }
                    continue;
                }
                float f[16];
                values16(c0, f);
                if (orow < 0) continue;
                const int64_t cb = col0 + c0;
                const bool full = cb + 16 <= p.cols;
                if (OUT == 2) {
                    float* dst = static_cast<float*>(out) + orow * p.ldo + cb;
                    if (full) {
#pragma unroll
                        for (int i = 0; i < 16; i += 4)
                            *reinterpret_cast<float4*>(dst + i) = make_float4(f[i], f[i + 1], f[i + 2], f[i + 3]);
                    } else {
                        for (int i = 0; i < 16; ++i)
                            if (cb + i < p.cols) dst[i] = f[i];
                    }
                } else {
                    using O = OutT<OUT == 1 ? 1 : 0>;
                    using T = typename O::T;
                    T* dst = static_cast<T*>(out) + orow * p.ldo + cb;
                    if (full) {
                        uint4 w0, w1;
                        w0.x = O::pack(f[0], f[1]);
                        w0.y = O::pack(f[2], f[3]);
                        w0.z = O::pack(f[4], f[5]);
                        w0.w = O::pack(f[6], f[7]);
                        w1.x = O::pack(f[8], f[9]);
                        w1.y = O::pack(f[10], f[11]);
                        w1.z = O::pack(f[12], f[13]);
                        w1.w = O::pack(f[14], f[15]);
                        reinterpret_cast<uint4*>(dst)[0] = w0;
                        reinterpret_cast<uint4*>(dst)[1] = w1;
                    } else {
                        for (int i = 0; i < 16; ++i)
                            if (cb + i < p.cols) O::store1(dst, i, f[i]);
                    }
                }
            }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(ab ? tempty_leader1 : tempty_leader0);
            if (++ab == NACC) { ab = 0; aph ^= 1u; }
          }
        }
    done_e:
        if (TMAO && lane == 0) bulk_wait<0>();  // this warp's stores are complete before the CTA exits
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    __syncwarp();
    cluster_sync();  // CTA 0's MMAs have finished reading both CTAs' shared memory
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(TMEM_COLS)
                     : "memory");
    }
}

// ---------------------------------------------------------------- dW chunk sum

__device__ __forceinline__ float4 add4(const float4 a, const float4 b) {
    return make_float4(__fadd_rn(a.x, b.x), __fadd_rn(a.y, b.y), __fadd_rn(a.z, b.z), __fadd_rn(a.w, b.w));
}

// dW tiles whose contraction ran as chunks: the chunks' f32 results c_0 ..
// c_{s-1} (s <= SMAX, a power of two at most 16) are added by the dW
// reduction's fixed pairwise tree (adjacent pairs level by level, an odd last
// entry carried up), all loaded first so the loads overlap and the tree runs
// in registers; then times *scale_a * *scale_b for FP8 (scales non-null), then
// for a contraction piece after the first the earlier pieces' sum in out plus
// that, rounded once to the output type.  One thread per 4 consecutive
// columns of a tile row.
constexpr int DW_MAX_CHUNKS = 16;
template <int OUT, int SMAX>
__global__ void __launch_bounds__(256) dw_chunk_sum_kernel(const float* __restrict__ partials, int split_from,
                                                           int split_s, int split_tiles, int units_m, int num_n,
                                                           int bn, void* out, int64_t ldo, int64_t rows,
                                                           int64_t cols, int accum_out, const float* scale_a,
                                                           const float* scale_b, int grouped) {
    grid_dep_wait();
    grid_dep_launch();
    const int64_t slot = 256 * static_cast<int64_t>(bn);
    const int64_t per_tile = slot / 4;
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= split_tiles * per_tile) return;
    const int ti = static_cast<int>(idx / per_tile);
    const int64_t e = (idx - ti * per_tile) * 4;  // row * bn + first column within the tile
    const int row = static_cast<int>(e / bn), col = static_cast<int>(e - static_cast<int64_t>(row) * bn);
    int mpair, nb;
    if (grouped) {  // grouped dweights: unit = (expert, row pair-tile, column tile), out [E][rows][ldo]
        const int t = split_from + ti, per = units_m * num_n;
        const int g = t / per, rr = t - g * per;
        mpair = rr / num_n;
        nb = rr - mpair * num_n;
        out = static_cast<float*>(out) + static_cast<int64_t>(g) * rows * ldo;
    } else {
        dense_raster(split_from + ti, units_m, num_n, mpair, nb);
    }
    const int64_t gr = static_cast<int64_t>(mpair) * 256 + row, gc = static_cast<int64_t>(nb) * bn + col;
    if (gr >= rows || gc >= cols) return;  // cols is a multiple of 8: the 4 columns are inside
    const float* src = partials + static_cast<int64_t>(ti) * split_s * slot + e;
    float4 v[SMAX];
#pragma unroll
    for (int j = 0; j < SMAX; ++j)
        v[j] = j < split_s ? *reinterpret_cast<const float4*>(src + j * slot) : make_float4(0.f, 0.f, 0.f, 0.f);
    int n = split_s;
#pragma unroll
    for (int w = SMAX; w > 1; w >>= 1) {
#pragma unroll
        for (int i = 0; i < w / 2; ++i) v[i] = (2 * i + 1 < n) ? add4(v[2 * i], v[2 * i + 1]) : v[2 * i];
        n = (n + 1) / 2;
    }
    float4 r = v[0];
    if (grouped && !accum_out) r = add4(r, make_float4(0.f, 0.f, 0.f, 0.f));  // an expert with no rows: +0
    if (scale_a != nullptr) {
        const float sc = __fmul_rn(__ldg(scale_a), __ldg(scale_b));
        r = make_float4(__fmul_rn(r.x, sc), __fmul_rn(r.y, sc), __fmul_rn(r.z, sc), __fmul_rn(r.w, sc));
    }
    if (OUT == 2) {
        float4* dst = reinterpret_cast<float4*>(static_cast<float*>(out) + gr * ldo + gc);
        *dst = accum_out ? add4(*dst, r) : r;
    } else {
        using O = OutT<OUT == 1 ? 1 : 0>;
        uint2 w;
        w.x = O::pack(r.x, r.y);
        w.y = O::pack(r.z, r.w);
        *reinterpret_cast<uint2*>(static_cast<typename O::T*>(out) + gr * ldo + gc) = w;
    }
}

template <int OUT>
cudaError_t launch_chunk_sum(const LaunchCtx& c, const float* ws, int split_from, int sp, int64_t split_tiles,
                             int units_m, int num_n, int bn, void* out, int64_t ldo, int64_t rows, int64_t cols,
                             int accum_out, const float* sa, const float* sb, int grouped = 0) {
    auto kern = sp <= 2 ? dw_chunk_sum_kernel<OUT, 2>
              : sp <= 4 ? dw_chunk_sum_kernel<OUT, 4>
              : sp <= 8 ? dw_chunk_sum_kernel<OUT, 8> : dw_chunk_sum_kernel<OUT, 16>;
    const int64_t threads = split_tiles * 256 * bn / 4;
    cudaError_t e = launch_pdl(kern, dim3(static_cast<unsigned>((threads + 255) / 256)), dim3(256), 0, c.stream, ws,
                               split_from, sp, static_cast<int>(split_tiles), units_m, num_n, bn, out, ldo, rows,
                               cols, accum_out, sa, sb, grouped);
    if (e == cudaSuccess) c.count();
    return e;
}

// ---------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 16-bit row-major tensor [outer][inner] (optionally [depth][outer][inner]),
// box {64, box_outer(, 1)}, 128-byte swizzle, zero fill out of bounds.
cudaError_t make_map(CUtensorMap* m, bi_dtype dt, const void* ptr, uint64_t inner, uint64_t outer,
                     uint64_t depth, uint32_t box_outer, bool rank3 = false) {
    auto enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const CUtensorMapDataType t =
        dt == BI_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    cuuint64_t dims[3] = {inner, outer, depth};
    cuuint64_t strides[2] = {inner * 2, inner * outer * 2};
    cuuint32_t box[3] = {64, box_outer, 1};
    cuuint32_t es[3] = {1, 1, 1};
    const cuuint32_t rank = rank3 ? 3 : 2;
    CUresult r = enc(m, t, rank, const_cast<void*>(ptr), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Output [depth][outer][inner] (row stride ld elements; out_fmt 0 f16, 1 bf16,
// 2 f32) for the TMA-store epilogue: box {128 bytes of columns, 32 rows (, 1)},
// 128-byte swizzle; stores past the extents are clipped.
cudaError_t make_out_map(CUtensorMap* m, int out_fmt, const void* ptr, uint64_t inner, uint64_t outer, uint64_t ld,
                         uint64_t depth = 1, bool rank3 = false) {
    auto enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const CUtensorMapDataType t = out_fmt == 2 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                : out_fmt == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                               : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const uint64_t es = out_fmt == 2 ? 4 : 2;
    cuuint64_t dims[3] = {inner, outer, depth};
    cuuint64_t strides[2] = {ld * es, ld * outer * es};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / es), 32, 1};
    cuuint32_t el[3] = {1, 1, 1};
    CUresult r = enc(m, t, rank3 ? 3 : 2, const_cast<void*>(ptr), dims, strides, box, el,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// units: work units (or an upper bound, for the grouped modes, whose count is
// known only on the device); -1 = the dense count.
// o: the output's tensor map for the TMA-store epilogue (every mode but the
// grouped rows, which pass null).
// pm: a map over the chunk partials (2-D [slots x 256][BN] f32) when the
// launch has chunk units.
template <int IN, int OUT, bool A_MN, bool B_MN, int MODE = DENSE, int BNT = BN>
cudaError_t launch_pair(const LaunchCtx& c, const CUtensorMap& a, const CUtensorMap& b, Params p,
                        const CUtensorMap* o, const CUtensorMap* a2 = nullptr, const CUtensorMap* b2 = nullptr,
                        int64_t units = -1, const CUtensorMap* pm = nullptr) {
    auto kern = tc_gemm_pair_kernel<IN, OUT, A_MN, B_MN, MODE, BNT>;
    constexpr int P_SMEM_BYTES = p_smem_bytes(IN, BNT, MODE != GROUPED_ROWS);
    if (MODE != GROUPED_ROWS && o == nullptr) return cudaErrorInvalidValue;
    static PerDeviceOnce setup;  // per device: the shared-memory opt-in and the co-resident clusters
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    const cudaError_t attr_err = setup.run(c.eng->device, [&](int& max_clusters) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, P_SMEM_BYTES);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t q = {};
        q.gridDim = dim3(128);
        q.blockDim = dim3(THREADS);
        q.dynamicSmemBytes = P_SMEM_BYTES;
        q.attrs = at;
        q.numAttrs = 1;
        e = cudaOccupancyMaxActiveClusters(&max_clusters, kern, &q);
        if (e == cudaSuccess && max_clusters < 1) e = cudaErrorInvalidConfiguration;
        return e;
    });
    if (attr_err != cudaSuccess) return attr_err;
    const int max_clusters = setup.value[c.eng->device];
    if (units < 0) units = int64_t((p.num_m + 1) / 2) * p.num_n;
    if (units <= 0) return cudaSuccess;
    p.status = c.status;
    p.wait_limit = c.wait_limit_ns;
    const int64_t clusters = units < max_clusters ? units : max_clusters;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(clusters * 2));
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = P_SMEM_BYTES;
    cfg.stream = c.stream;
    cudaLaunchAttribute la[2] = {at[0], {}};
    la[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see grid_dep_wait
    la[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = la;
    cfg.numAttrs = 2;
    if (p.split_s > 1 && pm == nullptr) return cudaErrorInvalidValue;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a, b, a2 ? *a2 : a, b2 ? *b2 : b, o ? *o : a, pm ? *pm : a, p);
    if (e != cudaSuccess) return e;
    c.count();
    return cudaGetLastError();
}

// Column tile of a pass: the engine's forced width (bi_engine_set_tile_cols)
// where the pass's B layout takes it, else the automatic choice.  Tile widths
// only decide how outputs are grouped into work units: every output element is
// the same ascending chain of 64-wide contraction blocks in one accumulator.
int pick_cols(const LaunchCtx& c, int automatic, bool b_mn_major) {
    const int f = c.eng ? c.eng->tile_cols : 0;
    if (f == 256 || f == 128) return f;
    if (!b_mn_major && (f == 176 || f == 192)) return f;
    return automatic;
}

template <int FMT, int BNT>
cudaError_t forward_impl(const LaunchCtx& c, bi_dtype dt, void* y, const void* x, const void* w,
                         const void* bias, int64_t M, int64_t K, int64_t N) {
    CUtensorMap a, b;
    cudaError_t e;
    if ((e = make_map(&a, dt, x, K, M, 1, BM)) != cudaSuccess) return e;   // X [M,K], K-major
    if ((e = make_map(&b, dt, w, N, K, 1, BK)) != cudaSuccess) return e;   // W [K,N], MN-major
    Params p{};
    p.out = y; p.ldo = N; p.rows = M; p.cols = N; p.bias = bias;
    p.num_m = static_cast<int>((M + BM - 1) / BM);
    p.num_n = static_cast<int>((N + BNT - 1) / BNT);
    p.num_kb = static_cast<int>((K + BK - 1) / BK);
    CUtensorMap o;
    if ((e = make_out_map(&o, FMT, y, N, M, N)) != cudaSuccess) return e;
    return launch_pair<FMT, FMT, false, true, DENSE, BNT>(c, a, b, p, &o);
}

template <int FMT>
cudaError_t forward_t(const LaunchCtx& c, bi_dtype dt, void* y, const void* x, const void* w,
                      const void* bias, int64_t M, int64_t K, int64_t N) {
    return pick_cols(c, BN, true) == 128 ? forward_impl<FMT, 128>(c, dt, y, x, w, bias, M, K, N)
                                         : forward_impl<FMT, 256>(c, dt, y, x, w, bias, M, K, N);
}

template <int FMT, int BNT>
cudaError_t dx_impl(const LaunchCtx& c, bi_dtype dt, void* dx, const void* dy, const void* w,
                    int64_t M, int64_t K, int64_t N) {
    CUtensorMap a, b;
    cudaError_t e;
    if ((e = make_map(&a, dt, dy, N, M, 1, BM)) != cudaSuccess) return e;  // dY [M,N], K-major
    if ((e = make_map(&b, dt, w, N, K, 1, BNT / 2)) != cudaSuccess) return e;  // W [K,N]: rows k, contraction n; half tile per CTA
    Params p{};
    p.out = dx; p.ldo = K; p.rows = M; p.cols = K;
    p.num_m = static_cast<int>((M + BM - 1) / BM);
    p.num_n = static_cast<int>((K + BNT - 1) / BNT);
    p.num_kb = static_cast<int>((N + BK - 1) / BK);
    CUtensorMap o;
    if ((e = make_out_map(&o, FMT, dx, K, M, K)) != cudaSuccess) return e;
    return launch_pair<FMT, FMT, false, false, DENSE, BNT>(c, a, b, p, &o);
}

template <int FMT>
cudaError_t dx_t(const LaunchCtx& c, bi_dtype dt, void* dx, const void* dy, const void* w,
                 int64_t M, int64_t K, int64_t N) {
    // (W is K-major here, but dX instantiates the 128- and 256-column tiles only)
    return pick_cols(c, BN, true) == 128 ? dx_impl<FMT, 128>(c, dt, dx, dy, w, M, K, N)
                                         : dx_impl<FMT, 256>(c, dt, dx, dy, w, M, K, N);
}

// Tile width of the 16-bit dW.  dW's output does not grow with the batch and
// the tile width does not enter the accumulation order (every output element
// is the same ascending chain of 64-wide contraction blocks, and the chunk
// split below is the same tree for either width), so the width may follow M,
// K and N: 256-column tiles, whose last partial wave runs in chunks, unless
// that gives fewer units than three quarters of a 152-SM GPU's 76 CTA pairs,
// in which case the 128-column tile (twice the tiles) keeps more pairs busy.
// Measured: GPT-2 up-projection dW (3 x 12 tiles of 256, 2 chunks each: 72
// units) 25.0 us with 256 columns against 27.0 with 128; the ragged 1000^3
// (16 tiles, 2 chunks: 32 units) 14.6 against 13.0.
constexpr int64_t DW_BUSY_UNITS = 57;
// dW's output tiles do not depend on M, and its contraction is the batch: the
// tiles of the last, partial wave (on a 152-SM GPU's 76 CTA pairs) run their
// contraction as s chunks of consecutive 64-row blocks, s pairs per tile, and
// dw_chunk_sum_kernel adds the chunks by the dW tree.  s = min(76 / tail tiles,
// 16, blocks / 8), a function of M, K and N only; 1 = no split.  Y and dX are
// never split: their rows must not depend on M.
constexpr int64_t DW_WAVE = 76;
constexpr int64_t DW_MIN_CHUNK_KB = 8;
int dw_split(int64_t tiles, int64_t nkb) {
    const int64_t tail = tiles % DW_WAVE;
    if (tail == 0) return 1;
    const int64_t sp = lmin(lmin(DW_WAVE / tail, DW_MAX_CHUNKS), nkb / DW_MIN_CHUNK_KB);
    return sp >= 2 ? static_cast<int>(sp) : 1;
}
struct DwShape {
    int bnt;        // tile columns
    int64_t tiles;  // output tiles of K x N
};
int64_t dw_tiles(int64_t K, int64_t N, int bnt) { return ((K + BM - 1) / BM + 1) / 2 * ((N + bnt - 1) / bnt); }
// len: rows of the first (longest) contraction piece
DwShape dw_shape(int64_t K, int64_t N, int64_t len, int forced = 0) {
    int bnt = forced;
    if (bnt != 128 && bnt != 256) {
        const int64_t t256 = dw_tiles(K, N, 256);
        bnt = t256 * dw_split(t256, (len + BK - 1) / BK) >= DW_BUSY_UNITS ? 256 : 128;
    }
    return {bnt, dw_tiles(K, N, bnt)};
}
int forced_cols(const LaunchCtx& c) { return c.eng ? c.eng->tile_cols : 0; }

template <int FMT, bool F32, int BNT>
cudaError_t dw_t(const LaunchCtx& c, bi_dtype dt, void* dw, const void* x, const void* dy,
                 int64_t M, int64_t K, int64_t N, float* ws) {
    // an f32 result over more than TC_PIECE_ROWS rows: pieces of that many rows,
    // each launch after the first adding its result to dW (a rounded dW takes
    // the whole contraction in one launch)
    const int64_t piece = F32 ? TC_PIECE_ROWS : M;  // M > 0 (the engine writes +0 for M = 0)
    for (int64_t d0 = 0; d0 < M; d0 += piece) {
        const int64_t len = lmin(piece, M - d0);
        CUtensorMap a, b;
        cudaError_t e;
        // X [M,K]: out k, contraction m; dY [M,N]: out n, contraction m (rows d0 .. d0 + len)
        if ((e = make_map(&a, dt, static_cast<const uint16_t*>(x) + d0 * K, K, len, 1, BK)) != cudaSuccess) return e;
        if ((e = make_map(&b, dt, static_cast<const uint16_t*>(dy) + d0 * N, N, len, 1, BK)) != cudaSuccess) return e;
        Params p{};
        p.out = dw; p.ldo = N; p.rows = K; p.cols = N;
        p.accum_out = d0 > 0 ? 1 : 0;
        p.num_m = static_cast<int>((K + BM - 1) / BM);
        p.num_n = static_cast<int>((N + BNT - 1) / BNT);
        p.num_kb = static_cast<int>((len + BK - 1) / BK);
        const int units_m = (p.num_m + 1) / 2;
        const int64_t tiles = static_cast<int64_t>(units_m) * p.num_n;
        const int sp = dw_split(tiles, p.num_kb);
        if (sp > 1 && ws == nullptr) return cudaErrorInvalidValue;
        p.split_s = sp;
        p.split_from = static_cast<int>(sp > 1 ? tiles - tiles % DW_WAVE : tiles);
        p.partials = ws;
        const int64_t split_tiles = tiles - p.split_from;
        CUtensorMap o, pmap;
        if ((e = make_out_map(&o, F32 ? 2 : FMT, dw, N, K, N)) != cudaSuccess) return e;
        if (sp > 1 && (e = make_out_map(&pmap, 2, ws, BNT, split_tiles * sp * 256, BNT)) != cudaSuccess) return e;
        if ((e = launch_pair<FMT, F32 ? 2 : FMT, true, true, DENSE, BNT>(c, a, b, p, &o, nullptr, nullptr,
                                                                          p.split_from + split_tiles * sp,
                                                                          sp > 1 ? &pmap : nullptr)) !=
            cudaSuccess)
            return e;
        if (sp > 1 && (e = launch_chunk_sum<F32 ? 2 : FMT>(c, ws, p.split_from, sp, split_tiles, units_m, p.num_n, BNT,
                                                           dw, p.ldo, p.rows, p.cols, p.accum_out, nullptr,
                                                           nullptr)) != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

template <int FMT, int BNT>
cudaError_t grouped_rows_impl(const LaunchCtx& c, bi_dtype dt, int dinput, void* out, const void* a_sorted,
                              const void* w, int64_t M, int64_t K, int64_t N, int64_t E, const uint32_t* seg,
                              const uint32_t* perm) {
    const int64_t L = dinput ? N : K;  // contraction
    const int64_t C = dinput ? K : N;  // output columns
    CUtensorMap a, b;
    cudaError_t e;
    // A = the row-sorted operand [M,L], K-major, 128 rows per CTA
    if ((e = make_map(&a, dt, a_sorted, L, M, 1, BM)) != cudaSuccess) return e;
    // B = W[g] [N,K] (3-D map): forward reads rows n (K-major, BNT / 2 per CTA);
    // dinput reads it with the output index k contiguous (MN-major)
    if ((e = make_map(&b, dt, w, K, N, E, dinput ? BK : BNT / 2, true)) != cudaSuccess) return e;
    Params p{};
    p.seg = seg; p.perm = perm; p.E = static_cast<int>(E);
    p.out = out; p.ldo = C; p.rows = M; p.cols = C;
    p.num_m = 0;
    p.num_n = static_cast<int>((C + BNT - 1) / BNT);
    p.num_kb = static_cast<int>((L + BK - 1) / BK);
    // the experts' 256-row tiles number at most floor(M / 256) + E
    const int64_t units = (M / GROUPED_TILE_ROWS + E) * p.num_n;
    if (dinput) {
        if constexpr (BNT == 128 || BNT == 256)
            return launch_pair<FMT, FMT, false, true, GROUPED_ROWS, BNT>(c, a, b, p, nullptr, nullptr, nullptr, units);
        return cudaErrorInvalidValue;
    }
    return launch_pair<FMT, FMT, false, false, GROUPED_ROWS, BNT>(c, a, b, p, nullptr, nullptr, nullptr, units);
}

template <int FMT>
cudaError_t grouped_rows_t(const LaunchCtx& c, bi_dtype dt, int dinput, void* out, const void* a_sorted,
                           const void* w, int64_t M, int64_t K, int64_t N, int64_t E, const uint32_t* seg,
                           const uint32_t* perm) {
    // 256 columns unless forced: narrower tiles measured slower for the grouped
    // workload (N = 1408 as 8 x 176 instead of 5.5 x 256: 112 against 103 us)
    const int cols = pick_cols(c, BN, dinput != 0);
    switch (cols) {
        case 128: return grouped_rows_impl<FMT, 128>(c, dt, dinput, out, a_sorted, w, M, K, N, E, seg, perm);
        case 176: return grouped_rows_impl<FMT, 176>(c, dt, dinput, out, a_sorted, w, M, K, N, E, seg, perm);
        case 192: return grouped_rows_impl<FMT, 192>(c, dt, dinput, out, a_sorted, w, M, K, N, E, seg, perm);
        default: return grouped_rows_impl<FMT, 256>(c, dt, dinput, out, a_sorted, w, M, K, N, E, seg, perm);
    }
}

// Grouped dweights: E x (N / 256) x (K / 256) units whatever the batch; the
// units of the last, partial wave on 76 CTA pairs contract in s chunks of
// consecutive 64-row blocks of the expert's rows in the piece (s = min(76 /
// tail units, 16, about 1 chunk per 8 blocks of an average expert), chosen
// from M, E, N and K), added by the dW tree in dw_chunk_sum_kernel.
struct GroupedDwSplit {
    int64_t units, split_from;
    int sp;
};
GroupedDwSplit grouped_dw_split(int64_t M, int64_t K, int64_t N, int64_t E) {
    const int64_t units_m = ((N + BM - 1) / BM + 1) / 2, num_n = (K + BN - 1) / BN;
    const int64_t units = E * units_m * num_n;
    const int64_t tail = units % DW_WAVE;
    const int64_t avg_kb = lmin(M / E, TC_PIECE_ROWS) / BK;  // blocks of an average expert in one piece
    int64_t sp = tail ? lmin(lmin(DW_WAVE / tail, DW_MAX_CHUNKS), avg_kb / DW_MIN_CHUNK_KB) : 1;
    if (sp < 2) sp = 1;
    return {units, sp > 1 ? units - tail : units, static_cast<int>(sp)};
}

template <int FMT>
cudaError_t grouped_dw_t(const LaunchCtx& c, bi_dtype dt, float* dw, const void* dy_sorted, const void* x_sorted,
                         const void* dy_tail, const void* x_tail, int64_t M, int64_t K, int64_t N, int64_t E,
                         const uint32_t* seg, float* ws) {
    // dW[g] [N,K] = sum over the expert's rows of dY^T X: both operands MN-major
    CUtensorMap a, b, a2, b2;
    cudaError_t e;
    if ((e = make_map(&a, dt, dy_sorted, N, M, 1, BK)) != cudaSuccess) return e;
    if ((e = make_map(&b, dt, x_sorted, K, M, 1, BK)) != cudaSuccess) return e;
    if ((e = make_map(&a2, dt, dy_tail, N, E * GROUPED_TAIL_ROWS, 1, BK)) != cudaSuccess) return e;
    if ((e = make_map(&b2, dt, x_tail, K, E * GROUPED_TAIL_ROWS, 1, BK)) != cudaSuccess) return e;
    Params p{};
    p.out = dw; p.ldo = K; p.rows = N; p.cols = K;
    p.seg = seg; p.E = static_cast<int>(E);
    p.num_m = static_cast<int>((N + BM - 1) / BM);
    p.num_n = static_cast<int>((K + BN - 1) / BN);
    p.num_kb = 0;
    const GroupedDwSplit sd = grouped_dw_split(M, K, N, E);
    if (sd.sp > 1 && ws == nullptr) return cudaErrorInvalidValue;
    p.split_s = sd.sp;
    p.split_from = static_cast<int>(sd.split_from);
    p.partials = ws;
    const int64_t split_units = sd.units - sd.split_from;
    const int64_t launch_units = sd.split_from + split_units * sd.sp;
    // one launch: each unit walks its expert's rows (or its chunk of them) in
    // pieces of TC_PIECE_ROWS rows counted from the expert's first row, adding
    // the pieces' results in order
    CUtensorMap o, pmap;  // dW [E][N][K]; the chunk partials
    if ((e = make_out_map(&o, 2, dw, K, N, K, E, true)) != cudaSuccess) return e;
    if (sd.sp > 1 && (e = make_out_map(&pmap, 2, ws, BN, split_units * sd.sp * 256, BN)) != cudaSuccess) return e;
    if ((e = launch_pair<FMT, 2, true, true, GROUPED_DW>(c, a, b, p, &o, &a2, &b2, launch_units,
                                                         sd.sp > 1 ? &pmap : nullptr)) != cudaSuccess)
        return e;
    if (sd.sp > 1)
        return launch_chunk_sum<2>(c, ws, p.split_from, sd.sp, split_units, (p.num_m + 1) / 2, p.num_n, BN, dw, p.ldo,
                                   p.rows, p.cols, 0, nullptr, nullptr, 1);
    return cudaSuccess;
}

// 8-bit row-major tensor [outer][inner], box {128, box_outer}, 128-byte swizzle.
cudaError_t make_map8(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_outer) {
    auto enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner};
    cuuint32_t box[2] = {128, box_outer};
    cuuint32_t es[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int OUT>
cudaError_t fp8_pass_t(const LaunchCtx& c, int pass, void* out, const uint8_t* a, const uint8_t* b,
                       const void* bias, const float* sa, const float* sb, int64_t M, int64_t K, int64_t N,
                       float* ws) {
    CUtensorMap ma, mb;
    cudaError_t e;
    Params p{};
    p.scale_a = sa; p.scale_b = sb; p.bias = bias;
    if (pass == 0) {         // y = xq wq: A = xq [M,K] K-major, B = wq [K,N] MN-major
        if ((e = make_map8(&ma, a, K, M, 128)) != cudaSuccess) return e;
        if ((e = make_map8(&mb, b, N, K, 128)) != cudaSuccess) return e;
        p.out = out; p.ldo = N; p.rows = M; p.cols = N;
        p.num_m = static_cast<int>((M + BM - 1) / BM);
        p.num_n = static_cast<int>((N + BN - 1) / BN);
        p.num_kb = static_cast<int>((K + 127) / 128);
        CUtensorMap o;
        if ((e = make_out_map(&o, OUT, out, N, M, N)) != cudaSuccess) return e;
        return launch_pair<2, OUT, false, true>(c, ma, mb, p, &o);
    }
    if (pass == 1) {         // dx = gq wq^T: A = gq [M,N] K-major, B = wq [K,N] rows k, contraction n
        if ((e = make_map8(&ma, a, N, M, 128)) != cudaSuccess) return e;
        if ((e = make_map8(&mb, b, N, K, 128)) != cudaSuccess) return e;
        p.out = out; p.ldo = K; p.rows = M; p.cols = K;
        p.num_m = static_cast<int>((M + BM - 1) / BM);
        p.num_n = static_cast<int>((K + BN - 1) / BN);
        p.num_kb = static_cast<int>((N + 127) / 128);
        CUtensorMap o;
        if ((e = make_out_map(&o, OUT, out, K, M, K)) != cudaSuccess) return e;
        return launch_pair<2, OUT, false, false>(c, ma, mb, p, &o);
    }
    // dw = xq^T gq: A = xq [M,K] (out k, contraction m), B = gq [M,N] (out n, contraction m);
    // an f32 result in pieces of TC_PIECE_ROWS rows, as for the 16-bit dW
    const int64_t piece = OUT == 2 ? TC_PIECE_ROWS : M;
    for (int64_t d0 = 0; d0 < M; d0 += piece) {
        const int64_t len = lmin(piece, M - d0);
        if ((e = make_map8(&ma, a + d0 * K, K, len, 128)) != cudaSuccess) return e;
        if ((e = make_map8(&mb, b + d0 * N, N, len, 128)) != cudaSuccess) return e;
        p.out = out; p.ldo = N; p.rows = K; p.cols = N; p.bias = nullptr;
        p.accum_out = d0 > 0 ? 1 : 0;
        p.num_m = static_cast<int>((K + BM - 1) / BM);
        p.num_n = static_cast<int>((N + BN - 1) / BN);
        p.num_kb = static_cast<int>((len + 127) / 128);
        // the last wave's tiles in chunks, as for the 16-bit dW
        const int units_m = (p.num_m + 1) / 2;
        const int64_t tiles = static_cast<int64_t>(units_m) * p.num_n;
        const int sp = dw_split(tiles, p.num_kb);
        if (sp > 1 && ws == nullptr) return cudaErrorInvalidValue;
        p.split_s = sp;
        p.split_from = static_cast<int>(sp > 1 ? tiles - tiles % DW_WAVE : tiles);
        p.partials = ws;
        const int64_t split_tiles = tiles - p.split_from;
        CUtensorMap o, pmap;
        if ((e = make_out_map(&o, OUT, out, N, K, N)) != cudaSuccess) return e;
        if (sp > 1 && (e = make_out_map(&pmap, 2, ws, BN, split_tiles * sp * 256, BN)) != cudaSuccess) return e;
        if ((e = launch_pair<2, OUT, true, true>(c, ma, mb, p, &o, nullptr, nullptr, p.split_from + split_tiles * sp,
                                                 sp > 1 ? &pmap : nullptr)) !=
            cudaSuccess)
            return e;
        if (sp > 1 && (e = launch_chunk_sum<OUT>(c, ws, p.split_from, sp, split_tiles, units_m, p.num_n, BN, out,
                                                 p.ldo, p.rows, p.cols, p.accum_out, sa, sb)) != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

// 32-bit K-major tensor [outer][inner] with row stride ld elements (ld >= inner,
// a multiple of 4), box {32, 128}, 128-byte swizzle.
cudaError_t make_map32(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint64_t ld) {
    auto enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {ld * 4};
    cuuint32_t box[2] = {32, 128};
    cuuint32_t es[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(ptr), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

cudaError_t tc_forward(const LaunchCtx& c, bi_dtype dt, void* y, const void* x, const void* w,
                       const void* bias, int64_t M, int64_t K, int64_t N) {
    return dt == BI_BF16 ? forward_t<1>(c, dt, y, x, w, bias, M, K, N)
                         : forward_t<0>(c, dt, y, x, w, bias, M, K, N);
}

cudaError_t tc_dx(const LaunchCtx& c, bi_dtype dt, void* dx, const void* dy, const void* w,
                  int64_t M, int64_t K, int64_t N) {
    return dt == BI_BF16 ? dx_t<1>(c, dt, dx, dy, w, M, K, N) : dx_t<0>(c, dt, dx, dy, w, M, K, N);
}

int64_t tc_dw_workspace_bytes(const LaunchCtx& c, int dw_f32, int64_t M, int64_t K, int64_t N) {
    const int64_t len = dw_f32 ? lmin(M, TC_PIECE_ROWS) : M;  // the first (longest) contraction piece
    const DwShape d = dw_shape(K, N, len, forced_cols(c));
    const int sp = dw_split(d.tiles, (len + BK - 1) / BK);
    return sp > 1 ? (d.tiles % DW_WAVE) * sp * 256 * d.bnt * 4 : 0;
}

cudaError_t tc_dw(const LaunchCtx& c, bi_dtype dt, void* dw, int dw_f32, const void* x,
                  const void* dy, int64_t M, int64_t K, int64_t N, float* ws) {
    const bool nw = dw_shape(K, N, dw_f32 ? lmin(M, TC_PIECE_ROWS) : M, forced_cols(c)).bnt == 128;
    if (dt == BI_BF16) {
        if (dw_f32) return nw ? dw_t<1, true, 128>(c, dt, dw, x, dy, M, K, N, ws) : dw_t<1, true, 256>(c, dt, dw, x, dy, M, K, N, ws);
        return nw ? dw_t<1, false, 128>(c, dt, dw, x, dy, M, K, N, ws) : dw_t<1, false, 256>(c, dt, dw, x, dy, M, K, N, ws);
    }
    if (dw_f32) return nw ? dw_t<0, true, 128>(c, dt, dw, x, dy, M, K, N, ws) : dw_t<0, true, 256>(c, dt, dw, x, dy, M, K, N, ws);
    return nw ? dw_t<0, false, 128>(c, dt, dw, x, dy, M, K, N, ws) : dw_t<0, false, 256>(c, dt, dw, x, dy, M, K, N, ws);
}

cudaError_t tc_grouped_rows(const LaunchCtx& c, bi_dtype dt, int pass_dinput, void* out, const void* a_sorted,
                            const void* w, int64_t M, int64_t K, int64_t N, int64_t E, const uint32_t* seg,
                            const uint32_t* perm) {
    return dt == BI_BF16 ? grouped_rows_t<1>(c, dt, pass_dinput, out, a_sorted, w, M, K, N, E, seg, perm)
                         : grouped_rows_t<0>(c, dt, pass_dinput, out, a_sorted, w, M, K, N, E, seg, perm);
}

cudaError_t tc_tf32x3_pass(const LaunchCtx& c, const float* a_hi, const float* a_lo, int64_t lda,
                           const float* b_hi, const float* b_lo, int64_t ldb, float* out, int64_t ldo,
                           const float* bias, int64_t rows, int64_t cols, int64_t depth) {
    // one launch per contraction piece: the first writes out, each later one adds
    // its result to out (in piece order), the last one adds the bias
    for (int64_t d0 = 0; d0 < depth; d0 += TF32X3_PIECE) {  // d0 % 4 == 0: 16-byte aligned bases
        const int64_t len = lmin(TF32X3_PIECE, depth - d0);
        CUtensorMap ah, al, bh, bl;
        cudaError_t e;
        if ((e = make_map32(&ah, a_hi + d0, len, rows, lda)) != cudaSuccess) return e;
        if ((e = make_map32(&al, a_lo + d0, len, rows, lda)) != cudaSuccess) return e;
        if ((e = make_map32(&bh, b_hi + d0, len, cols, ldb)) != cudaSuccess) return e;
        if ((e = make_map32(&bl, b_lo + d0, len, cols, ldb)) != cudaSuccess) return e;
        Params p{};
        p.out = out; p.ldo = ldo; p.rows = rows; p.cols = cols;
        p.bias = d0 + len == depth ? bias : nullptr;
        p.accum_out = d0 > 0 ? 1 : 0;
        p.num_m = static_cast<int>((rows + BM - 1) / BM);
        p.num_n = static_cast<int>((cols + BN - 1) / BN);
        p.num_kb = static_cast<int>((len + 31) / 32);
        CUtensorMap o;
        if ((e = make_out_map(&o, 2, out, cols, rows, ldo)) != cudaSuccess) return e;
        if ((e = launch_pair<3, 2, false, false>(c, ah, bh, p, &o, &al, &bl)) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

int64_t tc_fp8_dw_workspace_bytes(int out_f32, int64_t M, int64_t K, int64_t N) {
    const int64_t tiles = ((K + BM - 1) / BM + 1) / 2 * ((N + BN - 1) / BN);
    const int64_t len = out_f32 ? lmin(M, TC_PIECE_ROWS) : M;  // the first (longest) contraction piece
    const int sp = dw_split(tiles, (len + 127) / 128);
    return sp > 1 ? (tiles % DW_WAVE) * sp * 256 * BN * 4 : 0;
}

cudaError_t tc_fp8_pass(const LaunchCtx& c, int pass, bi_dtype out_dt, void* out, const uint8_t* a,
                       const uint8_t* b, const void* bias, const float* sa, const float* sb, int64_t M,
                       int64_t K, int64_t N, float* ws) {
    switch (out_dt) {
        case BI_BF16: return fp8_pass_t<1>(c, pass, out, a, b, bias, sa, sb, M, K, N, ws);
        case BI_F16: return fp8_pass_t<0>(c, pass, out, a, b, bias, sa, sb, M, K, N, ws);
        default: return fp8_pass_t<2>(c, pass, out, a, b, bias, sa, sb, M, K, N, ws);
    }
}

int64_t tc_grouped_dw_workspace_bytes(int64_t M, int64_t K, int64_t N, int64_t E) {
    const GroupedDwSplit sd = grouped_dw_split(M, K, N, E);
    return sd.sp > 1 ? (sd.units - sd.split_from) * sd.sp * 256 * BN * 4 : 0;
}

cudaError_t tc_grouped_dw(const LaunchCtx& c, bi_dtype dt, float* dw, const void* dy_sorted, const void* x_sorted,
                          const void* dy_tail, const void* x_tail, int64_t M, int64_t K, int64_t N, int64_t E,
                          const uint32_t* seg, float* ws) {
    return dt == BI_BF16 ? grouped_dw_t<1>(c, dt, dw, dy_sorted, x_sorted, dy_tail, x_tail, M, K, N, E, seg, ws)
                         : grouped_dw_t<0>(c, dt, dw, dy_sorted, x_sorted, dy_tail, x_tail, M, K, N, E, seg, ws);
}

}  // namespace bi
