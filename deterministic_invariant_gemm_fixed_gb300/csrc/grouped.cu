// Grouping of rows by expert id for the grouped matmul.
//
// Source: rublas 0.1.45 src/tensor_grouped/mod.rs -- ids outside [0,E) are
// padding and produce zero rows (fn grouped_matmul_nt); the segmented backward
// takes `offsets` [E+1] that describe the same grouping as `row_experts`
// (fn grouped_matmul_nt_backward_segmented_with_strategy).  Here the library
// builds that grouping itself, on the device, as a stable counting sort:
//
//   1. count:   each block counts the ids of its slice of rows per bucket
//               (bucket = id for id < E, bucket E = padding);
//   2. scan:    exclusive prefix over (bucket, block) in bucket-major order gives
//               every block its first output position per bucket, the group
//               offsets, and each expert's first 256-row tile (tensor-core tier);
//   3. scatter: each block walks its slice in row order, 256 rows at a time; a
//               row's position is its block's running base for its bucket plus
//               the number of earlier rows of that bucket in the same 256-row
//               step.  No atomics anywhere: positions are a pure function of the
//               ids, so the permutation is stable and run-to-run identical.
#include "bi_internal.h"

namespace bi {
namespace {

constexpr int SEG_THREADS = 256;
constexpr int SEG_ROWS_PER_BLOCK = 256;  // one step per block: many blocks in flight
constexpr uint32_t NONE = 0xffffffffu;

__device__ __forceinline__ uint32_t bucket_of(uint32_t id, uint32_t E) { return id < E ? id : E; }

// For the row held by thread `tid` in a 256-row step staged in sb[]: number of
// earlier rows with the same bucket, and whether no later row shares it.
__device__ __forceinline__ void rank_in_step(const uint32_t* sb, int tid, uint32_t g, uint32_t& rank,
                                             bool& last) {
    uint32_t before = 0, after = 0;
#pragma unroll 8
    for (int j = 0; j < SEG_THREADS; ++j) {
        const uint32_t same = sb[j] == g;
        before += (j < tid) & same;
        after += (j > tid) & same;
    }
    rank = before;
    last = after == 0;
}

// ---- fast path: E + 1 <= 1024 buckets and (E + 1) x blocks <= 16384 ------
//
// 512 rows per block, one per thread.  Within a warp, __match_any_sync finds
// the lanes holding the same bucket; a row's rank among them is the number of
// such lanes below it.  Each warp's count per bucket goes to shared memory,
// and a prefix over the 16 warps (per bucket, warp order) gives each warp's
// first rank in the block.  So a row's rank in its block is a pure function of
// the ids (rows in ascending order), without atomics, and two launches do the
// whole grouping: one writes every block's count per bucket, the other
// recomputes the ranks, adds the block's base (all rows of lower buckets plus
// the bucket's rows in earlier blocks) and scatters.
constexpr int SEGF_THREADS = 512;
constexpr int SEGF_WARPS = SEGF_THREADS / 32;
constexpr int SEGF_MAX_BUCKETS = 1024;
constexpr int64_t SEGF_MAX_TABLE = 16384;

// Ranks of this thread's row (row b * 512 + tid) within its warp and the warp's
// first rank per bucket: on return wc[w * (E + 1) + g] holds the number of
// rows of bucket g in warps 0 .. w-1 of the block, and tot[g] the block's
// count of bucket g.  Returns the row's bucket (NONE past M) and its rank
// among the block's rows of that bucket.
__device__ __forceinline__ uint32_t block_rank(const uint32_t* ids, int64_t M, uint32_t E, int64_t b, uint16_t* wc,
                                               uint32_t* tot, uint32_t& rank) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t nb = E + 1;
    const int64_t r = b * SEGF_THREADS + tid;
    const uint32_t g = r < M ? bucket_of(ids[r], E) : NONE;
    for (uint32_t i = tid; i < SEGF_WARPS * nb; i += SEGF_THREADS) wc[i] = 0;
    __syncthreads();
    const uint32_t peers = __match_any_sync(0xffffffffu, g);
    const uint32_t lower = peers & ((1u << lane) - 1u);
    if (g != NONE && lower == 0) wc[warp * nb + g] = static_cast<uint16_t>(__popc(peers));
    __syncthreads();
    for (uint32_t q = tid; q < nb; q += SEGF_THREADS) {
        uint32_t run = 0;
#pragma unroll
        for (int w = 0; w < SEGF_WARPS; ++w) {
            const uint32_t t = wc[w * nb + q];
            wc[w * nb + q] = static_cast<uint16_t>(run);
            run += t;
        }
        tot[q] = run;
    }
    __syncthreads();
    rank = g != NONE ? wc[warp * nb + g] + __popc(lower) : 0;
    return g;
}

// counts[b * (E + 1) + g] = rows of bucket g in block b.
__global__ void __launch_bounds__(SEGF_THREADS)
    seg_count_fast_kernel(const uint32_t* ids, int64_t M, uint32_t E, uint32_t* counts) {
    grid_dep_wait();
    grid_dep_launch();
    __shared__ uint16_t wc[SEGF_WARPS * SEGF_MAX_BUCKETS];
    __shared__ uint32_t tot[SEGF_MAX_BUCKETS];
    uint32_t rank;
    block_rank(ids, M, E, blockIdx.x, wc, tot, rank);
    for (uint32_t q = threadIdx.x; q <= E; q += SEGF_THREADS) counts[blockIdx.x * (E + 1) + q] = tot[q];
}

// In-place exclusive prefix sum of v[0 .. n) (n <= 1024) by one block of 512
// threads (two entries per thread); returns the total to every thread.
__device__ uint32_t block_exclusive_scan(uint32_t* v, uint32_t n, uint32_t* warp_tmp) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t i0 = 2 * tid, i1 = 2 * tid + 1;
    const uint32_t a = i0 < n ? v[i0] : 0, c = i1 < n ? v[i1] : 0;
    uint32_t x = a + c;  // inclusive scan of the pair sums within the warp
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_tmp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        uint32_t s = lane < SEGF_WARPS ? warp_tmp[lane] : 0;
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        if (lane < SEGF_WARPS) warp_tmp[lane] = s;  // inclusive over warps
    }
    __syncthreads();
    const uint32_t before = (warp ? warp_tmp[warp - 1] : 0) + x - (a + c);
    const uint32_t total = warp_tmp[SEGF_WARPS - 1];
    __syncthreads();
    if (i0 < n) v[i0] = before;
    if (i1 < n) v[i1] = before + a;
    __syncthreads();
    return total;
}

__device__ void write_tile_starts(uint32_t* seg, uint32_t E);

// perm[position] = row; block 0 also writes the segment table.
__global__ void __launch_bounds__(SEGF_THREADS)
    seg_scatter_fast_kernel(const uint32_t* ids, int64_t M, uint32_t E, const uint32_t* counts, int64_t NB,
                            uint32_t* seg, uint32_t* perm) {
    grid_dep_wait();
    grid_dep_launch();
    __shared__ __align__(16) uint16_t wc[SEGF_WARPS * SEGF_MAX_BUCKETS];  // later reused for 2 x 512 u32
    __shared__ uint32_t tot[SEGF_MAX_BUCKETS];
    __shared__ uint32_t base[SEGF_MAX_BUCKETS];
    __shared__ uint32_t warp_tmp[32];
    const int64_t b = blockIdx.x;
    uint32_t rank;
    const uint32_t g = block_rank(ids, M, E, b, wc, tot, rank);
    // all rows of bucket q (tot) and those in blocks before this one (base).
    // With at most 512 buckets, the threads split the blocks among them
    // (thread = bucket + nb * slice, blocks slice, slice + slices, ...; coalesced
    // rows of counts) and one thread per bucket adds the slices' sums.
    const uint32_t nb = E + 1;
    if (nb <= SEGF_THREADS) {
        const uint32_t slices = SEGF_THREADS / nb;
        uint32_t* red_all = reinterpret_cast<uint32_t*>(wc);  // the warp ranks are in registers now
        uint32_t* red_before = red_all + SEGF_THREADS;
        __syncthreads();
        if (threadIdx.x < slices * nb) {
            const uint32_t q = threadIdx.x % nb, sl = threadIdx.x / nb;
            uint32_t all = 0, before = 0;
            for (int64_t bb = sl; bb < NB; bb += slices) {
                const uint32_t v = counts[bb * nb + q];
                before += bb < b ? v : 0;
                all += v;
            }
            red_all[threadIdx.x] = all;
            red_before[threadIdx.x] = before;
        }
        __syncthreads();
        if (threadIdx.x < nb) {
            uint32_t all = 0, before = 0;
            for (uint32_t sl = 0; sl < slices; ++sl) {
                all += red_all[sl * nb + threadIdx.x];
                before += red_before[sl * nb + threadIdx.x];
            }
            tot[threadIdx.x] = all;
            base[threadIdx.x] = before;
        }
    } else {
        for (uint32_t q = threadIdx.x; q < nb; q += SEGF_THREADS) {
            uint32_t all = 0, before = 0;
#pragma unroll 8
            for (int64_t bb = 0; bb < NB; ++bb) {
                const uint32_t v = counts[bb * nb + q];
                before += bb < b ? v : 0;
                all += v;
            }
            tot[q] = all;
            base[q] = before;
        }
    }
    __syncthreads();
    block_exclusive_scan(tot, E + 1, warp_tmp);  // tot[q] = first sorted position of bucket q
    if (g != NONE) perm[tot[g] + base[g] + rank] = static_cast<uint32_t>(b * SEGF_THREADS + threadIdx.x);
    if (b == 0) {
        for (uint32_t q = threadIdx.x; q <= E; q += SEGF_THREADS) seg[q] = tot[q];
        __syncthreads();
        if (threadIdx.x == 0) {
            seg[E + 1] = static_cast<uint32_t>(M);
            write_tile_starts(seg, E);
        }
    }
}

__global__ void __launch_bounds__(SEG_THREADS)
    seg_count_kernel(const uint32_t* ids, int64_t M, uint32_t E, uint32_t* hist, int64_t NB) {
    grid_dep_wait();
    grid_dep_launch();
    __shared__ uint32_t sb[SEG_THREADS];
    const int64_t b = blockIdx.x;
    const int64_t begin = b * SEG_ROWS_PER_BLOCK;
    const int64_t end = lmin(M, begin + SEG_ROWS_PER_BLOCK);
    for (int64_t g = threadIdx.x; g <= E; g += SEG_THREADS) hist[g * NB + b] = 0;
    __syncthreads();
    for (int64_t base = begin; base < end; base += SEG_THREADS) {
        const int64_t r = base + threadIdx.x;
        sb[threadIdx.x] = r < end ? bucket_of(ids[r], E) : NONE;
        __syncthreads();
        const uint32_t g = sb[threadIdx.x];
        if (g != NONE) {
            uint32_t rank;
            bool last;
            rank_in_step(sb, threadIdx.x, g, rank, last);
            if (last) hist[g * NB + b] += rank + 1;  // the only writer of this entry in this step
        }
        __syncthreads();
    }
}

// First tile of each expert in the tensor-core grouped passes: the prefix sum of
// ceil(count / GROUPED_TILE_ROWS), written after the offsets (one thread).
__device__ void write_tile_starts(uint32_t* seg, uint32_t E) {
    uint32_t ts = 0;
    for (uint32_t g = 0; g < E; ++g) {
        seg[E + 2 + g] = ts;
        ts += (seg[g + 1] - seg[g] + GROUPED_TILE_ROWS - 1) / GROUPED_TILE_ROWS;
    }
    seg[E + 2 + E] = ts;
    seg[2 * E + 3] = ts;
}

// One block.  hist (bucket-major, (E+1)*NB entries) becomes its exclusive
// prefix sum; seg receives offsets[0..E+1] and the tile starts.
__global__ void __launch_bounds__(1024)
    seg_scan_kernel(uint32_t* hist, int64_t NB, uint32_t E, int64_t M, uint32_t* seg) {
    grid_dep_wait();
    grid_dep_launch();
    __shared__ uint32_t warp_sums[32];
    __shared__ uint32_t carry;
    const int64_t total = (static_cast<int64_t>(E) + 1) * NB;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    for (int64_t base = 0; base < total; base += 1024) {
        const int64_t i = base + threadIdx.x;
        const uint32_t v = i < total ? hist[i] : 0;
        uint32_t x = v;  // inclusive scan within the warp
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_sums[warp] = x;
        __syncthreads();
        if (warp == 0) {
            uint32_t s = warp_sums[lane];
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, s, o);
                if (lane >= o) s += y;
            }
            warp_sums[lane] = s;  // inclusive over warps
        }
        __syncthreads();
        const uint32_t before = carry + (warp ? warp_sums[warp - 1] : 0) + x - v;
        if (i < total) hist[i] = before;
        __syncthreads();
        if (threadIdx.x == 1023) carry = before + v;
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        for (uint32_t g = 0; g <= E; ++g) seg[g] = hist[static_cast<int64_t>(g) * NB];
        seg[E + 1] = static_cast<uint32_t>(M);
        write_tile_starts(seg, E);
    }
}

__global__ void __launch_bounds__(SEG_THREADS)
    seg_scatter_kernel(const uint32_t* ids, int64_t M, uint32_t E, uint32_t* base_pos, int64_t NB,
                       uint32_t* perm) {
    grid_dep_wait();
    grid_dep_launch();
    __shared__ uint32_t sb[SEG_THREADS];
    const int64_t b = blockIdx.x;
    const int64_t begin = b * SEG_ROWS_PER_BLOCK;
    const int64_t end = lmin(M, begin + SEG_ROWS_PER_BLOCK);
    for (int64_t base = begin; base < end; base += SEG_THREADS) {
        const int64_t r = base + threadIdx.x;
        sb[threadIdx.x] = r < end ? bucket_of(ids[r], E) : NONE;
        __syncthreads();
        const uint32_t g = sb[threadIdx.x];
        uint32_t rank = 0;
        bool last = false;
        if (g != NONE) {
            rank_in_step(sb, threadIdx.x, g, rank, last);
            perm[base_pos[g * NB + b] + rank] = static_cast<uint32_t>(r);
        }
        __syncthreads();  // every row of this step has read the old base
        if (g != NONE && last) base_pos[g * NB + b] += rank + 1;
        __syncthreads();
    }
}

// Segment table from caller offsets (block 0, thread 0) and the identity
// permutation (all threads).  The clamp keeps every later index in bounds
// whatever the caller passed.
__global__ void seg_from_offsets_kernel(const uint32_t* offsets, int64_t M, uint32_t E, uint32_t* seg,
                                        uint32_t* perm, int* status) {
    grid_dep_wait();
    grid_dep_launch();
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        const uint32_t m = static_cast<uint32_t>(M);
        bool bad = offsets[0] != 0;
        uint32_t prev = 0;
        seg[0] = 0;
        for (uint32_t g = 1; g <= E; ++g) {
            const uint32_t v = offsets[g];
            const uint32_t cl = v < prev ? prev : (v > m ? m : v);
            bad |= cl != v;
            seg[g] = cl;
            prev = cl;
        }
        seg[E + 1] = m;
        write_tile_starts(seg, E);
        if (bad && status) *reinterpret_cast<volatile int*>(status) = DEV_BAD_OFFSETS;
    }
    for (int64_t r = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; r < M;
         r += static_cast<int64_t>(gridDim.x) * blockDim.x)
        perm[r] = static_cast<uint32_t>(r);
}

// dst row s (s < offsets[E]) = src row perm[s]; one row per block step.  With
// zout, the padding rows (sorted positions offsets[E] .. M) of that output are
// zeroed too: the grouped GEMM never writes them.
__global__ void gather_sorted_kernel(const uint4* src, int64_t L16, uint32_t E, const uint32_t* seg,
                                     const uint32_t* perm, uint4* dst, uint4* zout, int64_t Z16) {
    grid_dep_wait();
    grid_dep_launch();
    const int64_t rows = seg[E];
    const int64_t all = zout ? static_cast<int64_t>(seg[E + 1]) : rows;
    for (int64_t r = blockIdx.x; r < all; r += gridDim.x) {
        if (r < rows) {
            const uint4* sp = src + static_cast<int64_t>(perm[r]) * L16;
            uint4* d = dst + r * L16;
            for (int64_t i = threadIdx.x; i < L16; i += blockDim.x) d[i] = __ldg(sp + i);
        } else {
            uint4* d = zout + static_cast<int64_t>(perm[r]) * Z16;
            const uint4 z = make_uint4(0, 0, 0, 0);
            for (int64_t i = threadIdx.x; i < Z16; i += blockDim.x) d[i] = z;
        }
    }
}

// dst row q = g*64 + l: expert g's sorted row (its last multiple of 64) + l, if
// the expert has it, else zeros.
__global__ void build_tails_kernel(const uint4* src, int64_t L16, uint32_t E, const uint32_t* seg,
                                   const uint32_t* perm, uint4* dst) {
    grid_dep_wait();
    grid_dep_launch();
    const int64_t rows = static_cast<int64_t>(E) * GROUPED_TAIL_ROWS;
    for (int64_t q = blockIdx.x; q < rows; q += gridDim.x) {
        const uint32_t g = static_cast<uint32_t>(q / GROUPED_TAIL_ROWS);
        const uint32_t l = static_cast<uint32_t>(q % GROUPED_TAIL_ROWS);
        const uint32_t cnt = seg[g + 1] - seg[g];
        const uint32_t pos = cnt / GROUPED_TAIL_ROWS * GROUPED_TAIL_ROWS + l;
        uint4* d = dst + q * L16;
        if (pos < cnt) {
            const uint4* sp = src + static_cast<int64_t>(perm[seg[g] + pos]) * L16;
            for (int64_t i = threadIdx.x; i < L16; i += blockDim.x) d[i] = __ldg(sp + i);
        } else {
            const uint4 z = make_uint4(0, 0, 0, 0);
            for (int64_t i = threadIdx.x; i < L16; i += blockDim.x) d[i] = z;
        }
    }
}

__global__ void zero_rows_kernel(uint8_t* out, int64_t row_bytes, uint32_t E, const uint32_t* seg,
                                 const uint32_t* perm) {
    grid_dep_wait();
    grid_dep_launch();
    const int64_t first = seg[E], end = seg[E + 1];
    for (int64_t s = first + blockIdx.x; s < end; s += gridDim.x) {
        uint8_t* d = out + static_cast<int64_t>(perm[s]) * row_bytes;
        for (int64_t i = threadIdx.x; i < row_bytes; i += blockDim.x) d[i] = 0;
    }
}

__device__ __forceinline__ unsigned long long gtimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits on an mbarrier that nothing ever completes, bounded by `limit`, then
// records the timeout the same way the GEMM pipeline does.
__global__ void selftest_wait_kernel(int* status, unsigned long long limit) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(&bar));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(a) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    const unsigned long long t0 = gtimer();
    for (;;) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n\t"
            "selp.b32 %0, 1, 0, p;\n\t}\n"
            : "=r"(ok)
            : "r"(a)
            : "memory");
        if (ok) return;
        if (gtimer() - t0 > limit) {
            *reinterpret_cast<volatile int*>(status) = DEV_TIMEOUT_SELFTEST;
            return;
        }
    }
}

int64_t num_seg_blocks(int64_t M) { return (M + SEG_ROWS_PER_BLOCK - 1) / SEG_ROWS_PER_BLOCK; }

}  // namespace

int64_t segment_scratch_bytes(int64_t M, int64_t E) {
    return (E + 1) * (num_seg_blocks(M) > 0 ? num_seg_blocks(M) : 1) * 4;
}

cudaError_t segment(const LaunchCtx& c, const uint32_t* ids, int64_t M, int64_t E, uint32_t* seg,
                    uint32_t* perm, void* scratch) {
    const int64_t NBF = (M + SEGF_THREADS - 1) / SEGF_THREADS;
    if (M > 0 && E + 1 <= SEGF_MAX_BUCKETS && (E + 1) * NBF <= SEGF_MAX_TABLE) {
        // two launches; counts[(E+1) * NBF] fits in the scratch of the general path
        uint32_t* counts = static_cast<uint32_t*>(scratch);
        cudaError_t e = launch_pdl(seg_count_fast_kernel, dim3(static_cast<unsigned>(NBF)), dim3(SEGF_THREADS), 0,
                                   c.stream, ids, M, static_cast<uint32_t>(E), counts);
        if (e != cudaSuccess) return e;
        c.count();
        e = launch_pdl(seg_scatter_fast_kernel, dim3(static_cast<unsigned>(NBF)), dim3(SEGF_THREADS), 0, c.stream,
                       ids, M, static_cast<uint32_t>(E), static_cast<const uint32_t*>(counts), NBF, seg, perm);
        if (e != cudaSuccess) return e;
        c.count();
        return cudaGetLastError();
    }
    const int64_t NB = num_seg_blocks(M) > 0 ? num_seg_blocks(M) : 1;
    uint32_t* hist = static_cast<uint32_t*>(scratch);
    if (M > 0) {
        const cudaError_t e = launch_pdl(seg_count_kernel, dim3(static_cast<unsigned>(NB)), dim3(SEG_THREADS), 0,
                                         c.stream, ids, M, static_cast<uint32_t>(E), hist, NB);
        if (e != cudaSuccess) return e;
        c.count();
    } else {
        cudaError_t e = cudaMemsetAsync(hist, 0, (E + 1) * NB * 4, c.stream);
        if (e != cudaSuccess) return e;
    }
    cudaError_t e = launch_pdl(seg_scan_kernel, dim3(1), dim3(1024), 0, c.stream, hist, NB, static_cast<uint32_t>(E),
                               M, seg);
    if (e != cudaSuccess) return e;
    c.count();
    if (M > 0) {
        e = launch_pdl(seg_scatter_kernel, dim3(static_cast<unsigned>(NB)), dim3(SEG_THREADS), 0, c.stream, ids, M,
                       static_cast<uint32_t>(E), hist, NB, perm);
        if (e != cudaSuccess) return e;
        c.count();
    }
    return cudaGetLastError();
}

cudaError_t segment_from_offsets(const LaunchCtx& c, const uint32_t* offsets, int64_t M, int64_t E,
                                 uint32_t* seg, uint32_t* perm) {
    int64_t blocks = (M + 255) / 256;
    if (blocks > static_cast<int64_t>(c.sm_count) * 8) blocks = static_cast<int64_t>(c.sm_count) * 8;
    if (blocks < 1) blocks = 1;
    const cudaError_t e = launch_pdl(seg_from_offsets_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0,
                                     c.stream, offsets, M, static_cast<uint32_t>(E), seg, perm, c.status);
    if (e != cudaSuccess) return e;
    c.count();
    return cudaGetLastError();
}

cudaError_t gather_sorted(const LaunchCtx& c, const void* src, int64_t M, int64_t L, int64_t E,
                          const uint32_t* seg, const uint32_t* perm, void* dst, void* zero_out, int64_t zero_C) {
    if (M == 0) return cudaSuccess;
    const int64_t L16 = L * 2 / 16;  // 16-bit data, L a multiple of 8
    const int64_t Z16 = zero_C * 2 / 16;  // 16-bit output rows, zero_C a multiple of 8
    const int64_t cap = static_cast<int64_t>(c.sm_count) * 16;
    const int64_t blocks = M < cap ? M : cap;
    const cudaError_t e = launch_pdl(gather_sorted_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, c.stream,
                                     static_cast<const uint4*>(src), L16, static_cast<uint32_t>(E), seg, perm,
                                     static_cast<uint4*>(dst), static_cast<uint4*>(zero_out), Z16);
    if (e != cudaSuccess) return e;
    c.count();
    return cudaGetLastError();
}

cudaError_t build_tails(const LaunchCtx& c, const void* src, int64_t L, int64_t E, const uint32_t* seg,
                        const uint32_t* perm, void* dst) {
    const int64_t L16 = L * 2 / 16;
    const int64_t rows = E * GROUPED_TAIL_ROWS;
    const int64_t cap = static_cast<int64_t>(c.sm_count) * 16;
    const int64_t blocks = rows < cap ? rows : cap;
    const cudaError_t e = launch_pdl(build_tails_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, c.stream,
                                     static_cast<const uint4*>(src), L16, static_cast<uint32_t>(E), seg, perm,
                                     static_cast<uint4*>(dst));
    if (e != cudaSuccess) return e;
    c.count();
    return cudaGetLastError();
}

cudaError_t zero_padding_rows(const LaunchCtx& c, void* out, int64_t C, int esize, int64_t E,
                              const uint32_t* seg, const uint32_t* perm) {
    const unsigned blocks = static_cast<unsigned>(c.sm_count * 4);
    const cudaError_t e = launch_pdl(zero_rows_kernel, dim3(blocks), dim3(256), 0, c.stream, static_cast<uint8_t*>(out),
                                     C * esize, static_cast<uint32_t>(E), seg, perm);
    if (e != cudaSuccess) return e;
    c.count();
    return cudaGetLastError();
}

cudaError_t selftest_wait(const LaunchCtx& c) {
    selftest_wait_kernel<<<1, 1, 0, c.stream>>>(c.status, c.wait_limit_ns);
    c.count();
    return cudaGetLastError();
}

}  // namespace bi
