// grouped_gemm.cuh -- the expert FFN as grouped GEMMs on the 5th-generation
// tensor cores (tcgen05 + TMEM, operands staged by TMA).
//
//   out[r, n] = epilogue( sum_k A[r, k] * B[g(r) * n_out + n, k] + bias[g(r), n] )
//
// A is the regrouped token buffer (one contiguous block of rows per expert,
// the dispatch's output), B the stacked expert weights in nn.Linear layout
// ([out, in], reduction dimension contiguous), g(r) the expert owning row r.
// The epilogue is GELU (first Linear) or identity (second Linear), then RNE to
// bf16. (Expert FFN = Linear -> GELU -> Linear: yunthe.com MoELayer listing;
// the page's remark that production code groups tokens per expert and runs
// grouped GEMMs is the prior art this replaces.)
//
// Work unit: a 128 x 256 output tile of one expert. The ragged per-expert row
// counts live only on the device: a tile list (row0, rows, expert) is built on
// the device from the expert offsets, and every block of a persistent grid
// walks the same list, so no host synchronisation is needed.
//
// Block = 6 warps, one block per SM:
//   warp 0     TMA producer (one lane): A tile 128x64 and B tile 256x64 per
//              stage, 128-byte swizzle, 4-stage ring in shared memory
//   warp 1     TMEM allocator + MMA issuer (one lane): tcgen05.mma
//              kind::f16, M=128 N=256 K=16, fp32 accumulators in TMEM, two
//              accumulator buffers (2 x 256 columns) so the epilogue of one
//              tile overlaps the main loop of the next
//   warps 2-5  epilogue: tcgen05.ld 32 lanes x 32 columns at a time, bias,
//              GELU, bf16; full 32-row blocks leave through a shared-memory
//              buffer and a TMA store, an expert's last partial block row by
//              row; rows past the expert's block and columns past n_out are
//              computed but not stored. A second mode
//              writes the raw fp32 accumulators of each K split (used for the
//              gate logits).
//
// Every wait is bounded (globaltimer). On a timeout the block sets
// MOE_DEVERR_TIMEOUT, stops issuing work, drains its own copies and MMAs in
// flight, frees its TMEM and returns.
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace moe {
namespace gg {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;  // 64 bf16 = 128 bytes = one swizzle row
constexpr int STAGES = 4;
constexpr int UMMA_K = 16;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;  // one k-block of both operands
// grouped_gemm_kernel's pipeline: G_STAGES stages of KPS k-blocks each (the
// MMA issuer waits once and commits once per stage)
#ifndef MOE_GEMM_KPS
#define MOE_GEMM_KPS 1
#endif
constexpr int KPS = MOE_GEMM_KPS;
constexpr int G_STAGES = STAGES / KPS;
constexpr int G_STAGE_BYTES = KPS * STAGE_BYTES;
static_assert(G_STAGES * KPS == STAGES, "k-blocks per stage must divide the ring");
constexpr int NUM_THREADS = 192;      // SM-pair kernel: producer, MMA, 4 epilogue warps
// Row-gather warps (gathered-A mode), taking the stage fills in turn. Measured
// on the Mixtral-shaped prefill and DeepSeek-V3-shaped layers: one warp
// (each fill arrived a fill late) made the first expert GEMM 1.2x / 1.5x
// slower than TMA boxes of a pre-permuted copy, two 1.1x / 1.0x, four (each
// arriving as soon as its own copies land) 1.03x / 1.0x, so the gather's
// saving (the dispatch no longer writes the copy) is kept.
#ifndef MOE_GATHER_WARPS
#define MOE_GATHER_WARPS 4
#endif
constexpr int GATHER_WARPS = MOE_GATHER_WARPS;
constexpr int NUM_THREADS_G = 192 + 32 * GATHER_WARPS;  // grouped_gemm_kernel: the same plus the row-gather warps
constexpr int GATHER_WARP = 6;
constexpr int ACC_COLS = BN;          // fp32 accumulator columns per buffer
constexpr int TMEM_COLS = 2 * ACC_COLS;
constexpr int BAR_BYTES = 256;
// Epilogue staging: each of the 4 epilogue warps owns two 32 x 32 bf16
// buffers (2 KB each) from which a TMA store writes full 32-row blocks.
constexpr int EPI_BUF_BYTES = 32 * 32 * 2;
constexpr int EPI_BYTES = 4 * 2 * EPI_BUF_BYTES;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + EPI_BYTES + BAR_BYTES + 1024;  // + alignment slack
#ifndef MOE_L2_PREFETCH_KBLOCKS
#define MOE_L2_PREFETCH_KBLOCKS 0
#endif
// Optional L2 prefetch of the weight (B) tile of k-block kb + PF_DIST while
// loading k-block kb (compile-time switch; 0 = off, the default). Measured on
// the Mixtral-shaped prefill layer, prefetching 4-16 k-blocks ahead was 6%
// slower than none: the raster groups already keep each weight tile's readers
// in step, so the first reader's fetch serves the others from L2.
constexpr int PF_DIST = MOE_L2_PREFETCH_KBLOCKS;
constexpr uint64_t WAIT_LIMIT_NS = 4000000000ull;   // 4 s
constexpr uint64_t DRAIN_LIMIT_NS = 200000000ull;   // 0.2 s

// Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A bf16 (bits 7-9 = 1),
// B bf16 (bits 10-12 = 1), both K-major (bits 15, 16 = 0), N >> 3 at bits 17-22,
// M >> 4 at bits 24-28.
constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                           ((uint32_t)(BM >> 4) << 24);

struct Params {
    const int4 *mtiles;       // [max_mtiles] {row0, rows, group, 0}; nullptr = dense mode
    const int *num_mtiles;    // device count of valid mtiles
    int max_mtiles;           // capacity of the list (bounds check)
    int dense_rows;           // dense mode: rows of A (one group)
    int n_out;                // output columns (multiple of 64)
    int k_dim;                // reduction length (multiple of 64)
    int num_groups;           // experts in B / bias
    int out_rows;             // rows of `out` (bounds check)
    const float *bias;        // [num_groups, n_out]
    uint16_t *out;            // [out_rows, n_out] bf16 (bf16 mode)
    int gelu;                 // 1: GELU epilogue
    float *out_f32;           // non-null: raw fp32 accumulators instead (no bias, no GELU),
                              // split s written to out_f32 + s * out_rows * n_out
    int k_splits;             // fp32 mode: the K range is cut into this many splits
    int raster;               // m-tiles per raster group (dense mode; the list mode stores groups)
    const int *k_ranges;      // fp32 mode: non-null = split s covers the reduction columns
                              // [k_ranges[s], k_ranges[s + 1]) (multiples of 64, device memory);
                              // an empty range writes zeros (per-expert weight gradients)
    const int32_t *a_rows;    // non-null: row r of A is row a_rows[r] of a_ptr (a gather by the
                              // copy warp; tmA is not read), [out_rows] device ints
    const uint16_t *a_ptr;    // the gathered tensor, [a_rows_limit, k_dim] bf16 row-major
    int a_rows_limit;         // rows of the gathered tensor (bounds check of a_rows)
    int q_rows;               // quantised channel-major kernel: the most rows any tile of the launch
                              // has (<= 32: half-size token stages, twice as many)
};

// ---------------------------------------------------------------- PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.b32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// The same with an L2 eviction-priority policy (createpolicy) for the loaded lines.
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap *map, uint32_t bar, int x, int y,
                                                 uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

#ifndef MOE_TMA_L2_HINTS
#define MOE_TMA_L2_HINTS 0
#endif
// L2 policies for the operand loads: activations (A, re-read by every n-tile)
// and weights (B, read by the m-tiles of one raster group at about the same
// time, then dead). 0 = none; 1 = A evict_last, B evict_first; 2 = A
// evict_last; 3 = B evict_first.
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_policy_normal() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 16 bytes global -> shared, asynchronous, through L2 only.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}


// Ask the TMA unit to pull a tile into L2 (no shared-memory destination).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap *map, int x, int y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y)
                 : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, 8-row
// groups 1024 bytes apart (SBO), version 1 (bits 46-47), layout 2 = SWIZZLE_128B.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;              // LBO (unused for swizzled K-major)
    d |= (uint64_t)(1024 >> 4) << 32;    // SBO
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Shared-memory descriptor of an MN-major operand with the 128-byte swizzle:
// 64 consecutive N elements (128 bytes) per row, 8 reduction rows per
// 1024-byte swizzle atom; the next 8 rows (SBO) 1024 bytes on, the next 64
// columns (LBO) one 64-row box (8 KB) on.
__device__ __forceinline__ uint64_t sdesc_mn(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((BK * 128) >> 4) << 16;  // LBO: the next 64-column box
    d |= (uint64_t)(1024 >> 4) << 32;        // SBO: the next 8 reduction rows
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

__device__ __forceinline__ void mma_bf16_id(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(IDESC), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- helpers

struct Shared {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    uint32_t tmem_base;
    volatile int abort_flag;
};
static_assert(sizeof(Shared) <= BAR_BYTES, "barrier block too large");

// Bounded wait: true when the phase with `parity` has completed; false on
// abort (another role gave up) or after `limit_ns` (then sets the abort flag
// and the device error bit).
__device__ __noinline__ bool wait_bounded(Shared *sh, uint32_t bar, uint32_t parity,
                                          uint64_t limit_ns, bool raise) {
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 255u) {
            if (raise && sh->abort_flag) return false;
            uint64_t now = globaltimer_ns();
            if (t0 == 0) {
                t0 = now;
            } else if (now - t0 > limit_ns) {
                if (raise) {
                    sh->abort_flag = 1;
                    flag_error(MOE_DEVERR_TIMEOUT);
                }
                return false;
            }
        }
    }
}

struct Tile {
    int row0, rows, group, n0;
    bool ok;
};

template <int TM>
__device__ __forceinline__ int num_m_tiles(const Params &p) {
    if (p.mtiles == nullptr) return (p.dense_rows + TM - 1) / TM;
    int n = *p.num_mtiles;
    return n < 0 ? 0 : (n > p.max_mtiles ? p.max_mtiles : n);
}

// Work item w -> (m-tile, n-tile). The m-tiles are cut into raster groups of
// at most `raster` consecutive m-tiles of ONE expert; group j with first
// m-tile m_j and g_j tiles owns the items [m_j * num_n, (m_j + g_j) * num_n),
// m running fastest inside the group. So the blocks in flight at any time
// work on a few experts' n-tiles at once and share their B (weight) tiles.
// Each m-tile entry carries its group as (m_j << 16) | g_j in .w; the dense
// mode (one group of rows) computes the same grouping arithmetically.
template <int TM>
__device__ __forceinline__ Tile tile_of(const Params &p, int w, int num_m, int num_n) {
    const int q = w / num_n;  // an m-tile of the group that owns item w
    int mj, gj;
    if (p.mtiles == nullptr) {
        mj = (q / p.raster) * p.raster;
        gj = min(p.raster, num_m - mj);
    } else {
        const int packed = p.mtiles[q].w;
        mj = packed >> 16;
        gj = packed & 0xFFFF;
    }
    Tile t;
    t.ok = false;
    if (gj <= 0 || mj < 0 || mj + gj > num_m) {
        t.row0 = t.rows = t.group = t.n0 = 0;
        return t;
    }
    const int local = w - mj * num_n;
    const int m = mj + local % gj;
    const int n = local / gj;

    if (p.mtiles == nullptr) {
        t.row0 = m * TM;
        t.rows = min(TM, p.dense_rows - t.row0);
        t.group = 0;
    } else {
        int4 v = p.mtiles[m];
        t.row0 = v.x;
        t.rows = v.y;
        t.group = v.z;
    }
    t.n0 = n * BN;
    t.ok = t.rows > 0 && t.rows <= TM && t.row0 >= 0 && t.row0 + t.rows <= p.out_rows &&
           t.group >= 0 && t.group < p.num_groups && n < num_n;
    return t;
}

__device__ __forceinline__ float gelu_erf(float v) {
    return 0.5f * v * (1.0f + erff(v * 0.70710678118654752440f));
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, uint32_t src, int x, int y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(src)
                 : "memory");
}

// Store one warp's 32 rows x 32 columns of bf16 results (lane = row; 16
// packed words per lane). A block whose 32 rows are all valid goes through
// the warp's shared-memory buffer and one TMA store (full 64-byte row
// segments); a partial block (an expert's last rows) is written row by row.
__device__ __forceinline__ void store_chunk_bf16(const CUtensorMap *tmC, uint8_t *ebuf, int &buf, int lane,
                                                 const uint32_t (&packed)[16], int rows_valid, int row_block,
                                                 int col, uint16_t *out_row) {
    if (rows_valid == 32) {
        if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
        __syncwarp();
        uint8_t *b = ebuf + buf * EPI_BUF_BYTES;
        uint4 *dst = reinterpret_cast<uint4 *>(b + lane * 64);
#pragma unroll
        for (int j = 0; j < 4; ++j)
            dst[j] = make_uint4(packed[4 * j], packed[4 * j + 1], packed[4 * j + 2], packed[4 * j + 3]);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(tmC, smem_u32(b), col, row_block);
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        }
        buf ^= 1;
    } else if (lane < rows_valid) {
        uint4 *dst = reinterpret_cast<uint4 *>(out_row + col);
#pragma unroll
        for (int j = 0; j < 4; ++j)
            dst[j] = make_uint4(packed[4 * j], packed[4 * j + 1], packed[4 * j + 2], packed[4 * j + 3]);
    }
}

// All TMA stores this warp issued have finished writing global memory.
__device__ __forceinline__ void store_drain(int lane) {
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    __syncwarp();
}

// ---------------------------------------------------------------- kernel

// A tile of at most 96 valid rows (an expert's last rows, or every tile of a
// decode batch) is loaded in 32-row chunks through tmA32, only the chunks that
// hold rows; the MMA still reads 128 rows, the rest are stale and their
// results are never stored.
constexpr int A_CHUNK_ROWS = 32;
constexpr int A_CHUNK_BYTES = A_CHUNK_ROWS * BK * 2;  // 4 KB: a multiple of the 1024-byte swizzle atom

__device__ __forceinline__ uint32_t a_tile_bytes(int rows) {
    return rows > 3 * A_CHUNK_ROWS ? (uint32_t)A_BYTES
                                   : (uint32_t)((rows + A_CHUNK_ROWS - 1) / A_CHUNK_ROWS) * A_CHUNK_BYTES;
}
__device__ __forceinline__ void load_a_tile(uint32_t dst, const CUtensorMap *tmA, const CUtensorMap *tmA32,
                                            uint32_t bar, int x, int row0, int rows, uint64_t policy = 0) {
    if (rows > 3 * A_CHUNK_ROWS) {
        if (policy) tma_load_2d_hint(dst, tmA, bar, x, row0, policy);
        else tma_load_2d(dst, tmA, bar, x, row0);
    } else {
        for (int c = 0; c * A_CHUNK_ROWS < rows; ++c) {
            if (policy) tma_load_2d_hint(dst + c * A_CHUNK_BYTES, tmA32, bar, x, row0 + c * A_CHUNK_ROWS, policy);
            else tma_load_2d(dst + c * A_CHUNK_BYTES, tmA32, bar, x, row0 + c * A_CHUNK_ROWS);
        }
    }
}

// BMN: B is given N-major, [num_groups * k_dim, n_out] (each group's matrix as
// stored, reduction rows by output columns), loaded as four 64-column boxes
// per stage and read by the MMA as an MN-major operand, so no transposed copy
// is needed (a separate instance: the K-major code is left as it was).
template <bool BMN>
__global__ void __launch_bounds__(NUM_THREADS_G, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmC, const Params p,
                    const __grid_constant__ CUtensorMap tmA32) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte alignment for the swizzled tiles
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    Shared *sh = reinterpret_cast<Shared *>(smem + G_STAGES * G_STAGE_BYTES + EPI_BYTES);

    const int warp = warp_id();
    const int lane = lane_id();

    if (threadIdx.x == 0) {
        for (int s = 0; s < G_STAGES; ++s) {
            // the B tile's arrive.expect_tx, plus one arrival per lane of the row-gather warp
            mbar_init(smem_u32(&sh->full[s]), p.a_rows != nullptr ? 33u : 1u);
            mbar_init(smem_u32(&sh->empty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&sh->tfull[a]), 1);
            mbar_init(smem_u32(&sh->tempty[a]), 4);
        }
        mbar_init(smem_u32(&sh->drain), 1);
        sh->abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&sh->tmem_base)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = sh->tmem_base;

    const int num_m = num_m_tiles<BM>(p);
    const int num_n = (p.n_out + BN - 1) / BN;
    const int splits = p.k_splits > 0 ? p.k_splits : 1;
    const int total = num_m * num_n * splits;
    const int kblocks = p.k_dim / BK;
    const int kb_per_split = (kblocks + splits - 1) / splits;
    // Balanced persistent schedule: the fewest blocks that finish the items
    // in as many rounds as the whole grid would take; block b takes items b,
    // b + stride, ... and blocks from stride on take none. A last round that
    // would leave most of the grid idle is spread over the rounds instead,
    // so a weight-streaming GEMM keeps every working block pulling from HBM
    // until the end.
    const int rounds = (total + (int)gridDim.x - 1) / (int)gridDim.x;
    const int stride = rounds > 0 ? (total + rounds - 1) / rounds : (int)gridDim.x;
    const int first = (int)blockIdx.x < stride ? (int)blockIdx.x : total;

    if (warp >= GATHER_WARP) {
        // ---------------------------------------------------- row-gather warps (a_rows mode)
        // Row i of the A tile is row a_rows[row0 + i] of a_ptr (for the first
        // expert GEMM: the token of each regrouped row, so the dispatch never
        // writes a regrouped copy of x). The GATHER_WARPS warps take the
        // stage fills in turn. For its fill a warp copies the tile's rows'
        // 128-byte segments of the k-block with 16-byte cp.async, lane l
        // taking chunk l % 8 of rows 4 j + l / 8, straight to the positions the
        // 128-byte swizzle gives them (chunk c of row i at i * 128 + (c ^ (i %
        // 8)) * 16), so the MMA reads them as it reads a TMA box. Rows past
        // the tile's rows are not copied (their accumulator rows are never
        // stored). The stage's full barrier counts the B tile's bytes and one
        // arrival per lane of the filling warp: a lane arrives once its copies
        // have landed (cp.async.wait_group) and it has fenced them for the
        // async proxy -- at once when the warps are many enough to keep every
        // stage's copies in flight, else one of its fills later.
        if (p.a_rows != nullptr) {
            const int c = lane & 7, rsub = lane >> 3;
            const int gw = warp - GATHER_WARP;  // this warp fills every GATHER_WARPS-th stage fill
            int fill = 0;
            // the source rows of a tile (rows 4 j + rsub, j < nj, this lane's):
            // all loads are issued first; check_rows, run when the rows are
            // used, validates them (a check right after each load would make
            // the 32 loads wait on one another)
            auto load_rows = [&](const Tile &t, int (&src)[32], int &nj) {
                nj = max(0, (t.rows - rsub + 3) / 4);
#pragma unroll
                for (int j = 0; j < 32; ++j) src[j] = j < nj ? __ldg(p.a_rows + t.row0 + 4 * j + rsub) : 0;
            };
            auto check_rows = [&](int (&src)[32], int nj) {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (j < nj && (src[j] < 0 || src[j] >= p.a_rows_limit)) {
                        flag_error(MOE_DEVERR_ROW_INDEX);
                        src[j] = 0;
                    }
            };
            auto next_tile = [&](int w, Tile &t) {
                for (; w < total; w += stride) {
                    t = tile_of<BM>(p, w / splits, num_m, num_n);
                    if (t.ok) return w;
                }
                return total;
            };
            uint32_t stage = 0, phase = 0;
            int prev = -1;  // stage of the previous fill, not yet arrived
            bool stop = false;
            Tile t, tn;
            int src[32], nsrc[32], nj = 0, nnj = 0;
            int w = next_tile(first, t);
            if (w < total) {
                load_rows(t, src, nj);
                check_rows(src, nj);
            }
            while (w < total && !stop) {
                // the next tile's rows load while this tile's copies are issued
                const int wn = next_tile(w + stride, tn);
                if (wn < total) load_rows(tn, nsrc, nnj);
                const int kb0 = p.k_ranges ? p.k_ranges[w % splits] / BK : (w % splits) * kb_per_split;
                const int kb1 = p.k_ranges ? p.k_ranges[w % splits + 1] / BK : min(kblocks, kb0 + kb_per_split);
                const uint32_t sw0 = (uint32_t)((c ^ rsub) << 4), sw1 = (uint32_t)((c ^ (rsub + 4)) << 4);
                for (int kb = kb0; kb < kb1; kb += KPS) {
                    if ((fill++ % GATHER_WARPS) != gw) {  // another gather warp's fill
                        if (++stage == G_STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                        continue;
                    }
                    bool ok = true;
                    if (lane == 0) ok = wait_bounded(sh, smem_u32(&sh->empty[stage]), phase ^ 1u, WAIT_LIMIT_NS, true);
                    if (__shfl_sync(0xffffffffu, ok ? 1 : 0, 0) == 0) {
                        stop = true;
                        break;
                    }
                    const int nk = min(KPS, kb1 - kb);
                    for (int part = 0; part < nk; ++part) {
                        const uint32_t a_s =
                            smem_u32(smem + stage * G_STAGE_BYTES + part * STAGE_BYTES) + (uint32_t)rsub * 128u;
                        const uint16_t *col = p.a_ptr + (size_t)(kb + part) * BK + c * 8;
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (j < nj) {
                                const uint32_t dst = a_s + (uint32_t)j * 512u + ((j & 1) ? sw1 : sw0);
                                const uint16_t *from = col + (size_t)src[j] * (size_t)p.k_dim;
                                cp_async16(dst, from);
                            }
                    }
                    asm volatile("cp.async.commit_group;" ::: "memory");
                    if (2 * GATHER_WARPS > G_STAGES) {
                        // arriving a fill late would hold the MMA back (with W gather warps and S
                        // stages, fill f + W needs the stage the MMA frees after fill f + W - S)
                        asm volatile("cp.async.wait_group 0;" ::: "memory");
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                        mbar_arrive(smem_u32(&sh->full[stage]));
                    } else {
                        if (prev >= 0) {
                            asm volatile("cp.async.wait_group 1;" ::: "memory");
                            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                            mbar_arrive(smem_u32(&sh->full[prev]));
                        }
                        prev = (int)stage;
                    }
                    if (++stage == G_STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                w = wn;
                nj = nnj;
#pragma unroll
                for (int j = 0; j < 32; ++j) src[j] = nsrc[j];
                check_rows(src, nj);
            }
            asm volatile("cp.async.wait_group 0;" ::: "memory");
            if (prev >= 0 && !stop) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                mbar_arrive(smem_u32(&sh->full[prev]));
            }
        }
    } else if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            const uint64_t pol_a = (MOE_TMA_L2_HINTS == 1 || MOE_TMA_L2_HINTS == 2) ? l2_policy_evict_last() : 0;
            const uint64_t pol_b = (MOE_TMA_L2_HINTS == 1 || MOE_TMA_L2_HINTS == 3) ? l2_policy_evict_first() : 0;
            uint32_t stage = 0, phase = 0;
            int issued_phase[G_STAGES];
            for (int s = 0; s < G_STAGES; ++s) issued_phase[s] = -1;
            bool stop = false;
            for (int w = first; w < total && !stop; w += stride) {
                Tile t = tile_of<BM>(p, w / splits, num_m, num_n);
                if (!t.ok) continue;
                const int brow = t.group * p.n_out + t.n0;
                const int kb0 = p.k_ranges ? p.k_ranges[w % splits] / BK : (w % splits) * kb_per_split;
                const int kb1 = p.k_ranges ? p.k_ranges[w % splits + 1] / BK : min(kblocks, kb0 + kb_per_split);
                if (PF_DIST > 0 && !BMN)
                    for (int kb = kb0; kb < kb1 && kb < kb0 + PF_DIST; ++kb) tma_prefetch_2d(&tmB, kb * BK, brow);
                for (int kb = kb0; kb < kb1; kb += KPS) {
                    if (PF_DIST > 0 && !BMN && kb + PF_DIST < kb1)
                        tma_prefetch_2d(&tmB, (kb + PF_DIST) * BK, brow);
                    if (!wait_bounded(sh, smem_u32(&sh->empty[stage]), phase ^ 1u, WAIT_LIMIT_NS, true)) {
                        stop = true;
                        break;
                    }
                    const uint32_t fb = smem_u32(&sh->full[stage]);
                    const int nk = min(KPS, kb1 - kb);
                    // with a_rows the row-gather warp fills the A tile (and arrives on fb itself)
                    mbar_arrive_expect_tx(fb, (uint32_t)nk * ((p.a_rows ? 0u : a_tile_bytes(t.rows)) + B_BYTES));
                    for (int part = 0; part < nk; ++part) {
                        uint8_t *a_s = smem + stage * G_STAGE_BYTES + part * STAGE_BYTES;
                        const int x = (kb + part) * BK;
                        if (!p.a_rows) load_a_tile(smem_u32(a_s), &tmA, &tmA32, fb, x, t.row0, t.rows, pol_a);
                        if constexpr (BMN) {  // reduction rows x..x+63 of the group, four 64-column boxes
#pragma unroll
                            for (int j = 0; j < BN / 64; ++j)
                                tma_load_2d(smem_u32(a_s + A_BYTES + j * (BK * 128)), &tmB, fb, t.n0 + 64 * j,
                                            t.group * p.k_dim + x);
                        } else if (pol_b) {
                            tma_load_2d_hint(smem_u32(a_s + A_BYTES), &tmB, fb, x, brow, pol_b);
                        } else {
                            tma_load_2d(smem_u32(a_s + A_BYTES), &tmB, fb, x, brow);
                        }
                    }
                    issued_phase[stage] = (int)phase;
                    if (++stage == G_STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (stop) {
                // let this block's copies in flight land before the block exits
                for (int s = 0; s < G_STAGES; ++s)
                    if (issued_phase[s] >= 0)
                        wait_bounded(sh, smem_u32(&sh->full[s]), (uint32_t)issued_phase[s],
                                     DRAIN_LIMIT_NS, false);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            uint32_t stage = 0, phase = 0;
            uint32_t acc = 0, acc_phase = 0;
            bool stop = false;
            for (int w = first; w < total && !stop; w += stride) {
                Tile t = tile_of<BM>(p, w / splits, num_m, num_n);
                if (!t.ok) continue;
                if (!wait_bounded(sh, smem_u32(&sh->tempty[acc]), acc_phase ^ 1u, WAIT_LIMIT_NS, true))
                    break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * ACC_COLS;
                const int kb0 = p.k_ranges ? p.k_ranges[w % splits] / BK : (w % splits) * kb_per_split;
                const int kb1 = p.k_ranges ? p.k_ranges[w % splits + 1] / BK : min(kblocks, kb0 + kb_per_split);
                for (int kb = kb0; kb < kb1; kb += KPS) {
                    if (!wait_bounded(sh, smem_u32(&sh->full[stage]), phase, WAIT_LIMIT_NS, true)) {
                        stop = true;
                        break;
                    }
                    tc_fence_after();
                    const int nk = min(KPS, kb1 - kb);
                    for (int part = 0; part < nk; ++part) {
                        const uint32_t a_addr = smem_u32(smem + stage * G_STAGE_BYTES + part * STAGE_BYTES);
                        const uint32_t b_addr = a_addr + A_BYTES;
                        if constexpr (BMN) {  // B MN-major: 16 reduction rows = two 1024-byte atoms per MMA
#pragma unroll
                            for (int kk = 0; kk < BK / UMMA_K; ++kk)
                                mma_bf16_id(d_tmem, sdesc(a_addr + kk * UMMA_K * 2), sdesc_mn(b_addr + kk * 2048),
                                            IDESC | (1u << 16), (kb != kb0 || part != 0 || kk != 0) ? 1u : 0u);
                        } else {
#pragma unroll
                            for (int kk = 0; kk < BK / UMMA_K; ++kk) {
                                mma_bf16(d_tmem, sdesc(a_addr + kk * UMMA_K * 2), sdesc(b_addr + kk * UMMA_K * 2),
                                         (kb != kb0 || part != 0 || kk != 0) ? 1u : 0u);
                            }
                        }
                    }
                    mma_commit(smem_u32(&sh->empty[stage]));
                    if (++stage == G_STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (stop) break;
                mma_commit(smem_u32(&sh->tfull[acc]));
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            // every MMA issued by this block has completed once `drain` fires
            mma_commit(smem_u32(&sh->drain));
            wait_bounded(sh, smem_u32(&sh->drain), 0, DRAIN_LIMIT_NS, false);
        }
    } else {
        // ---------------------------------------------------- epilogue (warps 2-5)
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const int row = q * 32 + lane;
        uint8_t *ebuf = smem + G_STAGES * G_STAGE_BYTES + (warp - 2) * 2 * EPI_BUF_BYTES;
        int ebuf_idx = 0;
        uint32_t acc = 0, acc_phase = 0;
        for (int w = first; w < total; w += stride) {
            Tile t = tile_of<BM>(p, w / splits, num_m, num_n);
            if (!t.ok) {
                if (threadIdx.x == 64) flag_error(MOE_DEVERR_TILE_LIST);
                continue;
            }
            if (!wait_bounded(sh, smem_u32(&sh->tfull[acc]), acc_phase, WAIT_LIMIT_NS, true)) break;
            tc_fence_after();
            const int rows_valid = max(0, min(32, t.rows - q * 32));
            uint16_t *out_row = p.out + (size_t)(t.row0 + row) * p.n_out;
            const float *bias = p.bias + (size_t)t.group * p.n_out;
            const uint32_t tbase = tmem_base + acc * ACC_COLS + ((uint32_t)(q * 32) << 16);
            for (int c0 = 0; c0 < BN; c0 += 32) {
                const int col = t.n0 + c0;
                if (col >= p.n_out) break;  // warp-uniform
                uint32_t r[32];
                tmem_ld32(tbase + c0, r);
                if (p.out_f32 != nullptr) {
                    // fp32 mode (raw accumulators of split w % splits). A full 32-row
                    // block goes row-major into the warp's 4 KB buffer with the
                    // 128-byte swizzle (conflict-free) and out with one TMA store
                    // (tmC is then the fp32 map of all split planes); an expert's
                    // last partial block is turned in the buffer (element (i, j) at
                    // word 32 i + (j ^ i)) and stored row by row, 128 contiguous
                    // bytes per instruction. Columns past n_out are not stored.
                    const bool empty = p.k_ranges && p.k_ranges[w % splits] == p.k_ranges[w % splits + 1];
                    if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
                    __syncwarp();  // the previous store has finished reading the buffer
                    if (rows_valid == 32) {
                        uint8_t *rowp = ebuf + lane * 128;
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            *reinterpret_cast<uint4 *>(rowp + ((c ^ (lane & 7)) << 4)) =
                                empty ? make_uint4(0u, 0u, 0u, 0u)  // nothing accumulated
                                      : make_uint4(r[4 * c], r[4 * c + 1], r[4 * c + 2], r[4 * c + 3]);
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_2d(&tmC, smem_u32(ebuf), col, (w % splits) * p.out_rows + t.row0 + q * 32);
                            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
                        }
                    } else {
                        uint32_t *tb = reinterpret_cast<uint32_t *>(ebuf);
#pragma unroll
                        for (int j = 0; j < 32; ++j) tb[lane * 32 + (j ^ lane)] = empty ? 0u : r[j];
                        __syncwarp();
                        float *base =
                            p.out_f32 + ((size_t)(w % splits) * p.out_rows + (t.row0 + q * 32)) * p.n_out + col;
                        const bool colok = lane < p.n_out - col;
                        for (int i = 0; i < rows_valid; ++i)
                            if (colok) base[(size_t)i * p.n_out + lane] = __uint_as_float(tb[i * 32 + (lane ^ i)]);
                        __syncwarp();
                    }
                    continue;
                }
                uint32_t packed[16];
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    const float4 b = __ldg(reinterpret_cast<const float4 *>(bias + col + j));
                    float v0 = __uint_as_float(r[j + 0]) + b.x;
                    float v1 = __uint_as_float(r[j + 1]) + b.y;
                    float v2 = __uint_as_float(r[j + 2]) + b.z;
                    float v3 = __uint_as_float(r[j + 3]) + b.w;
                    if (p.gelu) {
                        v0 = gelu_erf(v0);
                        v1 = gelu_erf(v1);
                        v2 = gelu_erf(v2);
                        v3 = gelu_erf(v3);
                    }
                    packed[j / 2] = pack_bf16x2(v0, v1);
                    packed[j / 2 + 1] = pack_bf16x2(v2, v3);
                }
                store_chunk_bf16(&tmC, ebuf, ebuf_idx, lane, packed, rows_valid, t.row0 + q * 32, col, out_row);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sh->tempty[acc]));
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        store_drain(lane);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(TMEM_COLS)
                     : "memory");
    }
}

// ============================================================================
// SM-pair variant: a cluster of 2 CTAs on two SMs runs tcgen05.mma.cta_group::2
// with M = 256 (128 rows per SM), N = 256, K = 16. Each CTA stages its own 128
// rows of A and its half (128 of the 256 output columns) of B per k-block, so
// a stage is 32 KB and the ring is 6 deep; each SM's TMEM holds its 128 rows
// of the 256 x 256 accumulator (two buffers of 256 columns).
//   rank 0 ("leader"): TMA for its halves, arms the stage barrier for the
//                      pair's 64 KB, issues the MMAs, commits to both CTAs
//   rank 1:            TMA for its halves, completing on the leader's barrier
//   both:              epilogue of their own 128 rows; arrive on the
//                      leader's accumulator-empty barrier
// Work unit: a 256 x 256 tile of one expert (m-tiles of 256 rows).
constexpr int PAIR_BM = 256;
#ifndef MOE_PAIR_STAGES
#define MOE_PAIR_STAGES 6
#endif
constexpr int P_STAGES = MOE_PAIR_STAGES;
constexpr int P_A_BYTES = 128 * BK * 2;
constexpr int P_B_BYTES = (BN / 2) * BK * 2;
constexpr int P_STAGE_BYTES = P_A_BYTES + P_B_BYTES;
constexpr int P_SMEM_BYTES = P_STAGES * P_STAGE_BYTES + EPI_BYTES + BAR_BYTES + 1024;
constexpr uint32_t IDESC_PAIR = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                                ((uint32_t)(PAIR_BM >> 4) << 24);

struct PairShared {
    uint64_t full[P_STAGES];
    uint64_t empty[P_STAGES];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    uint32_t tmem_base;
    volatile int abort_flag;
};
static_assert(sizeof(PairShared) <= BAR_BYTES, "barrier block too large");

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Address of the same shared-memory object in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.b32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// TMA load into this CTA's shared memory whose completion is counted on a
// barrier that may live in the peer CTA (cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *map, uint32_t bar_cluster,
                                                 int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster)
        : "memory");
}

__device__ __forceinline__ void mma_bf16_pair(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(IDESC_PAIR), "r"(acc)
        : "memory");
}

// Arrive (once the MMAs issued so far complete) on the barrier at this
// shared-memory offset in both CTAs of the pair.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar) {
    const uint16_t mask = 0x3;
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
        "h"(mask)
        : "memory");
}

__device__ __noinline__ bool wait_bounded_pair(PairShared *sh, uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                               bool raise, bool cluster_scope) {
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        // CTA-scope acquire for every barrier: cluster-scope waits measured
        // ~10% slower (the accumulator-empty barrier is still arrived with
        // release.cluster by the peer's epilogue)
        (void)cluster_scope;
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 255u) {
            if (raise && sh->abort_flag) return false;
            uint64_t now = globaltimer_ns();
            if (t0 == 0) {
                t0 = now;
            } else if (now - t0 > limit_ns) {
                if (raise) {
                    sh->abort_flag = 1;
                    flag_error(MOE_DEVERR_TIMEOUT);
                }
                return false;
            }
        }
    }
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                         const __grid_constant__ CUtensorMap tmC, const Params p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    PairShared *sh = reinterpret_cast<PairShared *>(smem + P_STAGES * P_STAGE_BYTES + EPI_BYTES);

    const int warp = warp_id();
    const int lane = lane_id();
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < P_STAGES; ++s) {
            mbar_init(smem_u32(&sh->full[s]), 1);
            mbar_init(smem_u32(&sh->empty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&sh->tfull[a]), 1);
            mbar_init(smem_u32(&sh->tempty[a]), 8);
        }
        mbar_init(smem_u32(&sh->drain), 1);
        sh->abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&sh->tmem_base)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    cluster_sync_all();  // both CTAs' barriers initialised, TMEM allocated
    tc_fence_after();
    const uint32_t tmem_base = sh->tmem_base;

    const int num_m = num_m_tiles<PAIR_BM>(p);
    const int num_n = (p.n_out + BN - 1) / BN;
    const int total = num_m * num_n;
    const int kblocks = p.k_dim / BK;
    // the single-SM kernel's balanced schedule, over clusters
    const int rounds = (total + (int)(gridDim.x >> 1) - 1) / (int)(gridDim.x >> 1);
    const int num_clusters = rounds > 0 ? (total + rounds - 1) / rounds : (int)(gridDim.x >> 1);
    const int cluster_id = (int)(blockIdx.x >> 1) < num_clusters ? (int)(blockIdx.x >> 1) : total;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer (both CTAs)
            uint32_t stage = 0, phase = 0;
            int issued_phase[P_STAGES];
            for (int s = 0; s < P_STAGES; ++s) issued_phase[s] = -1;
            bool stop = false;
            for (int w = cluster_id; w < total && !stop; w += num_clusters) {
                Tile t = tile_of<PAIR_BM>(p, w, num_m, num_n);
                if (!t.ok) continue;
                const int arow = t.row0 + (int)rank * 128;
                const int brow = t.group * p.n_out + t.n0 + (int)rank * (BN / 2);
                if (PF_DIST > 0)
                    for (int kb = 0; kb < kblocks && kb < PF_DIST; ++kb) tma_prefetch_2d(&tmB, kb * BK, brow);
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (PF_DIST > 0 && kb + PF_DIST < kblocks) tma_prefetch_2d(&tmB, (kb + PF_DIST) * BK, brow);
                    if (!wait_bounded_pair(sh, smem_u32(&sh->empty[stage]), phase ^ 1u, WAIT_LIMIT_NS, true,
                                           false)) {
                        stop = true;
                        break;
                    }
                    const uint32_t fb_local = smem_u32(&sh->full[stage]);
                    const uint32_t fb_leader = map_to_rank(fb_local, 0);
                    uint8_t *a_s = smem + stage * P_STAGE_BYTES;
                    if (leader) mbar_arrive_expect_tx(fb_local, 2 * P_STAGE_BYTES);
                    tma_load_2d_pair(smem_u32(a_s), &tmA, fb_leader, kb * BK, arow);
                    tma_load_2d_pair(smem_u32(a_s + P_A_BYTES), &tmB, fb_leader, kb * BK, brow);
                    issued_phase[stage] = (int)phase;
                    if (++stage == P_STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (stop && leader) {
                for (int s = 0; s < P_STAGES; ++s)
                    if (issued_phase[s] >= 0)
                        wait_bounded_pair(sh, smem_u32(&sh->full[s]), (uint32_t)issued_phase[s], DRAIN_LIMIT_NS,
                                          false, true);
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ------------------------------------------------ MMA issuer (leader only)
            uint32_t stage = 0, phase = 0;
            uint32_t acc = 0, acc_phase = 0;
            bool stop = false;
            for (int w = cluster_id; w < total && !stop; w += num_clusters) {
                Tile t = tile_of<PAIR_BM>(p, w, num_m, num_n);
                if (!t.ok) continue;
                if (!wait_bounded_pair(sh, smem_u32(&sh->tempty[acc]), acc_phase ^ 1u, WAIT_LIMIT_NS, true, true))
                    break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * ACC_COLS;
                for (int kb = 0; kb < kblocks; ++kb) {
                    // CTA-scope acquire: the peer's TMA bytes are counted on this barrier by the
                    // async proxy, which the MMA (also async proxy) then reads
                    if (!wait_bounded_pair(sh, smem_u32(&sh->full[stage]), phase, WAIT_LIMIT_NS, true, false)) {
                        stop = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(smem + stage * P_STAGE_BYTES);
                    const uint32_t b_addr = a_addr + P_A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < BK / UMMA_K; ++kk) {
                        mma_bf16_pair(d_tmem, sdesc(a_addr + kk * UMMA_K * 2), sdesc(b_addr + kk * UMMA_K * 2),
                                      (kb | kk) != 0 ? 1u : 0u);
                    }
                    mma_commit_pair(smem_u32(&sh->empty[stage]));
                    if (++stage == P_STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (stop) break;
                mma_commit_pair(smem_u32(&sh->tfull[acc]));
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            mma_commit_pair(smem_u32(&sh->drain));
            wait_bounded_pair(sh, smem_u32(&sh->drain), 0, DRAIN_LIMIT_NS, false, false);
        } else if (lane == 0) {
            // the leader's final commit also arrives here: wait for it so that no
            // arrival from this pair's MMAs is still in flight when the CTA exits
            wait_bounded_pair(sh, smem_u32(&sh->drain), 0, WAIT_LIMIT_NS, false, false);
        }
    } else {
        // ---------------------------------------------------- epilogue (warps 2-5, both CTAs)
        const int q = warp & 3;
        const int row = (int)rank * 128 + q * 32 + lane;  // row within the 256-row tile
        uint8_t *ebuf = smem + P_STAGES * P_STAGE_BYTES + (warp - 2) * 2 * EPI_BUF_BYTES;
        int ebuf_idx = 0;
        const uint32_t tempty_leader0 = map_to_rank(smem_u32(&sh->tempty[0]), 0);
        const uint32_t tempty_leader1 = map_to_rank(smem_u32(&sh->tempty[1]), 0);
        uint32_t acc = 0, acc_phase = 0;
        for (int w = cluster_id; w < total; w += num_clusters) {
            Tile t = tile_of<PAIR_BM>(p, w, num_m, num_n);
            if (!t.ok) {
                if (threadIdx.x == 64) flag_error(MOE_DEVERR_TILE_LIST);
                continue;
            }
            if (!wait_bounded_pair(sh, smem_u32(&sh->tfull[acc]), acc_phase, WAIT_LIMIT_NS, true, false)) break;
            tc_fence_after();
            const int rows_valid = max(0, min(32, t.rows - ((int)rank * 128 + q * 32)));
            uint16_t *out_row = p.out + (size_t)(t.row0 + row) * p.n_out;
            const float *bias = p.bias + (size_t)t.group * p.n_out;
            const uint32_t tbase = tmem_base + acc * ACC_COLS + ((uint32_t)(q * 32) << 16);
            for (int c0 = 0; c0 < BN; c0 += 32) {
                const int col = t.n0 + c0;
                if (col >= p.n_out) break;  // warp-uniform
                uint32_t r[32];
                tmem_ld32(tbase + c0, r);
                uint32_t packed[16];
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    const float4 b = __ldg(reinterpret_cast<const float4 *>(bias + col + j));
                    float v0 = __uint_as_float(r[j + 0]) + b.x;
                    float v1 = __uint_as_float(r[j + 1]) + b.y;
                    float v2 = __uint_as_float(r[j + 2]) + b.z;
                    float v3 = __uint_as_float(r[j + 3]) + b.w;
                    if (p.gelu) {
                        v0 = gelu_erf(v0);
                        v1 = gelu_erf(v1);
                        v2 = gelu_erf(v2);
                        v3 = gelu_erf(v3);
                    }
                    packed[j / 2] = pack_bf16x2(v0, v1);
                    packed[j / 2 + 1] = pack_bf16x2(v2, v3);
                }
                store_chunk_bf16(&tmC, ebuf, ebuf_idx, lane, packed, rows_valid,
                                 t.row0 + (int)rank * 128 + q * 32, col, out_row);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(acc == 0 ? tempty_leader0 : tempty_leader1);
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        store_drain(lane);
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // no remote arrive or multicast commit still targets either CTA
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                     : "memory");
    }
}

// The m-tile list of the routed experts, from the expert offsets:
// expert e owns rows [offsets[e], offsets[e+1]) and ceil(rows / tile_rows)
// tiles, grouped for rasterisation (see tile_of). Called by all threads of a
// block of blockDim.x >= N threads (at most 65535 tiles); `offsets` may be
// global or shared memory; sc is blockDim.x ints of shared scratch.
__device__ __forceinline__ void build_mtiles_block(const int32_t *offsets, int N, int total_rows, int tile_rows,
                                                   int raster, int max_tiles, int4 *__restrict__ mtiles,
                                                   int *__restrict__ num_mtiles, int *sc) {
    const int e = threadIdx.x;
    int cnt = 0, r0 = 0, r1 = 0;
    bool bad = false;
    if (e < N) {
        r0 = offsets[e];
        r1 = offsets[e + 1];
        if (r0 < 0 || r1 < r0 || r1 > total_rows) {
            bad = true;
        } else {
            cnt = (r1 - r0 + tile_rows - 1) / tile_rows;
        }
    }
    if (bad) flag_error(MOE_DEVERR_TILE_LIST);
    sc[e] = cnt;
    __syncthreads();
    // inclusive scan over the N experts (threads past N hold no tiles)
    int v = cnt;
    for (int o = 1; o < N; o <<= 1) {
        int add = (e >= o) ? sc[e - o] : 0;
        __syncthreads();
        sc[e] = v = v + add;
        __syncthreads();
    }
    const int start = v - cnt;
    // raster groups stay inside expert e: all of its tiles in one group when
    // there are at most 2 * raster of them (so an expert whose rows spill a
    // few rows into one more tile does not stream its weights a second time),
    // else ceil(cnt / raster) groups of balanced size
    const int ng = cnt <= 2 * raster ? 1 : (cnt + raster - 1) / raster;
    for (int i = 0; i < cnt; ++i) {
        int m = start + i;
        if (m < max_tiles) {
            int rr = r0 + i * tile_rows;
            int rows = r1 - rr < tile_rows ? r1 - rr : tile_rows;
            const int g = ((i + 1) * ng - 1) / cnt;           // group of tile i
            const int lo = (g * cnt) / ng, hi = ((g + 1) * cnt) / ng;
            mtiles[m] = make_int4(rr, rows, e, ((start + lo) << 16) | (hi - lo));
        }
    }
    if (e == N - 1) *num_mtiles = v < max_tiles ? v : max_tiles;
}

__global__ void __launch_bounds__(1024)
build_mtiles_kernel(const int32_t *__restrict__ offsets, int N, int total_rows, int tile_rows, int raster,
                    int max_tiles, int4 *__restrict__ mtiles, int *__restrict__ num_mtiles) {
    __shared__ int sc[1024];
    build_mtiles_block(offsets, N, total_rows, tile_rows, raster, max_tiles, mtiles, num_mtiles, sc);
}

}  // namespace gg
}  // namespace moe
