// gemm_quant.cuh -- the grouped expert GEMM with weight-only quantised expert
// weights (the 8- and 4-bit expert weights of the lmnt.cn/news/351908 sec.
// 4.3 remark; the CSDN page's sec. 3.2 one-byte FP8 weights; the yunthe.com
// page's 4-bit Mixtral), computed transposed so that the weights, not the
// tokens, fill the 128 rows of the MMA. Two formats:
//
//   FP8  E4M3 codes, one fp32 scale per output channel:
//        out[r, n] = epilogue( scale[g(r), n] * sum_k code(B[g(r) n_out + n, k]) A[r, k] + bias )
//   INT4 4-bit codes along k, eight columns 8m .. 8m + 7 to a little-endian
//        32-bit word (column 8m + 2j in bits 4j .. 4j + 3, column 8m + 2j + 1
//        in bits 16 + 4j .. 19 + 4j; code c stands for c - 8), one bf16 scale
//        per output channel and group of 128 reduction columns:
//        out[r, n] = epilogue( sum_k bf16((c - 8) * scale[g(r), k / 128, n]) A[r, k] + bias )
//
// A decode batch gives each expert a handful of rows, so a token-major tile
// (128 token rows) would spend almost all of its MMA work on padding. Here one
// tile is 128 output channels of one expert x up to 64 of its rows: the MMA
// is D[channel, row] = sum_k W[channel, k] * A[row, k] with M = 128 channels
// and N = the tile's row count rounded up to 16, so the tensor-core work
// scales with the real rows and the kernel is left to stream the codes.
//
// The codes cross HBM at one byte (FP8) or half a byte (INT4) per weight and
// are widened to bf16 in registers and written straight into tensor memory,
// which the MMA reads as its A operand (tcgen05.mma with A in TMEM); only the
// raw codes and the token tiles pass through shared memory. FP8 widening is
// exact (every E4M3 value is a bf16 value) and bf16 x bf16 products are exact
// in the fp32 accumulator, so the per-channel scale is applied in the
// epilogue, where it factors out of the sum over k. An INT4 scale changes
// every 128 columns, so it is applied while widening: (c - 8) is exact in
// bf16 and one bf16 multiply rounds the product once (RNE), which is the
// dequantised weight the format defines.
//
// The unit of the pipeline is a k-pair (128 reduction columns): one raw
// stage of codes, one TMEM A stage, one token stage, 8 MMAs and one commit.
// A narrow MMA is cheap, so the issuing thread's own instruction stream sets
// the pace: few barrier operations per 8 MMAs keep it short, and waiting
// warps sleep on their barrier instead of spinning for issue slots.
//
// Block = 16 warps, one block per SM, persistent over the tile list:
//   warp 0     raw producer (one lane): TMA of 128 channels x one k-pair of
//              codes (FP8: 128 bytes a row, 128-byte swizzle, 10-deep ring;
//              INT4: 64 bytes a row, 64-byte swizzle, 18-deep ring, each
//              stage also receiving the tile's 128 group scales by a bulk copy)
//   warps 1,15 TMEM allocator (warp 1) + two MMA issuers (one lane each):
//              even k-pairs into one accumulator, odd into another
//   warp 2     token producer (one lane): TMA of the tile's rows (16-row
//              boxes, only the boxes that hold rows) x 64 bf16, two per stage,
//              into a token ring of its own: 4 stages, or 8 half-size stages
//              when the launch's tiles have at most 32 rows (decode)
//   warps 3-6  epilogue: accumulator lane = channel, column = row; scale,
//              bias, GELU, bf16, stores (one 64-byte segment per row and warp)
//   warps 7-14 converters: warp w owns TMEM lanes 32 (w % 4) .. +31 (the
//              lanes its warp may address) and one k-block of each pair;
//              lane = channel, 64 codes -> 32 TMEM columns per stage (INT4:
//              times the channel's scale of the k-pair's group)
// TMEM: 4 A stages x 64 columns, then two buffers of two 64-column
// accumulators (one per issuer), summed in the epilogue.
// Split-K (few rows, so that 148 SMs get equal shares): work item = (tile,
// range of k-pairs); each split writes its raw fp32 sums to its own plane and
// quant_split_finalize_kernel adds the planes in a fixed order and applies
// the (FP8) scale, bias and GELU.
// Every wait is bounded (globaltimer); on a timeout the block sets
// MOE_DEVERR_TIMEOUT, stops, drains its own copies and MMAs and frees TMEM.
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "grouped_gemm.cuh"

namespace moe {
namespace gg {

constexpr int QT_CH = 128;                      // output channels per tile (MMA M)
constexpr int QT_ROWS = 64;                     // rows per tile at most (MMA N <= 64)
constexpr int QT_KPAIR = 2 * BK;                // reduction columns per pipeline stage (= an INT4 group)

// Weight formats (the kernel's template argument) and their raw-code rings.
constexpr int QF_FP8 = 0;
constexpr int QF_INT4 = 1;
template <int F>
struct QFormat;
template <>
struct QFormat<QF_FP8> {
    static constexpr int ROW_BYTES = QT_KPAIR;      // one byte a code
    static constexpr int RSTAGES = 10;
};
template <>
struct QFormat<QF_INT4> {
    static constexpr int ROW_BYTES = QT_KPAIR / 2;  // two codes a byte
    static constexpr int RSTAGES = 18;
};
constexpr int QT_RAW_K = QFormat<QF_FP8>::ROW_BYTES;        // FP8 raw row: 128 bytes
constexpr int QT_RAW_BYTES = QT_CH * QT_RAW_K;                // 16 KB
constexpr int QT_RSTAGES = QFormat<QF_FP8>::RSTAGES;         // the raw-ring budget (160 KB) both use:
constexpr int QT_SCALE_BYTES = QT_CH * 2;                    // INT4: a stage's 128 bf16 group scales
static_assert(QFormat<QF_INT4>::RSTAGES * (QT_CH * QFormat<QF_INT4>::ROW_BYTES + QT_SCALE_BYTES) <=
                  QT_RSTAGES * QT_RAW_BYTES,
              "raw ring budget");
constexpr int QT_MAX_RSTAGES = QFormat<QF_INT4>::RSTAGES;
constexpr int QT_TBOX = 16;                     // token rows per TMA box
constexpr int QT_TBOX_BYTES = QT_TBOX * BK * 2;       // 2 KB (two 1024-byte swizzle atoms)
constexpr int QT_TOK_HALF = QT_ROWS * BK * 2;         // 8 KB: one k-block of a 64-row token tile
constexpr int QT_TOK_BYTES = 2 * QT_TOK_HALF;         // a k-pair
constexpr int QT_NARROW_ROWS = 32;                    // launches whose tiles have at most 32 rows ...
constexpr int QT_NARROW_TSTAGES = 8;                  // ... keep twice as many (half-size) token stages
constexpr int QT_MAX_TSTAGES = QT_NARROW_TSTAGES;
constexpr int QT_STAGES = 4;                    // A (TMEM) + token (shared) stages
constexpr int QT_A_COLS = BK;                   // 128 bf16 per lane = 64 columns
constexpr int QT_ACC_COL0 = QT_STAGES * QT_A_COLS;    // 256
constexpr int QT_ACC_COLS = QT_ROWS;            // fp32 columns of one issuer's accumulator
constexpr int QT_TMEM_COLS = 512;
static_assert(QT_ACC_COL0 + 4 * QT_ACC_COLS <= QT_TMEM_COLS, "TMEM budget");
constexpr int QT_CONVERTERS = 256;              // warps 7-14
constexpr int QT_ISSUER2 = 15;                  // the second MMA issuer warp
constexpr int QT_NUM_THREADS = 16 * 32;
constexpr int QT_BAR_BYTES = 1024;
constexpr int QT_SMEM_BYTES = QT_RSTAGES * QT_RAW_BYTES + QT_STAGES * QT_TOK_BYTES + QT_BAR_BYTES + 1024;
static_assert(QT_SMEM_BYTES <= 227 * 1024, "shared memory");

struct QTShared {
    uint64_t raw_full[QT_MAX_RSTAGES];
    uint64_t raw_empty[QT_MAX_RSTAGES];
    uint64_t a_full[QT_STAGES];    // the 8 converter warps wrote the stage's A columns
    uint64_t tok_full[QT_MAX_TSTAGES];   // the token stage's boxes have landed
    uint64_t tok_empty[QT_MAX_TSTAGES];  // the MMAs reading the token stage have completed
    uint64_t empty[QT_STAGES];           // the MMAs reading the A stage have completed
    uint64_t tfull[2][2];          // [accumulator buffer][issuer]
    uint64_t tempty[2];
    uint64_t drain[2];
    uint32_t tmem_base;
    volatile int abort_flag;
};
static_assert(sizeof(QTShared) <= QT_BAR_BYTES, "barrier block too large");

// try_wait that lets the thread sleep up to `ns` while the phase is pending
// (a waiting warp then takes no issue slots from the working ones)
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.b32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}

__device__ __noinline__ bool qt_wait_slow(QTShared *sh, uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                          bool raise) {
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait_sleep(bar, parity, 2000u)) return true;
        if ((it & 15u) == 15u) {
            if (raise && sh->abort_flag) return false;
            const uint64_t now = globaltimer_ns();
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

// Bounded wait with an inline fast path for a phase that has already completed.
__device__ __forceinline__ bool qt_wait(QTShared *sh, uint32_t bar, uint32_t parity, uint64_t limit_ns, bool raise) {
    if (mbar_try_wait(bar, parity)) return true;
    return qt_wait_slow(sh, bar, parity, limit_ns, raise);
}

// Two E4M3 codes -> two bf16, exactly. `sel` picks the two code bytes of w
// into bits 0-7 and 16-23 and fills bits 8-15 and 24-31 with copies of each
// code's sign bit (prmt's sign-replicating byte select). Shifted left by 4
// and masked, each half is the bf16 pattern sign | (7 magnitude bits << 4):
// 2^(E-127) (1 + M/8) for E >= 1 and the subnormal (M/8) 2^-126 for E = 0,
// i.e. the E4M3 value times 2^-120 in every case; one packed bf16 multiply by
// 2^120 (exact: at most 4 significant bits, no overflow, subnormals kept)
// gives the E4M3 value with its sign. (E4M3 NaN, codes 0x7f / 0xff, come out
// as +-480.)
__device__ __forceinline__ uint32_t e4m3x2_bf16x2(uint32_t w, uint32_t sel) {
    uint32_t t;
    asm("prmt.b32 %0, %1, 0, %2;" : "=r"(t) : "r"(w), "r"(sel));
    uint32_t pat = (t << 4) & 0x87F087F0u;
    const __nv_bfloat162 m = *reinterpret_cast<const __nv_bfloat162 *>(&pat);
    const __nv_bfloat162 k120 = __halves2bfloat162(__ushort_as_bfloat16((unsigned short)0x7B80u),
                                                   __ushort_as_bfloat16((unsigned short)0x7B80u));  // 2^120
    const __nv_bfloat162 v = __hmul2(m, k120);
    return *reinterpret_cast<const uint32_t *>(&v);
}

// 16 codes (one 16-byte chunk, memory order) -> 8 packed bf16 pairs.
__device__ __forceinline__ void e4m3x16_to_bf16(const uint4 &in, uint32_t *o) {
    o[0] = e4m3x2_bf16x2(in.x, 0x9180u);
    o[1] = e4m3x2_bf16x2(in.x, 0xB3A2u);
    o[2] = e4m3x2_bf16x2(in.y, 0x9180u);
    o[3] = e4m3x2_bf16x2(in.y, 0xB3A2u);
    o[4] = e4m3x2_bf16x2(in.z, 0x9180u);
    o[5] = e4m3x2_bf16x2(in.z, 0xB3A2u);
    o[6] = e4m3x2_bf16x2(in.w, 0x9180u);
    o[7] = e4m3x2_bf16x2(in.w, 0xB3A2u);
}

// 32 INT4 codes (16 bytes = four words of eight columns) -> 16 packed bf16
// pairs (c - 8) * scale. The layout puts a word's columns 2j and 2j + 1 at
// bits 4j and 16 + 4j, so ((w >> 4j) & 0x000F000F) | 0x43004300 (one shift
// and one three-input logic op) is the pair as the bf16 patterns 0x4300 | c
// (= 128 + c, exact); 136 is subtracted (exact: c - 8) and one bf16 multiply
// by the scale rounds the product once (RNE).
__device__ __forceinline__ void int4x32_to_bf16(const uint4 &in, __nv_bfloat162 scale, uint32_t *o) {
    const uint32_t words[4] = {in.x, in.y, in.z, in.w};
    const __nv_bfloat162 k136 = __halves2bfloat162(__ushort_as_bfloat16((unsigned short)0x4308u),
                                                   __ushort_as_bfloat16((unsigned short)0x4308u));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t t = ((words[i] >> (4 * j)) & 0x000F000Fu) | 0x43004300u;  // columns 8i + 2j, 8i + 2j + 1
            __nv_bfloat162 v = __hsub2(*reinterpret_cast<const __nv_bfloat162 *>(&t), k136);
            v = __hmul2(v, scale);
            o[4 * i + j] = *reinterpret_cast<const uint32_t *>(&v);
        }
    }
}

// This thread's lane of 32 consecutive TMEM columns.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
        "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
        "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}

// This thread's lane of 16 consecutive TMEM columns, read.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// D (TMEM) [+]= A (TMEM, 128 lanes x 16 bf16) * B (shared memory descriptor)^T.
__device__ __forceinline__ void mma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                            uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

// Position in a ring of n stages (n known only at run time): stage index
// and phase parity, advanced one fill at a time, so no division.
struct RingPos {
    int n, s;
    uint32_t ph;
    __device__ __forceinline__ void next() {
        if (++s == n) {
            s = 0;
            ph ^= 1u;
        }
    }
};

// Work item -> tile: the bf16 kernels' raster order with 128-channel n-tiles
// (tile_of numbers n-tiles in units of its own 256-column width).
// A tile with more rows than the launch's token stages hold is invalid
// (every role skips it; the epilogue flags it).
__device__ __forceinline__ Tile qt_tile(const Params &p, int w, int num_m, int num_n) {
    Tile t = tile_of<QT_ROWS>(p, w, num_m, num_n);
    t.n0 = (t.n0 / BN) * QT_CH;
    if (p.q_rows > 0 && p.q_rows <= QT_NARROW_ROWS && t.rows > QT_NARROW_ROWS) t.ok = false;
    return t;
}

// 16 bytes from shared memory (a .shared address: the converters' reads of
// the raw stages stay on the shared-memory path)
__device__ __forceinline__ uint4 lds128(uint32_t saddr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(saddr)
                 : "memory");
    return v;
}

__device__ __forceinline__ uint16_t lds16(uint32_t saddr) {
    uint16_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(saddr) : "memory");
    return v;
}

// 1-D bulk copy global -> shared (both 16-byte aligned, a multiple of 16
// bytes) that completes on the mbarrier as transaction bytes.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// wscale: FP8, the per-channel fp32 scales [groups * n_out]; gscale: INT4,
// the bf16 group scales [groups][k_dim / 128][n_out].
template <int F>
__global__ void __launch_bounds__(QT_NUM_THREADS, 1)
grouped_gemm_quant_kernel(const __grid_constant__ CUtensorMap tmT, const __grid_constant__ CUtensorMap tmBq,
                          const Params p, const float *__restrict__ wscale, const uint16_t *__restrict__ gscale) {
    constexpr int RS = QFormat<F>::RSTAGES;     // raw ring stages
    constexpr int RB = QFormat<F>::ROW_BYTES;   // bytes of a channel's row per k-pair
    constexpr int RAWB = QT_CH * RB;            // bytes of a raw stage
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    uint8_t *rawbuf = smem;
    uint8_t *scalebuf = rawbuf + RS * RAWB;  // INT4: each raw stage's 128 group scales
    uint8_t *tokbuf = rawbuf + QT_RSTAGES * QT_RAW_BYTES;
    QTShared *sh = reinterpret_cast<QTShared *>(tokbuf + QT_STAGES * QT_TOK_BYTES);
    // Token ring: the MMA reads each k-pair's token tile from it. It is
    // decoupled from the A ring, and launches whose tiles have at most 32 rows
    // (decode) split its bytes into twice as many stages, so the token loads
    // run further ahead of the MMAs.
    const bool narrow = p.q_rows > 0 && p.q_rows <= QT_NARROW_ROWS;
    const int tstages = narrow ? QT_NARROW_TSTAGES : QT_STAGES;
    const int tok_half = (narrow ? QT_NARROW_ROWS : QT_ROWS) * BK * 2;
    const int tok_bytes = 2 * tok_half;

    const int warp = warp_id();
    const int lane = lane_id();

    if (threadIdx.x == 0) {
        for (int s = 0; s < RS; ++s) {
            mbar_init(smem_u32(&sh->raw_full[s]), 1);
            mbar_init(smem_u32(&sh->raw_empty[s]), QT_CONVERTERS / 32);
        }
        for (int s = 0; s < QT_STAGES; ++s) {
            mbar_init(smem_u32(&sh->a_full[s]), QT_CONVERTERS / 32);
            mbar_init(smem_u32(&sh->empty[s]), 1);
        }
        for (int s = 0; s < QT_MAX_TSTAGES; ++s) {
            mbar_init(smem_u32(&sh->tok_full[s]), 1);
            mbar_init(smem_u32(&sh->tok_empty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&sh->tfull[a][0]), 1);
            mbar_init(smem_u32(&sh->tfull[a][1]), 1);
            mbar_init(smem_u32(&sh->tempty[a]), 4);
            mbar_init(smem_u32(&sh->drain[a]), 1);
        }
        sh->abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        prefetch_tmap(&tmT);
        prefetch_tmap(&tmBq);
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&sh->tmem_base)),
                     "r"(QT_TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = sh->tmem_base;

    const int num_m = num_m_tiles<QT_ROWS>(p);
    const int num_n = (p.n_out + QT_CH - 1) / QT_CH;
    const int splits = p.out_f32 != nullptr && p.k_splits > 1 ? p.k_splits : 1;
    const int total = num_m * num_n * splits;
    const int kblocks = p.k_dim / BK;
    const int kpairs = (kblocks + 1) / 2;
    const int kgroups = p.k_dim / QT_KPAIR;  // INT4: scale groups per row (= k-pairs)
    // work item w: tile w / splits, k-pairs [split_k0(w), split_k0(w + 1)) of it
    // (the last split of a tile ends at kpairs); kpairs * splits < 2^31
    auto split_k0 = [&](int w) { return (w % splits) * kpairs / splits; };
    auto split_k1 = [&](int w) { return (w % splits + 1) * kpairs / splits; };

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ raw producer (codes)
            int j = 0;
            bool stop = false;
            for (int w = blockIdx.x; w < total && !stop; w += gridDim.x) {
                const Tile t = qt_tile(p, w / splits, num_m, num_n);
                if (!t.ok) continue;
                const int brow = t.group * p.n_out + t.n0;
                const int k1 = split_k1(w);
                for (int kp = split_k0(w); kp < k1; ++kp, ++j) {
                    const int r = j % RS;
                    if (!qt_wait(sh, smem_u32(&sh->raw_empty[r]), ((uint32_t)(j / RS) & 1u) ^ 1u,
                                 WAIT_LIMIT_NS, true)) {
                        stop = true;
                        break;
                    }
                    // the second half of an odd k count's last pair reads zeros past k_dim;
                    // channels past the tensor's last row read zeros too
                    mbar_arrive_expect_tx(smem_u32(&sh->raw_full[r]), RAWB + (F == QF_INT4 ? QT_SCALE_BYTES : 0));
                    tma_load_2d(smem_u32(rawbuf + r * RAWB), &tmBq, smem_u32(&sh->raw_full[r]), kp * RB, brow);
                    if (F == QF_INT4)  // the tile's 128 channel scales of this k-pair's group (contiguous)
                        bulk_g2s(smem_u32(scalebuf + r * QT_SCALE_BYTES),
                                 gscale + ((size_t)t.group * kgroups + kp) * p.n_out + t.n0, QT_SCALE_BYTES,
                                 smem_u32(&sh->raw_full[r]));
                }
            }
            if (stop) {
                for (int jj = max(0, j - RS); jj < j; ++jj)
                    qt_wait(sh, smem_u32(&sh->raw_full[jj % RS]), (uint32_t)(jj / RS) & 1u,
                            DRAIN_LIMIT_NS, false);
            }
        }
        __syncwarp();
    } else if (warp == 2) {
        if (lane == 0) {
            // ------------------------------------------------ token producer
            RingPos tp{tstages, 0, 0u};
            int issued_phase[QT_MAX_TSTAGES];
            for (int s = 0; s < QT_MAX_TSTAGES; ++s) issued_phase[s] = -1;
            bool stop = false;
            for (int w = blockIdx.x; w < total && !stop; w += gridDim.x) {
                const Tile t = qt_tile(p, w / splits, num_m, num_n);
                if (!t.ok) continue;
                const int boxes = (t.rows + QT_TBOX - 1) / QT_TBOX;
                const int k1 = split_k1(w);
                for (int kp = split_k0(w); kp < k1; ++kp, tp.next()) {
                    const int s = tp.s;
                    if (!qt_wait(sh, smem_u32(&sh->tok_empty[s]), tp.ph ^ 1u, WAIT_LIMIT_NS, true)) {
                        stop = true;
                        break;
                    }
                    const int halves = (2 * kp + 1 < kblocks) ? 2 : 1;
                    mbar_arrive_expect_tx(smem_u32(&sh->tok_full[s]), (uint32_t)(halves * boxes * QT_TBOX_BYTES));
                    for (int h = 0; h < halves; ++h)
                        for (int b = 0; b < boxes; ++b)
                            tma_load_2d(smem_u32(tokbuf + s * tok_bytes + h * tok_half + b * QT_TBOX_BYTES),
                                        &tmT, smem_u32(&sh->tok_full[s]), (2 * kp + h) * BK, t.row0 + b * QT_TBOX);
                    issued_phase[s] = (int)tp.ph;
                }
            }
            if (stop) {  // let this block's copies in flight land before it exits
                for (int s = 0; s < tstages; ++s)
                    if (issued_phase[s] >= 0)
                        qt_wait(sh, smem_u32(&sh->tok_full[s]), (uint32_t)issued_phase[s], DRAIN_LIMIT_NS, false);
            }
        }
        __syncwarp();
    } else if (warp == 1 || warp == QT_ISSUER2) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuers
            // Issuer e takes the k-pairs kp = e, e + 2, ... of every tile into
            // its own accumulator: a narrow MMA costs its issuing thread more
            // time than the tensor core, and two issuers overlap.
            const int e = warp == 1 ? 0 : 1;
            int i = 0;
            RingPos tp{tstages, 0, 0u};  // token stage of k-pair i
            uint32_t acc = 0, acc_phase = 0;
            bool stop = false;
            for (int w = blockIdx.x; w < total && !stop; w += gridDim.x) {
                const Tile t = qt_tile(p, w / splits, num_m, num_n);
                if (!t.ok) continue;
                const uint32_t ncols = (uint32_t)((t.rows + 15) & ~15);  // MMA N: 16 .. 64
                const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((ncols >> 3) << 17) |
                                       ((uint32_t)(QT_CH >> 4) << 24);
                if (!qt_wait(sh, smem_u32(&sh->tempty[acc]), acc_phase ^ 1u, WAIT_LIMIT_NS, true)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + QT_ACC_COL0 + (2 * acc + e) * QT_ACC_COLS;
                const int k0 = split_k0(w), k1 = split_k1(w);
                for (int kp = k0; kp < k1; ++kp, ++i, tp.next()) {
                    if (((kp - k0) & 1) != e) continue;
                    const int s = i % QT_STAGES;
                    const uint32_t ph = (uint32_t)(i / QT_STAGES) & 1u;
                    if (!qt_wait(sh, smem_u32(&sh->a_full[s]), ph, WAIT_LIMIT_NS, true) ||
                        !qt_wait(sh, smem_u32(&sh->tok_full[tp.s]), tp.ph, WAIT_LIMIT_NS, true)) {
                        stop = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_tmem = tmem_base + s * QT_A_COLS;
                    const uint32_t b_addr = smem_u32(tokbuf + tp.s * tok_bytes);
                    if (2 * kp + 1 < kblocks) {
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            mma_bf16_ta(d_tmem, a_tmem + kk * (UMMA_K / 2),
                                        sdesc(b_addr + (kk >> 2) * tok_half + (kk & 3) * UMMA_K * 2), idesc,
                                        (kp != k0 + e || kk != 0) ? 1u : 0u);
                    } else {  // an odd k count's last pair: its first k-block only
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_bf16_ta(d_tmem, a_tmem + kk * (UMMA_K / 2), sdesc(b_addr + kk * UMMA_K * 2), idesc,
                                        (kp != k0 + e || kk != 0) ? 1u : 0u);
                    }
                    mma_commit(smem_u32(&sh->empty[s]));
                    mma_commit(smem_u32(&sh->tok_empty[tp.s]));
                }
                if (stop) break;
                // (an issuer without pairs in this tile commits nothing new: the arrival is immediate)
                mma_commit(smem_u32(&sh->tfull[acc][e]));
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            mma_commit(smem_u32(&sh->drain[e]));
            qt_wait(sh, smem_u32(&sh->drain[e]), 0, DRAIN_LIMIT_NS, false);
        }
        __syncwarp();
    } else if (warp < 7) {
        // ---------------------------------------------------- epilogue (warps 3-6)
        const int q = warp & 3;
        const int ch = q * 32 + lane;  // channel within the tile = accumulator lane
        uint32_t acc = 0, acc_phase = 0;
        for (int w = blockIdx.x; w < total; w += gridDim.x) {
            const Tile t = qt_tile(p, w / splits, num_m, num_n);
            if (!t.ok) {
                if (threadIdx.x == 96) flag_error(MOE_DEVERR_TILE_LIST);
                continue;
            }
            if (!qt_wait(sh, smem_u32(&sh->tfull[acc][0]), acc_phase, WAIT_LIMIT_NS, true) ||
                !qt_wait(sh, smem_u32(&sh->tfull[acc][1]), acc_phase, WAIT_LIMIT_NS, true))
                break;
            tc_fence_after();
            const int n = t.n0 + ch;
            const int k0 = split_k0(w), k1 = split_k1(w);
            const bool live = n < p.n_out;
            float scl = 0.f, b = 0.f;
            if (live) {
                scl = F == QF_FP8 ? __ldg(wscale + (size_t)t.group * p.n_out + n) : 1.0f;
                b = __ldg(p.bias + (size_t)t.group * p.n_out + n);
            }
            uint16_t *outc = p.out + (size_t)t.row0 * p.n_out + n;
            const uint32_t tbase = tmem_base + QT_ACC_COL0 + 2 * acc * QT_ACC_COLS + ((uint32_t)(q * 32) << 16);
            for (int c0 = 0; c0 < t.rows; c0 += 16) {  // t.rows is warp-uniform
                uint32_t r[16];
                float sum[16];
                tmem_ld16(tbase + c0, r);
                const bool none = k1 == k0;  // an empty split (not launched so; zeros if it were)
#pragma unroll
                for (int j = 0; j < 16; ++j) sum[j] = none ? 0.f : __uint_as_float(r[j]);
                if (k1 - k0 > 1) {  // the second issuer's accumulator (odd k-pairs)
                    tmem_ld16(tbase + QT_ACC_COLS + c0, r);
#pragma unroll
                    for (int j = 0; j < 16; ++j) sum[j] += __uint_as_float(r[j]);
                }
                if (live) {
                    // split mode: raw partial sums of this split (scale, bias, GELU come after)
                    float *part = splits > 1 ? p.out_f32 + ((size_t)(w % splits) * p.out_rows + t.row0) * p.n_out + n
                                             : nullptr;
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        if (c0 + j < t.rows) {
                            const size_t off = (size_t)(c0 + j) * p.n_out;
                            if (part != nullptr) {
                                part[off] = sum[j];
                            } else {
                                float v = fmaf(sum[j], scl, b);
                                if (p.gelu) v = gelu_erf(v);
                                const __nv_bfloat16 h = __float2bfloat16_rn(v);
                                outc[off] = *reinterpret_cast<const uint16_t *>(&h);
                            }
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sh->tempty[acc]));
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
    } else if (warp < 7 + QT_CONVERTERS / 32) {
        // ---------------------------------------------------- converters (warps 7-14)
        const int q = warp & 3;            // TMEM lane quarter this warp may address
        const int half = (warp - 7) >> 2;  // which k-block of each pair
        const int ch = q * 32 + lane;      // channel = raw row = TMEM lane
        const uint32_t rrow = smem_u32(rawbuf) + (uint32_t)(ch * RB);
        // the raw tile's swizzle: FP8 rows of 128 bytes (128-byte swizzle: chunk c
        // of row ch at c ^ (ch % 8)); INT4 rows of 64 bytes (64-byte swizzle:
        // chunk c at c ^ ((ch / 2) % 4))
        const int sw = F == QF_FP8 ? (ch & 7) : ((ch >> 1) & 3);
        const uint32_t tlane = tmem_base + ((uint32_t)(q * 32) << 16) + half * (BK / 2);
        int i = 0;  // k-pairs converted (= raw stages consumed)
        bool stop = false;
        for (int w = blockIdx.x; w < total && !stop; w += gridDim.x) {
            const Tile t = qt_tile(p, w / splits, num_m, num_n);
            if (!t.ok) continue;
            const int k1 = split_k1(w);
            for (int kp = split_k0(w); kp < k1; ++kp, ++i) {
                const int r = i % RS, s = i % QT_STAGES;
                if (!qt_wait(sh, smem_u32(&sh->raw_full[r]), (uint32_t)(i / RS) & 1u, WAIT_LIMIT_NS, true)) {
                    stop = true;
                    break;
                }
                const uint32_t src = rrow + (uint32_t)(r * RAWB);
                uint32_t v[32];
                if (F == QF_FP8) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int chunk = half * 4 + c;  // 16-byte chunks (16 codes) of this k-block
                        const uint4 in = lds128(src + (uint32_t)((chunk ^ sw) << 4));
                        e4m3x16_to_bf16(in, v + 8 * c);
                    }
                } else {
                    // this channel's scale for the k-pair's group (landed with the codes)
                    const uint16_t g = lds16(smem_u32(scalebuf) + r * QT_SCALE_BYTES + ch * 2);
                    const __nv_bfloat162 gs = __halves2bfloat162(__ushort_as_bfloat16(g), __ushort_as_bfloat16(g));
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const int chunk = half * 2 + c;  // 16-byte chunks (32 codes) of this k-block
                        const uint4 in = lds128(src + (uint32_t)((chunk ^ sw) << 4));
                        int4x32_to_bf16(in, gs, v + 16 * c);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&sh->raw_empty[r]));
                if (!qt_wait(sh, smem_u32(&sh->empty[s]), ((uint32_t)(i / QT_STAGES) & 1u) ^ 1u, WAIT_LIMIT_NS,
                             true)) {
                    stop = true;
                    break;
                }
                tc_fence_after();
                tmem_st32(tlane + s * QT_A_COLS, v);
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&sh->a_full[s]));
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(QT_TMEM_COLS)
                     : "memory");
    }
}

// Split-K finalize: out[r, n] = epilogue( scale[g(r), n] * sum_s part[s, r, n] + bias[g(r), n] )
// (scale = nullptr: 1, the INT4 format, whose scales were applied while widening),
// the splits added in order. Block (x, y) = row x, columns
// [1024 y, 1024 y + 1024); g(r) from the expert offsets (offsets = nullptr:
// one group); rows past the last expert's block were not computed and are
// skipped.
__global__ void __launch_bounds__(256)
quant_split_finalize_kernel(const float *__restrict__ part, int splits, int rows, int n_out,
                          const int32_t *__restrict__ offsets, int groups, const float *__restrict__ scale,
                          const float *__restrict__ bias, int gelu, uint16_t *__restrict__ out) {
    const int r = blockIdx.x;
    if (r >= rows) return;
    int g = 0;
    if (offsets != nullptr) {
        if (r >= offsets[groups]) return;
        int lo = 0, hi = groups;  // largest g with offsets[g] <= r
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (offsets[mid] <= r) lo = mid;
            else hi = mid;
        }
        g = lo;
    }
    const size_t plane = (size_t)rows * n_out;
    const float *pr = part + (size_t)r * n_out;
    const float *sc = scale != nullptr ? scale + (size_t)g * n_out : nullptr;
    const float *bi = bias + (size_t)g * n_out;
    uint16_t *o = out + (size_t)r * n_out;
    const int n = blockIdx.y * 1024 + threadIdx.x * 4;
    if (n < n_out) {  // n_out is a multiple of 64
        float4 acc = *reinterpret_cast<const float4 *>(pr + n);
        for (int s = 1; s < splits; ++s) {
            const float4 v = *reinterpret_cast<const float4 *>(pr + s * plane + n);
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        const float4 c = sc != nullptr ? *reinterpret_cast<const float4 *>(sc + n) : make_float4(1.f, 1.f, 1.f, 1.f);
        const float4 b = *reinterpret_cast<const float4 *>(bi + n);
        float y0 = fmaf(acc.x, c.x, b.x), y1 = fmaf(acc.y, c.y, b.y);
        float y2 = fmaf(acc.z, c.z, b.z), y3 = fmaf(acc.w, c.w, b.w);
        if (gelu) {
            y0 = gelu_erf(y0);
            y1 = gelu_erf(y1);
            y2 = gelu_erf(y2);
            y3 = gelu_erf(y3);
        }
        *reinterpret_cast<uint2 *>(o + n) = make_uint2(pack_bf16x2(y0, y1), pack_bf16x2(y2, y3));
    }
}

}  // namespace gg
}  // namespace moe
