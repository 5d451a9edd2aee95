// gemm_fp8w.cuh -- the grouped expert GEMM with weight-only FP8 expert
// weights (E4M3 codes, one fp32 scale per output channel; the weight
// quantisation of the lmnt.cn/news/351908 sec. 4.3 remark and the CSDN page's
// sec. 3.2 one-byte FP8 weights):
//
//   out[r, n] = epilogue( scale[g(r), n] * sum_k A[r, k] * code(B[g(r) * n_out + n, k]) + bias[g(r), n] )
//
// The weights cross HBM as one byte per element. Every E4M3 value is exact in
// bf16, so the codes are widened to bf16 in shared memory and multiplied on
// the tensor cores (tcgen05.mma kind::f16, bf16 x bf16 products exact in the
// fp32 accumulator); the per-channel scale is applied to the accumulator in
// the epilogue, where it factors out of the sum over k.
//
// Block = 14 warps, one block per SM, persistent over the same tile list as
// the bf16 kernel:
//   warp 0     TMA producer (one lane): raw FP8 B tiles of 256 rows x 128
//              codes (two k-blocks, full 128-byte rows) into a 3-deep staging
//              ring, running ahead of everything else
//   warp 1     TMEM allocator + MMA issuer (one lane), two accumulators
//   warps 2-5  epilogue: scale, bias, GELU, bf16, stores
//   warps 6-13 converters: when an operand stage is free, one lane issues the
//              TMA load of the bf16 A tile (128x64, 128-byte swizzle; 32-row
//              chunks for short tiles) while all 256 threads widen one k-block
//              of codes to bf16 into the stage, in the 128-byte-swizzled
//              K-major layout the MMA reads
// Every wait is bounded (globaltimer); on a timeout the block sets
// MOE_DEVERR_TIMEOUT, stops, drains its own copies and MMAs and frees TMEM.
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "grouped_gemm.cuh"

namespace moe {
namespace gg {

#ifndef MOE_FP8_OPERAND_STAGES
#define MOE_FP8_OPERAND_STAGES 2
#endif
#ifndef MOE_FP8_RAW_STAGES
#define MOE_FP8_RAW_STAGES 3
#endif
constexpr int Q_STAGES = MOE_FP8_OPERAND_STAGES;  // operand stages (A + widened B, 48 KB each)
constexpr int Q_RSTAGES = MOE_FP8_RAW_STAGES;     // raw FP8 B stages, two k-blocks each
constexpr int Q_RAW_K = 2 * BK;             // codes per raw row: 128 bytes
constexpr int Q_RAW_BYTES = BN * Q_RAW_K;   // 256 rows x 128 codes = 32 KB
constexpr int Q_CONVERTERS = 256;           // threads of warps 6-13
constexpr int Q_NUM_THREADS = NUM_THREADS + Q_CONVERTERS;
constexpr int Q_SMEM_BYTES = Q_STAGES * STAGE_BYTES + Q_RSTAGES * Q_RAW_BYTES + EPI_BYTES + BAR_BYTES + 1024;
static_assert(Q_SMEM_BYTES <= 227 * 1024, "shared memory");

struct QShared {
    uint64_t a_full[Q_STAGES];
    uint64_t b_full[Q_STAGES];
    uint64_t empty[Q_STAGES];  // MMA done with the stage (A and widened B)
    uint64_t raw_full[Q_RSTAGES];
    uint64_t raw_empty[Q_RSTAGES];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    uint32_t tmem_base;
    volatile int abort_flag;
};
static_assert(sizeof(QShared) <= BAR_BYTES, "barrier block too large");

__device__ __noinline__ bool q_wait(QShared *sh, uint32_t bar, uint32_t parity, uint64_t limit_ns, bool raise) {
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 255u) {
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

// Two E4M3 codes (bytes 0 and 1 of w selected by `sel`) -> two bf16, exactly.
// The 7 magnitude bits shifted left by 4 are the bf16 pattern of
// 2^(E-127) (1 + M/8) for E >= 1 and of the bf16 subnormal (M/8) 2^-126 for
// E = 0; one packed bf16 multiply by 2^120 (exact: at most 4 significant bits,
// no overflow, subnormal inputs kept) gives 2^(E-7) (1 + M/8) and M 2^-9, the
// E4M3 values; the sign bit is put back last. (E4M3 NaN, codes 0x7f / 0xff,
// come out as 480.)
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t w, uint32_t sel) {
    const uint32_t x = __byte_perm(w, 0u, sel);  // code a in bits 0-7, code b in bits 16-23
    uint32_t mag = (x << 4) & 0x07F007F0u;
    const __nv_bfloat162 m = *reinterpret_cast<const __nv_bfloat162 *>(&mag);
    const __nv_bfloat162 k120 = __halves2bfloat162(__ushort_as_bfloat16((unsigned short)0x7B80u),
                                                   __ushort_as_bfloat16((unsigned short)0x7B80u));  // 2^120
    const __nv_bfloat162 v = __hmul2(m, k120);
    return *reinterpret_cast<const uint32_t *>(&v) | ((x << 8) & 0x80008000u);
}

// Four codes -> four bf16 (two packed pairs, memory order).
__device__ __forceinline__ void e4m3x4_to_bf16(uint32_t w, uint32_t &lo, uint32_t &hi) {
    lo = e4m3x2_to_bf16x2(w, 0x4140u);
    hi = e4m3x2_to_bf16x2(w, 0x4342u);
}

__global__ void __launch_bounds__(Q_NUM_THREADS, 1)
grouped_gemm_fp8w_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmBq,
                         const __grid_constant__ CUtensorMap tmC, const Params p, const float *__restrict__ wscale,
                         const __grid_constant__ CUtensorMap tmA32) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    uint8_t *rawbuf = smem + Q_STAGES * STAGE_BYTES;
    uint8_t *epibuf = rawbuf + Q_RSTAGES * Q_RAW_BYTES;
    QShared *sh = reinterpret_cast<QShared *>(epibuf + EPI_BYTES);

    const int warp = warp_id();
    const int lane = lane_id();

    if (threadIdx.x == 0) {
        for (int s = 0; s < Q_STAGES; ++s) {
            mbar_init(smem_u32(&sh->a_full[s]), 1);
            mbar_init(smem_u32(&sh->b_full[s]), Q_CONVERTERS / 32);
            mbar_init(smem_u32(&sh->empty[s]), 1);
        }
        for (int s = 0; s < Q_RSTAGES; ++s) {
            mbar_init(smem_u32(&sh->raw_full[s]), 1);
            mbar_init(smem_u32(&sh->raw_empty[s]), Q_CONVERTERS / 32);
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
        prefetch_tmap(&tmBq);
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
    const int total = num_m * num_n;
    const int kblocks = p.k_dim / BK;

    const int kpairs = (kblocks + 1) / 2;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer (raw FP8 B only)
            int j = 0;  // raw stages issued by this block
            bool stop = false;
            for (int w = blockIdx.x; w < total && !stop; w += gridDim.x) {
                Tile t = tile_of<BM>(p, w, num_m, num_n);
                if (!t.ok) continue;
                const int brow = t.group * p.n_out + t.n0;
                for (int kp = 0; kp < kpairs; ++kp, ++j) {
                    const int r = j % Q_RSTAGES;
                    const uint32_t rph = (uint32_t)(j / Q_RSTAGES) & 1u;
                    if (!q_wait(sh, smem_u32(&sh->raw_empty[r]), rph ^ 1u, WAIT_LIMIT_NS, true)) {
                        stop = true;
                        break;
                    }
                    // the last pair of an odd k count reads zeros past k_dim
                    mbar_arrive_expect_tx(smem_u32(&sh->raw_full[r]), Q_RAW_BYTES);
                    tma_load_2d(smem_u32(rawbuf + r * Q_RAW_BYTES), &tmBq, smem_u32(&sh->raw_full[r]), kp * Q_RAW_K,
                                brow);
                }
            }
            if (stop) {
                // let this block's copies in flight land before the block exits
                for (int jj = max(0, j - Q_RSTAGES); jj < j; ++jj)
                    q_wait(sh, smem_u32(&sh->raw_full[jj % Q_RSTAGES]), (uint32_t)(jj / Q_RSTAGES) & 1u,
                           DRAIN_LIMIT_NS, false);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            int i = 0;
            uint32_t acc = 0, acc_phase = 0;
            bool stop = false;
            for (int w = blockIdx.x; w < total && !stop; w += gridDim.x) {
                Tile t = tile_of<BM>(p, w, num_m, num_n);
                if (!t.ok) continue;
                if (!q_wait(sh, smem_u32(&sh->tempty[acc]), acc_phase ^ 1u, WAIT_LIMIT_NS, true)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * ACC_COLS;
                for (int kb = 0; kb < kblocks; ++kb, ++i) {
                    const int s = i % Q_STAGES;
                    const uint32_t ph = (uint32_t)(i / Q_STAGES) & 1u;
                    if (!q_wait(sh, smem_u32(&sh->a_full[s]), ph, WAIT_LIMIT_NS, true) ||
                        !q_wait(sh, smem_u32(&sh->b_full[s]), ph, WAIT_LIMIT_NS, true)) {
                        stop = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(smem + s * STAGE_BYTES);
                    const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < BK / UMMA_K; ++kk)
                        mma_bf16(d_tmem, sdesc(a_addr + kk * UMMA_K * 2), sdesc(b_addr + kk * UMMA_K * 2),
                                 (kb != 0 || kk != 0) ? 1u : 0u);
                    mma_commit(smem_u32(&sh->empty[s]));
                }
                if (stop) break;
                mma_commit(smem_u32(&sh->tfull[acc]));
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            mma_commit(smem_u32(&sh->drain));
            q_wait(sh, smem_u32(&sh->drain), 0, DRAIN_LIMIT_NS, false);
        }
        __syncwarp();
    } else if (warp < 6) {
        // ---------------------------------------------------- epilogue (warps 2-5)
        const int q = warp & 3;
        const int row = q * 32 + lane;
        uint8_t *ebuf = epibuf + (warp - 2) * 2 * EPI_BUF_BYTES;
        int ebuf_idx = 0;
        uint32_t acc = 0, acc_phase = 0;
        for (int w = blockIdx.x; w < total; w += gridDim.x) {
            Tile t = tile_of<BM>(p, w, num_m, num_n);
            if (!t.ok) {
                if (threadIdx.x == 64) flag_error(MOE_DEVERR_TILE_LIST);
                continue;
            }
            if (!q_wait(sh, smem_u32(&sh->tfull[acc]), acc_phase, WAIT_LIMIT_NS, true)) break;
            tc_fence_after();
            const int rows_valid = max(0, min(32, t.rows - q * 32));
            uint16_t *out_row = p.out + (size_t)(t.row0 + row) * p.n_out;
            const float *bias = p.bias + (size_t)t.group * p.n_out;
            const float *scl = wscale + (size_t)t.group * p.n_out;
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
                    const float4 sc = __ldg(reinterpret_cast<const float4 *>(scl + col + j));
                    float v0 = fmaf(__uint_as_float(r[j + 0]), sc.x, b.x);
                    float v1 = fmaf(__uint_as_float(r[j + 1]), sc.y, b.y);
                    float v2 = fmaf(__uint_as_float(r[j + 2]), sc.z, b.z);
                    float v3 = fmaf(__uint_as_float(r[j + 3]), sc.w, b.w);
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
    } else {
        // ---------------------------------------------------- converters (warps 6-13)
        // Unit u = ct + 256 m (m < 4): 16 codes of row u / 4, columns
        // 16 (u % 4) .. +15 of the k-block's half of the raw row, widened to
        // two 16-byte bf16 chunks 2 (u % 4) and 2 (u % 4) + 1 of that row in
        // the operand stage, each at chunk position (c ^ (row % 8)) of the
        // row's 128 bytes (the 128-byte swizzle the MMA descriptor declares).
        const int ct = threadIdx.x - NUM_THREADS;
        int i = 0, j = 0;  // k-blocks converted, raw stages consumed
        int last_a = -1;
        bool stop = false;
        for (int w = blockIdx.x; w < total && !stop; w += gridDim.x) {
            Tile t = tile_of<BM>(p, w, num_m, num_n);
            if (!t.ok) continue;
            for (int kb = 0; kb < kblocks; ++kb, ++i) {
                const int r = j % Q_RSTAGES, s = i % Q_STAGES;
                const uint32_t rph = (uint32_t)(j / Q_RSTAGES) & 1u, ph = (uint32_t)(i / Q_STAGES) & 1u;
                if (!q_wait(sh, smem_u32(&sh->empty[s]), ph ^ 1u, WAIT_LIMIT_NS, true)) {
                    stop = true;
                    break;
                }
                if (ct == 0) {
                    mbar_arrive_expect_tx(smem_u32(&sh->a_full[s]), a_tile_bytes(t.rows));
                    load_a_tile(smem_u32(smem + s * STAGE_BYTES), &tmA, &tmA32, smem_u32(&sh->a_full[s]), kb * BK,
                                t.row0, t.rows);
                    last_a = i;
                }
                if (!q_wait(sh, smem_u32(&sh->raw_full[r]), rph, WAIT_LIMIT_NS, true)) {
                    stop = true;
                    break;
                }
                const uint8_t *src = rawbuf + r * Q_RAW_BYTES + (kb & 1) * BK;
                uint8_t *dst = smem + s * STAGE_BYTES + A_BYTES;
#pragma unroll
                for (int m = 0; m < (BN * 4) / Q_CONVERTERS; ++m) {
                    const int u = ct + Q_CONVERTERS * m;
                    const int brow = u >> 2, grp = u & 3;
                    const uint4 in = *reinterpret_cast<const uint4 *>(src + brow * Q_RAW_K + grp * 16);
                    uint4 o0, o1;
                    e4m3x4_to_bf16(in.x, o0.x, o0.y);
                    e4m3x4_to_bf16(in.y, o0.z, o0.w);
                    e4m3x4_to_bf16(in.z, o1.x, o1.y);
                    e4m3x4_to_bf16(in.w, o1.z, o1.w);
                    uint8_t *drow = dst + brow * 128;
                    const int sw = brow & 7;
                    *reinterpret_cast<uint4 *>(drow + (((2 * grp) ^ sw) << 4)) = o0;
                    *reinterpret_cast<uint4 *>(drow + (((2 * grp + 1) ^ sw) << 4)) = o1;
                }
                // the widened tile is read by the tensor cores (async proxy):
                // every thread fences its own writes, then one arrival per warp
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                const bool pair_done = (kb & 1) || kb + 1 == kblocks;  // both halves of the raw stage consumed
                if (lane == 0) {
                    mbar_arrive(smem_u32(&sh->b_full[s]));
                    if (pair_done) mbar_arrive(smem_u32(&sh->raw_empty[r]));
                }
                if (pair_done) ++j;
            }
        }
        if (stop && ct == 0) {
            for (int ii = max(0, last_a - Q_STAGES + 1); ii <= last_a; ++ii)
                q_wait(sh, smem_u32(&sh->a_full[ii % Q_STAGES]), (uint32_t)(ii / Q_STAGES) & 1u, DRAIN_LIMIT_NS,
                       false);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                     : "memory");
    }
}

}  // namespace gg
}  // namespace moe
