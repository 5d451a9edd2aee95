// route.cuh -- gate logits, TopK-then-softmax routing and the balance-loss
// statistics (lmnt.cn/news/351908 sec. 2.1 score = Softmax(TopK(W_g x)),
// sec. 5.2 statistics; selection bias b_i from the yunthe.com MoE page).
//
// Logits are fp32 sums of bf16 x bf16 products on the CUDA cores. On the 1/64
// input grid every partial sum is an exact multiple of 2^-12 below 2^11, so the
// logits, and therefore the TopK decisions, do not depend on summation order.
#pragma once

#include "common.cuh"

namespace moe {
namespace route {

constexpr int kGateThreads = 256;

// ---------------------------------------------------------------------------
// Small N (<= 16): the whole router in one kernel.
//  * x streams through shared memory: thread 0 issues one bulk copy
//    (cp.async.bulk, mbarrier completion) per token row, 4 tokens per stage,
//    up to 4 stages in flight per block.
//  * Warp w owns the 8-element column chunks [w*CPW, (w+1)*CPW); its slice of
//    W_g (all N experts) is loaded into registers once per block.
//  * Per stage every warp forms partial logits of the 4 tokens over its
//    chunks; the 8 partials meet in shared memory. Warp tk (< 4) then adds
//    them in warp order for token tk, lane e holding expert e, and runs the
//    full softmax, K rounds of warp arg-max and the K-way softmax with
//    shuffles; lane k writes rank k.
constexpr int kRouterWarps = 8;
constexpr int kTokensPerStage = 4;
constexpr int kMaxK = 8;
constexpr int kMaxPartialRows = 1024;
constexpr int kRouterBlocks = 148;
constexpr int kRouterMaxStages = 4;
constexpr size_t kRouterSmemBudget = 192 * 1024;

// Blocks of the small-N router: a function of T only (not of the device), so
// the per-block partial probability sums are identical on every GPU.
inline int small_router_grid(int T) {
    int g = (T + kTokensPerStage - 1) / kTokensPerStage;
    return g < 1 ? 1 : (g > kRouterBlocks ? kRouterBlocks : g);
}
inline int small_router_stages(int d) {
    size_t per = (size_t)kTokensPerStage * d * 2;
    int s = (int)(kRouterSmemBudget / per);
    return s < 1 ? 1 : (s > kRouterMaxStages ? kRouterMaxStages : s);
}
inline size_t small_router_smem(int d) {
    return (size_t)small_router_stages(d) * kTokensPerStage * d * 2 + 64;
}

__device__ __forceinline__ uint32_t r_smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ bool r_try_wait(uint32_t bar, uint32_t parity) {
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

// Bounded wait (about 4 s): false after the limit, with the error bit set.
__device__ __noinline__ bool r_wait(uint32_t bar, uint32_t parity) {
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        if (r_try_wait(bar, parity)) return true;
        if ((it & 255u) == 255u) {
            uint64_t now = globaltimer_ns();
            if (t0 == 0) {
                t0 = now;
            } else if (now - t0 > 4000000000ull) {
                flag_error(MOE_DEVERR_TIMEOUT);
                return false;
            }
        }
    }
}

// Bulk copies of the stage's token rows (thread 0 only).
__device__ __forceinline__ void router_issue(uint32_t bar, uint8_t *dst, const uint16_t *x, int t0, int T,
                                             int d) {
    const uint32_t row_bytes = (uint32_t)d * 2;
    int n = T - t0;
    n = n < kTokensPerStage ? n : kTokensPerStage;
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(row_bytes * n)
                 : "memory");
    for (int i = 0; i < n; ++i) {
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                r_smem_u32(dst + (size_t)i * row_bytes)),
            "l"(reinterpret_cast<uint64_t>(x + (size_t)(t0 + i) * d)), "r"(row_bytes), "r"(bar)
            : "memory");
    }
}

template <int NMAX, int JMAX>
__global__ void __launch_bounds__(kRouterWarps * 32, 1)
router_smallN_kernel(const uint16_t *__restrict__ x, const uint16_t *__restrict__ Wg,
                     const float *__restrict__ sel_bias, int T, int d, int N, int K, int stages,
                     int32_t *__restrict__ topk_idx, float *__restrict__ topk_w,
                     int32_t *__restrict__ demand, float *__restrict__ prob_partial,
                     float *__restrict__ lse_partial) {
    extern __shared__ __align__(128) uint8_t xs[];  // [stages][4][d] bf16
    __shared__ __align__(8) uint64_t full[kRouterMaxStages];
    __shared__ float red[2][kRouterWarps][kTokensPerStage][NMAX];
    __shared__ int dcount[NMAX];
    __shared__ float psum_w[kTokensPerStage][NMAX];
    __shared__ float lsq_w[kTokensPerStage];
    __shared__ int abort_flag;
    const int chunks = d >> 3;
    const int lane = lane_id();
    const int warp = warp_id();
    constexpr int CPW = 32 * JMAX;  // chunks per warp
    const size_t stage_bytes = (size_t)kTokensPerStage * d * 2;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kRouterMaxStages; ++s)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(r_smem_u32(&full[s])), "r"(1) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        abort_flag = 0;
    }
    if (threadIdx.x < NMAX) dcount[threadIdx.x] = 0;
    __syncthreads();

    const int ngroups = (T + kTokensPerStage - 1) / kTokensPerStage;
    const int my_groups = blockIdx.x < ngroups ? (ngroups - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    if (threadIdx.x == 0) {
        for (int i = 0; i < stages && i < my_groups; ++i)
            router_issue(r_smem_u32(&full[i]), xs + i * stage_bytes, x,
                         (blockIdx.x + i * gridDim.x) * kTokensPerStage, T, d);
    }

    // this warp's W_g slice, all experts, in registers
    uint4 wreg[NMAX][JMAX];
#pragma unroll
    for (int e = 0; e < NMAX; ++e)
#pragma unroll
        for (int j = 0; j < JMAX; ++j) {
            const int c = warp * CPW + lane + 32 * j;
            wreg[e][j] = (e < N && c < chunks) ? __ldg(reinterpret_cast<const uint4 *>(Wg + (size_t)e * d) + c)
                                              : make_uint4(0u, 0u, 0u, 0u);
        }
    const float bias_lane = (sel_bias != nullptr && lane < N) ? sel_bias[lane] : 0.f;
    float pacc_lane = 0.f;  // routing warps: sum over their tokens of softmax_N[lane]
    float lsq = 0.f;        // routing warps: sum over their tokens of logsumexp^2 (z-loss)

    for (int i = 0; i < my_groups; ++i) {
        const int g = blockIdx.x + i * gridDim.x;
        const int t0 = g * kTokensPerStage;
        const int st = i % stages;
        if (!r_wait(r_smem_u32(&full[st]), (uint32_t)((i / stages) & 1))) abort_flag = 1;
        __syncthreads();
        if (abort_flag) break;  // block-uniform
        const uint16_t *xst = reinterpret_cast<const uint16_t *>(xs + st * stage_bytes);
        float acc[kTokensPerStage][NMAX];
#pragma unroll
        for (int tk = 0; tk < kTokensPerStage; ++tk)
#pragma unroll
            for (int e = 0; e < NMAX; ++e) acc[tk][e] = 0.f;
#pragma unroll
        for (int j = 0; j < JMAX; ++j) {
            const int c = warp * CPW + lane + 32 * j;
            if (c < chunks) {
                float xf[kTokensPerStage][8];
#pragma unroll
                for (int tk = 0; tk < kTokensPerStage; ++tk) {
                    uint4 xv = make_uint4(0u, 0u, 0u, 0u);
                    if (t0 + tk < T) xv = reinterpret_cast<const uint4 *>(xst + (size_t)tk * d)[c];
                    unpack_bf16x2(xv.x, xf[tk][0], xf[tk][1]);
                    unpack_bf16x2(xv.y, xf[tk][2], xf[tk][3]);
                    unpack_bf16x2(xv.z, xf[tk][4], xf[tk][5]);
                    unpack_bf16x2(xv.w, xf[tk][6], xf[tk][7]);
                }
#pragma unroll
                for (int e = 0; e < NMAX; ++e) {
                    if (e < N) {
                        float wf[8];
                        unpack_bf16x2(wreg[e][j].x, wf[0], wf[1]);
                        unpack_bf16x2(wreg[e][j].y, wf[2], wf[3]);
                        unpack_bf16x2(wreg[e][j].z, wf[4], wf[5]);
                        unpack_bf16x2(wreg[e][j].w, wf[6], wf[7]);
#pragma unroll
                        for (int tk = 0; tk < kTokensPerStage; ++tk)
#pragma unroll
                            for (int q = 0; q < 8; ++q) acc[tk][e] = fmaf(xf[tk][q], wf[q], acc[tk][e]);
                    }
                }
            }
        }
#pragma unroll
        for (int tk = 0; tk < kTokensPerStage; ++tk)
#pragma unroll
            for (int e = 0; e < NMAX; ++e)
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) acc[tk][e] += __shfl_xor_sync(0xffffffffu, acc[tk][e], o);
        if (lane == 0) {
#pragma unroll
            for (int tk = 0; tk < kTokensPerStage; ++tk)
#pragma unroll
                for (int e = 0; e < NMAX; ++e) red[i & 1][warp][tk][e] = acc[tk][e];
        }
        __syncthreads();  // stage consumed, partials visible
        if (threadIdx.x == 0 && i + stages < my_groups) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            router_issue(r_smem_u32(&full[st]), xs + st * stage_bytes, x,
                         (blockIdx.x + (i + stages) * gridDim.x) * kTokensPerStage, T, d);
        }
        if (warp < kTokensPerStage && t0 + warp < T) {
            // warp tk routes token t0 + tk; lane e holds expert e (N <= 16 < 32)
            const int t = t0 + warp;
            const bool live = lane < N;
            float sv = 0.f;
            if (live) {
                sv = red[i & 1][0][warp][lane];
#pragma unroll
                for (int w = 1; w < kRouterWarps; ++w) sv += red[i & 1][w][warp][lane];
            }
            // softmax over all N unbiased logits (balance-loss statistic)
            float m = live ? sv : -INFINITY;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            const float ex = live ? expf(sv - m) : 0.f;
            float z = ex;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
            pacc_lane += ex / z;
            const float lse = m + logf(z);
            lsq += lse * lse;
            // TopK on u = s + b: K rounds of warp arg-max, larger u first,
            // equal u -> smaller expert id first
            const float u = sv + bias_lane;
            bool taken = !live;
            int sel_e = 0;
            float sel_s = 0.f, mk = -INFINITY;
            float my_s = 0.f;
            int my_k = -1;
            for (int k = 0; k < K; ++k) {
                float bu = taken ? -INFINITY : u;
                int be = taken ? 0x7fffffff : lane;
                float bs = sv;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    const float ou = __shfl_xor_sync(0xffffffffu, bu, o);
                    const int oe = __shfl_xor_sync(0xffffffffu, be, o);
                    const float os = __shfl_xor_sync(0xffffffffu, bs, o);
                    if (ou > bu || (ou == bu && oe < be)) {
                        bu = ou;
                        be = oe;
                        bs = os;
                    }
                }
                if (lane == be) taken = true;
                if (lane == k) {
                    my_k = k;
                    my_s = bs;
                    sel_e = be;
                }
                mk = fmaxf(mk, bs);
                (void)sel_s;
            }
            // softmax over the K selected, unbiased logits; lane k owns rank k
            const float num = (my_k >= 0) ? expf(my_s - mk) : 0.f;
            float den = num;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
            if (my_k >= 0) {
                topk_idx[(size_t)t * K + my_k] = sel_e;
                topk_w[(size_t)t * K + my_k] = num / den;
                if ((unsigned)sel_e < (unsigned)N)
                    atomicAdd(&dcount[sel_e], 1);
                else
                    flag_error(MOE_DEVERR_EXPERT_ID);  // no orderable logit (NaN input)
            }
        }
    }
    // every bulk copy this block issued has landed before the block exits
    if (threadIdx.x == 0 && abort_flag) {
        for (int i2 = 0; i2 < stages && i2 < my_groups; ++i2) r_wait(r_smem_u32(&full[i2]), 0u);
    }
    __syncthreads();
    if (warp < kTokensPerStage && lane < N) psum_w[warp][lane] = pacc_lane;
    if (warp < kTokensPerStage && lane == 0) lsq_w[warp] = lsq;
    __syncthreads();
    if (warp == 0 && lane < N) {
        float a = psum_w[0][lane];
#pragma unroll
        for (int w = 1; w < kTokensPerStage; ++w) a += psum_w[w][lane];
        prob_partial[(size_t)blockIdx.x * N + lane] = a;
        if (dcount[lane]) atomicAdd(&demand[lane], dcount[lane]);
    }
    if (threadIdx.x == 0) {
        float a = lsq_w[0];
#pragma unroll
        for (int w = 1; w < kTokensPerStage; ++w) a += lsq_w[w];
        lse_partial[blockIdx.x] = a;
    }
}

// ---------------------------------------------------------------------------
// Gate GEMM, general N: 64 tokens x 64 experts per block, k-slabs of 32 staged
// in shared memory as fp32, 4 x 4 outputs per thread.
constexpr int kGBM = 64, kGBN = 64, kGBK = 32;

__global__ void __launch_bounds__(kGateThreads)
gate_logits_tiled_kernel(const uint16_t *__restrict__ x, const uint16_t *__restrict__ Wg, int T,
                         int d, int N, float *__restrict__ logits) {
    __shared__ __align__(16) float As[kGBK][kGBM + 4];
    __shared__ __align__(16) float Bs[kGBK][kGBN + 4];
    const int m0 = blockIdx.x * kGBM;
    const int n0 = blockIdx.y * kGBN;
    const int tid = threadIdx.x;
    const int tx = tid & 15;   // expert quad
    const int ty = tid >> 4;   // token quad
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

    // each thread stages one 8-element chunk of A and one of B per slab
    const int lr = tid >> 2;          // 0..63 row within tile
    const int lc = (tid & 3) * 8;     // 0,8,16,24 column within slab
    for (int k0 = 0; k0 < d; k0 += kGBK) {
        {
            float f[8];
            int r = m0 + lr;
            if (r < T) {
                uint4 v = __ldg(reinterpret_cast<const uint4 *>(x + (size_t)r * d + k0 + lc));
                unpack_bf16x2(v.x, f[0], f[1]);
                unpack_bf16x2(v.y, f[2], f[3]);
                unpack_bf16x2(v.z, f[4], f[5]);
                unpack_bf16x2(v.w, f[6], f[7]);
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) f[j] = 0.f;
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) As[lc + j][lr] = f[j];
            int e = n0 + lr;
            if (e < N) {
                uint4 v = __ldg(reinterpret_cast<const uint4 *>(Wg + (size_t)e * d + k0 + lc));
                unpack_bf16x2(v.x, f[0], f[1]);
                unpack_bf16x2(v.y, f[2], f[3]);
                unpack_bf16x2(v.z, f[4], f[5]);
                unpack_bf16x2(v.w, f[6], f[7]);
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) f[j] = 0.f;
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) Bs[lc + j][lr] = f[j];
        }
        __syncthreads();
#pragma unroll 8
        for (int k = 0; k < kGBK; ++k) {
            float4 a = *reinterpret_cast<const float4 *>(&As[k][ty * 4]);
            float4 b = *reinterpret_cast<const float4 *>(&Bs[k][tx * 4]);
            float av[4] = {a.x, a.y, a.z, a.w};
            float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        int r = m0 + ty * 4 + i;
        if (r >= T) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            int e = n0 + tx * 4 + j;
            if (e < N) logits[(size_t)r * N + e] = acc[i][j];
        }
    }
}

// ---------------------------------------------------------------------------
// TopK then softmax, one warp per token. `logits` holds `splits` partial-sum
// planes [splits][T][N] (1 for the CUDA-core gate). Lane l holds the logits of experts
// l, l+32, ... (LPL of them). K rounds of a warp arg-max on (u desc, id asc)
// pick the experts; the softmax runs over their unbiased logits. The full-N
// softmax probabilities are accumulated per lane (each lane owns its experts),
// reduced over the block's warps in a fixed order and written as one partial
// row per block: no floating-point atomics, so results are run-to-run stable.
constexpr int kTopkWarps = 8;

template <int LPL>
__global__ void __launch_bounds__(kTopkWarps * 32)
topk_softmax_kernel(const float *__restrict__ logits, int splits, const float *__restrict__ sel_bias, int T,
                    int N, int K, int32_t *__restrict__ topk_idx, float *__restrict__ topk_w,
                    int32_t *__restrict__ demand, float *__restrict__ prob_partial,
                    float *__restrict__ lse_partial) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    __shared__ float lsq_w[kTopkWarps];
    float *psum = reinterpret_cast<float *>(smem_raw);                       // [warps][N]
    int *dcount = reinterpret_cast<int *>(psum + kTopkWarps * N);            // [N]
    for (int e = threadIdx.x; e < N; e += blockDim.x) dcount[e] = 0;
    __syncthreads();

    const int lane = lane_id();
    const int warp = warp_id();
    float pacc[LPL];
#pragma unroll
    for (int i = 0; i < LPL; ++i) pacc[i] = 0.f;
    float bias[LPL];
#pragma unroll
    for (int i = 0; i < LPL; ++i) {
        int e = lane + 32 * i;
        bias[i] = (sel_bias != nullptr && e < N) ? sel_bias[e] : 0.f;
    }

    float lsq = 0.f;  // sum over this warp's tokens of logsumexp(s_t)^2 (z-loss)
    for (int t = blockIdx.x * kTopkWarps + warp; t < T; t += gridDim.x * kTopkWarps) {
        float s[LPL];
        float m = -INFINITY;
#pragma unroll
        for (int i = 0; i < LPL; ++i) {
            int e = lane + 32 * i;
            if (e < N) {
                // the gate GEMM may leave K-split partial sums: add them in split order
                float a = logits[(size_t)t * N + e];
                for (int sp = 1; sp < splits; ++sp) a += logits[((size_t)sp * T + t) * N + e];
                s[i] = a;
            } else {
                s[i] = -INFINITY;
            }
            m = fmaxf(m, s[i]);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float ex[LPL];
        float z = 0.f;
#pragma unroll
        for (int i = 0; i < LPL; ++i) {
            ex[i] = (lane + 32 * i < N) ? expf(s[i] - m) : 0.f;
            z += ex[i];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
        const float inv_z = 1.f / z;
        const float lse = m + logf(z);
        lsq += lse * lse;
#pragma unroll
        for (int i = 0; i < LPL; ++i) pacc[i] += ex[i] * inv_z;

        // K rounds of arg-max over the unselected experts
        unsigned taken = 0u;
        int sel_e[kMaxK];
        float sel_s[kMaxK];
#pragma unroll
        for (int k = 0; k < kMaxK; ++k) {
            sel_e[k] = 0;
            sel_s[k] = 0.f;
            if (k < K) {
                float bu = -INFINITY, bs = 0.f;
                int be = 0x7fffffff;
#pragma unroll
                for (int i = 0; i < LPL; ++i) {
                    int e = lane + 32 * i;
                    float u = s[i] + bias[i];
                    bool ok = (e < N) && !((taken >> i) & 1u);
                    if (ok && (u > bu || (u == bu && e < be))) {
                        bu = u;
                        be = e;
                        bs = s[i];
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    float ou = __shfl_xor_sync(0xffffffffu, bu, o);
                    int oe = __shfl_xor_sync(0xffffffffu, be, o);
                    float os = __shfl_xor_sync(0xffffffffu, bs, o);
                    if (ou > bu || (ou == bu && oe < be)) {
                        bu = ou;
                        be = oe;
                        bs = os;
                    }
                }
                sel_e[k] = be;
                sel_s[k] = bs;
                if ((be & 31) == lane) taken |= 1u << (be >> 5);
            }
        }
        float mk = -INFINITY;
#pragma unroll
        for (int k = 0; k < kMaxK; ++k)
            if (k < K) mk = fmaxf(mk, sel_s[k]);
        float den = 0.f;
        float num[kMaxK];
#pragma unroll
        for (int k = 0; k < kMaxK; ++k) {
            num[k] = (k < K) ? expf(sel_s[k] - mk) : 0.f;
            den += num[k];
        }
#pragma unroll
        for (int k = 0; k < kMaxK; ++k) {
            if (k < K && lane == k) {
                topk_idx[(size_t)t * K + k] = sel_e[k];
                topk_w[(size_t)t * K + k] = num[k] / den;
                if ((unsigned)sel_e[k] < (unsigned)N)
                    atomicAdd(&dcount[sel_e[k]], 1);
                else
                    flag_error(MOE_DEVERR_EXPERT_ID);  // no orderable logit (NaN input)
            }
        }
    }
#pragma unroll
    for (int i = 0; i < LPL; ++i) {
        int e = lane + 32 * i;
        if (e < N) psum[warp * N + e] = pacc[i];
    }
    if (lane == 0) lsq_w[warp] = lsq;
    __syncthreads();
    if (threadIdx.x == 0) {
        float a = 0.f;
        for (int w = 0; w < kTopkWarps; ++w) a += lsq_w[w];
        lse_partial[blockIdx.x] = a;
    }
    for (int e = threadIdx.x; e < N; e += blockDim.x) {
        float a = 0.f;
        for (int w = 0; w < kTopkWarps; ++w) a += psum[w * N + e];
        prob_partial[(size_t)blockIdx.x * N + e] = a;
        if (dcount[e]) atomicAdd(&demand[e], dcount[e]);
    }
}

// One balance-loss summand f_e P_e = (demand_e / (T K)) (prob_sum_e / T).
__device__ __forceinline__ float aux_term(int de, float ps, float TKf, float Tf) {
    return ((float)de / TKf) * (ps / Tf);
}

// One KL(u || f) summand in a form whose terms are all >= 0:
//   f h(u / f),  h(r) = r log r - r + 1,
// which adds (f - u) to u log(u / f); those extra pieces sum to zero over the
// experts because sum_e f_e = sum_e u = 1 (every token makes K assignments).
// r - 1 = (T K - N d_e) / (N d_e) is formed from exact integers; for
// |r - 1| < 1/2, h(1 + delta) = delta^2 sum_{n >= 2} (-delta)^(n-2) / (n (n - 1))
// (Taylor series of h at 1, 30 terms by Horner's rule: truncation below 1e-11
// relative) avoids the cancellation of the closed form. An idle expert gives +inf.
__device__ __forceinline__ float kl_summand(int de, long long TK, int N) {
    if (de <= 0) return INFINITY;
    const long long nd = (long long)N * de;
    const float f = (float)de / (float)TK;
    const float delta = (float)(TK - nd) / (float)nd;
    float h;
    if (fabsf(delta) < 0.5f) {
        float acc = 0.f;
#pragma unroll
        for (int n = 31; n >= 2; --n) acc = fmaf(acc, -delta, 1.0f / (float)(n * (n - 1)));
        h = delta * delta * acc;
    } else {
        const float r = (float)TK / (float)nd;
        h = r * logf(r) - r + 1.f;
    }
    return f * h;
}

// Compensated fp32 sum (Neumaier): s + c carries the running total with the
// rounding error of each addition kept in c. fp32 is used because fp64
// arithmetic is slow on this GPU; with the compensation the error stays at a
// few fp32 ulps of the total for the few thousand terms summed here.
struct KSum {
    float s = 0.f, c = 0.f;
    __device__ __forceinline__ void add(float x) {
        const float t = s + x;
        if (!isfinite(t)) {  // an infinite term (idle expert in the KL loss) or NaN: no compensation
            s = t;
            c = 0.f;
            return;
        }
        c += fabsf(s) >= fabsf(x) ? (s - t) + x : (x - t) + s;
        s = t;
    }
    __device__ __forceinline__ void add(const KSum &o) {
        add(o.s);
        add(o.c);
    }
    __device__ __forceinline__ float value() const { return s + c; }
};

__device__ __forceinline__ KSum shfl_xor_ksum(const KSum &v, int o) {
    KSum r;
    r.s = __shfl_xor_sync(0xffffffffu, v.s, o);
    r.c = __shfl_xor_sync(0xffffffffu, v.c, o);
    return r;
}

// Fixed-order block sums of three compensated sums per thread (any blockDim
// <= 1024, a multiple of 32); the results are valid in thread 0.
__device__ __forceinline__ void block_sum3(KSum &a, KSum &b, KSum &c, KSum *scratch /* 3 x 32 */) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        a.add(shfl_xor_ksum(a, o));
        b.add(shfl_xor_ksum(b, o));
        c.add(shfl_xor_ksum(c, o));
    }
    if (lane_id() == 0) {
        scratch[warp_id()] = a;
        scratch[32 + warp_id()] = b;
        scratch[64 + warp_id()] = c;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        a = b = c = KSum();
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
            a.add(scratch[w]);
            b.add(scratch[32 + w]);
            c.add(scratch[64 + w]);
        }
    }
}

// The losses from per-expert totals already in global memory (prob_sum as
// fp32 sums of probabilities, demand as counts) and `rows` per-block partial
// sums of logsumexp^2. Called by every thread of one block.
//   aux    = alpha N sum_e (demand_e / (T K)) (prob_sum_e / T)   (sec. 5.1-5.2)
//   z_loss = beta (1/T) sum_t logsumexp(s_t)^2                     (sec. 5.3)
//   aux_kl = kl_coef sum_e (1/N) log((1/N) / f_e)  (KL balance loss of the
//            CSDN "MoE逐token路由与活跃参数率实战解析" MoELayer listing)
__device__ void block_losses(int N, int T, int K, const int32_t *demand, const float *prob_sum,
                             const float *lse_partial, int rows, float alpha, float beta, float kl_coef,
                             float *aux, float *z_loss, float *aux_kl, KSum *scratch) {
    const long long TK = (long long)T * K;
    const float TKf = (float)TK, Tf = (float)T;
    KSum a_aux, a_kl, a_z;
    for (int e = threadIdx.x; e < N; e += blockDim.x) {
        const int de = __ldcg(demand + e);
        const float pe = __ldcg(prob_sum + e);
        if (aux != nullptr) a_aux.add(aux_term(de, pe, TKf, Tf));
        if (aux_kl != nullptr) a_kl.add(kl_summand(de, TK, N));
    }
    if (z_loss != nullptr)
        for (int r = threadIdx.x; r < rows; r += blockDim.x) a_z.add(__ldcg(lse_partial + r));
    block_sum3(a_aux, a_kl, a_z, scratch);
    if (threadIdx.x == 0) {
        if (aux != nullptr) aux[0] = alpha * (float)N * a_aux.value();
        if (z_loss != nullptr) z_loss[0] = beta * (a_z.value() / (float)T);
        if (aux_kl != nullptr) aux_kl[0] = kl_coef * a_kl.value();
    }
}

// prob_sum[e] = sum of the per-block partial rows, in double, in a fixed
// order. Block b owns experts [32 b, 32 b + 32): thread (x, y) adds rows
// y, y + 32, ... of expert 32 b + x (coalesced across x), then the 32 row
// lanes are added in y order. The last block to finish (counted on *done,
// which the caller zeroes) writes, when asked, the balance loss
//   aux = alpha * N * sum_e (demand[e] / (T K)) * (prob_sum[e] / T)
// (lmnt.cn/news/351908 sec. 5.1-5.2) and the router z-loss
//   z_loss = beta * (1/T) * sum_t logsumexp(s_t)^2       (sec. 5.3)
// from per-block partial sums, in a fixed order; which block is last does
// not change the result.
__global__ void __launch_bounds__(1024)
route_finalize_kernel(const float *__restrict__ prob_partial, const float *__restrict__ lse_partial, int rows,
                      int N, int T, int K, float alpha, float beta, float kl_coef,
                      const int32_t *__restrict__ demand, float *__restrict__ prob_sum, float *__restrict__ aux,
                      float *__restrict__ z_loss, float *__restrict__ aux_kl, unsigned int *__restrict__ done) {
    __shared__ double part[32][33];
    __shared__ bool last;
    const int x = threadIdx.x & 31, y = threadIdx.x >> 5;
    const int e = blockIdx.x * 32 + x;
    double a = 0.0;
    if (e < N) {
#pragma unroll 4
        for (int r = y; r < rows; r += 32) a += (double)prob_partial[(size_t)r * N + e];
    }
    part[y][x] = a;
    __syncthreads();
    if (y == 0 && e < N) {
        double s = 0.0;
        for (int j = 0; j < 32; ++j) s += part[j][x];
        prob_sum[e] = (float)s;
    }
    if (aux == nullptr && z_loss == nullptr && aux_kl == nullptr) return;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) last = atomicAdd(done, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!last) return;
    __threadfence();
    __shared__ KSum scratch[96];
    block_losses(N, T, K, demand, prob_sum, lse_partial, rows, alpha, beta, kl_coef, aux, z_loss, aux_kl, scratch);
}

// Number of blocks of the TopK kernel (general N): a function of T only.
inline int topk_grid(int T) {
    int g = (T + kTopkWarps - 1) / kTopkWarps;
    return g < 1 ? 1 : (g > 256 ? 256 : g);
}

}  // namespace route
}  // namespace moe
