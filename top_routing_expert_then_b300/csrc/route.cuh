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
// Small N (<= 16): the whole router in one kernel. A block of 4 warps takes 4
// tokens at a time; warp w owns the 8-element column chunks c with
// (c / 32) % 4 == w, lane j the chunks with c % 32 == j, and accumulates all N
// logits of the 4 tokens over its chunks (W_g is read through L1: it is small
// and shared by every block on the SM). The partial sums meet in shared memory
// and warp 0 adds them in warp order, then runs TopK / softmax for the 4
// tokens (every lane computes the same values; lane k writes rank k).
constexpr int kRouterWarps = 4;
constexpr int kTokensPerBlock = 4;
constexpr int kMaxK = 8;
constexpr int kMaxPartialRows = 1024;

// Blocks of the small-N router: a function of T only, so the partial
// probability sums (and hence prob_sum) are identical on every device.
inline int small_router_grid(int T) {
    int g = (T + kTokensPerBlock - 1) / kTokensPerBlock;
    return g < 1 ? 1 : (g > kMaxPartialRows ? kMaxPartialRows : g);
}

template <int NMAX>
__global__ void __launch_bounds__(kRouterWarps * 32)
router_smallN_kernel(const uint16_t *__restrict__ x, const uint16_t *__restrict__ Wg,
                     const float *__restrict__ sel_bias, int T, int d, int N, int K,
                     int32_t *__restrict__ topk_idx, float *__restrict__ topk_w,
                     int32_t *__restrict__ demand, float *__restrict__ prob_partial) {
    __shared__ float red[kRouterWarps][kTokensPerBlock][NMAX];
    __shared__ int dcount[NMAX];
    const int chunks = d >> 3;
    const int lane = lane_id();
    const int warp = warp_id();
    if (threadIdx.x < NMAX) dcount[threadIdx.x] = 0;
    float bias[NMAX];
    float pacc[NMAX];
#pragma unroll
    for (int e = 0; e < NMAX; ++e) {
        bias[e] = (sel_bias != nullptr && e < N) ? sel_bias[e] : 0.f;
        pacc[e] = 0.f;
    }
    const uint4 *wg = reinterpret_cast<const uint4 *>(Wg);

    for (int t0 = blockIdx.x * kTokensPerBlock; t0 < T; t0 += gridDim.x * kTokensPerBlock) {
        float acc[kTokensPerBlock][NMAX];
#pragma unroll
        for (int i = 0; i < kTokensPerBlock; ++i)
#pragma unroll
            for (int e = 0; e < NMAX; ++e) acc[i][e] = 0.f;
#pragma unroll 2
        for (int c = warp * 32 + lane; c < chunks; c += kRouterWarps * 32) {
            uint4 xv[kTokensPerBlock];
#pragma unroll
            for (int i = 0; i < kTokensPerBlock; ++i)
                xv[i] = (t0 + i < T) ? __ldg(reinterpret_cast<const uint4 *>(x + (size_t)(t0 + i) * d) + c)
                                     : make_uint4(0u, 0u, 0u, 0u);
            uint4 wv[NMAX];
#pragma unroll
            for (int e = 0; e < NMAX; ++e) wv[e] = (e < N) ? __ldg(wg + (size_t)e * chunks + c) : make_uint4(0u, 0u, 0u, 0u);
            float xf[kTokensPerBlock][8];
#pragma unroll
            for (int i = 0; i < kTokensPerBlock; ++i) {
                unpack_bf16x2(xv[i].x, xf[i][0], xf[i][1]);
                unpack_bf16x2(xv[i].y, xf[i][2], xf[i][3]);
                unpack_bf16x2(xv[i].z, xf[i][4], xf[i][5]);
                unpack_bf16x2(xv[i].w, xf[i][6], xf[i][7]);
            }
#pragma unroll
            for (int e = 0; e < NMAX; ++e) {
                float wf[8];
                unpack_bf16x2(wv[e].x, wf[0], wf[1]);
                unpack_bf16x2(wv[e].y, wf[2], wf[3]);
                unpack_bf16x2(wv[e].z, wf[4], wf[5]);
                unpack_bf16x2(wv[e].w, wf[6], wf[7]);
#pragma unroll
                for (int i = 0; i < kTokensPerBlock; ++i)
#pragma unroll
                    for (int j = 0; j < 8; ++j) acc[i][e] = fmaf(xf[i][j], wf[j], acc[i][e]);
            }
        }
#pragma unroll
        for (int i = 0; i < kTokensPerBlock; ++i)
#pragma unroll
            for (int e = 0; e < NMAX; ++e) {
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) acc[i][e] += __shfl_xor_sync(0xffffffffu, acc[i][e], o);
            }
        if (lane == 0) {
#pragma unroll
            for (int i = 0; i < kTokensPerBlock; ++i)
#pragma unroll
                for (int e = 0; e < NMAX; ++e) red[warp][i][e] = acc[i][e];
        }
        __syncthreads();
        if (warp == 0) {
#pragma unroll
            for (int i = 0; i < kTokensPerBlock; ++i) {
                const int t = t0 + i;
                if (t >= T) break;  // warp-uniform
                float s[NMAX];
#pragma unroll
                for (int e = 0; e < NMAX; ++e) {
                    float a = red[0][i][e];
#pragma unroll
                    for (int w = 1; w < kRouterWarps; ++w) a += red[w][i][e];
                    s[e] = a;
                }
                // softmax over all N unbiased logits (balance-loss statistic)
                float m = -INFINITY;
#pragma unroll
                for (int e = 0; e < NMAX; ++e)
                    if (e < N) m = fmaxf(m, s[e]);
                float ex[NMAX];
                float z = 0.f;
#pragma unroll
                for (int e = 0; e < NMAX; ++e) {
                    ex[e] = (e < N) ? expf(s[e] - m) : 0.f;
                    z += ex[e];
                }
                const float inv_z = 1.f / z;
#pragma unroll
                for (int e = 0; e < NMAX; ++e) pacc[e] += ex[e] * inv_z;
                // TopK on u = s + b: larger u first, equal u -> smaller id first
                unsigned taken = 0u;
                int sel_e[kMaxK];
                float sel_s[kMaxK];
#pragma unroll
                for (int k = 0; k < kMaxK; ++k) {
                    sel_e[k] = 0;
                    sel_s[k] = 0.f;
                    if (k < K) {
                        float bu = -INFINITY, bs = 0.f;
                        int be = -1;
#pragma unroll
                        for (int e = 0; e < NMAX; ++e) {
                            const float u = s[e] + bias[e];
                            if (e < N && !((taken >> e) & 1u) && (be < 0 || u > bu)) {
                                bu = u;
                                be = e;
                                bs = s[e];
                            }
                        }
                        sel_e[k] = be;
                        sel_s[k] = bs;
                        taken |= 1u << be;
                    }
                }
                float mk = -INFINITY;
#pragma unroll
                for (int k = 0; k < kMaxK; ++k)
                    if (k < K) mk = fmaxf(mk, sel_s[k]);
                float num[kMaxK];
                float den = 0.f;
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
                        atomicAdd(&dcount[sel_e[k]], 1);
                    }
                }
            }
        }
        __syncthreads();
    }
    if (warp == 0 && lane < N) {
        float a = 0.f;
#pragma unroll
        for (int e = 0; e < NMAX; ++e)
            if (e == lane) a = pacc[e];
        prob_partial[(size_t)blockIdx.x * N + lane] = a;
        if (dcount[lane]) atomicAdd(&demand[lane], dcount[lane]);
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
// TopK then softmax, one warp per token. Lane l holds the logits of experts
// l, l+32, ... (LPL of them). K rounds of a warp arg-max on (u desc, id asc)
// pick the experts; the softmax runs over their unbiased logits. The full-N
// softmax probabilities are accumulated per lane (each lane owns its experts),
// reduced over the block's warps in a fixed order and written as one partial
// row per block: no floating-point atomics, so results are run-to-run stable.
constexpr int kTopkWarps = 8;

template <int LPL>
__global__ void __launch_bounds__(kTopkWarps * 32)
topk_softmax_kernel(const float *__restrict__ logits, const float *__restrict__ sel_bias, int T,
                    int N, int K, int32_t *__restrict__ topk_idx, float *__restrict__ topk_w,
                    int32_t *__restrict__ demand, float *__restrict__ prob_partial) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
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

    for (int t = blockIdx.x * kTopkWarps + warp; t < T; t += gridDim.x * kTopkWarps) {
        float s[LPL];
        float m = -INFINITY;
#pragma unroll
        for (int i = 0; i < LPL; ++i) {
            int e = lane + 32 * i;
            s[i] = (e < N) ? logits[(size_t)t * N + e] : -INFINITY;
            m = fmaxf(m, s[i]);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float ex[LPL];
        float z = 0.f;
#pragma unroll
        for (int i = 0; i < LPL; ++i) {
            ex[i] = (lane + 32 * i < N) ? __expf(s[i] - m) : 0.f;
            z += ex[i];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
        const float inv_z = 1.f / z;
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
                atomicAdd(&dcount[sel_e[k]], 1);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < LPL; ++i) {
        int e = lane + 32 * i;
        if (e < N) psum[warp * N + e] = pacc[i];
    }
    __syncthreads();
    for (int e = threadIdx.x; e < N; e += blockDim.x) {
        float a = 0.f;
        for (int w = 0; w < kTopkWarps; ++w) a += psum[w * N + e];
        prob_partial[(size_t)blockIdx.x * N + e] = a;
        if (dcount[e]) atomicAdd(&demand[e], dcount[e]);
    }
}

// One block of 1024 threads. prob_sum[e] = sum of the per-block partial rows
// in double, each expert reduced by one warp in a fixed lane/shuffle order.
// With aux != nullptr it also writes the balance loss
//   aux = alpha * N * sum_e (demand[e] / (T K)) * (prob_sum[e] / T)
// (lmnt.cn/news/351908 sec. 5.1-5.2) from the same fp32 prob_sum values.
__global__ void __launch_bounds__(1024)
route_finalize_kernel(const float *__restrict__ prob_partial, int rows, int N, int T, int K, float alpha,
                      const int32_t *__restrict__ demand, float *__restrict__ prob_sum, float *__restrict__ aux) {
    const int lane = lane_id(), warp = warp_id();
    const int warps = blockDim.x >> 5;
    for (int e = warp; e < N; e += warps) {
        double a = 0.0;
        for (int r = lane; r < rows; r += 32) a += (double)prob_partial[(size_t)r * N + e];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
        if (lane == 0) prob_sum[e] = (float)a;
    }
    if (aux == nullptr) return;
    __syncthreads();
    if (warp == 0) {
        double s = 0.0;
        for (int e = lane; e < N; e += 32)
            s += ((double)demand[e] / ((double)T * (double)K)) * ((double)prob_sum[e] / (double)T);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) aux[0] = (float)((double)alpha * (double)N * s);
    }
}

// Number of blocks of the TopK kernel (general N): a function of T only.
inline int topk_grid(int T) {
    int g = (T + kTopkWarps - 1) / kTopkWarps;
    return g < 1 ? 1 : (g > kMaxPartialRows ? kMaxPartialRows : g);
}

}  // namespace route
}  // namespace moe
