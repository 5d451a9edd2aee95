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
constexpr int kMaxK = 8;
constexpr int kMaxPartialRows = 1024;

// Fixed-point unit of the per-expert sums of probabilities and routing
// weights (values in [0, 1] rounded to this grid, then summed as integers).
constexpr float kFixUnit = 1.0f / 2147483648.0f;  // 2^-31

// Per-block partial statistics: [rows][4] = sum of logsumexp^2, sum of
// routing entropies, max |logit|, unused.
constexpr int kPartialStride = 4;


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
                    float *__restrict__ lse_partial, unsigned long long *__restrict__ w_acc) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    __shared__ float lsq_w[kTopkWarps], ent_w[kTopkWarps], amax_w[kTopkWarps];
    unsigned long long *wacc = reinterpret_cast<unsigned long long *>(smem_raw);  // [N]
    float *psum = reinterpret_cast<float *>(wacc + N);                       // [warps][N]
    int *dcount = reinterpret_cast<int *>(psum + kTopkWarps * N);            // [N]
    for (int e = threadIdx.x; e < N; e += blockDim.x) {
        dcount[e] = 0;
        wacc[e] = 0ull;
    }
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

    float lsq = 0.f;   // sum over this warp's tokens of logsumexp(s_t)^2 (z-loss)
    float ent = 0.f;   // sum of routing entropies
    float amax = 0.f;  // max |logit|
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
        // entropy lse - sum_e p_e s_e, and the logit range
        float ps = 0.f, am = 0.f;
#pragma unroll
        for (int i = 0; i < LPL; ++i)
            if (lane + 32 * i < N) {
                ps += ex[i] * s[i];
                am = fmaxf(am, fabsf(s[i]));
            }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            ps += __shfl_xor_sync(0xffffffffu, ps, o);
            am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
        }
        ent += lse - ps * inv_z;
        amax = fmaxf(amax, am);
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
                if ((unsigned)sel_e[k] < (unsigned)N) {
                    atomicAdd(&dcount[sel_e[k]], 1);
                    atomicAdd(&wacc[sel_e[k]], (unsigned long long)__float2uint_rn(num[k] / den * 2147483648.0f));
                }
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
    if (lane == 0) {
        lsq_w[warp] = lsq;
        ent_w[warp] = ent;
        amax_w[warp] = amax;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float a = 0.f, b = 0.f, c = 0.f;
        for (int w = 0; w < kTopkWarps; ++w) {
            a += lsq_w[w];
            b += ent_w[w];
            c = fmaxf(c, amax_w[w]);
        }
        lse_partial[(size_t)blockIdx.x * kPartialStride] = a;
        lse_partial[(size_t)blockIdx.x * kPartialStride + 1] = b;
        lse_partial[(size_t)blockIdx.x * kPartialStride + 2] = c;
    }
    for (int e = threadIdx.x; e < N; e += blockDim.x)
        if (wacc[e] != 0ull) atomicAdd(w_acc + e, wacc[e]);
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

// Fixed-order block sums of NV compensated sums per thread (any blockDim <=
// 1024, a multiple of 32); the results are valid in thread 0.
template <int NV>
__device__ __forceinline__ void block_sums(KSum (&v)[NV], KSum *scratch /* NV x 32 */) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int i = 0; i < NV; ++i) v[i].add(shfl_xor_ksum(v[i], o));
    if (lane_id() == 0)
#pragma unroll
        for (int i = 0; i < NV; ++i) scratch[32 * i + warp_id()] = v[i];
    __syncthreads();
    if (threadIdx.x == 0) {
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            v[i] = KSum();
            for (int w = 0; w < (int)(blockDim.x >> 5); ++w) v[i].add(scratch[32 * i + w]);
        }
    }
}

// Block maximum (valid in thread 0).
__device__ __forceinline__ float block_max(float v, float *scratch /* 32 */) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    __syncthreads();
    if (lane_id() == 0) scratch[warp_id()] = v;
    __syncthreads();
    if (threadIdx.x == 0)
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) v = fmaxf(v, scratch[w]);
    return v;
}

// The losses and the router health statistics from per-expert totals in
// global memory (prob_sum as fp32 sums of probabilities, demand as counts,
// w_acc as fixed-point sums of routing weights) and `rows` per-block partials.
// Called by every thread of one block; every output may be null.
//   aux    = alpha N sum_e (demand_e / (T K)) (prob_sum_e / T)   (lmnt.cn/news/351908 sec. 5.1-5.2)
//   z_loss = beta (1/T) sum_t logsumexp(s_t)^2                     (sec. 5.3)
//   aux_kl = kl_coef sum_e (1/N) log((1/N) / f_e)  (KL balance loss of the
//            CSDN "MoE逐token路由与活跃参数率实战解析" MoELayer listing)
//   health[0] = population std over experts of f_e = demand_e / (T K)
//               (the CSDN page's sec. 3.3 expert_util_std)
//   health[2] = mean routing entropy (nats) of softmax_N(s_t),
//   health[3] = max |logit|  (lmnt sec. 8.2 / 9.3 routing monitors;
//               health[1], the drop rate, is written by the dispatch)
//   mean_weight[e] = mean routing weight of the assignments to e (0 if none)
// With prob_acc / dem_acc given (the fused router's fixed-point totals),
// prob_sum[e] = prob_acc[e] * prob_unit and demand[e] = dem_acc[e] are
// computed here and written out; otherwise demand and prob_sum are read.
// The per-block partial rows are loaded first, so that their loads and the
// per-expert ones are in flight together.
__device__ void block_losses(int N, int T, int K, int32_t *demand, float *prob_sum, const float *partials,
                             int rows, const unsigned long long *w_acc, float alpha, float beta, float kl_coef,
                             float *aux, float *z_loss, float *aux_kl, float *health, float *mean_weight,
                             KSum *scratch /* 5 x 32 */, float *mscratch /* 32 */,
                             const unsigned long long *prob_acc = nullptr, const int32_t *dem_acc = nullptr,
                             float prob_unit = 0.f) {
    const long long TK = (long long)T * K;
    const float TKf = (float)TK, Tf = (float)T, inv_n = 1.0f / (float)N;
    KSum v[5];  // aux, kl, z, entropy, load variance
    float amax = 0.f;
    for (int r = threadIdx.x; r < rows; r += blockDim.x) {
        v[2].add(__ldcg(partials + (size_t)r * kPartialStride));
        v[3].add(__ldcg(partials + (size_t)r * kPartialStride + 1));
        amax = fmaxf(amax, __ldcg(partials + (size_t)r * kPartialStride + 2));
    }
    for (int e = threadIdx.x; e < N; e += blockDim.x) {
        int de;
        float pe;
        if (prob_acc != nullptr) {
            pe = __ull2float_rn(__ldcg(prob_acc + e)) * prob_unit;
            de = __ldcg(dem_acc + e);
            prob_sum[e] = pe;
            demand[e] = de;
        } else {
            de = __ldcg(demand + e);
            pe = __ldcg(prob_sum + e);
        }
        v[0].add(aux_term(de, pe, TKf, Tf));
        if (aux_kl != nullptr) v[1].add(kl_summand(de, TK, N));
        const float df = (float)de / TKf - inv_n;
        v[4].add(df * df);
        if (mean_weight != nullptr)
            mean_weight[e] = de > 0 ? __ull2float_rn(__ldcg(w_acc + e)) * kFixUnit / (float)de : 0.f;
    }
    block_sums<5>(v, scratch);
    amax = block_max(amax, mscratch);
    if (threadIdx.x == 0) {
        if (aux != nullptr) aux[0] = alpha * (float)N * v[0].value();
        if (z_loss != nullptr) z_loss[0] = beta * (v[2].value() / Tf);
        if (aux_kl != nullptr) aux_kl[0] = kl_coef * v[1].value();
        if (health != nullptr) {
            health[0] = sqrtf(v[4].value() * inv_n);
            health[2] = v[3].value() / Tf;
            health[3] = amax;
        }
    }
}

// prob_sum[e] = sum of the per-block partial rows, in double, in a fixed
// order. Block b owns experts [32 b, 32 b + 32): thread (x, y) adds rows
// y, y + 32, ... of expert 32 b + x (coalesced across x), then the 32 row
// lanes are added in y order. The last block to finish (counted on *done,
// which the caller zeroes) writes, when asked, the router health statistics,
// the balance loss
//   aux = alpha * N * sum_e (demand[e] / (T K)) * (prob_sum[e] / T)
// (lmnt.cn/news/351908 sec. 5.1-5.2) and the router z-loss
//   z_loss = beta * (1/T) * sum_t logsumexp(s_t)^2       (sec. 5.3)
// from per-block partial sums, in a fixed order; which block is last does
// not change the result.
__global__ void __launch_bounds__(1024)
route_finalize_kernel(const float *__restrict__ prob_partial, const float *__restrict__ lse_partial, int rows,
                      int N, int T, int K, float alpha, float beta, float kl_coef,
                      const int32_t *__restrict__ demand, float *__restrict__ prob_sum, float *__restrict__ aux,
                      float *__restrict__ z_loss, float *__restrict__ aux_kl,
                      const unsigned long long *__restrict__ w_acc, float *__restrict__ health,
                      float *__restrict__ mean_weight, unsigned int *__restrict__ done) {
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
    if (aux == nullptr && z_loss == nullptr && aux_kl == nullptr && health == nullptr && mean_weight == nullptr)
        return;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) last = atomicAdd(done, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!last) return;
    __threadfence();
    __shared__ KSum scratch[5 * 32];
    __shared__ float mscratch[32];
    block_losses(N, T, K, const_cast<int32_t *>(demand), prob_sum, lse_partial, rows, w_acc, alpha, beta, kl_coef, aux, z_loss, aux_kl,
                 health, mean_weight, scratch, mscratch);
}

// Number of blocks of the TopK kernel (general N): a function of T only.
inline int topk_grid(int T) {
    int g = (T + kTopkWarps - 1) / kTopkWarps;
    return g < 1 ? 1 : (g > 256 ? 256 : g);
}

}  // namespace route
}  // namespace moe
