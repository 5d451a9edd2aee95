// plan.cuh -- the single-block step between the fused router and the
// dispatch's assign kernel: it turns the router's per-tile rows (one row of
// per-expert counts and fixed-point sums per 128-token tile) into
//   the dispatch plan  (lmnt.cn/news/351908 sec. 3.1, 3.3)
//     base[c][e]  = assignments to e in tiles before c (exclusive prefix),
//     demand[e]   = all assignments to e, kept[e] = min(demand[e], C),
//     offsets     = exclusive prefix of kept (offsets[N] = kept rows R),
//     the grouped GEMMs' m-tile list over those blocks;
//   the routing statistics and losses  (sec. 5.1-5.3)
//     prob_sum[e] = sum_t softmax_N(s_t)[e],
//     aux    = alpha N sum_e (demand_e / (T K)) (prob_sum_e / T),
//     z_loss = beta (1/T) sum_t logsumexp(s_t)^2,
//     aux_kl = kl_coef sum_e (1/N) log((1/N) / f_e), f_e = demand_e / (T K)
//              (the CSDN page's MoELayer KL balance loss; +inf for an idle expert),
//     health = [std_e f_e, drop rate, mean routing entropy, max |logit|],
//     mean_weight[e] = mean routing weight of the assignments to e.
// Every sum runs in a fixed order, so results do not depend on scheduling:
// integers for the counts and the fixed-point probability and weight sums;
// fp32 for the few hundred loss terms, each a non-negative quantity added in a
// pairwise tree (error about log2(terms) fp32 ulps of the total). fp64 is
// avoided: on this GPU its rate is a small fraction of fp32's, and a block of
// 1024 threads doing a few fp64 reductions took tens of microseconds. The code
// is kept short on purpose: it runs once per layer with a cold instruction cache.
#pragma once

#include "common.cuh"
#include "grouped_gemm.cuh"
#include "route.cuh"

namespace moe {
namespace plan {

constexpr int kThreads = 1024;
constexpr float kFixUnit = 1.0f / 2147483648.0f;  // 2^-31, the routers' fixed-point unit

struct Params {
    int T, N, K, C;
    int tiles;                        // rows of the tile tables (128-token tiles)
    int route_blocks;                 // rows of lse_partial
    const int32_t *tile_hist;         // [tiles][N]
    const unsigned long long *tile_prob, *tile_w;  // [tiles][N]
    const float *lse_partial;         // [route_blocks][route::kPartialStride]
    // dispatch plan (base == nullptr: statistics only)
    int32_t *base, *kept, *offsets;
    // m-tile list (mtiles == nullptr: none)
    int tile_rows, raster, max_tiles;
    int4 *mtiles;
    int *num_mtiles;
    // statistics (demand and prob_sum required; the rest may be null)
    int32_t *demand;
    float *prob_sum, *aux, *z_loss, *aux_kl, *health, *mean_weight;
    float alpha, beta, kl_coef;
};

// Pairwise sum over the 32 lanes of a warp (fixed order; valid in every lane).
__device__ __forceinline__ float warp_tree_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__global__ void __launch_bounds__(kThreads) plan_kernel(const Params p) {
    __shared__ int s_kept[1024];
    __shared__ int s_off[1025];
    __shared__ int sc[1024];
    __shared__ float t_aux[1024], t_kl[1024], t_var[1024];  // per-expert loss terms
    const int N = p.N, tid = threadIdx.x;

    // ---- per expert: counts and sums over the tiles. G lanes (a power of two
    // <= 32) share an expert; lane j of the group takes a contiguous run of
    // tiles, so the tile order is kept by an exclusive scan across the group.
    int G = 32;
    while (G > 1 && G * N > kThreads) G >>= 1;
    const int e = tid / G, j = tid % G;
    const int per = (p.tiles + G - 1) / G;
    const int c0 = min(p.tiles, j * per), c1 = min(p.tiles, c0 + per);
    int cnt = 0;
    unsigned long long pr = 0ull, wr = 0ull;
    if (e < N)
        for (int c = c0; c < c1; ++c) {
            const size_t i = (size_t)c * N + e;
            cnt += __ldcg(p.tile_hist + i);
            pr += __ldcg(p.tile_prob + i);
            wr += __ldcg(p.tile_w + i);
        }
    int incl = cnt;
    for (int o = 1; o < G; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o, G);
        if (j >= o) incl += t;
    }
    for (int o = G / 2; o > 0; o >>= 1) {
        pr += __shfl_xor_sync(0xffffffffu, pr, o, G);
        wr += __shfl_xor_sync(0xffffffffu, wr, o, G);
    }
    const int dem = __shfl_sync(0xffffffffu, incl, G - 1, G);
    if (e < N && p.base != nullptr) {
        int run = incl - cnt;
        for (int c = c0; c < c1; ++c) {
            const size_t i = (size_t)c * N + e;
            p.base[i] = run;
            run += __ldcg(p.tile_hist + i);
        }
    }
    const float prob = __ull2float_rn(pr) * kFixUnit;  // the integer total rounded once, then scaled exactly
    if (e < N && j == 0) {
        p.demand[e] = dem;
        p.prob_sum[e] = prob;
        if (p.mean_weight != nullptr) p.mean_weight[e] = dem > 0 ? __ull2float_rn(wr) * kFixUnit / (float)dem : 0.f;
    }

    // ---- kept rows and the expert offsets (exclusive scan over the experts)
    const bool lead = e < N && j == 0;
    if (p.base != nullptr) {
        if (tid < N) s_kept[tid] = 0;
        __syncthreads();
        if (lead) s_kept[e] = min(dem, p.C);
        __syncthreads();
        int v = tid < N ? s_kept[tid] : 0;
        sc[tid] = v;
        __syncthreads();
        for (int o = 1; o < N; o <<= 1) {
            const int add = tid >= o ? sc[tid - o] : 0;
            __syncthreads();
            sc[tid] = v = v + add;
            __syncthreads();
        }
        if (tid < N) {
            s_off[tid + 1] = v;
            p.kept[tid] = s_kept[tid];
            p.offsets[tid + 1] = v;
        }
        if (tid == 0) {
            s_off[0] = 0;
            p.offsets[0] = 0;
        }
        __syncthreads();
        if (p.mtiles != nullptr)
            gg::build_mtiles_block(s_off, N, p.T * p.K, p.tile_rows, p.raster, p.max_tiles, p.mtiles, p.num_mtiles,
                                   sc);
    }

    // ---- losses and health: per-expert terms, then warp 0 adds the expert
    // terms and warp 1 the router blocks' partial sums, each in a fixed order
    const float TKf = (float)p.T * (float)p.K, Tf = (float)p.T, inv_n = 1.0f / (float)N;
    if (lead) {
        const float f = (float)dem / TKf;
        t_aux[e] = f * (prob / Tf);
        t_kl[e] = p.aux_kl != nullptr ? route::kl_summand(dem, (long long)p.T * p.K, N) : 0.f;
        t_var[e] = (f - inv_n) * (f - inv_n);
    }
    __syncthreads();
    const int warp = warp_id(), lane = lane_id();
    if (warp == 0) {
        float a = 0.f, k = 0.f, v = 0.f;
        for (int i = lane; i < N; i += 32) {
            a += t_aux[i];
            k += t_kl[i];
            v += t_var[i];
        }
        a = warp_tree_sum(a);
        k = warp_tree_sum(k);
        v = warp_tree_sum(v);
        if (lane == 0) {
            if (p.aux != nullptr) p.aux[0] = p.alpha * (float)N * a;
            if (p.aux_kl != nullptr) p.aux_kl[0] = p.kl_coef * k;
            if (p.health != nullptr) {
                p.health[0] = sqrtf(v * inv_n);
                if (p.base != nullptr) p.health[1] = (float)(p.T * p.K - s_off[N]) / TKf;
            }
        }
    } else if (warp == 1) {
        float l = 0.f, en = 0.f, am = 0.f;
        for (int r = lane; r < p.route_blocks; r += 32) {
            l += __ldcg(p.lse_partial + (size_t)r * route::kPartialStride);
            en += __ldcg(p.lse_partial + (size_t)r * route::kPartialStride + 1);
            am = fmaxf(am, __ldcg(p.lse_partial + (size_t)r * route::kPartialStride + 2));
        }
        l = warp_tree_sum(l);
        en = warp_tree_sum(en);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
        if (lane == 0) {
            if (p.z_loss != nullptr) p.z_loss[0] = p.beta * (l / Tf);
            if (p.health != nullptr) {
                p.health[2] = en / Tf;
                p.health[3] = am;
            }
        }
    }
}

}  // namespace plan
}  // namespace moe
