// plan.cuh -- the step between the fused router and the expert GEMMs: from
// the router's per-tile rows (one row of per-expert counts and fixed-point
// sums per 128-token tile) it forms
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
// plan_kernel does this with blocks of 1024 threads for any number of tiles:
// block 0 the dispatch plan and the m-tile lists, block 1 (or block 0 when
// there is no plan to form) the statistics and losses, which no later kernel
// waits for, at the same time; a single-tile batch (decode) does it inside
// the router kernel with the block-level pieces below, which also place its
// assignments.
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

// What the statistics need and where they go (demand and prob_sum required;
// the rest may be null).
struct Stats {
    int T, N, K;
    int route_blocks;            // rows of lse_partial
    const float *lse_partial;    // [route_blocks][route::kPartialStride]
    int32_t *demand;
    float *prob_sum, *aux, *z_loss, *aux_kl, *health, *mean_weight;
    float alpha, beta, kl_coef;
};

// The dispatch plan's outputs (base == nullptr: statistics only).
struct Dispatch {
    int C;
    int32_t *base, *kept, *offsets;
    int tile_rows, raster, max_tiles;  // m-tile list (mtiles == nullptr: none)
    int4 *mtiles;
    int *num_mtiles;
    int32_t *slot_of, *row_token;      // single-tile batches placed by the router itself
    int tile_rows2, raster2;           // a second m-tile list (mtiles2 == nullptr: none)
    int4 *mtiles2;
    int *num_mtiles2;
};

struct Params {
    Stats st;
    Dispatch dp;
    int tiles;                                     // rows of the tile tables
    const int32_t *tile_hist;                      // [tiles][N]
    const unsigned long long *tile_prob, *tile_w;  // [tiles][N]
};

// Pairwise sum over the 32 lanes of a warp (fixed order; valid in every lane).
__device__ __forceinline__ float warp_tree_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// kept[e] = min(demand[e], C) and the expert offsets (exclusive scan; s_off
// in shared memory gets offsets[0..N]). All threads of a block of
// blockDim.x >= N; sc: blockDim.x ints of shared scratch.
__device__ __forceinline__ void expert_offsets(const int *s_dem, int N, int C, int *s_off, int *sc,
                                               int32_t *kept, int32_t *offsets) {
    const int tid = threadIdx.x;
    int v = tid < N ? min(s_dem[tid], C) : 0;
    if (tid < N) kept[tid] = v;
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
        offsets[tid + 1] = v;
    }
    if (tid == 0) {
        s_off[0] = 0;
        offsets[0] = 0;
    }
    __syncthreads();
}

// The losses and health statistics from the per-expert totals s_dem / s_prob
// (shared) and the router blocks' partial sums. kept_rows >= 0 also gives the
// drop rate. All threads of a block of blockDim.x >= max(N, 64); t_aux, t_kl,
// t_var: N floats of shared scratch each.
__device__ __forceinline__ void losses(const Stats &q, const int *s_dem, const float *s_prob, float *t_aux,
                                       float *t_kl, float *t_var, int kept_rows) {
    const int N = q.N, tid = threadIdx.x;
    const float TKf = (float)q.T * (float)q.K, Tf = (float)q.T, inv_n = 1.0f / (float)N;
    if (tid < N) {
        const int dem = s_dem[tid];
        const float f = (float)dem / TKf;
        t_aux[tid] = f * (s_prob[tid] / Tf);
        t_kl[tid] = q.aux_kl != nullptr ? route::kl_summand(dem, (long long)q.T * q.K, N) : 0.f;
        t_var[tid] = (f - inv_n) * (f - inv_n);
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
            if (q.aux != nullptr) q.aux[0] = q.alpha * (float)N * a;
            if (q.aux_kl != nullptr) q.aux_kl[0] = q.kl_coef * k;
            if (q.health != nullptr) {
                q.health[0] = sqrtf(v * inv_n);
                if (kept_rows >= 0) q.health[1] = (float)(q.T * q.K - kept_rows) / TKf;
            }
        }
    } else if (warp == 1) {
        float l = 0.f, en = 0.f, am = 0.f;
        for (int r = lane; r < q.route_blocks; r += 32) {
            l += __ldcg(q.lse_partial + (size_t)r * route::kPartialStride);
            en += __ldcg(q.lse_partial + (size_t)r * route::kPartialStride + 1);
            am = fmaxf(am, __ldcg(q.lse_partial + (size_t)r * route::kPartialStride + 2));
        }
        l = warp_tree_sum(l);
        en = warp_tree_sum(en);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
        if (lane == 0) {
            if (q.z_loss != nullptr) q.z_loss[0] = q.beta * (l / Tf);
            if (q.health != nullptr) {
                q.health[2] = en / Tf;
                q.health[3] = am;
            }
        }
    }
}

// Places the assignments of a batch of T <= blockDim.x tokens in token order
// (the dispatch's position rule: assignment (t, k) to expert e gets position
// p = number of tokens t' < t that chose e, and is kept iff p < C): thread t
// owns token t; bits (blockDim.x / 32 x N words of shared scratch) mark, per
// warp and expert, the warp's tokens that chose it. Writes slot_of, and
// row_token (-1 past offsets[N], up to `rows`). All threads.
__device__ __forceinline__ void assign_tokens(const int32_t *topk_idx, int T, int K, int N, int C, const int *s_off,
                                              unsigned *bits, int32_t *slot_of, int32_t *row_token, int rows) {
    const int tid = threadIdx.x, w = warp_id(), lane = lane_id(), nw = blockDim.x / 32;
    for (int i = tid; i < nw * N; i += blockDim.x) bits[i] = 0u;
    for (int r = s_off[N] + tid; r < rows; r += blockDim.x) row_token[r] = -1;
    __syncthreads();
    if (tid < T)
        for (int k = 0; k < K; ++k) {
            const int e = __ldcg(topk_idx + (size_t)tid * K + k);
            if (e >= 0 && e < N) atomicOr(&bits[w * N + e], 1u << lane);
        }
    __syncthreads();
    const unsigned below = (1u << lane) - 1u;
    for (int k = 0; k < (tid < T ? K : 0); ++k) {
        const int e = __ldcg(topk_idx + (size_t)tid * K + k);
        int slot = -1;
        if (e >= 0 && e < N) {
            int pos = __popc(bits[w * N + e] & below);
            for (int w2 = 0; w2 < w; ++w2) pos += __popc(bits[w2 * N + e]);
            if (pos < C) {
                slot = s_off[e] + pos;
                row_token[slot] = tid;
            }
        } else {
            flag_error(MOE_DEVERR_EXPERT_ID);
        }
        slot_of[(size_t)tid * K + k] = slot;
    }
}

// Blocks of 1024 threads: per-expert totals over the tiles (G lanes, a power
// of two <= 32, share an expert; lane j of the group takes a contiguous run of
// tiles, so the tile order is kept by an exclusive scan across the group);
// then block 0 forms the plan and the m-tile lists, and the last block
// (block 1 of two, or block 0 alone) the statistics and losses.
__global__ void __launch_bounds__(kThreads) plan_kernel(const Params p) {
    __shared__ int s_dem[1024], s_off[1025], sc[1024];
    __shared__ float s_prob[1024], t_aux[1024], t_kl[1024], t_var[1024];
    const int N = p.st.N, tid = threadIdx.x;
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
    const bool plan_here = blockIdx.x == 0 && p.dp.base != nullptr;
    const bool stats_here = blockIdx.x == gridDim.x - 1;
    if (e < N && plan_here) {
        int run = incl - cnt;
        for (int c = c0; c < c1; ++c) {
            const size_t i = (size_t)c * N + e;
            p.dp.base[i] = run;
            run += __ldcg(p.tile_hist + i);
        }
    }
    if (e < N && j == 0) {
        const float prob = __ull2float_rn(pr) * kFixUnit;  // the integer total rounded once, then scaled exactly
        s_dem[e] = dem;
        s_prob[e] = prob;
        if (stats_here) {
            p.st.demand[e] = dem;
            p.st.prob_sum[e] = prob;
            if (p.st.mean_weight != nullptr)
                p.st.mean_weight[e] = dem > 0 ? __ull2float_rn(wr) * kFixUnit / (float)dem : 0.f;
        }
    }
    __syncthreads();
    int kept_rows = -1;
    if (plan_here) {
        expert_offsets(s_dem, N, p.dp.C, s_off, sc, p.dp.kept, p.dp.offsets);
        kept_rows = s_off[N];
        if (p.dp.mtiles != nullptr)
            gg::build_mtiles_block(s_off, N, p.st.T * p.st.K, p.dp.tile_rows, p.dp.raster, p.dp.max_tiles,
                                   p.dp.mtiles, p.dp.num_mtiles, sc);
        __syncthreads();
        if (p.dp.mtiles2 != nullptr)
            gg::build_mtiles_block(s_off, N, p.st.T * p.st.K, p.dp.tile_rows2, p.dp.raster2, p.dp.max_tiles,
                                   p.dp.mtiles2, p.dp.num_mtiles2, sc);
    } else if (p.dp.base != nullptr) {  // rows kept = sum of min(demand, C), an integer sum (any order)
        int v = tid < N ? min(s_dem[tid], p.dp.C) : 0;
        v = __reduce_add_sync(0xffffffffu, v);
        if ((tid & 31) == 0) sc[tid >> 5] = v;
        __syncthreads();
        kept_rows = 0;
        for (int w = 0; w < kThreads / 32; ++w) kept_rows += sc[w];
    }
    if (stats_here) losses(p.st, s_dem, s_prob, t_aux, t_kl, t_var, kept_rows);
}

}  // namespace plan
}  // namespace moe
