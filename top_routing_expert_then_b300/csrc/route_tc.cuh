// route_tc.cuh -- the whole router for up to 256 experts in one kernel, with
// the gate contraction on the tensor cores:
//   s = W_g x                      (lmnt.cn/news/351908 sec. 2.1)
//   TopK over s + b, then softmax over the K kept unbiased logits
//   demand[e], sum_t softmax_N(s_t)[e], sum_t logsumexp(s_t)^2   (sec. 5.2-5.3)
// and per-tile rows of the statistics from which the plan kernel forms the
// balance loss, the router z-loss and the KL(uniform || f) loss variant.
//
// Work split. A tile is 128 tokens. The d_model reduction of one tile is split
// over a cluster of S CTAs (S in {1, 2, 4, 8}, chosen from T and d_model only,
// so results do not depend on the device). CTA r of the cluster:
//   warp 0     TMA producer (one lane): x tile 128 x 64 and W_g tile Npad x 64
//              (rows past N and tokens past T read as zeros), 128-byte swizzle
//   warp 1     TMEM allocator + MMA issuer (one lane): tcgen05.mma kind::f16,
//              M = 128, N = Npad (N rounded up to 16), fp32 accumulator in TMEM
//   warps 4-7  copy the partial logits TMEM -> shared memory, [expert][token]
//              with a padded stride, over the freed operand ring
// After a cluster barrier CTA r owns the tokens [r * 128 / S, (r + 1) * 128 / S)
// of the tile: all 256 threads add the S CTAs' partial logits of those tokens
// (16-byte loads from distributed shared memory, in CTA-rank order) into a
// local buffer; a second cluster barrier releases the peers' buffers; then
// tokens are routed by groups of G = max(2 S, N / 32) lanes, one token per
// group, lane g holding experts g, g + G, ... (all groups of the CTA in one
// pass when the lanes hold at most 32 experts each).
//
// On the 1/64 input grid every partial sum is an exact fp32 multiple of 2^-12,
// so logits, TopK and dispatch decisions are independent of the split.
//
// Statistics without floating-point atomics: per-expert probability sums are
// accumulated as unsigned 64-bit fixed point (2^-31 units; each fp32
// probability rounds to that grid with a 32-bit conversion, then integer
// additions in any order give the same total), demand as integers. The CTAs
// of a cluster add theirs into one row per 128-token tile (the dispatch's
// per-chunk histogram is that row's counts); a single-block plan kernel
// (dispatch.cuh) reduces the rows into demand, prob_sum and the losses.
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "grouped_gemm.cuh"
#include "plan.cuh"
#include "route.cuh"

namespace moe {
namespace rtc {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTile = 128;                 // tokens per tile (MMA M)
constexpr int kBK = 64;                    // d_model columns per stage (one 128-byte swizzle row)
constexpr int kXBytes = kTile * kBK * 2;   // 16 KB
constexpr int kMaxSplits = 8;
constexpr int kMaxStages = 12;
constexpr int kMaxN = 256;
constexpr int kRefSMs = 148;               // the split choice assumes one wave on 148 SMs
constexpr float kProbScale = 2147483648.0f;          // 2^31
constexpr float kProbUnit = 1.0f / 2147483648.0f;    // 2^-31
constexpr size_t kMaxSmem = 214 * 1024;  // + the static block below stays within 227 KB

// Partial-logit buffer [expert][token]: with one split the routing reads it
// directly (odd stride: conflict-free across experts); with several, rows are
// 16-byte aligned for the peers' vector loads.
__host__ __device__ constexpr int pstride(int S) { return S == 1 ? kTile + 1 : kTile + 4; }
// Local buffer of the summed logits of a CTA's own tokens (S > 1), odd stride.
__host__ __device__ constexpr int lstride(int S) { return kTile / S + 1; }
// Lanes that route one token together: enough groups for the CTA's 128 / S
// tokens in one pass of 256 threads, and at most 32 experts per lane.
__host__ __device__ constexpr int route_group(int LPL, int S) {
    return (2 * S > LPL ? 2 * S : LPL) > 32 ? 32 : (2 * S > LPL ? 2 * S : LPL);
}

struct Params {
    int T, d, N, Npad, K, stages;
    uint32_t idesc, tmem_cols;
    uint32_t l_offset;             // bytes from the aligned dynamic shared base to the local buffer
    const float *sel_bias;
    int32_t *topk_idx;
    float *topk_w;
    // per 128-token tile (row = tile, the S CTAs of its cluster added up in rank
    // order; every row is written, nothing needs zeroing beforehand):
    int32_t *tile_hist;             // [tiles][N] assignments to e among the tile's tokens
    unsigned long long *tile_prob;  // [tiles][N] sum of softmax_N(s_t)[e], 2^-31 units
    unsigned long long *tile_w;     // [tiles][N] sum of the routing weights given to e, 2^-31 units
    float *lse_partial;             // [gridDim.x][4] per-CTA sums of logsumexp^2 and entropy, max |logit|
    // a single-tile batch (T <= 128) with fuse_plan: CTA rank 0 also forms the
    // statistics, the dispatch plan and the m-tile list and places the
    // assignments (slot_of, row_token), so no plan or assign kernel follows
    int fuse_plan;
    plan::Stats st;
    plan::Dispatch dp;
};

struct Shared {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t acc_full;
    uint64_t drain;
    uint32_t tmem_base;
    volatile int abort_flag;
    float lsq_w[kWarps], ent_w[kWarps], amax_w[kWarps];
    float bias[kMaxN];
    int dcount[kMaxN];
    unsigned long long pacc[kMaxN];
    unsigned long long wacc[kMaxN];
};

// Tiles, splits and shared memory of a launch: functions of (T, d, N) only.
inline int num_tiles(int T) { return (T + kTile - 1) / kTile; }
inline int splits(int T, int d) {
    const int tiles = num_tiles(T), kb = d / kBK;
    int s = kMaxSplits;
    while (s > 1 && ((long long)tiles * s > kRefSMs || s > kb)) s >>= 1;
    return s;
}
inline int npad(int N) { return (N + 15) / 16 * 16; }
inline uint32_t tmem_cols(int N) {
    const int np = npad(N);
    uint32_t c = 32;
    while ((int)c < np) c <<= 1;
    return c;
}
inline size_t stage_bytes(int N) { return (size_t)kXBytes + (size_t)npad(N) * kBK * 2; }
inline size_t align16(size_t v) { return (v + 15) & ~(size_t)15; }
inline size_t l_offset(int T, int d, int N, int stages) {
    const int S = splits(T, d);
    const size_t ring = (size_t)stages * stage_bytes(N);
    const size_t pbuf = (size_t)N * pstride(S) * sizeof(float);
    return align16(ring > pbuf ? ring : pbuf);
}
inline size_t l_bytes(int T, int d, int N) {
    const int S = splits(T, d);
    return S == 1 ? 0 : (size_t)N * lstride(S) * sizeof(float);
}
inline size_t smem_for(int T, int d, int N, int stages) {
    return l_offset(T, d, N, stages) + l_bytes(T, d, N) + 1024;  // + alignment slack
}
// Operand ring: about 184 KB in flight when one wave covers the grid, 96 KB
// (two CTAs per SM) otherwise, within the shared-memory limit.
inline int stages(int T, int d, int N) {
    const size_t sb = stage_bytes(N);
    const bool one_wave = (long long)num_tiles(T) * splits(T, d) <= kRefSMs;
    const size_t budget = one_wave ? 184 * 1024 : 96 * 1024;
    int s = (int)(budget / sb);
    if (s > kMaxStages) s = kMaxStages;
    if (s < 2) s = 2;
    while (s > 2 && smem_for(T, d, N, s) > kMaxSmem) --s;
    return s;
}
inline size_t smem_bytes(int T, int d, int N) { return smem_for(T, d, N, stages(T, d, N)); }
inline uint32_t idesc(int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(npad(N) >> 3) << 17) | ((uint32_t)(kTile >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16_id(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(id), "r"(acc)
        : "memory");
}

__device__ __forceinline__ uint32_t ld_dsmem_u32(uint32_t cluster_addr) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(cluster_addr) : "memory");
    return v;
}
__device__ __forceinline__ unsigned long long ld_dsmem_u64(uint32_t cluster_addr) {
    unsigned long long v;
    asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(cluster_addr) : "memory");
    return v;
}

__device__ __forceinline__ float4 ld_dsmem_v4(uint32_t cluster_addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(cluster_addr)
                 : "memory");
    return v;
}

// Order-preserving map of a float onto the unsigned integers (for redux.sync
// max/min); NaN maps to 0, below every number.
__device__ __forceinline__ unsigned okey(float v) {
    const unsigned b = __float_as_uint(v);
    if (v != v) return 0u;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float okey_inv(unsigned k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Bounded wait on an mbarrier phase (about 4 s); false on abort or timeout.
__device__ __noinline__ bool wait_b(Shared *sh, uint32_t bar, uint32_t parity, uint64_t limit_ns, bool raise) {
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        if (gg::mbar_try_wait(bar, parity)) return true;
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

template <int LPL, int S>
__global__ void __launch_bounds__(kThreads, 1)
route_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW, const Params p) {
    constexpr int PS = pstride(S);
    constexpr int RT = kTile / S;            // tokens this CTA routes
    constexpr int LS = S == 1 ? PS : lstride(S);
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ Shared sh;
    const uint32_t raw_addr = gg::smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    float *P = reinterpret_cast<float *>(smem);                                  // [N][PS]
    float *Lb = S == 1 ? P : reinterpret_cast<float *>(smem + p.l_offset);      // [N][LS]

    const int warp = warp_id(), lane = lane_id();
    const uint32_t rank = S == 1 ? 0u : gg::cluster_rank();
    const int m0 = (int)(blockIdx.x / (unsigned)S) * kTile;
    const int r0 = (int)rank * RT;           // first tile row this CTA routes
    const int kblocks = p.d / kBK;
    const int kb0 = (int)rank * kblocks / S, kb1 = ((int)rank + 1) * kblocks / S;
    const uint32_t sbytes = (uint32_t)kXBytes + (uint32_t)p.Npad * kBK * 2;
    const int K = p.K, N = p.N;

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            gg::mbar_init(gg::smem_u32(&sh.full[s]), 1);
            gg::mbar_init(gg::smem_u32(&sh.empty[s]), 1);
        }
        gg::mbar_init(gg::smem_u32(&sh.acc_full), 1);
        gg::mbar_init(gg::smem_u32(&sh.drain), 1);
        sh.abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        // first fill of the operand ring: no stage has been used yet
        for (int i = 0; i < p.stages && kb0 + i < kb1; ++i) {
            const uint32_t fb = gg::smem_u32(&sh.full[i]);
            uint8_t *xs = smem + (size_t)i * sbytes;
            gg::mbar_arrive_expect_tx(fb, sbytes);
            gg::tma_load_2d(gg::smem_u32(xs), &tmX, fb, (kb0 + i) * kBK, m0);
            gg::tma_load_2d(gg::smem_u32(xs + kXBytes), &tmW, fb, (kb0 + i) * kBK, 0);
        }
    }
    for (int e = threadIdx.x; e < N; e += kThreads) {
        sh.dcount[e] = 0;
        sh.pacc[e] = 0ull;
        sh.wacc[e] = 0ull;
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         gg::smem_u32(&sh.tmem_base)),
                     "r"(p.tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    gg::tc_fence_before();
    __syncthreads();
    gg::tc_fence_after();
    const uint32_t tmem = sh.tmem_base;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            const int first = min(p.stages, kb1 - kb0);  // issued in the prologue
            uint32_t stage = (uint32_t)(first % p.stages), phase = first == p.stages ? 1u : 0u;
            int issued[kMaxStages];
            for (int s = 0; s < kMaxStages; ++s) issued[s] = s < first ? 0 : -1;
            bool stop = false;
            for (int kb = kb0 + first; kb < kb1; ++kb) {
                if (!wait_b(&sh, gg::smem_u32(&sh.empty[stage]), phase ^ 1u, gg::WAIT_LIMIT_NS, true)) {
                    stop = true;
                    break;
                }
                const uint32_t fb = gg::smem_u32(&sh.full[stage]);
                uint8_t *xs = smem + (size_t)stage * sbytes;
                gg::mbar_arrive_expect_tx(fb, sbytes);
                gg::tma_load_2d(gg::smem_u32(xs), &tmX, fb, kb * kBK, m0);
                gg::tma_load_2d(gg::smem_u32(xs + kXBytes), &tmW, fb, kb * kBK, 0);
                issued[stage] = (int)phase;
                if (++stage == (uint32_t)p.stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (stop) {
                for (int s = 0; s < p.stages; ++s)
                    if (issued[s] >= 0)
                        wait_b(&sh, gg::smem_u32(&sh.full[s]), (uint32_t)issued[s], gg::DRAIN_LIMIT_NS, false);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            uint32_t stage = 0, phase = 0;
            bool stop = false;
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!wait_b(&sh, gg::smem_u32(&sh.full[stage]), phase, gg::WAIT_LIMIT_NS, true)) {
                    stop = true;
                    break;
                }
                gg::tc_fence_after();
                const uint32_t a_addr = gg::smem_u32(smem + (size_t)stage * sbytes);
                const uint32_t b_addr = a_addr + kXBytes;
#pragma unroll
                for (int kk = 0; kk < kBK / gg::UMMA_K; ++kk)
                    mma_bf16_id(tmem, gg::sdesc(a_addr + kk * gg::UMMA_K * 2), gg::sdesc(b_addr + kk * gg::UMMA_K * 2),
                                p.idesc, (kb != kb0 || kk != 0) ? 1u : 0u);
                gg::mma_commit(gg::smem_u32(&sh.empty[stage]));
                if (++stage == (uint32_t)p.stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!stop) gg::mma_commit(gg::smem_u32(&sh.acc_full));
            // every MMA of this block has completed once `drain` fires
            gg::mma_commit(gg::smem_u32(&sh.drain));
            wait_b(&sh, gg::smem_u32(&sh.drain), 0, gg::DRAIN_LIMIT_NS, false);
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ---------------------------------------------------- TMEM -> shared memory
        const int q = warp & 3;
        const int row = q * 32 + lane;
        if (wait_b(&sh, gg::smem_u32(&sh.acc_full), 0, gg::WAIT_LIMIT_NS, true)) {
            gg::tc_fence_after();
            for (int c0 = 0; c0 < p.Npad; c0 += 32) {
                uint32_t r[32];
                gg::tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)c0, r);
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (c0 + j < N) P[(c0 + j) * PS + row] = __uint_as_float(r[j]);
            }
        }
    }
    gg::tc_fence_before();
    __syncthreads();

    if (S > 1) {
        gg::cluster_sync_all();  // every split's partial logits are visible cluster-wide
        // ---------------------------------------------------- split sum into the local buffer
        if (!sh.abort_flag) {
            constexpr int QPR = RT / 4;  // float4 groups per expert row
            const uint32_t pbase = gg::smem_u32(P);
            uint32_t peer[S];
#pragma unroll
            for (int sp = 0; sp < S; ++sp) peer[sp] = gg::map_to_rank(pbase, (uint32_t)sp);
            const int items = N * QPR;
            constexpr int IPP = 8 / S;  // items per pass: 8 vector loads in flight per thread
            for (int base = threadIdx.x; base < items; base += IPP * kThreads) {
                float4 v[IPP][S];
                int dst[IPP];
#pragma unroll
                for (int u = 0; u < IPP; ++u) {
                    const int it = base + u * kThreads;
                    const int itc = it < items ? it : base;
                    const int e = itc / QPR, q = itc - e * QPR;
                    dst[u] = it < items ? e * LS + 4 * q : -1;
                    const uint32_t off = (uint32_t)(e * PS + r0 + 4 * q) * 4u;
#pragma unroll
                    for (int sp = 0; sp < S; ++sp) v[u][sp] = ld_dsmem_v4(peer[sp] + off);
                }
#pragma unroll
                for (int u = 0; u < IPP; ++u) {
                    float4 a = v[u][0];
#pragma unroll
                    for (int sp = 1; sp < S; ++sp) {
                        a.x += v[u][sp].x;
                        a.y += v[u][sp].y;
                        a.z += v[u][sp].z;
                        a.w += v[u][sp].w;
                    }
                    if (dst[u] >= 0) {
                        float *d = Lb + dst[u];
                        d[0] = a.x;
                        d[1] = a.y;
                        d[2] = a.z;
                        d[3] = a.w;
                    }
                }
            }
        }
        __syncthreads();
        gg::cluster_sync_all();  // the peers have finished reading this block's partial logits
    }
    if (warp == 1) {
        gg::tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(p.tmem_cols)
                     : "memory");
    }

    // -------------------------------------------------------- routing
    // G consecutive lanes route one token; lane g of the group holds experts
    // g, g + G, ... (EPT of them). Group shuffles reduce within the group.
    {
        constexpr int NMAX = 32 * LPL;
        constexpr int G = route_group(LPL, S);
        constexpr int EPT = NMAX / G;
        constexpr int TPP = kThreads / G;  // tokens per pass
        static_assert(EPT <= 32 && (G & (G - 1)) == 0 && G <= 32, "group shape");
        const int gl = threadIdx.x % G;
        const int col0 = S == 1 ? r0 : 0;
        for (int e = threadIdx.x; e < N; e += kThreads) sh.bias[e] = p.sel_bias != nullptr ? p.sel_bias[e] : 0.f;
        __syncthreads();
        float lsq = 0.f, ent = 0.f, amax = 0.f;
        for (int i = threadIdx.x / G; i < RT && !sh.abort_flag; i += TPP) {
            // the loop bound is warp-uniform (RT is a multiple of the groups per
            // warp); tokens past T run along with zero logits and write nothing,
            // so every lane joins the full-warp shuffles
            const int t = m0 + r0 + i;
            const bool live = t < p.T;
            float sv[EPT], u[EPT];
            float m = -INFINITY;
#pragma unroll
            for (int j = 0; j < EPT; ++j) {
                const int e = gl + G * j;
                sv[j] = (live && e < N) ? Lb[e * LS + col0 + i] : 0.f;
                u[j] = e < N ? (sv[j] + sh.bias[e]) + 0.0f : -INFINITY;  // + 0.0f: -0 -> +0
                if (e < N) m = fmaxf(m, sv[j]);
            }
#pragma unroll
            for (int o = G / 2; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            float ex[EPT];
            float z = 0.f;
#pragma unroll
            for (int j = 0; j < EPT; ++j) {
                ex[j] = (gl + G * j < N) ? expf(sv[j] - m) : 0.f;
                z += ex[j];
            }
#pragma unroll
            for (int o = G / 2; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
            const float inv_z = 1.f / z;
            // routing entropy lse - sum_e p_e s_e and the logit range (health statistics)
            float ps = 0.f, am = 0.f;
#pragma unroll
            for (int j = 0; j < EPT; ++j)
                if (gl + G * j < N) {
                    ps += ex[j] * sv[j];
                    am = fmaxf(am, fabsf(sv[j]));
                }
#pragma unroll
            for (int o = G / 2; o > 0; o >>= 1) {
                ps += __shfl_xor_sync(0xffffffffu, ps, o);
                am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
            }
            if (gl == 0 && live) {
                const float lse = m + logf(z);
                lsq += lse * lse;
                ent += lse - ps * inv_z;
                amax = fmaxf(amax, am);
            }
            // this token's softmax probabilities replace its logits in the column
#pragma unroll
            for (int j = 0; j < EPT; ++j)
                if (live && gl + G * j < N) Lb[(gl + G * j) * LS + col0 + i] = ex[j] * inv_z;

            // K rounds of arg-max on u = s + b over the unselected experts:
            // larger u first, equal u -> smaller expert id first
            // (the rounds are not unrolled: with up to 8 rounds over up to 32
            // experts per lane the unrolled body was large enough that
            // instruction fetch, from a cold cache every layer, dominated)
            unsigned taken = 0u;
            int sel_e[route::kMaxK];
            float sel_s[route::kMaxK];
#pragma unroll
            for (int k = 0; k < route::kMaxK; ++k) {
                sel_e[k] = -1;
                sel_s[k] = 0.f;
            }
#pragma unroll 1
            for (int k = 0; k < K; ++k) {
                {
                    float bu = -INFINITY, bs = 0.f;
                    int be = 0x7fffffff;
#pragma unroll
                    for (int j = 0; j < EPT; ++j) {
                        const int e = gl + G * j;
                        if (e < N && !((taken >> j) & 1u) && (u[j] > bu || be == 0x7fffffff)) {
                            bu = u[j];
                            be = e;
                            bs = sv[j];
                        }
                    }
#pragma unroll
                    for (int o = G / 2; o > 0; o >>= 1) {
                        const float ou = __shfl_xor_sync(0xffffffffu, bu, o);
                        const int oe = __shfl_xor_sync(0xffffffffu, be, o);
                        const float os = __shfl_xor_sync(0xffffffffu, bs, o);
                        if (ou > bu || (ou == bu && oe < be)) {
                            bu = ou;
                            be = oe;
                            bs = os;
                        }
                    }
                    if (be != 0x7fffffff && be % G == gl) taken |= 1u << (be / G);
#pragma unroll
                    for (int q = 0; q < route::kMaxK; ++q)  // keeps the arrays in registers
                        if (q == k) {
                            sel_e[q] = be;
                            sel_s[q] = bs;
                        }
                }
            }
            if (gl == 0 && live) {
                // softmax over the K selected, unbiased logits
                float mk = -INFINITY;
#pragma unroll
                for (int k = 0; k < route::kMaxK; ++k)
                    if (k < K) mk = fmaxf(mk, sel_s[k]);
                float nu[route::kMaxK];
                float den = 0.f;
#pragma unroll
                for (int k = 0; k < route::kMaxK; ++k) {
                    nu[k] = k < K ? expf(sel_s[k] - mk) : 0.f;
                    den += nu[k];
                }
#pragma unroll
                for (int k = 0; k < route::kMaxK; ++k) {
                    if (k < K) {
                        const bool ok = (unsigned)sel_e[k] < (unsigned)N;
                        p.topk_idx[(size_t)t * K + k] = ok ? sel_e[k] : -1;
                        p.topk_w[(size_t)t * K + k] = nu[k] / den;
                        if (ok) {
                            atomicAdd(&sh.dcount[sel_e[k]], 1);
                            atomicAdd(&sh.wacc[sel_e[k]], (unsigned long long)__float2uint_rn(nu[k] / den * kProbScale));
                        } else
                            flag_error(MOE_DEVERR_EXPERT_ID);  // no orderable logit (NaN input)
                    }
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            lsq += __shfl_xor_sync(0xffffffffu, lsq, o);
            ent += __shfl_xor_sync(0xffffffffu, ent, o);
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        }
        if (lane == 0) {
            sh.lsq_w[warp] = lsq;
            sh.ent_w[warp] = ent;
            sh.amax_w[warp] = amax;
        }
        __syncthreads();
        // per-expert sums of this block's probabilities, in fixed point
        const int nlive = sh.abort_flag ? 0 : max(0, min(RT, p.T - (m0 + r0)));
        for (int e = threadIdx.x; e < N; e += kThreads) {
            unsigned long long a = 0ull;
            const float *row = Lb + e * LS + col0;
            for (int j = 0; j < nlive; ++j) a += __float2uint_rn(row[j] * kProbScale);
            sh.pacc[e] = a;
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float a = 0.f, b = 0.f, c = 0.f;
        for (int w = 0; w < kWarps; ++w) {
            a += sh.lsq_w[w];
            b += sh.ent_w[w];
            c = fmaxf(c, sh.amax_w[w]);
        }
        p.lse_partial[(size_t)blockIdx.x * route::kPartialStride] = a;
        p.lse_partial[(size_t)blockIdx.x * route::kPartialStride + 1] = b;
        p.lse_partial[(size_t)blockIdx.x * route::kPartialStride + 2] = c;
    }

    // -------------------------------------------------------- the tile's per-expert row
    // The S CTAs of the cluster route disjoint token ranges of one 128-token
    // tile; CTA r adds their counts and fixed-point sums for experts
    // r, r + S, ... in rank order (integers: any order gives the same total)
    // and writes them. No global atomics, no zeroed counters, no ticket.
    const size_t row = (size_t)(blockIdx.x / (unsigned)S) * N;
    if (S == 1) {
        for (int e = threadIdx.x; e < N; e += kThreads) {
            p.tile_hist[row + e] = sh.dcount[e];
            p.tile_prob[row + e] = sh.pacc[e];
            p.tile_w[row + e] = sh.wacc[e];
        }
    } else {
        gg::cluster_sync_all();  // every CTA's per-expert totals are visible cluster-wide
        for (int e = (int)rank + S * (int)threadIdx.x; e < N; e += S * kThreads) {
            uint32_t dc = 0;
            unsigned long long pa = 0ull, wa = 0ull;
#pragma unroll
            for (int sp = 0; sp < S; ++sp) {
                dc += ld_dsmem_u32(gg::map_to_rank(gg::smem_u32(&sh.dcount[e]), (uint32_t)sp));
                pa += ld_dsmem_u64(gg::map_to_rank(gg::smem_u32(&sh.pacc[e]), (uint32_t)sp));
                wa += ld_dsmem_u64(gg::map_to_rank(gg::smem_u32(&sh.wacc[e]), (uint32_t)sp));
            }
            p.tile_hist[row + e] = (int32_t)dc;
            p.tile_prob[row + e] = pa;
            p.tile_w[row + e] = wa;
        }
        gg::cluster_sync_all();  // the peers have finished reading this CTA's totals
    }

    // -------------------------------------------------------- single tile: the plan here
    // Every CTA's rows, routing weights and expert ids are visible to the
    // cluster after the barrier above (release / acquire at cluster scope);
    // the operand ring is free, so its shared memory is the scratch. CTA 0
    // forms the dispatch plan and the tile lists the GEMMs wait for; the
    // statistics and losses feed no later kernel, so with a cluster of two or
    // more CTAs rank 1 forms them at the same time.
    const uint32_t loss_rank = S > 1 ? 1u : 0u;
    if (p.fuse_plan && (rank == 0 || rank == loss_rank)) {
        __syncthreads();  // (one CTA: its own row writes)
        int *s_dem = reinterpret_cast<int *>(smem);
        float *s_prob = reinterpret_cast<float *>(s_dem + kMaxN);
        int *s_off = reinterpret_cast<int *>(s_prob + kMaxN);  // kMaxN + 1
        int *sc = s_off + kMaxN + 4;                             // kThreads
        float *t_aux = reinterpret_cast<float *>(sc + kThreads);
        float *t_kl = t_aux + kMaxN, *t_var = t_kl + kMaxN;
        unsigned *bits = reinterpret_cast<unsigned *>(t_var + kMaxN);  // kWarps x N
        const bool stats_here = rank == loss_rank;
        for (int e = threadIdx.x; e < N; e += kThreads) {
            const int dem = __ldcg(p.tile_hist + e);
            s_dem[e] = dem;
            if (stats_here) {
                const float prob = __ull2float_rn(__ldcg(p.tile_prob + e)) * plan::kFixUnit;
                s_prob[e] = prob;
                p.st.demand[e] = dem;
                p.st.prob_sum[e] = prob;
                if (p.st.mean_weight != nullptr)
                    p.st.mean_weight[e] =
                        dem > 0 ? __ull2float_rn(__ldcg(p.tile_w + e)) * plan::kFixUnit / (float)dem : 0.f;
            }
        }
        __syncthreads();
        int kept_rows = -1;
        if (rank == 0) {
            plan::expert_offsets(s_dem, N, p.dp.C, s_off, sc, p.dp.kept, p.dp.offsets);
            plan::assign_tokens(p.topk_idx, p.T, K, N, p.dp.C, s_off, bits, p.dp.slot_of, p.dp.row_token,
                                p.T * K);
            __syncthreads();
            if (p.dp.mtiles != nullptr)
                gg::build_mtiles_block(s_off, N, p.T * K, p.dp.tile_rows, p.dp.raster, p.dp.max_tiles, p.dp.mtiles,
                                       p.dp.num_mtiles, sc);
            __syncthreads();
            if (p.dp.mtiles2 != nullptr)
                gg::build_mtiles_block(s_off, N, p.T * K, p.dp.tile_rows2, p.dp.raster2, p.dp.max_tiles,
                                       p.dp.mtiles2, p.dp.num_mtiles2, sc);
            kept_rows = s_off[N];
        } else {  // rows kept = sum of min(demand, C), an integer sum (any order)
            int v = threadIdx.x < N ? min(s_dem[threadIdx.x], p.dp.C) : 0;
            v = __reduce_add_sync(0xffffffffu, v);
            if ((threadIdx.x & 31) == 0) sc[threadIdx.x >> 5] = v;
            __syncthreads();
            kept_rows = 0;
            for (int w = 0; w < kWarps; ++w) kept_rows += sc[w];
        }
        if (stats_here) plan::losses(p.st, s_dem, s_prob, t_aux, t_kl, t_var, kept_rows);
    }
}

}  // namespace rtc
}  // namespace moe
