// dispatch.cuh -- capacity-limited, token-ordered dispatch and the combine
// (lmnt.cn/news/351908 sec. 3.1: regroup token order into one contiguous block
// per expert; sec. 3.2: combine through the same index table, same order;
// sec. 3.3: capacity = ceil(T/N * capacity_factor), overflow dropped).
//
// Position of assignment (t, k) with expert e inside e's block:
//   p = #{t' < t : e in topk_idx[t']}     (each token names an expert at most once)
// computed as   base[chunk][e]              exclusive scan over 128-token chunks
//             + popc(bits[w'][e]) for the chunk's earlier warps
//             + popc(bits[w][e] & lanes below this one)
// where bits[w][e] has bit l set iff token (chunk, w, l) chose e. Integer work
// only: bit-exact and independent of scheduling.
#pragma once

#include "common.cuh"

namespace moe {
namespace dispatch {

constexpr int kChunk = 128;  // tokens per block (4 warps x 32 lanes)

inline int num_chunks(int rows) { return (rows + kChunk - 1) / kChunk; }

// Capacity priority. Token order (the default): the assignments of token t
// come before those of every later token. Rank order: every token's k-th
// choice comes before any token's (k+1)-th choice. Both are handled as one
// scan over "virtual tokens" v that name one expert each at most once:
//   token order  v = t, entries (t, 0..K-1)
//   rank order   v = k * T + t, entry (t, k) alone
struct Order {
    int T, K, rank_major;
    __device__ __forceinline__ int tv() const { return rank_major ? T * K : T; }
    __device__ __forceinline__ int kv() const { return rank_major ? 1 : K; }
    // flat index (t * K + k) of the j-th entry of virtual token v
    __device__ __forceinline__ int entry(int v, int j) const {
        return rank_major ? (v % T) * K + v / T : v * K + j;
    }
    __device__ __forceinline__ int token(int v) const { return rank_major ? v % T : v; }
};

// hist[chunk][e] = assignments to e among the chunk's virtual tokens.
__global__ void __launch_bounds__(kChunk)
count_kernel(const int32_t *__restrict__ topk_idx, Order o, int N, int32_t *__restrict__ hist) {
    extern __shared__ int cnt[];  // [N]
    for (int e = threadIdx.x; e < N; e += blockDim.x) cnt[e] = 0;
    __syncthreads();
    const int v = blockIdx.x * kChunk + threadIdx.x;
    if (v < o.tv()) {
        for (int j = 0; j < o.kv(); ++j) {
            int e = topk_idx[o.entry(v, j)];
            if (e >= 0 && e < N)
                atomicAdd(&cnt[e], 1);
            else
                flag_error(MOE_DEVERR_EXPERT_ID);
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < N; e += blockDim.x) hist[(size_t)blockIdx.x * N + e] = cnt[e];
}

// One block. base[c][e] = sum_{c' < c} hist[c'][e]; kept[e] = min(total, C);
// offsets = exclusive prefix of kept (offsets[N] = kept rows R). drop_rate
// (optional): the fraction of the `total` assignments past capacity (the
// token drop rate the lmnt.cn/news/351908 sec. 8.2 / 9.3 monitors watch).
__global__ void __launch_bounds__(1024)
scan_kernel(const int32_t *__restrict__ hist, int chunks, int N, int C, int32_t *__restrict__ base,
            int32_t *__restrict__ kept, int32_t *__restrict__ offsets, float *__restrict__ drop_rate, int total) {
    extern __shared__ int sh[];  // [N] kept, then scan buffer [N]
    int *kv = sh;
    for (int e = threadIdx.x; e < N; e += blockDim.x) {
        int run = 0;
#pragma unroll 8
        for (int c = 0; c < chunks; ++c) {
            int h = hist[(size_t)c * N + e];
            base[(size_t)c * N + e] = run;
            run += h;
        }
        int kp = run < C ? run : C;
        kept[e] = kp;
        kv[e] = kp;
    }
    __syncthreads();
    // inclusive Hillis-Steele scan over N <= 1024 entries, one per thread
    const int e = threadIdx.x;
    int v = (e < N) ? kv[e] : 0;
    for (int o = 1; o < N; o <<= 1) {
        int add = (e >= o && e < N) ? kv[e - o] : 0;
        __syncthreads();
        if (e < N) kv[e] = v = v + add;
        __syncthreads();
    }
    if (e < N) offsets[e + 1] = v;
    if (e == 0) offsets[0] = 0;
    if (drop_rate != nullptr && e == N - 1) drop_rate[0] = (float)((double)(total - v) / (double)total);
}

// slot_of[t, k] = offsets[e] + p if p < C else -1; row_token[slot] = t, and
// row_token[r] = -1 for the rows r in [offsets[N], rows) that nothing keeps.
__global__ void __launch_bounds__(kChunk)
assign_kernel(const int32_t *__restrict__ topk_idx, Order o, int N, int C, const int32_t *__restrict__ base,
              const int32_t *__restrict__ offsets, int32_t *__restrict__ slot_of, int32_t *__restrict__ row_token,
              int rows) {
    extern __shared__ unsigned bits[];  // [4][N]
    for (int i = threadIdx.x; i < 4 * N; i += blockDim.x) bits[i] = 0u;
    for (int r = __ldg(offsets + N) + blockIdx.x * blockDim.x + threadIdx.x; r < rows; r += gridDim.x * blockDim.x)
        row_token[r] = -1;
    __syncthreads();
    const int w = warp_id(), lane = lane_id();
    const int v = blockIdx.x * kChunk + threadIdx.x;
    if (v < o.tv()) {
        for (int j = 0; j < o.kv(); ++j) {
            int e = topk_idx[o.entry(v, j)];
            if (e >= 0 && e < N) atomicOr(&bits[w * N + e], 1u << lane);
        }
    }
    __syncthreads();
    if (v >= o.tv()) return;
    const unsigned below = (1u << lane) - 1u;
    for (int j = 0; j < o.kv(); ++j) {
        const int ent = o.entry(v, j);
        int e = topk_idx[ent];
        int slot = -1;
        if (e >= 0 && e < N) {
            int p = base[(size_t)blockIdx.x * N + e];
            for (int w2 = 0; w2 < w; ++w2) p += __popc(bits[w2 * N + e]);
            p += __popc(bits[w * N + e] & below);
            if (p < C) {
                slot = offsets[e] + p;
                row_token[slot] = o.token(v);
            }
        }
        slot_of[ent] = slot;
    }
}

// The count, scan and assign kernels in one launch, for a dispatch of at most
// kChunk virtual tokens (decode batches): one block of kChunk threads, with
// the same counts, the same exclusive scan of the kept counts (one warp,
// ceil(N / 32) experts per lane) and the same positions
// p = popc of the earlier warps' and lanes' bits, so every output is the one
// the three kernels write; row_token is filled with -1 first.
__global__ void __launch_bounds__(kChunk)
dispatch_small_kernel(const int32_t *__restrict__ topk_idx, Order o, int N, int C, int32_t *__restrict__ kept,
                      int32_t *__restrict__ offsets, int32_t *__restrict__ slot_of, int32_t *__restrict__ row_token,
                      float *__restrict__ drop_rate, int total) {
    extern __shared__ int sh[];  // cnt[N], off[N + 1], bits[4][N]
    int *cnt = sh;
    int *off = sh + N;
    unsigned *bits = reinterpret_cast<unsigned *>(sh + 2 * N + 1);
    for (int e = threadIdx.x; e < N; e += blockDim.x) cnt[e] = 0;
    for (int i = threadIdx.x; i < 4 * N; i += blockDim.x) bits[i] = 0u;
    for (int i = threadIdx.x; i < total; i += blockDim.x) row_token[i] = -1;
    __syncthreads();
    const int w = warp_id(), lane = lane_id();
    const int v = threadIdx.x;
    if (v < o.tv()) {
        for (int j = 0; j < o.kv(); ++j) {
            const int e = topk_idx[o.entry(v, j)];
            if (e >= 0 && e < N) {
                atomicAdd(&cnt[e], 1);
                atomicOr(&bits[w * N + e], 1u << lane);
            } else {
                flag_error(MOE_DEVERR_EXPERT_ID);
            }
        }
    }
    __syncthreads();
    if (w == 0) {
        const int per = (N + 31) / 32, e0 = min(N, lane * per), e1 = min(N, e0 + per);
        int sum = 0;
        for (int e = e0; e < e1; ++e) sum += min(cnt[e], C);
        int incl = sum;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int t = __shfl_up_sync(0xFFFFFFFFu, incl, d);
            if (lane >= d) incl += t;
        }
        int run = incl - sum;
        for (int e = e0; e < e1; ++e) {
            const int k = min(cnt[e], C);
            kept[e] = k;
            off[e] = run;
            offsets[e] = run;
            run += k;
        }
        if (lane == 31) {
            offsets[N] = incl;
            if (drop_rate != nullptr) drop_rate[0] = (float)((double)(total - incl) / (double)total);
        }
    }
    __syncthreads();
    if (v >= o.tv()) return;
    const unsigned below = (1u << lane) - 1u;
    for (int j = 0; j < o.kv(); ++j) {
        const int ent = o.entry(v, j);
        const int e = topk_idx[ent];
        int slot = -1;
        if (e >= 0 && e < N) {
            int p = 0;
            for (int w2 = 0; w2 < w; ++w2) p += __popc(bits[w2 * N + e]);
            p += __popc(bits[w * N + e] & below);
            if (p < C) {
                slot = off[e] + p;
                row_token[slot] = o.token(v);
            }
        }
        slot_of[ent] = slot;
    }
}

// Tokens per block in the permute and combine kernels: a thread owns one
// 16-byte column chunk of kRowTok consecutive tokens, so one block issues all
// of its loads after a single round trip for the dispatch table.
constexpr int kRowTok = 8;

// x_perm[slot_of[t, k]] = x[t].
__global__ void __launch_bounds__(256)
permute_kernel(const uint16_t *__restrict__ x, const int32_t *__restrict__ slot_of, int T, int K, int d,
               int rows, uint16_t *__restrict__ x_perm) {
    const int t0 = blockIdx.x * kRowTok;
    const int c = blockIdx.y * blockDim.x + threadIdx.x;
    const int vec = d >> 3;
    __shared__ int slots[kRowTok][8];
    if (threadIdx.x < kRowTok * K) {
        const int i = threadIdx.x / K, k = threadIdx.x % K;
        int s = -1;
        if (t0 + i < T) {
            s = slot_of[(size_t)(t0 + i) * K + k];
            if (s >= rows) {
                flag_error(MOE_DEVERR_ROW_INDEX);
                s = -1;
            }
        }
        slots[i][k] = s;
    }
    __syncthreads();
    if (c >= vec) return;
    uint4 v[kRowTok];
#pragma unroll
    for (int i = 0; i < kRowTok; ++i)
        if (t0 + i < T) v[i] = __ldg(reinterpret_cast<const uint4 *>(x + (size_t)(t0 + i) * d) + c);
#pragma unroll
    for (int i = 0; i < kRowTok; ++i) {
        if (t0 + i >= T) break;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if (k < K) {
                const int s = slots[i][k];
                if (s >= 0) reinterpret_cast<uint4 *>(x_perm + (size_t)s * d)[c] = v[i];
            }
        }
    }
}

// y[t] = bf16(z[t] + sum_k w[t,k] * y_perm[slot_of[t,k]]), fp32, increasing k.
// A thread owns one 16-byte column chunk of TOK = 8 / KMAX consecutive tokens
// and issues all TOK * KMAX row loads before any arithmetic.
template <int KMAX>
__global__ void __launch_bounds__(256)
combine_kernel(const uint16_t *__restrict__ y_perm, const int32_t *__restrict__ slot_of,
               const float *__restrict__ topk_w, const uint16_t *__restrict__ z, int T, int K, int d, int rows,
               uint16_t *__restrict__ y) {
    constexpr int TOK = 8 / KMAX;
    const int t0 = blockIdx.x * TOK;
    const int c = blockIdx.y * blockDim.x + threadIdx.x;
    const int vec = d >> 3;
    __shared__ int slots[TOK][KMAX];
    __shared__ float wts[TOK][KMAX];
    if (threadIdx.x < TOK * KMAX) {
        const int i = threadIdx.x / KMAX, k = threadIdx.x % KMAX;
        int s = -1;
        float w = 0.f;
        if (t0 + i < T && k < K) {
            s = slot_of[(size_t)(t0 + i) * K + k];
            w = topk_w[(size_t)(t0 + i) * K + k];
            if (s >= rows) {
                flag_error(MOE_DEVERR_ROW_INDEX);
                s = -1;
            }
        }
        slots[i][k] = s;
        wts[i][k] = w;
    }
    __syncthreads();
    if (c >= vec) return;
    uint4 v[TOK][KMAX];
#pragma unroll
    for (int i = 0; i < TOK; ++i)
#pragma unroll
        for (int k = 0; k < KMAX; ++k) {
            const int sl = slots[i][k];
            v[i][k] = sl >= 0 ? __ldg(reinterpret_cast<const uint4 *>(y_perm + (size_t)sl * d) + c)
                              : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
    for (int i = 0; i < TOK; ++i) {
        const int t = t0 + i;
        if (t >= T) break;
        float acc[8];
        if (z != nullptr) {
            uint4 zv = __ldg(reinterpret_cast<const uint4 *>(z + (size_t)t * d) + c);
            unpack_bf16x2(zv.x, acc[0], acc[1]);
            unpack_bf16x2(zv.y, acc[2], acc[3]);
            unpack_bf16x2(zv.z, acc[4], acc[5]);
            unpack_bf16x2(zv.w, acc[6], acc[7]);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] = 0.f;
        }
#pragma unroll
        for (int k = 0; k < KMAX; ++k) {
            if (slots[i][k] >= 0) {
                const float wk = wts[i][k];
                float f[8];
                unpack_bf16x2(v[i][k].x, f[0], f[1]);
                unpack_bf16x2(v[i][k].y, f[2], f[3]);
                unpack_bf16x2(v[i][k].z, f[4], f[5]);
                unpack_bf16x2(v[i][k].w, f[6], f[7]);
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[j] = fmaf(wk, f[j], acc[j]);
            }
        }
        uint4 o;
        o.x = pack_bf16x2(acc[0], acc[1]);
        o.y = pack_bf16x2(acc[2], acc[3]);
        o.z = pack_bf16x2(acc[4], acc[5]);
        o.w = pack_bf16x2(acc[6], acc[7]);
        reinterpret_cast<uint4 *>(y + (size_t)t * d)[c] = o;
    }
}

// aux = alpha * N * sum_e (demand[e] / (T K)) * (prob_sum[e] / T), in double,
// fixed reduction order (lmnt.cn/news/351908 sec. 5.1-5.2).
__global__ void aux_loss_kernel(const int32_t *__restrict__ demand, const float *__restrict__ prob_sum,
                                int T, int N, int K, float alpha, float *__restrict__ aux) {
    __shared__ double part[32];
    double a = 0.0;
    for (int e = threadIdx.x; e < N; e += blockDim.x)
        a += ((double)demand[e] / ((double)T * (double)K)) * ((double)prob_sum[e] / (double)T);
    for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
    if (lane_id() == 0) part[warp_id()] = a;
    __syncthreads();
    if (threadIdx.x == 0) {
        double s = 0.0;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) s += part[w];
        aux[0] = (float)((double)alpha * (double)N * s);
    }
}

}  // namespace dispatch
}  // namespace moe
