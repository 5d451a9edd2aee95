// backward.cuh -- the layer's backward pass: everything but the four big
// contractions, which run on the grouped tcgen05 GEMM (grouped_gemm.cuh):
//   dh  = dO W2            (grouped over experts, W2 read as stored: N-major B)
//   dx' = da W1            (grouped over experts, W1 read as stored: N-major B)
//   dW2 = dO^T h, dW1 = da^T x    (per expert, the expert's tokens as the
//                           reduction: transposed, 64-padded activation copies)
// Definitions (the gradient of the forward with the routing held fixed; the
// training signal of lmnt.cn/news/351908 sec. 5):
//   combine   dw_tk = <dy_t, o_tk>,  dO_tk = bf16(w_tk dy_t)
//   expert    da = bf16(dh * GELU'(a)), a = x W1^T + b1 recomputed in fp32
//   biases    db1 = sum da, db2 = sum dO per expert (fixed-order column sums)
//   gate      ds_t = softmax Jacobian of the K kept weights applied to dw_t
//             + balance-loss and z-loss terms; dW_g = ds^T x, dx += ds W_g
// Every reduction runs in a fixed order: results are run-to-run identical.
#pragma once

#include "common.cuh"

namespace moe {
namespace bwd {

constexpr int kThreads = 256;

// Expert owning row r of the regrouped buffer (offsets[N] = rows).
__device__ __forceinline__ int expert_of_row(const int32_t *__restrict__ offsets, int N, int r) {
    int lo = 0, hi = N - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (offsets[mid] <= r)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ float gelu_grad(float v) {
    // d/dv [v Phi(v)] = Phi(v) + v phi(v)
    return 0.5f * (1.0f + erff(v * 0.70710678118654752440f)) + v * 0.39894228040143267794f * expf(-0.5f * v * v);
}

// Fixed-order block sum (blockDim = kThreads); valid in thread 0.
__device__ __forceinline__ float block_sum(float v, float *scratch) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    __syncthreads();
    if (lane_id() == 0) scratch[warp_id()] = v;
    __syncthreads();
    float s = 0.f;
    if (threadIdx.x == 0)
        for (int w = 0; w < kThreads / 32; ++w) s += scratch[w];
    return s;
}

// One block per token: dw[t, k] = <dy_t, y_perm[slot]> (0 when dropped) and
// dO[slot] = bf16(w[t, k] * dy_t).
__global__ void __launch_bounds__(kThreads)
combine_backward_kernel(const uint16_t *__restrict__ dy, const uint16_t *__restrict__ y_perm,
                        const int32_t *__restrict__ slot_of, const float *__restrict__ topk_w, int K, int d,
                        float *__restrict__ dw, uint16_t *__restrict__ dO) {
    __shared__ float scratch[kThreads / 32];
    const int t = blockIdx.x;
    const uint16_t *g = dy + (size_t)t * d;
    for (int k = 0; k < K; ++k) {
        const int r = slot_of[(size_t)t * K + k];
        if (r < 0) {  // block-uniform
            if (threadIdx.x == 0) dw[(size_t)t * K + k] = 0.f;
            continue;
        }
        const float wk = topk_w[(size_t)t * K + k];
        const uint16_t *o = y_perm + (size_t)r * d;
        uint16_t *dst = dO + (size_t)r * d;
        float acc = 0.f;
        for (int c = threadIdx.x; c < d; c += kThreads) {
            const float gv = bf16_bits_to_float(g[c]);
            acc = fmaf(gv, bf16_bits_to_float(o[c]), acc);
            dst[c] = (uint16_t)(__bfloat16_as_ushort(__float2bfloat16_rn(wk * gv)));
        }
        const float s = block_sum(acc, scratch);
        if (threadIdx.x == 0) dw[(size_t)t * K + k] = s;
    }
}

// da[r, j] = bf16(dh[r, j] * GELU'(a[r, j] + b1[e(r), j])), a and dh fp32
// (raw GEMM accumulators). One block per row.
__global__ void __launch_bounds__(kThreads)
gelu_backward_kernel(const float *__restrict__ dh, const float *__restrict__ a, const float *__restrict__ b1,
                     const int32_t *__restrict__ offsets, int N, int f, uint16_t *__restrict__ da) {
    const int r = blockIdx.x;
    if (r >= offsets[N]) return;  // the grid covers the largest possible row count
    const int e = expert_of_row(offsets, N, r);
    const float *dhr = dh + (size_t)r * f;
    const float *ar = a + (size_t)r * f;
    const float *br = b1 + (size_t)e * f;
    uint16_t *out = da + (size_t)r * f;
    for (int j = threadIdx.x; j < f; j += kThreads)
        out[j] = __bfloat16_as_ushort(__float2bfloat16_rn(dhr[j] * gelu_grad(ar[j] + br[j])));
}

// out[e, c] = sum over the rows of expert e of in[r, c] (bf16 in, fp32 sum in
// row order). grid = (ceil(C / kThreads), N).
__global__ void __launch_bounds__(kThreads)
expert_colsum_kernel(const uint16_t *__restrict__ in, const int32_t *__restrict__ offsets, int C,
                     float *__restrict__ out) {
    const int e = blockIdx.y;
    const int c = blockIdx.x * kThreads + threadIdx.x;
    if (c >= C) return;
    float s = 0.f;
    for (int r = offsets[e]; r < offsets[e + 1]; ++r) s += bf16_bits_to_float(in[(size_t)r * C + c]);
    out[(size_t)e * C + c] = s;
}

// The single group {0, rows} and its padded form {0, roundup64(rows)}.
__global__ void single_group_kernel(int rows, int32_t *__restrict__ off, int32_t *__restrict__ poff) {
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    off[0] = 0;
    off[1] = rows;
    poff[0] = 0;
    poff[1] = (rows + 63) / 64 * 64;
}

// Padded group offsets: poff[e + 1] = poff[e] + roundup64(rows of group e).
__global__ void padded_offsets_kernel(const int32_t *__restrict__ offsets, int N, int32_t *__restrict__ poff) {
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    int acc = 0;
    poff[0] = 0;
    for (int e = 0; e < N; ++e) {
        const int rows = offsets[e + 1] - offsets[e];
        acc += (rows + 63) / 64 * 64;
        poff[e + 1] = acc;
    }
}

// out[c, poff[e] + r - offsets[e]] = in[r, c] for the rows r of group e:
// the regrouped rows become the columns of a [C, ld] matrix whose groups
// start at 64-aligned columns (padding columns are zeroed by the caller).
// 32 x 32 tiles through shared memory; grid = (ceil(C / 32), ceil(R / 32)).
__global__ void __launch_bounds__(kThreads)
transpose_grouped_kernel(const uint16_t *__restrict__ in, int R, int C, const int32_t *__restrict__ offsets,
                         const int32_t *__restrict__ poff, int N, uint16_t *__restrict__ out, size_t ld) {
    __shared__ uint16_t tile[32][33];
    const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 8 rows of 32 threads
    for (int i = ty; i < 32; i += 8) {
        const int r = r0 + i, c = c0 + tx;
        tile[i][tx] = (r < R && c < C) ? in[(size_t)r * C + c] : (uint16_t)0;
    }
    __syncthreads();
    const int r = r0 + tx;
    if (r >= R || r >= offsets[N]) return;
    const int e = expert_of_row(offsets, N, r);
    const size_t col = (size_t)poff[e] + (size_t)(r - offsets[e]);
    for (int i = ty; i < 32; i += 8) {
        const int c = c0 + i;
        if (c < C) out[(size_t)c * ld + col] = tile[tx][i];
    }
}

// Gate gradient, one warp per token (lane l: experts l, l + 32, ...):
//   p = softmax(s_t) over all N, lse = logsumexp(s_t)
//   ds[e] = g_aux alpha N / T p_e (f_e - sum_e' f_e' p_e') + g_z 2 beta / T lse p_e
//         + [e in TopK] w_e (dw_e - sum_k w_k dw_k)
// with f = demand / (T K) (constant: counts carry no gradient).
__global__ void __launch_bounds__(kThreads)
gate_backward_kernel(const float *__restrict__ logits, const int32_t *__restrict__ topk_idx,
                     const float *__restrict__ topk_w, const float *__restrict__ dw,
                     const int32_t *__restrict__ demand, int T, int N, int K, float alpha, float beta, float g_aux,
                     float g_z, float *__restrict__ ds) {
    const int t = blockIdx.x * (kThreads / 32) + warp_id();
    if (t >= T) return;  // warp-uniform
    const int lane = lane_id();
    const float *s = logits + (size_t)t * N;
    float m = -INFINITY;
    for (int e = lane; e < N; e += 32) m = fmaxf(m, s[e]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float z = 0.f;
    for (int e = lane; e < N; e += 32) z += expf(s[e] - m);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    const float inv_z = 1.f / z, lse = m + logf(z);
    const float inv_tk = 1.f / ((float)T * (float)K);
    float fp = 0.f;
    for (int e = lane; e < N; e += 32) fp += ((float)demand[e] * inv_tk) * (expf(s[e] - m) * inv_z);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) fp += __shfl_xor_sync(0xffffffffu, fp, o);
    const float ca = g_aux * alpha * (float)N / (float)T, cz = g_z * 2.f * beta / (float)T * lse;
    float sdw = 0.f;
    for (int k = 0; k < K; ++k) sdw += topk_w[(size_t)t * K + k] * dw[(size_t)t * K + k];
    float *out = ds + (size_t)t * N;
    for (int e = lane; e < N; e += 32) {
        const float p = expf(s[e] - m) * inv_z;
        float g = ca * p * ((float)demand[e] * inv_tk - fp) + cz * p;
        for (int k = 0; k < K; ++k)
            if (topk_idx[(size_t)t * K + k] == e)
                g += topk_w[(size_t)t * K + k] * (dw[(size_t)t * K + k] - sdw);
        out[e] = g;
    }
}

// C[M, N] (fp32, row-major) = sum_k A(m, k) B(k, n), SIMT, 64 x 64 tiles, k in
// slabs of 32 staged in shared memory; 4 x 4 outputs per thread. The operand
// accessors are the two gate contractions:
//   dW_g[e, i] = sum_t ds[t, e] x[t, i]     (A = ds^T fp32, B = x bf16, k = t)
//   dx[t, i]  = sum_e ds[t, e] W_g[e, i]    (A = ds fp32, B = W_g bf16, k = e)
// Both read A as a [k][m]... strided view and B as [k][n] rows: A(m, k) =
// a[k * a_ks + m * a_ms], B(k, n) = b[k * ldb + n].
constexpr int kSB = 64, kSK = 32;

__global__ void __launch_bounds__(kThreads)
simt_gemm_kernel(const float *__restrict__ a, size_t a_ks, size_t a_ms, const uint16_t *__restrict__ b,
                 size_t ldb, int M, int Nn, int Kk, float *__restrict__ c, size_t ldc) {
    __shared__ __align__(16) float As[kSK][kSB + 4];
    __shared__ __align__(16) float Bs[kSK][kSB + 4];
    const int m0 = blockIdx.y * kSB, n0 = blockIdx.x * kSB;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    for (int k0 = 0; k0 < Kk; k0 += kSK) {
        for (int q = threadIdx.x; q < kSK * kSB; q += kThreads) {
            const int kk = q / kSB, mm = q % kSB;
            const int k = k0 + kk;
            As[kk][mm] = (k < Kk && m0 + mm < M) ? a[(size_t)k * a_ks + (size_t)(m0 + mm) * a_ms] : 0.f;
            Bs[kk][mm] = (k < Kk && n0 + mm < Nn) ? bf16_bits_to_float(b[(size_t)k * ldb + n0 + mm]) : 0.f;
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < kSK; ++kk) {
            const float4 av = *reinterpret_cast<const float4 *>(&As[kk][ty * 4]);
            const float4 bv = *reinterpret_cast<const float4 *>(&Bs[kk][tx * 4]);
            const float ar[4] = {av.x, av.y, av.z, av.w}, br[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(ar[i], br[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int m = m0 + ty * 4 + i;
        if (m >= M) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = n0 + tx * 4 + j;
            if (n < Nn) c[(size_t)m * ldc + n] = acc[i][j];
        }
    }
}

// dx[t, i] += sum_k dx_perm[slot(t, k), i] (kept slots, k order) + dx_shared[t, i].
__global__ void __launch_bounds__(kThreads)
dx_gather_kernel(const float *__restrict__ dx_perm, const int32_t *__restrict__ slot_of,
                 const float *__restrict__ dx_shared, int K, int d, float *__restrict__ dx) {
    const int t = blockIdx.x;
    float *o = dx + (size_t)t * d;
    for (int i = threadIdx.x; i < d; i += kThreads) {
        float acc = dx_shared ? dx_shared[(size_t)t * d + i] : 0.f;
        for (int k = 0; k < K; ++k) {
            const int r = slot_of[(size_t)t * K + k];
            if (r >= 0) acc += dx_perm[(size_t)r * d + i];
        }
        o[i] += acc;
    }
}

}  // namespace bwd
}  // namespace moe
