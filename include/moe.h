/*
 * moe.h -- C ABI of libmoe.so: the forward pass of one Mixture-of-Experts
 * layer on one NVIDIA B300 (sm_103a).
 *
 * The layer (as the MoE pages define it):
 *   logits  s = W_g x                       (one linear map, no bias)
 *   select  the K largest of s (+ optional selection bias b), ties to the
 *           lower expert id
 *   weights softmax over only the K kept, unbiased logits
 *   dispatch token order -> one contiguous block per expert, at most
 *           capacity = ceil(T / N * capacity_factor) tokens per expert, the
 *           rest dropped (they pass through the residual outside the layer);
 *           which ones survive: earlier tokens first, or (drop_policy)
 *           earlier ranks first
 *   experts E_e(x) = Linear(d_model -> d_ff) -> GELU -> Linear(d_ff -> d_model)
 *   combine y[t] = z[t] + sum_k w[t,k] E_{idx[t,k]}(x[t]) in fixed k order
 *           (z = optional always-on shared expert, weight 1)
 *   aux     alpha * N * sum_i f_i P_i (Switch-style balance loss)
 *   z-loss  beta * mean_t logsumexp(s_t)^2 (router logit magnitude penalty)
 * Sources: lmnt.cn/news/351908 (sec. 2.1 score equation, sec. 3.1-3.3
 * dispatch/combine/capacity, sec. 5.1-5.2 balance loss); "MoE混合专家模型实战：
 * 专家路由与稀疏激活的推理成本优化方案" (yunthe.com: output equation, expert
 * FFN listing, selection bias b_i); "MoE 专家路由如何实现稀疏激活" (wiblog.cn:
 * shared expert).
 *
 * Conventions for every entry point
 *  - Tensors are row-major. bf16 tensors are passed as moe_bf16 (raw bits).
 *    Weights use the nn.Linear layout [out, in], so the reduction dimension is
 *    contiguous for both operands of every matrix product.
 *  - Every tensor pointer is caller-owned DEVICE memory unless its comment says
 *    HOST. The library allocates and frees nothing and keeps no per-call state;
 *    scratch comes from the caller's workspace (see moe_workspace_bytes).
 *  - All work is enqueued asynchronously on `stream` (a cudaStream_t, NULL =
 *    legacy default stream). Outputs are valid once the stream reaches that
 *    point. No entry point synchronises except moe_get_device_error.
 *  - Errors: arguments are validated on the host before anything is enqueued.
 *    MOE_ERR_INVALID_ARG: a NULL required pointer, a non-positive size,
 *    K > N, a misaligned pointer (bf16/fp32 tensors need 16-byte alignment).
 *    MOE_ERR_UNSUPPORTED: d_model or d_ff not a multiple of 64, K > 8,
 *    N > 1024, ceil(T * K / 128) + N > 65535. MOE_ERR_WORKSPACE: workspace NULL or smaller than
 *    required. MOE_ERR_CUDA: a CUDA launch error (the CUDA error is consumed).
 *  - Device-side consistency checks (an expert id outside [0, N), a row index
 *    outside its buffer, a pipeline wait that exceeds its time limit) never
 *    trap: the offending element is skipped and a bit is set in a device error
 *    word that moe_get_device_error reads.
 *  - Inputs must be finite. Results on NaN or Inf inputs are unspecified.
 *  - Kernel variants (environment variables read once per process; every
 *    variant computes the same function and passes the same parity tests,
 *    the defaults are the measured fastest): MOE_GEMM_VARIANT=pair (bf16
 *    expert GEMM on SM pairs, cta_group::2, 256-row tiles); MOE_ROUTE_VARIANT=
 *    legacy (gate GEMM + TopK + finalize kernels for every N instead of the
 *    fused router for N <= 256); MOE_FP8_GEMM=token_major (FP8 expert GEMM
 *    with token rows as the MMA's M and the weights widened in shared memory
 *    instead of the channel-major kernel).
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

typedef uint16_t moe_bf16; /* bfloat16 bit pattern */

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,
    MOE_ERR_UNSUPPORTED = 2,
    MOE_ERR_WORKSPACE = 3,
    MOE_ERR_CUDA = 4,
    MOE_ERR_DEVICE = 5
} moe_status;

/* Device error word bits (moe_get_device_error). */
#define MOE_DEVERR_EXPERT_ID 0x1u   /* a top-k expert id outside [0, N) was skipped */
#define MOE_DEVERR_ROW_INDEX 0x2u   /* a slot / row index outside its buffer was skipped */
#define MOE_DEVERR_TIMEOUT   0x4u   /* a GEMM pipeline wait ran out; that tile was abandoned */
#define MOE_DEVERR_TILE_LIST 0x8u   /* the expert offsets were inconsistent; tiles were skipped */

/* Problem statement (lmnt.cn/news/351908 sec. 2.1 and 3.3; selection bias and
 * shared expert from the yunthe.com and wiblog.cn pages). */
typedef struct {
    int32_t T;               /* tokens in the batch */
    int32_t d_model;         /* hidden size (multiple of 64) */
    int32_t d_ff;            /* expert inner size (multiple of 64) */
    int32_t N;               /* routed experts (1..1024) */
    int32_t K;               /* experts per token (1..min(8, N)) */
    float capacity_factor;   /* <= 0: dropless, capacity = T */
    int32_t has_shared;      /* 1: one always-on shared expert of shape (d_model, d_ff) */
    float aux_alpha;         /* balance-loss coefficient alpha */
    float z_beta;            /* router z-loss coefficient beta (lmnt.cn/news/351908 sec. 5.3) */
    int32_t drop_policy;     /* which assignments a full expert keeps: MOE_DROP_TOKEN_ORDER
                                (earlier tokens first) or MOE_DROP_RANK_ORDER (every token's
                                first choice before any second choice, ...) */
    float kl_coef;           /* coefficient of the KL(uniform || f) balance loss variant */
} moe_shape;

#define MOE_DROP_TOKEN_ORDER 0
#define MOE_DROP_RANK_ORDER 1

#define MOE_WEIGHTS_BF16 0
#define MOE_WEIGHTS_FP8_E4M3 1
#define MOE_WEIGHTS_INT4_G128 2

/* Layer weights, all DEVICE pointers. */
typedef struct {
    const moe_bf16 *Wg;   /* [N, d_model]         gate */
    const moe_bf16 *W1;   /* [N, d_ff, d_model]   expert first Linear */
    const float *b1;      /* [N, d_ff] */
    const moe_bf16 *W2;   /* [N, d_model, d_ff]   expert second Linear */
    const float *b2;      /* [N, d_model] */
    const moe_bf16 *Ws1;  /* [d_ff, d_model] shared expert (NULL unless has_shared) */
    const float *bs1;     /* [d_ff] */
    const moe_bf16 *Ws2;  /* [d_model, d_ff] */
    const float *bs2;     /* [d_model] */
    /* Expert weight format. MOE_WEIGHTS_BF16 (0): W1, W2, Ws1, Ws2 above.
     * MOE_WEIGHTS_FP8_E4M3: weight-only quantised experts (the 8/4-bit expert
     * weights of lmnt.cn/news/351908 sec. 4.3 and the one-byte FP8 weights of
     * the CSDN "MoE逐token路由与活跃参数率实战解析" sec. 3.2): the bf16 expert
     * matrices are ignored (may be NULL) and each is given as FP8 E4M3 codes
     * (the "e4m3fn" encoding) in the same nn.Linear layout with one fp32 scale
     * per output channel; the dequantised weight is code value * scale. The
     * gate W_g and all biases stay as above. NaN codes (0x7f, 0xff) are not
     * supported.
     * MOE_WEIGHTS_INT4_G128: weight-only 4-bit experts (the 4-bit expert
     * weights of lmnt.cn/news/351908 sec. 4.3; the yunthe.com page measures a
     * 4-bit Mixtral): W1q / W2q / Ws1q / Ws2q hold 4-bit codes along the
     * reduction dimension, half a byte each: the eight columns 8m .. 8m + 7
     * of a row form one little-endian 32-bit word (bytes 4m .. 4m + 3 of the
     * row) with column 8m + 2j in bits 4j .. 4j + 3 and column 8m + 2j + 1 in
     * bits 16 + 4j .. 19 + 4j, j = 0 .. 3 (so the bytes hold the column pairs
     * (0, 2), (4, 6), (1, 3), (5, 7), low nibble first); code c stands for the
     * integer c - 8. Shapes [N, d_ff, d_model / 2], [N, d_model, d_ff / 2],
     * [d_ff, d_model / 2], [d_model, d_ff / 2]; g1 / g2 / gs1 / gs2 hold one
     * bf16 scale per output channel and group of 128 consecutive reduction
     * columns, group-major: [N, d_model / 128, d_ff], [N, d_ff / 128, d_model],
     * [d_model / 128, d_ff], [d_ff / 128, d_model]. The dequantised weight is
     * (c - 8) * scale rounded once to bf16 (round to nearest even). s1, s2,
     * ss1, ss2 are ignored. d_model and d_ff must be multiples of 128
     * (MOE_ERR_UNSUPPORTED otherwise). */
    int32_t format;
    const uint8_t *W1q;   /* FP8 [N, d_ff, d_model]; INT4 [N, d_ff, d_model / 2] */
    const float *s1;      /* FP8 [N, d_ff] */
    const uint8_t *W2q;   /* FP8 [N, d_model, d_ff]; INT4 [N, d_model, d_ff / 2] */
    const float *s2;      /* FP8 [N, d_model] */
    const uint8_t *Ws1q;  /* (has_shared) FP8 [d_ff, d_model]; INT4 [d_ff, d_model / 2] */
    const float *ss1;     /* FP8 [d_ff] */
    const uint8_t *Ws2q;  /* FP8 [d_model, d_ff]; INT4 [d_model, d_ff / 2] */
    const float *ss2;     /* FP8 [d_model] */
    const moe_bf16 *g1;   /* INT4 [N, d_model / 128, d_ff] */
    const moe_bf16 *g2;   /* INT4 [N, d_ff / 128, d_model] */
    const moe_bf16 *gs1;  /* INT4 (has_shared) [d_model / 128, d_ff] */
    const moe_bf16 *gs2;  /* INT4 (has_shared) [d_ff / 128, d_model] */
} moe_weights;

/* Gradients written by moe_backward, all DEVICE fp32 buffers in the layout
 * of the corresponding parameter (each is overwritten, not accumulated). */
typedef struct {
    float *dx;            /* [T, d_model] */
    float *dWg;           /* [N, d_model] */
    float *dW1;           /* [N, d_ff, d_model] */
    float *db1;           /* [N, d_ff] */
    float *dW2;           /* [N, d_model, d_ff] */
    float *db2;           /* [N, d_model] */
    float *dWs1;          /* [d_ff, d_model] (has_shared) */
    float *dbs1;          /* [d_ff] */
    float *dWs2;          /* [d_model, d_ff] */
    float *dbs2;          /* [d_model] */
    float *dw;            /* [T, K] gradient of the routing weights (optional, NULL) */
} moe_grads;

/* Optional outputs of moe_forward, all DEVICE pointers; any member may be NULL
 * (the value is then kept in the workspace only). */
typedef struct {
    int32_t *topk_idx;       /* [T, K] selected experts, rank order */
    float *topk_w;           /* [T, K] routing weights (sum to 1 per token) */
    int32_t *demand;         /* [N] assignments per expert before capacity */
    float *prob_sum;         /* [N] sum over tokens of softmax over all N logits */
    int32_t *kept;           /* [N] min(demand, capacity) */
    int32_t *expert_offsets; /* [N + 1] exclusive prefix sum of kept */
    int32_t *slot_of;        /* [T, K] row of (t, k) in the per-expert blocks, -1 = dropped */
    float *aux;              /* [1] balance loss */
    float *z_loss;           /* [1] router z-loss beta * (1/T) * sum_t logsumexp(s_t)^2
                                (lmnt.cn/news/351908 sec. 5.3): fp32 per token, per-block fp32
                                partial sums added in block order with compensated (Neumaier)
                                fp32 summation */
    float *aux_kl;           /* [1] kl_coef * sum_e (1/N) (log(1/N) - log f_e), f_e = demand_e/(T K)
                                (KL-to-uniform balance loss of the CSDN MoELayer listing);
                                +inf when an expert receives nothing */
    float *health;           /* [4] router health statistics (lmnt.cn/news/351908 sec. 8.2 and
                                9.3 monitors; the CSDN page's sec. 3.3 expert_util_std):
                                [0] population std over experts of f_e = demand_e / (T K),
                                [1] fraction of the T K assignments dropped by capacity,
                                [2] mean routing entropy (nats) of the full softmax,
                                [3] max |gate logit| */
    float *mean_weight;      /* [N] mean routing weight of the assignments to each expert
                                (0 for an idle expert) */
} moe_route_out;

/* Workspace sizes. */
typedef enum {
    MOE_WS_FORWARD = 0,  /* moe_forward and moe_forward_hostio */
    MOE_WS_ROUTE = 1,    /* moe_route */
    MOE_WS_DISPATCH = 2, /* moe_dispatch */
    MOE_WS_FFN = 3,      /* moe_expert_ffn */
    MOE_WS_BACKWARD = 4  /* moe_backward */
} moe_ws_kind;

/* capacity = ceil(T / N * capacity_factor), evaluated in double, clamped to
 * [0, T]; T when capacity_factor <= 0 (lmnt.cn/news/351908 sec. 3.3 capacity
 * equation). Returns -1 for an invalid shape. */
MOE_API int32_t moe_capacity(const moe_shape *shape);

/* Bytes of workspace the given entry point needs for this shape (0 for an
 * invalid shape). Workspace must be 256-byte aligned device memory. */
MOE_API size_t moe_workspace_bytes(const moe_shape *shape, int32_t kind);

MOE_API const char *moe_status_string(int32_t status);

/* Gate and routing (lmnt.cn/news/351908 sec. 2.1: score = Softmax(TopK(W_g x));
 * selection bias b_i from yunthe.com; statistics for the balance loss, sec. 5.2).
 *   x        [T, d_model] bf16
 *   Wg       [N, d_model] bf16
 *   sel_bias [N] fp32 or NULL; added to the logits for the selection only
 * Outputs:
 *   topk_idx [T, K] int32   experts ordered by (s + b) descending, id ascending
 *   topk_w   [T, K] fp32    softmax over the K selected unbiased logits
 *   demand   [N] int32      count of (t, k) with topk_idx == e
 *   prob_sum [N] fp32       sum over t of softmax over all N unbiased logits
 * Logits are fp32 sums of bf16 products (exact when inputs lie on the 1/64
 * grid the tests use). Deterministic: no floating-point atomics. */
MOE_API moe_status moe_route(const moe_shape *shape, const moe_bf16 *x, const moe_bf16 *Wg,
                     const float *sel_bias, int32_t *topk_idx, float *topk_w, int32_t *demand,
                     float *prob_sum, void *workspace, size_t workspace_bytes, void *stream);

/* moe_route without a caller workspace. The pages have no counterpart of
 * this entry point; it exists for callers that cannot hand the library device
 * scratch memory (a plugin whose host framework plans all device memory up
 * front and has no slot for per-operator scratch, or a latency-critical loop
 * that must not call cudaMalloc once it runs, since cudaMalloc can
 * synchronise the device and can fail when memory is fragmented).
 * Same arguments (minus the workspace), outputs and results as moe_route.
 * Scratch: one fixed 8 MiB array inside libmoe.so's device memory, present
 * on every GPU that loads the library until the process exits. A shape may
 * use it when moe_workspace_bytes(shape, MOE_WS_ROUTE) <= 8 MiB; larger
 * shapes return MOE_ERR_UNSUPPORTED. The function allocates
 * nothing: no cudaMalloc, cudaFree or allocating library call.
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture. Only a successful lookup is kept: if the first
 * call fails (MOE_ERR_CUDA), a later call on that device retries it. All calls share the one array: calls whose work
 * overlaps on the GPU (different streams, or different host threads on one
 * device) race on it and must be serialised by the caller. */
MOE_API moe_status moe_route_noalloc(const moe_shape *shape, const moe_bf16 *x, const moe_bf16 *Wg,
                                     const float *sel_bias, int32_t *topk_idx, float *topk_w,
                                     int32_t *demand, float *prob_sum, void *stream);

/* Dispatch (lmnt.cn/news/351908 sec. 3.1 regroup by expert, sec. 3.3 capacity):
 * assignment (t, k) with e = topk_idx[t, k] gets position p = number of
 * earlier tokens t' < t that also chose e; it is kept iff p < capacity and
 * then lives at row expert_offsets[e] + p of the regrouped buffer.
 *   topk_idx [T, K] int32; x [T, d_model] bf16
 * Outputs:
 *   kept [N], expert_offsets [N + 1], slot_of [T, K] (-1 = dropped),
 *   row_token [T * K] (token of each kept row; -1 past the last kept row),
 *   x_perm [T * K, d_model] bf16 (rows >= expert_offsets[N] are untouched).
 * Bit-exact and deterministic (integer work only). */
MOE_API moe_status moe_dispatch(const moe_shape *shape, const int32_t *topk_idx, const moe_bf16 *x,
                        int32_t *kept, int32_t *expert_offsets, int32_t *slot_of,
                        int32_t *row_token, moe_bf16 *x_perm, void *workspace,
                        size_t workspace_bytes, void *stream);

/* Expert FFNs as grouped GEMMs on the tensor cores (yunthe.com MoELayer
 * listing: Linear -> GELU -> Linear per expert; grouped-GEMM remark there):
 *   for every row r of expert e's block [expert_offsets[e], expert_offsets[e+1]):
 *     h = bf16(GELU(x_perm[r] W1[e]^T + b1[e]))      (erf GELU, fp32 epilogue)
 *     y_perm[r] = bf16(h W2[e]^T + b2[e])            (fp32 accumulation)
 *   with has_shared, also z[t] = the same FFN with Ws1/bs1/Ws2/bs2 on x[t].
 *   x_perm [T * K, d_model] bf16, expert_offsets [N + 1] int32 (device)
 *   x [T, d_model] bf16 (read only when has_shared)
 * Outputs: y_perm [T * K, d_model] bf16 (rows >= expert_offsets[N] untouched),
 *          z_shared [T, d_model] bf16 (required iff has_shared). */
MOE_API moe_status moe_expert_ffn(const moe_shape *shape, const moe_bf16 *x_perm,
                          const int32_t *expert_offsets, const moe_weights *weights,
                          const moe_bf16 *x, moe_bf16 *y_perm, moe_bf16 *z_shared,
                          void *workspace, size_t workspace_bytes, void *stream);

/* Combine (lmnt.cn/news/351908 sec. 3.2 combine equation; same order as the
 * dispatch): y[t] = bf16(z[t] + sum_{k=0..K-1, slot_of[t,k] >= 0}
 *                        topk_w[t,k] * y_perm[slot_of[t,k]]), fp32 accumulation
 * in increasing k. z_shared may be NULL (then z = 0).
 *   y_perm [rows, d_model] bf16 with rows = T * K; slot_of [T, K]; topk_w [T, K]
 * Output: y [T, d_model] bf16. */
MOE_API moe_status moe_combine(const moe_shape *shape, const moe_bf16 *y_perm, const int32_t *slot_of,
                       const float *topk_w, const moe_bf16 *z_shared, moe_bf16 *y, void *stream);

/* Balance loss (lmnt.cn/news/351908 sec. 5.1 equation and sec. 5.2 code):
 *   aux = alpha * N * sum_e (demand[e] / (T K)) * (prob_sum[e] / T)
 * demand [N] int32, prob_sum [N] fp32 (as moe_route writes them);
 * aux [1] fp32 DEVICE. Evaluated in double, stored fp32. */
MOE_API moe_status moe_aux_loss(const moe_shape *shape, const int32_t *demand, const float *prob_sum,
                        float *aux, void *stream);

/* The whole layer: route -> dispatch -> expert FFN -> combine -> aux, all
 * enqueued on `stream`, no host synchronisation.
 *   x [T, d_model] bf16, sel_bias [N] fp32 or NULL, y [T, d_model] bf16.
 *   out may be NULL. workspace >= moe_workspace_bytes(shape, MOE_WS_FORWARD). */
MOE_API moe_status moe_forward(const moe_shape *shape, const moe_weights *weights, const moe_bf16 *x,
                       const float *sel_bias, moe_bf16 *y, const moe_route_out *out,
                       void *workspace, size_t workspace_bytes, void *stream);

/* moe_forward that also records timing marks on `stream`: events[i] is a
 * cudaEvent_t created by the caller (a NULL entry is skipped), recorded
 *   0 before routing, 1 after routing (with the aux loss), 2 after dispatch,
 *   3 after the first grouped GEMM (tile list, x W1^T, shared expert's first
 *     Linear), 4 after the second grouped GEMM, 5 after combine.
 * events must point to 6 entries. The kernels launched are those of
 * moe_forward (which computes the aux loss inside its routing stage). */
MOE_API moe_status moe_forward_marked(const moe_shape *shape, const moe_weights *weights, const moe_bf16 *x,
                                      const float *sel_bias, moe_bf16 *y, const moe_route_out *out,
                                      void *workspace, size_t workspace_bytes, void *const *events,
                                      void *stream);

/* moe_forward with the token batch in HOST memory: copies x_host -> x_dev,
 * runs the layer, copies y_dev -> y_host, all asynchronously on `stream`
 * (use pinned host buffers for overlap; the copies are complete once the
 * stream is). x_dev and y_dev are caller-owned DEVICE buffers of T * d_model
 * bf16 each. */
MOE_API moe_status moe_forward_hostio(const moe_shape *shape, const moe_weights *weights,
                              const moe_bf16 *x_host, moe_bf16 *x_dev, const float *sel_bias,
                              moe_bf16 *y_dev, moe_bf16 *y_host, const moe_route_out *out,
                              void *workspace, size_t workspace_bytes, void *stream);

/* Host-to-host forward over a sequence of nbatch batches of T tokens with the
 * transfers overlapped: batch i is read from x_host + i * host_stride and
 * written to y_host + i * host_stride (host_stride in elements; 0 = the same
 * host buffers for every batch); host buffers should be pinned. x_dev and
 * y_dev each hold TWO device buffers of [T, d_model] bf16 (double buffering).
 * The copies run on two copy streams owned by the library and are ordered
 * against the forwards on `stream` with events, so batch i+1's input copy and
 * batch i-1's output copy overlap batch i's forward. Asynchronous: every copy
 * and forward has finished once `stream` has. One call at a time per device
 * (a mutex serialises callers). workspace as for moe_forward. */
MOE_API moe_status moe_forward_hostio_batches(const moe_shape *shape, const moe_weights *weights, int32_t nbatch,
                                              const moe_bf16 *x_host, moe_bf16 *y_host, size_t host_stride,
                                              const float *sel_bias, moe_bf16 *x_dev, moe_bf16 *y_dev,
                                              void *workspace, size_t workspace_bytes, void *stream);

/* Backward pass of the layer (training; the pages' sec. 5 training signal,
 * lmnt.cn/news/351908). Recomputes the forward for (x, sel_bias) and writes
 * the gradients of
 *     L = <dy, y> + g_aux * aux + g_z * z_loss
 * with respect to x and every weight and bias, for the forward's routing
 * decisions (TopK sets, capacity drops and dispatch are piecewise constant:
 * no gradient flows through them, through sel_bias or the KL variant):
 *   combine   dw_tk = <dy_t, o_tk> (0 when dropped), dO = bf16(w_tk dy_t)
 *   experts   dh = dO W2, da = bf16(dh * GELU'(a)) with a = x W1^T + b1,
 *             dW2 = dO^T h, db2 = sum dO, dW1 = da^T x, db1 = sum da,
 *             dx += da W1 through the dispatch; shared expert with dO = dy
 *   gate      ds_t = w (dw - <w, dw>) on the TopK set (softmax over the kept
 *             logits, sec. 2.1) + g_aux alpha N / T p (f - <f, p>) + g_z 2 beta
 *             / T lse p (sec. 5.2-5.3), dWg = ds^T x, dx += ds Wg
 * dO and da are stored in bf16 between the tensor-core GEMMs, every other
 * intermediate and every gradient in fp32. dy: [T, d_model] bf16 (device).
 * grads: see moe_grads. BF16 expert weights only (FP8, INT4: MOE_ERR_UNSUPPORTED).
 * workspace >= moe_workspace_bytes(shape, MOE_WS_BACKWARD). Asynchronous on
 * `stream`. */
MOE_API moe_status moe_backward(const moe_shape *shape, const moe_weights *weights, const moe_bf16 *x,
                                const float *sel_bias, const moe_bf16 *dy, float g_aux, float g_z,
                                const moe_grads *grads, void *workspace, size_t workspace_bytes, void *stream);

/* Reads (and, if clear != 0, resets) the device error word of the current
 * device. Synchronises the device. *code_out receives the MOE_DEVERR_* bits. */
MOE_API moe_status moe_get_device_error(int32_t clear, int32_t *code_out);

/* Number of kernels this library has launched in this process (all devices,
 * all threads). Used to count launches inside a timed region. */
MOE_API uint64_t moe_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
