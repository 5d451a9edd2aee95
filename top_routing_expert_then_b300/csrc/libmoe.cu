// libmoe.cu -- the C ABI of include/moe.h: host-side validation, workspace
// layout and kernel launches for the MoE layer forward pass on sm_103a.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <initializer_list>
#include <mutex>

#include "../../include/moe.h"
#include "common.cuh"
#include "dispatch.cuh"
#include "grouped_gemm.cuh"
#include "route.cuh"
#include "route_tc.cuh"
#include "gemm_fp8w.cuh"
#include "gemm_quant.cuh"
#include "backward.cuh"
#include "plan.cuh"

namespace {

using moe::gg::BM;

std::atomic<uint64_t> g_launches{0};

inline void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

inline cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr size_t kAlign = 256;
inline size_t align_up(size_t v) { return (v + kAlign - 1) & ~(kAlign - 1); }

// Sequential carve of a workspace (or, with base == nullptr, only its size).
struct Carve {
    char *base;
    size_t off = 0;
    explicit Carve(void *b) : base(static_cast<char *>(b)) {}
    template <typename T>
    T *take(size_t count) {
        off = align_up(off);
        T *p = base ? reinterpret_cast<T *>(base + off) : nullptr;
        off += count * sizeof(T);
        return p;
    }
    size_t bytes() const { return align_up(off); }
};

// ------------------------------------------------------------------ shape checks

moe_status check_shape(const moe_shape *s) {
    if (s == nullptr) return MOE_ERR_INVALID_ARG;
    if (s->T <= 0 || s->d_model <= 0 || s->d_ff <= 0 || s->N <= 0 || s->K <= 0)
        return MOE_ERR_INVALID_ARG;
    if (s->K > s->N) return MOE_ERR_INVALID_ARG;
    if (std::isnan(s->capacity_factor) || std::isnan(s->aux_alpha) || std::isnan(s->z_beta)) return MOE_ERR_INVALID_ARG;
    if (s->has_shared != 0 && s->has_shared != 1) return MOE_ERR_INVALID_ARG;
    if (s->drop_policy != MOE_DROP_TOKEN_ORDER && s->drop_policy != MOE_DROP_RANK_ORDER) return MOE_ERR_INVALID_ARG;
    if (std::isnan(s->kl_coef)) return MOE_ERR_INVALID_ARG;
    if (s->d_model % 64 != 0 || s->d_ff % 64 != 0) return MOE_ERR_UNSUPPORTED;
    if (s->K > moe::route::kMaxK || s->N > 1024) return MOE_ERR_UNSUPPORTED;
    if ((int64_t)s->T * s->K >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
    if ((int64_t)s->N * s->d_ff >= (int64_t(1) << 31) || (int64_t)s->N * s->d_model >= (int64_t(1) << 31))
        return MOE_ERR_UNSUPPORTED;
    if (((int64_t)s->T * s->K + 127) / 128 + s->N > 65535) return MOE_ERR_UNSUPPORTED;  // m-tile list index
    return MOE_OK;
}

int capacity_of(const moe_shape *s) {
    // lmnt.cn/news/351908 sec. 3.3: capacity = ceil(T / N * capacity_factor)
    if (s->capacity_factor <= 0.f) return s->T;
    double c = std::ceil((double)s->T / (double)s->N * (double)s->capacity_factor);
    if (c > (double)s->T) c = (double)s->T;
    if (c < 0.0) c = 0.0;
    return (int)c;
}

// Capacity of the device tile list: m-tiles of 64 rows (the FP8 kernel's
// height; the bf16 kernels' 128- and 256-row tiles need fewer).
// m-tiles of the smallest height any kernel uses (32 rows): an expert's block
// of r rows takes at most r / 32 + 1 of them
int max_mtiles(const moe_shape *s) {
    return (int)(((int64_t)s->T * s->K + 31) / 32) + s->N;
}

// ------------------------------------------------------------------ workspace layouts

struct RouteWs {
    float *logits;                 // general path: gate logits (K-split planes)
    float *partial;                // general path: per-block probability sums
    float *lse_partial;            // per-block sums of logsumexp^2, entropy, max |logit|
    unsigned long long *wacc;      // general path: fixed-point routing-weight sums (zeroed per call)
    unsigned int *done;            // general path: finished-block ticket (zeroed per call)
    int32_t *tile_hist;            // fused path: per 128-token tile, [tiles][N] assignments
    unsigned long long *tile_prob; // fused path: [tiles][N] fixed-point probability sums
    unsigned long long *tile_w;    // fused path: [tiles][N] fixed-point routing-weight sums
};

// Routing for N <= 256 runs as one fused kernel (tensor-core gate, TopK,
// softmax, statistics and losses). N > 256 takes the general path: gate GEMM
// (tensor cores when N % 32 == 0, else CUDA-core tiles) + TopK kernel +
// finalize kernel; MOE_ROUTE_VARIANT=legacy (environment, read once) selects
// the general path for every N.
bool legacy_route() {
    static const bool v = []() {
        const char *e = std::getenv("MOE_ROUTE_VARIANT");
        return e != nullptr && std::strcmp(e, "legacy") == 0;
    }();
    return v;
}
bool fused_route(const moe_shape *s) { return s->N <= moe::rtc::kMaxN && !legacy_route(); }
int fused_route_grid(const moe_shape *s) {
    return moe::rtc::num_tiles(s->T) * moe::rtc::splits(s->T, s->d_model);
}

// General path: the gate runs on the tensor cores (grouped GEMM, fp32 output)
// when N > 16 and N % 32 == 0; with few 128 x 256 tiles it splits K so that
// about one wave of blocks (148 SMs) has work. The split count depends on the
// shape only, so results are the same on every device.
bool tensor_gate(const moe_shape *s) { return s->N > 16 && s->N % 32 == 0; }

int gate_splits(const moe_shape *s) {
    if (!tensor_gate(s)) return 1;
    const int64_t tiles = (int64_t)((s->T + 127) / 128) * ((s->N + 255) / 256);
    int64_t sp = 148 / (tiles > 0 ? tiles : 1);
    if (sp > 4) sp = 4;
    if (sp < 1) sp = 1;
    const int kb = s->d_model / 64;
    // no empty split: every split keeps at least one 64-wide k-block
    const int per = (int)((kb + sp - 1) / sp);
    return (kb + per - 1) / per;
}

RouteWs carve_route(Carve &c, const moe_shape *s) {
    RouteWs w{};
    if (fused_route(s)) {
        const size_t tiles = (size_t)moe::rtc::num_tiles(s->T);
        w.lse_partial = c.take<float>((size_t)fused_route_grid(s) * moe::route::kPartialStride);
        w.tile_hist = c.take<int32_t>(tiles * s->N);
        w.tile_prob = c.take<unsigned long long>(tiles * s->N);
        w.tile_w = c.take<unsigned long long>(tiles * s->N);
        return w;
    }
    w.logits = c.take<float>((size_t)gate_splits(s) * s->T * s->N);
    w.partial = c.take<float>((size_t)moe::route::kMaxPartialRows * s->N);
    w.lse_partial = c.take<float>((size_t)moe::route::kMaxPartialRows * moe::route::kPartialStride);
    w.wacc = c.take<unsigned long long>(s->N);
    w.done = c.take<unsigned int>(4);
    return w;
}

struct DispatchWs {
    int32_t *hist;
    int32_t *base;
};
DispatchWs carve_dispatch(Carve &c, const moe_shape *s) {
    DispatchWs w;
    size_t n = (size_t)moe::dispatch::num_chunks(s->T * s->K) * s->N;  // enough for either priority
    w.hist = c.take<int32_t>(n);
    w.base = c.take<int32_t>(n);
    return w;
}

// FP8 split-K partial sums: batches of at most kSplitRows routed rows (decode)
// get kMaxFp8Splits fp32 planes of [rows, max(d_ff, d_model)].
constexpr int kSplitRows = 128;
constexpr int kMaxFp8Splits = 4;

struct FfnWs {
    int4 *mtiles;       // m-tile list of the first expert GEMM
    int *num_mtiles;
    int4 *mtiles2;      // of the second, when its tiles differ (SM-pair kernel)
    int *num_mtiles2;
    uint16_t *H;
    uint16_t *Hs;
    float *part;  // nullptr: no split-K
};
FfnWs carve_ffn(Carve &c, const moe_shape *s) {
    FfnWs w;
    w.mtiles = c.take<int4>((size_t)max_mtiles(s));
    w.num_mtiles = c.take<int>(4);
    w.mtiles2 = c.take<int4>((size_t)max_mtiles(s));
    w.num_mtiles2 = c.take<int>(4);
    w.H = c.take<uint16_t>((size_t)s->T * s->K * s->d_ff);
    w.Hs = s->has_shared ? c.take<uint16_t>((size_t)s->T * s->d_ff) : nullptr;
    const int64_t rows = (int64_t)s->T * s->K;
    w.part = rows <= kSplitRows
                 ? c.take<float>((size_t)kMaxFp8Splits * rows * (size_t)std::max(s->d_ff, s->d_model))
                 : nullptr;
    return w;
}

struct ForwardWs {
    RouteWs route;
    DispatchWs disp;
    FfnWs ffn;
    int32_t *topk_idx, *demand, *kept, *offsets, *slot_of, *row_token;
    float *topk_w, *prob_sum, *aux;
    uint16_t *x_perm, *y_perm, *z;
};
ForwardWs carve_forward(Carve &c, const moe_shape *s) {
    ForwardWs w;
    const size_t TK = (size_t)s->T * s->K;
    w.route = carve_route(c, s);
    w.disp = carve_dispatch(c, s);
    w.ffn = carve_ffn(c, s);
    w.topk_idx = c.take<int32_t>(TK);
    w.topk_w = c.take<float>(TK);
    w.demand = c.take<int32_t>(s->N);
    w.prob_sum = c.take<float>(s->N);
    w.kept = c.take<int32_t>(s->N);
    w.offsets = c.take<int32_t>((size_t)s->N + 1);
    w.slot_of = c.take<int32_t>(TK);
    w.row_token = c.take<int32_t>(TK);
    w.aux = c.take<float>(4);
    w.x_perm = c.take<uint16_t>(TK * s->d_model);
    w.y_perm = c.take<uint16_t>(TK * s->d_model);
    w.z = s->has_shared ? c.take<uint16_t>((size_t)s->T * s->d_model) : nullptr;
    return w;
}

// Backward workspace: the forward's, plus the recomputed pre-activations, the
// backward intermediates and the transposed, 64-padded activation copies the
// per-expert weight-gradient GEMMs reduce over (the weights are read as stored).
struct BackwardWs {
    ForwardWs fwd;
    int4 *mtiles;
    int *num_mtiles;
    float *A1, *DH, *DXP, *L, *DS, *dw;
    uint16_t *DA, *dO, *dOT, *HT, *DAT, *XPT;
    int32_t *poff;
    size_t ldp;  // columns of the padded transposed copies
    // shared expert
    float *As1, *DHs, *DXs;
    uint16_t *DAs, *dyT, *HsT, *DAsT, *xT;
    int32_t *soff, *spoff;
    size_t ldt;
};
BackwardWs carve_backward(Carve &c, const moe_shape *s) {
    BackwardWs w{};
    const size_t T = s->T, d = s->d_model, f = s->d_ff, N = s->N, R = (size_t)s->T * s->K;
    w.fwd = carve_forward(c, s);
    w.mtiles = c.take<int4>((size_t)max_mtiles(s));
    w.num_mtiles = c.take<int>(4);
    w.A1 = c.take<float>(R * f);
    w.DH = c.take<float>(R * f);
    w.DXP = c.take<float>(R * d);
    w.L = c.take<float>(T * N);
    w.DS = c.take<float>(T * N);
    w.dw = c.take<float>(R);
    w.DA = c.take<uint16_t>(R * f);
    w.dO = c.take<uint16_t>(R * d);
    w.ldp = (R + 63) / 64 * 64 + 64 * N;  // >= sum of the 64-padded groups; rows 16-byte aligned
    w.dOT = c.take<uint16_t>(d * w.ldp);
    w.HT = c.take<uint16_t>(f * w.ldp);
    w.DAT = c.take<uint16_t>(f * w.ldp);
    w.XPT = c.take<uint16_t>(d * w.ldp);
    w.poff = c.take<int32_t>(N + 1);
    if (s->has_shared) {
        w.ldt = (T + 63) / 64 * 64;
        w.As1 = c.take<float>(T * f);
        w.DHs = c.take<float>(T * f);
        w.DXs = c.take<float>(T * d);
        w.DAs = c.take<uint16_t>(T * f);
        w.dyT = c.take<uint16_t>(d * w.ldt);
        w.HsT = c.take<uint16_t>(f * w.ldt);
        w.DAsT = c.take<uint16_t>(f * w.ldt);
        w.xT = c.take<uint16_t>(d * w.ldt);
        w.soff = c.take<int32_t>(2);
        w.spoff = c.take<int32_t>(2);
    }
    return w;
}

size_t ws_bytes(const moe_shape *s, int kind) {
    Carve c(nullptr);
    switch (kind) {
        case MOE_WS_ROUTE: carve_route(c, s); break;
        case MOE_WS_DISPATCH: carve_dispatch(c, s); break;
        case MOE_WS_FFN: carve_ffn(c, s); break;
        case MOE_WS_FORWARD: carve_forward(c, s); break;
        case MOE_WS_BACKWARD: carve_backward(c, s); break;
        default: return 0;
    }
    return c.bytes();
}

moe_status check_ws(const moe_shape *s, int kind, void *ws, size_t bytes) {
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0)
        return MOE_ERR_WORKSPACE;
    if (bytes < ws_bytes(s, kind)) return MOE_ERR_WORKSPACE;
    return MOE_OK;
}

// ------------------------------------------------------------------ per-device state

constexpr int kMaxDevices = 64;
struct DeviceState {
    std::once_flag once;
    int num_sms = 0;
    cudaError_t init_err = cudaSuccess;
    // batched host I/O: two copy streams and per-buffer events, created on first use
    std::once_flag io_once;
    cudaError_t io_err = cudaSuccess;
    std::mutex io_mutex;
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t ev_start = nullptr, ev_in[2] = {}, ev_fwd[2] = {}, ev_out[2] = {};
};
DeviceState g_dev[kMaxDevices];

// The fused router instantiated per (lanes' experts, cluster size).
template <int L>
const void *fused_route_kernel_s(int S) {
    switch (S) {
        case 1: return (const void *)moe::rtc::route_tc_kernel<L, 1>;
        case 2: return (const void *)moe::rtc::route_tc_kernel<L, 2>;
        case 4: return (const void *)moe::rtc::route_tc_kernel<L, 4>;
        default: return (const void *)moe::rtc::route_tc_kernel<L, 8>;
    }
}
const void *fused_route_kernel(int lpl, int S) {
    if (lpl <= 1) return fused_route_kernel_s<1>(S);
    if (lpl <= 2) return fused_route_kernel_s<2>(S);
    if (lpl <= 4) return fused_route_kernel_s<4>(S);
    return fused_route_kernel_s<8>(S);
}


moe_status device_state(DeviceState **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    DeviceState &st = g_dev[dev];
    std::call_once(st.once, [&st, dev]() {
        cudaError_t e = cudaDeviceGetAttribute(&st.num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(moe::gg::grouped_gemm_kernel<false>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, moe::gg::SMEM_BYTES);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(moe::gg::grouped_gemm_kernel<true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, moe::gg::SMEM_BYTES);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(moe::gg::grouped_gemm_pair_kernel,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, moe::gg::P_SMEM_BYTES);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(moe::gg::grouped_gemm_fp8w_kernel,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, moe::gg::Q_SMEM_BYTES);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(moe::gg::grouped_gemm_quant_kernel<moe::gg::QF_FP8>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, moe::gg::QT_SMEM_BYTES);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(moe::gg::grouped_gemm_quant_kernel<moe::gg::QF_INT4>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, moe::gg::QT_SMEM_BYTES);
        for (int lpl = 1; lpl <= 8; lpl <<= 1)
            for (int sp = 1; sp <= moe::rtc::kMaxSplits; sp <<= 1)
                if (e == cudaSuccess)
                    e = cudaFuncSetAttribute(fused_route_kernel(lpl, sp), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)moe::rtc::kMaxSmem);
        st.init_err = e;
    });
    if (st.init_err != cudaSuccess) return MOE_ERR_CUDA;
    *out = &st;
    return MOE_OK;
}

moe_status launch_status() {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// ------------------------------------------------------------------ TMA descriptors

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encoder() {
    std::call_once(g_encode_once, []() {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        cudaGetLastError();
    });
    return g_encode != nullptr;
}

// Row-major bf16 [rows, cols] tensor. Operand maps: box = box_rows x 64
// columns with the 128-byte swizzle the MMA descriptors expect. Output maps
// (epilogue TMA stores): box = 32 x 32, no swizzle.
bool make_tmap(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows,
               uint32_t box_cols = moe::gg::BK, bool swizzle128 = true) {
    if (!get_encoder()) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
                          box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Row-major fp32 [rows, cols] tensor (cols a multiple of 4): the raw
// accumulator planes the fp32 GEMM mode stores, 32 x 32 boxes with the
// 128-byte swizzle its epilogue buffers use.
bool make_tmap_f32(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols) {
    if (!get_encoder()) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 4};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Row-major one-byte [rows, cols] tensor (FP8 codes): box_rows x box_cols
// bytes land densely, rows box_cols bytes apart; with swizzle128 (box_cols =
// 128) the 16-byte chunks of row r are permuted by r % 8 as for bf16 tiles.
bool make_tmap_u8(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                  uint32_t box_cols, CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_NONE) {
    if (!get_encoder()) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// ------------------------------------------------------------------ stage launchers (no validation)

moe_status launch_gemm(DeviceState *dev, bool pair, const void *A, uint64_t a_rows_n, const void *B, uint64_t b_rows,
                       int k_dim, int n_out, int groups, const float *bias, uint16_t *out, int out_rows,
                       const int4 *mtiles, const int *num_mtiles, int max_tiles, int dense_rows, bool gelu,
                       cudaStream_t st, float *out_f32 = nullptr, int k_splits = 1, const int *k_ranges = nullptr,
                       const int32_t *a_rows = nullptr, bool b_mn = false);

// The dispatch plan the fused router's plan kernel also forms (forward path):
// per-chunk bases, kept counts, expert offsets and the grouped GEMMs' m-tile list.
using DispatchPlan = moe::plan::Dispatch;

moe::plan::Stats plan_stats(const moe_shape *s, const RouteWs &w, int32_t *demand, float *prob_sum, float *aux,
                            float *z_loss, float *aux_kl, float *health, float *mean_weight) {
    moe::plan::Stats q{};
    q.T = s->T;
    q.N = s->N;
    q.K = s->K;
    q.route_blocks = fused_route_grid(s);
    q.lse_partial = w.lse_partial;
    q.demand = demand;
    q.prob_sum = prob_sum;
    q.aux = aux;
    q.z_loss = z_loss;
    q.aux_kl = aux_kl;
    q.health = health;
    q.mean_weight = mean_weight;
    q.alpha = s->aux_alpha;
    q.beta = s->z_beta;
    q.kl_coef = s->kl_coef;
    return q;
}

moe_status run_route(const moe_shape *s, DeviceState *dev, const uint16_t *x, const uint16_t *Wg,
                     const float *sel_bias, int32_t *topk_idx, float *topk_w, int32_t *demand,
                     float *prob_sum, float *aux, const RouteWs &w, cudaStream_t st, float *z_loss = nullptr,
                     float *aux_kl = nullptr, float *health = nullptr, float *mean_weight = nullptr,
                     const DispatchPlan *dplan = nullptr) {
    const int T = s->T, d = s->d_model, N = s->N, K = s->K;
    if (fused_route(s)) {
        CUtensorMap tx, tw;
        if (!make_tmap(&tx, x, (uint64_t)T, (uint64_t)d, moe::rtc::kTile)) return MOE_ERR_CUDA;
        if (!make_tmap(&tw, Wg, (uint64_t)N, (uint64_t)d, (uint32_t)moe::rtc::npad(N))) return MOE_ERR_CUDA;
        moe::rtc::Params p;
        p.T = T;
        p.d = d;
        p.N = N;
        p.Npad = moe::rtc::npad(N);
        p.K = K;
        const int S = moe::rtc::splits(T, d);
        p.stages = moe::rtc::stages(T, d, N);
        p.l_offset = (uint32_t)moe::rtc::l_offset(T, d, N, p.stages);
        p.idesc = moe::rtc::idesc(N);
        p.tmem_cols = moe::rtc::tmem_cols(N);
        p.sel_bias = sel_bias;
        p.topk_idx = topk_idx;
        p.topk_w = topk_w;
        p.tile_hist = w.tile_hist;
        p.tile_prob = w.tile_prob;
        p.tile_w = w.tile_w;
        p.lse_partial = w.lse_partial;
        // a single-tile batch on the forward path: the router forms the plan itself
        const bool in_router = dplan != nullptr && moe::rtc::num_tiles(T) == 1;
        p.fuse_plan = in_router ? 1 : 0;
        p.st = plan_stats(s, w, demand, prob_sum, aux, z_loss, aux_kl, health, mean_weight);
        if (dplan != nullptr) p.dp = *dplan;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)fused_route_grid(s));
        cfg.blockDim = dim3(moe::rtc::kThreads);
        cfg.dynamicSmemBytes = moe::rtc::smem_bytes(T, d, N);
        cfg.stream = st;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = (unsigned)S;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        const int lpl = (p.Npad + 31) / 32;
        const void *fn = fused_route_kernel(lpl, S);
        void *args[] = {&tx, &tw, &p};
        cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
        count_launch();
        if (e != cudaSuccess) {
            cudaGetLastError();
            return MOE_ERR_CUDA;
        }
        if (in_router) return launch_status();
        // statistics and losses from the per-tile rows; on the forward path a
        // second block forms the dispatch plan and the m-tile lists meanwhile
        moe::plan::Params q{};
        q.st = plan_stats(s, w, demand, prob_sum, aux, z_loss, aux_kl, health, mean_weight);
        if (dplan != nullptr) q.dp = *dplan;
        q.tiles = moe::rtc::num_tiles(T);
        q.tile_hist = w.tile_hist;
        q.tile_prob = w.tile_prob;
        q.tile_w = w.tile_w;
        moe::plan::plan_kernel<<<dplan != nullptr ? 2 : 1, moe::plan::kThreads, 0, st>>>(q);
        count_launch();
        return launch_status();
    }
    const int splits = gate_splits(s);
    if (cudaMemsetAsync(demand, 0, sizeof(int32_t) * N, st) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemsetAsync(w.wacc, 0, sizeof(unsigned long long) * N, st) != cudaSuccess) return MOE_ERR_CUDA;
    if (tensor_gate(s)) {
        // logits = x Wg^T on the tensor cores, raw fp32 K-split partials
        moe_status g = launch_gemm(dev, false, x, (uint64_t)T, Wg, (uint64_t)N, d, N, 1, nullptr, nullptr, T,
                                   nullptr, nullptr, 0, T, false, st, w.logits, splits);
        if (g != MOE_OK) return g;
    } else {
        dim3 grid((T + moe::route::kGBM - 1) / moe::route::kGBM, (N + moe::route::kGBN - 1) / moe::route::kGBN);
        moe::route::gate_logits_tiled_kernel<<<grid, moe::route::kGateThreads, 0, st>>>(x, Wg, T, d, N, w.logits);
        count_launch();
    }
    const int rows = moe::route::topk_grid(T);
    const size_t smem = (size_t)N * sizeof(unsigned long long) + (size_t)moe::route::kTopkWarps * N * sizeof(float) +
                        (size_t)N * sizeof(int);
    const int lpl = (N + 31) / 32;
    const int thr = moe::route::kTopkWarps * 32;
#define MOE_TOPK(L)                                                                                     \
    moe::route::topk_softmax_kernel<L><<<rows, thr, smem, st>>>(w.logits, splits, sel_bias, T, N, K, topk_idx, \
                                                                topk_w, demand, w.partial, w.lse_partial, w.wacc)
    if (lpl <= 1) MOE_TOPK(1);
    else if (lpl <= 2) MOE_TOPK(2);
    else if (lpl <= 4) MOE_TOPK(4);
    else if (lpl <= 8) MOE_TOPK(8);
    else if (lpl <= 16) MOE_TOPK(16);
    else MOE_TOPK(32);
#undef MOE_TOPK
    count_launch();
    if ((aux != nullptr || z_loss != nullptr || aux_kl != nullptr || health != nullptr || mean_weight != nullptr) &&
        cudaMemsetAsync(w.done, 0, sizeof(unsigned int), st) != cudaSuccess)
        return MOE_ERR_CUDA;
    moe::route::route_finalize_kernel<<<(N + 31) / 32, 1024, 0, st>>>(
        w.partial, w.lse_partial, rows, N, T, K, s->aux_alpha, s->z_beta, s->kl_coef, demand, prob_sum, aux, z_loss,
        aux_kl, w.wacc, health, mean_weight, w.done);
    count_launch();
    return launch_status();
}

moe_status run_dispatch(const moe_shape *s, const int32_t *topk_idx, const uint16_t *x, int32_t *kept,
                        int32_t *offsets, int32_t *slot_of, int32_t *row_token, uint16_t *x_perm,
                        const DispatchWs &w, cudaStream_t st, float *drop_rate = nullptr, bool permute = true,
                        bool planned = false, bool placed = false) {
    const int T = s->T, N = s->N, K = s->K, d = s->d_model;
    const int C = capacity_of(s);
    const moe::dispatch::Order order{T, K, s->drop_policy == MOE_DROP_RANK_ORDER ? 1 : 0};
    const int chunks = moe::dispatch::num_chunks(order.rank_major ? T * K : T);
    const int rows = T * K;
    if (placed) {
        // the router has placed the assignments itself (a single-tile batch)
    } else if (planned) {
        // the router's plan kernel has formed w.base, kept and offsets (token order)
        moe::dispatch::assign_kernel<<<chunks, moe::dispatch::kChunk, 4 * N * sizeof(unsigned), st>>>(
            topk_idx, order, N, C, w.base, offsets, slot_of, row_token, rows);
        count_launch();
    } else if (chunks == 1) {
        // a decode-sized batch: count, scan and assign in one block
        moe::dispatch::dispatch_small_kernel<<<1, moe::dispatch::kChunk, (6 * (size_t)N + 1) * sizeof(int), st>>>(
            topk_idx, order, N, C, kept, offsets, slot_of, row_token, drop_rate, rows);
        count_launch();
    } else {
        moe::dispatch::count_kernel<<<chunks, moe::dispatch::kChunk, N * sizeof(int), st>>>(topk_idx, order, N,
                                                                                            w.hist);
        count_launch();
        moe::dispatch::scan_kernel<<<1, 1024, N * sizeof(int), st>>>(w.hist, chunks, N, C, w.base, kept, offsets,
                                                                     drop_rate, rows);
        count_launch();
        moe::dispatch::assign_kernel<<<chunks, moe::dispatch::kChunk, 4 * N * sizeof(unsigned), st>>>(
            topk_idx, order, N, C, w.base, offsets, slot_of, row_token, rows);
        count_launch();
    }
    if (permute) {
        const int vec = d / 8;
        const int thr = vec < 256 ? 64 : 256;
        dim3 grid((T + moe::dispatch::kRowTok - 1) / moe::dispatch::kRowTok, (vec + thr - 1) / thr);
        moe::dispatch::permute_kernel<<<grid, thr, 0, st>>>(x, slot_of, T, K, d, rows, x_perm);
        count_launch();
    }
    return launch_status();
}

// Which grouped-GEMM kernel runs. The SM-pair kernel (256-row tiles) cuts the
// operand traffic per SM by a third but pads each expert's last tile to 256
// rows; measured on the Mixtral-shaped layer it is slower than the single-SM
// kernel (128-row tiles), so the default is the single-SM kernel.
// MOE_GEMM_VARIANT=single|pair (environment, read once) forces one of them.
enum GemmVariant { kAuto = 0, kSingle = 1, kPair = 2 };
constexpr int kRasterSingle = 8;  // m-tiles (128 rows) per raster group
constexpr int kRasterPair = 4;    // m-tiles (256 rows) per raster group
int gemm_variant_override() {
    static const int v = []() {
        const char *e = std::getenv("MOE_GEMM_VARIANT");
        if (e == nullptr) return (int)kAuto;
        if (std::strcmp(e, "single") == 0) return (int)kSingle;
        if (std::strcmp(e, "pair") == 0) return (int)kPair;
        return (int)kAuto;
    }();
    return v;
}

bool use_pair(int64_t expected_rows_per_group) {
    const int o = gemm_variant_override();
    if (o == kSingle) return false;
    if (o == kPair) return true;
    (void)expected_rows_per_group;
    return false;
}

// The second expert GEMM on the SM-pair kernel by default when its tiles are
// long and the experts' blocks large: measured on the Mixtral-shaped prefill
// layer (about 1024 rows per expert, reduction 14336) it took 688 us against
// 748 us on the single-SM kernel; with 640-row blocks (capacity factor 1.25,
// each padded to 768) or a 4096-long reduction the single-SM kernel is faster.
bool use_pair_gemm2(int64_t expected_rows_per_group, int k_dim) {
    const int o = gemm_variant_override();
    if (o == kSingle) return false;
    if (o == kPair) return true;
    return expected_rows_per_group >= 1024 && k_dim >= 8192;
}

moe_status launch_gemm(DeviceState *dev, bool pair, const void *A, uint64_t a_rows_n, const void *B, uint64_t b_rows,
                       int k_dim, int n_out, int groups, const float *bias, uint16_t *out, int out_rows,
                       const int4 *mtiles, const int *num_mtiles, int max_tiles, int dense_rows, bool gelu,
                       cudaStream_t st, float *out_f32, int k_splits, const int *k_ranges, const int32_t *a_rows,
                       bool b_mn) {
    CUtensorMap ta, tb, tc, ta32;
    const uint32_t b_box = pair ? moe::gg::BN / 2 : moe::gg::BN;
    // fp32 mode, gathered A and an N-major B: single-SM kernel
    if (out_f32 != nullptr || a_rows != nullptr || b_mn) pair = false;
    if (!make_tmap(&ta, A, a_rows_n, (uint64_t)k_dim, 128)) return MOE_ERR_CUDA;
    if (b_mn) {  // B as stored: [groups * k_dim, n_out], 64 x 64 boxes
        (void)b_rows;
        if (!make_tmap(&tb, B, (uint64_t)groups * (uint64_t)k_dim, (uint64_t)n_out, 64, 64)) return MOE_ERR_CUDA;
    } else if (!make_tmap(&tb, B, b_rows, (uint64_t)k_dim, b_box)) {
        return MOE_ERR_CUDA;
    }
    if (out != nullptr) {
        if (!make_tmap(&tc, out, (uint64_t)out_rows, (uint64_t)n_out, 32, 32, false)) return MOE_ERR_CUDA;
    } else if (out_f32 != nullptr) {
        // fp32 mode: every split's plane, [k_splits * out_rows, n_out]
        if (!make_tmap_f32(&tc, out_f32, (uint64_t)k_splits * (uint64_t)out_rows, (uint64_t)n_out))
            return MOE_ERR_CUDA;
    } else {
        return MOE_ERR_INVALID_ARG;
    }
    moe::gg::Params p{};
    p.mtiles = mtiles;
    p.num_mtiles = num_mtiles;
    p.max_mtiles = max_tiles;
    p.dense_rows = dense_rows;
    p.n_out = n_out;
    p.k_dim = k_dim;
    p.num_groups = groups;
    p.out_rows = out_rows;
    p.bias = bias;
    p.out = out;
    p.gelu = gelu ? 1 : 0;
    p.out_f32 = out_f32;
    p.k_splits = k_splits;
    p.k_ranges = k_ranges;
    p.a_rows = a_rows;  // gathered A: the row-gather warp copies rows a_rows[r] of A
    p.a_ptr = static_cast<const uint16_t *>(A);
    p.a_rows_limit = (int)a_rows_n;
    if (pair && (out_f32 != nullptr || k_splits != 1)) return MOE_ERR_UNSUPPORTED;
    const int tile_m = pair ? moe::gg::PAIR_BM : moe::gg::BM;
    p.raster = pair ? kRasterPair : kRasterSingle;
    const int m_upper = mtiles ? max_tiles : (dense_rows + tile_m - 1) / tile_m;
    const int n_tiles = (n_out + moe::gg::BN - 1) / moe::gg::BN;
    const int64_t work = (int64_t)m_upper * n_tiles * k_splits;
    if (pair) {
        int clusters = dev->num_sms / 2;
        if (work < clusters) clusters = (int)work;
        if (clusters < 1) clusters = 1;
        moe::gg::grouped_gemm_pair_kernel<<<2 * clusters, moe::gg::NUM_THREADS, moe::gg::P_SMEM_BYTES, st>>>(ta, tb, tc,
                                                                                                        p);
    } else {
        int grid = dev->num_sms;
        if (work < grid) grid = (int)work;
        if (grid < 1) grid = 1;
        if (!make_tmap(&ta32, A, a_rows_n, (uint64_t)k_dim, moe::gg::A_CHUNK_ROWS)) return MOE_ERR_CUDA;
        if (b_mn)
            moe::gg::grouped_gemm_kernel<true><<<grid, moe::gg::NUM_THREADS_G, moe::gg::SMEM_BYTES, st>>>(ta, tb, tc, p,
                                                                                                       ta32);
        else
            moe::gg::grouped_gemm_kernel<false><<<grid, moe::gg::NUM_THREADS_G, moe::gg::SMEM_BYTES, st>>>(ta, tb, tc,
                                                                                                        p, ta32);
    }
    count_launch();
    return MOE_OK;
}

// FP8 expert GEMM variant: the channel-major kernel (gemm_fp8t.cuh, weights
// widened into tensor memory, default) or the token-major one (gemm_fp8w.cuh,
// weights widened into shared memory), MOE_FP8_GEMM=token_major
// (environment, read once).
bool fp8_token_major() {
    static const bool v = []() {
        const char *e = std::getenv("MOE_FP8_GEMM");
        return e != nullptr && std::strcmp(e, "token_major") == 0;
    }();
    return v;
}

moe::gg::Params fp8_params(int k_dim, int n_out, int groups, const float *bias, uint16_t *out, int out_rows,
                           const int4 *mtiles, const int *num_mtiles, int max_tiles, int dense_rows, bool gelu) {
    moe::gg::Params p{};
    p.mtiles = mtiles;
    p.num_mtiles = num_mtiles;
    p.max_mtiles = max_tiles;
    p.dense_rows = dense_rows;
    p.n_out = n_out;
    p.k_dim = k_dim;
    p.num_groups = groups;
    p.out_rows = out_rows;
    p.bias = bias;
    p.out = out;
    p.gelu = gelu ? 1 : 0;
    p.out_f32 = nullptr;
    p.k_splits = 1;
    p.raster = kRasterSingle;
    return p;
}

// The grouped GEMM with FP8 expert weights: A bf16 [a_rows, k_dim], Bq codes
// [groups * n_out, k_dim], scale [groups * n_out].
// Split count for the channel-major FP8 GEMM: the S (<= kMaxFp8Splits, each
// split at least one k-pair) that minimises the busiest SM's time,
// ceil(units / SMs) * (ceil(pairs / S) + kFp8ItemOverhead), for the expected
// m-tile count; the smaller S on ties. The per-item overhead (about four
// k-pairs' time) is measured: Mixtral-shaped decode with 4 splits took 6%
// longer on the first GEMM (32 k-pairs per tile) and 3% less on the second
// (112 k-pairs per tile) than without.
constexpr int kFp8ItemOverhead = 4;
int fp8_splits(int m_est, int n_tiles, int kpairs, int num_sms) {
    int best = 1;
    int64_t best_cost = INT64_MAX;
    for (int S = 1; S <= kMaxFp8Splits && S <= kpairs; ++S) {
        const int64_t units = (int64_t)m_est * n_tiles * S;
        const int64_t cost = ((units + num_sms - 1) / num_sms) * ((kpairs + S - 1) / S + kFp8ItemOverhead);
        if (cost < best_cost) {
            best_cost = cost;
            best = S;
        }
    }
    return best;
}

// The grouped GEMM with quantised expert weights: A bf16 [a_rows, k_dim];
// FP8 (is_int4 false): codes Bq [groups * n_out, k_dim], scale [groups * n_out];
// INT4: codes Bq [groups * n_out, k_dim / 2], gscale [groups, k_dim / 128, n_out] bf16.
moe_status launch_gemm_quant(DeviceState *dev, bool is_int4, const void *A, uint64_t a_rows, const void *Bq,
                             uint64_t b_rows, int k_dim, int n_out, int groups, const float *scale,
                             const uint16_t *gscale, const float *bias, uint16_t *out, int out_rows,
                             const int4 *mtiles, const int *num_mtiles, int max_tiles, int dense_rows, bool gelu,
                             cudaStream_t st, float *part = nullptr, const int32_t *offsets = nullptr,
                             int tile_rows = moe::gg::QT_ROWS) {
    if (is_int4 || !fp8_token_major()) {
        CUtensorMap tt, tb;
        if (!make_tmap(&tt, A, a_rows, (uint64_t)k_dim, moe::gg::QT_TBOX)) return MOE_ERR_CUDA;
        const bool ok = is_int4 ? make_tmap_u8(&tb, Bq, b_rows, (uint64_t)k_dim / 2, moe::gg::QT_CH,
                                            moe::gg::QFormat<moe::gg::QF_INT4>::ROW_BYTES, CU_TENSOR_MAP_SWIZZLE_64B)
                             : make_tmap_u8(&tb, Bq, b_rows, (uint64_t)k_dim, moe::gg::QT_CH,
                                            moe::gg::QFormat<moe::gg::QF_FP8>::ROW_BYTES, CU_TENSOR_MAP_SWIZZLE_128B);
        if (!ok) return MOE_ERR_CUDA;
        moe::gg::Params p = fp8_params(k_dim, n_out, groups, bias, out, out_rows, mtiles, num_mtiles, max_tiles,
                                       dense_rows, gelu);
        // the most rows of any tile: the list's tile height, or the dense rows' (64-row tiles)
        p.q_rows = mtiles ? tile_rows : std::min(dense_rows, moe::gg::QT_ROWS);
        const int n_tiles = (n_out + moe::gg::QT_CH - 1) / moe::gg::QT_CH;
        const int kpairs = (k_dim / moe::gg::BK + 1) / 2;
        const int m_upper = mtiles ? max_tiles : (dense_rows + moe::gg::QT_ROWS - 1) / moe::gg::QT_ROWS;
        int splits = 1;
        if (part != nullptr && out_rows <= kSplitRows) {
            // routed rows: about one m-tile per expert that receives rows
            const int m_est = mtiles ? std::min(groups, out_rows) : m_upper;
            splits = fp8_splits(m_est, n_tiles, kpairs, dev->num_sms);
        }
        if (splits > 1) {
            p.out_f32 = part;
            p.k_splits = splits;
        }
        const int64_t work = (int64_t)m_upper * n_tiles * splits;
        int grid = dev->num_sms;
        if (work < grid) grid = (int)work;
        if (grid < 1) grid = 1;
        if (is_int4)
            moe::gg::grouped_gemm_quant_kernel<moe::gg::QF_INT4>
                <<<grid, moe::gg::QT_NUM_THREADS, moe::gg::QT_SMEM_BYTES, st>>>(tt, tb, p, nullptr, gscale);
        else
            moe::gg::grouped_gemm_quant_kernel<moe::gg::QF_FP8>
                <<<grid, moe::gg::QT_NUM_THREADS, moe::gg::QT_SMEM_BYTES, st>>>(tt, tb, p, scale, nullptr);
        count_launch();
        if (splits > 1) {
            const dim3 fgrid((unsigned)out_rows, (unsigned)((n_out + 1023) / 1024));
            moe::gg::quant_split_finalize_kernel<<<fgrid, 256, 0, st>>>(part, splits, out_rows, n_out, offsets,
                                                                           groups, is_int4 ? nullptr : scale, bias,
                                                                           gelu ? 1 : 0, out);
            count_launch();
        }
        return MOE_OK;
    }
    CUtensorMap ta, tb, tc, ta32;
    if (!make_tmap(&ta, A, a_rows, (uint64_t)k_dim, moe::gg::BM)) return MOE_ERR_CUDA;
    if (!make_tmap(&ta32, A, a_rows, (uint64_t)k_dim, moe::gg::A_CHUNK_ROWS)) return MOE_ERR_CUDA;
    if (!make_tmap_u8(&tb, Bq, b_rows, (uint64_t)k_dim, moe::gg::BN, moe::gg::Q_RAW_K)) return MOE_ERR_CUDA;
    if (!make_tmap(&tc, out, (uint64_t)out_rows, (uint64_t)n_out, 32, 32, false)) return MOE_ERR_CUDA;
    const moe::gg::Params p = fp8_params(k_dim, n_out, groups, bias, out, out_rows, mtiles, num_mtiles, max_tiles,
                                         dense_rows, gelu);
    const int m_upper = mtiles ? max_tiles : (dense_rows + moe::gg::BM - 1) / moe::gg::BM;
    const int64_t work = (int64_t)m_upper * ((n_out + moe::gg::BN - 1) / moe::gg::BN);
    int grid = dev->num_sms;
    if (work < grid) grid = (int)work;
    if (grid < 1) grid = 1;
    moe::gg::grouped_gemm_fp8w_kernel<<<grid, moe::gg::Q_NUM_THREADS, moe::gg::Q_SMEM_BYTES, st>>>(ta, tb, tc, p,
                                                                                                   scale, ta32);
    count_launch();
    return MOE_OK;
}

// x_perm: the regrouped rows; or, with gather_rows (bf16 weights only), the
// first GEMM reads row gather_rows[r] of x for regrouped row r instead (x_perm
// is then not read).
// The routed experts' GEMM kernel and its m-tile shape: FP8 (64-row tiles, or
// 128 token-major), the SM-pair kernel (256) or the single-SM kernel (128).
struct FfnTiling {
    bool quant, pair_routed, pair_routed2, pair_shared;  // quant: FP8 or INT4 expert weights
    int tile_rows, raster;    // first expert GEMM's m-tiles
    int tile_rows2, raster2;  // second's (a second list is built when they differ)
};
FfnTiling ffn_tiling(const moe_shape *s, const moe_weights *wt, bool gather) {
    FfnTiling t;
    int64_t per_expert = (int64_t)s->T * s->K / s->N;
    const int C = capacity_of(s);
    if (per_expert > C) per_expert = C;
    t.quant = wt->format != MOE_WEIGHTS_BF16;
    t.pair_routed = !t.quant && !gather && use_pair(per_expert);
    t.pair_routed2 = !t.quant && use_pair_gemm2(per_expert, s->d_ff);
    t.pair_shared = !t.quant && use_pair(s->T);
    // quantised channel-major kernel: 32-row tiles (more, half-size token
    // stages) when the experts get at most 32 rows each on average (decode)
    const int qt_rows = per_expert <= moe::gg::QT_NARROW_ROWS ? moe::gg::QT_NARROW_ROWS : moe::gg::QT_ROWS;
    t.tile_rows = t.quant ? (wt->format == MOE_WEIGHTS_FP8_E4M3 && fp8_token_major() ? moe::gg::BM : qt_rows)
                        : (t.pair_routed ? moe::gg::PAIR_BM : moe::gg::BM);
    t.raster = t.pair_routed ? kRasterPair : kRasterSingle;
    t.tile_rows2 = t.quant ? t.tile_rows : (t.pair_routed2 ? moe::gg::PAIR_BM : moe::gg::BM);
    t.raster2 = t.quant ? t.raster : (t.pair_routed2 ? kRasterPair : kRasterSingle);
    return t;
}

// tiles_ready: w.mtiles already holds the m-tile list of ffn_tiling(s, wt,
// gather_rows != nullptr) (the router's plan kernel built it).
moe_status run_ffn(const moe_shape *s, DeviceState *dev, const uint16_t *x_perm, const int32_t *offsets,
                   const moe_weights *wt, const uint16_t *x, uint16_t *y_perm, uint16_t *z,
                   const FfnWs &w, cudaStream_t st, cudaEvent_t mid = nullptr, const int32_t *gather_rows = nullptr,
                   bool tiles_ready = false) {
    const int T = s->T, N = s->N, K = s->K, d = s->d_model, f = s->d_ff;
    const int rows = T * K;
    const int mt = max_mtiles(s);
    const FfnTiling tl = ffn_tiling(s, wt, gather_rows != nullptr);
    const bool quant = tl.quant, pair_routed = tl.pair_routed, pair_shared = tl.pair_shared;
    const bool two_lists = tl.tile_rows2 != tl.tile_rows;
    const int4 *mtiles2 = two_lists ? w.mtiles2 : w.mtiles;
    const int *num_mtiles2 = two_lists ? w.num_mtiles2 : w.num_mtiles;
    if (!tiles_ready) {
        moe::gg::build_mtiles_kernel<<<1, 1024, 0, st>>>(offsets, N, rows, tl.tile_rows, tl.raster, mt, w.mtiles,
                                                         w.num_mtiles);
        count_launch();
        if (two_lists) {
            moe::gg::build_mtiles_kernel<<<1, 1024, 0, st>>>(offsets, N, rows, tl.tile_rows2, tl.raster2, mt,
                                                             w.mtiles2, w.num_mtiles2);
            count_launch();
        }
    }
    moe_status r;
    if (quant) {
        // the same four GEMMs with quantised expert weights (FP8 per-channel or INT4 group-wise scales)
        const bool i4 = wt->format == MOE_WEIGHTS_INT4_G128;
        r = launch_gemm_quant(dev, i4, x_perm, rows, wt->W1q, (uint64_t)N * f, d, f, N, wt->s1, wt->g1, wt->b1, w.H,
                              rows, w.mtiles, w.num_mtiles, mt, 0, true, st, w.part, offsets, tl.tile_rows);
        if (r != MOE_OK) return r;
        if (s->has_shared) {
            r = launch_gemm_quant(dev, i4, x, T, wt->Ws1q, f, d, f, 1, wt->ss1, wt->gs1, wt->bs1, w.Hs, T, nullptr,
                                  nullptr, 0, T, true, st, w.part);
            if (r != MOE_OK) return r;
        }
        if (mid != nullptr && cudaEventRecord(mid, st) != cudaSuccess) return MOE_ERR_CUDA;
        r = launch_gemm_quant(dev, i4, w.H, rows, wt->W2q, (uint64_t)N * d, f, d, N, wt->s2, wt->g2, wt->b2, y_perm,
                              rows, w.mtiles, w.num_mtiles, mt, 0, false, st, w.part, offsets, tl.tile_rows);
        if (r != MOE_OK) return r;
        if (s->has_shared) {
            r = launch_gemm_quant(dev, i4, w.Hs, T, wt->Ws2q, d, f, d, 1, wt->ss2, wt->gs2, wt->bs2, z, T, nullptr,
                                  nullptr, 0, T, false, st, w.part);
            if (r != MOE_OK) return r;
        }
        return launch_status();
    }
    // routed experts: H = GELU(x_perm W1^T + b1), y_perm = H W2^T + b2
    if (gather_rows != nullptr)
        r = launch_gemm(dev, false, x, T, wt->W1, (uint64_t)N * f, d, f, N, wt->b1, w.H, rows, w.mtiles,
                        w.num_mtiles, mt, 0, true, st, nullptr, 1, nullptr, gather_rows);
    else
        r = launch_gemm(dev, pair_routed, x_perm, rows, wt->W1, (uint64_t)N * f, d, f, N, wt->b1, w.H, rows,
                        w.mtiles, w.num_mtiles, mt, 0, true, st);
    if (r != MOE_OK) return r;
    if (s->has_shared) {
        r = launch_gemm(dev, pair_shared, x, T, wt->Ws1, f, d, f, 1, wt->bs1, w.Hs, T, nullptr, nullptr, 0, T, true,
                        st);
        if (r != MOE_OK) return r;
    }
    if (mid != nullptr && cudaEventRecord(mid, st) != cudaSuccess) return MOE_ERR_CUDA;
    r = launch_gemm(dev, tl.pair_routed2, w.H, rows, wt->W2, (uint64_t)N * d, f, d, N, wt->b2, y_perm, rows,
                    mtiles2, num_mtiles2, mt, 0, false, st);
    if (r != MOE_OK) return r;
    if (s->has_shared) {
        r = launch_gemm(dev, pair_shared, w.Hs, T, wt->Ws2, d, f, d, 1, wt->bs2, z, T, nullptr, nullptr, 0, T, false,
                        st);
        if (r != MOE_OK) return r;
    }
    return launch_status();
}

moe_status run_combine(const moe_shape *s, const uint16_t *y_perm, const int32_t *slot_of,
                       const float *topk_w, const uint16_t *z, uint16_t *y, cudaStream_t st) {
    const int vec = s->d_model / 8;
    const int thr = vec < 256 ? 64 : 256;
    const int K = s->K;
    const int kmax = K <= 1 ? 1 : (K <= 2 ? 2 : (K <= 4 ? 4 : 8));
    dim3 grid((s->T + 8 / kmax - 1) / (8 / kmax), (vec + thr - 1) / thr);
#define MOE_COMBINE(KM)                                                                                    \
    moe::dispatch::combine_kernel<KM><<<grid, thr, 0, st>>>(y_perm, slot_of, topk_w, z, s->T, K, s->d_model, \
                                                            s->T * K, y)
    if (kmax == 1) MOE_COMBINE(1);
    else if (kmax == 2) MOE_COMBINE(2);
    else if (kmax == 4) MOE_COMBINE(4);
    else MOE_COMBINE(8);
#undef MOE_COMBINE
    count_launch();
    return launch_status();
}

moe_status run_aux(const moe_shape *s, const int32_t *demand, const float *prob_sum, float *aux,
                   cudaStream_t st) {
    moe::dispatch::aux_loss_kernel<<<1, 256, 0, st>>>(demand, prob_sum, s->T, s->N, s->K, s->aux_alpha, aux);
    count_launch();
    return launch_status();
}

// Transposes of the grouped rows in[rows(offsets), C] into out[C, ld] (zeroed
// first: padding columns must read as zeros).
moe_status transpose_grouped(const uint16_t *in, int R, int C, const int32_t *offsets, const int32_t *poff, int N,
                             uint16_t *out, size_t ld, cudaStream_t st) {
    if (cudaMemsetAsync(out, 0, (size_t)C * ld * sizeof(uint16_t), st) != cudaSuccess) return MOE_ERR_CUDA;
    if (R <= 0) return MOE_OK;
    dim3 grid((C + 31) / 32, (R + 31) / 32);
    moe::bwd::transpose_grouped_kernel<<<grid, moe::bwd::kThreads, 0, st>>>(in, R, C, offsets, poff, N, out, ld);
    count_launch();
    return launch_status();
}

moe_status simt_gemm(const float *a, size_t a_ks, size_t a_ms, const uint16_t *b, size_t ldb, int M, int Nn, int Kk,
                     float *c, size_t ldc, cudaStream_t st) {
    dim3 grid((Nn + moe::bwd::kSB - 1) / moe::bwd::kSB, (M + moe::bwd::kSB - 1) / moe::bwd::kSB);
    moe::bwd::simt_gemm_kernel<<<grid, moe::bwd::kThreads, 0, st>>>(a, a_ks, a_ms, b, ldb, M, Nn, Kk, c, ldc);
    count_launch();
    return launch_status();
}

moe_status run_backward(const moe_shape *s, DeviceState *dev, const moe_weights *wt, const uint16_t *x,
                        const float *sel_bias, const uint16_t *dy, float g_aux, float g_z, const moe_grads *g,
                        const BackwardWs &w, cudaStream_t st) {
    const int T = s->T, N = s->N, K = s->K, d = s->d_model, f = s->d_ff;
    const int rows = T * K;
    const int mt = max_mtiles(s);
    const ForwardWs &fw = w.fwd;
    float *dw = g->dw ? g->dw : w.dw;
    moe_status r;
    // ---- forward recompute (routing decisions, H = h, y_perm = o)
    if ((r = run_route(s, dev, x, wt->Wg, sel_bias, fw.topk_idx, fw.topk_w, fw.demand, fw.prob_sum, nullptr, fw.route,
                       st)) != MOE_OK)
        return r;
    if ((r = run_dispatch(s, fw.topk_idx, x, fw.kept, fw.offsets, fw.slot_of, fw.row_token, fw.x_perm, fw.disp,
                          st)) != MOE_OK)
        return r;
    if ((r = run_ffn(s, dev, fw.x_perm, fw.offsets, wt, x, fw.y_perm, fw.z, fw.ffn, st)) != MOE_OK) return r;
    // the 128-row tile list for the single-SM fp32 GEMMs below
    moe::gg::build_mtiles_kernel<<<1, 1024, 0, st>>>(fw.offsets, N, rows, moe::gg::BM, kRasterSingle, mt, w.mtiles,
                                                     w.num_mtiles);
    count_launch();
    // pre-activations a = x W1^T (raw fp32; the bias is added where GELU' is taken)
    if ((r = launch_gemm(dev, false, fw.x_perm, rows, wt->W1, (uint64_t)N * f, d, f, N, wt->b1, nullptr, rows,
                         w.mtiles, w.num_mtiles, mt, 0, false, st, w.A1)) != MOE_OK)
        return r;
    // gate logits in fp32 (exact on the input grid, any order)
    {
        dim3 grid((T + moe::route::kGBM - 1) / moe::route::kGBM, (N + moe::route::kGBN - 1) / moe::route::kGBN);
        moe::route::gate_logits_tiled_kernel<<<grid, moe::route::kGateThreads, 0, st>>>(x, wt->Wg, T, d, N, w.L);
        count_launch();
    }
    // ---- combine backward
    moe::bwd::combine_backward_kernel<<<T, moe::bwd::kThreads, 0, st>>>(dy, fw.y_perm, fw.slot_of, fw.topk_w, K, d,
                                                                        dw, w.dO);
    count_launch();
    // ---- routed experts
    // dh = dO W2_e and dx' = da W1_e read the weights as stored (N-major B): no transposed copies
    if ((r = launch_gemm(dev, false, w.dO, rows, wt->W2, (uint64_t)N * d, d, f, N, wt->b1, nullptr, rows, w.mtiles,
                         w.num_mtiles, mt, 0, false, st, w.DH, 1, nullptr, nullptr, true)) != MOE_OK)
        return r;
    moe::bwd::gelu_backward_kernel<<<rows, moe::bwd::kThreads, 0, st>>>(w.DH, w.A1, wt->b1, fw.offsets, N, f, w.DA);
    count_launch();
    if ((r = launch_gemm(dev, false, w.DA, rows, wt->W1, (uint64_t)N * f, f, d, N, wt->b2, nullptr, rows, w.mtiles,
                         w.num_mtiles, mt, 0, false, st, w.DXP, 1, nullptr, nullptr, true)) != MOE_OK)
        return r;
    moe::bwd::expert_colsum_kernel<<<dim3((f + 255) / 256, N), moe::bwd::kThreads, 0, st>>>(w.DA, fw.offsets, f,
                                                                                           g->db1);
    moe::bwd::expert_colsum_kernel<<<dim3((d + 255) / 256, N), moe::bwd::kThreads, 0, st>>>(w.dO, fw.offsets, d,
                                                                                           g->db2);
    moe::bwd::padded_offsets_kernel<<<1, 32, 0, st>>>(fw.offsets, N, w.poff);
    count_launch();
    count_launch();
    count_launch();
    if ((r = transpose_grouped(w.dO, rows, d, fw.offsets, w.poff, N, w.dOT, w.ldp, st)) != MOE_OK) return r;
    if ((r = transpose_grouped(fw.ffn.H, rows, f, fw.offsets, w.poff, N, w.HT, w.ldp, st)) != MOE_OK) return r;
    if ((r = transpose_grouped(w.DA, rows, f, fw.offsets, w.poff, N, w.DAT, w.ldp, st)) != MOE_OK) return r;
    if ((r = transpose_grouped(fw.x_perm, rows, d, fw.offsets, w.poff, N, w.XPT, w.ldp, st)) != MOE_OK) return r;
    // dW2[e] = dO_e^T H_e: [d, f], dW1[e] = DA_e^T X_e: [f, d] -- the expert's rows are the reduction
    if ((r = launch_gemm(dev, false, w.dOT, d, w.HT, f, (int)w.ldp, f, 1, wt->b1, nullptr, d, nullptr, nullptr, 0, d,
                         false, st, g->dW2, N, w.poff)) != MOE_OK)
        return r;
    if ((r = launch_gemm(dev, false, w.DAT, f, w.XPT, d, (int)w.ldp, d, 1, wt->b1, nullptr, f, nullptr, nullptr, 0, f,
                         false, st, g->dW1, N, w.poff)) != MOE_OK)
        return r;
    // ---- shared expert (weight 1: dO = dy)
    const float *dxs = nullptr;
    if (s->has_shared) {
        moe::bwd::single_group_kernel<<<1, 32, 0, st>>>(T, w.soff, w.spoff);
        count_launch();
        if ((r = launch_gemm(dev, false, x, T, wt->Ws1, f, d, f, 1, wt->bs1, nullptr, T, nullptr, nullptr, 0, T, false,
                             st, w.As1)) != MOE_OK)
            return r;
        if ((r = launch_gemm(dev, false, dy, T, wt->Ws2, d, d, f, 1, wt->bs1, nullptr, T, nullptr, nullptr, 0, T, false,
                             st, w.DHs, 1, nullptr, nullptr, true)) != MOE_OK)
            return r;
        moe::bwd::gelu_backward_kernel<<<T, moe::bwd::kThreads, 0, st>>>(w.DHs, w.As1, wt->bs1, w.soff, 1, f, w.DAs);
        count_launch();
        if ((r = launch_gemm(dev, false, w.DAs, T, wt->Ws1, f, f, d, 1, wt->bs2, nullptr, T, nullptr, nullptr, 0, T,
                             false, st, w.DXs, 1, nullptr, nullptr, true)) != MOE_OK)
            return r;
        moe::bwd::expert_colsum_kernel<<<dim3((f + 255) / 256, 1), moe::bwd::kThreads, 0, st>>>(w.DAs, w.soff, f,
                                                                                               g->dbs1);
        moe::bwd::expert_colsum_kernel<<<dim3((d + 255) / 256, 1), moe::bwd::kThreads, 0, st>>>(dy, w.soff, d,
                                                                                               g->dbs2);
        count_launch();
        count_launch();
        if ((r = transpose_grouped(dy, T, d, w.soff, w.spoff, 1, w.dyT, w.ldt, st)) != MOE_OK) return r;
        if ((r = transpose_grouped(fw.ffn.Hs, T, f, w.soff, w.spoff, 1, w.HsT, w.ldt, st)) != MOE_OK) return r;
        if ((r = transpose_grouped(w.DAs, T, f, w.soff, w.spoff, 1, w.DAsT, w.ldt, st)) != MOE_OK) return r;
        if ((r = transpose_grouped(x, T, d, w.soff, w.spoff, 1, w.xT, w.ldt, st)) != MOE_OK) return r;
        if ((r = launch_gemm(dev, false, w.dyT, d, w.HsT, f, (int)w.ldt, f, 1, wt->bs1, nullptr, d, nullptr, nullptr, 0,
                             d, false, st, g->dWs2, 1, w.spoff)) != MOE_OK)
            return r;
        if ((r = launch_gemm(dev, false, w.DAsT, f, w.xT, d, (int)w.ldt, d, 1, wt->bs1, nullptr, f, nullptr, nullptr, 0,
                             f, false, st, g->dWs1, 1, w.spoff)) != MOE_OK)
            return r;
        dxs = w.DXs;
    }
    // ---- gate
    moe::bwd::gate_backward_kernel<<<(T + 7) / 8, moe::bwd::kThreads, 0, st>>>(
        w.L, fw.topk_idx, fw.topk_w, dw, fw.demand, T, N, K, s->aux_alpha, s->z_beta, g_aux, g_z, w.DS);
    count_launch();
    // dWg[e, i] = sum_t DS[t, e] x[t, i];  dx[t, i] = sum_e DS[t, e] Wg[e, i]
    if ((r = simt_gemm(w.DS, (size_t)N, 1, x, (size_t)d, N, d, T, g->dWg, (size_t)d, st)) != MOE_OK) return r;
    if ((r = simt_gemm(w.DS, 1, (size_t)N, wt->Wg, (size_t)d, T, d, N, g->dx, (size_t)d, st)) != MOE_OK) return r;
    moe::bwd::dx_gather_kernel<<<T, moe::bwd::kThreads, 0, st>>>(w.DXP, fw.slot_of, dxs, K, d, g->dx);
    count_launch();
    return launch_status();
}

bool weights_ok(const moe_shape *s, const moe_weights *w, bool need_gate) {
    if (w == nullptr) return false;
    const int fmt = w->format;
    if (fmt != MOE_WEIGHTS_BF16 && fmt != MOE_WEIGHTS_FP8_E4M3 && fmt != MOE_WEIGHTS_INT4_G128) return false;
    if (need_gate && (w->Wg == nullptr || !aligned16(w->Wg))) return false;
    auto all = [](std::initializer_list<const void *> ps) {
        for (const void *p : ps)
            if (p == nullptr || !aligned16(p)) return false;
        return true;
    };
    bool ok = fmt == MOE_WEIGHTS_BF16        ? all({w->W1, w->b1, w->W2, w->b2})
              : fmt == MOE_WEIGHTS_FP8_E4M3 ? all({w->W1q, w->s1, w->b1, w->W2q, w->s2, w->b2})
                                             : all({w->W1q, w->g1, w->b1, w->W2q, w->g2, w->b2});
    if (ok && s->has_shared)
        ok = fmt == MOE_WEIGHTS_BF16        ? all({w->Ws1, w->bs1, w->Ws2, w->bs2})
             : fmt == MOE_WEIGHTS_FP8_E4M3 ? all({w->Ws1q, w->ss1, w->bs1, w->Ws2q, w->ss2, w->bs2})
                                            : all({w->Ws1q, w->gs1, w->bs1, w->Ws2q, w->gs2, w->bs2});
    return ok;
}

// INT4 scales come in groups of 128 reduction columns: both reductions (d_model
// for the first Linear, d_ff for the second) must hold whole groups.
bool weights_shape_supported(const moe_shape *s, const moe_weights *w) {
    return w->format != MOE_WEIGHTS_INT4_G128 || (s->d_model % 128 == 0 && s->d_ff % 128 == 0);
}

}  // namespace

// ==================================================================== routing without a workspace
// Some callers cannot pass us device scratch memory: a plugin inside a host
// framework whose memory planner has no slot for per-operator scratch, or a
// latency-critical loop that must not call cudaMalloc after start-up
// (cudaMalloc can synchronise the device and fail under fragmentation).
// moe_route_noalloc serves them from one fixed array in the library's own
// device memory. The array is a file-scope __device__ object, so every GPU
// that loads this library holds it until the process exits.
constexpr size_t kRouteScratchBytes = size_t(8) << 20;  // 8 MiB
static __device__ __align__(256) unsigned char moe_route_scratch[kRouteScratchBytes];

namespace {
struct ScratchAddress {
    std::mutex mu;
    void *ptr = nullptr;  // set once a lookup has succeeded; a failed lookup is retried on the next call
};
ScratchAddress g_route_scratch_addr[kMaxDevices];

// Device address of moe_route_scratch on the current device. In host code the
// symbol's name is only a host-side stand-in; the address must come from
// cudaGetSymbolAddress, with that device current. Only a successful lookup is
// kept, so a first call that failed (for example one made during a stream
// capture) does not poison later calls on that device.
moe_status route_scratch(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    ScratchAddress &a = g_route_scratch_addr[dev];
    std::lock_guard<std::mutex> lock(a.mu);
    if (a.ptr == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, moe_route_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return MOE_ERR_CUDA;
        }
        a.ptr = p;
    }
    *out = a.ptr;
    return MOE_OK;
}
}  // namespace

// ==================================================================== C ABI

extern "C" {

int32_t moe_capacity(const moe_shape *shape) {
    if (check_shape(shape) != MOE_OK) return -1;
    return capacity_of(shape);
}

size_t moe_workspace_bytes(const moe_shape *shape, int32_t kind) {
    if (check_shape(shape) != MOE_OK) return 0;
    return ws_bytes(shape, kind);
}

const char *moe_status_string(int32_t status) {
    switch (status) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported shape";
        case MOE_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case MOE_ERR_CUDA: return "CUDA error";
        case MOE_ERR_DEVICE: return "device-side error";
        default: return "unknown status";
    }
}

moe_status moe_route(const moe_shape *shape, const moe_bf16 *x, const moe_bf16 *Wg, const float *sel_bias,
                     int32_t *topk_idx, float *topk_w, int32_t *demand, float *prob_sum, void *workspace,
                     size_t workspace_bytes, void *stream) {
    moe_status r = check_shape(shape);
    if (r != MOE_OK) return r;
    if (!x || !Wg || !topk_idx || !topk_w || !demand || !prob_sum) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(Wg)) return MOE_ERR_INVALID_ARG;
    if ((r = check_ws(shape, MOE_WS_ROUTE, workspace, workspace_bytes)) != MOE_OK) return r;
    DeviceState *dev;
    if ((r = device_state(&dev)) != MOE_OK) return r;
    Carve c(workspace);
    RouteWs w = carve_route(c, shape);
    return run_route(shape, dev, x, Wg, sel_bias, topk_idx, topk_w, demand, prob_sum, nullptr, w,
                     as_stream(stream));
}

moe_status moe_route_noalloc(const moe_shape *shape, const moe_bf16 *x, const moe_bf16 *Wg, const float *sel_bias,
                             int32_t *topk_idx, float *topk_w, int32_t *demand, float *prob_sum, void *stream) {
    moe_status r = check_shape(shape);
    if (r != MOE_OK) return r;
    if (!x || !Wg || !topk_idx || !topk_w || !demand || !prob_sum) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(Wg)) return MOE_ERR_INVALID_ARG;
    if (ws_bytes(shape, MOE_WS_ROUTE) > kRouteScratchBytes) return MOE_ERR_UNSUPPORTED;
    DeviceState *dev;
    if ((r = device_state(&dev)) != MOE_OK) return r;
    void *scratch = nullptr;
    if ((r = route_scratch(&scratch)) != MOE_OK) return r;
    // every scratch word the kernels read is written earlier in the same call
    Carve c(scratch);
    RouteWs w = carve_route(c, shape);
    return run_route(shape, dev, x, Wg, sel_bias, topk_idx, topk_w, demand, prob_sum, nullptr, w,
                     as_stream(stream));
}

moe_status moe_dispatch(const moe_shape *shape, const int32_t *topk_idx, const moe_bf16 *x, int32_t *kept,
                        int32_t *expert_offsets, int32_t *slot_of, int32_t *row_token, moe_bf16 *x_perm,
                        void *workspace, size_t workspace_bytes, void *stream) {
    moe_status r = check_shape(shape);
    if (r != MOE_OK) return r;
    if (!topk_idx || !x || !kept || !expert_offsets || !slot_of || !row_token || !x_perm)
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(x_perm)) return MOE_ERR_INVALID_ARG;
    if ((r = check_ws(shape, MOE_WS_DISPATCH, workspace, workspace_bytes)) != MOE_OK) return r;
    DeviceState *dev;
    if ((r = device_state(&dev)) != MOE_OK) return r;
    Carve c(workspace);
    DispatchWs w = carve_dispatch(c, shape);
    return run_dispatch(shape, topk_idx, x, kept, expert_offsets, slot_of, row_token, x_perm, w,
                        as_stream(stream));
}

moe_status moe_expert_ffn(const moe_shape *shape, const moe_bf16 *x_perm, const int32_t *expert_offsets,
                          const moe_weights *weights, const moe_bf16 *x, moe_bf16 *y_perm, moe_bf16 *z_shared,
                          void *workspace, size_t workspace_bytes, void *stream) {
    moe_status r = check_shape(shape);
    if (r != MOE_OK) return r;
    if (!x_perm || !expert_offsets || !y_perm || !weights_ok(shape, weights, false)) return MOE_ERR_INVALID_ARG;
    if (!weights_shape_supported(shape, weights)) return MOE_ERR_UNSUPPORTED;
    if (!aligned16(x_perm) || !aligned16(y_perm)) return MOE_ERR_INVALID_ARG;
    if (shape->has_shared && (!x || !z_shared || !aligned16(x) || !aligned16(z_shared)))
        return MOE_ERR_INVALID_ARG;
    if ((r = check_ws(shape, MOE_WS_FFN, workspace, workspace_bytes)) != MOE_OK) return r;
    DeviceState *dev;
    if ((r = device_state(&dev)) != MOE_OK) return r;
    Carve c(workspace);
    FfnWs w = carve_ffn(c, shape);
    return run_ffn(shape, dev, x_perm, expert_offsets, weights, x, y_perm, z_shared, w, as_stream(stream));
}

moe_status moe_combine(const moe_shape *shape, const moe_bf16 *y_perm, const int32_t *slot_of,
                       const float *topk_w, const moe_bf16 *z_shared, moe_bf16 *y, void *stream) {
    moe_status r = check_shape(shape);
    if (r != MOE_OK) return r;
    if (!y_perm || !slot_of || !topk_w || !y) return MOE_ERR_INVALID_ARG;
    if (!aligned16(y_perm) || !aligned16(y) || (z_shared && !aligned16(z_shared))) return MOE_ERR_INVALID_ARG;
    return run_combine(shape, y_perm, slot_of, topk_w, z_shared, y, as_stream(stream));
}

moe_status moe_aux_loss(const moe_shape *shape, const int32_t *demand, const float *prob_sum, float *aux,
                        void *stream) {
    moe_status r = check_shape(shape);
    if (r != MOE_OK) return r;
    if (!demand || !prob_sum || !aux) return MOE_ERR_INVALID_ARG;
    return run_aux(shape, demand, prob_sum, aux, as_stream(stream));
}

}  // extern "C"

namespace {

moe_status forward_impl(const moe_shape *shape, const moe_weights *weights, const moe_bf16 *x,
                        const float *sel_bias, moe_bf16 *y, const moe_route_out *out, void *workspace,
                        size_t workspace_bytes, void *const *events, void *stream) {
    moe_status r = check_shape(shape);
    if (r != MOE_OK) return r;
    if (!x || !y || !aligned16(x) || !aligned16(y) || !weights_ok(shape, weights, true)) return MOE_ERR_INVALID_ARG;
    if (!weights_shape_supported(shape, weights)) return MOE_ERR_UNSUPPORTED;
    if ((r = check_ws(shape, MOE_WS_FORWARD, workspace, workspace_bytes)) != MOE_OK) return r;
    DeviceState *dev;
    if ((r = device_state(&dev)) != MOE_OK) return r;
    cudaStream_t st = as_stream(stream);
    Carve c(workspace);
    ForwardWs w = carve_forward(c, shape);
    moe_route_out o;
    std::memset(&o, 0, sizeof o);
    if (out) o = *out;
    int32_t *topk_idx = o.topk_idx ? o.topk_idx : w.topk_idx;
    float *topk_w = o.topk_w ? o.topk_w : w.topk_w;
    int32_t *demand = o.demand ? o.demand : w.demand;
    float *prob_sum = o.prob_sum ? o.prob_sum : w.prob_sum;
    int32_t *kept = o.kept ? o.kept : w.kept;
    int32_t *offsets = o.expert_offsets ? o.expert_offsets : w.offsets;
    int32_t *slot_of = o.slot_of ? o.slot_of : w.slot_of;
    float *aux = o.aux ? o.aux : w.aux;
    float *z_loss = o.z_loss ? o.z_loss : w.aux + 1;
    float *aux_kl = o.aux_kl ? o.aux_kl : w.aux + 2;
    float *health = o.health;
    float *mean_weight = o.mean_weight;

    auto mark = [&](int i) -> bool {
        return events == nullptr || events[i] == nullptr ||
               cudaEventRecord(reinterpret_cast<cudaEvent_t>(events[i]), st) == cudaSuccess;
    };
    // bf16 experts: the first expert GEMM gathers its rows from x by row_token,
    // so the regrouped copy of x is never written (FP8 experts read x_perm)
    const bool gather = weights->format == MOE_WEIGHTS_BF16;
    // the fused router's plan kernel also forms the dispatch plan (token-order
    // capacity) and the m-tile list
    const bool planned = fused_route(shape) && shape->drop_policy == MOE_DROP_TOKEN_ORDER;
    const bool placed = planned && moe::rtc::num_tiles(shape->T) == 1;  // the router places them itself
    const FfnTiling tl = ffn_tiling(shape, weights, gather);
    const bool two_lists = tl.tile_rows2 != tl.tile_rows;
    const DispatchPlan dplan{capacity_of(shape), w.disp.base, kept, offsets, tl.tile_rows, tl.raster,
                             max_mtiles(shape), w.ffn.mtiles, w.ffn.num_mtiles, slot_of, w.row_token,
                             tl.tile_rows2, tl.raster2, two_lists ? w.ffn.mtiles2 : nullptr, w.ffn.num_mtiles2};
    if (!mark(0)) return MOE_ERR_CUDA;
    if ((r = run_route(shape, dev, x, weights->Wg, sel_bias, topk_idx, topk_w, demand, prob_sum, aux, w.route,
                       st, z_loss, aux_kl, health, mean_weight, planned ? &dplan : nullptr)) != MOE_OK)
        return r;
    if (!mark(1)) return MOE_ERR_CUDA;
    if ((r = run_dispatch(shape, topk_idx, x, kept, offsets, slot_of, w.row_token, w.x_perm, w.disp, st,
                          health ? health + 1 : nullptr, !gather, planned, placed)) != MOE_OK)
        return r;
    if (!mark(2)) return MOE_ERR_CUDA;
    cudaEvent_t mid = events ? reinterpret_cast<cudaEvent_t>(events[3]) : nullptr;
    if ((r = run_ffn(shape, dev, w.x_perm, offsets, weights, x, w.y_perm, w.z, w.ffn, st, mid,
                     gather ? w.row_token : nullptr, planned)) != MOE_OK)
        return r;
    if (!mark(4)) return MOE_ERR_CUDA;
    if ((r = run_combine(shape, w.y_perm, slot_of, topk_w, w.z, y, st)) != MOE_OK) return r;
    if (!mark(5)) return MOE_ERR_CUDA;
    return MOE_OK;
}

}  // namespace

extern "C" {

moe_status moe_forward(const moe_shape *shape, const moe_weights *weights, const moe_bf16 *x,
                       const float *sel_bias, moe_bf16 *y, const moe_route_out *out, void *workspace,
                       size_t workspace_bytes, void *stream) {
    return forward_impl(shape, weights, x, sel_bias, y, out, workspace, workspace_bytes, nullptr, stream);
}

moe_status moe_forward_marked(const moe_shape *shape, const moe_weights *weights, const moe_bf16 *x,
                              const float *sel_bias, moe_bf16 *y, const moe_route_out *out, void *workspace,
                              size_t workspace_bytes, void *const *events, void *stream) {
    if (events == nullptr) return MOE_ERR_INVALID_ARG;
    return forward_impl(shape, weights, x, sel_bias, y, out, workspace, workspace_bytes, events, stream);
}

moe_status moe_forward_hostio(const moe_shape *shape, const moe_weights *weights, const moe_bf16 *x_host,
                              moe_bf16 *x_dev, const float *sel_bias, moe_bf16 *y_dev, moe_bf16 *y_host,
                              const moe_route_out *out, void *workspace, size_t workspace_bytes, void *stream) {
    moe_status r = check_shape(shape);
    if (r != MOE_OK) return r;
    if (!x_host || !y_host) return MOE_ERR_INVALID_ARG;
    if (!x_dev || !y_dev || !aligned16(x_dev) || !aligned16(y_dev)) return MOE_ERR_INVALID_ARG;
    cudaStream_t st = as_stream(stream);
    const size_t bytes = (size_t)shape->T * shape->d_model * sizeof(moe_bf16);
    if (cudaMemcpyAsync(x_dev, x_host, bytes, cudaMemcpyHostToDevice, st) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    if ((r = moe_forward(shape, weights, x_dev, sel_bias, y_dev, out, workspace, workspace_bytes, stream)) != MOE_OK)
        return r;
    if (cudaMemcpyAsync(y_host, y_dev, bytes, cudaMemcpyDeviceToHost, st) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    return MOE_OK;
}

moe_status moe_forward_hostio_batches(const moe_shape *shape, const moe_weights *weights, int32_t nbatch,
                                      const moe_bf16 *x_host, moe_bf16 *y_host, size_t host_stride,
                                      const float *sel_bias, moe_bf16 *x_dev, moe_bf16 *y_dev, void *workspace,
                                      size_t workspace_bytes, void *stream) {
    moe_status r = check_shape(shape);
    if (r != MOE_OK) return r;
    if (nbatch < 1 || !x_host || !y_host || !x_dev || !y_dev || !aligned16(x_dev) || !aligned16(y_dev))
        return MOE_ERR_INVALID_ARG;
    if (!weights_ok(shape, weights, true)) return MOE_ERR_INVALID_ARG;
    if (!weights_shape_supported(shape, weights)) return MOE_ERR_UNSUPPORTED;
    if ((r = check_ws(shape, MOE_WS_FORWARD, workspace, workspace_bytes)) != MOE_OK) return r;
    DeviceState *dev;
    if ((r = device_state(&dev)) != MOE_OK) return r;
    std::call_once(dev->io_once, [dev]() {
        cudaError_t e = cudaStreamCreateWithFlags(&dev->h2d, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&dev->d2h, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&dev->ev_start, cudaEventDisableTiming);
        for (int b = 0; b < 2 && e == cudaSuccess; ++b) {
            e = cudaEventCreateWithFlags(&dev->ev_in[b], cudaEventDisableTiming);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&dev->ev_fwd[b], cudaEventDisableTiming);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&dev->ev_out[b], cudaEventDisableTiming);
        }
        dev->io_err = e;
    });
    if (dev->io_err != cudaSuccess) return MOE_ERR_CUDA;
    // one caller at a time per device: the copy streams and events are shared
    std::lock_guard<std::mutex> lock(dev->io_mutex);
    cudaStream_t st = as_stream(stream);
    const size_t elems = (size_t)shape->T * shape->d_model, bytes = elems * sizeof(moe_bf16);
    auto ok = [](cudaError_t e) { return e == cudaSuccess; };
    // earlier work on `stream` may still use the device buffers
    if (!ok(cudaEventRecord(dev->ev_start, st)) || !ok(cudaStreamWaitEvent(dev->h2d, dev->ev_start, 0)) ||
        !ok(cudaStreamWaitEvent(dev->d2h, dev->ev_start, 0))) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    for (int32_t i = 0; i < nbatch; ++i) {
        const int b = i & 1;
        moe_bf16 *xb = x_dev + (size_t)b * elems, *yb = y_dev + (size_t)b * elems;
        // input copy into buffer b once batch i-2's forward has consumed it
        if (i >= 2 && !ok(cudaStreamWaitEvent(dev->h2d, dev->ev_fwd[b], 0))) break;
        if (!ok(cudaMemcpyAsync(xb, x_host + (size_t)i * host_stride, bytes, cudaMemcpyHostToDevice, dev->h2d)) ||
            !ok(cudaEventRecord(dev->ev_in[b], dev->h2d)))
            break;
        // forward once the input has landed and batch i-2's output copy has left buffer b
        if (!ok(cudaStreamWaitEvent(st, dev->ev_in[b], 0))) break;
        if (i >= 2 && !ok(cudaStreamWaitEvent(st, dev->ev_out[b], 0))) break;
        if ((r = moe_forward(shape, weights, xb, sel_bias, yb, nullptr, workspace, workspace_bytes, stream)) !=
            MOE_OK)
            return r;
        if (!ok(cudaEventRecord(dev->ev_fwd[b], st))) break;
        // output copy after the forward
        if (!ok(cudaStreamWaitEvent(dev->d2h, dev->ev_fwd[b], 0)) ||
            !ok(cudaMemcpyAsync(y_host + (size_t)i * host_stride, yb, bytes, cudaMemcpyDeviceToHost, dev->d2h)) ||
            !ok(cudaEventRecord(dev->ev_out[b], dev->d2h)))
            break;
        if (i + 1 == nbatch) {
            // `stream` completes after every copy
            if (!ok(cudaStreamWaitEvent(st, dev->ev_out[b], 0))) break;
            if (nbatch > 1 && !ok(cudaStreamWaitEvent(st, dev->ev_out[b ^ 1], 0))) break;
            return launch_status();
        }
    }
    cudaGetLastError();
    return MOE_ERR_CUDA;
}

moe_status moe_backward(const moe_shape *shape, const moe_weights *weights, const moe_bf16 *x,
                        const float *sel_bias, const moe_bf16 *dy, float g_aux, float g_z, const moe_grads *grads,
                        void *workspace, size_t workspace_bytes, void *stream) {
    moe_status r = check_shape(shape);
    if (r != MOE_OK) return r;
    if (!x || !dy || !aligned16(x) || !aligned16(dy) || !grads || !weights_ok(shape, weights, true))
        return MOE_ERR_INVALID_ARG;
    if (weights->format != MOE_WEIGHTS_BF16) return MOE_ERR_UNSUPPORTED;
    if (std::isnan(g_aux) || std::isnan(g_z)) return MOE_ERR_INVALID_ARG;
    const void *req[] = {grads->dx, grads->dWg, grads->dW1, grads->db1, grads->dW2, grads->db2};
    for (const void *p : req)
        if (p == nullptr || !aligned16(p)) return MOE_ERR_INVALID_ARG;
    if (shape->has_shared) {
        const void *sh[] = {grads->dWs1, grads->dbs1, grads->dWs2, grads->dbs2};
        for (const void *p : sh)
            if (p == nullptr || !aligned16(p)) return MOE_ERR_INVALID_ARG;
    }
    if ((r = check_ws(shape, MOE_WS_BACKWARD, workspace, workspace_bytes)) != MOE_OK) return r;
    DeviceState *dev;
    if ((r = device_state(&dev)) != MOE_OK) return r;
    Carve c(workspace);
    BackwardWs w = carve_backward(c, shape);
    return run_backward(shape, dev, weights, x, sel_bias, dy, g_aux, g_z, grads, w, as_stream(stream));
}

moe_status moe_get_device_error(int32_t clear, int32_t *code_out) {
    if (code_out == nullptr) return MOE_ERR_INVALID_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, moe::g_device_error, sizeof v) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    if (clear) {
        unsigned int zero = 0;
        if (cudaMemcpyToSymbol(moe::g_device_error, &zero, sizeof zero) != cudaSuccess) {
            cudaGetLastError();
            return MOE_ERR_CUDA;
        }
    }
    *code_out = (int32_t)v;
    return MOE_OK;
}

uint64_t moe_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
