"""Thin ctypes binding of libmoe.so (include/moe.h).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels. torch supplies device memory and the current stream. A missing or
unloadable library raises MoELibraryError; nothing here falls back to a CPU
or PyTorch implementation.
"""

from __future__ import annotations

import ctypes
import os
import re
from dataclasses import dataclass
from typing import Optional

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIBRARY = os.path.join(HERE, "libmoe.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "moe.h")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE, MOE_ERR_CUDA, MOE_ERR_DEVICE = range(6)
MOE_WS_FORWARD, MOE_WS_ROUTE, MOE_WS_DISPATCH, MOE_WS_FFN, MOE_WS_BACKWARD = range(5)
DEVERR_EXPERT_ID, DEVERR_ROW_INDEX, DEVERR_TIMEOUT, DEVERR_TILE_LIST = 1, 2, 4, 8


class MoELibraryError(RuntimeError):
    pass


class MoEError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {status} ({status_string(status)})")


class MoeShape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d_model", ctypes.c_int32), ("d_ff", ctypes.c_int32),
                ("N", ctypes.c_int32), ("K", ctypes.c_int32), ("capacity_factor", ctypes.c_float),
                ("has_shared", ctypes.c_int32), ("aux_alpha", ctypes.c_float), ("z_beta", ctypes.c_float),
                ("drop_policy", ctypes.c_int32), ("kl_coef", ctypes.c_float)]


MOE_WEIGHTS_BF16, MOE_WEIGHTS_FP8_E4M3, MOE_WEIGHTS_INT4_G128 = 0, 1, 2


class MoeWeights(ctypes.Structure):
    _fields_ = ([(n, ctypes.c_void_p) for n in ("Wg", "W1", "b1", "W2", "b2", "Ws1", "bs1", "Ws2", "bs2")]
                + [("format", ctypes.c_int32)]
                + [(n, ctypes.c_void_p) for n in ("W1q", "s1", "W2q", "s2", "Ws1q", "ss1", "Ws2q", "ss2")]
                + [(n, ctypes.c_void_p) for n in ("g1", "g2", "gs1", "gs2")])


class MoeGrads(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("dx", "dWg", "dW1", "db1", "dW2", "db2", "dWs1", "dbs1", "dWs2",
                                               "dbs2", "dw")]


class MoeRouteOut(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("topk_idx", "topk_w", "demand", "prob_sum", "kept",
                                               "expert_offsets", "slot_of", "aux", "z_loss", "aux_kl",
                                               "health", "mean_weight")]


_lib = None


def declared_functions() -> list:
    """Names of the entry points include/moe.h declares."""
    with open(HEADER) as fh:
        return re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", fh.read())


def load():
    """Load libmoe.so (built in-tree by ``python -m top_routing_expert_then_b300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIBRARY):
        raise MoELibraryError(f"{LIBRARY} is missing: build it with "
                              "`python -m top_routing_expert_then_b300.build` (needs nvcc)")
    try:
        lib = ctypes.CDLL(LIBRARY)
    except OSError as e:
        raise MoELibraryError(f"cannot load {LIBRARY}: {e}") from e
    P, S = ctypes.c_void_p, ctypes.POINTER(MoeShape)
    i32, sz = ctypes.c_int32, ctypes.c_size_t
    sig = {
        "moe_capacity": ([S], i32),
        "moe_workspace_bytes": ([S, i32], sz),
        "moe_status_string": ([i32], ctypes.c_char_p),
        "moe_route": ([S, P, P, P, P, P, P, P, P, sz, P], i32),
        "moe_route_noalloc": ([S, P, P, P, P, P, P, P, P], i32),
        "moe_dispatch": ([S, P, P, P, P, P, P, P, P, sz, P], i32),
        "moe_expert_ffn": ([S, P, P, ctypes.POINTER(MoeWeights), P, P, P, P, sz, P], i32),
        "moe_combine": ([S, P, P, P, P, P, P], i32),
        "moe_aux_loss": ([S, P, P, P, P], i32),
        "moe_forward": ([S, ctypes.POINTER(MoeWeights), P, P, P, ctypes.POINTER(MoeRouteOut), P, sz, P], i32),
        "moe_forward_marked": ([S, ctypes.POINTER(MoeWeights), P, P, P, ctypes.POINTER(MoeRouteOut), P, sz,
                                ctypes.POINTER(ctypes.c_void_p), P], i32),
        "moe_forward_hostio": ([S, ctypes.POINTER(MoeWeights), P, P, P, P, P, ctypes.POINTER(MoeRouteOut),
                                P, sz, P], i32),
        "moe_forward_hostio_batches": ([S, ctypes.POINTER(MoeWeights), i32, P, P, sz, P, P, P, P, sz, P], i32),
        "moe_backward": ([S, ctypes.POINTER(MoeWeights), P, P, P, ctypes.c_float, ctypes.c_float,
                          ctypes.POINTER(MoeGrads), P, sz, P], i32),
        "moe_get_device_error": ([i32, ctypes.POINTER(i32)], i32),
        "moe_launch_count": ([], ctypes.c_uint64),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().moe_status_string(status).decode()


def _check(fn: str, status: int):
    if status != MOE_OK:
        raise MoEError(fn, status)


def _ptr(t: Optional[torch.Tensor], dtype=None, what="tensor", numel=None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{what} must be {dtype}, got {t.dtype}")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{what} has {t.numel()} elements, needs {numel}")
    return t.data_ptr()


def _stream(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


MOE_DROP_TOKEN_ORDER, MOE_DROP_RANK_ORDER = 0, 1


def make_shape(T, d_model, d_ff, N, K, capacity_factor=0.0, has_shared=False, aux_alpha=0.01,
               z_beta=1e-3, rank_major=False, kl_coef=0.02) -> MoeShape:
    return MoeShape(int(T), int(d_model), int(d_ff), int(N), int(K), float(capacity_factor),
                    1 if has_shared else 0, float(aux_alpha), float(z_beta),
                    MOE_DROP_RANK_ORDER if rank_major else MOE_DROP_TOKEN_ORDER, float(kl_coef))


def shape_of(cfg) -> MoeShape:
    """moe_shape of an object with T, d_model, d_ff, N, K, capacity_factor,
    has_shared, aux_alpha (e.g. an inputs.MoEConfig)."""
    return make_shape(cfg.T, cfg.d_model, cfg.d_ff, cfg.N, cfg.K, cfg.capacity_factor, cfg.has_shared,
                      cfg.aux_alpha, getattr(cfg, "z_beta", 1e-3), getattr(cfg, "rank_major", False),
                      getattr(cfg, "kl_coef", 0.02))


def capacity(shape: MoeShape) -> int:
    return int(load().moe_capacity(ctypes.byref(shape)))


def workspace_bytes(shape: MoeShape, kind: int = MOE_WS_FORWARD) -> int:
    return int(load().moe_workspace_bytes(ctypes.byref(shape), kind))


def workspace(shape: MoeShape, kind: int = MOE_WS_FORWARD, device="cuda") -> torch.Tensor:
    n = workspace_bytes(shape, kind)
    if n == 0:
        raise MoEError("moe_workspace_bytes", MOE_ERR_INVALID_ARG)
    return torch.empty(n, dtype=torch.uint8, device=device)


def _ws(shape, kind, ws):
    if ws is None:
        ws = workspace(shape, kind)
    return ws, ws.data_ptr(), ws.numel()


# ------------------------------------------------------------------ stages

def route(shape: MoeShape, x, Wg, sel_bias=None, ws=None, stream=None):
    """-> (topk_idx [T,K] int32, topk_w [T,K] fp32, demand [N] int32, prob_sum [N] fp32)"""
    T, N, K = shape.T, shape.N, shape.K
    dev = x.device
    idx = torch.empty((T, K), dtype=torch.int32, device=dev)
    w = torch.empty((T, K), dtype=torch.float32, device=dev)
    demand = torch.empty((N,), dtype=torch.int32, device=dev)
    psum = torch.empty((N,), dtype=torch.float32, device=dev)
    ws, wp, wn = _ws(shape, MOE_WS_ROUTE, ws)
    _check("moe_route", load().moe_route(
        ctypes.byref(shape), _ptr(x, torch.bfloat16, "x", T * shape.d_model),
        _ptr(Wg, torch.bfloat16, "Wg", N * shape.d_model), _ptr(sel_bias, torch.float32, "sel_bias", N),
        idx.data_ptr(), w.data_ptr(), demand.data_ptr(), psum.data_ptr(), wp, wn, _stream(stream)))
    return idx, w, demand, psum


def route_noalloc(shape: MoeShape, x, Wg, sel_bias=None, stream=None):
    """moe_route without a workspace: the library's own fixed scratch array
    serves as scratch (for callers that cannot allocate device memory).
    -> (topk_idx, topk_w, demand, prob_sum)"""
    T, N, K = shape.T, shape.N, shape.K
    dev = x.device
    idx = torch.empty((T, K), dtype=torch.int32, device=dev)
    w = torch.empty((T, K), dtype=torch.float32, device=dev)
    demand = torch.empty((N,), dtype=torch.int32, device=dev)
    psum = torch.empty((N,), dtype=torch.float32, device=dev)
    _check("moe_route_noalloc", load().moe_route_noalloc(
        ctypes.byref(shape), _ptr(x, torch.bfloat16, "x", T * shape.d_model),
        _ptr(Wg, torch.bfloat16, "Wg", N * shape.d_model), _ptr(sel_bias, torch.float32, "sel_bias", N),
        idx.data_ptr(), w.data_ptr(), demand.data_ptr(), psum.data_ptr(), _stream(stream)))
    return idx, w, demand, psum


def dispatch(shape: MoeShape, topk_idx, x, ws=None, stream=None):
    """-> (kept [N], expert_offsets [N+1], slot_of [T,K], row_token [T*K], x_perm [T*K,d])"""
    T, N, K, d = shape.T, shape.N, shape.K, shape.d_model
    dev = x.device
    kept = torch.empty((N,), dtype=torch.int32, device=dev)
    offsets = torch.empty((N + 1,), dtype=torch.int32, device=dev)
    slot_of = torch.empty((T, K), dtype=torch.int32, device=dev)
    row_token = torch.empty((T * K,), dtype=torch.int32, device=dev)
    x_perm = torch.zeros((T * K, d), dtype=torch.bfloat16, device=dev)
    ws, wp, wn = _ws(shape, MOE_WS_DISPATCH, ws)
    _check("moe_dispatch", load().moe_dispatch(
        ctypes.byref(shape), _ptr(topk_idx, torch.int32, "topk_idx", T * K), _ptr(x, torch.bfloat16, "x", T * d),
        kept.data_ptr(), offsets.data_ptr(), slot_of.data_ptr(), row_token.data_ptr(), x_perm.data_ptr(),
        wp, wn, _stream(stream)))
    return kept, offsets, slot_of, row_token, x_perm


def weights_struct(W1, b1, W2, b2, Wg=None, Ws1=None, bs1=None, Ws2=None, bs2=None, quant=None) -> MoeWeights:
    """The C struct; with ``quant`` (codes and scales W1q, s1, W2q, s2 and the
    shared expert's Ws1q, ss1, Ws2q, ss2) the expert matrices are FP8 with fp32
    channel scales, or (quant.format == "int4_g128") INT4 with bf16 group
    scales (passed as g1, g2, gs1, gs2)."""
    bf, f32, u8 = torch.bfloat16, torch.float32, torch.uint8
    w = MoeWeights(_ptr(Wg, bf, "Wg"), _ptr(W1, bf, "W1"), _ptr(b1, f32, "b1"), _ptr(W2, bf, "W2"),
                   _ptr(b2, f32, "b2"), _ptr(Ws1, bf, "Ws1"), _ptr(bs1, f32, "bs1"), _ptr(Ws2, bf, "Ws2"),
                   _ptr(bs2, f32, "bs2"), MOE_WEIGHTS_BF16)
    if quant is not None and getattr(quant, "format", "fp8_e4m3") == "int4_g128":
        w.format = MOE_WEIGHTS_INT4_G128
        for n, dt, field in (("W1q", u8, "W1q"), ("s1", bf, "g1"), ("W2q", u8, "W2q"), ("s2", bf, "g2"),
                             ("Ws1q", u8, "Ws1q"), ("ss1", bf, "gs1"), ("Ws2q", u8, "Ws2q"), ("ss2", bf, "gs2")):
            setattr(w, field, _ptr(getattr(quant, n), dt, n))
    elif quant is not None:
        w.format = MOE_WEIGHTS_FP8_E4M3
        for n, dt in (("W1q", u8), ("s1", f32), ("W2q", u8), ("s2", f32), ("Ws1q", u8), ("ss1", f32),
                      ("Ws2q", u8), ("ss2", f32)):
            setattr(w, n, _ptr(getattr(quant, n), dt, n))
    return w


def _check_weights(shape: MoeShape, W1, b1, W2, b2, Ws1=None, bs1=None, Ws2=None, bs2=None, Wg=None, quant=None):
    N, d, f = shape.N, shape.d_model, shape.d_ff
    want = {"b1": (b1, (N, f)), "b2": (b2, (N, d))}
    int4 = quant is not None and getattr(quant, "format", "fp8_e4m3") == "int4_g128"
    if quant is None:
        want.update({"W1": (W1, (N, f, d)), "W2": (W2, (N, d, f))})
    elif int4:
        want.update({"W1q": (quant.W1q, (N, f, d // 2)), "s1": (quant.s1, (N, d // 128, f)),
                     "W2q": (quant.W2q, (N, d, f // 2)), "s2": (quant.s2, (N, f // 128, d))})
    else:
        want.update({"W1q": (quant.W1q, (N, f, d)), "s1": (quant.s1, (N, f)), "W2q": (quant.W2q, (N, d, f)),
                     "s2": (quant.s2, (N, d))})
    if Wg is not None:
        want["Wg"] = (Wg, (N, d))
    if shape.has_shared:
        want.update({"bs1": (bs1, (f,)), "bs2": (bs2, (d,))})
        if quant is None:
            want.update({"Ws1": (Ws1, (f, d)), "Ws2": (Ws2, (d, f))})
        elif int4:
            want.update({"Ws1q": (quant.Ws1q, (f, d // 2)), "ss1": (quant.ss1, (d // 128, f)),
                         "Ws2q": (quant.Ws2q, (d, f // 2)), "ss2": (quant.ss2, (f // 128, d))})
        else:
            want.update({"Ws1q": (quant.Ws1q, (f, d)), "ss1": (quant.ss1, (f,)), "Ws2q": (quant.Ws2q, (d, f)),
                         "ss2": (quant.ss2, (d,))})
    for name, (t, shp) in want.items():
        if t is None or tuple(t.shape) != shp:
            raise ValueError(f"{name} must have shape {shp}, got {None if t is None else tuple(t.shape)}")


def expert_ffn(shape: MoeShape, x_perm, expert_offsets, W1, b1, W2, b2, x=None, Ws1=None, bs1=None, Ws2=None,
               bs2=None, ws=None, stream=None, quant=None):
    """-> (y_perm [T*K, d], z [T, d] or None); ``quant``: quantised expert weights."""
    T, K, d = shape.T, shape.K, shape.d_model
    _check_weights(shape, W1, b1, W2, b2, Ws1, bs1, Ws2, bs2, quant=quant)
    dev = x_perm.device
    y_perm = torch.zeros((T * K, d), dtype=torch.bfloat16, device=dev)
    z = torch.empty((T, d), dtype=torch.bfloat16, device=dev) if shape.has_shared else None
    wts = weights_struct(W1, b1, W2, b2, None, Ws1, bs1, Ws2, bs2, quant=quant)
    ws, wp, wn = _ws(shape, MOE_WS_FFN, ws)
    _check("moe_expert_ffn", load().moe_expert_ffn(
        ctypes.byref(shape), _ptr(x_perm, torch.bfloat16, "x_perm", T * K * d),
        _ptr(expert_offsets, torch.int32, "expert_offsets", shape.N + 1), ctypes.byref(wts),
        _ptr(x, torch.bfloat16, "x", T * d), y_perm.data_ptr(), None if z is None else z.data_ptr(),
        wp, wn, _stream(stream)))
    return y_perm, z


def combine(shape: MoeShape, y_perm, slot_of, topk_w, z=None, stream=None):
    T, K, d = shape.T, shape.K, shape.d_model
    y = torch.empty((T, d), dtype=torch.bfloat16, device=y_perm.device)
    _check("moe_combine", load().moe_combine(
        ctypes.byref(shape), _ptr(y_perm, torch.bfloat16, "y_perm", T * K * d),
        _ptr(slot_of, torch.int32, "slot_of", T * K), _ptr(topk_w, torch.float32, "topk_w", T * K),
        _ptr(z, torch.bfloat16, "z", T * d), y.data_ptr(), _stream(stream)))
    return y


def aux_loss(shape: MoeShape, demand, prob_sum, stream=None):
    aux = torch.empty((1,), dtype=torch.float32, device=demand.device)
    _check("moe_aux_loss", load().moe_aux_loss(
        ctypes.byref(shape), _ptr(demand, torch.int32, "demand", shape.N),
        _ptr(prob_sum, torch.float32, "prob_sum", shape.N), aux.data_ptr(), _stream(stream)))
    return aux


def device_error(clear: bool = True) -> int:
    code = ctypes.c_int32(0)
    _check("moe_get_device_error", load().moe_get_device_error(1 if clear else 0, ctypes.byref(code)))
    return int(code.value)


def launch_count() -> int:
    return int(load().moe_launch_count())


# ------------------------------------------------------------------ the whole layer

@dataclass
class RouteOutputs:
    topk_idx: torch.Tensor
    topk_w: torch.Tensor
    demand: torch.Tensor
    prob_sum: torch.Tensor
    kept: torch.Tensor
    expert_offsets: torch.Tensor
    slot_of: torch.Tensor
    aux: torch.Tensor
    z_loss: torch.Tensor
    aux_kl: torch.Tensor
    health: torch.Tensor
    mean_weight: torch.Tensor


class MoELayer:
    """One MoE layer's weights plus a forward workspace, all on one device."""

    def __init__(self, shape: MoeShape, Wg, W1, b1, W2, b2, Ws1=None, bs1=None, Ws2=None, bs2=None, quant=None):
        _check_weights(shape, W1, b1, W2, b2, Ws1, bs1, Ws2, bs2, Wg=Wg, quant=quant)
        self.shape = shape
        self.tensors = (Wg, W1, b1, W2, b2, Ws1, bs1, Ws2, bs2, quant)  # keep alive
        self.weights = weights_struct(W1, b1, W2, b2, Wg, Ws1, bs1, Ws2, bs2, quant=quant)
        self.device = Wg.device
        self.ws = workspace(shape, MOE_WS_FORWARD, self.device)

    @classmethod
    def from_inputs(cls, inp) -> "MoELayer":
        """From an inputs.MoEInputs already on the GPU."""
        return cls(shape_of(inp.cfg), inp.Wg, inp.W1, inp.b1, inp.W2, inp.b2, inp.Ws1, inp.bs1, inp.Ws2, inp.bs2,
                   quant=getattr(inp, "quant", None))

    def route_outputs(self) -> RouteOutputs:
        T, N, K, dev = self.shape.T, self.shape.N, self.shape.K, self.device
        i32, f32 = torch.int32, torch.float32
        return RouteOutputs(torch.empty((T, K), dtype=i32, device=dev), torch.empty((T, K), dtype=f32, device=dev),
                            torch.empty((N,), dtype=i32, device=dev), torch.empty((N,), dtype=f32, device=dev),
                            torch.empty((N,), dtype=i32, device=dev), torch.empty((N + 1,), dtype=i32, device=dev),
                            torch.empty((T, K), dtype=i32, device=dev), torch.empty((1,), dtype=f32, device=dev),
                            torch.empty((1,), dtype=f32, device=dev), torch.empty((1,), dtype=f32, device=dev),
                            torch.empty((4,), dtype=f32, device=dev), torch.empty((N,), dtype=f32, device=dev))

    @staticmethod
    def _out_struct(ro: Optional[RouteOutputs]):
        if ro is None:
            return None
        return ctypes.byref(MoeRouteOut(*(getattr(ro, n).data_ptr() for n in (
            "topk_idx", "topk_w", "demand", "prob_sum", "kept", "expert_offsets", "slot_of", "aux", "z_loss",
            "aux_kl", "health", "mean_weight"))))

    def forward(self, x, sel_bias=None, y=None, route_out: Optional[RouteOutputs] = None, stream=None):
        s = self.shape
        if y is None:
            y = torch.empty((s.T, s.d_model), dtype=torch.bfloat16, device=self.device)
        _check("moe_forward", load().moe_forward(
            ctypes.byref(s), ctypes.byref(self.weights), _ptr(x, torch.bfloat16, "x", s.T * s.d_model),
            _ptr(sel_bias, torch.float32, "sel_bias", s.N), _ptr(y, torch.bfloat16, "y", s.T * s.d_model),
            self._out_struct(route_out), self.ws.data_ptr(), self.ws.numel(), _stream(stream)))
        return y

    def forward_hostio_batches(self, x_host, y_host, nbatch: int, x_dev, y_dev, sel_bias=None, same_host=False,
                               stream=None):
        """moe_forward_hostio_batches: nbatch host-to-host forwards with the copies
        overlapped. x_host / y_host: pinned CPU bf16 tensors [nbatch, T, d] (or
        [T, d] with same_host=True: every batch reuses them); x_dev / y_dev:
        device bf16 tensors [2, T, d]."""
        s = self.shape
        td = s.T * s.d_model
        for name, t in (("x_host", x_host), ("y_host", y_host)):
            if t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous CPU bf16 tensor")
            if t.numel() != (td if same_host else nbatch * td):
                raise ValueError(f"{name} has {t.numel()} elements")
        _check("moe_forward_hostio_batches", load().moe_forward_hostio_batches(
            ctypes.byref(s), ctypes.byref(self.weights), int(nbatch), x_host.data_ptr(), y_host.data_ptr(),
            0 if same_host else td, _ptr(sel_bias, torch.float32, "sel_bias", s.N),
            _ptr(x_dev, torch.bfloat16, "x_dev", 2 * td), _ptr(y_dev, torch.bfloat16, "y_dev", 2 * td),
            self.ws.data_ptr(), self.ws.numel(), _stream(stream)))

    def backward(self, x, dy, sel_bias=None, g_aux: float = 1.0, g_z: float = 1.0, ws=None, stream=None) -> dict:
        """moe_backward: fp32 gradients {dx, dWg, dW1, db1, dW2, db2, dw (+ dWs1, dbs1, dWs2, dbs2)} of
        <dy, y> + g_aux * aux + g_z * z_loss for this layer at x."""
        s = self.shape
        T, d, f, N, K, dev = s.T, s.d_model, s.d_ff, s.N, s.K, self.device
        e = lambda *shape: torch.empty(shape, dtype=torch.float32, device=dev)  # noqa: E731
        g = {"dx": e(T, d), "dWg": e(N, d), "dW1": e(N, f, d), "db1": e(N, f), "dW2": e(N, d, f), "db2": e(N, d),
             "dw": e(T, K)}
        if s.has_shared:
            g.update({"dWs1": e(f, d), "dbs1": e(f), "dWs2": e(d, f), "dbs2": e(d)})
        gs = MoeGrads(*(g[n].data_ptr() if n in g else None for n in (
            "dx", "dWg", "dW1", "db1", "dW2", "db2", "dWs1", "dbs1", "dWs2", "dbs2", "dw")))
        ws, wp, wn = _ws(s, MOE_WS_BACKWARD, ws)
        _check("moe_backward", load().moe_backward(
            ctypes.byref(s), ctypes.byref(self.weights), _ptr(x, torch.bfloat16, "x", T * d),
            _ptr(sel_bias, torch.float32, "sel_bias", N), _ptr(dy, torch.bfloat16, "dy", T * d), float(g_aux),
            float(g_z), ctypes.byref(gs), wp, wn, _stream(stream)))
        return g

    def forward_marked(self, x, events, sel_bias=None, y=None, route_out: Optional[RouteOutputs] = None,
                       stream=None):
        """forward() that records 6 torch.cuda.Event marks at the stage boundaries
        (before routing, after routing, after dispatch, after the first grouped
        GEMM, after the second, after combine + aux)."""
        s = self.shape
        if len(events) != 6:
            raise ValueError("need 6 events")
        if y is None:
            y = torch.empty((s.T, s.d_model), dtype=torch.bfloat16, device=self.device)
        ev = (ctypes.c_void_p * 6)(*[None if e is None else e.cuda_event for e in events])
        _check("moe_forward_marked", load().moe_forward_marked(
            ctypes.byref(s), ctypes.byref(self.weights), _ptr(x, torch.bfloat16, "x", s.T * s.d_model),
            _ptr(sel_bias, torch.float32, "sel_bias", s.N), _ptr(y, torch.bfloat16, "y", s.T * s.d_model),
            self._out_struct(route_out), self.ws.data_ptr(), self.ws.numel(), ev, _stream(stream)))
        return y

    def forward_hostio(self, x_host: torch.Tensor, y_host: torch.Tensor, x_dev, y_dev, sel_bias=None,
                       route_out: Optional[RouteOutputs] = None, stream=None):
        """x_host / y_host: CPU bf16 tensors (pin them for asynchronous copies)."""
        s = self.shape
        for name, t in (("x_host", x_host), ("y_host", y_host)):
            if t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous() or t.numel() < s.T * s.d_model:
                raise ValueError(f"{name} must be a contiguous CPU bf16 tensor of T*d_model elements")
        _check("moe_forward_hostio", load().moe_forward_hostio(
            ctypes.byref(s), ctypes.byref(self.weights), x_host.data_ptr(),
            _ptr(x_dev, torch.bfloat16, "x_dev", s.T * s.d_model), _ptr(sel_bias, torch.float32, "sel_bias", s.N),
            _ptr(y_dev, torch.bfloat16, "y_dev", s.T * s.d_model), y_host.data_ptr(), self._out_struct(route_out),
            self.ws.data_ptr(), self.ws.numel(), _stream(stream)))
        return y_host
