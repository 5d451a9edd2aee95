"""CPU oracle of the MoE layer forward pass -- TEST INFRASTRUCTURE.

A ctypes shim over ``moe_oracle.c`` (plain C, IEEE double). Only the test
suite, the package smoke check and the benchmark's CPU-baseline leg may import
this module; the product path never does, and nothing here imports the product
package. ``moe_oracle.c`` names the page passage each step follows.

bf16 tensors cross this boundary as their raw 16-bit patterns (numpy uint16).
Torch CPU tensors are accepted and converted.

``Oracle(path)`` wraps any build of the C source; the module-level functions use
the default build next to this file. (The test suite also builds deliberately
broken copies of the source to show that its pins catch planted mistakes.)
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass
from typing import Optional

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "moe_oracle.c")
LIBRARY = os.path.join(HERE, "libmoe_oracle.so")
CFLAGS = ["-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-Wall", "-Wextra"]


def compile_source(src: str, out: str) -> str:
    """gcc build of an oracle source file (no -ffast-math: IEEE semantics)."""
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, src, "-lm"])
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    if force or not os.path.exists(LIBRARY) or os.path.getmtime(LIBRARY) < os.path.getmtime(SOURCE):
        compile_source(SOURCE, LIBRARY)
    return LIBRARY


# ------------------------------------------------------------------ marshalling

def _np(a, dtype):
    """Contiguous numpy array of ``dtype``; bf16 torch tensors -> uint16 bits."""
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor
        import torch
        a = a.detach().cpu().contiguous()
        if a.dtype == torch.bfloat16:
            a = a.view(torch.int16).numpy().view(np.uint16)
        else:
            a = a.numpy()
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        if dtype == np.uint16:
            raise TypeError("bf16 operands must be bf16 tensors or uint16 bit patterns")
        a = np.ascontiguousarray(a.astype(dtype))
    return a


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def bf16_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns -> float64 values (exact)."""
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@dataclass
class OracleResult:
    logits: np.ndarray     # [T, N] float64
    topk_idx: np.ndarray   # [T, K] int32
    topk_w: np.ndarray     # [T, K] float32
    demand: np.ndarray     # [N] int32
    P: np.ndarray          # [N] float64 (mean over tokens of the full softmax)
    capacity: int
    kept: np.ndarray       # [N] int32
    offsets: np.ndarray    # [N+1] int32
    slot_of: np.ndarray    # [T, K] int32
    row_token: np.ndarray  # [T*K] int32
    y_perm: Optional[np.ndarray]  # [R, d] uint16 (bf16 bits); rows of unwanted tokens are 0
    z: Optional[np.ndarray]       # [T, d] uint16 or None
    y: Optional[np.ndarray]       # [T, d] uint16; rows of unwanted tokens are 0
    aux: float
    z_loss: float
    aux_kl: float = 0.0
    health: Optional[np.ndarray] = None      # util_std, drop_rate, mean entropy, max |logit|
    mean_weight: Optional[np.ndarray] = None  # [N]


class Oracle:
    def __init__(self, path: Optional[str] = None):
        lib = ctypes.CDLL(path or build())
        P = ctypes.c_void_p
        i32, f64 = ctypes.c_int32, ctypes.c_double
        lib.oracle_bf16_value.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_value.restype = f64
        lib.oracle_bf16_round.argtypes = [f64]
        lib.oracle_bf16_round.restype = ctypes.c_uint16
        lib.oracle_gelu.argtypes = [f64]
        lib.oracle_gelu.restype = f64
        lib.oracle_capacity.argtypes = [i32, i32, f64]
        lib.oracle_capacity.restype = i32
        lib.oracle_gate_logits.argtypes = [i32, i32, i32, P, P, P]
        lib.oracle_route.argtypes = [i32, i32, i32, P, P, P, P, P, P]
        lib.oracle_dispatch.argtypes = [i32, i32, i32, i32, P, P, P, P, P]
        lib.oracle_dispatch_ordered.argtypes = [i32, i32, i32, i32, i32, P, P, P, P, P]
        lib.oracle_aux_kl.argtypes = [i32, i32, i32, f64, P]
        lib.oracle_aux_kl.restype = f64
        lib.oracle_expert_rows.argtypes = [i32, i32, i32, P, P, P, P, P, P, P]
        lib.oracle_expert_ffn.argtypes = [i32, i32, i32, i32, P, P, P, P, P, P, P, P, P]
        lib.oracle_shared_ffn.argtypes = [i32, i32, i32, P, P, P, P, P, P, P]
        lib.oracle_expert_ffn_fp8.argtypes = [i32, i32, i32, i32, P, P, P, P, P, P, P, P, P, P, P]
        lib.oracle_shared_ffn_fp8.argtypes = [i32, i32, i32, P, P, P, P, P, P, P, P, P]
        lib.oracle_expert_ffn_int4.argtypes = [i32, i32, i32, i32, P, P, P, P, P, P, P, P, P, P, P]
        lib.oracle_shared_ffn_int4.argtypes = [i32, i32, i32, P, P, P, P, P, P, P, P, P]
        lib.oracle_int4_dequant.restype = f64
        lib.oracle_int4_dequant.argtypes = [i32, ctypes.c_uint16]
        lib.oracle_backward.argtypes = [i32, i32, i32, i32, i32] + [P] * 17 + [f64, f64, f64, f64, i32] + [P] * 12
        lib.oracle_combine_backward.argtypes = [i32, i32, i32, P, P, P, P]
        lib.oracle_gate_backward.argtypes = [i32, i32, i32, i32, P, P, P, P, P, f64, f64, f64, f64, P]
        lib.oracle_expert_backward.argtypes = [i32, i32, i32, i32, i32, i32] + [P] * 11 + [i32] + [P] * 4
        lib.oracle_health.argtypes = [i32, i32, i32, P, P, P, P, P, P, P]
        lib.oracle_fp8_value.restype = f64
        lib.oracle_fp8_value.argtypes = [ctypes.c_uint8]
        lib.oracle_combine.argtypes = [i32, i32, i32, P, P, P, P, P, P]
        lib.oracle_aux_loss.argtypes = [i32, i32, i32, f64, P, P]
        lib.oracle_aux_loss.restype = f64
        lib.oracle_z_loss.argtypes = [i32, i32, P, f64]
        lib.oracle_z_loss.restype = f64
        self.lib = lib

    # ---- scalar helpers
    def bf16_round(self, v: float) -> int:
        return int(self.lib.oracle_bf16_round(float(v)))

    def gelu(self, v: float) -> float:
        return float(self.lib.oracle_gelu(float(v)))

    def capacity(self, T: int, N: int, capacity_factor: float) -> int:
        return int(self.lib.oracle_capacity(T, N, float(capacity_factor)))

    # ---- stages
    def gate_logits(self, x, Wg) -> np.ndarray:
        x = _np(x, np.uint16)
        Wg = _np(Wg, np.uint16)
        T, d = x.shape
        N = Wg.shape[0]
        s = np.empty((T, N), dtype=np.float64)
        self.lib.oracle_gate_logits(T, d, N, _p(x), _p(Wg), _p(s))
        return s

    def route(self, s, K: int, sel_bias=None):
        s = _np(s, np.float64)
        T, N = s.shape
        sb = _np(sel_bias, np.float32)
        idx = np.empty((T, K), dtype=np.int32)
        w = np.empty((T, K), dtype=np.float32)
        demand = np.empty((N,), dtype=np.int32)
        P = np.empty((N,), dtype=np.float64)
        self.lib.oracle_route(T, N, K, _p(s), _p(sb), _p(idx), _p(w), _p(demand), _p(P))
        return idx, w, demand, P

    def dispatch(self, idx, N: int, C: int, rank_major: bool = False):
        idx = _np(idx, np.int32)
        T, K = idx.shape
        kept = np.empty((N,), dtype=np.int32)
        offsets = np.empty((N + 1,), dtype=np.int32)
        slot_of = np.empty((T, K), dtype=np.int32)
        row_token = np.empty((T * K,), dtype=np.int32)
        if rank_major:
            self.lib.oracle_dispatch_ordered(T, N, K, C, 1, _p(idx), _p(kept), _p(offsets), _p(slot_of),
                                             _p(row_token))
        else:
            self.lib.oracle_dispatch(T, N, K, C, _p(idx), _p(kept), _p(offsets), _p(slot_of), _p(row_token))
        return kept, offsets, slot_of, row_token

    def aux_kl(self, demand, T: int, K: int, coef: float) -> float:
        demand = _np(demand, np.int32)
        return float(self.lib.oracle_aux_kl(T, demand.shape[0], K, float(coef), _p(demand)))

    def expert_rows(self, x, rows, W1e, b1e, W2e, b2e) -> np.ndarray:
        """One expert's FFN on x[rows[i]]."""
        x = _np(x, np.uint16)
        rows = _np(rows, np.int32)
        W1e, W2e = _np(W1e, np.uint16), _np(W2e, np.uint16)
        b1e, b2e = _np(b1e, np.float32), _np(b2e, np.float32)
        d = x.shape[1]
        f = W1e.shape[0]
        out = np.empty((rows.shape[0], d), dtype=np.uint16)
        self.lib.oracle_expert_rows(d, f, rows.shape[0], _p(rows), _p(x), _p(W1e), _p(b1e),
                                    _p(W2e), _p(b2e), _p(out))
        return out

    def expert_ffn(self, x, offsets, row_token, W1, b1, W2, b2, want=None) -> np.ndarray:
        x = _np(x, np.uint16)
        offsets, row_token = _np(offsets, np.int32), _np(row_token, np.int32)
        W1, W2 = _np(W1, np.uint16), _np(W2, np.uint16)
        b1, b2 = _np(b1, np.float32), _np(b2, np.float32)
        want = _np(want, np.uint8)
        T, d = x.shape
        N, f = W1.shape[0], W1.shape[1]
        y_perm = np.zeros((max(int(offsets[N]), 0), d), dtype=np.uint16)
        self.lib.oracle_expert_ffn(T, d, f, N, _p(offsets), _p(row_token), _p(x), _p(W1), _p(b1),
                                   _p(W2), _p(b2), _p(want), _p(y_perm))
        return y_perm

    def health(self, s, demand, kept, idx, w):
        """-> (h [4]: util_std, drop_rate, mean entropy, max |logit|; mean_w [N])."""
        s = np.ascontiguousarray(s, dtype=np.float64)
        T, N = s.shape
        idx = _np(idx, np.int32)
        K = idx.shape[1]
        h = np.zeros(4)
        mw = np.zeros(N)
        self.lib.oracle_health(T, N, K, _p(s), _p(_np(demand, np.int32)), _p(_np(kept, np.int32)), _p(idx),
                               _p(_np(w, np.float32)), _p(h), _p(mw))
        return h, mw

    def fp8_value(self, code: int) -> float:
        return float(self.lib.oracle_fp8_value(int(code)))

    def expert_ffn_fp8(self, x, offsets, row_token, W1q, s1, b1, W2q, s2, b2, want=None) -> np.ndarray:
        """expert_ffn with FP8 E4M3 weight codes (uint8) and per-output-channel scales."""
        x = _np(x, np.uint16)
        offsets, row_token = _np(offsets, np.int32), _np(row_token, np.int32)
        W1q, W2q = _np(W1q, np.uint8), _np(W2q, np.uint8)
        s1, s2 = _np(s1, np.float32), _np(s2, np.float32)
        b1, b2 = _np(b1, np.float32), _np(b2, np.float32)
        want = _np(want, np.uint8)
        T, d = x.shape
        N, f = W1q.shape[0], W1q.shape[1]
        y_perm = np.zeros((max(int(offsets[N]), 0), d), dtype=np.uint16)
        self.lib.oracle_expert_ffn_fp8(T, d, f, N, _p(offsets), _p(row_token), _p(x), _p(W1q), _p(s1), _p(b1),
                                       _p(W2q), _p(s2), _p(b2), _p(want), _p(y_perm))
        return y_perm

    def shared_ffn_fp8(self, x, Ws1q, ss1, bs1, Ws2q, ss2, bs2, want=None) -> np.ndarray:
        x = _np(x, np.uint16)
        Ws1q, Ws2q = _np(Ws1q, np.uint8), _np(Ws2q, np.uint8)
        ss1, ss2 = _np(ss1, np.float32), _np(ss2, np.float32)
        bs1, bs2 = _np(bs1, np.float32), _np(bs2, np.float32)
        want = _np(want, np.uint8)
        T, d = x.shape
        f = Ws1q.shape[0]
        z = np.zeros((T, d), dtype=np.uint16)
        self.lib.oracle_shared_ffn_fp8(T, d, f, _p(x), _p(Ws1q), _p(ss1), _p(bs1), _p(Ws2q), _p(ss2), _p(bs2),
                                       _p(want), _p(z))
        return z

    def int4_dequant(self, code: int, scale_bits: int) -> float:
        """The dequantised INT4 weight: bf16(RNE) of (code - 8) * scale."""
        return float(self.lib.oracle_int4_dequant(int(code), int(scale_bits)))

    def expert_ffn_int4(self, x, offsets, row_token, W1q4, g1, b1, W2q4, g2, b2, want=None) -> np.ndarray:
        """expert_ffn with INT4 group-wise weights: packed codes [N, out, in / 2]
        (eight columns to a little-endian 32-bit word, column 2j of the run in
        bits 4j.., 2j + 1 in bits 16 + 4j..) and bf16 group scales [N, in / 128, out]."""
        x = _np(x, np.uint16)
        offsets, row_token = _np(offsets, np.int32), _np(row_token, np.int32)
        W1q4, W2q4 = _np(W1q4, np.uint8), _np(W2q4, np.uint8)
        g1, g2 = _np(g1, np.uint16), _np(g2, np.uint16)
        b1, b2 = _np(b1, np.float32), _np(b2, np.float32)
        want = _np(want, np.uint8)
        T, d = x.shape
        N, f = W1q4.shape[0], W1q4.shape[1]
        y_perm = np.zeros((max(int(offsets[N]), 0), d), dtype=np.uint16)
        self.lib.oracle_expert_ffn_int4(T, d, f, N, _p(offsets), _p(row_token), _p(x), _p(W1q4), _p(g1), _p(b1),
                                        _p(W2q4), _p(g2), _p(b2), _p(want), _p(y_perm))
        return y_perm

    def shared_ffn_int4(self, x, Ws1q4, gs1, bs1, Ws2q4, gs2, bs2, want=None) -> np.ndarray:
        x = _np(x, np.uint16)
        Ws1q4, Ws2q4 = _np(Ws1q4, np.uint8), _np(Ws2q4, np.uint8)
        gs1, gs2 = _np(gs1, np.uint16), _np(gs2, np.uint16)
        bs1, bs2 = _np(bs1, np.float32), _np(bs2, np.float32)
        want = _np(want, np.uint8)
        T, d = x.shape
        f = Ws1q4.shape[0]
        z = np.zeros((T, d), dtype=np.uint16)
        self.lib.oracle_shared_ffn_int4(T, d, f, _p(x), _p(Ws1q4), _p(gs1), _p(bs1), _p(Ws2q4), _p(gs2), _p(bs2),
                                        _p(want), _p(z))
        return z

    def shared_ffn(self, x, Ws1, bs1, Ws2, bs2, want=None) -> np.ndarray:
        x = _np(x, np.uint16)
        Ws1, Ws2 = _np(Ws1, np.uint16), _np(Ws2, np.uint16)
        bs1, bs2 = _np(bs1, np.float32), _np(bs2, np.float32)
        want = _np(want, np.uint8)
        T, d = x.shape
        f = Ws1.shape[0]
        z = np.zeros((T, d), dtype=np.uint16)
        self.lib.oracle_shared_ffn(T, d, f, _p(x), _p(Ws1), _p(bs1), _p(Ws2), _p(bs2), _p(want), _p(z))
        return z

    def combine(self, y_perm, slot_of, w, d: int, z=None, want=None) -> np.ndarray:
        y_perm = _np(y_perm, np.uint16)
        if y_perm.size == 0:
            y_perm = np.zeros((1, d), dtype=np.uint16)  # never read: every slot is -1
        slot_of = _np(slot_of, np.int32)
        w = _np(w, np.float32)
        z = _np(z, np.uint16)
        want = _np(want, np.uint8)
        T, K = slot_of.shape
        y = np.zeros((T, d), dtype=np.uint16)
        self.lib.oracle_combine(T, d, K, _p(y_perm), _p(slot_of), _p(w), _p(z), _p(want), _p(y))
        return y

    def aux_loss(self, demand, P, T: int, K: int, alpha: float) -> float:
        demand = _np(demand, np.int32)
        P = _np(P, np.float64)
        return float(self.lib.oracle_aux_loss(T, demand.shape[0], K, float(alpha), _p(demand), _p(P)))

    def z_loss(self, s, beta: float) -> float:
        s = _np(s, np.float64)
        T, N = s.shape
        return float(self.lib.oracle_z_loss(T, N, _p(s), float(beta)))

    def backward(self, x, Wg, W1, b1, W2, b2, fwd: "OracleResult", dy, aux_alpha: float, z_beta: float,
                 g_aux: float = 1.0, g_z: float = 1.0, Ws1=None, bs1=None, Ws2=None, bs2=None,
                 round_stored: bool = True, want=None) -> dict:
        """Gradients of the layer (see oracle_backward in moe_oracle.c) for the
        routing decisions of ``fwd`` and the upstream gradient ``dy`` [T, d]
        (bf16). Returns float64 arrays dx, dWg, dW1, db1, dW2, db2, dw (and
        dWs1, dbs1, dWs2, dbs2 with a shared expert). ``want`` (bool [T])
        limits the work to those tokens' dx and dw."""
        x, Wg = _np(x, np.uint16), _np(Wg, np.uint16)
        W1, W2 = _np(W1, np.uint16), _np(W2, np.uint16)
        b1, b2 = _np(b1, np.float32), _np(b2, np.float32)
        dy = _np(dy, np.uint16)
        T, d = x.shape
        N, f = W1.shape[0], W1.shape[1]
        K = fwd.topk_idx.shape[1]
        shared = Ws1 is not None
        if shared:
            Ws1, Ws2 = _np(Ws1, np.uint16), _np(Ws2, np.uint16)
            bs1, bs2 = _np(bs1, np.float32), _np(bs2, np.float32)
        out = {"dx": np.zeros((T, d)), "dw": np.zeros((T, K))}
        if want is None:
            out.update({"dWg": np.zeros((N, d)), "dW1": np.zeros((N, f, d)), "db1": np.zeros((N, f)),
                        "dW2": np.zeros((N, d, f)), "db2": np.zeros((N, d))})
        if shared and want is None:
            out.update({"dWs1": np.zeros((f, d)), "dbs1": np.zeros(f), "dWs2": np.zeros((d, f)),
                        "dbs2": np.zeros(d)})
        s = np.ascontiguousarray(fwd.logits, dtype=np.float64)
        self.lib.oracle_backward(
            T, d, f, N, K, _p(x), _p(Wg), _p(W1), _p(b1), _p(W2), _p(b2), _p(Ws1), _p(bs1), _p(Ws2), _p(bs2),
            _p(s), _p(np.ascontiguousarray(fwd.topk_idx, np.int32)), _p(np.ascontiguousarray(fwd.slot_of, np.int32)),
            _p(np.ascontiguousarray(fwd.offsets, np.int32)), _p(np.ascontiguousarray(fwd.row_token, np.int32)),
            _p(np.ascontiguousarray(fwd.demand, np.int32)), _p(dy), float(aux_alpha), float(z_beta), float(g_aux),
            float(g_z), 1 if round_stored else 0,
            _p(None if want is None else np.ascontiguousarray(np.asarray(want).astype(np.uint8))),
            _p(out["dx"]), _p(out.get("dWg")), _p(out.get("dW1")), _p(out.get("db1")),
            _p(out.get("dW2")), _p(out.get("db2")), _p(out.get("dWs1")), _p(out.get("dbs1")), _p(out.get("dWs2")),
            _p(out.get("dbs2")), _p(out["dw"]))
        return out

    # ---- pieces of the backward (for full-size checks)
    def combine_backward(self, dy, y_perm, slot_of) -> np.ndarray:
        """dw [T, K] = <dy_t, o_tk> from the forward's stored expert outputs."""
        dy = _np(dy, np.uint16)
        y_perm = _np(y_perm, np.uint16)
        if y_perm.size == 0:
            y_perm = np.zeros((1, dy.shape[1]), dtype=np.uint16)  # never read: every slot is -1
        slot_of = _np(slot_of, np.int32)
        T, d = dy.shape
        K = slot_of.shape[1]
        dw = np.zeros((T, K))
        self.lib.oracle_combine_backward(T, d, K, _p(dy), _p(y_perm), _p(slot_of), _p(dw))
        return dw

    def gate_backward(self, x, fwd: "OracleResult", dw, aux_alpha: float, z_beta: float, g_aux: float = 1.0,
                      g_z: float = 1.0) -> np.ndarray:
        """dW_g [N, d] from the slot gradients dw [T, K] and the forward's routing."""
        x = _np(x, np.uint16)
        T, d = x.shape
        s = np.ascontiguousarray(fwd.logits, dtype=np.float64)
        N = s.shape[1]
        K = fwd.topk_idx.shape[1]
        dWg = np.zeros((N, d))
        self.lib.oracle_gate_backward(T, d, N, K, _p(x), _p(s), _p(np.ascontiguousarray(fwd.topk_idx, np.int32)),
                                      _p(np.ascontiguousarray(dw, np.float64)),
                                      _p(np.ascontiguousarray(fwd.demand, np.int32)), float(aux_alpha),
                                      float(z_beta), float(g_aux), float(g_z), _p(dWg))
        return dWg

    def expert_backward(self, x, fwd: "OracleResult", e: int, W1e, b1e, W2e, b2e, dy,
                        round_stored: bool = True) -> dict:
        """Weight and bias gradients of routed expert e (e >= 0) or of the
        shared expert (e < 0, weight 1 on every token): dW1 [f, d], db1 [f],
        dW2 [d, f], db2 [d]."""
        x = _np(x, np.uint16)
        W1e, W2e = _np(W1e, np.uint16), _np(W2e, np.uint16)
        b1e, b2e = _np(b1e, np.float32), _np(b2e, np.float32)
        dy = _np(dy, np.uint16)
        T, d = x.shape
        f = W1e.shape[0]
        s = np.ascontiguousarray(fwd.logits, dtype=np.float64)
        N = s.shape[1]
        K = fwd.topk_idx.shape[1]
        out = {"dW1": np.zeros((f, d)), "db1": np.zeros(f), "dW2": np.zeros((d, f)), "db2": np.zeros(d)}
        self.lib.oracle_expert_backward(
            T, d, f, N, K, int(e), _p(s), _p(np.ascontiguousarray(fwd.topk_idx, np.int32)),
            _p(np.ascontiguousarray(fwd.slot_of, np.int32)), _p(np.ascontiguousarray(fwd.offsets, np.int32)),
            _p(np.ascontiguousarray(fwd.row_token, np.int32)), _p(x), _p(W1e), _p(b1e), _p(W2e), _p(b2e), _p(dy),
            1 if round_stored else 0, _p(out["dW1"]), _p(out["db1"]), _p(out["dW2"]), _p(out["db2"]))
        return out

    # ---- the whole layer
    def forward(self, x, Wg, W1, b1, W2, b2, K: int, capacity_factor: float, aux_alpha: float,
                sel_bias=None, Ws1=None, bs1=None, Ws2=None, bs2=None, want=None,
                skip_ffn: bool = False, z_beta: float = 1e-3, rank_major: bool = False,
                kl_coef: float = 0.02, quant=None) -> OracleResult:
        """Full layer forward. Routing, dispatch and the aux loss always cover
        every token; ``want`` (bool/uint8 [T], optional) limits the FFN and the
        combine to a sample of tokens (the others' outputs are left 0).
        ``quant`` (optional) holds quantised expert weights instead of
        W1/W2/Ws1/Ws2: an object with ``format`` "fp8_e4m3" and W1q, s1, W2q,
        s2 (and Ws1q, ss1, Ws2q, ss2 with a shared expert), or "int4_g128" and
        the packed codes and bf16 group scales in the same fields."""
        x = _np(x, np.uint16)
        T, d = x.shape
        N = _np(Wg, np.uint16).shape[0]
        s = self.gate_logits(x, Wg)
        idx, w, demand, P = self.route(s, K, sel_bias)
        C = self.capacity(T, N, capacity_factor)
        kept, offsets, slot_of, row_token = self.dispatch(idx, N, C, rank_major)
        aux = self.aux_loss(demand, P, T, K, aux_alpha)
        zl = self.z_loss(s, z_beta)
        akl = self.aux_kl(demand, T, K, kl_coef)
        y_perm = z = y = None
        if not skip_ffn:
            want_u8 = None if want is None else np.ascontiguousarray(np.asarray(want).astype(np.uint8))
            if quant is None:
                y_perm = self.expert_ffn(x, offsets, row_token, W1, b1, W2, b2, want_u8)
                if Ws1 is not None:
                    z = self.shared_ffn(x, Ws1, bs1, Ws2, bs2, want_u8)
            elif getattr(quant, "format", "fp8_e4m3") == "int4_g128":
                q = quant
                y_perm = self.expert_ffn_int4(x, offsets, row_token, q.W1q, q.s1, b1, q.W2q, q.s2, b2, want_u8)
                if bs1 is not None:
                    z = self.shared_ffn_int4(x, q.Ws1q, q.ss1, bs1, q.Ws2q, q.ss2, bs2, want_u8)
            else:
                q = quant
                y_perm = self.expert_ffn_fp8(x, offsets, row_token, q.W1q, q.s1, b1, q.W2q, q.s2, b2, want_u8)
                if bs1 is not None:
                    z = self.shared_ffn_fp8(x, q.Ws1q, q.ss1, bs1, q.Ws2q, q.ss2, bs2, want_u8)
            y = self.combine(y_perm, slot_of, w, d, z, want_u8)
        hl, mw = self.health(s, demand, kept, idx, w)
        return OracleResult(s, idx, w, demand, P, C, kept, offsets, slot_of, row_token, y_perm, z, y, aux, zl, akl,
                            hl, mw)


_default: Optional[Oracle] = None
_lock = threading.Lock()


def default() -> Oracle:
    global _default
    with _lock:
        if _default is None:
            _default = Oracle()
    return _default


def forward(*args, **kw) -> OracleResult:
    return default().forward(*args, **kw)


def backward_inputs(inp, fwd: OracleResult, dy, g_aux: float = 1.0, g_z: float = 1.0,
                    round_stored: bool = True, want=None) -> dict:
    """Backward over the fields of the seeded input generator (bf16 experts)."""
    c = inp.cfg
    return default().backward(inp.x, inp.Wg, inp.W1, inp.b1, inp.W2, inp.b2, fwd, dy, c.aux_alpha,
                              getattr(c, "z_beta", 1e-3), g_aux, g_z, inp.Ws1, inp.bs1, inp.Ws2, inp.bs2,
                              round_stored=round_stored, want=want)


def forward_inputs(inp, want=None, skip_ffn: bool = False) -> OracleResult:
    """Forward over an object with the fields of the seeded input generator
    (x, Wg, W1, b1, W2, b2, sel_bias, Ws1, bs1, Ws2, bs2 and cfg)."""
    c = inp.cfg
    return default().forward(inp.x, inp.Wg, inp.W1, inp.b1, inp.W2, inp.b2, c.K, c.capacity_factor,
                             c.aux_alpha, inp.sel_bias, inp.Ws1, inp.bs1, inp.Ws2, inp.bs2,
                             want=want, skip_ffn=skip_ffn, z_beta=getattr(c, "z_beta", 1e-3),
                             rank_major=getattr(c, "rank_major", False), kl_coef=getattr(c, "kl_coef", 0.02),
                             quant=getattr(inp, "quant", None))
