"""Host-side checks of libmoe.so that need no GPU: the library loads, exports
every entry point include/moe.h declares, and rejects bad arguments with the
documented status before touching CUDA (fake, never-dereferenced addresses)."""

import ctypes
import subprocess

import pytest

from top_routing_expert_then_b300 import lib
from top_routing_expert_then_b300.build import LIBRARY, build

FAKE = 0x10000  # 16-byte aligned, never dereferenced by the host checks


@pytest.fixture(scope="module")
def L():
    build()
    return lib.load()


def test_exports_every_declared_symbol(L):
    names = lib.declared_functions()
    assert len(names) >= 12
    out = subprocess.check_output(["nm", "-D", "--defined-only", LIBRARY], text=True)
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    for n in names:
        assert n in exported, n
        assert getattr(L, n) is not None
    # nothing but the declared API is exported
    assert {e for e in exported if e.startswith("moe_")} == set(names)


def test_capacity_closed_form(L):
    # lmnt.cn/news/351908 sec. 3.3: ceil(T / N * capacity_factor); dropless = T
    assert lib.capacity(lib.make_shape(256, 128, 256, 8, 2, 1.25)) == 40
    assert lib.capacity(lib.make_shape(4096, 4096, 14336, 8, 2, 1.25)) == 640
    assert lib.capacity(lib.make_shape(8192, 2048, 1408, 64, 2, 1.0)) == 128
    assert lib.capacity(lib.make_shape(4096, 7168, 2048, 256, 8, 0.0)) == 4096
    assert lib.capacity(lib.make_shape(10, 64, 64, 3, 1, 1.0)) == 4
    assert lib.capacity(lib.make_shape(5, 64, 64, 8, 1, 100.0)) == 5
    assert lib.capacity(lib.make_shape(0, 64, 64, 8, 1, 1.0)) == -1


def test_workspace_sizes(L):
    s = lib.make_shape(4096, 4096, 14336, 8, 2, 0.0)
    fw = lib.workspace_bytes(s, lib.MOE_WS_FORWARD)
    parts = [lib.workspace_bytes(s, k) for k in (lib.MOE_WS_ROUTE, lib.MOE_WS_DISPATCH, lib.MOE_WS_FFN)]
    assert all(p > 0 for p in parts) and fw >= sum(parts)
    # the hidden activation alone: T*K rows of d_ff bf16
    assert lib.workspace_bytes(s, lib.MOE_WS_FFN) >= 4096 * 2 * 14336 * 2
    assert fw % 256 == 0
    assert lib.workspace_bytes(lib.make_shape(16, 100, 64, 8, 2), 0) == 0   # d_model % 64
    assert lib.workspace_bytes(s, 99) == 0


def _route(L, shape, x=FAKE, wg=FAKE, ws=FAKE, ws_bytes=1 << 40):
    return L.moe_route(ctypes.byref(shape), x, wg, None, FAKE, FAKE, FAKE, FAKE, ws, ws_bytes, None)


def test_invalid_arguments(L):
    ok = lib.make_shape(256, 128, 256, 8, 2, 1.25)
    assert _route(L, lib.make_shape(256, 128, 256, 8, 9)) == lib.MOE_ERR_INVALID_ARG       # K > N
    assert _route(L, lib.make_shape(0, 128, 256, 8, 2)) == lib.MOE_ERR_INVALID_ARG         # T = 0
    assert _route(L, lib.make_shape(256, 128, 256, 8, 0)) == lib.MOE_ERR_INVALID_ARG       # K = 0
    assert _route(L, lib.make_shape(256, 96, 256, 8, 2)) == lib.MOE_ERR_UNSUPPORTED        # d % 64
    assert _route(L, lib.make_shape(256, 128, 200, 8, 2)) == lib.MOE_ERR_UNSUPPORTED       # f % 64
    assert _route(L, lib.make_shape(256, 128, 256, 16, 9)) == lib.MOE_ERR_UNSUPPORTED      # K > 8
    assert _route(L, lib.make_shape(256, 128, 256, 2048, 2)) == lib.MOE_ERR_UNSUPPORTED    # N > 1024
    s = lib.make_shape(256, 128, 256, 8, 2, 1.25)
    s.has_shared = 3
    assert _route(L, s) == lib.MOE_ERR_INVALID_ARG
    s = lib.make_shape(256, 128, 256, 8, 2, 1.25)
    s.drop_policy = 2                                                                      # unknown priority
    assert _route(L, s) == lib.MOE_ERR_INVALID_ARG
    s = lib.make_shape(256, 128, 256, 8, 2, 1.25, kl_coef=float("nan"))
    assert _route(L, s) == lib.MOE_ERR_INVALID_ARG
    assert _route(L, ok, x=None) == lib.MOE_ERR_INVALID_ARG
    assert _route(L, ok, x=FAKE + 2) == lib.MOE_ERR_INVALID_ARG                            # misaligned
    assert _route(L, ok, ws=None) == lib.MOE_ERR_WORKSPACE
    assert _route(L, ok, ws=FAKE + 16) == lib.MOE_ERR_WORKSPACE                            # not 256-aligned
    assert _route(L, ok, ws_bytes=16) == lib.MOE_ERR_WORKSPACE
    assert L.moe_route(None, FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 40, None) == lib.MOE_ERR_INVALID_ARG
    # other entry points
    assert L.moe_dispatch(ctypes.byref(ok), FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE, 1 << 40, None) \
        == lib.MOE_ERR_INVALID_ARG
    assert L.moe_dispatch(ctypes.byref(ok), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 8, None) \
        == lib.MOE_ERR_WORKSPACE
    w = lib.MoeWeights(FAKE, FAKE, FAKE, None, FAKE, None, None, None, None)                 # W2 missing
    assert L.moe_expert_ffn(ctypes.byref(ok), FAKE, FAKE, ctypes.byref(w), FAKE, FAKE, None, FAKE, 1 << 40,
                            None) == lib.MOE_ERR_INVALID_ARG
    sh = lib.make_shape(256, 128, 256, 8, 2, 0.0, has_shared=True)
    w = lib.MoeWeights(FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None, None)                 # shared missing
    assert L.moe_expert_ffn(ctypes.byref(sh), FAKE, FAKE, ctypes.byref(w), FAKE, FAKE, FAKE, FAKE, 1 << 40,
                            None) == lib.MOE_ERR_INVALID_ARG
    # FP8 expert weights: the bf16 matrices may be absent, the codes and scales may not
    w = lib.MoeWeights(FAKE, None, FAKE, None, FAKE, None, None, None, None, 7)              # unknown format
    assert L.moe_expert_ffn(ctypes.byref(ok), FAKE, FAKE, ctypes.byref(w), FAKE, FAKE, None, FAKE, 1 << 40,
                            None) == lib.MOE_ERR_INVALID_ARG
    w = lib.MoeWeights(FAKE, None, FAKE, None, FAKE, None, None, None, None, lib.MOE_WEIGHTS_FP8_E4M3,
                       FAKE, None, FAKE, FAKE)                                                 # s1 missing
    assert L.moe_expert_ffn(ctypes.byref(ok), FAKE, FAKE, ctypes.byref(w), FAKE, FAKE, None, FAKE, 1 << 40,
                            None) == lib.MOE_ERR_INVALID_ARG
    w = lib.MoeWeights(FAKE, None, FAKE, None, FAKE, None, FAKE, None, FAKE, lib.MOE_WEIGHTS_FP8_E4M3,
                       FAKE, FAKE, FAKE, FAKE)                                                 # shared codes missing
    assert L.moe_expert_ffn(ctypes.byref(sh), FAKE, FAKE, ctypes.byref(w), FAKE, FAKE, FAKE, FAKE, 1 << 40,
                            None) == lib.MOE_ERR_INVALID_ARG
    # INT4 group-wise expert weights: codes and bf16 group scales, reductions in whole groups of 128
    w = lib.MoeWeights(FAKE, None, FAKE, None, FAKE, None, None, None, None, lib.MOE_WEIGHTS_INT4_G128,
                       FAKE, None, FAKE, None, None, None, None, None, FAKE, None)             # g2 missing
    assert L.moe_expert_ffn(ctypes.byref(ok), FAKE, FAKE, ctypes.byref(w), FAKE, FAKE, None, FAKE, 1 << 40,
                            None) == lib.MOE_ERR_INVALID_ARG
    w = lib.MoeWeights(FAKE, None, FAKE, None, FAKE, None, None, None, None, lib.MOE_WEIGHTS_INT4_G128,
                       FAKE, None, FAKE, None, None, None, None, None, FAKE, FAKE)
    d192 = lib.make_shape(256, 192, 256, 8, 2, 1.25)                                       # 192 = 1.5 groups
    assert L.moe_expert_ffn(ctypes.byref(d192), FAKE, FAKE, ctypes.byref(w), FAKE, FAKE, None, FAKE, 1 << 40,
                            None) == lib.MOE_ERR_UNSUPPORTED
    assert L.moe_forward(ctypes.byref(d192), ctypes.byref(w), FAKE, None, FAKE, None, FAKE, 1 << 40, None) \
        == lib.MOE_ERR_UNSUPPORTED
    assert L.moe_combine(ctypes.byref(ok), FAKE, FAKE, None, None, FAKE, None) == lib.MOE_ERR_INVALID_ARG
    assert L.moe_combine(ctypes.byref(ok), FAKE, FAKE, FAKE, FAKE + 8, FAKE, None) == lib.MOE_ERR_INVALID_ARG
    assert L.moe_aux_loss(ctypes.byref(ok), FAKE, None, FAKE, None) == lib.MOE_ERR_INVALID_ARG
    w = lib.MoeWeights(None, FAKE, FAKE, FAKE, FAKE, None, None, None, None)                 # Wg missing
    assert L.moe_forward(ctypes.byref(ok), ctypes.byref(w), FAKE, None, FAKE, None, FAKE, 1 << 40, None) \
        == lib.MOE_ERR_INVALID_ARG
    w = lib.MoeWeights(FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None, None)
    assert L.moe_forward(ctypes.byref(ok), ctypes.byref(w), FAKE, None, FAKE, None, FAKE, 64, None) \
        == lib.MOE_ERR_WORKSPACE
    assert L.moe_forward_hostio(ctypes.byref(ok), ctypes.byref(w), None, FAKE, None, FAKE, FAKE, None, FAKE,
                                1 << 40, None) == lib.MOE_ERR_INVALID_ARG
    assert L.moe_get_device_error(0, None) == lib.MOE_ERR_INVALID_ARG


def test_status_strings(L):
    for code in range(6):
        assert lib.status_string(code)
    assert "unknown" in lib.status_string(42)


def test_product_path_has_no_fallback():
    """The binding and the package never import the oracle or call torch math
    on the data path: the layer exists only as libmoe.so."""
    import inspect
    import top_routing_expert_then_b300.lib as m
    src = inspect.getsource(m)
    assert "oracle" not in src.replace("no CPU", "")
    for forbidden in ("torch.matmul", "F.linear", "torch.topk", "softmax(", "gelu("):
        assert forbidden not in src


def test_int4_pack_layout():
    """The input generator's INT4 packing: codes 0..7 of one run of eight
    columns form the little-endian word 0x75316420 (column 2j in bits 4j ..,
    column 2j + 1 in bits 16 + 4j ..), the same bytes the oracle's pins pack
    bit by bit, and a second run continues at byte 4."""
    import numpy as np
    import torch
    from top_routing_expert_then_b300.inputs import int4_pack
    from oracle_pins import _int4_pack
    codes = torch.arange(16, dtype=torch.int32).remainder(16).reshape(1, 16)
    got = int4_pack(codes).numpy()
    assert got.tolist() == [[0x20, 0x64, 0x31, 0x75, 0xA8, 0xEC, 0xB9, 0xFD]]
    rng = np.random.default_rng(5)
    c = rng.integers(0, 16, size=(3, 5, 256)).astype(np.uint8)
    assert np.array_equal(int4_pack(torch.from_numpy(c)).numpy(), _int4_pack(c))
