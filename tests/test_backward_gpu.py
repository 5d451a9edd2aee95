"""moe_backward (through the C ABI) against the oracle's fp64 backward.

The oracle mirrors the two bf16 storage points of the GPU backward (dO and da
between the GEMMs) and otherwise computes in fp64; the GPU accumulates in
fp32. Every gradient must agree within rel-L2 1e-2 and max |diff| <= 5e-2 of
the tensor's largest magnitude (fp32 accumulation order and occasional one-ulp
bf16 flips of dO / da; the gate gradients go through fp32 softmax Jacobians).
"""

import numpy as np
import pytest
import torch

import oracle
from top_routing_expert_then_b300 import lib
from top_routing_expert_then_b300.inputs import MoEConfig, make_dy, make_inputs

pytestmark = pytest.mark.gpu

REL_L2 = 1e-2
MAX_FRAC = 5e-2

CASES = [
    MoEConfig("bwd_tiny_drops", 256, 128, 256, 8, 2, 1.25),
    MoEConfig("bwd_ragged", 300, 192, 320, 6, 2, 0.0),
    MoEConfig("bwd_shared_bias_k4", 200, 128, 192, 16, 4, 0.0, has_shared=True, sel_bias=True),
    MoEConfig("bwd_n64_skewed", 512, 128, 128, 64, 2, 1.0, zipf=True),
    MoEConfig("bwd_one_token", 1, 64, 64, 4, 2, 0.0),
]


def _compare(name, got, ref):
    g = got.detach().double().cpu().numpy()
    assert g.shape == ref.shape, (name, g.shape, ref.shape)
    assert np.all(np.isfinite(g)), name
    scale = max(np.abs(ref).max(), 1e-30)
    rel = np.linalg.norm(g - ref) / max(np.linalg.norm(ref), 1e-30)
    worst = np.abs(g - ref).max() / scale
    assert rel <= REL_L2 and worst <= MAX_FRAC, (name, rel, worst)


@pytest.mark.parametrize("cfg", CASES, ids=[c.name for c in CASES])
def test_backward_parity(cfg):
    inp = make_inputs(cfg, 2, device="cuda")
    dy = make_dy(cfg, 2, device="cuda")
    g_aux, g_z = 2.0, 3.0
    layer = lib.MoELayer.from_inputs(inp)
    got = layer.backward(inp.x, dy, inp.sel_bias, g_aux, g_z)
    torch.cuda.synchronize()
    assert lib.device_error() == 0
    cpu = inp.to("cpu")
    fwd = oracle.forward_inputs(cpu)
    ref = oracle.backward_inputs(cpu, fwd, dy.cpu(), g_aux, g_z)
    for name, r in ref.items():
        _compare(name, got[name], r)


def test_backward_deterministic():
    cfg = CASES[2]
    inp = make_inputs(cfg, 5, device="cuda")
    dy = make_dy(cfg, 5, device="cuda")
    layer = lib.MoELayer.from_inputs(inp)
    a = layer.backward(inp.x, dy, inp.sel_bias)
    b = layer.backward(inp.x, dy, inp.sel_bias)
    torch.cuda.synchronize()
    for k in a:
        assert torch.equal(a[k], b[k]), k


@pytest.mark.parametrize("name", ["mixtral_prefill", "skewed"])
def test_backward_full_size_sampled(name):
    """Full-size workload: dx and dw of 12 sampled tokens against the oracle
    (each computable one token at a time); the rest finite and run-to-run
    identical."""
    from top_routing_expert_then_b300.inputs import CONFIGS
    from parity_util import sample_tokens
    cfg = CONFIGS[name]
    inp = make_inputs(cfg, 0, device="cuda")
    dy = make_dy(cfg, 0, device="cuda")
    layer = lib.MoELayer.from_inputs(inp)
    got = layer.backward(inp.x, dy, inp.sel_bias, 1.0, 1.0)
    again = layer.backward(inp.x, dy, inp.sel_bias, 1.0, 1.0)
    torch.cuda.synchronize()
    assert lib.device_error() == 0
    for k in got:
        assert torch.isfinite(got[k]).all(), k
        assert torch.equal(got[k], again[k]), k
    del again
    cpu = inp.to("cpu")
    fwd = oracle.forward_inputs(cpu, skip_ffn=True)
    toks = sample_tokens(cfg.T, 12, 3)
    want = np.zeros(cfg.T, dtype=bool)
    want[toks] = True
    ref = oracle.backward_inputs(cpu, fwd, dy.cpu(), 1.0, 1.0, want=want)
    _compare("dx", got["dx"][torch.from_numpy(toks).cuda()], ref["dx"][toks])
    _compare("dw", got["dw"][torch.from_numpy(toks).cuda()], ref["dw"][toks])
