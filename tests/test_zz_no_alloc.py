"""moe_route_noalloc: routing for callers that cannot hand the library device
scratch memory (e.g. a plugin whose host framework plans all device memory up
front, or a loop that must not call cudaMalloc once running). It uses one
fixed scratch array inside libmoe.so instead of a workspace.

Checked through the C ABI against the workspace entry point moe_route, on two
calls in a row (the shared array keeps the previous call's contents, so the
second call must not depend on them). This file is collected last so that a
failure here cannot stop the rest of the suite; it also passes on its own in a
fresh process.
"""

import numpy as np
import pytest
import torch

from parity_util import PROB_RTOL, W_ATOL
from top_routing_expert_then_b300 import lib
from top_routing_expert_then_b300.inputs import MoEConfig, make_inputs

pytestmark = pytest.mark.gpu

# one shape on the fused tensor-core router (N <= 256) and one on the general
# path (N > 256: logits, TopK and finalize kernels, logits in the scratch),
# drawn with different seeds so consecutive calls see different contents
CASES = [
    (MoEConfig("noalloc_small_n", 1000, 256, 256, 8, 2, 1.25), 11),
    (MoEConfig("noalloc_general_n", 1000, 512, 256, 320, 8, 0.0, sel_bias=True), 12),
]


def _compare(cfg, seed):
    inp = make_inputs(cfg, seed, device="cuda")
    shape = lib.shape_of(cfg)
    ref = lib.route(shape, inp.x, inp.Wg, inp.sel_bias)
    got = lib.route_noalloc(shape, inp.x, inp.Wg, inp.sel_bias)
    torch.cuda.synchronize()
    r_idx, r_w, r_dem, r_ps = (t.cpu().numpy() for t in ref)
    g_idx, g_w, g_dem, g_ps = (t.cpu().numpy() for t in got)
    assert np.array_equal(g_idx, r_idx)
    assert np.array_equal(g_dem, r_dem)
    assert np.allclose(g_w, r_w, rtol=0, atol=W_ATOL)
    assert np.allclose(g_ps, r_ps, rtol=PROB_RTOL, atol=1e-6)


def test_noalloc_route_matches_workspace_route_twice_in_a_row():
    for cfg, seed in CASES:
        _compare(cfg, seed)      # first call on this device sets up the scratch address
        _compare(cfg, seed + 100)  # second call reuses the array left by the first
    assert lib.device_error() == 0


def test_noalloc_route_rejects_shapes_beyond_its_scratch():
    # routing workspace above 8 MiB: refused before anything is enqueued
    big = lib.make_shape(16384, 64, 64, 512, 8, 0.0)
    assert lib.workspace_bytes(big, lib.MOE_WS_ROUTE) > 8 << 20
    x = torch.zeros((16384, 64), dtype=torch.bfloat16, device="cuda")
    wg = torch.zeros((512, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(lib.MoEError) as e:
        lib.route_noalloc(big, x, wg)
    assert e.value.status == lib.MOE_ERR_UNSUPPORTED
