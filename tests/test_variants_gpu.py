"""The opt-in kernel variants against the oracle. Each is selected by an
environment variable that the library reads once per process, so each runs
in a child process of its own:

  MOE_FP8_GEMM=token_major   FP8 expert GEMM with the weights widened in
                             shared memory (token rows as the MMA's M)
  MOE_GEMM_VARIANT=pair      bf16 expert GEMM on SM pairs (cta_group::2, M=256)
  MOE_ROUTE_VARIANT=legacy   the general router (gate GEMM, TopK, finalize
                             kernels) for every N instead of the fused kernel
"""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

CHILD = r"""
import sys
sys.path[:0] = [{here!r}, {root!r}]
from parity_util import check_layer
from top_routing_expert_then_b300.inputs import MoEConfig
for cfg in [{configs}]:
    check_layer(cfg, seed=1)
print("ok")
"""

VARIANTS = {
    "fp8_token_major": ("MOE_FP8_GEMM", "token_major", [
        'MoEConfig("fp8_experts", 700, 256, 640, 8, 2, 1.25, weights="fp8_e4m3")',
        'MoEConfig("fp8_decode_small", 24, 256, 384, 8, 2, 0.0, has_shared=True, weights="fp8_e4m3")']),
    "gemm_pair": ("MOE_GEMM_VARIANT", "pair", [
        'MoEConfig("ragged", 300, 192, 320, 6, 2, 0.0)',
        'MoEConfig("multi_tile_shared", 1500, 256, 512, 4, 2, 0.0, has_shared=True, sel_bias=True)']),
    "route_legacy": ("MOE_ROUTE_VARIANT", "legacy", [
        'MoEConfig("n37_pad", 700, 192, 128, 37, 3, 1.1)',
        'MoEConfig("n128_k6_bias", 600, 256, 128, 128, 6, 0.0, sel_bias=True)']),
}


@pytest.mark.parametrize("name", sorted(VARIANTS))
def test_variant_parity(name):
    var, value, configs = VARIANTS[name]
    env = dict(os.environ, **{var: value})
    code = CHILD.format(here=HERE, root=ROOT, configs=", ".join(configs))
    r = subprocess.run([sys.executable, "-c", code], env=env, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:] + r.stderr[-4000:]
