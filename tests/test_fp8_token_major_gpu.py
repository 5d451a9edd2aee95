"""The token-major FP8 expert GEMM (weights widened in shared memory, selected
with MOE_FP8_GEMM=token_major, read once per process) against the oracle, in
a child process so the selection does not leak into the other tests."""

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
for cfg in [MoEConfig("fp8_experts", 700, 256, 640, 8, 2, 1.25, weights="fp8_e4m3"),
            MoEConfig("fp8_decode_small", 24, 256, 384, 8, 2, 0.0, has_shared=True, weights="fp8_e4m3")]:
    check_layer(cfg, seed=1)
print("ok")
"""


def test_token_major_fp8_gemm_parity():
    env = dict(os.environ, MOE_FP8_GEMM="token_major")
    r = subprocess.run([sys.executable, "-c", CHILD.format(here=HERE, root=ROOT)], env=env, cwd=ROOT,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:] + r.stderr[-4000:]
