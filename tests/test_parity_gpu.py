"""CUDA path (through the C ABI) against the CPU oracle, element by element.

Indices, drops, offsets and the dispatch table must match bit for bit (the
inputs lie on the 1/64 grid, so every gate logit is exact in fp32 and fp64);
bf16 values must agree within rel-L2 5e-3 and |d| <= 3e-2 (1 + |ref|); the
aux loss within 1e-5 relative.
"""

import numpy as np
import pytest
import torch

import oracle
from parity_util import assert_bf16_tol, bits_np, check_layer, gpu_inputs
from top_routing_expert_then_b300 import lib
from top_routing_expert_then_b300.inputs import CONFIGS, MoEConfig

pytestmark = pytest.mark.gpu

# Small shapes the oracle finishes in seconds. They span several GEMM tiles,
# ragged row / column / chunk tails, drops, the shared expert, the selection
# bias and the extreme N / K the ABI accepts.
SMALL = [
    CONFIGS["tiny"],
    MoEConfig("ragged", 300, 192, 320, 6, 2, 0.0),
    MoEConfig("drops_k4", 1000, 256, 512, 16, 4, 1.0),
    MoEConfig("shared_bias_k8", 513, 128, 384, 32, 8, 0.0, has_shared=True, sel_bias=True),
    MoEConfig("wide_n256", 200, 64, 128, 256, 8, 1.5),
    MoEConfig("dense_n1k1", 130, 64, 64, 1, 1, 0.0),
    MoEConfig("one_token", 1, 128, 128, 8, 2, 0.0),
    MoEConfig("n1024_k8", 64, 64, 64, 1024, 8, 0.0),
    MoEConfig("n20_gate_tiled", 257, 64, 192, 20, 3, 2.0),
    MoEConfig("soft_router_k_eq_n", 100, 128, 128, 8, 8, 0.0),
    MoEConfig("tight_capacity", 500, 128, 256, 8, 2, 0.05),
    MoEConfig("multi_tile", 2048, 512, 1024, 8, 2, 0.0),
    MoEConfig("skewed_small", 1024, 256, 192, 64, 2, 1.0, zipf=True),
    MoEConfig("rank_major_drops", 1000, 256, 512, 16, 4, 1.0, rank_major=True),
    MoEConfig("rank_major_skewed", 2048, 256, 192, 64, 2, 1.0, zipf=True, rank_major=True),
    MoEConfig("rank_major_ties", 300, 128, 128, 8, 3, 0.5, rank_major=True),
    # one dispatch chunk (the single-block dispatch kernel), rank order with drops
    MoEConfig("rank_major_small", 40, 128, 128, 8, 3, 0.5, rank_major=True),
    # fused tensor-core router: N padded to 16 (37 -> 48, 200 -> 208), several
    # lanes per warp (N = 128, 200), more tiles than one wave (T = 20000: one
    # split, two blocks per SM)
    MoEConfig("n37_pad", 700, 192, 128, 37, 3, 1.1),
    MoEConfig("n128_k6_bias", 600, 256, 128, 128, 6, 0.0, sel_bias=True),
    MoEConfig("n200_bias", 400, 320, 128, 200, 8, 1.0, sel_bias=True),
    MoEConfig("multi_wave", 20000, 128, 128, 8, 2, 1.0),
    # general path (N > 256): CUDA-core tiled gate when N % 32 != 0
    MoEConfig("n300_gate_tiled", 257, 64, 64, 300, 3, 2.0),
    # a shared expert whose dense GEMMs span several raster groups of 128-row
    # tiles (17 and 32 m-tiles), long reductions, a ragged last shared tile
    MoEConfig("shared_groups", 2100, 1024, 512, 16, 4, 0.0, has_shared=True, sel_bias=True),
    MoEConfig("shared_groups_n64", 4096, 512, 256, 64, 2, 1.0, has_shared=True),
    # >= 1024 rows per expert and a long second reduction: the second expert
    # GEMM runs on the SM-pair kernel (256-row tiles, ragged last tiles)
    MoEConfig("pair_gemm2", 1100, 256, 8192, 2, 2, 0.0),
    # decode-sized bf16 batches (a few rows per expert, x rows gathered): a
    # shared expert; odd k-block counts and a ragged n tile
    MoEConfig("bf16_decode_split", 24, 256, 384, 8, 2, 0.0, has_shared=True),
    MoEConfig("bf16_decode_odd", 40, 192, 320, 6, 2, 0.0, sel_bias=True),
    # FP8 E4M3 expert weights (per-output-channel scales): several n-tiles, a
    # ragged expert, the shared expert, drops
    MoEConfig("fp8_experts", 700, 256, 640, 8, 2, 1.25, weights="fp8_e4m3"),
    MoEConfig("fp8_shared_bias", 300, 192, 320, 16, 4, 0.0, has_shared=True, sel_bias=True, weights="fp8_e4m3"),
    # a few rows per expert (decode: MMA N = 16), three channel tiles
    MoEConfig("fp8_decode_small", 24, 256, 384, 8, 2, 0.0, weights="fp8_e4m3"),
    # several 128-row tiles per expert with a ragged last one, a half channel
    # tile (192 = 128 + 64), an odd k-block count, the dense shared expert
    MoEConfig("fp8_many_rows", 700, 128, 192, 2, 1, 0.0, has_shared=True, weights="fp8_e4m3"),
    # decode-sized batch: split-K over the k-pairs with an odd k-block count
    # (192 = 3 x 64, 320 = 5 x 64), the shared expert split too
    MoEConfig("fp8_split_k", 40, 192, 320, 4, 2, 0.0, has_shared=True, sel_bias=True, weights="fp8_e4m3"),
    # a decode-sized batch with a Zipf-skewed gate: a few experts hold most rows
    MoEConfig("fp8_decode_zipf", 120, 256, 384, 8, 2, 0.0, zipf=True, weights="fp8_e4m3"),
    # INT4 group-wise expert weights (4-bit codes, a bf16 scale per 128 columns):
    # several channel tiles and groups, drops, a ragged expert
    MoEConfig("int4_experts", 700, 256, 640, 8, 2, 1.25, weights="int4_g128"),
    # the shared expert and the selection bias, K = 4
    MoEConfig("int4_shared_bias", 300, 256, 384, 16, 4, 0.0, has_shared=True, sel_bias=True, weights="int4_g128"),
    # decode-sized: split-K over the k-pairs with odd k-pair counts (384 = 3 x 128,
    # 640 = 5 x 128), the shared expert split too
    MoEConfig("int4_split_k", 40, 384, 640, 4, 2, 0.0, has_shared=True, weights="int4_g128"),
    # several 64-row tiles per expert with a ragged last one, one group per row
    MoEConfig("int4_many_rows", 700, 128, 256, 2, 1, 0.0, weights="int4_g128"),
]


@pytest.mark.parametrize("cfg", SMALL, ids=[c.name for c in SMALL])
def test_small_layer_parity(cfg):
    check_layer(cfg, seed=1)


def test_all_ties_heavy_drops():
    """Every logit equal: each token selects experts 0..K-1 (ties go to the
    lower id), so experts 0..K-1 overflow capacity and the rest stay empty."""
    cfg = MoEConfig("ties", 300, 128, 128, 8, 2, 1.25)
    inp = gpu_inputs(cfg, 3)
    inp.Wg.zero_()
    layer = lib.MoELayer.from_inputs(inp)
    ro = layer.route_outputs()
    y = layer.forward(inp.x, route_out=ro)
    torch.cuda.synchronize()
    ref = oracle.forward_inputs(inp.to("cpu"))
    assert np.array_equal(ro.topk_idx.cpu().numpy(), np.tile([0, 1], (300, 1)))
    assert np.array_equal(ro.slot_of.cpu().numpy(), ref.slot_of)
    assert ref.kept.tolist() == [47, 47, 0, 0, 0, 0, 0, 0]
    assert np.allclose(ro.topk_w.cpu().numpy(), 0.5)
    assert_bf16_tol(bits_np(y), ref.y, "ties y")
    assert abs(float(ro.aux.cpu()[0]) - 0.01) < 1e-7   # uniform P -> alpha
    assert lib.device_error() == 0


def test_deterministic_reruns():
    """Two runs of the layer give identical bytes (no order-dependent atomics)."""
    cfg = MoEConfig("rerun", 700, 256, 384, 16, 4, 1.25, has_shared=True, sel_bias=True)
    inp = gpu_inputs(cfg, 5)
    layer = lib.MoELayer.from_inputs(inp)
    outs = []
    for _ in range(2):
        ro = layer.route_outputs()
        y = layer.forward(inp.x, inp.sel_bias, route_out=ro)
        torch.cuda.synchronize()
        outs.append([y.clone()] + [getattr(ro, n).clone() for n in ("topk_idx", "topk_w", "prob_sum", "slot_of",
                                                                     "aux")])
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_hostio_matches_device_path():
    cfg = MoEConfig("hostio", 384, 128, 256, 8, 2, 1.25)
    inp = gpu_inputs(cfg, 6)
    layer = lib.MoELayer.from_inputs(inp)
    y_dev = layer.forward(inp.x)
    x_host = inp.x.cpu().pin_memory()
    y_host = torch.empty_like(x_host).pin_memory()
    xd = torch.empty_like(inp.x)
    yd = torch.empty_like(inp.x)
    layer.forward_hostio(x_host, y_host, xd, yd)
    torch.cuda.synchronize()
    assert torch.equal(y_host, y_dev.cpu())


def test_out_of_range_expert_ids_are_flagged_not_trapped():
    """Corrupted top-k ids (written from the host) are skipped by the dispatch
    kernels and reported through the device error word."""
    cfg = MoEConfig("badids", 64, 64, 64, 8, 2, 0.0)
    inp = gpu_inputs(cfg, 7)
    shape = lib.shape_of(cfg)
    lib.device_error(clear=True)
    idx = torch.randint(0, 8, (64, 2), dtype=torch.int32, device="cuda")
    idx[:, 1] = (idx[:, 0] + 1) % 8
    idx[5, 0] = 99
    idx[9, 1] = -3
    kept, offsets, slot_of, row_token, x_perm = lib.dispatch(shape, idx, inp.x)
    torch.cuda.synchronize()
    assert lib.device_error() & lib.DEVERR_EXPERT_ID
    so = slot_of.cpu().numpy()
    assert so[5, 0] == -1 and so[9, 1] == -1
    assert int(offsets[-1]) == 64 * 2 - 2
    assert lib.device_error() == 0   # cleared by the previous read


# ---------------------------------------------------------------- full-size workloads
# Routing and dispatch compared on every token. FFN outputs: every token where
# the oracle finishes in a few minutes (the decode and skewed workloads, and
# -- slow -- the Mixtral prefill and DeepSeek-V3-shaped layers); on the
# capacity-limited prefill, the tokens of covering_tokens (every expert's
# first and last kept row and both sides of each 128/256-row tile edge).
FULL = {
    "mixtral_prefill": None, "mixtral_prefill_cf125": "cover", "mixtral_decode16": None,
    "mixtral_decode64": None, "skewed": None, "dsv3": None, "mixtral_decode16_fp8": None,
    "mixtral_decode64_fp8": None, "mixtral_decode16_int4": None, "mixtral_decode64_int4": None,
}
SLOW = {"mixtral_prefill", "dsv3"}


@pytest.mark.parametrize("name", [pytest.param(n, marks=pytest.mark.slow) if n in SLOW else n for n in FULL])
def test_full_size_parity(name):
    cfg = CONFIGS[name]
    ref = check_layer(cfg, seed=0, sample=FULL[name], stages=True, cache=name in SLOW)
    if name == "skewed":
        # the Zipf-skewed gate makes the first experts hot; capacity 128 drops tokens
        mean = cfg.T * cfg.K / cfg.N
        assert ref.demand[0] > 4 * mean and ref.demand[1] > 2 * mean
        assert (ref.slot_of < 0).sum() >= 8192


# ---------------------------------------------------------------- gate exactness on the tensor cores
def adversarial_gate_inputs(cfg: MoEConfig, seed: int):
    """x and W_g on the 1/64 grid whose gate logits all lie near +-1000..1792
    and differ between the experts of a token only by a few multiples of
    2^-12, so every TopK choice and capacity drop hangs on the lowest bits of
    a large sum (ties included).

    The d_model coordinates split into "big" ones, where every expert's gate
    row holds the same +-8/64 and the token holds +-2 (each product +-1/4; the
    token's flips set its common part B_t), and 48 "small" ones, 16 in each of
    the first, a middle and the last 64-wide block, interleaved with big ones
    (every fourth coordinate), where both the gate rows and the tokens hold
    -1/64, 0 or +1/64 (products of 2^-12). So s[t, e] = B_t + m_te 2^-12 with
    |m_te| <= 48: exact in fp32 only if every partial sum keeps all 23 bits
    below the leading one. Each token switches on the small coordinates of
    one, two or all three blocks, so the small products meet accumulators of
    every size."""
    g = torch.Generator().manual_seed(seed)
    T, d, N = cfg.T, cfg.d_model, cfg.N
    small = torch.cat([torch.arange(0, 64, 4), torch.arange(d // 2, d // 2 + 64, 4),
                       torch.arange(d - 64 + 1, d, 4)])
    big = torch.ones(d, dtype=torch.bool)
    big[small] = False
    tau = torch.randint(0, 2, (d,), generator=g) * 2 - 1
    wg = torch.zeros((N, d), dtype=torch.int32)
    wg[:, big] = (8 * tau[big]).to(torch.int32)
    wg[:, small] = torch.randint(-1, 2, (N, small.numel()), generator=g, dtype=torch.int32)
    nbig = int(big.sum())
    xi = torch.zeros((T, d), dtype=torch.int32)
    for t in range(T):
        flips = int(torch.randint(0, (nbig - 4000) // 2 + 1, (1,), generator=g))  # B_t in [1000, 1780]
        sign = 1 if int(torch.randint(0, 2, (1,), generator=g)) else -1
        v = 128 * tau[big].to(torch.int32) * sign
        v[torch.randperm(nbig, generator=g)[:flips]] *= -1
        xi[t, big] = v
        on = int(torch.randint(1, 8, (1,), generator=g))  # which of the three small blocks are on
        vals = torch.randint(-1, 2, (small.numel(),), generator=g, dtype=torch.int32)
        mask = torch.tensor([(on >> (i // 16)) & 1 for i in range(small.numel())], dtype=torch.int32)
        xi[t, small] = vals * mask
    x = (xi.to(torch.float32) / 64).to(torch.bfloat16)
    Wg = (wg.to(torch.float32) / 64).to(torch.bfloat16)
    return x, Wg


ADVERSARIAL = [
    # fused tensor-core router: d_model split over an 8-CTA cluster
    MoEConfig("adv_gate_n8", 512, 7168, 64, 8, 2, 1.0),
    MoEConfig("adv_gate_n256_k8", 256, 7168, 64, 256, 8, 1.0),
    # N > 256: the tensor-core gate GEMM with K-split partial planes
    MoEConfig("adv_gate_n320_k4", 512, 7168, 64, 320, 4, 1.0),
    # N > 256, N % 32 != 0: the CUDA-core tiled gate
    MoEConfig("adv_gate_n300_k3", 256, 7168, 64, 300, 3, 1.0),
]


@pytest.mark.parametrize("cfg", ADVERSARIAL, ids=[c.name for c in ADVERSARIAL])
def test_gate_exact_near_ties(cfg):
    """TopK, drops and max|logit| bit-exact on logits near 1000-1792 that
    differ by single multiples of 2^-12 (see adversarial_gate_inputs)."""
    inp = gpu_inputs(cfg, 11)
    x, Wg = adversarial_gate_inputs(cfg, 11)
    inp.x.copy_(x)
    inp.Wg.copy_(Wg)
    cpu = inp.to("cpu")
    ref = oracle.forward_inputs(cpu)
    s = ref.logits
    assert np.abs(s).min() >= 1000 - 1 and np.abs(s).max() <= 1792
    top = np.sort(s, axis=1)[:, ::-1]
    gaps = np.round((top[:, :-1] - top[:, 1:]) * 4096).astype(np.int64)
    assert (gaps == 1).sum() >= cfg.T // 4 and (gaps == 0).sum() >= cfg.T // 4, "want many 1-step gaps and ties"
    check_layer_on(cfg, inp, ref)


def check_layer_on(cfg, inp, ref):
    """check_layer's whole-layer comparison for explicitly given inputs."""
    layer = lib.MoELayer.from_inputs(inp)
    ro = layer.route_outputs()
    y = layer.forward(inp.x, inp.sel_bias, route_out=ro)
    torch.cuda.synchronize()
    assert lib.device_error() == 0
    assert np.array_equal(ro.topk_idx.cpu().numpy(), ref.topk_idx), "topk_idx"
    assert np.array_equal(ro.demand.cpu().numpy(), ref.demand), "demand"
    assert np.array_equal(ro.kept.cpu().numpy(), ref.kept), "kept"
    assert np.array_equal(ro.slot_of.cpu().numpy(), ref.slot_of), "slot_of"
    assert float(ro.health.cpu()[3]) == np.float32(ref.health[3]), "max|logit|"
    assert np.allclose(ro.topk_w.cpu().numpy(), ref.topk_w, rtol=0, atol=2e-6), "topk_w"
    assert_bf16_tol(bits_np(y), ref.y, "forward y")
    idx, w, demand, psum = lib.route(lib.shape_of(cfg), inp.x, inp.Wg, inp.sel_bias)
    torch.cuda.synchronize()
    assert np.array_equal(idx.cpu().numpy(), ref.topk_idx), "moe_route topk_idx"


def test_hostio_batches_match_forward():
    """moe_forward_hostio_batches (overlapped copies, double-buffered device
    buffers) gives, for every batch, the bytes moe_forward gives."""
    cfg = MoEConfig("hostio_batches", 300, 128, 256, 8, 2, 1.25, has_shared=True)
    inp = gpu_inputs(cfg, 4)
    layer = lib.MoELayer.from_inputs(inp)
    nb = 5
    xs = torch.stack([(torch.randint(-128, 129, (cfg.T, cfg.d_model), device="cuda").float() / 64).to(torch.bfloat16)
                      for _ in range(nb)])
    x_host = xs.cpu().pin_memory()
    y_host = torch.empty_like(x_host).pin_memory()
    xd = torch.empty((2, cfg.T, cfg.d_model), dtype=torch.bfloat16, device="cuda")
    yd = torch.empty_like(xd)
    layer.forward_hostio_batches(x_host, y_host, nb, xd, yd)
    torch.cuda.synchronize()
    for i in range(nb):
        ref = layer.forward(xs[i])
        torch.cuda.synchronize()
        assert torch.equal(y_host[i], ref.cpu()), i
    assert lib.device_error() == 0
