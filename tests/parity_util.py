"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
and compare it with the CPU oracle on the same seeded inputs."""

from __future__ import annotations

import numpy as np
import torch

import oracle
from oracle import bf16_to_f64
from top_routing_expert_then_b300 import lib
from top_routing_expert_then_b300.inputs import MoEConfig, make_inputs

# Tolerances for bf16 outputs with fp32 accumulation (vs the fp64 oracle):
# relative L2 over the tensor and a per-element bound.
REL_L2 = 5e-3
ELEM_ABS = 3e-2
AUX_RTOL = 1e-5
W_ATOL = 2e-6       # routing weights (fp32 softmax vs fp64 softmax rounded to fp32)
PROB_RTOL = 2e-5    # per-expert sums of full-softmax probabilities


def bits_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def assert_bf16_tol(got_bits, ref_bits, what=""):
    g = bf16_to_f64(got_bits)
    r = bf16_to_f64(ref_bits)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    if g.size == 0:
        return
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    err = np.abs(g - r)
    bound = ELEM_ABS * (1.0 + np.abs(r))
    worst = np.argmax(err - bound)
    assert np.all(err <= bound), (f"{what}: element {np.unravel_index(worst, g.shape)} got {g.flat[worst]} "
                                  f"ref {r.flat[worst]}")
    rel = np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30)
    assert rel <= REL_L2, f"{what}: rel-L2 {rel:.3e}"


def sample_tokens(T: int, n: int, seed: int = 0) -> np.ndarray:
    """n token ids spread over [0, T): both ends plus seeded random picks."""
    rng = np.random.default_rng(seed)
    pick = {0, T - 1} | set(rng.choice(T, size=min(n, T), replace=False).tolist())
    return np.array(sorted(pick)[:max(n, 2)], dtype=np.int64)


def covering_tokens(ref, T: int, n_random: int = 16, seed: int = 0, tile_rows=(128, 256)) -> np.ndarray:
    """Tokens whose outputs exercise every tile boundary of the expert GEMMs:
    for each expert that keeps rows, the tokens of its first and last kept
    row (its last, partial m-tile) and of the rows on both sides of every
    128- and 256-row tile edge inside its block; the first and the last token
    (the shared expert's tail tile); plus seeded random picks."""
    N = len(ref.kept)
    pick = {0, T - 1}
    for e in range(N):
        r0, r1 = int(ref.offsets[e]), int(ref.offsets[e + 1])
        if r1 <= r0:
            continue
        rows = {r0, r1 - 1}
        for tr in tile_rows:
            for edge in range(r0 + tr, r1, tr):
                rows |= {edge - 1, edge}
        pick |= {int(ref.row_token[r]) for r in rows}
    rng = np.random.default_rng(seed)
    pick |= set(rng.choice(T, size=min(n_random, T), replace=False).tolist())
    return np.array(sorted(pick), dtype=np.int64)


_ORACLE_CACHE = {}


def oracle_forward_cached(cfg: MoEConfig, seed: int, cpu):
    """The oracle's full forward (every token) of (cfg, seed), computed once
    per test process: the full-size workloads' forward and backward checks
    share it."""
    key = (cfg, seed)
    if key not in _ORACLE_CACHE:
        _ORACLE_CACHE[key] = oracle.forward_inputs(cpu)
    return _ORACLE_CACHE[key]


def gpu_inputs(cfg: MoEConfig, seed: int = 0):
    inp = make_inputs(cfg, seed, device="cuda")
    torch.cuda.synchronize()
    return inp


def check_layer(cfg: MoEConfig, seed: int = 0, sample=None, stages: bool = True, cache: bool = False):
    """Full comparison of one configuration.

    Routing, dispatch, kept counts, drops, prob sums and the aux loss are
    compared on every token. FFN outputs are compared on every row
    (sample=None), on the rows of `sample` random tokens (an int), or on
    sample="cover": the tokens of covering_tokens (every expert's first and
    last kept row, both sides of every 128/256-row tile edge, the first and
    last token). With `stages`, each ABI stage is also run on oracle-produced
    inputs, isolating it from the stages before it. With `cache`, the oracle's
    full forward is kept for later tests of the same (cfg, seed).
    """
    inp = gpu_inputs(cfg, seed)
    cpu = inp.to("cpu")
    T, K, N, d = cfg.T, cfg.K, cfg.N, cfg.d_model
    want = None
    if sample == "cover":
        routing = oracle.forward_inputs(cpu, skip_ffn=True)
        want = np.zeros(T, dtype=np.uint8)
        want[covering_tokens(routing, T, seed=seed)] = 1
    elif sample is not None and sample < T:
        want = np.zeros(T, dtype=np.uint8)
        want[sample_tokens(T, sample, seed)] = 1
    if want is None and cache:
        ref = oracle_forward_cached(cfg, seed, cpu)
    else:
        ref = oracle.forward_inputs(cpu, want=want)
    shape = lib.shape_of(cfg)
    assert lib.capacity(shape) == ref.capacity

    # ---- the whole layer through moe_forward
    layer = lib.MoELayer.from_inputs(inp)
    ro = layer.route_outputs()
    y = layer.forward(inp.x, inp.sel_bias, route_out=ro)
    torch.cuda.synchronize()
    assert lib.device_error() == 0

    assert np.array_equal(ro.topk_idx.cpu().numpy(), ref.topk_idx), "topk_idx"
    assert np.allclose(ro.topk_w.cpu().numpy(), ref.topk_w, rtol=0, atol=W_ATOL), "topk_w"
    assert np.array_equal(ro.demand.cpu().numpy(), ref.demand), "demand"
    assert np.allclose(ro.prob_sum.cpu().numpy().astype(np.float64), ref.P * T, rtol=PROB_RTOL, atol=1e-6), "prob_sum"
    assert np.array_equal(ro.kept.cpu().numpy(), ref.kept), "kept"
    assert np.array_equal(ro.expert_offsets.cpu().numpy(), ref.offsets), "expert_offsets"
    assert np.array_equal(ro.slot_of.cpu().numpy(), ref.slot_of), "slot_of"
    aux = float(ro.aux.cpu()[0])
    assert abs(aux - ref.aux) <= AUX_RTOL * abs(ref.aux), ("aux", aux, ref.aux)
    zl = float(ro.z_loss.cpu()[0])
    assert abs(zl - ref.z_loss) <= AUX_RTOL * abs(ref.z_loss), ("z_loss", zl, ref.z_loss)
    kl = float(ro.aux_kl.cpu()[0])
    if np.isfinite(ref.aux_kl):
        assert abs(kl - ref.aux_kl) <= AUX_RTOL * abs(ref.aux_kl) + 1e-7, ("aux_kl", kl, ref.aux_kl)
    else:
        assert kl == ref.aux_kl, ("aux_kl", kl, ref.aux_kl)

    hl = ro.health.cpu().numpy().astype(np.float64)
    assert abs(hl[0] - ref.health[0]) <= 1e-5 * ref.health[0] + 1e-7, ("util_std", hl[0], ref.health[0])
    assert abs(hl[1] - ref.health[1]) <= 1e-6, ("drop_rate", hl[1], ref.health[1])
    assert abs(hl[2] - ref.health[2]) <= 1e-5 * abs(ref.health[2]) + 1e-6, ("entropy", hl[2], ref.health[2])
    assert hl[3] == np.float32(ref.health[3]), ("max|logit|", hl[3], ref.health[3])
    assert np.allclose(ro.mean_weight.cpu().numpy(), ref.mean_weight, rtol=0, atol=W_ATOL), "mean_weight"

    yb = bits_np(y)
    rows = slice(None) if want is None else want.astype(bool)
    assert_bf16_tol(yb[rows], ref.y[rows], "forward y")

    if not stages:
        return ref
    # ---- stage by stage, each fed with oracle-produced inputs
    idx, w, demand, psum = lib.route(shape, inp.x, inp.Wg, inp.sel_bias)
    torch.cuda.synchronize()
    assert np.array_equal(idx.cpu().numpy(), ref.topk_idx)
    assert np.allclose(w.cpu().numpy(), ref.topk_w, rtol=0, atol=W_ATOL)
    assert np.array_equal(demand.cpu().numpy(), ref.demand)

    ref_idx = torch.from_numpy(ref.topk_idx).cuda()
    kept, offsets, slot_of, row_token, x_perm = lib.dispatch(shape, ref_idx, inp.x)  # policy from shape
    torch.cuda.synchronize()
    assert np.array_equal(kept.cpu().numpy(), ref.kept)
    assert np.array_equal(offsets.cpu().numpy(), ref.offsets)
    assert np.array_equal(slot_of.cpu().numpy(), ref.slot_of)
    assert np.array_equal(row_token.cpu().numpy(), ref.row_token)
    R = int(ref.offsets[N])
    xb = bits_np(inp.x)
    assert np.array_equal(bits_np(x_perm)[:R], xb[ref.row_token[:R]]), "x_perm = x[row_token]"

    # FFN on the oracle's regrouped rows
    xp = torch.zeros((T * K, d), dtype=torch.bfloat16, device="cuda")
    if R:
        xp[:R] = inp.x[torch.from_numpy(ref.row_token[:R].astype(np.int64)).cuda()]
    y_perm, z = lib.expert_ffn(shape, xp, torch.from_numpy(ref.offsets).cuda(), inp.W1, inp.b1, inp.W2, inp.b2,
                               inp.x, inp.Ws1, inp.bs1, inp.Ws2, inp.bs2, quant=inp.quant)
    torch.cuda.synchronize()
    ypb = bits_np(y_perm)[:R]
    if want is None:
        assert_bf16_tol(ypb, ref.y_perm, "y_perm")
    else:
        live = want[ref.row_token[:R]].astype(bool)
        assert_bf16_tol(ypb[live], ref.y_perm[live], "y_perm (sampled)")
    if cfg.has_shared:
        assert_bf16_tol(bits_np(z)[rows], ref.z[rows], "z_shared")

    # combine on the oracle's expert outputs and weights
    if want is None:
        yp_ref = torch.zeros((T * K, d), dtype=torch.bfloat16, device="cuda")
        if R:
            yp_ref[:R] = torch.from_numpy(ref.y_perm.view(np.int16)).cuda().view(torch.bfloat16)
        z_ref = None
        if cfg.has_shared:
            z_ref = torch.from_numpy(ref.z.view(np.int16)).cuda().view(torch.bfloat16)
        yc = lib.combine(shape, yp_ref, torch.from_numpy(ref.slot_of).cuda(), torch.from_numpy(ref.topk_w).cuda(),
                         z_ref)
        torch.cuda.synchronize()
        assert_bf16_tol(bits_np(yc), ref.y, "combine")

    a = lib.aux_loss(shape, torch.from_numpy(ref.demand).cuda(),
                     torch.from_numpy((ref.P * T).astype(np.float32)).cuda())
    assert abs(float(a.cpu()[0]) - ref.aux) <= AUX_RTOL * abs(ref.aux)
    assert lib.device_error() == 0
    return ref
