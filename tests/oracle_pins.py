"""Pins of the CPU oracle against facts that do not come from the oracle.

Each ``pin_*`` takes an ``Oracle`` and raises AssertionError when the oracle
disagrees with a closed form, an invariant, a library routine on a special
case, brute force on a tiny input, or the worked example printed on the pages.
``test_oracle.py`` runs them on the real oracle; ``test_oracle_mutations.py``
runs them on deliberately broken copies of the oracle to show each planted
mistake is caught.
"""

from __future__ import annotations

import itertools
import json
import math
import os

import numpy as np
import scipy.special
import torch
import torch.nn.functional as F

from oracle import bf16_to_f64

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ------------------------------------------------------------------ helpers

def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def grid_x(rng, T, d):
    return bits(torch.from_numpy(rng.integers(-128, 129, (T, d)) / 64.0).to(torch.bfloat16))


def grid_wg(rng, N, d, lo=-8, hi=8):
    return bits(torch.from_numpy(rng.integers(lo, hi + 1, (N, d)) / 64.0).to(torch.bfloat16))


def randn_bf16(rng, shape, std):
    return bits(torch.from_numpy(rng.standard_normal(shape) * std).to(torch.float32).to(torch.bfloat16))


def torch_expert(xb, W1e, b1e, W2e, b2e) -> np.ndarray:
    """Dense FFN through torch's float64 library ops: Linear -> GELU (erf) ->
    bf16 -> Linear -> bf16. Independent of the oracle's C code."""
    x = torch.from_numpy(bf16_to_f64(xb))
    W1 = torch.from_numpy(bf16_to_f64(W1e))
    W2 = torch.from_numpy(bf16_to_f64(W2e))
    b1 = torch.from_numpy(np.asarray(b1e, np.float64))
    b2 = torch.from_numpy(np.asarray(b2e, np.float64))
    h = F.gelu(F.linear(x, W1, b1)).to(torch.bfloat16).to(torch.float64)
    return F.linear(h, W2, b2).numpy()


def to_bf16_bits_f64(v: np.ndarray) -> np.ndarray:
    return bits(torch.from_numpy(np.asarray(v, np.float64)).to(torch.bfloat16))


def assert_bf16_close(got_bits, ref_bits, max_mismatch_frac=1e-3, what=""):
    """bf16 results equal bit for bit, except a small fraction (double rounding
    through float32 in torch's float64->bf16 cast) which must lie within one
    bf16 ulp."""
    got_bits = np.asarray(got_bits, np.uint16)
    ref_bits = np.asarray(ref_bits, np.uint16)
    assert got_bits.shape == ref_bits.shape, what
    diff = got_bits != ref_bits
    frac = diff.mean() if diff.size else 0.0
    assert frac <= max_mismatch_frac, f"{what}: {frac:.4%} of bf16 values differ"
    if diff.any():
        g = bf16_to_f64(got_bits[diff])
        r = bf16_to_f64(ref_bits[diff])
        ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(r), 1e-30))) - 7)
        assert np.all(np.abs(g - r) <= ulp * 1.0001), f"{what}: a differing value is more than 1 ulp off"


# ------------------------------------------------------------------ bf16 rounding

def pin_bf16_round(orc):
    """Double -> bf16 RNE matches torch's float32 -> bf16 cast on values that
    float32 holds exactly, including exact halfway cases (ties to even)."""
    rng = np.random.default_rng(1)
    v = rng.standard_normal(4000).astype(np.float32) * np.exp2(rng.integers(-20, 20, 4000)).astype(np.float32)
    # exact midpoints between neighbouring bf16 values: low 16 bits = 0x8000
    mids = (rng.integers(0x3000, 0x5000, 200).astype(np.uint32) << 16 | 0x8000).view(np.float32)
    v = np.concatenate([v, mids, np.float32([0.0, -0.0, 1.0, -3.5])])
    ref = bits(torch.from_numpy(v).to(torch.bfloat16))
    got = np.array([orc.bf16_round(float(a)) for a in v], dtype=np.uint16)
    assert np.array_equal(got, ref), "bf16 rounding differs from torch's RNE cast"
    assert orc.bf16_round(1 + 2 ** -8) == 0x3F80       # halfway -> even (1.0)
    assert orc.bf16_round(1 + 3 * 2 ** -8) == 0x3F82   # halfway -> even (1 + 2^-6)


# ------------------------------------------------------------------ GELU

def pin_gelu(orc):
    """erf-form GELU: torch's exact GELU in float64 and the limits."""
    xs = np.linspace(-8, 8, 401)
    ref = F.gelu(torch.from_numpy(xs), approximate="none").numpy()
    got = np.array([orc.gelu(float(a)) for a in xs])
    assert np.allclose(got, ref, rtol=1e-14, atol=1e-15)
    assert orc.gelu(0.0) == 0.0
    assert abs(orc.gelu(30.0) - 30.0) < 1e-12 and abs(orc.gelu(-30.0)) < 1e-12
    assert abs(orc.gelu(1.0) - 0.5 * (1 + math.erf(1 / math.sqrt(2)))) < 1e-15


# ------------------------------------------------------------------ capacity

def pin_capacity(orc):
    """capacity = ceil(T / N * capacity_factor); dropless (cf <= 0) = T."""
    assert orc.capacity(256, 8, 1.25) == 40
    assert orc.capacity(4096, 8, 1.25) == 640
    assert orc.capacity(8192, 64, 1.0) == 128
    assert orc.capacity(4096, 256, 0.0) == 4096
    assert orc.capacity(10, 3, 1.0) == 4      # ceil(3.33)
    assert orc.capacity(7, 2, 1.5) == 6       # ceil(5.25)
    assert orc.capacity(16, 8, 2.0) == 4
    assert orc.capacity(5, 8, 100.0) == 5     # never above T


# ------------------------------------------------------------------ gate

def pin_gate_exact(orc):
    """On the 1/64 grid every logit is an integer multiple of 2^-12: check it
    against int64 matrix arithmetic (exact)."""
    rng = np.random.default_rng(2)
    T, d, N = 37, 96, 5
    x = grid_x(rng, T, d)
    Wg = grid_wg(rng, N, d)
    s = orc.gate_logits(x, Wg)
    xi = np.rint(bf16_to_f64(x) * 64).astype(np.int64)
    wi = np.rint(bf16_to_f64(Wg) * 64).astype(np.int64)
    ref = (xi @ wi.T).astype(np.float64) / 4096.0
    assert s.shape == (T, N)
    assert np.array_equal(s, ref)


# ------------------------------------------------------------------ route

def _brute_topk(u_row, K):
    """Lexicographically smallest id set among the K-subsets of maximal sum."""
    best, best_set = None, None
    for comb in itertools.combinations(range(len(u_row)), K):  # lexicographic order
        sm = sum(u_row[i] for i in comb)
        if best is None or sm > best:
            best, best_set = sm, comb
    return set(best_set)


def pin_route_bruteforce(orc):
    """Selection = the maximal-sum K-subset (smallest ids on ties), ranked by
    value then id; weights = softmax of the K unbiased logits (scipy)."""
    rng = np.random.default_rng(3)
    for N, K, with_bias in [(6, 1, False), (6, 2, False), (6, 3, True), (5, 5, False), (7, 2, True)]:
        T = 48
        s = rng.integers(-3, 4, (T, N)).astype(np.float64)  # small range: ties are common
        bias = (rng.integers(-2, 3, N) / 2.0).astype(np.float32) if with_bias else None
        idx, w, demand, P = orc.route(s, K, bias)
        u = s + (bias.astype(np.float64) if with_bias else 0.0)
        for t in range(T):
            assert set(idx[t].tolist()) == _brute_topk(u[t], K), (N, K, t)
            assert len(set(idx[t].tolist())) == K
            for k in range(K - 1):
                a, b = idx[t, k], idx[t, k + 1]
                assert u[t, a] > u[t, b] or (u[t, a] == u[t, b] and a < b)
            ref = scipy.special.softmax(s[t, idx[t]])
            assert np.allclose(w[t], ref, rtol=2e-7, atol=1e-12)
        assert np.array_equal(demand, np.bincount(idx.ravel(), minlength=N))
        assert np.allclose(P, scipy.special.softmax(s, axis=1).mean(0), rtol=1e-13, atol=1e-15)


def pin_route_closed_forms(orc):
    """K=2: w0 = sigmoid(s_a - s_b); K=1: w = 1; sum of weights = 1; all-equal
    logits select experts 0..K-1; a selection bias moves the choice but not
    the weights."""
    rng = np.random.default_rng(4)
    s = rng.standard_normal((64, 8)) * 3
    idx, w, _, _ = orc.route(s, 2)
    d = s[np.arange(64), idx[:, 0]] - s[np.arange(64), idx[:, 1]]
    assert np.allclose(w[:, 0], scipy.special.expit(d), rtol=2e-7)
    assert np.all(d >= 0)
    assert np.all(np.abs(w.sum(1) - 1) < 2e-7)
    idx1, w1, _, _ = orc.route(s, 1)
    assert np.all(w1 == 1.0) and np.array_equal(idx1[:, 0], np.argmax(s, axis=1))
    idxe, _, _, _ = orc.route(np.zeros((3, 8)), 4)
    assert np.array_equal(idxe, np.tile(np.arange(4), (3, 1)))
    sb = np.array([[1.0, 0.0, 0.5]])
    idxb, wb, _, _ = orc.route(sb, 2, np.float32([0.0, 2.0, 0.0]))
    assert idxb.tolist() == [[1, 0]]
    assert np.allclose(wb[0], [scipy.special.expit(-1.0), scipy.special.expit(1.0)], rtol=2e-7)


def pin_worked_example(orc):
    """The pages' worked top-2 example (the selection; the weights follow the
    formula -- see the fixture for why the printed 0.62 is not pinned)."""
    with open(os.path.join(GOLDEN, "worked_example_top2.json")) as fh:
        g = json.load(fh)
    idx, w, _, _ = orc.route(np.array([g["logits"]]), g["K"])
    assert idx[0].tolist() == g["expected_idx"]
    assert [i + 1 for i in idx[0]] == g["page_selected_1based"]
    assert np.allclose(w[0], g["expected_weights"], rtol=1e-7)


# ------------------------------------------------------------------ dispatch

def _brute_dispatch(idx, N, C):
    """Stable sort of all (expert, token) pairs, keep the first C per expert."""
    T, K = idx.shape
    pairs = sorted(((int(idx[t, k]), t, k) for t in range(T) for k in range(K)),
                   key=lambda p: (p[0], p[1]))
    slot = -np.ones((T, K), np.int64)
    rows = []
    per = {}
    for e, t, k in pairs:
        if per.get(e, 0) < C:
            per[e] = per.get(e, 0) + 1
            slot[t, k] = len(rows)
            rows.append(t)
    kept = np.array([per.get(e, 0) for e in range(N)])
    return slot, np.array(rows, dtype=np.int64), kept


def _brute_dispatch_rank_major(idx, N, C):
    """Stable sort of all (expert, rank, token) triples, first C per expert."""
    T, K = idx.shape
    triples = sorted(((int(idx[t, k]), k, t) for t in range(T) for k in range(K)))
    slot = -np.ones((T, K), np.int64)
    rows, per = [], {}
    for e, k, t in triples:
        if per.get(e, 0) < C:
            per[e] = per.get(e, 0) + 1
            slot[t, k] = len(rows)
            rows.append(t)
    return slot, np.array(rows, dtype=np.int64), np.array([per.get(e, 0) for e in range(N)])


def pin_dispatch_rank_major(orc):
    """Rank-major capacity priority: every first choice is served before any
    second choice; brute force over (expert, rank, token) triples, and with
    room for everyone it keeps the same rows as token order."""
    rng = np.random.default_rng(14)
    for T, N, K, C in [(40, 5, 2, 6), (33, 8, 3, 4), (20, 4, 1, 3), (30, 6, 3, 30)]:
        idx, _, demand, _ = orc.route(rng.standard_normal((T, N)), K)
        kept, offsets, slot_of, row_token = orc.dispatch(idx, N, C, rank_major=True)
        slot, rows, kept_ref = _brute_dispatch_rank_major(idx, N, C)
        assert np.array_equal(slot_of, slot)
        R = len(rows)
        assert np.array_equal(row_token[:R], rows) and np.all(row_token[R:] == -1)
        assert np.array_equal(kept, kept_ref) and np.array_equal(kept, np.minimum(demand, C))
        tok = orc.dispatch(idx, N, C)
        assert np.array_equal(tok[0], kept)           # kept counts never depend on the order
        if C >= T:
            assert np.array_equal(tok[2] >= 0, slot_of >= 0)
    # a case where the orders disagree: token 0's second choice vs token 1's first
    idx = np.array([[0, 1], [1, 0]], np.int32)
    _, _, s_tok, _ = orc.dispatch(idx, 2, 1)
    _, _, s_rank, _ = orc.dispatch(idx, 2, 1, rank_major=True)
    assert s_tok.tolist() == [[0, 1], [-1, -1]]      # token 0 takes both seats
    assert s_rank.tolist() == [[0, -1], [1, -1]]     # first choices take them


def pin_aux_kl(orc):
    """coef * KL(uniform || f): 0 for uniform demand; torch's kl_div on the
    same frequencies (the listing's own call); +inf for an idle expert."""
    assert abs(orc.aux_kl(np.array([5, 5, 5, 5], np.int32), 10, 2, 0.02)) < 1e-15
    rng = np.random.default_rng(15)
    demand = rng.integers(1, 50, 7).astype(np.int32)
    T, K = int(demand.sum()), 1
    f = torch.from_numpy(demand.astype(np.float64) / (T * K))
    ref = 0.02 * float(F.kl_div(f.log(), torch.full((7,), 1 / 7, dtype=torch.float64), reduction="sum"))
    assert abs(orc.aux_kl(demand, T, K, 0.02) - ref) < 1e-14
    assert orc.aux_kl(np.array([4, 0], np.int32), 2, 2, 0.02) == math.inf


def pin_dispatch_bruteforce(orc):
    rng = np.random.default_rng(5)
    for T, N, K, C in [(40, 5, 2, 6), (40, 5, 2, 40), (33, 8, 3, 4), (20, 4, 1, 3), (16, 6, 6, 9)]:
        s = rng.standard_normal((T, N))
        idx, _, demand, _ = orc.route(s, K)
        kept, offsets, slot_of, row_token = orc.dispatch(idx, N, C)
        slot, rows, kept_ref = _brute_dispatch(idx, N, C)
        assert np.array_equal(slot_of, slot)
        R = len(rows)
        assert offsets[N] == R and np.array_equal(row_token[:R], rows)
        assert np.all(row_token[R:] == -1)
        assert np.array_equal(kept, kept_ref) and np.array_equal(kept, np.minimum(demand, C))
        assert np.array_equal(offsets, np.concatenate([[0], np.cumsum(kept)]))
        # round trip: kept slots form a bijection onto [0, R) and point back to their token
        live = slot_of[slot_of >= 0]
        assert np.array_equal(np.sort(live), np.arange(R))
        tt = np.repeat(np.arange(T)[:, None], K, 1)
        assert np.array_equal(row_token[slot_of[slot_of >= 0]], tt[slot_of >= 0])


def pin_permutation_roundtrip(orc):
    """Gathering x by row_token and scattering back through slot_of restores x."""
    rng = np.random.default_rng(6)
    T, d, N, K = 50, 16, 6, 2
    x = grid_x(rng, T, d)
    idx, _, _, _ = orc.route(rng.standard_normal((T, N)), K)
    kept, offsets, slot_of, row_token = orc.dispatch(idx, N, T)
    R = offsets[N]
    assert R == T * K
    x_perm = x[row_token[:R]]
    for e in range(N):  # contiguous per-expert blocks, tokens increasing
        blk = row_token[offsets[e]:offsets[e + 1]]
        assert np.all(np.diff(blk) > 0)
        assert np.all((idx[blk] == e).any(axis=1))
    for k in range(K):
        assert np.array_equal(x_perm[slot_of[:, k]], x)


# ------------------------------------------------------------------ FFN and combine

def _small_layer(rng, T, d, f, N):
    x = grid_x(rng, T, d)
    Wg = grid_wg(rng, N, d)
    W1 = randn_bf16(rng, (N, f, d), d ** -0.5)
    b1 = (rng.standard_normal((N, f)) * 0.02).astype(np.float32)
    W2 = randn_bf16(rng, (N, d, f), f ** -0.5)
    b2 = (rng.standard_normal((N, d)) * 0.02).astype(np.float32)
    return x, Wg, W1, b1, W2, b2


def pin_dense_special_case(orc):
    """N = 1, K = 1, dropless: the layer is one dense FFN (torch float64 ops)."""
    rng = np.random.default_rng(7)
    T, d, f = 24, 32, 48
    x, Wg, W1, b1, W2, b2 = _small_layer(rng, T, d, f, 1)
    r = orc.forward(x, Wg, W1, b1, W2, b2, K=1, capacity_factor=0.0, aux_alpha=0.01)
    ref = to_bf16_bits_f64(torch_expert(x, W1[0], b1[0], W2[0], b2[0]))
    assert np.all(r.topk_w == 1.0)
    assert_bf16_close(r.y, ref, what="dense FFN")


def pin_identical_experts(orc):
    """All experts share weights and nothing is dropped: the weights sum to 1
    within fp32 rounding, which cannot move a bf16 value, so y == E(x)."""
    rng = np.random.default_rng(8)
    T, d, f, N, K = 40, 32, 64, 4, 2
    x, Wg, W1, b1, W2, b2 = _small_layer(rng, T, d, f, 1)
    W1n, b1n = np.repeat(W1, N, 0), np.repeat(b1, N, 0)
    W2n, b2n = np.repeat(W2, N, 0), np.repeat(b2, N, 0)
    Wg = grid_wg(rng, N, d)
    r = orc.forward(x, Wg, W1n, b1n, W2n, b2n, K=K, capacity_factor=0.0, aux_alpha=0.01)
    single = orc.expert_rows(x, np.arange(T, dtype=np.int32), W1[0], b1[0], W2[0], b2[0])
    assert np.array_equal(r.y, single)
    assert_bf16_close(single, to_bf16_bits_f64(torch_expert(x, W1[0], b1[0], W2[0], b2[0])),
                      what="shared-weight expert")


def pin_token_major(orc):
    """Dropless, distinct experts: y[t] = bf16(sum_k w[t,k] E_{idx[t,k]}(x_t)),
    evaluated token by token with torch, no permutation at all."""
    rng = np.random.default_rng(9)
    T, d, f, N, K = 30, 32, 48, 5, 2
    x, Wg, W1, b1, W2, b2 = _small_layer(rng, T, d, f, N)
    r = orc.forward(x, Wg, W1, b1, W2, b2, K=K, capacity_factor=0.0, aux_alpha=0.01)
    out = np.zeros((T, d))
    for e in range(N):
        o = bf16_to_f64(to_bf16_bits_f64(torch_expert(x, W1[e], b1[e], W2[e], b2[e])))
        for k in range(K):
            sel = r.topk_idx[:, k] == e
            out[sel] += r.topk_w[sel, k].astype(np.float64)[:, None] * o[sel]
    assert_bf16_close(r.y, to_bf16_bits_f64(out), max_mismatch_frac=3e-3, what="token-major")


def pin_soft_router(orc):
    """K = N ('soft router'): y = sum_e softmax(s)_e E_e(x)."""
    rng = np.random.default_rng(10)
    T, d, f, N = 20, 32, 32, 4
    x, Wg, W1, b1, W2, b2 = _small_layer(rng, T, d, f, N)
    r = orc.forward(x, Wg, W1, b1, W2, b2, K=N, capacity_factor=0.0, aux_alpha=0.01)
    s = r.logits
    p = scipy.special.softmax(s, axis=1).astype(np.float32).astype(np.float64)
    out = np.zeros((T, d))
    for e in range(N):
        out += p[:, e:e + 1] * bf16_to_f64(to_bf16_bits_f64(torch_expert(x, W1[e], b1[e], W2[e], b2[e])))
    assert_bf16_close(r.y, to_bf16_bits_f64(out), max_mismatch_frac=3e-3, what="soft router")


def pin_drops_and_shared(orc):
    """Capacity drops leave only the kept assignments; with the routed experts
    silenced (W2 = 0, b2 = 0) the output is exactly the shared expert's."""
    rng = np.random.default_rng(11)
    T, d, f, N, K = 32, 32, 48, 4, 2
    x, Wg, W1, b1, W2, b2 = _small_layer(rng, T, d, f, N)
    Ws1, bs1 = W1[0].copy(), b1[0].copy()
    Ws2, bs2 = W2[1].copy(), b2[1].copy()
    zero2, zb2 = np.zeros_like(W2), np.zeros_like(b2)
    r = orc.forward(x, Wg, W1, b1, zero2, zb2, K=K, capacity_factor=1.0, aux_alpha=0.01,
                    Ws1=Ws1, bs1=bs1, Ws2=Ws2, bs2=bs2)
    z_ref = to_bf16_bits_f64(torch_expert(x, Ws1, bs1, Ws2, bs2))
    assert_bf16_close(r.z, z_ref, what="shared expert")
    assert np.array_equal(r.y, r.z)
    # routed only, with drops: the dropped assignment contributes nothing
    r2 = orc.forward(x, Wg, W1, b1, W2, b2, K=K, capacity_factor=1.0, aux_alpha=0.01)
    assert r2.capacity == 8 and (r2.slot_of < 0).any()
    out = np.zeros((T, d))
    for e in range(N):
        o = bf16_to_f64(to_bf16_bits_f64(torch_expert(x, W1[e], b1[e], W2[e], b2[e])))
        for k in range(K):
            sel = (r2.topk_idx[:, k] == e) & (r2.slot_of[:, k] >= 0)
            out[sel] += r2.topk_w[sel, k].astype(np.float64)[:, None] * o[sel]
    assert_bf16_close(r2.y, to_bf16_bits_f64(out), max_mismatch_frac=3e-3, what="dropped")


# ------------------------------------------------------------------ aux loss

def pin_aux(orc):
    """alpha * N * sum f P: equals alpha for uniform logits (any f) and for
    uniform f (any P); lies in [0, alpha N]; f and P are distributions."""
    rng = np.random.default_rng(12)
    alpha = 0.01
    for N, K in [(8, 2), (6, 1), (16, 4)]:
        T = 64
        idx, w, demand, P = orc.route(np.zeros((T, N)), K)
        assert abs(orc.aux_loss(demand, P, T, K, alpha) - alpha) < 1e-15
        # uniform f: token t prefers experts t, t+1, ..., t+K-1 (mod N), T = N
        s = np.zeros((N, N))
        for t in range(N):
            for j in range(K):
                s[t, (t + j) % N] = 10.0 - j
        s += rng.standard_normal((N, N)) * 0.01
        idx, w, demand, P = orc.route(s, K)
        assert np.all(demand == K)
        assert abs(orc.aux_loss(demand, P, N, K, alpha) - alpha) < 1e-14
        s = rng.standard_normal((T, N)) * 4
        idx, w, demand, P = orc.route(s, K)
        a = orc.aux_loss(demand, P, T, K, alpha)
        assert 0.0 <= a <= alpha * N
        assert demand.sum() == T * K and abs(P.sum() - 1) < 1e-12
    # all mass on one expert: f = P = 1 for it -> alpha * N
    idx, w, demand, P = orc.route(np.tile([[50.0, 0, 0, 0]], (10, 1)), 1)
    assert abs(orc.aux_loss(demand, P, 10, 1, alpha) - alpha * 4) < 1e-12


# ------------------------------------------------------------------ router z-loss

def pin_z_loss(orc):
    """beta * mean_t logsumexp(s_t)^2: scipy's logsumexp on random logits;
    equal logits c give (c + log N)^2; one expert gives mean(s^2); large
    logits stay finite (max-shifted evaluation)."""
    rng = np.random.default_rng(13)
    beta = 1e-3
    s = rng.standard_normal((50, 7)) * 5
    ref = beta * np.mean(scipy.special.logsumexp(s, axis=1) ** 2)
    assert abs(orc.z_loss(s, beta) - ref) <= 1e-13 * abs(ref)
    c = 2.5
    assert abs(orc.z_loss(np.full((9, 16), c), 1.0) - (c + math.log(16)) ** 2) < 1e-12
    one = rng.standard_normal((20, 1))
    assert abs(orc.z_loss(one, 1.0) - float(np.mean(one[:, 0] ** 2))) < 1e-12
    big = np.array([[800.0, 799.0, 0.0]])
    v = orc.z_loss(big, 1.0)
    assert math.isfinite(v) and abs(v - scipy.special.logsumexp(big[0]) ** 2) < 1e-9 * v
    assert orc.z_loss(s, 0.0) == 0.0


def pin_fp8_decode(orc):
    """FP8 E4M3 decoding of every code against torch's float8_e4m3fn."""
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = np.array([orc.fp8_value(int(c)) for c in codes])
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(mine[ok], ref[ok])
    assert orc.fp8_value(0x7E) == 448.0 and orc.fp8_value(0x01) == 2.0 ** -9


def _fp8_exact_weights(rng, shape):
    """FP8 codes with one power-of-two scale per output row (rows differ), and
    the same weights as bf16 (code * 2^k has at most 4 significant bits)."""
    codes = rng.integers(0, 256, size=shape).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x3F   # no NaN codes
    k = rng.integers(-9, -3, size=shape[:-1])
    scale = np.ldexp(1.0, k).astype(np.float32)
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy() * scale[..., None]
    bf = torch.from_numpy(vals).to(torch.bfloat16)
    assert np.array_equal(bf.to(torch.float64).numpy(), vals)   # exactly representable
    return codes, scale, bits(bf)


def pin_fp8_experts(orc):
    """Quantised experts whose dequantised weights are exactly a bf16 weight
    set give bit-identical outputs to the bf16 experts (routed and shared),
    so the quantised path inherits the bf16 path's pins; per-row scales differ,
    so a scale taken from the wrong row or column fails."""
    rng = np.random.default_rng(17)
    T, d, f, N, K = 48, 32, 48, 4, 2
    x = grid_x(rng, T, d)
    Wg = grid_wg(rng, N, d)
    W1q, s1, W1 = _fp8_exact_weights(rng, (N, f, d))
    W2q, s2, W2 = _fp8_exact_weights(rng, (N, d, f))
    Ws1q, ss1, Ws1 = _fp8_exact_weights(rng, (f, d))
    Ws2q, ss2, Ws2 = _fp8_exact_weights(rng, (d, f))
    b1 = (rng.standard_normal((N, f)) * 0.02).astype(np.float32)
    b2 = (rng.standard_normal((N, d)) * 0.02).astype(np.float32)
    bs1 = (rng.standard_normal(f) * 0.02).astype(np.float32)
    bs2 = (rng.standard_normal(d) * 0.02).astype(np.float32)
    ref = orc.forward(x, Wg, W1, b1, W2, b2, K=K, capacity_factor=0.0, aux_alpha=0.01,
                      Ws1=Ws1, bs1=bs1, Ws2=Ws2, bs2=bs2)

    class Q:
        pass
    q = Q()
    q.W1q, q.s1, q.W2q, q.s2, q.Ws1q, q.ss1, q.Ws2q, q.ss2 = W1q, s1, W2q, s2, Ws1q, ss1, Ws2q, ss2
    got = orc.forward(x, Wg, None, b1, None, b2, K=K, capacity_factor=0.0, aux_alpha=0.01,
                      bs1=bs1, bs2=bs2, quant=q)
    assert np.array_equal(got.y_perm, ref.y_perm)
    assert np.array_equal(got.z, ref.z)
    assert np.array_equal(got.y, ref.y)
    # and the dense special case through torch: one quantised expert = one Linear/GELU/Linear
    e_rows = orc.expert_ffn_fp8(x, np.array([0, T], np.int32), np.arange(T, dtype=np.int32),
                                W1q[:1], s1[:1], b1[:1], W2q[:1], s2[:1], b2[:1])
    assert_bf16_close(e_rows, to_bf16_bits_f64(torch_expert(x, W1[0], b1[0], W2[0], b2[0])),
                      what="fp8 dense expert")


def pin_int4_dequant(orc):
    """INT4 dequantisation: every code c in 0..15 stands for c - 8, and the
    weight is (c - 8) * scale rounded to bf16 (RNE), checked against torch's
    float32 product (exact: at most 11 significant bits) cast to bfloat16, for
    scales that need rounding, including an exact halfway case."""
    scales = torch.tensor([1.0, 1.0078125, 1.9921875, 0.3359375, 3.0e-3, -0.75, 117.0], dtype=torch.bfloat16)
    for sb in scales:
        sbits = int(sb.view(torch.int16).item()) & 0xFFFF
        for c in range(16):
            want = (torch.tensor(float(c - 8), dtype=torch.float32) * sb.to(torch.float32)).to(torch.bfloat16)
            assert orc.int4_dequant(c, sbits) == float(want.to(torch.float64)), (c, float(sb))
    # (11 - 8) * 1.0078125 = 3.0234375 lies halfway between bf16 3.015625 and
    # 3.03125: round to the even mantissa
    half_bits = int(torch.tensor(1.0078125, dtype=torch.bfloat16).view(torch.int16).item()) & 0xFFFF
    assert orc.int4_dequant(11, half_bits) == 3.03125
    assert orc.int4_dequant(8, half_bits) == 0.0 and orc.int4_dequant(0, 0x3F80) == -8.0


def _int4_pack(codes):
    """The INT4 byte layout written out bit by bit: each run of eight columns
    becomes one little-endian 32-bit word whose bits 4j .. 4j + 3 take column
    2j of the run and bits 16 + 4j .. 19 + 4j column 2j + 1."""
    *lead, inn = codes.shape
    runs = codes.reshape(*lead, inn // 8, 8).astype(np.uint32)
    word = np.zeros(runs.shape[:-1], np.uint32)
    for j in range(4):
        word |= runs[..., 2 * j] << np.uint32(4 * j)
        word |= runs[..., 2 * j + 1] << np.uint32(16 + 4 * j)
    return word.astype("<u4").view(np.uint8).reshape(*lead, inn // 2)


def _int4_weights(rng, out, inn, lead=()):
    """Random INT4 codes in the packed layout and random bf16 group scales
    [..., inn / 128, out]; returns them with the dequantised bf16 weights
    [..., out, inn] computed independently in torch."""
    codes = rng.integers(0, 16, size=lead + (out, inn)).astype(np.uint8)
    packed = _int4_pack(codes)
    sc = torch.from_numpy(rng.uniform(0.004, 0.06, size=lead + (inn // 128, out))).to(torch.bfloat16)
    s_full = sc.to(torch.float32).transpose(-1, -2).repeat_interleave(128, dim=-1)   # [..., out, inn]
    w = ((torch.from_numpy(codes.astype(np.float32)) - 8.0) * s_full).to(torch.bfloat16)
    return packed, bits(sc), bits(w)


def pin_int4_experts(orc):
    """INT4 group-wise experts give bit-identical outputs to bf16 experts
    holding their dequantised weights (routed and shared), the dequantisation
    done independently in torch from the packed layout: so the INT4 path
    inherits the bf16 path's pins, and a swapped nibble, a scale from the
    wrong row or group, or an unrounded weight fails."""
    rng = np.random.default_rng(23)
    T, d, f, N, K = 40, 256, 384, 4, 2
    x = grid_x(rng, T, d)
    Wg = grid_wg(rng, N, d)
    W1q, g1, W1 = _int4_weights(rng, f, d, (N,))
    W2q, g2, W2 = _int4_weights(rng, d, f, (N,))
    Ws1q, gs1, Ws1 = _int4_weights(rng, f, d)
    Ws2q, gs2, Ws2 = _int4_weights(rng, d, f)
    b1 = (rng.standard_normal((N, f)) * 0.02).astype(np.float32)
    b2 = (rng.standard_normal((N, d)) * 0.02).astype(np.float32)
    bs1 = (rng.standard_normal(f) * 0.02).astype(np.float32)
    bs2 = (rng.standard_normal(d) * 0.02).astype(np.float32)
    ref = orc.forward(x, Wg, W1, b1, W2, b2, K=K, capacity_factor=0.0, aux_alpha=0.01,
                      Ws1=Ws1, bs1=bs1, Ws2=Ws2, bs2=bs2)

    class Q:
        format = "int4_g128"
    q = Q()
    q.W1q, q.s1, q.W2q, q.s2, q.Ws1q, q.ss1, q.Ws2q, q.ss2 = W1q, g1, W2q, g2, Ws1q, gs1, Ws2q, gs2
    got = orc.forward(x, Wg, None, b1, None, b2, K=K, capacity_factor=0.0, aux_alpha=0.01,
                      bs1=bs1, bs2=bs2, quant=q)
    assert np.array_equal(got.y_perm, ref.y_perm)
    assert np.array_equal(got.z, ref.z)
    assert np.array_equal(got.y, ref.y)


def _torch_layer_grads(x, Wg, W1, b1, W2, b2, fwd, dy, alpha, beta, g_aux, g_z, shared=None):
    """torch autograd in float64 of a plain restatement of the layer with the
    forward's routing decisions held fixed; the bf16 storage points (h, o, y)
    round the value and pass the gradient through unchanged."""
    f64 = torch.float64

    def t64(a):
        return torch.from_numpy(bf16_to_f64(a) if a.dtype == np.uint16 else a.astype(np.float64)).to(f64)

    def rb(v):  # bf16 rounding with an identity gradient
        return v + (v.to(torch.bfloat16).to(f64) - v).detach()

    xs, Wgs = t64(x).requires_grad_(), t64(Wg).requires_grad_()
    W1s, b1s, W2s, b2s = (t64(a).requires_grad_() for a in (W1, b1, W2, b2))
    T, d = xs.shape
    N, K = Wgs.shape[0], fwd.topk_idx.shape[1]
    idx = torch.from_numpy(fwd.topk_idx.astype(np.int64))
    s = xs @ Wgs.T
    w = torch.softmax(s.gather(1, idx), dim=1)
    y = torch.zeros((T, d), dtype=f64)
    for t in range(T):
        for k in range(K):
            if fwd.slot_of[t, k] < 0:
                continue
            e = int(idx[t, k])
            h = rb(torch.nn.functional.gelu(xs[t] @ W1s[e].T + b1s[e]))
            o = rb(h @ W2s[e].T + b2s[e])
            y[t] = y[t] + w[t, k] * o
    extra = []
    if shared is not None:
        Ws1s, bs1s, Ws2s, bs2s = (t64(a).requires_grad_() for a in shared)
        hs = rb(torch.nn.functional.gelu(xs @ Ws1s.T + bs1s))
        y = y + rb(hs @ Ws2s.T + bs2s)
        extra = [Ws1s, bs1s, Ws2s, bs2s]
    p = torch.softmax(s, dim=1)
    fr = torch.from_numpy(fwd.demand.astype(np.float64)) / (T * K)
    aux = alpha * N * (fr * p.mean(0)).sum()
    zl = beta * (torch.logsumexp(s, dim=1) ** 2).mean()
    L = (rb(y) * t64(dy)).sum() + g_aux * aux + g_z * zl
    L.backward()
    g = {"dx": xs.grad, "dWg": Wgs.grad, "dW1": W1s.grad, "db1": b1s.grad, "dW2": W2s.grad, "db2": b2s.grad}
    if extra:
        g.update({"dWs1": extra[0].grad, "dbs1": extra[1].grad, "dWs2": extra[2].grad, "dbs2": extra[3].grad})
    return {k: v.numpy() for k, v in g.items()}


def pin_backward_autograd(orc):
    """The backward against torch autograd in float64 (routing held fixed),
    with drops (capacity 0.75), a shared expert and non-unit loss weights;
    dw checked against <dy, o> by its definition through torch as well."""
    rng = np.random.default_rng(19)
    T, d, f, N, K = 20, 16, 24, 4, 2
    x, Wg, W1, b1, W2, b2 = _small_layer(rng, T, d, f, N)
    Ws1 = randn_bf16(rng, (f, d), d ** -0.5)
    Ws2 = randn_bf16(rng, (d, f), f ** -0.5)
    bs1 = (rng.standard_normal(f) * 0.02).astype(np.float32)
    bs2 = (rng.standard_normal(d) * 0.02).astype(np.float32)
    dy = bits(torch.from_numpy(rng.standard_normal((T, d))).to(torch.bfloat16))
    alpha, beta, g_aux, g_z = 0.01, 1e-3, 3.0, 5.0
    fwd = orc.forward(x, Wg, W1, b1, W2, b2, K=K, capacity_factor=0.75, aux_alpha=alpha, z_beta=beta,
                      Ws1=Ws1, bs1=bs1, Ws2=Ws2, bs2=bs2)
    assert (fwd.slot_of < 0).any(), "the case should drop some assignments"
    got = orc.backward(x, Wg, W1, b1, W2, b2, fwd, dy, alpha, beta, g_aux, g_z, Ws1, bs1, Ws2, bs2,
                       round_stored=False)
    ref = _torch_layer_grads(x, Wg, W1, b1, W2, b2, fwd, dy, alpha, beta, g_aux, g_z, (Ws1, bs1, Ws2, bs2))
    for name, r in ref.items():
        scale = max(np.abs(r).max(), 1e-30)
        assert np.abs(got[name] - r).max() <= 1e-10 * scale, name
    yp = bf16_to_f64(fwd.y_perm)
    dyv = bf16_to_f64(dy)
    for t in range(T):
        for k in range(K):
            r = fwd.slot_of[t, k]
            want = 0.0 if r < 0 else float(np.dot(dyv[t], yp[r]))
            assert abs(got["dw"][t, k] - want) <= 1e-12 * (1 + abs(want))
    # rounding dO and da to bf16 moves the gradients by about bf16 precision only
    rnd = orc.backward(x, Wg, W1, b1, W2, b2, fwd, dy, alpha, beta, g_aux, g_z, Ws1, bs1, Ws2, bs2)
    for name in ("dx", "dW1", "dW2"):
        rel = np.linalg.norm(rnd[name] - got[name]) / np.linalg.norm(got[name])
        assert 0 < rel < 1e-2, (name, rel)


def pin_backward_token_mask(orc):
    """The token-masked backward (used on full-size workloads) gives the same
    dx and dw on the wanted tokens as the full backward."""
    rng = np.random.default_rng(23)
    T, d, f, N, K = 30, 16, 32, 4, 2
    x, Wg, W1, b1, W2, b2 = _small_layer(rng, T, d, f, N)
    dy = bits(torch.from_numpy(rng.standard_normal((T, d))).to(torch.bfloat16))
    fwd = orc.forward(x, Wg, W1, b1, W2, b2, K=K, capacity_factor=1.0, aux_alpha=0.01)
    full = orc.backward(x, Wg, W1, b1, W2, b2, fwd, dy, 0.01, 1e-3)
    want = np.zeros(T, dtype=bool)
    want[[0, 7, 29]] = True
    part = orc.backward(x, Wg, W1, b1, W2, b2, fwd, dy, 0.01, 1e-3, want=want)
    assert np.array_equal(part["dx"][want], full["dx"][want])
    assert np.array_equal(part["dw"][want], full["dw"][want])


def pin_backward_pieces(orc):
    """The per-part backward functions used on full-size workloads agree with
    the whole backward (itself pinned to torch autograd): dw from the stored
    expert outputs, dW_g from dw, and each expert's weight and bias gradients
    (routed experts with drops, and the shared expert)."""
    rng = np.random.default_rng(31)
    T, d, f, N, K = 40, 16, 24, 5, 2
    x, Wg, W1, b1, W2, b2 = _small_layer(rng, T, d, f, N)
    Ws1 = randn_bf16(rng, (f, d), d ** -0.5)
    Ws2 = randn_bf16(rng, (d, f), f ** -0.5)
    bs1 = (rng.standard_normal(f) * 0.02).astype(np.float32)
    bs2 = (rng.standard_normal(d) * 0.02).astype(np.float32)
    dy = bits(torch.from_numpy(rng.standard_normal((T, d))).to(torch.bfloat16))
    alpha, beta, g_aux, g_z = 0.01, 1e-3, 2.0, 3.0
    fwd = orc.forward(x, Wg, W1, b1, W2, b2, K=K, capacity_factor=0.8, aux_alpha=alpha, z_beta=beta,
                      Ws1=Ws1, bs1=bs1, Ws2=Ws2, bs2=bs2)
    assert (fwd.slot_of < 0).any() and (fwd.kept > 0).sum() >= 3
    full = orc.backward(x, Wg, W1, b1, W2, b2, fwd, dy, alpha, beta, g_aux, g_z, Ws1, bs1, Ws2, bs2)

    def close(a, b, what):
        scale = max(np.abs(b).max(), 1e-30)
        assert np.abs(a - b).max() <= 1e-12 * scale, what

    dw = orc.combine_backward(dy, fwd.y_perm, fwd.slot_of)
    close(dw, full["dw"], "dw")
    close(orc.gate_backward(x, fwd, dw, alpha, beta, g_aux, g_z), full["dWg"], "dWg")
    for e in range(N):
        g = orc.expert_backward(x, fwd, e, W1[e], b1[e], W2[e], b2[e], dy)
        for k in ("dW1", "db1", "dW2", "db2"):
            close(g[k], full[k][e], f"{k}[{e}]")
    g = orc.expert_backward(x, fwd, -1, Ws1, bs1, Ws2, bs2, dy)
    for k, ks in (("dW1", "dWs1"), ("db1", "dbs1"), ("dW2", "dWs2"), ("db2", "dbs2")):
        close(g[k], full[ks], f"shared {k}")


def pin_health(orc):
    """Router health statistics: entropy vs scipy.stats.entropy per token;
    equal logits give log N and a spread of 0 over equal loads; a closed-form
    two-level load; drop rate from the dispatch counts; mean weights vs
    numpy.bincount; max |logit| vs numpy."""
    import scipy.stats
    rng = np.random.default_rng(29)
    T, N, K = 40, 6, 2
    s = rng.standard_normal((T, N)) * 3
    idx, w, demand, _ = orc.route(s, K)
    C = 9
    kept = orc.dispatch(idx, N, C)[0]
    h, mw = orc.health(s, demand, kept, idx, w)
    p = scipy.special.softmax(s, axis=1)
    assert abs(h[2] - np.mean(scipy.stats.entropy(p, axis=1))) < 1e-12
    f = demand / (T * K)
    assert abs(h[0] - np.std(f)) < 1e-15
    assert abs(h[1] - (1 - kept.sum() / (T * K))) < 1e-15 and h[1] > 0
    assert abs(h[3] - np.abs(s).max()) == 0
    ref_mw = np.bincount(idx.ravel(), weights=w.ravel().astype(np.float64), minlength=N)
    ref_mw = np.where(demand > 0, ref_mw / np.maximum(demand, 1), 0.0)
    assert np.allclose(mw, ref_mw, rtol=1e-15, atol=1e-15)
    # equal logits: entropy log N, every token on experts 0..K-1
    s0 = np.full((8, 4), 1.5)
    idx0, w0, d0, _ = orc.route(s0, 2)
    h0, _ = orc.health(s0, d0, d0, idx0, w0)
    assert abs(h0[2] - math.log(4)) < 1e-14 and h0[1] == 0.0
    # loads (1/2, 1/2, 0, 0) -> std 1/4
    assert abs(h0[0] - 0.25) < 1e-15


ALL_PINS = [
    pin_bf16_round, pin_gelu, pin_capacity, pin_gate_exact, pin_route_bruteforce,
    pin_route_closed_forms, pin_worked_example, pin_dispatch_bruteforce,
    pin_permutation_roundtrip, pin_dense_special_case, pin_identical_experts, pin_fp8_decode,
    pin_fp8_experts, pin_backward_autograd, pin_backward_token_mask, pin_backward_pieces, pin_health,
    pin_token_major, pin_soft_router, pin_drops_and_shared, pin_aux, pin_z_loss,
    pin_dispatch_rank_major, pin_aux_kl, pin_int4_dequant, pin_int4_experts,
]
