"""Seeded synthetic inputs for the MoE layer forward pass.

This module is shared by the CUDA path's callers and by the CPU oracle's
tests. It holds none of the layer's arithmetic: it only names the workload
shapes and draws random tensors for them. Everything here is plain torch RNG
on a caller-chosen device with a seeded generator, so a (config, seed, device)
triple always produces the same bytes.

Value recipe (the workloads of the MoE pages: Mixtral-shaped and
DeepSeek-V3-shaped layers, a tiny layer and a skewed fine-grained layer):

* ``x``  = randint(-128, 128 inclusive) / 64, stored bf16 (exact): multiples
  of 1/64 uniform in [-2, 2].
* ``Wg`` = randint(-8, 8 inclusive) / 64, stored bf16 (exact): multiples of
  1/64 in [-0.125, 0.125]. Layout ``[N, d_model]`` (nn.Linear ``[out, in]``).
  With these grids every gate logit is a multiple of 2^-12 of magnitude
  below 2^11, so any fp32 or fp64 summation order gives the same logit.
* Expert weights ``W1 [N, d_ff, d_model]``, ``W2 [N, d_model, d_ff]`` drawn
  N(0, 1/fan_in) and rounded to bf16 (torch's RNE cast); biases N(0, 0.02^2)
  in fp32.
* Skewed routing: expert e's gate row gets an additive Zipf(s=1.2) offset
  ``round(16 * (e+1)^-1.2) / 64`` on every entry. It stays on the 1/64 grid
  (|W_g| <= 0.375, so logits stay exact multiples of 2^-12 below 2^12) and
  makes experts 0 and 1 hot: about 9x and 3x the mean demand at
  T=8192, N=64, K=2.
* Aux-loss-free selection bias ``b_i`` ~ U(-0.05, 0.05) rounded to a multiple
  of 2^-12 (so ``s + b`` stays exact in fp32), fp32.
* Shared expert weights drawn like the routed ones.
"""

from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Dict, Optional

import torch


@dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int
    d_model: int
    d_ff: int
    N: int
    K: int
    capacity_factor: float  # <= 0 means dropless (capacity = T)
    has_shared: bool = False
    sel_bias: bool = False
    zipf: bool = False
    aux_alpha: float = 0.01
    z_beta: float = 1e-3
    rank_major: bool = False   # capacity priority: earlier ranks first instead of earlier tokens
    kl_coef: float = 0.02      # KL-to-uniform balance-loss variant
    weights: str = "bf16"      # expert weight format: "bf16", "fp8_e4m3" (per-output-channel scales)
                               # or "int4_g128" (4-bit codes, a bf16 scale per 128 reduction columns)
    note: str = ""

    def with_(self, **kw) -> "MoEConfig":
        return replace(self, **kw)


# The named workloads. capacity_factor <= 0 encodes "dropless" (capacity = T).
CONFIGS: Dict[str, MoEConfig] = {
    "tiny": MoEConfig("tiny", 256, 128, 256, 8, 2, 1.25,
                      note="tiny layer, top-2 of 8, capacity factor 1.25"),
    "mixtral_prefill": MoEConfig("mixtral_prefill", 4096, 4096, 14336, 8, 2, 0.0,
                                 note="Mixtral-shaped prefill, dropless"),
    "mixtral_prefill_cf125": MoEConfig("mixtral_prefill_cf125", 4096, 4096, 14336, 8, 2, 1.25,
                                       note="Mixtral-shaped prefill, capacity factor 1.25"),
    "mixtral_decode16": MoEConfig("mixtral_decode16", 16, 4096, 14336, 8, 2, 0.0,
                                  note="Mixtral-shaped decode, 16 tokens, dropless"),
    "mixtral_decode64": MoEConfig("mixtral_decode64", 64, 4096, 14336, 8, 2, 0.0,
                                  note="Mixtral-shaped decode, 64 tokens, dropless"),
    "skewed": MoEConfig("skewed", 8192, 2048, 1408, 64, 2, 1.0, zipf=True,
                        note="fine-grained 64 experts, Zipf-skewed gate, capacity factor 1.0"),
    "dsv3": MoEConfig("dsv3", 4096, 7168, 2048, 256, 8, 0.0, has_shared=True, sel_bias=True,
                      note="DeepSeek-V3-shaped: 256 routed + 1 shared expert, top-8, selection bias"),
    # a slice of the DeepSeek-V3-shaped layer for profiling: 16 routed experts
    # of the same shape and the same 128 rows per expert on average (2 GB of
    # weights instead of 15)
    "dsv3_slice16": MoEConfig("dsv3_slice16", 256, 7168, 2048, 16, 8, 0.0, has_shared=True, sel_bias=True,
                              note="16 experts of the DeepSeek-V3 shape, 128 rows per expert"),
    # a larger slice (64 experts, 128 rows each) whose GEMMs run several waves of tiles
    "dsv3_slice64": MoEConfig("dsv3_slice64", 1024, 7168, 2048, 64, 8, 0.0, has_shared=True, sel_bias=True,
                              note="64 experts of the DeepSeek-V3 shape, 128 rows per expert"),
    "mixtral_decode16_fp8": MoEConfig("mixtral_decode16_fp8", 16, 4096, 14336, 8, 2, 0.0, weights="fp8_e4m3",
                                      note="Mixtral-shaped decode, 16 tokens, FP8 E4M3 expert weights"),
    "mixtral_decode16_int4": MoEConfig("mixtral_decode16_int4", 16, 4096, 14336, 8, 2, 0.0, weights="int4_g128",
                                       note="Mixtral-shaped decode, 16 tokens, INT4 group-wise expert weights"),
    "mixtral_decode64_int4": MoEConfig("mixtral_decode64_int4", 64, 4096, 14336, 8, 2, 0.0, weights="int4_g128",
                                       note="Mixtral-shaped decode, 64 tokens, INT4 group-wise expert weights"),
    "mixtral_decode64_fp8": MoEConfig("mixtral_decode64_fp8", 64, 4096, 14336, 8, 2, 0.0, weights="fp8_e4m3",
                                      note="Mixtral-shaped decode, 64 tokens, FP8 E4M3 expert weights"),
}


@dataclass
class MoEInputs:
    cfg: MoEConfig
    x: torch.Tensor            # [T, d] bf16
    Wg: torch.Tensor           # [N, d] bf16
    W1: torch.Tensor           # [N, f, d] bf16
    b1: torch.Tensor           # [N, f] fp32
    W2: torch.Tensor           # [N, d, f] bf16
    b2: torch.Tensor           # [N, d] fp32
    sel_bias: Optional[torch.Tensor] = None  # [N] fp32
    Ws1: Optional[torch.Tensor] = None       # [f, d] bf16
    bs1: Optional[torch.Tensor] = None       # [f] fp32
    Ws2: Optional[torch.Tensor] = None       # [d, f] bf16
    bs2: Optional[torch.Tensor] = None       # [d] fp32
    extra: Dict[str, torch.Tensor] = field(default_factory=dict)
    quant: Optional["QuantWeights"] = None   # quantised expert weights (cfg.weights != "bf16")

    def to(self, device) -> "MoEInputs":
        def mv(t):
            return None if t is None else t.to(device)
        return MoEInputs(self.cfg, mv(self.x), mv(self.Wg), mv(self.W1), mv(self.b1),
                         mv(self.W2), mv(self.b2), mv(self.sel_bias), mv(self.Ws1),
                         mv(self.bs1), mv(self.Ws2), mv(self.bs2),
                         {k: mv(v) for k, v in self.extra.items()},
                         None if self.quant is None else self.quant.to(device))


@dataclass
class QuantWeights:
    """Quantised expert weights.

    format "fp8_e4m3": uint8 E4M3 codes in nn.Linear layout and one fp32 scale
    per output channel (dequantised weight = code value * scale):
    W1q [N, f, d], s1 [N, f], W2q [N, d, f], s2 [N, d] (shared: [f, d], [f],
    [d, f], [d]).
    format "int4_g128": 4-bit codes, eight consecutive reduction columns
    8m .. 8m + 7 of a row in one little-endian 32-bit word (bytes 4m .. 4m + 3
    of the row), column 8m + 2j in bits 4j .. 4j + 3 and column 8m + 2j + 1 in
    bits 16 + 4j .. 19 + 4j (code c stands for c - 8), and one bf16 scale per
    output channel and group of 128 reduction columns, stored group-major
    (dequantised weight = bf16(RNE) of (c - 8) * scale):
    W1q [N, f, d / 2], s1 [N, d / 128, f], W2q [N, d, f / 2], s2 [N, f / 128, d]
    (shared: [f, d / 2], [d / 128, f], [d, f / 2], [f / 128, d])."""
    W1q: torch.Tensor
    s1: torch.Tensor
    W2q: torch.Tensor
    s2: torch.Tensor
    Ws1q: Optional[torch.Tensor] = None
    ss1: Optional[torch.Tensor] = None
    Ws2q: Optional[torch.Tensor] = None
    ss2: Optional[torch.Tensor] = None
    format: str = "fp8_e4m3"

    def to(self, device) -> "QuantWeights":
        def mv(t):
            return None if t is None else t.to(device)
        return QuantWeights(mv(self.W1q), mv(self.s1), mv(self.W2q), mv(self.s2), mv(self.Ws1q),
                            mv(self.ss1), mv(self.Ws2q), mv(self.ss2), self.format)


FP8_E4M3_MAX = 448.0


def fp8_codes(W: torch.Tensor):
    """Synthetic FP8 weights for a stack of nn.Linear matrices [..., out, in]:
    one fp32 scale per output row mapping the row's largest magnitude to 448,
    codes = torch's float8_e4m3fn cast of W / scale. (Data preparation only:
    calibrated quantisers need real data and are not part of this package.)"""
    w = W.to(torch.float32)
    amax = w.abs().amax(dim=-1).clamp_min(1e-30)
    scale = (amax / FP8_E4M3_MAX).to(torch.float32)
    q = (w / scale[..., None]).to(torch.float8_e4m3fn).view(torch.uint8)
    return q.contiguous(), scale.contiguous()


INT4_GROUP = 128


def int4_codes(W: torch.Tensor):
    """Synthetic INT4 group-wise weights for a stack of nn.Linear matrices
    [..., out, in] (in a multiple of 128): per output row and group of 128
    reduction columns, scale = bf16(largest magnitude / 7) and code = clamp(
    round(W / scale), -8, 7) + 8, packed eight to a 32-bit word as
    `int4_pack` says; scales returned group-major [..., in / 128, out]. (Data
    preparation only: calibrated quantisers need real data.)"""
    w = W.to(torch.float32)
    *lead, out, inn = w.shape
    g = w.reshape(*lead, out, inn // INT4_GROUP, INT4_GROUP)
    scale = (g.abs().amax(dim=-1).clamp_min(1e-30) / 7.0).to(torch.bfloat16)
    q = torch.round(g / scale.to(torch.float32)[..., None]).clamp(-8, 7).to(torch.int32) + 8
    return int4_pack(q.reshape(*lead, out, inn)), scale.transpose(-1, -2).contiguous()


def int4_pack(codes: torch.Tensor) -> torch.Tensor:
    """Pack 4-bit codes [..., in] (in a multiple of 8, values 0..15) into the
    int4_g128 byte layout [..., in / 2]: columns 8m .. 8m + 7 form one
    little-endian 32-bit word whose bits 4j .. 4j + 3 hold column 8m + 2j and
    bits 16 + 4j .. 19 + 4j hold column 8m + 2j + 1 (j = 0 .. 3), so that
    (word >> 4j) & 0x000F000F is the pair (2j, 2j + 1) in two 16-bit halves."""
    q = codes.to(torch.int32)
    *lead, inn = q.shape
    g = q.reshape(*lead, inn // 8, 8)
    # byte b of the word: bits 8b .. 8b + 7, i.e. nibbles 2b (low) and 2b + 1
    word_bytes = [g[..., 0] | (g[..., 2] << 4), g[..., 4] | (g[..., 6] << 4),
                  g[..., 1] | (g[..., 3] << 4), g[..., 5] | (g[..., 7] << 4)]
    return torch.stack(word_bytes, dim=-1).to(torch.uint8).reshape(*lead, inn // 2).contiguous()


ZIPF_AMPLITUDE_64THS = 16
ZIPF_S = 1.2


def zipf_offsets_64ths(N: int) -> torch.Tensor:
    """Per-expert integer offsets (in units of 1/64) for the skewed gate."""
    e = torch.arange(1, N + 1, dtype=torch.float64)
    return torch.round(ZIPF_AMPLITUDE_64THS * e.pow(-ZIPF_S)).to(torch.int64)


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn_bf16(shape, std: float, g, device, chunk_rows: int = 1024) -> torch.Tensor:
    """N(0, std^2) rounded to bf16, drawn chunk by chunk to bound fp32 scratch."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1, shape[-1])
    for r0 in range(0, flat.shape[0], chunk_rows):
        r1 = min(flat.shape[0], r0 + chunk_rows)
        tmp = torch.randn((r1 - r0, shape[-1]), generator=g, device=device, dtype=torch.float32)
        flat[r0:r1] = (tmp * std).to(torch.bfloat16)
    return out


def make_inputs(cfg: MoEConfig | str, seed: int = 0, device="cpu") -> MoEInputs:
    """Draw every input of one MoE layer forward for ``cfg`` on ``device``."""
    if isinstance(cfg, str):
        cfg = CONFIGS[cfg]
    device = torch.device(device)
    g = _gen(device, seed)
    T, d, f, N = cfg.T, cfg.d_model, cfg.d_ff, cfg.N

    x = (torch.randint(-128, 129, (T, d), generator=g, device=device, dtype=torch.int32)
         .to(torch.float32) / 64).to(torch.bfloat16)
    wg_int = torch.randint(-8, 9, (N, d), generator=g, device=device, dtype=torch.int32)
    if cfg.zipf:
        wg_int = wg_int + zipf_offsets_64ths(N).to(device=device, dtype=torch.int32)[:, None]
    Wg = (wg_int.to(torch.float32) / 64).to(torch.bfloat16)

    W1 = _randn_bf16((N, f, d), d ** -0.5, g, device)
    b1 = torch.randn((N, f), generator=g, device=device, dtype=torch.float32) * 0.02
    W2 = _randn_bf16((N, d, f), f ** -0.5, g, device)
    b2 = torch.randn((N, d), generator=g, device=device, dtype=torch.float32) * 0.02

    sel_bias = None
    if cfg.sel_bias:
        u = torch.rand((N,), generator=g, device=device, dtype=torch.float64) * 0.1 - 0.05
        sel_bias = (torch.round(u * 4096) / 4096).to(torch.float32)

    Ws1 = bs1 = Ws2 = bs2 = None
    if cfg.has_shared:
        Ws1 = _randn_bf16((f, d), d ** -0.5, g, device)
        bs1 = torch.randn((f,), generator=g, device=device, dtype=torch.float32) * 0.02
        Ws2 = _randn_bf16((d, f), f ** -0.5, g, device)
        bs2 = torch.randn((d,), generator=g, device=device, dtype=torch.float32) * 0.02

    quant = None
    if cfg.weights == "int4_g128":
        W1q, s1 = int4_codes(W1)
        W2q, s2 = int4_codes(W2)
        quant = QuantWeights(W1q, s1, W2q, s2, format="int4_g128")
        if cfg.has_shared:
            quant.Ws1q, quant.ss1 = int4_codes(Ws1)
            quant.Ws2q, quant.ss2 = int4_codes(Ws2)
    if cfg.weights == "fp8_e4m3":
        W1q, s1 = fp8_codes(W1)
        W2q, s2 = fp8_codes(W2)
        quant = QuantWeights(W1q, s1, W2q, s2)
        if cfg.has_shared:
            quant.Ws1q, quant.ss1 = fp8_codes(Ws1)
            quant.Ws2q, quant.ss2 = fp8_codes(Ws2)
    elif cfg.weights not in ("bf16", "int4_g128"):
        raise ValueError(f"unknown weight format {cfg.weights!r}")

    return MoEInputs(cfg, x, Wg, W1, b1, W2, b2, sel_bias, Ws1, bs1, Ws2, bs2, quant=quant)


def make_x(cfg: MoEConfig, seed: int, device="cpu") -> torch.Tensor:
    """A fresh batch of tokens on the 1/64 grid (used for multi-batch runs)."""
    g = _gen(torch.device(device), seed)
    return (torch.randint(-128, 129, (cfg.T, cfg.d_model), generator=g, device=device,
                          dtype=torch.int32).to(torch.float32) / 64).to(torch.bfloat16)


def make_dy(cfg: MoEConfig, seed: int, device="cpu") -> torch.Tensor:
    """A seeded upstream gradient for the layer output: N(0, 1) rounded to bf16."""
    g = _gen(torch.device(device), seed + 1000)
    return torch.randn((cfg.T, cfg.d_model), generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
