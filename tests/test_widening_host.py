"""The quantised GEMM's widening arithmetic, restated on the host.

The channel-major quantised kernel turns weight codes into bf16 with a few
integer operations and one or two packed bf16 operations per pair of codes.
These tests restate those steps bit by bit in numpy (they share no code with
the kernel) and check them, for every code, against independent decoders:
torch's float8_e4m3fn for FP8 and the oracle's INT4 dequantisation for INT4
(itself pinned to torch's float32 product rounded to bfloat16). The GPU parity
tests then check the kernel against the oracle end to end.
"""

import numpy as np
import torch


def _bf16_value(bits):
    """bf16 bit patterns (uint16 array) -> float64 values (exact)."""
    b = np.asarray(bits, dtype=np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def _prmt_sign_replicating(word, sel):
    """PTX prmt.b32 d, a, 0, sel (default mode) on one 32-bit word: result
    byte i takes byte (sel >> 4i) & 7 of {a, 0} (a is bytes 0-3), or, when
    bit 3 of that nibble is set, that byte's top bit replicated over 8 bits."""
    src = [(word >> (8 * k)) & 0xFF for k in range(4)] + [0, 0, 0, 0]
    out = 0
    for i in range(4):
        nib = (sel >> (4 * i)) & 0xF
        byte = src[nib & 7]
        if nib & 8:
            byte = 0xFF if byte & 0x80 else 0x00
        out |= byte << (8 * i)
    return out


def test_e4m3_widening_every_code():
    """Two codes per step: a sign-replicating byte select puts code k of the
    pair in the low bits of its 16-bit half with copies of its sign above;
    shifting left by 4 and masking with 0x87F0 per half gives the bf16 pattern
    sign | (E, M) << 4 = the E4M3 value times 2^-120, and one bf16 multiply by
    2^120 (exact) gives the value, for normal and subnormal codes alike."""
    codes = [c for c in range(256) if c not in (0x7F, 0xFF)]  # the two NaN codes are unsupported
    want = torch.tensor(codes, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    k120 = _bf16_value(np.array([0x7B80], np.uint16))[0]
    assert k120 == 2.0 ** 120
    got = []
    for c in codes:
        # the code as byte 0 (selector 0x9180, low half) and as byte 2 (0xB3A2, low half)
        for word, sel in ((c, 0x9180), (c << 16, 0xB3A2)):
            t = _prmt_sign_replicating(word, sel)
            pat = ((t << 4) & 0x87F087F0) & 0xFFFF
            got_v = _bf16_value(np.array([pat], np.uint16))[0] * k120
            got.append(got_v)
    got = np.array(got).reshape(-1, 2)
    assert np.array_equal(got[:, 0], want) and np.array_equal(got[:, 1], want)


def test_e4m3_widening_high_half():
    """The second code of each pair lands in the high half (byte 1 with
    selector 0x9180, byte 3 with 0xB3A2), and nothing of the low half leaks
    into it through the shift."""
    rng = np.random.default_rng(3)
    ok = [c for c in range(256) if c not in (0x7F, 0xFF)]
    for _ in range(200):
        b = rng.choice(ok, size=4)
        word = int(b[0]) | int(b[1]) << 8 | int(b[2]) << 16 | int(b[3]) << 24
        dec = torch.tensor(b.astype(np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()
        for sel, (lo, hi) in ((0x9180, (0, 1)), (0xB3A2, (2, 3))):
            pat = (_prmt_sign_replicating(word, sel) << 4) & 0x87F087F0
            v = _bf16_value(np.array([pat & 0xFFFF, pat >> 16], np.uint16)) * 2.0 ** 120
            assert v[0] == dec[lo] and v[1] == dec[hi]


def _bf16_round(x):
    return torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).to(torch.float64).numpy()


def test_int4_widening_every_code_and_position(orc):
    """Eight codes per 32-bit word: (w >> 4j) & 0x000F000F | 0x43004300 is the
    pair (columns 2j, 2j + 1 of the word's run) as the bf16 values 128 + c;
    subtracting 136 is exact and one bf16 multiply by the scale rounds once,
    which is the oracle's dequantised weight for every code, position and a
    spread of scales."""
    scales = torch.tensor([1.0, 1.0078125, 0.3359375, 3.0e-3, -0.75, 117.0], dtype=torch.bfloat16)
    rng = np.random.default_rng(11)
    words = [int(w) for w in rng.integers(0, 2 ** 32, size=64, dtype=np.uint64)]
    words += [0x76543210, 0xFEDCBA98, 0x00000000, 0xFFFFFFFF]
    for sb in scales:
        sbits = int(sb.view(torch.int16).item()) & 0xFFFF
        s = float(sb.to(torch.float64))
        for w in words:
            for j in range(4):
                t = ((w >> (4 * j)) & 0x000F000F) | 0x43004300
                halves = _bf16_value(np.array([t & 0xFFFF, t >> 16], np.uint16))
                cm8 = halves - 136.0                      # exact: c - 8
                got = _bf16_round(cm8 * s)                 # exact product, one rounding
                # the layout: column 2j of the run in nibble j, column 2j + 1 in nibble j + 4
                c_lo, c_hi = (w >> (4 * j)) & 15, (w >> (16 + 4 * j)) & 15
                want = [orc.int4_dequant(c_lo, sbits), orc.int4_dequant(c_hi, sbits)]
                assert got.tolist() == want, (hex(w), j, s)


def test_int4_widening_follows_the_packed_layout(orc):
    """Codes packed by the input generator's int4_pack come out of the
    widening step in column order: pair j of a word is columns 2j and 2j + 1
    of its run of eight."""
    from top_routing_expert_then_b300.inputs import int4_pack
    rng = np.random.default_rng(17)
    codes = rng.integers(0, 16, size=(32, 8)).astype(np.int32)
    packed = int4_pack(torch.from_numpy(codes)).numpy()  # [32, 4] bytes
    sbits = int(torch.tensor(0.3359375, dtype=torch.bfloat16).view(torch.int16).item()) & 0xFFFF
    s = 0.3359375
    for run, b in zip(codes, packed):
        w = int.from_bytes(bytes(b.tolist()), "little")
        for j in range(4):
            t = ((w >> (4 * j)) & 0x000F000F) | 0x43004300
            got = _bf16_round((_bf16_value(np.array([t & 0xFFFF, t >> 16], np.uint16)) - 136.0) * s)
            want = [orc.int4_dequant(int(run[2 * j]), sbits), orc.int4_dequant(int(run[2 * j + 1]), sbits)]
            assert got.tolist() == want, (run.tolist(), j)
