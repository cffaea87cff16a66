"""Pins for the oracle's INT4 group-32 variant with fp16 group scales (2/3/5/6-bit article §2.1 costs an fp16 scale
per 32 weights at 0.5 bpw; the quantization rule is the DBHOO-CIM INT4 article's, §3.1, with the scale stored in
fp16 and used rounded). Exact lattices, clamp and zero cases, the range flag, byte accounting and round trips."""
import numpy as np
import pytest
from conftest import read_golden

RULE = {r[0]: r[1] for r in read_golden("int4_rule.txt")}


def lattice(rng, n_groups):
    """w = s * t, s a power of two inside fp16's normal range, t in [-8, 7] with -8 present: max|w| / 8 = s exactly,
    fp16(s) = s, and w / s = t exactly."""
    t = rng.integers(-8, 8, (n_groups, 32))
    t[np.arange(n_groups), rng.integers(0, 32, n_groups)] = -8
    s = np.exp2(rng.integers(-14, 12, n_groups)).astype(np.float32)
    return (t * s[:, None]).astype(np.float32), t, s


def test_lattice_is_reproduced_exactly(orc):
    rng = np.random.default_rng(31)
    w, t, s = lattice(rng, 48 * 8)
    W = w.reshape(48, 256)
    parts = orc.quantize(orc.Q4G32H, W)
    assert parts["flags"] == 0
    assert np.array_equal(parts["q"].reshape(-1, 32), t)
    assert np.array_equal(parts["d"].reshape(-1), s.astype(np.float16).view(np.uint16))
    packed, gs = orc.pack(orc.Q4G32H, 48, 256, parts)
    assert gs.dtype == np.uint16
    assert np.array_equal(orc.dequant(orc.Q4G32H, 48, 256, packed, gs), W)


def test_positive_extreme_clamps_to_7_and_codes_match_q4g32(orc):
    """A group whose max is positive (w = 8 s) gives 8 -> clamped to 7; with power-of-two scales the codes and the
    packed bytes are those of the fp32-scale format (same rule, same nibbles)."""
    rng = np.random.default_rng(32)
    w, t, s = lattice(rng, 64)
    w = -w                                               # the extreme is now +8 s
    W = w.reshape(8, 256)
    ph = orc.quantize(orc.Q4G32H, W)
    pf = orc.quantize(orc.Q4G32, W)
    assert np.array_equal(ph["q"], pf["q"])
    assert np.array_equal(ph["q"].reshape(-1, 32), np.minimum(-t, 7))
    a, _ = orc.pack(orc.Q4G32H, 8, 256, ph)
    b, _ = orc.pack(orc.Q4G32, 8, 256, pf)
    assert np.array_equal(a, b)


def test_zero_tiny_and_overflowing_groups(orc):
    W = np.zeros((1, 96), np.float32)
    W[0, 32:64] = 1e-9                                   # max/8 rounds to fp16 zero: zero codes, zero scale
    W[0, 64] = 1e6                                       # max/8 = 125000 overflows fp16: RANGE flag
    parts = orc.quantize(orc.Q4G32H, W)
    assert parts["flags"] == 1
    d = parts["d"].reshape(-1)
    assert d[0] == 0 and d[1] == 0 and (d[2] & 0x7FFF) == 0x7C00
    assert not parts["q"][0, :64].any()


def test_rounding_is_half_to_even_against_the_rounded_scale(orc):
    """The codes use the fp16-rounded scale D: w = (k + 1/2) D ties round to even."""
    D = np.float32(2.0 ** -6)
    w = np.zeros((1, 32), np.float32)
    w[0, 0] = -8 * D                                     # sets s = D exactly
    w[0, 1:7] = np.array([0.5, 1.5, 2.5, -0.5, -1.5, 6.5], np.float32) * D
    q = orc.quantize(orc.Q4G32H, w)["q"][0]
    assert list(q[:7]) == [-8, 0, 2, 2, 0, -2, 6]


def test_error_bound(orc):
    """|w - w'| <= D / 2 inside the code range, where D = fp16(max|w| / 8); the positive extreme may clamp, which
    costs at most D / 2 + (8 s - 7.5 D)."""
    rng = np.random.default_rng(33)
    W = (rng.standard_normal((64, 1024)) * np.exp(rng.uniform(-6, 3, (64, 1)))).astype(np.float32)
    parts = orc.quantize(orc.Q4G32H, W)
    packed, gs = orc.pack(orc.Q4G32H, 64, 1024, parts)
    deq = orc.dequant(orc.Q4G32H, 64, 1024, packed, gs).astype(np.float64)
    D = parts["d"].view(np.float16).astype(np.float64).repeat(32, axis=1)
    amax = np.abs(W.astype(np.float64)).reshape(64, 32, 32).max(axis=2).repeat(32, axis=1)
    bound = D / 2 + np.maximum(0.0, amax - 7.5 * D)
    assert np.all(np.abs(deq - W) <= bound * (1 + 1e-12))


def test_byte_accounting(orc):
    assert float(RULE["FP16_SCALE_BPW_G32"]) == 16 / 32
    lay = orc.layout(orc.Q4G32H, 128, 4096)
    bpw = 8 * (lay["packed_bytes"] + lay["scale_bytes"]) / (128 * 4096)
    assert bpw == 4.0 + float(RULE["FP16_SCALE_BPW_G32"])
    assert lay["scale_stride"] * 2 % 16 == 0
    # scale rows are padded to 16 bytes: K = 96 has 3 groups, stored in a row of 8
    assert orc.layout(orc.Q4G32H, 1, 96)["scale_stride"] == 8


def test_pack_unpack_round_trip(orc):
    rng = np.random.default_rng(34)
    N, K = 61, 32 * 512                                  # ~1M codes
    parts = dict(q=rng.integers(-8, 8, (N, K)).astype(np.int8), gscale=None, sub_scale=None, sub_min=None,
                 d=rng.integers(0, 0x7C00, (N, K // 32)).astype(np.uint16), dmin=None)
    packed, gs = orc.pack(orc.Q4G32H, N, K, parts)
    back = orc.unpack(orc.Q4G32H, N, K, packed, gs)
    assert np.array_equal(back["q"], parts["q"])
    assert np.array_equal(back["d"], parts["d"])
