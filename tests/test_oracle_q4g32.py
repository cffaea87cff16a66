"""Pins for the oracle's INT4 symmetric group-32 path (DBHOO-CIM INT4 article, pwwt.cn/news/4452170,
§2.1, §3.1, §3.2, §4.1) — built from exact lattices and closed forms, never from the oracle itself."""
import numpy as np
import pytest
from conftest import read_golden

RULE = {r[0]: r[1] for r in read_golden("int4_rule.txt")}
G = int(RULE["GROUP"])
QMIN, QMAX = int(RULE["QMIN"]), int(RULE["QMAX"])
DIV = float(RULE["DIVISOR"])
FLOOR = np.float32(float(RULE["SCALE_FLOOR"]))


def lattice(rng, n_groups, with_min=True):
    """Weights w = s * t with s a power of two and integer t in [-8, 7] containing -8 (the group's |w| max
    sits on the negative extreme, so max|w|/8 = s exactly and w/s = t exactly)."""
    t = rng.integers(QMIN, QMAX + 1, (n_groups, G))
    if with_min:
        t[np.arange(n_groups), rng.integers(0, G, n_groups)] = QMIN
    s = np.exp2(rng.integers(-20, 4, n_groups)).astype(np.float32)
    return (t * s[:, None]).astype(np.float32), t, s


def test_constants_match_page():
    assert (G, QMIN, QMAX, DIV) == (32, -8, 7, 8.0)
    assert int(RULE["BYTES_PER_GROUP_CODES"]) == G * 4 // 8


def test_lattice_is_reproduced_exactly(orc):
    rng = np.random.default_rng(10)
    w, t, s = lattice(rng, 64 * 8)
    W = w.reshape(64, 8 * G)
    parts = orc.quantize(orc.Q4G32, W)
    assert np.array_equal(parts["q"].reshape(-1, G), t)
    assert np.array_equal(parts["gscale"].reshape(-1), s)
    packed, gs = orc.pack(orc.Q4G32, 64, 8 * G, parts)
    deq = orc.dequant(orc.Q4G32, 64, 8 * G, packed, gs)
    assert np.array_equal(deq, W)


def test_positive_extreme_is_clamped_to_7(orc):
    # max |w| on a positive element: w/s = +8 must clamp to 7 ("-8..7, not -7..7", §3.1)
    w = np.zeros((1, G), np.float32)
    w[0, 0] = 2.0
    w[0, 1] = -1.0
    w[0, 2] = 0.5
    parts = orc.quantize(orc.Q4G32, w)
    assert parts["gscale"][0, 0] == np.float32(0.25)
    assert parts["q"][0, 0] == QMAX and parts["q"][0, 1] == -4 and parts["q"][0, 2] == 2
    # the clamped extreme's dequant error is one full scale, every other element's at most half a scale
    packed, gs = orc.pack(orc.Q4G32, 1, G, parts)
    deq = orc.dequant(orc.Q4G32, 1, G, packed, gs)
    assert deq[0, 0] == np.float32(1.75)


def test_zero_and_tiny_groups_use_the_floor(orc):
    w = np.zeros((1, 2 * G), np.float32)
    w[0, G:] = 1e-13
    parts = orc.quantize(orc.Q4G32, w)
    assert np.array_equal(parts["gscale"][0], np.array([FLOOR, FLOOR], np.float32))
    assert not parts["q"].any()


def test_round_half_to_even(orc):
    # s = 1 (max |w| = 8 on a negative element): w = k + 1/2 must round to the even neighbour (torch.round)
    w = np.zeros((1, G), np.float32)
    w[0, 0] = -8.0
    w[0, 1:7] = [0.5, 1.5, 2.5, -0.5, -1.5, -2.5]
    parts = orc.quantize(orc.Q4G32, w)
    assert list(parts["q"][0, :7]) == [-8, 0, 2, 2, 0, -2, -2]


def test_clamp_round_order_equivalence(orc):
    # §2.1 writes round(clamp(w/s)), §3.1 clamp(round(w/s)); both orders give the oracle's integers
    rng = np.random.default_rng(11)
    W = (rng.laplace(0, 0.02, (256, 32 * 32))).astype(np.float32)
    W[rng.random(W.shape) < 0.01] *= 40
    parts = orc.quantize(orc.Q4G32, W)
    s = np.repeat(parts["gscale"], G, axis=1)
    ratio = (W / s).astype(np.float32)
    a = np.rint(np.clip(ratio, QMIN, QMAX))
    b = np.clip(np.rint(ratio), QMIN, QMAX)
    assert np.array_equal(a, b)
    assert np.array_equal(parts["q"].astype(np.float64), b)


def test_nibble_order_closed_form(orc):
    # codes q_k = (k mod 16) - 8 -> stored u_k = k mod 16; byte j = u_2j + 16 * u_2j+1 (low nibble = even index)
    K = 4 * G
    q = ((np.arange(K) % 16) - 8).astype(np.int8)[None, :]
    parts = dict(q=q, gscale=np.ones((1, K // G), np.float32))
    packed, gs = orc.pack(orc.Q4G32, 1, K, parts)
    u = np.arange(K) % 16
    expect = (u[0::2] + 16 * u[1::2]).astype(np.uint8)
    assert np.array_equal(packed[0], expect)
    assert packed.shape[1] == K // 2
    back = orc.unpack(orc.Q4G32, 1, K, packed, gs)
    assert np.array_equal(back["q"], q)


def test_dequant_error_bound(orc):
    # §3.4 self-check of the 2/3/5/6-bit article: |w - w'| <= scale / 2 for in-range elements; the clamped
    # positive extreme (w/s in (7.5, 8]) may be off by up to one scale.
    rng = np.random.default_rng(12)
    W = rng.laplace(0, 0.02, (128, 1024)).astype(np.float32)
    packed, gs, _ = orc.quantize_pack(orc.Q4G32, W)
    deq = orc.dequant(orc.Q4G32, 128, 1024, packed, gs)
    s = np.repeat(gs[:, :1024 // G], G, axis=1).astype(np.float64)
    err = np.abs(W.astype(np.float64) - deq)
    in_range = (W / s) <= 7.5
    assert np.all(err[in_range] <= s[in_range] / 2 * (1 + 1e-6))
    assert np.all(err <= s * (1 + 1e-6))


def test_layout_bytes(orc):
    lay = orc.layout(orc.Q4G32, 4096, 4096)
    assert lay["row_stride"] == 2048 and lay["packed_bytes"] == 4096 * 2048
    assert lay["scale_stride"] == 128 and lay["scale_bytes"] == 4096 * 128 * 4
    assert (lay["packed_bytes"] + lay["scale_bytes"]) / (4096 * 4096) == 0.625
    # scale rows padded to 16 bytes; padding written as zero
    lay = orc.layout(orc.Q4G32, 3, 96)
    assert lay["scale_stride"] == 4
    W = np.ones((3, 96), np.float32)
    packed, gs, _ = orc.quantize_pack(orc.Q4G32, W)
    assert gs.shape == (3, 4) and not gs[:, 3].any()
    with pytest.raises(ValueError):
        orc.layout(orc.Q4G32, 3, 48)
