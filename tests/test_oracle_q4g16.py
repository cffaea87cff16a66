"""Pins for the oracle's INT4 variant with groups of 16 (DBHOO-CIM INT4 article, pwwt.cn/news/4452170, §5.1: for a
model with many outlier weights, change the group size from 32 to 16; the rule is that article's §3.1 with fp32
scales, §4.1). Exact lattices, the clamp and floor edges, agreement with group 32 where it must agree, the error
bound, byte accounting and a round trip."""
import numpy as np
from conftest import read_golden

RULE = {r[0]: r[1] for r in read_golden("int4_rule.txt")}
FLOOR = np.float32(float(RULE["SCALE_FLOOR"]))


def lattice(rng, n_groups):
    t = rng.integers(-8, 8, (n_groups, 16))
    t[np.arange(n_groups), rng.integers(0, 16, n_groups)] = -8
    s = np.exp2(rng.integers(-20, 4, n_groups)).astype(np.float32)
    return (t * s[:, None]).astype(np.float32), t, s


def test_lattice_is_reproduced_exactly(orc):
    rng = np.random.default_rng(41)
    w, t, s = lattice(rng, 32 * 16)
    W = w.reshape(32, 256)
    parts = orc.quantize(orc.Q4G16, W)
    assert np.array_equal(parts["q"].reshape(-1, 16), t)
    assert np.array_equal(parts["gscale"].reshape(-1), s)
    packed, gs = orc.pack(orc.Q4G16, 32, 256, parts)
    assert np.array_equal(orc.dequant(orc.Q4G16, 32, 256, packed, gs), W)


def test_agrees_with_group_32_when_both_halves_share_a_max(orc):
    """If both 16-weight halves of every 32-group reach the same max |w|, the two rules give the same scale for
    every weight, hence identical codes and identical packed code bytes."""
    rng = np.random.default_rng(42)
    W = rng.standard_normal((8, 512)).astype(np.float32)
    g = W.reshape(8, 16, 2, 16)
    m = np.abs(g).max(axis=(2, 3), keepdims=True)
    g[:, :, 0, 0] = m[:, :, 0, 0]
    g[:, :, 1, 0] = -m[:, :, 0, 0]
    W = g.reshape(8, 512)
    a, b = orc.quantize(orc.Q4G16, W), orc.quantize(orc.Q4G32, W)
    assert np.array_equal(a["q"], b["q"])
    assert np.array_equal(a["gscale"][:, ::2], b["gscale"])
    assert np.array_equal(orc.pack(orc.Q4G16, 8, 512, a)[0], orc.pack(orc.Q4G32, 8, 512, b)[0])


def test_clamp_floor_and_zero(orc):
    W = np.zeros((1, 64), np.float32)
    W[0, 0:16] = np.linspace(-1.0, 1.0, 16, dtype=np.float32)      # max positive: +8 s -> clamped to 7
    W[0, 16:32] = 1e-20                                               # max/8 below the floor
    parts = orc.quantize(orc.Q4G16, W)
    s = parts["gscale"][0]
    assert s[0] == np.float32(1.0) / np.float32(8.0) and parts["q"][0, 15] == 7 and parts["q"][0, 0] == -8
    assert s[1] == FLOOR and not parts["q"][0, 16:32].any()
    assert s[2] == FLOOR and s[3] == FLOOR and not parts["q"][0, 32:].any()


def test_error_bound(orc):
    rng = np.random.default_rng(43)
    W = (rng.standard_normal((32, 1024)) * np.exp(rng.uniform(-6, 3, (32, 1)))).astype(np.float32)
    W[rng.random(W.shape) < 0.003] *= 40.0                            # outliers
    parts = orc.quantize(orc.Q4G16, W)
    packed, gs = orc.pack(orc.Q4G16, 32, 1024, parts)
    deq = orc.dequant(orc.Q4G16, 32, 1024, packed, gs).astype(np.float64)
    s = parts["gscale"].astype(np.float64).repeat(16, axis=1)
    clamped = W / s > 7.5                               # positive codes past 7.5 clamp to 7: at most s off
    bound = np.where(clamped, s, s / 2) * (1 + 1e-6)
    assert np.all(np.abs(deq - W) <= bound)
    # the point of §5.1: on outlier-heavy weights group 16 has the smaller error
    p32 = orc.quantize(orc.Q4G32, W)
    pk, g32 = orc.pack(orc.Q4G32, 32, 1024, p32)
    e32 = np.abs(orc.dequant(orc.Q4G32, 32, 1024, pk, g32) - W).mean()
    assert np.abs(deq - W).mean() < e32


def test_byte_accounting(orc):
    lay = orc.layout(orc.Q4G16, 64, 4096)
    assert 8 * (lay["packed_bytes"] + lay["scale_bytes"]) / (64 * 4096) == 4.0 + 32 / 16
    assert orc.layout(orc.Q4G16, 1, 96)["scale_stride"] == 8          # 6 groups, rows padded to 16 bytes


def test_pack_unpack_round_trip(orc):
    rng = np.random.default_rng(44)
    N, K = 61, 32 * 512
    parts = dict(q=rng.integers(-8, 8, (N, K)).astype(np.int8),
                 gscale=rng.standard_normal((N, K // 16)).astype(np.float32),
                 sub_scale=None, sub_min=None, d=None, dmin=None)
    packed, gs = orc.pack(orc.Q4G16, N, K, parts)
    back = orc.unpack(orc.Q4G16, N, K, packed, gs)
    assert np.array_equal(back["q"], parts["q"])
    assert np.array_equal(back["gscale"].view(np.uint32), parts["gscale"].view(np.uint32))
