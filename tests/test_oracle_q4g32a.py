"""Pins for the oracle's asymmetric INT4 variant Q4G32A (DBHOO-CIM INT4 article, pwwt.cn/news/4452170, §5.1: a
layer whose weight maxima stand out is quantized asymmetrically; 2/3/5/6-bit article, lpnh.cn/news/2857666, §2.1:
q = rint(w / s) + z, w' = s (q - z)). Per group of 32: the range [min(0, min w), max(0, max w)] spread over 15
steps, an integer zero point z in 0..15, codes stored as unsigned nibbles, (s, z) kept as an fp32 pair.
Exact lattices, zero and one-sided groups, the error bound, the gain over the symmetric rule on one-sided groups,
byte accounting and a round trip."""
import numpy as np


def lattice(rng, n_groups):
    """w = s (u - z) with s a power of two, z in 0..15 and u in 0..15 with both 0 and 15 present: the group range is
    [-s z, s (15 - z)], so s = 15 s / 15 and z = s z / s come back exactly, codes equal u and the dequantized
    weights equal w."""
    u = rng.integers(0, 16, (n_groups, 32))
    for gi in range(n_groups):
        i0, i1 = rng.permutation(32)[:2]
        u[gi, i0], u[gi, i1] = 0, 15
    s = np.exp2(rng.integers(-16, 2, n_groups)).astype(np.float32)
    z = rng.integers(0, 16, n_groups)
    return ((u - z[:, None]) * s[:, None]).astype(np.float32), u, s, z


def test_lattice_is_reproduced_exactly(orc):
    rng = np.random.default_rng(51)
    w, u, s, z = lattice(rng, 24 * 8)
    W = w.reshape(24, 256)
    parts = orc.quantize(orc.Q4G32A, W)
    assert np.array_equal(parts["q"].reshape(-1, 32), u)
    sz = parts["gscale"].reshape(-1, 2)
    assert np.array_equal(sz[:, 0], s) and np.array_equal(sz[:, 1], z.astype(np.float32))
    packed, gs = orc.pack(orc.Q4G32A, 24, 256, parts)
    assert np.array_equal(orc.dequant(orc.Q4G32A, 24, 256, packed, gs), W)
    # the stored nibbles are the codes themselves (no offset); low nibble = even index
    uu = u.reshape(24, 256)
    assert np.array_equal(packed, (uu[:, 0::2] + 16 * uu[:, 1::2]).astype(np.uint8))


def test_zero_weights_come_back_exactly(orc):
    """Zero maps to the code z and dequantizes to exactly 0 in every group, whatever its skew (the reason for an
    integer zero point)."""
    rng = np.random.default_rng(54)
    W = (rng.standard_normal((16, 512)) + rng.uniform(-3, 3, (16, 1))).astype(np.float32)
    W[rng.random(W.shape) < 0.2] = 0.0
    parts = orc.quantize(orc.Q4G32A, W)
    packed, gs = orc.pack(orc.Q4G32A, 16, 512, parts)
    deq = orc.dequant(orc.Q4G32A, 16, 512, packed, gs)
    z = parts["gscale"].reshape(16, -1, 2)[:, :, 1].repeat(32, axis=1)
    assert np.all(parts["q"][W == 0] == z[W == 0])
    assert np.all(deq[W == 0] == 0.0)


def test_one_sided_constant_and_zero_groups(orc):
    W = np.zeros((1, 96), np.float32)
    W[0, :32] = np.linspace(0.5, 2.0, 32, dtype=np.float32)        # no negative weight: z = 0, s = 2 / 15
    W[0, 32:64] = -0.75                                            # constant negative: z = 15, codes 0
    parts = orc.quantize(orc.Q4G32A, W)
    sz = parts["gscale"][0]
    assert sz[0] == np.float32(2.0) / np.float32(15.0) and sz[1].view(np.uint32) == 0    # z = +0
    assert parts["q"][0, 31] == 15 and parts["q"][0, 0] == 4       # 0.5 / (2 / 15) = 3.75 -> 4
    assert sz[3] == 15.0 and not parts["q"][0, 32:64].any()
    assert sz[4] == np.float32(1e-12) and sz[5] == 0.0 and not parts["q"][0, 64:].any()   # all-zero group: floor
    packed, gs = orc.pack(orc.Q4G32A, 1, 96, parts)
    deq = orc.dequant(orc.Q4G32A, 1, 96, packed, gs)[0]
    assert np.allclose(deq[32:64], -0.75, rtol=2 ** -22, atol=0) and np.all(deq[64:] == 0.0)


def test_error_bound_and_gain_over_symmetric(orc):
    """|w - w'| <= s / 2 (plus the fp32 roundings of w / s, -lo / s and s (q - z), a few ulps of the group range),
    also where the top code clamps. On one-sided groups the asymmetric rule spends all 16 codes on the range and
    beats the symmetric rule's mean error (P1 §2.1's argument for the asymmetric form)."""
    rng = np.random.default_rng(52)
    W = (rng.standard_normal((32, 1024)) * np.exp(rng.uniform(-6, 3, (32, 1)))).astype(np.float32)
    W += (np.float32(0.7) * np.abs(W).max(axis=1, keepdims=True) * rng.uniform(-1, 1, (32, 1))).astype(np.float32)
    parts = orc.quantize(orc.Q4G32A, W)
    packed, gs = orc.pack(orc.Q4G32A, 32, 1024, parts)
    deq = orc.dequant(orc.Q4G32A, 32, 1024, packed, gs).astype(np.float64)
    s = parts["gscale"].astype(np.float64).reshape(32, 32, 2)[:, :, 0].repeat(32, axis=1)
    assert np.all(np.abs(deq - W) <= s / 2 + 15 * s * 2.0 ** -21)
    assert (np.abs(deq - W) > 0.45 * s).any()                       # the bound is reached, not vacuous

    P = np.abs(rng.standard_normal((32, 1024))).astype(np.float32)  # one-sided weights
    pa = orc.quantize(orc.Q4G32A, P)
    ps = orc.quantize(orc.Q4G32, P)
    ea = np.abs(orc.dequant(orc.Q4G32A, 32, 1024, *orc.pack(orc.Q4G32A, 32, 1024, pa)) - P).mean()
    es = np.abs(orc.dequant(orc.Q4G32, 32, 1024, *orc.pack(orc.Q4G32, 32, 1024, ps)) - P).mean()
    assert ea < 0.6 * es


def test_byte_accounting(orc):
    lay = orc.layout(orc.Q4G32A, 64, 4096)
    assert lay["row_stride"] == 2048 and lay["scale_stride"] == 256
    assert 8 * (lay["packed_bytes"] + lay["scale_bytes"]) / (64 * 4096) == 4.0 + 64 / 32     # 6 bpw
    assert orc.layout(orc.Q4G32A, 1, 96)["scale_stride"] == 8        # 3 pairs, rows padded to 16 bytes


def test_pack_unpack_round_trip(orc):
    rng = np.random.default_rng(53)
    N, K = 61, 32 * 512
    sz = np.stack([rng.standard_normal((N, K // 32)), rng.integers(0, 16, (N, K // 32))], -1)
    parts = dict(q=rng.integers(0, 16, (N, K)).astype(np.int8), gscale=sz.reshape(N, K // 16).astype(np.float32),
                 sub_scale=None, sub_min=None, d=None, dmin=None)
    packed, gs = orc.pack(orc.Q4G32A, N, K, parts)
    back = orc.unpack(orc.Q4G32A, N, K, packed, gs)
    assert np.array_equal(back["q"], parts["q"])
    assert np.array_equal(back["gscale"].view(np.uint32), parts["gscale"].view(np.uint32))
