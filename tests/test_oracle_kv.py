"""Pins of the oracle's 8-bit KV-cache quantizer (2/3/5/6-bit article §4.1: 8 bits, one fp16 scale per 32 elements;
Mix-Quant article §2.3: dequantized back to fp16). Exact lattices, the rounding and clamp rules, the error bound and
the page's byte accounting, none of which re-derive the oracle's own formula."""
import numpy as np
import pytest

from conftest import kv, read_golden


def f16(x):
    return np.asarray(x, np.float16).view(np.uint16)


def test_exact_lattice_round_trips(orc):
    """v = d * q with d a power of two and |q| = 127 present in every group: the quantizer returns d and q exactly and
    dequantization gives v back bit for bit."""
    rng = np.random.default_rng(1)
    G = 257
    q = rng.integers(-127, 128, size=(G, 32))
    q[np.arange(G), rng.integers(0, 32, G)] = rng.choice([-127, 127], G)
    e = rng.integers(-14, -2, G)                      # d = 2^e: v = q * 2^e stays a normal fp16
    d = np.ldexp(1.0, e)
    v = (q * d[:, None]).astype(np.float16)
    assert np.array_equal(v.astype(np.float64), q * d[:, None])      # the lattice itself is exact in fp16
    qo, so = orc.kv_quantize(f16(v))
    assert np.array_equal(qo.reshape(G, 32), q)
    assert np.array_equal(so, f16(d))
    assert np.array_equal(orc.kv_dequant(qo, so), f16(v))


def test_ties_round_to_even_and_zero_group(orc):
    d = 2.0 ** -6
    vals = np.zeros(32)
    vals[0] = 127 * d                                  # sets d exactly
    vals[1:6] = np.array([0.5, 1.5, 2.5, -2.5, -0.5]) * d
    q, s = orc.kv_quantize(f16(np.concatenate([vals, np.zeros(32)])))
    assert list(q[:6]) == [127, 0, 2, 2, -2, 0]
    assert s[1] == 0 and not q[32:].any()
    assert not orc.kv_dequant(q, s)[32:].any()


def test_clamp_when_the_rounded_scale_is_smaller(orc):
    """max|v| / 127 rounded to fp16 can land below the true quotient (for small groups the scale is subnormal and
    coarse), so max|v| / d exceeds 127: the code clamps to 127, never wraps."""
    found = 0
    for m in np.unique(np.geomspace(2.0 ** -16, 2.0 ** -8, 3000).astype(np.float16)):
        a = float(m)
        d = float(np.float16(np.float32(a) / np.float32(127.0)))
        if d > 0 and a / d > 127.5:
            v = np.zeros(32, np.float16)
            v[3] = m
            v[4] = -m
            q, s = orc.kv_quantize(f16(v))
            assert q[3] == 127 and q[4] == -127
            found += 1
    assert found > 0


def test_error_bound(orc):
    """|v - v'| <= d/2 (rounding to the code lattice, the clamp only ever shortens a step) plus the fp16 rounding of
    v' (at most half an fp16 ulp of |v'|), with d the group's stored scale."""
    rng = np.random.default_rng(2)
    v = (rng.standard_normal((4096, 32)) * np.exp(rng.uniform(-8, 4, (4096, 1)))).astype(np.float16)
    q, s = orc.kv_quantize(f16(v))
    vd = orc.kv_dequant(q, s).view(np.float16).astype(np.float64).reshape(4096, 32)
    d = s.view(np.float16).astype(np.float64)[:, None]
    ulp = np.spacing(np.abs(vd).astype(np.float16)).astype(np.float64)
    a = np.abs(v.astype(np.float64)).max(axis=1, keepdims=True)
    err = np.abs(vd - v.astype(np.float64))
    # an element that clamps is within (a - 127 d) of the lattice end, which the first term covers when d >= a / 127.5
    bound = np.maximum(d / 2, a - 127 * d) + ulp / 2
    assert np.all(err <= bound * (1 + 1e-12))


def test_page_byte_accounting(orc):
    g = {r[0]: kv(r[1:]) for r in read_golden("kv_cache.txt")}
    k = g["KV"]
    elems = 2 * k["layers"] * k["kv_heads"] * k["head_dim"] * k["context"]
    assert abs(elems * 2 / 1e9 - k["fp16_GB"]) < 0.005
    # the layout stores one int8 code per element and one fp16 scale per 32 elements
    n = 32 * 64
    q, s = orc.kv_quantize(np.zeros(n, np.uint16))
    bytes_per_elem = (q.nbytes + s.nbytes) / n
    assert bytes_per_elem == 34 / 32
    assert abs(bytes_per_elem - g["INT8"]["bytes_per_elem"]) < 0.005
    assert abs(elems * 1.0 / 1e9 - g["INT8"]["half_GB"]) < 0.005      # the codes alone: the page's "half"


def test_size_must_be_whole_groups(orc):
    with pytest.raises(ValueError):
        orc.kv_quantize(np.zeros(48, np.uint16))
