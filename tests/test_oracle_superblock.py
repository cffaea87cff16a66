"""Pins for the oracle's 256-weight super-block formats (2/3/5/6-bit quantization article,
lpnh.cn/news/2857666, §2.1 two-level scales, §2.2 cross-byte packing, §2.3 byte table, §3.4 self-checks):
byte accounting against the page's table, exact lattices, closed-form bit layouts, 1e6-value round trips,
error bounds and the overflow status."""
import numpy as np
import pytest
from conftest import read_golden

FMTS = ["Q2S", "Q3S", "Q5S", "Q6S"]


def table():
    rows = [r for r in read_golden("superblock_bytes.txt") if r[0] != "PLANES"]
    return {r[0]: dict(codes=int(r[1]), sub=int(r[2]), sup=int(r[3]), total=int(r[4]), bpw=float(r[5])) for r in rows}


@pytest.mark.parametrize("name", FMTS)
def test_byte_accounting_matches_page_table(orc, name):
    t = table()[name]
    fmt = orc.FORMATS[name]
    bits, nsub, sublen, lmax, asym, nbytes = orc.SB[fmt]
    assert t["codes"] + t["sub"] + t["sup"] == t["total"] == nbytes
    assert 8 * nbytes / 256 == t["bpw"]
    assert t["codes"] == 256 * bits // 8
    assert nsub * sublen == 256
    lay = orc.layout(fmt, 3, 512)
    assert lay["block_bytes"] == nbytes
    assert lay["row_stride"] == -(-2 * nbytes // 16) * 16 and lay["packed_bytes"] == 3 * lay["row_stride"]


def test_model_sizes_match_page(orc):
    for name, bpw, gb in read_golden("model_sizes.txt"):
        fmt = orc.FORMATS[name]
        exact_bpw = 8 * orc.SB[fmt][5] / 256
        assert abs(exact_bpw - float(bpw)) < 0.05
        assert abs(7e9 * exact_bpw / 8 / 1e9 - float(gb)) < 0.05


def test_plane_split_matches_page():
    planes = {r[1]: (int(r[2]), int(r[3])) for r in read_golden("superblock_bytes.txt") if r[0] == "PLANES"}
    assert planes["Q5S"] == (128, 32) and planes["Q6S"] == (128, 64)
    assert sum(planes["Q5S"]) == table()["Q5S"]["codes"] and sum(planes["Q6S"]) == table()["Q6S"]["codes"]


def make_lattice(orc, fmt, rows, nb, rng):
    """W = d * L_j * q_i (- dmin * M_j) with d, dmin powers of two, max L_j = Lmax, and every sub-block holding its
    extreme codes, so the two-level quantizer must return exactly (d, L, M, q) and dequant(W) == W."""
    bits, nsub, sublen, lmax, asym, nbytes = orc.SB[fmt]
    K = 256 * nb
    W = np.zeros((rows, K), np.float32)
    q = np.zeros((rows, K), np.int64)
    L = np.zeros((rows, nb * nsub), np.int64)
    M = np.zeros((rows, nb * nsub), np.int64)
    d = np.zeros((rows, nb), np.float32)
    dm = np.zeros((rows, nb), np.float32)
    for r in range(rows):
        for b in range(nb):
            e = rng.integers(-12, 6)
            dv = np.float32(2.0 ** e)
            dmv = np.float32(2.0 ** (e + rng.integers(-3, 4)))
            Lb = rng.integers(1, lmax + 1, nsub)
            jmax = rng.integers(nsub)
            Lb[jmax] = lmax
            Mb = rng.integers(0, lmax + 1, nsub)
            Mb[rng.integers(nsub)] = lmax
            if b % 3 == 1:                      # one all-zero-scale sub-block now and then
                Lb[(jmax + 1 + rng.integers(nsub - 1)) % nsub] = 0
            for j in range(nsub):
                sl = slice(256 * b + sublen * j, 256 * b + sublen * (j + 1))
                if asym:
                    qs = rng.integers(0, 2 ** bits, sublen)
                    qs[0], qs[1] = 0, 2 ** bits - 1
                    if Lb[j] == 0:
                        qs[:] = 0
                    # stored M for a zero-L sub-block still decodes to -dmin*M
                    W[r, sl] = (dv * Lb[j] * qs - dmv * Mb[j]).astype(np.float32)
                else:
                    qs = rng.integers(-(2 ** (bits - 1)), 2 ** (bits - 1), sublen)
                    qs[0] = -(2 ** (bits - 1))
                    if Lb[j] == 0:
                        qs[:] = 0
                    W[r, sl] = (dv * Lb[j] * qs).astype(np.float32)
                q[r, sl] = qs
            L[r, b * nsub:(b + 1) * nsub] = Lb
            M[r, b * nsub:(b + 1) * nsub] = Mb
            d[r, b] = dv
            dm[r, b] = dmv
    return W, q, L, M, d, dm


@pytest.mark.parametrize("name", FMTS)
def test_exact_lattice(orc, name):
    fmt = orc.FORMATS[name]
    bits, nsub, sublen, lmax, asym, nbytes = orc.SB[fmt]
    rng = np.random.default_rng(20 + fmt)
    W, q, L, M, d, dm = make_lattice(orc, fmt, 6, 3, rng)
    parts = orc.quantize(fmt, W)
    assert parts["flags"] == 0
    assert np.array_equal(orc.f16_bits_to_f32(parts["d"]), d)
    zero_sub = (L == 0)
    if asym:
        assert np.array_equal(orc.f16_bits_to_f32(parts["dmin"]), dm)
        assert np.array_equal(parts["sub_min"].astype(np.int64), M)
        # a zero-scale sub-block quantizes to q = 0 regardless of the construction
        assert np.array_equal(parts["sub_scale"].astype(np.int64), L)
    else:
        assert np.array_equal(parts["sub_scale"].astype(np.int64), L)
    assert np.array_equal(parts["q"].astype(np.int64), q)
    packed, _ = orc.pack(fmt, 6, W.shape[1], parts)
    deq = orc.dequant(fmt, 6, W.shape[1], packed)
    assert np.array_equal(deq, W)
    assert not zero_sub.all()


def test_q3s_code_layout_closed_form(orc):
    # P1 §2.2 unpack3: 8 codes in 3 bytes, code t at bits 3t -> the 24-bit value is the base-8 number with
    # digit t = u_t; stored u = q + 4 (offset binary for the symmetric 3-bit codes).
    rng = np.random.default_rng(30)
    u = rng.integers(0, 8, 256)
    parts = dict(q=(u - 4).astype(np.int8)[None, :], sub_scale=np.arange(16, dtype=np.uint8)[None, :] * 4 + 1,
                 d=np.array([[0x3C00]], np.uint16))
    packed, _ = orc.pack(orc.Q3S, 1, 256, parts)
    p = packed[0].astype(np.int64)
    for g in range(32):
        v = p[3 * g] + 256 * p[3 * g + 1] + 65536 * p[3 * g + 2]
        assert v == sum(int(u[8 * g + t]) * 8 ** t for t in range(8))
    for r in range(4):
        v = p[96 + 3 * r] + 256 * p[97 + 3 * r] + 65536 * p[98 + 3 * r]
        assert v == sum(int(parts["sub_scale"][0, 4 * r + f]) * 64 ** f for f in range(4))
    assert p[108] + 256 * p[109] == 0x3C00


def test_q2s_q5s_q6s_layout_closed_form(orc):
    rng = np.random.default_rng(31)
    # Q2S: weight i at bits 2(i&3) of byte i>>2 -> byte = sum_k u_{4b+k} * 4^k
    u = rng.integers(0, 4, 256)
    Ls, Ms = rng.integers(0, 16, 16), rng.integers(0, 16, 16)
    parts = dict(q=u.astype(np.int8)[None], sub_scale=Ls.astype(np.uint8)[None], sub_min=Ms.astype(np.uint8)[None],
                 d=np.array([[0x1234]], np.uint16), dmin=np.array([[0x5678]], np.uint16))
    p = orc.pack(orc.Q2S, 1, 256, parts)[0][0].astype(np.int64)
    assert all(p[b] == sum(int(u[4 * b + k]) * 4 ** k for k in range(4)) for b in range(64))
    assert all(p[64 + j] == Ls[j] + 16 * Ms[j] for j in range(16))
    assert p[80] + 256 * p[81] == 0x1234 and p[82] + 256 * p[83] == 0x5678
    # Q5S: low plane byte = lo(u_2b) + 16 lo(u_2b+1); high plane byte m of the 4-byte word of weights 32c .. 32c + 31:
    # bit 4 + j = hi(u_{32c+8j+2m}), bit j = hi(u_{32c+8j+2((m+3) mod 4)+1}); 16 six-bit fields
    u = rng.integers(0, 32, 256)
    Ls, Ms = rng.integers(0, 64, 8), rng.integers(0, 64, 8)
    parts = dict(q=u.astype(np.int8)[None], sub_scale=Ls.astype(np.uint8)[None], sub_min=Ms.astype(np.uint8)[None],
                 d=np.array([[0x0101]], np.uint16), dmin=np.array([[0x0202]], np.uint16))
    p = orc.pack(orc.Q5S, 1, 256, parts)[0][0].astype(np.int64)
    assert all(p[b] == u[2 * b] % 16 + 16 * (u[2 * b + 1] % 16) for b in range(128))
    for c in range(8):
        for m in range(4):
            even = sum(int(u[32 * c + 8 * j + 2 * m] // 16) * 2 ** (4 + j) for j in range(4))
            odd = sum(int(u[32 * c + 8 * j + 2 * ((m + 3) % 4) + 1] // 16) * 2 ** j for j in range(4))
            assert p[128 + 4 * c + m] == even + odd, (c, m)
    fields = list(Ls) + list(Ms)
    for r in range(4):
        v = p[160 + 3 * r] + 256 * p[161 + 3 * r] + 65536 * p[162 + 3 * r]
        assert v == sum(int(fields[4 * r + f]) * 64 ** f for f in range(4))
    assert p[172] + 256 * p[173] == 0x0101 and p[174] + 256 * p[175] == 0x0202
    # Q6S: stored u = q + 32; low plane as Q5S; high plane byte = sum_k (u_{4c+k} >> 4) 4^k; int8 scales
    u = rng.integers(0, 64, 256)
    Ls = rng.integers(0, 256, 16)
    parts = dict(q=(u - 32).astype(np.int8)[None], sub_scale=Ls.astype(np.uint8)[None], d=np.array([[0x3C00]], np.uint16))
    p = orc.pack(orc.Q6S, 1, 256, parts)[0][0].astype(np.int64)
    assert all(p[b] == u[2 * b] % 16 + 16 * (u[2 * b + 1] % 16) for b in range(128))
    assert all(p[128 + c] == sum(int(u[4 * c + k] // 16) * 4 ** k for k in range(4)) for c in range(64))
    assert all(p[192 + j] == Ls[j] for j in range(16))
    assert p[208] + 256 * p[209] == 0x3C00


def _random_parts(orc, fmt, N, K, rng):
    bits, nsub, sublen, lmax, asym, nbytes = orc.SB[fmt]
    nb = K // 256
    lo, hi = (0, 2 ** bits) if asym else (-(2 ** (bits - 1)), 2 ** (bits - 1))
    parts = dict(q=rng.integers(lo, hi, (N, K)).astype(np.int8),
                 sub_scale=rng.integers(0, 256 if fmt == orc.Q6S else (16 if fmt == orc.Q2S else 64),
                                        (N, nb * nsub)).astype(np.uint8),
                 d=rng.integers(0, 65536, (N, nb)).astype(np.uint16))
    if asym:
        parts["sub_min"] = rng.integers(0, 16 if fmt == orc.Q2S else 64, (N, nb * nsub)).astype(np.uint8)
        parts["dmin"] = rng.integers(0, 65536, (N, nb)).astype(np.uint16)
    return parts


@pytest.mark.parametrize("name", FMTS)
def test_million_value_roundtrip(orc, name):
    # P1 §2.2 / §3.4: pack then unpack 1,000,000 random integers, all equal.
    count = int(read_golden("selfcheck.txt")[0][1])
    fmt = orc.FORMATS[name]
    K = 4096
    N = -(-count // K)
    rng = np.random.default_rng(40 + fmt)
    parts = _random_parts(orc, fmt, N, K, rng)
    packed, _ = orc.pack(fmt, N, K, parts)
    back = orc.unpack(fmt, N, K, packed)
    for key in ("q", "sub_scale", "sub_min", "d", "dmin"):
        if parts.get(key) is not None:
            assert np.array_equal(back[key], parts[key]), key
    assert N * K >= count


def test_bit_runs_closed_form_and_roundtrip(orc):
    """P1 §2.2 cross-byte packing as bit runs: 8 three-bit codes in 3 bytes, 8 five-bit codes in 5 bytes and 4
    six-bit fields in 3 bytes. A million random fields per width round-trip, and on a prefix each group's
    little-endian byte value is the base-2^width number whose digit i is field i."""
    rng = np.random.default_rng(50)
    for width, per_group, group_bytes in ((3, 8, 3), (5, 8, 5), (6, 4, 3), (2, 4, 1), (4, 2, 1), (1, 8, 1)):
        n = (1_000_000 // per_group + 1) * per_group
        c = rng.integers(0, 2 ** width, n).astype(np.uint8)
        p = orc.run_pack(c, width)
        assert p.size == n // per_group * group_bytes
        assert np.array_equal(orc.run_unpack(p, width, n), c)
        for g in range(200):
            v = sum(int(p[group_bytes * g + b]) << (8 * b) for b in range(group_bytes))
            assert v == sum(int(c[per_group * g + i]) * (2 ** width) ** i for i in range(per_group))


@pytest.mark.parametrize("name", FMTS)
def test_error_bound_and_clamp_invariants(orc, name):
    fmt = orc.FORMATS[name]
    bits, nsub, sublen, lmax, asym, nbytes = orc.SB[fmt]
    rng = np.random.default_rng(60 + fmt)
    W = rng.laplace(0, 0.02, (64, 1024)).astype(np.float32)
    parts = orc.quantize(fmt, W)
    packed, _ = orc.pack(fmt, 64, 1024, parts)
    deq = orc.dequant(fmt, 64, 1024, packed).astype(np.float64)
    D = np.repeat(orc.f16_bits_to_f32(parts["d"]), 256, axis=1).astype(np.float64)
    L = np.repeat(parts["sub_scale"].astype(np.float64), sublen, axis=1)
    es = D * L
    q = parts["q"].astype(np.float64)
    if asym:
        Dm = np.repeat(orc.f16_bits_to_f32(parts["dmin"]), 256, axis=1).astype(np.float64)
        em = Dm * np.repeat(parts["sub_min"].astype(np.float64), sublen, axis=1)
        t = (W + em) / es
        qlo, qhi = 0, 2 ** bits - 1
    else:
        t = W / es
        qlo, qhi = -(2 ** (bits - 1)), 2 ** (bits - 1) - 1
    err = np.abs(W - deq)
    inr = (t >= qlo - 0.5) & (t <= qhi + 0.5)
    assert np.all(err[inr] <= es[inr] / 2 * (1 + 1e-5) + 1e-12)
    assert np.all(q[t < qlo - 0.5] == qlo) and np.all(q[t > qhi + 0.5] == qhi)
    assert inr.mean() > 0.9      # symmetric 3-bit clamps its positive extremes (range -4..3)


@pytest.mark.parametrize("name", FMTS)
def test_zero_block_and_range_flag(orc, name):
    fmt = orc.FORMATS[name]
    W = np.zeros((2, 512), np.float32)
    W[1, 256:] = 1e9            # d = 1e9 / 2^(b-1) / Lmax or (max-lo)/(2^b-1)/Lmax: beyond fp16 for every format
    W[1, 300] = -1e9
    parts = orc.quantize(fmt, W)
    assert parts["flags"] == 1
    assert np.all(parts["d"][0] == 0) and not parts["q"][0].any()
    packed, _ = orc.pack(fmt, 2, 512, parts)
    deq = orc.dequant(fmt, 2, 512, packed)
    assert not deq[0].any()
    assert np.all(parts["d"][1, 1] & 0x7FFF == 0x7C00) or np.all(parts["dmin"][1, 1] & 0x7FFF == 0x7C00)
