"""GPU parity of quantize / pack / fused quantize+pack / unpack / dequantize: every code, packed byte, scale and
dequantized value must equal the oracle's bit for bit (DBHOO-CIM article §3.1-§3.2 for INT4,
2/3/5/6-bit article §2.1-§2.3 for the super-block formats)."""
import numpy as np
import pytest
import torch

from conftest import to_np_fp32

pytestmark = pytest.mark.gpu

ALL = ["Q4G32", "Q2S", "Q3S", "Q5S", "Q6S", "Q4G32H", "Q4G16", "Q4G32A"]
DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def weights(N, K, seed, dtype=torch.float32):
    from bit_weight_quantized_qpack_gb300 import synth
    W = synth.laplace((N, K), 0.02, seed)
    g = torch.Generator().manual_seed(seed + 1)
    mask = torch.rand(N, K, generator=g) < 0.002
    W[mask] *= 25.0                                      # outliers
    if N > 2:
        W[1] = 0.0                                       # an all-zero row
        W[2, : min(K, 256)] = -W[2, : min(K, 256)].abs()  # a negative-only block
    return W.to(dtype)


def shapes(name):
    out = [(1, 256), (37, 1024), (5, 4096 + 256)]
    if name in ("Q4G32", "Q4G32H", "Q4G16", "Q4G32A"):
        out += [(9, 96), (3, 32), (6, 4096 + 160)]       # rows ending inside a 256-weight block
    return out


def cmp_parts(got, ref):
    for k in ("q", "gscale", "sub_scale", "sub_min", "d", "dmin"):
        if ref.get(k) is None:
            continue
        g = got[k].cpu().numpy()
        r = ref[k]
        if g.dtype == np.int16:
            g = g.view(np.uint16)
        if g.dtype == np.float32:
            assert np.array_equal(g.view(np.uint32), r.view(np.uint32)), k
        else:
            assert np.array_equal(g, r), k


@pytest.mark.parametrize("name", ALL)
@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
def test_quantize_parts_and_packed_bit_exact(qpg, orc, name, dt):
    fmt = qpg.FORMATS[name]
    for i, (N, K) in enumerate(shapes(name)):
        W = weights(N, K, 100 + i, DT[dt])
        Wd = W.cuda()
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        parts = qpg.qpack_quantize(fmt, Wd, status=st)
        packed, gs = qpg.qpack_quantize_pack(fmt, Wd, status=st)
        torch.cuda.synchronize()
        Wn = to_np_fp32(W)
        ref = orc.quantize(fmt, Wn)
        cmp_parts(parts, ref)
        rp, rgs = orc.pack(fmt, N, K, ref)
        assert np.array_equal(packed.cpu().numpy(), rp)
        if rgs is not None:                                # fp32 (Q4G32) or fp16 (Q4G32H) scales, bit for bit
            assert np.array_equal(gs.cpu().numpy().view(np.uint8), rgs.view(np.uint8))
        assert int(st.item()) == ref["flags"] == 0


@pytest.mark.parametrize("name", ALL)
def test_pack_unpack_dequant_bit_exact(qpg, orc, name):
    fmt = qpg.FORMATS[name]
    for i, (N, K) in enumerate(shapes(name)):
        Wn = to_np_fp32(weights(N, K, 200 + i))
        ref = orc.quantize(fmt, Wn)
        rp, rgs = orc.pack(fmt, N, K, ref)
        # pack the oracle's parts on the GPU
        parts = {k: (None if v is None or k == "flags" else torch.from_numpy(
            v.view(np.int16) if v.dtype == np.uint16 else v).cuda()) for k, v in ref.items()}
        packed, gs = qpg.qpack_pack(fmt, N, K, parts)
        torch.cuda.synchronize()
        assert np.array_equal(packed.cpu().numpy(), rp)
        # unpack and dequantize the oracle's bytes on the GPU
        pd = torch.from_numpy(rp).cuda()
        gd = None if rgs is None else torch.from_numpy(rgs.view(np.int16) if rgs.dtype == np.uint16 else rgs).cuda()
        back = qpg.qpack_unpack(fmt, N, K, pd, gd)
        deq = qpg.qpack_dequant(fmt, N, K, pd, gd)
        torch.cuda.synchronize()
        cmp_parts(back, ref)
        rdeq = orc.dequant(fmt, N, K, rp, rgs)
        assert np.array_equal(deq.cpu().numpy().view(np.uint32), rdeq.view(np.uint32))


@pytest.mark.parametrize("name", ["Q2S", "Q3S", "Q5S", "Q6S", "Q4G32H"])
def test_range_flag(qpg, orc, name):
    fmt = qpg.FORMATS[name]
    W = torch.zeros(3, 512)
    W[1, 256:] = 1e9
    W[1, 300] = -1e9
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    packed, _ = qpg.qpack_quantize_pack(fmt, W.cuda(), status=st)
    torch.cuda.synchronize()
    ref_packed, _, flags = orc.quantize_pack(fmt, W.numpy())
    assert flags == 1 and int(st.item()) == 1
    assert np.array_equal(packed.cpu().numpy(), ref_packed)
    st.zero_()
    qpg.qpack_quantize_pack(fmt, torch.ones(2, 256, device="cuda") * 0.5, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0


def test_int4_config_matrix_bit_exact(qpg, orc):
    """4096x4096 fp32 W ~ N(0, 0.02^2) with 0.1% ±U(0.1, 0.5) outliers (seed 0), INT4 group 32."""
    from bit_weight_quantized_qpack_gb300 import synth
    W = synth.normal_with_outliers((4096, 4096), 0.02, 0.001, 0.1, 0.5, seed=0)
    packed, gs = qpg.qpack_quantize_pack(qpg.Q4G32, W.cuda())
    torch.cuda.synchronize()
    rp, rgs, _ = orc.quantize_pack(orc.Q4G32, W.numpy())
    assert np.array_equal(packed.cpu().numpy(), rp)
    assert np.array_equal(gs.cpu().numpy().view(np.uint32), rgs.view(np.uint32))


def test_q3s_config_matrix_bit_exact(qpg, orc):
    """11008x4096 Laplace(0, 0.015) weights (seed 0), 3-bit 110-byte super-blocks."""
    from bit_weight_quantized_qpack_gb300 import synth
    W = synth.laplace((11008, 4096), 0.015, seed=0)
    packed, _ = qpg.qpack_quantize_pack(qpg.Q3S, W.cuda())
    torch.cuda.synchronize()
    rp, _, _ = orc.quantize_pack(orc.Q3S, W.numpy())
    assert np.array_equal(packed.cpu().numpy(), rp)


def test_int4_quotients_at_rounding_boundaries(qpg, orc):
    """Weights whose quotient w / s sits on or next to a half-integer (ties round to even, P2 §3.1's torch.round): the
    codes must still equal the oracle's (IEEE division, then round half to even)."""
    s = np.float32(0.01)
    rng = np.random.default_rng(5)
    N, K = 64, 4096
    W = np.empty((N, K), np.float32)
    for r in range(N):
        k = rng.integers(-8, 7, K).astype(np.float32) + np.float32(0.5)
        w = (k * s).astype(np.float32)
        step = rng.integers(-2, 3, K)                    # the tie itself and its fp32 neighbours
        w = np.where(step > 0, np.nextafter(w, np.float32(np.inf)), w)
        w = np.where(step < 0, np.nextafter(w, np.float32(-np.inf)), w)
        w = np.where(step == 2, np.nextafter(w, np.float32(np.inf)), w)
        w = np.where(step == -2, np.nextafter(w, np.float32(-np.inf)), w)
        W[r] = w
    W[:, ::32] = np.float32(8) * s                        # every group's max: s = max / 8 exactly
    Wt = torch.from_numpy(W)
    packed, gs = qpg.qpack_quantize_pack(qpg.Q4G32, Wt.cuda())
    torch.cuda.synchronize()
    rp, rgs, _ = orc.quantize_pack(orc.Q4G32, W)
    assert np.array_equal(packed.cpu().numpy(), rp)
    assert np.array_equal(gs.cpu().numpy().view(np.uint32), rgs.view(np.uint32))


@pytest.mark.parametrize("name,G", [("Q4G16", 16), ("Q4G32H", 32)])
def test_int4_variants_quotients_at_rounding_boundaries(qpg, orc, name, G):
    """As above for group 16 and for the fp16 group scale, with s = 2^-7 (exact in fp16, so the fp16-rounded scale is s
    itself): quotients on and next to half-integers, every group's maximum 8 s."""
    s = np.float32(2.0 ** -7)
    rng = np.random.default_rng(6)
    N, K = 64, 4096
    k = rng.integers(-8, 7, (N, K)).astype(np.float32) + np.float32(0.5)
    W = (k * s).astype(np.float32)
    step = rng.integers(-1, 2, (N, K))
    W = np.where(step > 0, np.nextafter(W, np.float32(np.inf)), W)
    W = np.where(step < 0, np.nextafter(W, np.float32(-np.inf)), W).astype(np.float32)
    W[:, ::G] = np.float32(8) * s
    fmt = qpg.FORMATS[name]
    packed, gs = qpg.qpack_quantize_pack(fmt, torch.from_numpy(W).cuda())
    torch.cuda.synchronize()
    rp, rgs, _ = orc.quantize_pack(fmt, W)
    assert np.array_equal(packed.cpu().numpy(), rp)
    g = gs.cpu().numpy()
    assert np.array_equal(g.view(np.uint16 if g.dtype == np.int16 or g.dtype == np.float16 else np.uint32),
                          rgs.view(np.uint16 if rgs.dtype in (np.uint16, np.float16) else np.uint32))


@pytest.mark.parametrize("name", ["Q2S", "Q3S", "Q5S", "Q6S"])
def test_superblock_quotients_at_rounding_boundaries(qpg, orc, name):
    """Weights on and next to the half-integer quotients of their sub-block's rounded scale: w = (k + 1/2) e, or
    (k + 1/2) e_s - e_m for the asymmetric formats (the quotient is (w + e_m) / e_s), with e the oracle's own
    d16 * L_j. Each sub-block keeps its smallest and largest weight and the others stay between them, so every
    scale is unchanged; the codes, where the quantizer's quotient from a reciprocal defers to the true division, must
    equal the oracle's (2/3/5/6-bit article §2.1, rounding half to even)."""
    from bit_weight_quantized_qpack_gb300 import synth
    fmt = qpg.FORMATS[name]
    bits, nsub, sublen, lmax, asym, _ = orc.SB[fmt]
    N, K = 32, 1024
    W = synth.laplace((N, K), 0.02, seed=61).numpy().astype(np.float32)
    P = orc.quantize(fmt, W)
    D = orc.f16_bits_to_f32(P["d"])
    Dm = orc.f16_bits_to_f32(P["dmin"]) if asym else None
    rng = np.random.default_rng(62)
    placed = 0
    for r in range(N):
        for j in range((K // 256) * nsub):
            seg = slice(j * sublen, (j + 1) * sublen)
            w = W[r, seg].copy()
            lo_i, hi_i = int(np.argmin(w)), int(np.argmax(w))
            Lj = np.float32(np.int8(P["sub_scale"][r, j]) if name == "Q6S" else P["sub_scale"][r, j])
            e = np.float32(np.float32(D[r, j // nsub]) * Lj)
            if not e > 0:
                continue
            if asym:
                em = np.float32(np.float32(Dm[r, j // nsub]) * np.float32(P["sub_min"][r, j]))
                k = rng.integers(0, 2 ** bits - 1, sublen).astype(np.float32) + np.float32(0.5)
                v = (k * e - em).astype(np.float32)
            else:
                k = rng.integers(-(2 ** (bits - 1)), 2 ** (bits - 1) - 1, sublen).astype(np.float32) + np.float32(0.5)
                v = (k * e).astype(np.float32)
            step = rng.integers(-1, 2, sublen)
            v = np.where(step > 0, np.nextafter(v, np.float32(np.inf)), v)
            v = np.where(step < 0, np.nextafter(v, np.float32(-np.inf)), v).astype(np.float32)
            v = np.clip(v, w[lo_i], w[hi_i]).astype(np.float32)
            v[lo_i], v[hi_i] = w[lo_i], w[hi_i]
            W[r, seg] = v
            placed += sublen - 2
    assert placed > N * K // 2
    P2 = orc.quantize(fmt, W)
    for key in ("sub_scale", "sub_min", "d", "dmin"):          # the construction kept every scale
        if P[key] is not None:
            assert np.array_equal(P[key], P2[key]), key
    packed, _ = qpg.qpack_quantize_pack(fmt, torch.from_numpy(W).cuda())
    torch.cuda.synchronize()
    rp, _, _ = orc.quantize_pack(fmt, W)
    assert np.array_equal(packed.cpu().numpy(), rp)


@pytest.mark.parametrize("name", ALL)
def test_quantize_pack_large_bit_exact(qpg, orc, name):
    """16.7 M weights per format (random weights rarely come near a rounding boundary, where the quantizer's quotient
    from a reciprocal defers to the true division; the boundary tests take that path on purpose): packed bytes and
    scales bit-exact."""
    from bit_weight_quantized_qpack_gb300 import synth
    fmt = qpg.FORMATS[name]
    W = synth.laplace((4096, 4096), 0.02, 77)
    packed, gs = qpg.qpack_quantize_pack(fmt, W.cuda())
    torch.cuda.synchronize()
    rp, rgs, _ = orc.quantize_pack(fmt, W.numpy())
    assert np.array_equal(packed.cpu().numpy(), rp)
    if rgs is not None:
        assert np.array_equal(gs.cpu().numpy().view(np.uint32), rgs.view(np.uint32))


@pytest.mark.parametrize("name", ["Q4G32", "Q2S", "Q3S", "Q5S", "Q6S"])
@pytest.mark.parametrize("shape", [(14336, 4096), (4096, 14336)], ids=["14336x4096", "4096x14336"])
def test_prefill_config_fp16_matrices_bit_exact(qpg, orc, name, shape):
    """The prefill workload's weights exactly as the benchmark quantizes them: Laplace(0, 0.02), seed 7, held as fp16,
    14336x4096 and 4096x14336, each of the five base formats, fused quantize+pack from fp16 on the GPU. The oracle
    quantizes the same values widened to fp32 (exact), so packed bytes and scales must match bit for bit."""
    from bit_weight_quantized_qpack_gb300 import synth
    fmt = qpg.FORMATS[name]
    N, K = shape
    W16 = synth.laplace((N, K), 0.02, seed=7, dtype=torch.float16)
    packed, gs = qpg.qpack_quantize_pack(fmt, W16.cuda())
    torch.cuda.synchronize()
    rp, rgs, flags = orc.quantize_pack(fmt, W16.float().numpy())
    assert flags == 0
    assert np.array_equal(packed.cpu().numpy(), rp)
    if rgs is not None:
        assert np.array_equal(gs.cpu().numpy().view(np.uint32), rgs.view(np.uint32))


def test_q4g32a_skewed_and_degenerate_groups_bit_exact(qpg, orc):
    """Asymmetric INT4 groups of every shape the zero-point rule distinguishes (DBHOO-CIM article §5.1; 2/3/5/6-bit
    article §2.1): positive-only (z = 0), negative-only (z = 15), constant, all-zero (the 1e-12 floor), exact lattices
    w = s (u - z) whose quotients land on integers, half-integer quotients (ties to even), subnormal and huge
    magnitudes (a range near the fp32 limit), and zeros mixed into skewed groups."""
    rng = np.random.default_rng(77)
    G = []
    G.append(np.abs(rng.standard_normal(32)) + 0.1)
    G.append(-np.abs(rng.standard_normal(32)) - 0.1)
    G.append(np.full(32, 0.3))
    G.append(np.full(32, -2.5))
    G.append(np.zeros(32))
    for _ in range(8):
        s, z = 2.0 ** rng.integers(-12, 3), rng.integers(0, 16)
        u = rng.integers(0, 16, 32)
        u[:2] = (0, 15)
        G.append(s * (u - z))
        G.append(s * (u - z + 0.5 * rng.choice([-1, 1], 32)).clip(-z, 15 - z))
    G.append(rng.standard_normal(32) * 1e-41)
    G.append(np.concatenate([[1.5e38, -1.5e38], rng.standard_normal(30) * 1e37]))
    g = rng.standard_normal(32) + 2.0
    g[rng.random(32) < 0.3] = 0.0
    G.append(g)
    while len(G) % 8:
        G.append(rng.standard_normal(32))
    W = np.concatenate(G).astype(np.float32).reshape(-1, 256)
    N, K = W.shape
    fmt = qpg.Q4G32A
    parts = qpg.qpack_quantize(fmt, torch.from_numpy(W).cuda())
    packed, gs = qpg.qpack_quantize_pack(fmt, torch.from_numpy(W).cuda())
    deq = qpg.qpack_dequant(fmt, N, K, packed, gs)
    torch.cuda.synchronize()
    ref = orc.quantize(fmt, W)
    cmp_parts(parts, ref)
    rp, rgs = orc.pack(fmt, N, K, ref)
    assert np.array_equal(packed.cpu().numpy(), rp)
    assert np.array_equal(gs.cpu().numpy().view(np.uint32), rgs.view(np.uint32))
    rdeq = orc.dequant(fmt, N, K, rp, rgs)
    assert np.array_equal(deq.cpu().numpy().view(np.uint32), rdeq.view(np.uint32))
