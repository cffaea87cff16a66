"""GPU parity of the tensor-core prefill dequant GEMM against the oracle's fp64 reference with bf16 weights:
||Y - Y_ref|| / ||Y_ref|| <= 2e-2 (the bound of the prefill path), plus a tight per-element check that the only
error sources are fp32 accumulation and the final bf16 rounding of Y (2/3/5/6-bit article §1.2: prefill is a
dense contraction)."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

ALL = ["Q4G32", "Q2S", "Q3S", "Q5S", "Q6S", "Q4G32H", "Q4G16", "Q4G32A"]


def corner_tiles(M, N, T=128):
    """Every element of the four T x T output tiles at the corners of Y (clipped to M x N): whole CTA tiles at the
    first and last token and weight-row positions, where a per-tile descriptor or epilogue fault would show."""
    ms, ns = [], []
    for m0 in sorted({0, max(0, M - T)}):
        for n0 in sorted({0, max(0, N - T)}):
            mm, nn = np.meshgrid(np.arange(m0, min(M, m0 + T)), np.arange(n0, min(N, n0 + T)), indexing="ij")
            ms.append(mm.ravel()); ns.append(nn.ravel())
    return np.concatenate(ms), np.concatenate(ns)


def run_case(qpg, orc, fmt, M, N, K, seed, full=True, nsample=512):
    from bit_weight_quantized_qpack_gb300 import synth
    W = synth.laplace((N, K), 0.02, seed)
    rp, rgs, _ = orc.quantize_pack(fmt, W.numpy())
    X = synth.normal((M, K), 1.0, seed + 1).to(torch.bfloat16)
    pd = torch.from_numpy(rp).cuda()
    gd = None if rgs is None else torch.from_numpy(rgs.view(np.int16) if rgs.dtype == np.uint16 else rgs).cuda()
    Y = qpg.qgemm_prefill(fmt, pd, gd, N, K, X.cuda())
    torch.cuda.synchronize()
    Yg = Y.float().cpu().numpy()
    Xb = X.view(torch.int16).numpy().view(np.uint16)
    if full:
        ms, ns = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
        ms, ns = ms.ravel(), ns.ravel()
    else:
        rng = np.random.default_rng(seed)
        cm, cn = corner_tiles(M, N)
        ms = np.concatenate([rng.integers(0, M, nsample), cm])
        ns = np.concatenate([rng.integers(0, N, nsample), cn])
    order = np.argsort(ns, kind="stable")
    ms, ns = ms[order], ns[order]
    ref = orc.prefill_sample(fmt, N, K, rp, rgs, Xb, ms, ns, round_w=True)
    got = Yg[ms, ns].astype(np.float64)
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
    assert rel <= 2e-2, rel
    # per element: bf16 output rounding (at most 2^-8 relative) plus an accumulation term scaled like the GEMV
    # bound, 2e-5 * ||x_m|| * ||w'_n|| (fp32 accumulation error is absolute, so cancelled outputs need it)
    xn = np.linalg.norm(X.float().numpy().astype(np.float64), axis=1)
    wb = torch.from_numpy(orc.dequant(fmt, N, K, rp, rgs)).to(torch.bfloat16).double().numpy()
    wn = np.linalg.norm(wb, axis=1)
    bound = 2.0 ** -8 * np.abs(ref) + 2e-5 * xn[ms] * wn[ns]
    err = np.abs(got - ref)
    assert np.all(err <= bound), f"worst err/bound {np.max(err / bound):.3f}, norm rel {rel:.2e}"
    assert qpg.qpack_fetch_fault_flags() == 0
    return rel


def test_prefill_single_tile_int4(qpg, orc):
    run_case(qpg, orc, qpg.Q4G32, 128, 256, 64, 10)


@pytest.fixture(params=[0, 256, 224, 112, 128], ids=["tile-auto", "tile-pair", "tile-pair-224", "tile-112", "tile-128"])
def tile_rows(request, qpg):
    """The prefill tiling: chosen per launch (the default), forced to CTA pairs of 256 or 224 weight rows (one
    cluster of two CTAs sharing each tensor-core instruction), or forced to single CTAs of 112 or 128 weight rows."""
    qpg.qpack_set_option(qpg.OPT_PREFILL_TILE_ROWS, request.param)
    yield request.param
    qpg.qpack_set_option(qpg.OPT_PREFILL_TILE_ROWS, 0)


@pytest.mark.parametrize("name", ALL)
def test_prefill_ragged(qpg, orc, name, tile_rows):
    fmt = qpg.FORMATS[name]
    for i, (M, N, K) in enumerate([(128, 256, 256), (1, 300, 512), (130, 512, 256), (257, 260, 768)]):
        run_case(qpg, orc, fmt, M, N, K, 20 + i)


def test_prefill_tile_rows_option_values(qpg):
    L = qpg.lib()
    assert L.qpack_set_option(qpg.OPT_PREFILL_TILE_ROWS, 96) == -1
    assert L.qpack_set_option(99, 0) == -1
    for v in (256, 224, 112, 128, 0):
        assert L.qpack_set_option(qpg.OPT_PREFILL_TILE_ROWS, v) == 0


def test_prefill_config_int4_14336x4096(qpg, orc, tile_rows):
    """The prefill workload's INT4 matrix at M = 2048, with each tiling: 512 random outputs plus the four corner
    128 x 128 tiles."""
    run_case(qpg, orc, qpg.Q4G32, 2048, 14336, 4096, 7, full=False)


def test_prefill_config_q6s_4096x14336(qpg, orc, tile_rows):
    """The prefill workload's 6-bit matrix at M = 2048, with each tiling: 512 random outputs plus the four corner
    128 x 128 tiles (with 112-row tiles, single or in pairs, the last corner spans two CTAs and a ragged 64-row
    tile)."""
    run_case(qpg, orc, qpg.Q6S, 2048, 4096, 14336, 7, full=False)
