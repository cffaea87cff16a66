"""GPU parity of the fused dequant-GEMV and the small-batch GEMM against the oracle's fp64 products:
max |y - y_ref| / (||w'_r|| * ||x||) <= 1e-4 (2/3/5/6-bit article §1.2 / §3.3; DBHOO-CIM article §3.3)."""
import numpy as np
import pytest
import torch

from conftest import gemv_bound_check, to_np_fp32

pytestmark = pytest.mark.gpu

ALL = ["Q4G32", "Q2S", "Q3S", "Q5S", "Q6S", "Q4G32H", "Q4G16", "Q4G32A"]


def case(orc, fmt, N, K, seed, b=0.02):
    from bit_weight_quantized_qpack_gb300 import synth
    W = synth.laplace((N, K), b, seed)
    rp, rgs, _ = orc.quantize_pack(fmt, W.numpy())
    return rp, rgs


def run_gemv(qpg, fmt, rp, rgs, N, K, x):
    pd = torch.from_numpy(rp).cuda()
    gd = None if rgs is None else torch.from_numpy(rgs.view(np.int16) if rgs.dtype == np.uint16 else rgs).cuda()
    y = qpg.qgemv(fmt, pd, gd, N, K, x.cuda())
    torch.cuda.synchronize()
    return y.cpu().numpy()


def shapes(name):
    s = [(1, 256), (3, 512), (4, 4096), (37, 4096 + 768), (130, 8192 + 256), (9, 12288)]
    if name in ("Q4G32", "Q4G32H", "Q4G16", "Q4G32A"):
        s += [(5, 96), (7, 4096 + 32)]
    return s


@pytest.mark.parametrize("name", ALL)
def test_gemv_tiles_and_ragged_tails(qpg, orc, name):
    from bit_weight_quantized_qpack_gb300 import synth
    fmt = qpg.FORMATS[name]
    for i, (N, K) in enumerate(shapes(name)):
        rp, rgs = case(orc, fmt, N, K, 300 + i)
        x = synth.normal((K,), 1.0, 400 + i, dtype=torch.float16)
        y = run_gemv(qpg, fmt, rp, rgs, N, K, x)
        xb = x.numpy().view(np.uint16)
        y_ref = orc.gemv(fmt, N, K, rp, rgs, xb)
        deq = orc.dequant(fmt, N, K, rp, rgs)
        gemv_bound_check(y, y_ref, deq, x.numpy().astype(np.float64)[None, :])
    assert qpg.qpack_fetch_fault_flags() == 0


@pytest.mark.parametrize("name", ALL)
def test_gemv_one_hot_columns(qpg, orc, name):
    fmt = qpg.FORMATS[name]
    N, K = 21, 4096 + 256
    rp, rgs = case(orc, fmt, N, K, 500)
    deq = orc.dequant(fmt, N, K, rp, rgs)
    for k in (0, 1, 31, 255, 4096, K - 1):
        x = torch.zeros(K, dtype=torch.float16)
        x[k] = 1.0
        y = run_gemv(qpg, fmt, rp, rgs, N, K, x)
        # the staged 1.0 is 32767 steps of fl(1/32767): exact to 2.4e-7, and the asymmetric formats subtract the
        # minimum term separately, so a small w' can carry the roundings of its two larger terms
        tol = 1e-6 * np.abs(deq[:, k]) + 1e-6 * np.abs(deq).max(axis=1)
        assert np.all(np.abs(y - deq[:, k]) <= tol)


@pytest.mark.parametrize("name", ALL)
def test_gemv_tiny_and_mixed_magnitude_activations(qpg, orc, name):
    """The bound scales with ||x||, so it must hold for activations near the fp16 subnormal range and for vectors
    whose entries span many binades (the staged activations carry one step per 16 activations)."""
    from bit_weight_quantized_qpack_gb300 import synth
    fmt = qpg.FORMATS[name]
    N, K = 19, 4096 + 512
    rp, rgs = case(orc, fmt, N, K, 620)
    deq = orc.dequant(fmt, N, K, rp, rgs)
    base = synth.normal((K,), 1.0, 621)
    mixed = base.clone()
    mixed[::7] *= 1e-4
    mixed[::11] *= 300.0
    for x32 in (base * 1e-5, base * 3e-7, mixed):
        x = x32.to(torch.float16)
        y = run_gemv(qpg, fmt, rp, rgs, N, K, x)
        y_ref = orc.gemv(fmt, N, K, rp, rgs, x.numpy().view(np.uint16))
        gemv_bound_check(y, y_ref, deq, x.numpy().astype(np.float64)[None, :])
    y = run_gemv(qpg, fmt, rp, rgs, N, K, torch.zeros(K, dtype=torch.float16))
    assert np.all(y == 0.0)


@pytest.mark.parametrize("name", ALL)
def test_gemv_rows_spread_over_all_sms(qpg, orc, name):
    """More rows than SMs but not a multiple of the tile: every CTA ends its row range with a ragged tile."""
    from bit_weight_quantized_qpack_gb300 import synth
    fmt = qpg.FORMATS[name]
    N, K = 1000, 4096
    rp, rgs = case(orc, fmt, N, K, 640)
    x = synth.normal((K,), 1.0, 641, dtype=torch.float16)
    y = run_gemv(qpg, fmt, rp, rgs, N, K, x)
    y_ref = orc.gemv(fmt, N, K, rp, rgs, x.numpy().view(np.uint16))
    deq = orc.dequant(fmt, N, K, rp, rgs)
    gemv_bound_check(y, y_ref, deq, x.numpy().astype(np.float64)[None, :])
    assert qpg.qpack_fetch_fault_flags() == 0


# (N, K): many rows per CTA with ragged stages; more than 256 rows per CTA (several partial-sum rounds); the
# 7B down-projection width; long rows (one row class, eight K parts); and the largest K the batch-1 path takes.
STAGE_SHAPES = [(1531, 4096), (45613, 256), (613, 11008), (311, 20480), (160, 32768)]


@pytest.mark.parametrize("name", ALL)
@pytest.mark.parametrize("shape", STAGE_SHAPES, ids=[f"{n}x{k}" for n, k in STAGE_SHAPES])
def test_gemv_stage_shapes(qpg, orc, name, shape):
    from bit_weight_quantized_qpack_gb300 import synth
    fmt = qpg.FORMATS[name]
    N, K = shape
    rp, rgs = case(orc, fmt, N, K, 660 + N % 97)
    x = synth.normal((K,), 1.0, 661 + K % 89, dtype=torch.float16)
    y = run_gemv(qpg, fmt, rp, rgs, N, K, x)
    y_ref = orc.gemv(fmt, N, K, rp, rgs, x.numpy().view(np.uint16), nthreads=8)
    deq = orc.dequant(fmt, N, K, rp, rgs)
    gemv_bound_check(y, y_ref, deq, x.numpy().astype(np.float64)[None, :])
    assert qpg.qpack_fetch_fault_flags() == 0


@pytest.mark.parametrize("name", ALL)
@pytest.mark.parametrize("K", [32768 + 256, 65536 + 4096 + 256])
def test_gemv_long_rows_in_k_splits(qpg, orc, name, K):
    """Batch-1 rows longer than one SM can stage beside the weight ring: the product is taken in K splits whose partial
    products are added to y in split order."""
    from bit_weight_quantized_qpack_gb300 import synth
    fmt = qpg.FORMATS[name]
    N = 157
    rp, rgs = case(orc, fmt, N, K, 680 + K % 13)
    x = synth.normal((K,), 1.0, 681, dtype=torch.float16)
    y = run_gemv(qpg, fmt, rp, rgs, N, K, x)
    y_ref = orc.gemv(fmt, N, K, rp, rgs, x.numpy().view(np.uint16), nthreads=8)
    deq = orc.dequant(fmt, N, K, rp, rgs)
    gemv_bound_check(y, y_ref, deq, x.numpy().astype(np.float64)[None, :])
    assert qpg.qpack_fetch_fault_flags() == 0


@pytest.mark.parametrize("name", ALL)
def test_gemv_large_activations_and_zero_rows(qpg, orc, name):
    from bit_weight_quantized_qpack_gb300 import synth
    fmt = qpg.FORMATS[name]
    N, K = 16, 2048
    W = synth.laplace((N, K), 0.02, 600)
    W[3] = 0
    rp, rgs, _ = orc.quantize_pack(fmt, W.numpy())
    x = (synth.normal((K,), 1.0, 601) * 30).to(torch.float16)   # |x| up to ~150
    y = run_gemv(qpg, fmt, rp, rgs, N, K, x)
    y_ref = orc.gemv(fmt, N, K, rp, rgs, x.numpy().view(np.uint16))
    deq = orc.dequant(fmt, N, K, rp, rgs)
    gemv_bound_check(y, y_ref, deq, x.numpy().astype(np.float64)[None, :])
    assert y[3] == 0.0 or abs(y[3]) < 1e-6


@pytest.mark.parametrize("name", ALL)
@pytest.mark.parametrize("M", [2, 3, 4, 6, 8, 11, 16])
def test_small_batch(qpg, orc, name, M):
    from bit_weight_quantized_qpack_gb300 import synth
    fmt = qpg.FORMATS[name]
    N, K = 45, 4096 + 512
    rp, rgs = case(orc, fmt, N, K, 700 + M)
    X = synth.normal((M, K), 1.0, 800 + M, dtype=torch.float16)
    pd = torch.from_numpy(rp).cuda()
    gd = None if rgs is None else torch.from_numpy(rgs.view(np.int16) if rgs.dtype == np.uint16 else rgs).cuda()
    Y = qpg.qgemm_small(fmt, pd, gd, N, K, X.cuda())
    torch.cuda.synchronize()
    Y_ref = orc.gemm(fmt, N, K, rp, rgs, X.numpy().view(np.uint16))
    deq = orc.dequant(fmt, N, K, rp, rgs)
    gemv_bound_check(Y.cpu().numpy(), Y_ref, deq, X.numpy().astype(np.float64))


# (N, K, M): rows whose staged activations do not fit one SM's shared memory beside the weight ring go in K splits
# (one launch per split, the later ones adding to Y), at the 70B MLP widths, with a ragged last split; at M = 2 the
# 8-rows-per-warp tiles are full (613 rows over the SMs) and ragged (211 rows), and 28672 takes a 3-way K split.
SMALL_BATCH_SHAPES = [(613, 8192, 16), (613, 8192, 5), (613, 8192, 2), (211, 28672, 16), (211, 28672, 3),
                      (211, 28672, 2), (97, 28672 + 256, 16), (97, 28672 + 256, 7)]


@pytest.mark.parametrize("name", ALL)
@pytest.mark.parametrize("shape", SMALL_BATCH_SHAPES, ids=[f"{n}x{k}xM{m}" for n, k, m in SMALL_BATCH_SHAPES])
def test_small_batch_groups(qpg, orc, name, shape):
    from bit_weight_quantized_qpack_gb300 import synth
    fmt = qpg.FORMATS[name]
    N, K, M = shape
    rp, rgs = case(orc, fmt, N, K, 720 + M + N % 7)
    X = synth.normal((M, K), 1.0, 820 + M, dtype=torch.float16)
    pd = torch.from_numpy(rp).cuda()
    gd = None if rgs is None else torch.from_numpy(rgs.view(np.int16) if rgs.dtype == np.uint16 else rgs).cuda()
    Y = qpg.qgemm_small(fmt, pd, gd, N, K, X.cuda())
    torch.cuda.synchronize()
    Y_ref = orc.gemm(fmt, N, K, rp, rgs, X.numpy().view(np.uint16), nthreads=8)
    deq = orc.dequant(fmt, N, K, rp, rgs)
    gemv_bound_check(Y.cpu().numpy(), Y_ref, deq, X.numpy().astype(np.float64))
    assert qpg.qpack_fetch_fault_flags() == 0


def test_small_batch_strided(qpg, orc):
    from bit_weight_quantized_qpack_gb300 import synth
    fmt = qpg.Q5S
    N, K, M = 19, 1024, 5
    rp, rgs = case(orc, fmt, N, K, 900)
    Xfull = synth.normal((M, K + 64), 1.0, 901, dtype=torch.float16)
    X = Xfull[:, :K]
    Yfull = torch.full((M, N + 13), 7.0, device="cuda")
    qpg.qgemm_small(fmt, torch.from_numpy(rp).cuda(), None, N, K, Xfull.cuda()[:, :K], Y=Yfull[:, :N])
    torch.cuda.synchronize()
    Yn = Yfull.cpu().numpy()
    assert np.all(Yn[:, N:] == 7.0)                         # nothing written past ldy's valid columns
    Y_ref = orc.gemm(fmt, N, K, rp, rgs, X.contiguous().numpy().view(np.uint16))
    gemv_bound_check(Yn[:, :N], Y_ref, orc.dequant(fmt, N, K, rp, rgs), X.numpy().astype(np.float64))


def test_config_int4_4096(qpg, orc):
    from bit_weight_quantized_qpack_gb300 import synth
    W = synth.normal_with_outliers((4096, 4096), 0.02, 0.001, 0.1, 0.5, seed=0)
    x = synth.normal((4096,), 1.0, seed=1, dtype=torch.float16)
    packed, gs = qpg.qpack_quantize_pack(qpg.Q4G32, W.cuda())
    y = qpg.qgemv(qpg.Q4G32, packed, gs, 4096, 4096, x.cuda())
    torch.cuda.synchronize()
    rp, rgs, _ = orc.quantize_pack(orc.Q4G32, W.numpy())
    y_ref = orc.gemv(orc.Q4G32, 4096, 4096, rp, rgs, x.numpy().view(np.uint16), nthreads=8)
    gemv_bound_check(y.cpu().numpy(), y_ref, orc.dequant(orc.Q4G32, 4096, 4096, rp, rgs),
                     x.numpy().astype(np.float64)[None, :])


def test_config_q3s_11008(qpg, orc):
    from bit_weight_quantized_qpack_gb300 import synth
    W = synth.laplace((11008, 4096), 0.015, seed=0)
    x = synth.normal((4096,), 1.0, seed=1, dtype=torch.float16)
    packed, _ = qpg.qpack_quantize_pack(qpg.Q3S, W.cuda())
    y = qpg.qgemv(qpg.Q3S, packed, None, 11008, 4096, x.cuda())
    torch.cuda.synchronize()
    rp, _, _ = orc.quantize_pack(orc.Q3S, W.numpy())
    y_ref = orc.gemv(orc.Q3S, 11008, 4096, rp, None, x.numpy().view(np.uint16), nthreads=8)
    gemv_bound_check(y.cpu().numpy(), y_ref, orc.dequant(orc.Q3S, 11008, 4096, rp, None),
                     x.numpy().astype(np.float64)[None, :])
    assert qpg.qpack_fetch_fault_flags() == 0


def test_weight_prefetch_dependent_chain(qpg, orc):
    """With QPACK_OPT_WEIGHT_PREFETCH each product may stream its weights before the previous kernel ends, but its
    activations must still come from the finished previous kernel: a chain where every x is produced by the
    kernel launched just before the product."""
    from bit_weight_quantized_qpack_gb300 import synth
    fmt, N, K = qpg.Q3S, 4096, 4096
    mats = []
    for i in range(3):
        W = synth.laplace((N, K), 0.02, 950 + i)
        rp, rgs, _ = orc.quantize_pack(fmt, W.numpy())
        mats.append((rp, torch.from_numpy(rp).cuda()))
    qpg.qpack_set_option(qpg.OPT_WEIGHT_PREFETCH, 1)
    try:
        x = synth.normal((K,), 1.0, 960, dtype=torch.float16).cuda()
        xs, ys = [], []
        for rp, pd in mats:
            xs.append(x.clone())
            y = qpg.qgemv(fmt, pd, None, N, K, x)
            ys.append(y)
            x = (y * 0.05).to(torch.float16)          # next activation depends on this product's output
        torch.cuda.synchronize()
    finally:
        qpg.qpack_set_option(qpg.OPT_WEIGHT_PREFETCH, 0)
    for (rp, _), xin, y in zip(mats, xs, ys):
        xb = xin.cpu().numpy().view(np.uint16)
        y_ref = orc.gemv(fmt, N, K, rp, None, xb, nthreads=8)
        gemv_bound_check(y.cpu().numpy(), y_ref, orc.dequant(fmt, N, K, rp, None), xin.cpu().numpy().astype(np.float64)[None, :])


@pytest.mark.parametrize("seed", range(12))
def test_random_differential_sweep(qpg, orc, seed):
    """Differential sweep with fixed seeds: a random format, shape and batch per case (rows 1..3000, K up to ~12K in
    whole groups or super-blocks, M 1..16, Laplace scale over three decades); the GPU quantizes and packs (bytes
    compared with the oracle's) and multiplies (products within the bound)."""
    from bit_weight_quantized_qpack_gb300 import synth
    rng = np.random.default_rng(9000 + seed)
    name = ALL[int(rng.integers(len(ALL)))]
    fmt = qpg.FORMATS[name]
    blk = 32 if name.startswith("Q4G") else 256
    N = int(rng.integers(1, 3001))
    K = blk * int(rng.integers(1, 12288 // blk + 1))
    if name.startswith("Q4G") and rng.random() < 0.5:
        K = 64 * max(1, K // 64)
    M = int(rng.integers(1, 17))
    b = float(10.0 ** rng.uniform(-3, 0))
    W = synth.laplace((N, K), b, 9100 + seed)
    p, g = qpg.qpack_quantize_pack(fmt, W.cuda())
    rp, rgs, _ = orc.quantize_pack(fmt, W.numpy())
    torch.cuda.synchronize()
    assert np.array_equal(p.cpu().numpy(), rp), name
    if rgs is not None:
        assert np.array_equal(g.cpu().numpy().view(np.uint8), rgs.view(np.uint8)), name
    X = synth.normal((M, K), float(10.0 ** rng.uniform(-2, 2)), 9200 + seed, dtype=torch.float16)
    Y = qpg.qgemm_small(fmt, p, g, N, K, X.cuda()) if M > 1 else qpg.qgemv(fmt, p, g, N, K, X[0].cuda())[None, :]
    torch.cuda.synchronize()
    Y_ref = orc.gemm(fmt, N, K, rp, rgs, X.numpy().view(np.uint16), nthreads=8)
    deq = orc.dequant(fmt, N, K, rp, rgs)
    gemv_bound_check(Y.cpu().numpy(), Y_ref, deq, X.numpy().astype(np.float64))
    assert qpg.qpack_fetch_fault_flags() == 0
