"""Worst-case activations for the decode products' 16-bit activation staging.

The decode kernels turn each fp16 activation into a 16-bit integer before the integer multiply-adds. The pages take
activations in floating point (the 2/3/5/6-bit article, lpnh.cn/news/2857666, §3.3 multiplies codes with float x;
the DBHOO-CIM article, pwwt.cn/news/4452170, §2.2 keeps activations in fp16/fp32), so the rounding of x must stay
inside the product bound max |y - y_ref| / (||w'_r|| ||x||) <= 1e-4 for every finite fp16 x, not just for random x.

The worst case for a staging with step h per block of n activations is a weight row of one sign, a block holding
one large entry and n - 1 entries that each lose half a step in the same direction: the error approaches
(n - 1) * h/2 * |w| against ||w|| ||x||. Two input families reach it:

* BLOCK32: the family that breaks a power-of-two step per 32 activations (step 2^-14 for a unit whose largest entry
  is 1.0): one entry 1.0 and 31 entries 1.5 * 2^-14 per 32, which round to 2 * 2^-14. Against a constant positive
  row it gives 1.67e-4 (the CPU test below emulates that staging exactly and checks that it exceeds 1e-4).
* HALF16: the family aimed at the library's staging (step m / 32767 per 16 activations, m = the half's largest
  |x|): one entry m and 15 fp16 values chosen to sit just below a half-step of that grid, with the signs of the
  target weight row. The CPU test emulates the staging exactly and checks that it comes within 5% of the bound
  sqrt(15) / 65534 (a constant row reaches sqrt(15) / 4 = 96.8% of it). For m whose grid step is close to the fp16
  spacing of the small values (tiny m) no fp16 value sits near a half-step, so the magnitudes used are ones where
  the family is adversarial.

The GPU tests run both families through the C ABI for every format at M = 1, 2, 8 and 16, at K = 4096 (the
register-staged batch-1 path for the chunk widths of every format) and K = 12288 (shared-memory staging), and check
the product bound against the oracle's fp64 sums. A last test covers non-finite activations: every output of the
affected activation row is nan and the fault word reports it.
"""
import numpy as np
import pytest
import torch

from conftest import gemv_bound_check

ALL = ["Q4G32", "Q2S", "Q3S", "Q5S", "Q6S", "Q4G32H", "Q4G16", "Q4G32A"]
INV32767 = np.float32(1.0) / np.float32(32767.0)


def fp16_values(x):
    return np.asarray(x, np.float16).astype(np.float64)


def stage_block32_pow2(x):
    """Exact emulation of a power-of-two staging step per 32 activations: E with max|x| 2^E in [2^14, 2^15),
    xi = rint(x 2^E) (half to even). Returns the staged values xi 2^-E."""
    x = np.asarray(x, np.float64).reshape(-1, 32)
    out = np.zeros_like(x)
    for u in range(x.shape[0]):
        m = np.abs(x[u]).max()
        if m == 0:
            continue
        E = 14 - int(np.floor(np.log2(m)))
        out[u] = np.rint(x[u] * 2.0 ** E) * 2.0 ** -E
    return out.reshape(-1)


def stage_half16(x16):
    """Exact emulation of the library's staging (fp32 arithmetic as the kernel does it): per 16 activations
    sigma = fl(m * fl(1/32767)), inv = fl(1/sigma), xi = rint(x * inv) with the product rounded once (a fused
    multiply-add; in fp64 the product of an fp16 and an fp32 value is exact). Returns xi * sigma in fp64."""
    x = np.asarray(x16, np.float16).astype(np.float32).reshape(-1, 16)
    out = np.zeros(x.shape, np.float64)
    for h in range(x.shape[0]):
        m = np.float32(np.abs(x[h]).max())
        if m == 0:
            continue
        sigma = np.float32(m * INV32767)
        inv = np.float32(np.float32(1.0) / sigma)
        xi = np.rint(x[h].astype(np.float64) * np.float64(inv))
        out[h] = xi * np.float64(sigma)
    return out.reshape(-1)


def block32_family(K, signs):
    """One entry 1.0 at a rotating position and 31 entries 1.5 * 2^-14 per 32 activations, with the given signs."""
    x = np.full(K, 1.5 * 2.0 ** -14)
    for u in range(K // 32):
        x[32 * u + (u * 7) % 32] = 1.0
    return fp16_values(x * signs)


def half16_small_value(m):
    """The fp16 value v in (0, m / 8) that the half16 staging of a half with maximum m rounds down the most."""
    m32 = np.float32(m)
    sigma = np.float32(m32 * INV32767)
    inv = np.float32(np.float32(1.0) / sigma)
    hi = float(m) / 8
    bits = np.arange(1, np.float16(hi).view(np.uint16) + 1, dtype=np.uint16)
    v = bits.view(np.float16).astype(np.float32)
    xi = np.rint(v.astype(np.float64) * np.float64(inv))
    err = v.astype(np.float64) - xi * np.float64(sigma)
    return float(v[int(np.argmax(err))])


def half16_family(K, signs, m=1.0):
    """Per 16 activations: one entry m at a rotating position, 15 entries at the worst-rounded value, signs given."""
    a = half16_small_value(m)
    x = np.full(K, a)
    for h in range(K // 16):
        x[16 * h + (h * 5) % 16] = m
    return fp16_values(x * signs)


def quantized_rows(orc, fmt, K, n_random=3, seed=0):
    """Row 0 constant positive (every format quantizes it to a constant row), rows 1.. Laplace(0, 0.02)."""
    from bit_weight_quantized_qpack_gb300 import synth
    W = np.empty((1 + n_random, K), np.float32)
    W[0] = 0.02
    W[1:] = synth.laplace((n_random, K), 0.02, seed).numpy()
    rp, rgs, _ = orc.quantize_pack(fmt, W)
    deq = orc.dequant(fmt, W.shape[0], K, rp, rgs).astype(np.float64)
    return W.shape[0], rp, rgs, deq


def ratio(y, y_ref, deq_row, x):
    return abs(y - y_ref) / (np.linalg.norm(deq_row) * np.linalg.norm(x))


def test_families_are_adversarial(orc):
    """CPU: the exact emulations show that BLOCK32 breaks a power-of-two step per 32 (1.67e-4 > 1e-4) while the
    library's staging keeps it small, and that HALF16 drives the library's staging to within 5% of its bound."""
    K = 4096
    N, rp, rgs, deq = quantized_rows(orc, orc.Q4G32, K)
    w = deq[0]
    assert np.all(w == w[0]) and w[0] > 0                  # constant positive row (all codes clamp to 7)
    xb = block32_family(K, np.ones(K))
    y = w @ xb
    r_old = ratio(w @ stage_block32_pow2(xb), y, w, xb)
    r_new = ratio(w @ stage_half16(xb), y, w, xb)
    assert 1.6e-4 < r_old < 1.7e-4
    assert r_new < 1e-6
    bound = np.sqrt(15) / 65534
    for m in (1.0, 0.125, 300.0):
        xh = half16_family(K, np.ones(K), m)
        r = ratio(w @ stage_half16(xh), w @ xh, w, xh)
        assert 0.95 * bound < r <= 1.02 * bound, (m, r, bound)
    # signs aligned with a Laplace row: the emulated error still stays inside the bound
    xs = half16_family(K, np.where(deq[1] < 0, -1.0, 1.0))
    assert ratio(deq[1] @ stage_half16(xs), deq[1] @ xs, deq[1], xs) <= 1.02 * bound


def _to_dev(qpg, rp, rgs):
    pd = torch.from_numpy(rp).cuda()
    gd = None if rgs is None else torch.from_numpy(rgs.view(np.int16) if rgs.dtype == np.uint16 else rgs).cuda()
    return pd, gd


@pytest.mark.gpu
@pytest.mark.parametrize("name", ALL)
@pytest.mark.parametrize("K", [4096, 12288])
@pytest.mark.parametrize("M", [1, 2, 8, 16])
def test_adversarial_activations_within_bound(qpg, orc, name, K, M):
    fmt = qpg.FORMATS[name]
    N, rp, rgs, deq = quantized_rows(orc, fmt, K, seed=1000 + K % 7)
    rows = []
    for m in range(M):
        target = m % N                                     # activation row m aims at weight row m mod N
        signs = np.where(deq[target] < 0, -1.0, 1.0)
        fam = half16_family if m % 2 == 0 else block32_family
        rows.append(fam(K, signs) if fam is block32_family else fam(K, signs, [1.0, 0.3, 40.0][m % 3]))
    X = np.stack(rows)
    Xt = torch.from_numpy(X.astype(np.float16))
    pd, gd = _to_dev(qpg, rp, rgs)
    if M == 1:
        Y = qpg.qgemv(fmt, pd, gd, N, K, Xt[0].cuda())[None, :]
    else:
        Y = qpg.qgemm_small(fmt, pd, gd, N, K, Xt.cuda())
    torch.cuda.synchronize()
    Y_ref = orc.gemm(fmt, N, K, rp, rgs, Xt.numpy().view(np.uint16))
    worst = gemv_bound_check(Y.cpu().numpy(), Y_ref, deq, X)
    assert worst <= 7e-5, worst                           # the staging's own bound is 6.0e-5
    assert qpg.qpack_fetch_fault_flags() == 0


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["Q4G32", "Q3S", "Q5S", "Q2S"])
@pytest.mark.parametrize("K", [4096, 12288])
def test_nonfinite_activation_policy(qpg, orc, name, K):
    """An inf or nan activation: every output of its activation row is nan (the IEEE sum would be nan or +-inf;
    the call does not pick one) and QPACK_FAULT_NONFINITE_X is set; the other activation rows are unaffected."""
    from bit_weight_quantized_qpack_gb300 import synth
    fmt = qpg.FORMATS[name]
    N = 37
    W = synth.laplace((N, K), 0.02, 1100)
    rp, rgs, _ = orc.quantize_pack(fmt, W.numpy())
    deq = orc.dequant(fmt, N, K, rp, rgs)
    pd, gd = _to_dev(qpg, rp, rgs)
    assert qpg.qpack_fetch_fault_flags() == 0
    for bad in (float("inf"), float("-inf"), float("nan")):
        X = synth.normal((3, K), 1.0, 1101, dtype=torch.float16)
        X[1, K - 5] = bad
        y = qpg.qgemv(fmt, pd, gd, N, K, X[1].cuda())
        torch.cuda.synchronize()
        assert torch.isnan(y).all()
        assert qpg.qpack_fetch_fault_flags() & qpg.FAULT_NONFINITE_X
        Y = qpg.qgemm_small(fmt, pd, gd, N, K, X.cuda())
        torch.cuda.synchronize()
        Yn = Y.cpu().numpy()
        assert np.isnan(Yn[1]).all()
        assert qpg.qpack_fetch_fault_flags() & qpg.FAULT_NONFINITE_X
        good = X[[0, 2]]
        Y_ref = orc.gemm(fmt, N, K, rp, rgs, good.numpy().view(np.uint16))
        gemv_bound_check(Yn[[0, 2]], Y_ref, deq, good.numpy().astype(np.float64))
    assert qpg.qpack_fetch_fault_flags() == 0
