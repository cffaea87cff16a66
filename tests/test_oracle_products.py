"""Pins for the oracle's fp64-accumulated products y = dequant(W)·x (2/3/5/6-bit article §3.3 gemv_q3 semantics,
DBHOO-CIM article §3.3 fused dequant) and the prefill reference: one-hot columns, row sums, numpy/torch
library products on small random cases, and thread-count independence."""
import numpy as np
import pytest
import torch

ALL = ["Q4G32", "Q2S", "Q3S", "Q5S", "Q6S"]


def _packed(orc, fmt, N, K, seed):
    rng = np.random.default_rng(seed)
    W = rng.laplace(0, 0.02, (N, K)).astype(np.float32)
    packed, gs, _ = orc.quantize_pack(fmt, W)
    return packed, gs


@pytest.mark.parametrize("name", ALL)
def test_one_hot_gives_columns_exactly(orc, name):
    fmt = orc.FORMATS[name]
    N, K = 5, 512
    packed, gs = _packed(orc, fmt, N, K, 70 + fmt)
    deq = orc.dequant(fmt, N, K, packed, gs)
    for k in (0, 1, 255, 256, 511):
        x = np.zeros(K, np.uint16)
        x[k] = 0x3C00                       # fp16 1.0
        y = orc.gemv(fmt, N, K, packed, gs, x)
        assert np.array_equal(y, deq[:, k].astype(np.float64))
        x[k] = 0xC000                       # fp16 -2.0
        y = orc.gemv(fmt, N, K, packed, gs, x)
        assert np.array_equal(y, -2.0 * deq[:, k].astype(np.float64))


@pytest.mark.parametrize("name", ALL)
def test_against_numpy_matmul(orc, name):
    fmt = orc.FORMATS[name]
    N, K, M = 7, 768, 3
    packed, gs = _packed(orc, fmt, N, K, 80 + fmt)
    deq = orc.dequant(fmt, N, K, packed, gs).astype(np.float64)
    rng = np.random.default_rng(90)
    X = rng.standard_normal((M, K)).astype(np.float16)
    Y = orc.gemm(fmt, N, K, packed, gs, X.view(np.uint16))
    ref = X.astype(np.float64) @ deq.T
    scale = np.abs(X.astype(np.float64)) @ np.abs(deq).T
    assert np.all(np.abs(Y - ref) <= 1e-13 * scale + 1e-300)
    ones = np.full(K, 0x3C00, np.uint16)
    rs = orc.gemv(fmt, N, K, packed, gs, ones)
    assert np.allclose(rs, deq.sum(axis=1), rtol=1e-13, atol=1e-15)


def test_row_window_and_threads(orc):
    fmt = orc.Q5S
    N, K = 33, 512
    packed, gs = _packed(orc, fmt, N, K, 91)
    x = np.random.default_rng(92).standard_normal(K).astype(np.float16).view(np.uint16)
    full = orc.gemv(fmt, N, K, packed, gs, x, nthreads=1)
    assert np.array_equal(orc.gemv(fmt, N, K, packed, gs, x, nthreads=4), full)
    assert np.array_equal(orc.gemv(fmt, N, K, packed, gs, x, r0=10, nrows=7), full[10:17])


@pytest.mark.parametrize("name", ["Q4G32", "Q6S"])
def test_prefill_sample_against_torch(orc, name):
    fmt = orc.FORMATS[name]
    N, K, M = 9, 512, 6
    packed, gs = _packed(orc, fmt, N, K, 93)
    deq = orc.dequant(fmt, N, K, packed, gs)
    X = torch.randn(M, K, generator=torch.Generator().manual_seed(94)).to(torch.bfloat16)
    Xb = X.view(torch.int16).numpy().view(np.uint16)
    ms, ns = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    order = np.argsort(ns.ravel(), kind="stable")
    ms, ns = ms.ravel()[order], ns.ravel()[order]
    got = orc.prefill_sample(fmt, N, K, packed, gs, Xb, ms, ns, round_w=True)
    Wb = torch.from_numpy(deq).to(torch.bfloat16).double()
    ref = (X.double() @ Wb.T).numpy()[ms, ns]
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)
    got_unrounded = orc.prefill_sample(fmt, N, K, packed, gs, Xb, ms, ns, round_w=False)
    ref2 = (X.double() @ torch.from_numpy(deq).double().T).numpy()[ms, ns]
    assert np.allclose(got_unrounded, ref2, rtol=1e-12, atol=1e-12)
