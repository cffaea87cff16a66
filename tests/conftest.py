import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built libqpack")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def read_golden(name):
    """Non-comment lines of a golden fixture, split into tokens."""
    rows = []
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append(line.split())
    return rows


def kv(tokens):
    """Parse 'key=value' tokens into a dict of floats."""
    out = {}
    for t in tokens:
        if "=" in t:
            k, v = t.split("=", 1)
            out[k] = float(v)
    return out


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.lib()
    return oracle


@pytest.fixture(scope="session")
def qpg():
    """The built CUDA library on cuda:0 (GPU tests only)."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_weight_quantized_qpack_gb300 import _build
    _build.build()
    import bit_weight_quantized_qpack_gb300 as qp
    qp.lib()
    return qp


def to_np_fp32(t):
    """Exact fp32 numpy copy of a CPU/GPU tensor of dtype fp32/fp16/bf16."""
    import torch
    return t.detach().to("cpu", torch.float32).numpy()


def gemv_bound_check(y_gpu, y_ref, deq_rows, X, tol=1e-4):
    """max |y - y_ref| / (||w'_r|| * ||x_m||) <= tol over every (m, r); returns the worst ratio."""
    import numpy as np
    deq = np.asarray(deq_rows, np.float64)
    Xd = np.atleast_2d(np.asarray(X, np.float64))
    bound = tol * np.outer(np.linalg.norm(Xd, axis=1), np.linalg.norm(deq, axis=1))
    # An all-zero dequantized row makes the ratio 0/0; there the output must be zero up to 1e-9 * ||x||
    # (an INT4 zero group keeps the 1e-12 scale floor, so offset cancellation may leave ~1e-13).
    zero_rows = np.linalg.norm(deq, axis=1) == 0
    bound[:, zero_rows] = 1e-9 * np.linalg.norm(Xd, axis=1)[:, None]
    err = np.abs(np.atleast_2d(np.asarray(y_gpu, np.float64)) - np.atleast_2d(y_ref))
    ratio = err / np.maximum(bound, 1e-300) * tol
    assert np.all(err <= bound), f"worst |err|/(||w||*||x||) = {ratio.max():.3e} > {tol}"
    return float(ratio.max())
