"""CPU-side checks of the C ABI: the library loads, exports every function include/qpack.h declares, and its
host-only entry points (layout, status strings, argument validation that rejects before any launch) behave."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def qp():
    from bit_weight_quantized_qpack_gb300 import _build
    _build.build()
    import bit_weight_quantized_qpack_gb300 as qp
    qp.lib()
    return qp


def declared_functions():
    names = []
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            text = open(os.path.join(ROOT, "include", f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?(?:int|void|char\s*\*|const char\s*\*)\s*\*?\s*(\w+)\s*\(",
                                text, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(qp):
    names = declared_functions()
    assert {"qpack_quantize", "qpack_pack", "qgemv", "qgemm_small", "qgemm_prefill"} <= set(names)
    L = ctypes.CDLL(qp.LIB_PATH)
    for n in names:
        assert hasattr(L, n), f"{n} declared in include/ but not exported"


def test_layout_matches_oracle(qp, orc):
    for name, fmt in qp.FORMATS.items():
        for N, K in ((1, 256), (7, 4096), (11008, 4096), (4096, 11008), (3, 28672)):
            a = qp.layout(fmt, N, K)
            b = orc.layout(fmt, N, K)
            assert a["row_stride"] == b["row_stride"] and a["packed_bytes"] == b["packed_bytes"]
            assert a["scale_stride"] == b["scale_stride"] and a["scale_bytes"] == b["scale_bytes"]
            assert a["weight_bytes"] == a["packed_bytes"] + a["scale_bytes"]


def test_config_byte_counts(qp):
    # 4096x4096 INT4: 8,388,608 code bytes + 2,097,152 scale bytes; 11008x4096 3-bit: 19,374,080 bytes
    assert qp.layout(qp.Q4G32, 4096, 4096)["weight_bytes"] == 10_485_760
    assert qp.layout(qp.Q3S, 11008, 4096)["weight_bytes"] == 19_374_080
    # padded rows for K = 11008
    assert qp.layout(qp.Q2S, 1, 11008)["row_stride"] == 3616
    assert qp.layout(qp.Q3S, 1, 11008)["row_stride"] == 4736
    assert qp.layout(qp.Q6S, 1, 11008)["row_stride"] == 9040


def test_argument_validation_rejects_before_launch(qp):
    L = qp.lib()
    P = ctypes.c_void_p
    good = P(1 << 20)          # never dereferenced: every call below fails validation first
    odd = P((1 << 20) + 4)
    SHAPE, ALIGN, ARG = -2, -3, -1
    assert L.qgemv(qp.Q4G32, good, good, 8, 48, good, good, None) == SHAPE
    assert L.qgemv(qp.Q3S, good, None, 8, 4096 + 32, good, good, None) == SHAPE
    assert L.qgemv(qp.Q3S, odd, None, 8, 4096, good, good, None) == ALIGN
    assert L.qgemv(qp.Q4G32, good, None, 8, 4096, good, good, None) == ARG
    assert L.qgemv(qp.Q4G32A, good, None, 8, 4096, good, good, None) == ARG
    assert L.qpack_pack(qp.Q4G32A, 8, 4096, good, None, None, None, None, None, good, good, None) == ARG
    assert L.qgemv(9, good, good, 8, 4096, good, good, None) == ARG
    assert L.qgemv(qp.Q3S, good, None, 8, 4096, odd, good, None) == ALIGN
    assert L.qgemm_small(qp.Q5S, good, None, 8, 4096, 17, good, 4096, good, 8, None) == SHAPE
    assert L.qgemm_small(qp.Q5S, good, None, 8, 4096, 2, good, 4095, good, 8, None) == SHAPE
    assert L.qgemm_small(qp.Q5S, good, None, 8, 4096, 2, good, 4100, good, 8, None) == ALIGN
    assert L.qgemm_prefill(qp.Q4G32, good, good, 8, 96, 4, good, 96, good, 8, None) == SHAPE
    assert L.qpack_quantize_pack(qp.Q2S, good, 7, 8, 256, good, None, None, None) == ARG
    assert L.qpack_quantize_pack(qp.Q2S, odd, 0, 8, 256, good, None, None, None) == ALIGN
    assert L.qpack_dequant(qp.Q6S, -1, 256, good, None, good, None) == ARG
    assert L.qpack_kv_quantize(good, 48, good, good, None) == SHAPE
    assert L.qpack_kv_quantize(good, 64, None, good, None) == ARG
    assert L.qpack_kv_quantize(odd, 64, good, good, None) == ALIGN
    assert L.qpack_kv_dequant(good, good, 64, odd, None) == ALIGN
    assert L.qpack_kv_dequant(good, good, -32, good, None) == SHAPE
    # empty problems are accepted and launch nothing
    assert L.qpack_kv_quantize(good, 0, good, good, None) == 0
    assert L.qpack_kv_dequant(good, good, 0, good, None) == 0
    assert L.qgemv(qp.Q3S, good, None, 0, 4096, good, good, None) == 0
    assert L.qgemm_small(qp.Q3S, good, None, 8, 4096, 0, good, 4096, good, 8, None) == 0
    # options: an unknown option or tiling is refused before any device query; the five tilings are accepted (on a
    # host without a GPU the device query behind them then fails with ERR_CUDA)
    assert L.qpack_set_option(99, 0) == ARG
    for v in (96, 64, 240, -1):
        assert L.qpack_set_option(qp.OPT_PREFILL_TILE_ROWS, v) == ARG
    for v in (112, 128, 224, 256, 0):          # ends on the default, so later calls on a GPU host are unaffected
        assert L.qpack_set_option(qp.OPT_PREFILL_TILE_ROWS, v) in (0, -5)


def test_status_strings(qp):
    for s in (0, -1, -2, -3, -4, -5, -6, 12345):
        assert qp.qpack_status_string(s)
    assert qp.qpack_version() >= 10000


def test_binding_checks_types_and_sizes_before_any_launch(qp):
    """The Python binding rejects tensors whose element type, size or layout the C ABI cannot see (it takes bare
    pointers) before anything reaches the device; CPU tensors suffice since the checks come first."""
    import pytest
    import torch
    N, K = 8, 256
    L = qp.layout(qp.Q3S, N, K)
    packed = torch.zeros((N, L["row_stride"]), dtype=torch.uint8)
    x16 = torch.zeros(K, dtype=torch.float16)
    with pytest.raises(qp.QpackError, match="x: expected torch.float16"):
        qp.qgemv(qp.Q3S, packed, None, N, K, torch.zeros(K, dtype=torch.float32))
    with pytest.raises(qp.QpackError, match="packed"):
        qp.qgemv(qp.Q3S, packed[: N - 1], None, N, K, x16)
    with pytest.raises(qp.QpackError, match="group_scales: required"):
        qp.qgemv(qp.Q4G32, torch.zeros((N, K // 2), dtype=torch.uint8), None, N, K, x16)
    with pytest.raises(qp.QpackError, match="y: expected"):
        qp.qgemv(qp.Q3S, packed, None, N, K, x16, torch.zeros(N, dtype=torch.float16))
    with pytest.raises(qp.QpackError, match="X: expected torch.bfloat16"):
        qp.qgemm_prefill(qp.Q3S, packed, None, N, K, torch.zeros((4, K), dtype=torch.float16))
    with pytest.raises(qp.QpackError, match="X: expected a row-major matrix"):
        qp.qgemm_small(qp.Q3S, packed, None, N, K, torch.zeros((K, 4), dtype=torch.float16).t())
    with pytest.raises(qp.QpackError, match="v: expected torch.float16"):
        qp.qpack_kv_quantize(torch.zeros(64, dtype=torch.float32))
    with pytest.raises(qp.QpackError, match="W: expected float32"):
        qp.qpack_quantize_pack(qp.Q3S, torch.zeros((N, K), dtype=torch.int8))
    with pytest.raises(qp.QpackError, match="CUDA tensors"):
        qp.qgemv(qp.Q3S, packed, None, N, K, x16)
