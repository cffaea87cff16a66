"""qpack oracle — TEST INFRASTRUCTURE ONLY.

Python (ctypes + numpy) front of the plain C++ oracle in ``qpack_oracle.cpp``: the five weight formats'
quantizers, packers, unpackers, dequantization and fp64-accumulated products, and the 8-bit KV-cache quantizer and
dequantizer (P1 §4.1; the Mix-Quant article, lnrk.cn/news/34246, §2.3), written from the source pages
(P1 = the 2/3/5/6-bit quantization article, lpnh.cn/news/2857666; P2 = the DBHOO-CIM INT4 CPU inference
article, pwwt.cn/news/4452170), with the readings of what they leave open stated in ``qpack_oracle.cpp``.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may import this package.
It never imports the CUDA package and the CUDA package never imports it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

Q4G32, Q2S, Q3S, Q5S, Q6S, Q4G32H, Q4G16, Q4G32A = 0, 1, 2, 3, 4, 5, 6, 7
FORMATS = {"Q4G32": Q4G32, "Q2S": Q2S, "Q3S": Q3S, "Q5S": Q5S, "Q6S": Q6S, "Q4G32H": Q4G32H, "Q4G16": Q4G16,
           "Q4G32A": Q4G32A}
FLAG_RANGE = 1

# (bits, sub-blocks, weights per sub-block, Lmax, asymmetric, bytes per super-block) — P1 §2.3 byte table (Q5S:
# 8 sub-blocks of 32 with 6-bit scale and minimum; Q2S: 4-bit scale and minimum; Q3S / Q6S symmetric).
SB = {
    Q2S: (2, 16, 16, 15, True, 84),
    Q3S: (3, 16, 16, 63, False, 110),
    Q5S: (5, 8, 32, 63, True, 176),
    Q6S: (6, 16, 16, 127, False, 210),
}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qpack_oracle.cpp")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle_qpack.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle shared library (plain g++, no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call([
            "g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
            "-pthread", "-o", tmp, _SRC,
        ])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
            sigs = {
                "orc_f32_to_f16": [P, P, I64], "orc_f16_to_f32": [P, P, I64],
                "orc_f32_to_bf16": [P, P, I64], "orc_bf16_to_f32": [P, P, I64],
                "orc_run_pack": [P, I, I64, P], "orc_run_unpack": [P, I, I64, P],
                "orc_layout": [I, I64, I64, P],
                "orc_quantize": [I, P, I64, I64, P, P, P, P, P, P],
                "orc_pack": [I, I64, I64, P, P, P, P, P, P, P, P],
                "orc_unpack": [I, I64, I64, P, P, P, P, P, P, P, P],
                "orc_dequant_rows": [I, I64, I64, P, P, I64, I64, P],
                "orc_gemm_rows": [I, I64, I64, P, P, I64, P, I64, I64, I64, P, I],
                "orc_prefill_sample": [I, I64, I64, P, P, P, I64, I64, P, P, I64, I, P],
                "orc_kv_quantize": [P, I64, P, P],
                "orc_kv_dequant": [P, P, I64, P],
            }
            for name, args in sigs.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = I if name not in ("orc_f32_to_f16", "orc_f16_to_f32", "orc_f32_to_bf16",
                                               "orc_bf16_to_f32", "orc_run_pack", "orc_run_unpack") else None
            _lib = L
    return _lib


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------------------------------------------------
# converters
# ---------------------------------------------------------------------------------------------------------
def f32_to_f16_bits(x):
    x = _c(x, np.float32); y = np.empty(x.shape, np.uint16)
    lib().orc_f32_to_f16(_p(x), _p(y), x.size); return y


def f16_bits_to_f32(h):
    h = _c(h, np.uint16); y = np.empty(h.shape, np.float32)
    lib().orc_f16_to_f32(_p(h), _p(y), h.size); return y


def f32_to_bf16_bits(x):
    x = _c(x, np.float32); y = np.empty(x.shape, np.uint16)
    lib().orc_f32_to_bf16(_p(x), _p(y), x.size); return y


def bf16_bits_to_f32(h):
    h = _c(h, np.uint16); y = np.empty(h.shape, np.float32)
    lib().orc_bf16_to_f32(_p(h), _p(y), h.size); return y


# ---------------------------------------------------------------------------------------------------------
# generic cross-byte packers (P1 §2.2)
# ---------------------------------------------------------------------------------------------------------
def run_pack(fields, width):
    """n fields of `width` bits laid end to end, least significant bit first (field i at bits width*i..): P1 §2.2's
    cross-byte packing (width 3: 8 codes in 3 bytes; width 6: 4 fields in 3 bytes; width 5: 8 codes in 5 bytes)."""
    f = _c(fields, np.uint8); n = f.size; p = np.empty((width * n + 7) // 8, np.uint8)
    lib().orc_run_pack(_p(f), int(width), n, _p(p)); return p


def run_unpack(packed, width, n):
    p = _c(packed, np.uint8); f = np.empty(n, np.uint8)
    lib().orc_run_unpack(_p(p), int(width), int(n), _p(f)); return f


# ---------------------------------------------------------------------------------------------------------
# formats
# ---------------------------------------------------------------------------------------------------------
def _gs(fmt, group_scales):
    """The INT4 group-scale array in its stored type: fp32 (Q4G32) or fp16 bit patterns (Q4G32H)."""
    if group_scales is None:
        return None
    return _c(group_scales, np.uint16 if fmt == Q4G32H else np.float32)


def _parts(fmt, N, K):
    q = np.zeros((N, K), np.int8)
    parts = dict(q=q, gscale=None, sub_scale=None, sub_min=None, d=None, dmin=None)
    if fmt in (Q4G32, Q4G16, Q4G32A):   # Q4G32A: (scale, zero point) pairs, [N, K/16]
        parts["gscale"] = np.zeros((N, K // (32 if fmt == Q4G32 else 16)), np.float32)
    elif fmt == Q4G32H:
        parts["d"] = np.zeros((N, K // 32), np.uint16)          # the fp16 group scales
    else:
        bits, nsub, sublen, lmax, asym, nbytes = SB[fmt]
        nb = K // 256
        parts["sub_scale"] = np.zeros((N, nb * nsub), np.uint8)
        parts["d"] = np.zeros((N, nb), np.uint16)
        if asym:
            parts["sub_min"] = np.zeros((N, nb * nsub), np.uint8)
            parts["dmin"] = np.zeros((N, nb), np.uint16)
    return parts


def layout(fmt, N, K):
    """dict(row_stride, packed_bytes, scale_stride, scale_bytes, block_bytes); raises ValueError on bad K."""
    out = np.zeros(5, np.int64)
    rc = lib().orc_layout(int(fmt), int(N), int(K), _p(out))
    if rc != 0:
        raise ValueError(f"shape N={N} K={K} not accepted by format {fmt}")
    return dict(row_stride=int(out[0]), packed_bytes=int(out[1]), scale_stride=int(out[2]),
                scale_bytes=int(out[3]), block_bytes=int(out[4]))


def quantize(fmt, W):
    """Quantize fp32 W [N, K] into unpacked parts: dict(q, gscale | sub_scale, sub_min, d, dmin, flags); Q4G32H keeps
    its fp16 group scales in d [N, K/32]."""
    W = _c(W, np.float32)
    N, K = W.shape
    parts = _parts(fmt, N, K)
    q = parts["q"]
    rc = lib().orc_quantize(int(fmt), _p(W), N, K, _p(q), _p(parts["gscale"]), _p(parts["sub_scale"]),
                            _p(parts["sub_min"]), _p(parts["d"]), _p(parts["dmin"]))
    if rc < 0:
        raise ValueError(f"orc_quantize rc={rc}")
    parts["flags"] = rc
    return parts


def pack(fmt, N, K, parts):
    """Pack unpacked parts -> (packed uint8 [N, row_stride], group scales [N, S] (fp32 for Q4G32, fp16 bit patterns
    for Q4G32H) or None)."""
    lay = layout(fmt, N, K)
    packed = np.zeros((N, lay["row_stride"]), np.uint8)
    gs = None
    if fmt in (Q4G32, Q4G16, Q4G32A):
        gs = np.zeros((N, lay["scale_stride"]), np.float32)
    elif fmt == Q4G32H:
        gs = np.zeros((N, lay["scale_stride"]), np.uint16)
    g = lambda k, dt: None if parts.get(k) is None else _c(parts[k], dt)
    rc = lib().orc_pack(int(fmt), N, K, _p(_c(parts["q"], np.int8)), _p(g("gscale", np.float32)),
                        _p(g("sub_scale", np.uint8)), _p(g("sub_min", np.uint8)), _p(g("d", np.uint16)),
                        _p(g("dmin", np.uint16)), _p(packed), _p(gs))
    if rc != 0:
        raise ValueError(f"orc_pack rc={rc}")
    return packed, gs


def unpack(fmt, N, K, packed, group_scales=None):
    packed = _c(packed, np.uint8)
    gs = _gs(fmt, group_scales)
    parts = _parts(fmt, N, K)
    q = parts["q"]
    rc = lib().orc_unpack(int(fmt), N, K, _p(packed), _p(gs), _p(q), _p(parts["gscale"]), _p(parts["sub_scale"]),
                          _p(parts["sub_min"]), _p(parts["d"]), _p(parts["dmin"]))
    if rc != 0:
        raise ValueError(f"orc_unpack rc={rc}")
    return parts


def dequant(fmt, N, K, packed, group_scales=None, r0=0, nrows=None):
    """fp32 dequantized rows [r0, r0 + nrows) of a packed matrix."""
    nrows = N - r0 if nrows is None else nrows
    out = np.zeros((nrows, K), np.float32)
    gs = _gs(fmt, group_scales)
    rc = lib().orc_dequant_rows(int(fmt), N, K, _p(_c(packed, np.uint8)), _p(gs), r0, nrows, _p(out))
    if rc != 0:
        raise ValueError(f"orc_dequant_rows rc={rc}")
    return out


def gemm(fmt, N, K, packed, group_scales, X_f16_bits, r0=0, nrows=None, nthreads=1):
    """fp64 Y [M, nrows] = X · dequant(W)[r0:r0+nrows]ᵀ; X given as fp16 bit patterns [M, K]."""
    X = _c(X_f16_bits, np.uint16)
    if X.ndim == 1:
        X = X[None, :]
    M = X.shape[0]
    nrows = N - r0 if nrows is None else nrows
    Y = np.zeros((M, nrows), np.float64)
    gs = _gs(fmt, group_scales)
    rc = lib().orc_gemm_rows(int(fmt), N, K, _p(_c(packed, np.uint8)), _p(gs), M, _p(X), X.shape[1], r0, nrows,
                             _p(Y), int(nthreads))
    if rc != 0:
        raise ValueError(f"orc_gemm_rows rc={rc}")
    return Y


def gemv(fmt, N, K, packed, group_scales, x_f16_bits, r0=0, nrows=None, nthreads=1):
    return gemm(fmt, N, K, packed, group_scales, np.asarray(x_f16_bits)[None, :], r0, nrows, nthreads)[0]


def prefill_sample(fmt, N, K, packed, group_scales, X_bf16_bits, ms, ns, round_w=True):
    """fp64 Y[m_i, n_i] = Σ_k bf16(X)[m_i, k] · bf16(w')[n_i, k] for the sampled pairs (sorted by n for speed)."""
    X = _c(X_bf16_bits, np.uint16)
    ms = _c(ms, np.int64); ns = _c(ns, np.int64)
    out = np.zeros(ms.size, np.float64)
    gs = _gs(fmt, group_scales)
    rc = lib().orc_prefill_sample(int(fmt), N, K, _p(_c(packed, np.uint8)), _p(gs), _p(X), X.shape[1], X.shape[0],
                                  _p(ms), _p(ns), ms.size, int(bool(round_w)), _p(out))
    if rc != 0:
        raise ValueError(f"orc_prefill_sample rc={rc}")
    return out


def quantize_pack(fmt, W):
    """Quantize fp32 W and pack it: (packed, group_scales, flags)."""
    W = _c(W, np.float32)
    parts = quantize(fmt, W)
    packed, gs = pack(fmt, W.shape[0], W.shape[1], parts)
    return packed, gs, parts["flags"]


# ---------------------------------------------------------------------------------------------------------
# 8-bit KV cache (2/3/5/6-bit article §4.1; Mix-Quant article §2.3)
# ---------------------------------------------------------------------------------------------------------
def kv_quantize(v_f16_bits):
    """fp16 bit patterns (any shape, size a multiple of 32, groups of 32 consecutive elements) ->
    (int8 codes of the same shape, fp16 scale bit patterns [size / 32])."""
    v = _c(v_f16_bits, np.uint16)
    q = np.empty(v.shape, np.int8)
    s = np.empty(v.size // 32, np.uint16)
    if lib().orc_kv_quantize(_p(v), v.size, _p(q), _p(s)) != 0:
        raise ValueError("kv_quantize: size must be a multiple of 32")
    return q, s


def kv_dequant(q, scales):
    """int8 codes + fp16 scale bit patterns -> fp16 bit patterns of the codes' shape."""
    q = _c(q, np.int8)
    s = _c(scales, np.uint16)
    out = np.empty(q.shape, np.uint16)
    if lib().orc_kv_dequant(_p(q), _p(s), q.size, _p(out)) != 0:
        raise ValueError("kv_dequant: size must be a multiple of 32")
    return out
