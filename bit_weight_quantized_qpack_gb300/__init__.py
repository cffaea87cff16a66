"""qpack for GB300: fused dequantization + matrix-vector / small-batch / prefill products over group-quantized
low-bit weights (INT4 group-32 and the 2/3/5/6-bit 256-weight super-block formats).

This module is a thin ctypes binding over the C ABI of ``libqpack.so`` (declared in ``include/qpack.h``). It
only marshals arguments: every computation runs in the library's CUDA kernels. PyTorch supplies device memory
and streams. There is no CPU fallback: importing works anywhere, but every compute call raises ``QpackError``
when the CUDA library is not built or no GPU is present.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

Q4G32, Q2S, Q3S, Q5S, Q6S, Q4G32H, Q4G16, Q4G32A = 0, 1, 2, 3, 4, 5, 6, 7
FORMATS = {"Q4G32": Q4G32, "Q2S": Q2S, "Q3S": Q3S, "Q5S": Q5S, "Q6S": Q6S, "Q4G32H": Q4G32H, "Q4G16": Q4G16,
           "Q4G32A": Q4G32A}
F32, F16, BF16 = 0, 1, 2
FLAG_RANGE = 1
FAULT_NONFINITE_X = 16
# (sub-blocks per super-block, asymmetric) for the super-block formats
_SB = {Q2S: (16, True), Q3S: (16, False), Q5S: (8, True), Q6S: (16, False)}

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqpack.so")
_lock = threading.Lock()
_lib = None


class QpackError(RuntimeError):
    pass


class Layout(ctypes.Structure):
    _fields_ = [("row_stride", ctypes.c_int64), ("packed_bytes", ctypes.c_int64),
                ("scale_stride", ctypes.c_int64), ("scale_bytes", ctypes.c_int64),
                ("block_bytes", ctypes.c_int64), ("nsub", ctypes.c_int64),
                ("weight_bytes", ctypes.c_int64)]


def lib():
    """Load libqpack.so (raises QpackError if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise QpackError(f"libqpack.so not built ({LIB_PATH}); run __graft_entry__.build()")
            L = ctypes.CDLL(LIB_PATH)
            P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
            sigs = {
                "qpack_layout": ([I, I64, I64, ctypes.POINTER(Layout)], I),
                "qpack_quantize": ([I, P, I, I64, I64, P, P, P, P, P, P, P, P], I),
                "qpack_pack": ([I, I64, I64, P, P, P, P, P, P, P, P, P], I),
                "qpack_quantize_pack": ([I, P, I, I64, I64, P, P, P, P], I),
                "qpack_unpack": ([I, I64, I64, P, P, P, P, P, P, P, P, P], I),
                "qpack_dequant": ([I, I64, I64, P, P, P, P], I),
                "qgemv": ([I, P, P, I64, I64, P, P, P], I),
                "qgemm_small": ([I, P, P, I64, I64, I, P, I64, P, I64, P], I),
                "qgemm_prefill": ([I, P, P, I64, I64, I64, P, I64, P, I64, P], I),
                "qpack_kv_quantize": ([P, I64, P, P, P], I),
                "qpack_kv_dequant": ([P, P, I64, P, P], I),
                "qpack_status_string": ([I], ctypes.c_char_p),
                "qpack_fetch_fault_flags": ([ctypes.POINTER(ctypes.c_int32)], I),
                "qpack_version": ([], I),
                "qpack_set_option": ([I, I], I),
            }
            for name, (args, res) in sigs.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = res
            _lib = L
    return _lib


def _check(rc: int, what: str):
    if rc != 0:
        msg = lib().qpack_status_string(rc).decode()
        raise QpackError(f"{what}: {msg} (status {rc})")


def _need(t, dtype, what, numel=None, rows=None, cols=None):
    """Argument checks the C ABI cannot make (it sees only pointers): element type, size and, for matrices, a row-major
    layout with unit column stride. Raises QpackError before anything is launched."""
    if t.dtype != dtype:
        raise QpackError(f"{what}: expected {dtype}, got {t.dtype}")
    if rows is not None:
        if t.dim() != 2 or t.shape[0] < rows or t.shape[1] < cols or (t.shape[1] > 1 and t.stride(1) != 1):
            raise QpackError(f"{what}: expected a row-major matrix of at least {rows} x {cols}, got {tuple(t.shape)} "
                             f"with strides {tuple(t.stride())}")
    elif numel is not None:
        if not t.is_contiguous() or t.numel() < numel:
            raise QpackError(f"{what}: expected a contiguous tensor of at least {numel} elements, got "
                             f"{tuple(t.shape)}")


def _need_packed(fmt, N, K, packed, group_scales):
    L = layout(fmt, N, K)
    _need(packed, torch.uint8, "packed", numel=L["packed_bytes"])
    if L["scale_bytes"]:
        if group_scales is None:
            raise QpackError("group_scales: required by this format")
        gdt = torch.float16 if int(fmt) == Q4G32H else torch.float32
        if group_scales.dtype == torch.int16 and gdt == torch.float16:
            gdt = torch.int16                                   # fp16 bit patterns held as int16
        _need(group_scales, gdt, "group_scales", numel=L["scale_bytes"] // group_scales.element_size())


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise QpackError("qpack kernels take CUDA tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dt(t):
    d = {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16}.get(t.dtype)
    if d is None:
        raise QpackError(f"W: expected float32, float16 or bfloat16, got {t.dtype}")
    if t.dim() != 2 or not t.is_contiguous():
        raise QpackError(f"W: expected a contiguous [N, K] matrix, got {tuple(t.shape)}")
    return d


def layout(fmt: int, N: int, K: int) -> dict:
    out = Layout()
    _check(lib().qpack_layout(int(fmt), int(N), int(K), ctypes.byref(out)), "qpack_layout")
    return {f: getattr(out, f) for f, _ in Layout._fields_}


def alloc_packed(fmt, N, K, device="cuda"):
    """Caller-owned packed buffers of the right sizes: (packed uint8 [N, row_stride], scales or None)."""
    L = layout(fmt, N, K)
    packed = torch.empty((N, L["row_stride"]), dtype=torch.uint8, device=device)
    gs = None
    if fmt in (Q4G32, Q4G32H, Q4G16, Q4G32A):   # fp32 or fp16 group scales (Q4G32A: fp32 (s, z) pairs)
        gs = torch.empty((N, L["scale_stride"]), dtype=torch.float16 if fmt == Q4G32H else torch.float32, device=device)
    return packed, gs


def alloc_parts(fmt, N, K, device="cuda"):
    parts = dict(q=torch.empty((N, K), dtype=torch.int8, device=device), gscale=None, sub_scale=None,
                 sub_min=None, d=None, dmin=None)
    if fmt in (Q4G32, Q4G16, Q4G32A):
        parts["gscale"] = torch.empty((N, K // (32 if fmt == Q4G32 else 16)), dtype=torch.float32, device=device)
    elif fmt == Q4G32H:
        parts["d"] = torch.empty((N, K // 32), dtype=torch.int16, device=device)   # fp16 group-scale bits
    else:
        nsub, asym = _SB[fmt]
        nb = K // 256
        parts["sub_scale"] = torch.empty((N, nb * nsub), dtype=torch.uint8, device=device)
        parts["d"] = torch.empty((N, nb), dtype=torch.int16, device=device)
        if asym:
            parts["sub_min"] = torch.empty((N, nb * nsub), dtype=torch.uint8, device=device)
            parts["dmin"] = torch.empty((N, nb), dtype=torch.int16, device=device)
    return parts


def qpack_quantize(fmt, W, parts=None, status=None, stream=None):
    wdt = _dt(W)
    N, K = W.shape
    parts = alloc_parts(fmt, N, K, W.device) if parts is None else parts
    rc = lib().qpack_quantize(int(fmt), _ptr(W), wdt, N, K, _ptr(parts["q"]), _ptr(parts["gscale"]),
                              _ptr(parts["sub_scale"]), _ptr(parts["sub_min"]), _ptr(parts["d"]),
                              _ptr(parts["dmin"]), _ptr(status), _stream(stream))
    _check(rc, "qpack_quantize")
    return parts


def qpack_pack(fmt, N, K, parts, packed=None, group_scales=None, stream=None):
    if packed is None:
        packed, group_scales = alloc_packed(fmt, N, K, parts["q"].device)
    rc = lib().qpack_pack(int(fmt), N, K, _ptr(parts["q"]), _ptr(parts["gscale"]), _ptr(parts["sub_scale"]),
                          _ptr(parts["sub_min"]), _ptr(parts["d"]), _ptr(parts["dmin"]), _ptr(packed),
                          _ptr(group_scales), _stream(stream))
    _check(rc, "qpack_pack")
    return packed, group_scales


def qpack_quantize_pack(fmt, W, packed=None, group_scales=None, status=None, stream=None):
    wdt = _dt(W)
    N, K = W.shape
    if packed is None:
        packed, group_scales = alloc_packed(fmt, N, K, W.device)
    rc = lib().qpack_quantize_pack(int(fmt), _ptr(W), wdt, N, K, _ptr(packed), _ptr(group_scales),
                                   _ptr(status), _stream(stream))
    _check(rc, "qpack_quantize_pack")
    return packed, group_scales


def qpack_unpack(fmt, N, K, packed, group_scales=None, parts=None, stream=None):
    parts = alloc_parts(fmt, N, K, packed.device) if parts is None else parts
    rc = lib().qpack_unpack(int(fmt), N, K, _ptr(packed), _ptr(group_scales), _ptr(parts["q"]),
                            _ptr(parts["gscale"]), _ptr(parts["sub_scale"]), _ptr(parts["sub_min"]),
                            _ptr(parts["d"]), _ptr(parts["dmin"]), _stream(stream))
    _check(rc, "qpack_unpack")
    return parts


def qpack_dequant(fmt, N, K, packed, group_scales=None, out=None, stream=None):
    out = torch.empty((N, K), dtype=torch.float32, device=packed.device) if out is None else out
    rc = lib().qpack_dequant(int(fmt), N, K, _ptr(packed), _ptr(group_scales), _ptr(out), _stream(stream))
    _check(rc, "qpack_dequant")
    return out


def qgemv(fmt, packed, group_scales, N, K, x, y=None, stream=None):
    _need_packed(fmt, N, K, packed, group_scales)
    _need(x, torch.float16, "x", numel=K)
    y = torch.empty(N, dtype=torch.float32, device=x.device) if y is None else y
    _need(y, torch.float32, "y", numel=N)
    rc = lib().qgemv(int(fmt), _ptr(packed), _ptr(group_scales), N, K, _ptr(x), _ptr(y), _stream(stream))
    _check(rc, "qgemv")
    return y


def qgemm_small(fmt, packed, group_scales, N, K, X, Y=None, stream=None):
    _need_packed(fmt, N, K, packed, group_scales)
    M = X.shape[0]
    _need(X, torch.float16, "X", rows=M, cols=K)
    Y = torch.empty((M, N), dtype=torch.float32, device=X.device) if Y is None else Y
    _need(Y, torch.float32, "Y", rows=M, cols=N)
    rc = lib().qgemm_small(int(fmt), _ptr(packed), _ptr(group_scales), N, K, M, _ptr(X), X.stride(0), _ptr(Y),
                           Y.stride(0), _stream(stream))
    _check(rc, "qgemm_small")
    return Y


def qgemm_prefill(fmt, packed, group_scales, N, K, X, Y=None, stream=None):
    _need_packed(fmt, N, K, packed, group_scales)
    M = X.shape[0]
    _need(X, torch.bfloat16, "X", rows=M, cols=K)
    Y = torch.empty((M, N), dtype=torch.bfloat16, device=X.device) if Y is None else Y
    _need(Y, torch.bfloat16, "Y", rows=M, cols=N)
    rc = lib().qgemm_prefill(int(fmt), _ptr(packed), _ptr(group_scales), N, K, M, _ptr(X), X.stride(0),
                             _ptr(Y), Y.stride(0), _stream(stream))
    _check(rc, "qgemm_prefill")
    return Y


def qpack_kv_quantize(v, codes=None, scales=None, stream=None):
    """fp16 KV tensor (any shape, contiguous, numel a multiple of 32) -> (int8 codes of its shape, fp16 scales
    [numel / 32]): one fp16 scale per 32 consecutive elements."""
    n = v.numel()
    _need(v, torch.float16, "v", numel=n)
    codes = torch.empty(v.shape, dtype=torch.int8, device=v.device) if codes is None else codes
    scales = torch.empty(n // 32, dtype=torch.float16, device=v.device) if scales is None else scales
    _need(codes, torch.int8, "codes", numel=n)
    _need(scales, torch.float16, "scales", numel=n // 32)
    _check(lib().qpack_kv_quantize(_ptr(v), n, _ptr(codes), _ptr(scales), _stream(stream)), "qpack_kv_quantize")
    return codes, scales


def qpack_kv_dequant(codes, scales, out=None, stream=None):
    """int8 codes + fp16 scales -> fp16 tensor of the codes' shape."""
    _need(codes, torch.int8, "codes", numel=codes.numel())
    _need(scales, torch.float16, "scales", numel=codes.numel() // 32)
    out = torch.empty(codes.shape, dtype=torch.float16, device=codes.device) if out is None else out
    _need(out, torch.float16, "out", numel=codes.numel())
    _check(lib().qpack_kv_dequant(_ptr(codes), _ptr(scales), codes.numel(), _ptr(out), _stream(stream)),
           "qpack_kv_dequant")
    return out


def qpack_fetch_fault_flags() -> int:
    v = ctypes.c_int32(0)
    _check(lib().qpack_fetch_fault_flags(ctypes.byref(v)), "qpack_fetch_fault_flags")
    return int(v.value)


def qpack_status_string(status: int) -> str:
    return lib().qpack_status_string(int(status)).decode()


OPT_WEIGHT_PREFETCH = 1
OPT_PREFILL_TILE_ROWS = 2


def qpack_set_option(option: int, value: int) -> None:
    _check(lib().qpack_set_option(int(option), int(value)), "qpack_set_option")


def qpack_version() -> int:
    return int(lib().qpack_version())
