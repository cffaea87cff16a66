"""Decode-phase bandwidth arithmetic (2/3/5/6-bit article, lpnh.cn/news/2857666, §1.2: time per token = weight
bytes / effective bandwidth; DBHOO-CIM article, pwwt.cn/news/4452170, §4.4: effective bandwidth = weight bytes /
latency, utilisation = effective / peak)."""
from __future__ import annotations


def effective_gbps(weight_bytes: float, seconds: float) -> float:
    """Effective weight bandwidth in GB/s (decimal) for streaming `weight_bytes` in `seconds`."""
    return weight_bytes / seconds / 1e9


def utilisation(eff_gbps: float, peak_gbps: float) -> float:
    return eff_gbps / peak_gbps


def seconds_per_sweep(weight_bytes: float, gbps: float) -> float:
    """Time to read every weight once at `gbps` (the decode-step floor)."""
    return weight_bytes / (gbps * 1e9)


def tokens_per_second(weight_bytes_per_token: float, gbps: float) -> float:
    """Decode ceiling: one full weight sweep per generated token."""
    return 1.0 / seconds_per_sweep(weight_bytes_per_token, gbps)


def tflops(flops: float, seconds: float) -> float:
    return flops / seconds / 1e12
