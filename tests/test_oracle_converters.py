"""Pins for the oracle's hand-written fp16 / bf16 converters against numpy / torch library conversions
(IEEE round-to-nearest-even), exhaustive over all 65,536 fp16 patterns."""
import numpy as np
import torch


def test_f16_to_f32_exhaustive(orc):
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = orc.f16_bits_to_f32(h)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_f32_to_f16_roundtrip_exhaustive(orc):
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = h.view(np.float16).astype(np.float32)
    back = orc.f32_to_f16_bits(f)
    ok = ~np.isnan(f)
    assert np.array_equal(back[ok], h[ok])


def test_f32_to_f16_random_and_ties(orc):
    rng = np.random.default_rng(1)
    # wide magnitude range incl. subnormal fp16 outputs and overflow
    x = (rng.standard_normal(400_000) * np.exp2(rng.integers(-30, 20, 400_000))).astype(np.float32)
    # exact ties between consecutive fp16 values (midpoints), incl. subnormal midpoints
    h = rng.integers(0, 0x7BFF, 200_000).astype(np.uint16)
    a = h.view(np.float16).astype(np.float64)
    b = (h + 1).view(np.float16).astype(np.float64)
    mid = ((a + b) / 2).astype(np.float32)
    x = np.concatenate([x, mid, -mid, np.float32([65504, 65519.99, 65520, 1e-8, 2.9802322e-08, 5.96e-8])])
    got = orc.f32_to_f16_bits(x)
    ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_against_torch(orc):
    rng = np.random.default_rng(2)
    x = (rng.standard_normal(300_000) * np.exp2(rng.integers(-60, 60, 300_000))).astype(np.float32)
    u = rng.integers(0, 1 << 15, 100_000).astype(np.uint32)
    ties = ((u << 16) | 0x8000).view(np.float32)      # exact midpoints between bf16 neighbours
    x = np.concatenate([x, ties[np.isfinite(ties)]])
    got = orc.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)
    back = orc.bf16_bits_to_f32(got)
    assert np.array_equal(back, torch.from_numpy(got.view(np.int16)).view(torch.bfloat16).float().numpy())
