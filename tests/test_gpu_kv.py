"""GPU parity of the 8-bit KV-cache kernels: codes, scales and the dequantized fp16 cache bit for bit against the
oracle (2/3/5/6-bit article §4.1; Mix-Quant article §2.3)."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def check(qpg, orc, v):
    """v: CPU fp16 tensor."""
    q, s = qpg.qpack_kv_quantize(v.cuda())
    out = qpg.qpack_kv_dequant(q, s)
    torch.cuda.synchronize()
    rq, rs = orc.kv_quantize(v.numpy().view(np.uint16))
    assert np.array_equal(q.cpu().numpy().reshape(-1), rq.reshape(-1)), "codes differ"
    assert np.array_equal(s.cpu().numpy().view(np.uint16), rs), "scales differ"
    assert np.array_equal(out.cpu().numpy().view(np.uint16).reshape(-1), orc.kv_dequant(rq, rs).reshape(-1))


@pytest.mark.parametrize("n", [32, 32 * 33, 1024, 1024 * 7 + 96, 1 << 20, (1 << 22) + 32 * 5])
def test_kv_sizes(qpg, orc, n):
    from bit_weight_quantized_qpack_gb300 import synth
    v = synth.normal((n,), 1.0, seed=n % 997, dtype=torch.float16)
    check(qpg, orc, v)


def test_kv_magnitudes(qpg, orc):
    """Groups spanning many binades, fp16 extremes, subnormals, all-zero and single-element groups."""
    from bit_weight_quantized_qpack_gb300 import synth
    g = 4096
    base = synth.normal((g, 32), 1.0, seed=5)
    scale = torch.exp(torch.linspace(-20.0, 10.0, g))[:, None]
    v = (base * scale).clamp(-65504, 65504)
    v[0] = 0.0
    v[1] = 0.0
    v[1, 7] = -65504.0
    v[2] = 6e-8                                        # fp16 subnormals
    v[3, ::2] = 1e-3
    v[3, 1::2] = -300.0
    check(qpg, orc, v.to(torch.float16))


def test_kv_7b_cache_shape(qpg, orc):
    """The 7B grouped-query cache of the page (2 x 32 layers x 8 heads x 128 x 8192 tokens, 1.07 GB fp16) in one call;
    the oracle checks 64 sampled 4096-element slices (groups are independent)."""
    from bit_weight_quantized_qpack_gb300 import synth
    shape = (2, 32, 8, 8192, 128)
    v = synth.normal(shape, 1.0, seed=21, device="cuda", dtype=torch.float16)
    q, s = qpg.qpack_kv_quantize(v)
    out = qpg.qpack_kv_dequant(q, s)
    torch.cuda.synchronize()
    n = v.numel()
    starts = np.random.default_rng(3).integers(0, n // 4096, 64) * 4096
    vf, qf, sf, of = v.view(-1), q.view(-1), s.view(-1), out.view(-1)
    for st in starts:
        st = int(st)
        rq, rs = orc.kv_quantize(vf[st:st + 4096].cpu().numpy().view(np.uint16))
        assert np.array_equal(qf[st:st + 4096].cpu().numpy(), rq)
        assert np.array_equal(sf[st // 32:(st + 4096) // 32].cpu().numpy().view(np.uint16), rs)
        assert np.array_equal(of[st:st + 4096].cpu().numpy().view(np.uint16), orc.kv_dequant(rq, rs))
    assert qpg.qpack_fetch_fault_flags() == 0


def test_kv_rounding_boundaries(qpg, orc):
    """Elements on and next to the half-integer multiples (k + 1/2) d of their group's scale, over scales spanning the
    fp16 range: the codes must equal rint of the correctly rounded quotient (ties to even), as in the oracle."""
    rng = np.random.default_rng(9)
    G = 8192
    m = np.exp(rng.uniform(np.log(1e-3), np.log(6e4), G)).astype(np.float16)          # each group's max |v|
    d = (m.astype(np.float32) / np.float32(127)).astype(np.float16).astype(np.float64)
    k = rng.integers(-127, 127, (G, 31))
    v = ((k + 0.5) * d[:, None]).astype(np.float16)             # the tie itself where fp16 holds it, else a neighbour
    bits = v.view(np.uint16).astype(np.int32) + rng.integers(-1, 2, (G, 31))            # and adjacent fp16 values
    v = (bits & 0xFFFF).astype(np.uint16).view(np.float16)
    v = np.where(np.isfinite(v.astype(np.float32)), v, np.float16(0))
    grp = np.concatenate([m[:, None], v], axis=1).reshape(-1)
    check(qpg, orc, torch.from_numpy(grp.copy()))
