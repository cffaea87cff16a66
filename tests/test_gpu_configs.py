"""Full-size parity of the decode workloads in the launch configuration the benchmark times, on sampled rows.

- 7B-Llama decode step, every super-block format: the four launches of a layer (q|k|v, o, gate|up and down).
  q|k|v and gate|up are row-concatenated packed matrices.
- 70B MLP small-batch decode, INT4 and Q5S, M = 1, 2, 4, 8, 16: gate and up (28672 x 8192) and down (8192 x 28672)
  of layers 0 and 79.

Weights and activations are generated on the GPU from the benchmark's seeds. The GPU quantizes and multiplies the
full matrices. The oracle quantizes only the sampled rows of the same weights (rows quantize independently), checks
those packed bytes against the GPU's bit for bit, and takes the fp64 products of those rows. The products must meet
max |y - y_ref| / (||w'_r|| * ||x||) <= 1e-4 (2/3/5/6-bit article §1.2, §3.3; DBHOO-CIM article §3.3)."""
import numpy as np
import pytest
import torch

from conftest import gemv_bound_check

pytestmark = pytest.mark.gpu

SAMPLE = 48


def sampled_rows(N, seed):
    g = np.random.default_rng(seed)
    rows = np.sort(g.choice(N, size=min(SAMPLE, N), replace=False))
    return np.unique(np.concatenate([[0, N - 1], rows]))


def check_rows(qpg, orc, fmt, W_rows, p, g, rows, X, Y):
    """W_rows: fp32 numpy [r, K] (the sampled rows); p / g: GPU packed matrix (and Q4G32 scales); X: fp16 [M, K];
    Y: GPU products [M, N]."""
    K = W_rows.shape[1]
    n = len(rows)
    rp, rgs, _ = orc.quantize_pack(fmt, W_rows)
    gp = p[torch.as_tensor(rows, device=p.device)].cpu().numpy()
    assert np.array_equal(gp.reshape(-1), np.asarray(rp).reshape(-1)), "packed rows differ from the oracle"
    if g is not None:
        gg = g[torch.as_tensor(rows, device=g.device)].cpu().numpy()
        assert np.array_equal(gg.reshape(-1).view(np.uint32), np.asarray(rgs).reshape(-1).view(np.uint32))
    Xb = X.cpu().numpy().view(np.uint16)
    Y_ref = orc.gemm(fmt, n, K, rp, rgs, Xb, nthreads=8)
    deq = orc.dequant(fmt, n, K, rp, rgs)
    Yg = Y.cpu().numpy()[:, rows]
    return gemv_bound_check(Yg, Y_ref, deq, X.cpu().numpy().astype(np.float64))


@pytest.mark.parametrize("name", ["Q2S", "Q3S", "Q5S", "Q6S"])
def test_config3_decode_step_layers(qpg, orc, name):
    from bit_weight_quantized_qpack_gb300 import synth
    fmt = qpg.FORMATS[name]
    shapes = [(4096, 4096)] * 4 + [(11008, 4096)] * 2 + [(4096, 11008)]
    groups = [[0, 1, 2], [3], [4, 5], [6]]
    x4 = synth.normal((4096,), 1.0, seed=11, device="cuda", dtype=torch.float16)
    x11 = synth.normal((11008,), 1.0, seed=12, device="cuda", dtype=torch.float16)
    for layer in (0, 31):
        Ws, packed = [], []
        for mi, (N, K) in enumerate(shapes):
            W = synth.laplace((N, K), 0.02, seed=synth.seed_for(3, layer, mi), device="cuda")
            p, _ = qpg.qpack_quantize_pack(fmt, W)
            Ws.append(W)
            packed.append(p)
        for gi, gidx in enumerate(groups):
            K = shapes[gidx[0]][1]
            N = sum(shapes[i][0] for i in gidx)
            pc = torch.cat([packed[i] for i in gidx], 0)
            x = x4 if K == 4096 else x11
            y = qpg.qgemv(fmt, pc, None, N, K, x)
            torch.cuda.synchronize()
            rows = sampled_rows(N, 1000 * layer + gi)
            Wc = torch.cat([Ws[i] for i in gidx], 0)
            W_rows = Wc[torch.as_tensor(rows, device="cuda")].cpu().numpy()
            check_rows(qpg, orc, fmt, W_rows, pc, None, rows, x[None, :], y[None, :])
        del Ws, packed
        torch.cuda.empty_cache()
    assert qpg.qpack_fetch_fault_flags() == 0


@pytest.mark.parametrize("name,layers", [("Q4G32", (0, 79)), ("Q5S", (0, 79)), ("Q4G32H", (0,)), ("Q4G16", (0,)),
                                         ("Q4G32A", (0,))])
def test_config4_70b_mlp_small_batch(qpg, orc, name, layers):
    """The INT4 variants (fp16 scales, group 16, asymmetric) run the same launches on layer 0."""
    from bit_weight_quantized_qpack_gb300 import synth
    fmt = qpg.FORMATS[name]
    shapes = [(28672, 8192), (28672, 8192), (8192, 28672)]
    for layer in layers:
        for mi, (N, K) in enumerate(shapes):
            W = synth.laplace((N, K), 0.01, seed=synth.seed_for(4, layer, mi), device="cuda")
            p, g = qpg.qpack_quantize_pack(fmt, W)
            rows = sampled_rows(N, 7000 + 10 * layer + mi)
            W_rows = W[torch.as_tensor(rows, device="cuda")].cpu().numpy()
            del W
            for M in (1, 2, 4, 8, 16):
                X = synth.normal((M, K), 1.0, seed=100 + M + K, device="cuda", dtype=torch.float16)
                Y = qpg.qgemm_small(fmt, p, g, N, K, X)
                torch.cuda.synchronize()
                check_rows(qpg, orc, fmt, W_rows, p, g, rows, X, Y)
            del p, g
            torch.cuda.empty_cache()
    assert qpg.qpack_fetch_fault_flags() == 0


def test_config3_mixed_format_layer(qpg, orc):
    """The mixed-format decode step (q and k Q5S, v and o Q6S, feed-forward Q3S; 2/3/5/6-bit article §2.4): every
    launch of layer 0, with q|k and gate|up row-concatenated."""
    from bit_weight_quantized_qpack_gb300 import synth
    shapes = [(4096, 4096)] * 4 + [(11008, 4096)] * 2 + [(4096, 11008)]
    fmts = ["Q5S", "Q5S", "Q6S", "Q6S", "Q3S", "Q3S", "Q3S"]
    groups = [[0, 1], [2], [3], [4, 5], [6]]
    x4 = synth.normal((4096,), 1.0, seed=11, device="cuda", dtype=torch.float16)
    x11 = synth.normal((11008,), 1.0, seed=12, device="cuda", dtype=torch.float16)
    Ws = [synth.laplace((N, K), 0.02, seed=synth.seed_for(3, 0, mi), device="cuda") for mi, (N, K) in enumerate(shapes)]
    for gi, gidx in enumerate(groups):
        fmt = qpg.FORMATS[fmts[gidx[0]]]
        K = shapes[gidx[0]][1]
        N = sum(shapes[i][0] for i in gidx)
        pc = torch.cat([qpg.qpack_quantize_pack(fmt, Ws[i])[0] for i in gidx], 0)
        x = x4 if K == 4096 else x11
        y = qpg.qgemv(fmt, pc, None, N, K, x)
        torch.cuda.synchronize()
        rows = sampled_rows(N, 500 + gi)
        W_rows = torch.cat([Ws[i] for i in gidx], 0)[torch.as_tensor(rows, device="cuda")].cpu().numpy()
        check_rows(qpg, orc, fmt, W_rows, pc, None, rows, x[None, :], y[None, :])
    assert qpg.qpack_fetch_fault_flags() == 0
