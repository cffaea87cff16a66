"""Hand-computed products of tiny matrices for every format (tests/golden/tiny_products.txt).

Each row of K = 256 weights is an exact lattice of its format's dequantization rule, built from a few integers per
block (which code sits where, the sub-block scale and minimum integers or the INT4 scale and zero point) with unit
super-scales, so every dequantized weight is an integer; the activations are small integers constant on a block. The
fixture lists, per row, every block's code sum S_j and its contribution to y, worked out by hand from the closed forms
in its header (the 2/3/5/6-bit article, lpnh.cn/news/2857666, §3.4: quantize a known block and check what comes
back). The oracle must return exactly these integers; the CUDA products must stay within their bound of them.
"""
import numpy as np
import pytest
import torch

from conftest import gemv_bound_check, read_golden


def parse():
    cases, cur = [], None
    for tok in read_golden("tiny_products.txt"):
        if tok[0] == "FORMAT":
            cur = dict(name=tok[1], B=int(tok[2]), A=int(tok[3]), C=int(tok[4]), rows=[])
            cases.append(cur)
        elif tok[0] == "ROW":
            cur["rows"].append(dict({k: [int(v) for v in val.split(",")] for k, val in (t.split("=") for t in tok[2:])},
                                    terms=[]))
        elif tok[0] == "TERM":
            cur["rows"][-1]["terms"].append((int(tok[1]), int(tok[2]), int(tok[3])))
        elif tok[0] == "Y":
            cur["rows"][-1]["y"] = int(tok[1])
    return cases


def build(case):
    """The weight rows and the activation vector of one format's case."""
    B, A, C = case["B"], case["A"], case["C"]
    nb = 256 // B
    x = np.repeat(np.array([(j % 4) - 1 for j in range(nb)], np.float64), B)
    W = np.zeros((len(case["rows"]), 256), np.float64)
    for r, row in enumerate(case["rows"]):
        for j in range(nb):
            code = np.where(np.arange(B) < row["k"][j], A, C).astype(np.float64)
            if "L" in row:                                     # super-block formats, d = dmin = 1
                w = row["L"][j] * code - (row["M"][j] if "M" in row else 0)
            elif "z" in row:                                   # INT4 asymmetric: s (u - z)
                w = row["s"][j] * (code - row["z"][j])
            else:                                              # INT4 symmetric: s q
                w = row["s"][j] * code
            W[r, B * j:B * (j + 1)] = w
    return W.astype(np.float32), x


CASES = parse()


def test_fixture_terms_add_up():
    """The fixture's own arithmetic: each block's S_j and contribution follow from the row parameters, and the
    contributions sum to Y (so a typo in a literal is caught before the oracle is compared with it)."""
    assert [c["name"] for c in CASES] == ["Q3S", "Q6S", "Q2S", "Q5S", "Q4G32", "Q4G32H", "Q4G16", "Q4G32A"]
    for case in CASES:
        B, A, C = case["B"], case["A"], case["C"]
        for row in case["rows"]:
            assert sum(t for _, _, t in row["terms"]) == row["y"]
            for j, S, t in row["terms"]:
                assert S == row["k"][j] * A + (B - row["k"][j]) * C
                c = (j % 4) - 1
                if "L" in row:
                    assert t == c * (row["L"][j] * S - B * (row["M"][j] if "M" in row else 0))
                elif "z" in row:
                    assert t == c * row["s"][j] * (S - B * row["z"][j])
                else:
                    assert t == c * row["s"][j] * S


@pytest.mark.parametrize("case", CASES, ids=[c["name"] for c in CASES])
def test_oracle_gemv_equals_hand_computed(orc, case):
    fmt = orc.FORMATS[case["name"]]
    W, x = build(case)
    N, K = W.shape
    packed, gs, _ = orc.quantize_pack(fmt, W)
    deq = orc.dequant(fmt, N, K, packed, gs)
    assert np.array_equal(deq, W)                             # exact lattice: quantize + dequantize is the identity
    xb = x.astype(np.float16).view(np.uint16)
    y = orc.gemv(fmt, N, K, packed, gs, xb)
    assert list(y) == [float(row["y"]) for row in case["rows"]]
    Y = orc.gemm(fmt, N, K, packed, gs, np.stack([xb, xb]))
    assert np.array_equal(Y, np.stack([y, y]))


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES, ids=[c["name"] for c in CASES])
def test_gpu_products_on_hand_computed_rows(qpg, case):
    fmt = qpg.FORMATS[case["name"]]
    W, x = build(case)
    N, K = W.shape
    p, g = qpg.qpack_quantize_pack(fmt, torch.from_numpy(W).cuda())
    X = torch.from_numpy(np.stack([x, -x, 2 * x]).astype(np.float16)).cuda()
    y1 = qpg.qgemv(fmt, p, g, N, K, X[0])
    Y = qpg.qgemm_small(fmt, p, g, N, K, X)
    torch.cuda.synchronize()
    yh = np.array([row["y"] for row in case["rows"]], np.float64)
    gemv_bound_check(y1.cpu().numpy()[None, :], yh[None, :], W, x[None, :])
    gemv_bound_check(Y.cpu().numpy(), np.stack([yh, -yh, 2 * yh]), W, np.stack([x, -x, 2 * x]))
