"""The benchmark's metric helpers reproduce the decode arithmetic the pages print (golden fixture)."""
from conftest import kv, read_golden

from bit_weight_quantized_qpack_gb300 import metrics


def test_decode_arithmetic_matches_pages():
    for row in read_golden("decode_arithmetic.txt"):
        k = kv(row[1:])
        if row[0] == "CEILING":
            assert round(metrics.tokens_per_second(k["weight_GB"] * 1e9, k["bw_GBps"]), 1) == k["tok_per_s"]
        elif row[0] == "SWEEP":
            assert round(metrics.seconds_per_sweep(k["weight_GB"] * 1e9, k["bw_GBps"]), 2) == k["seconds"]
        elif row[0] == "EFFECTIVE":
            eff = metrics.effective_gbps(k["weight_GB"] * 1e9, k["latency_s"])
            assert round(eff, 1) == k["eff_GBps"]
            assert round(metrics.utilisation(eff, k["peak_GBps"]), 2) == k["utilisation"]
