"""The page's printed figures pin the shapes and the traffic formula the bench uses."""
import json
import os

from hyper_connection_mix_gb300 import traffic as bench_model

HERE = os.path.dirname(os.path.abspath(__file__))


def _fig():
    with open(os.path.join(HERE, "golden", "hc_fused_page_figures.json")) as f:
        return json.load(f)


def test_shape_constants():
    f = _fig()["figures"]
    assert f["num_slices"]["value"] * f["slice_width"]["value"] == f["K"]["value"]
    assert f["K"]["value"] // f["block_k"]["value"] == f["k_walk_chunks"]["value"]
    assert f["mix"]["value"] == 2 * f["hc"]["value"] + f["hc"]["value"] ** 2
    assert f["calls_per_forward"]["value"] == 2 * f["layers"]["value"]


def test_activation_bytes_match_page():
    f = _fig()["figures"]
    M, K = f["prefill_rows"]["value"], f["K"]["value"]
    x_mb = bench_model.activation_bytes(M, K) / 1e6
    assert round(x_mb) == f["activation_mb_at_4096"]["value"]


def test_stock_partial_round_trip_matches_page():
    f = _fig()["figures"]
    mb = bench_model.stock_partial_round_trip_bytes(
        f["prefill_rows"]["value"], f["num_slices"]["value"], f["mix"]["value"]) / 1e6
    assert round(mb) == f["partial_round_trip_mb_at_4096"]["value"]


def test_algorithmic_bytes_formula():
    # x once (bf16) plus W once (fp32); outputs excluded
    assert bench_model.algorithmic_bytes(4096, 20480) == 4096 * 20480 * 2 + 24 * 20480 * 4
