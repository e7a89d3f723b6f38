"""Numbers printed on the pages pin the work accounting and the kernels'
base-2 constants (tests/golden/page_numbers.json, each entry cited there)."""
import json
import math
import os

from exact_attention_flashattention_gb300 import flops

G = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_numbers.json")))


def test_backward_flop_count():
    g = G["bwd_flops_causal_8_16_4096_128"]
    s = g["shape"]
    f = flops.bwd_flops(s["B"], s["H"], s["N"], s["d"], s["causal"])
    assert abs(f / g["value"] - 1) < g["rel_tol"]


def test_backward_min_bytes():
    r, w = flops.bwd_min_bytes(8, 16, 4096, 128)
    assert abs(r / 1e6 - G["bwd_bytes_read_MB"]["value"]) < G["bwd_bytes_read_MB"]["abs_tol_MB"]
    assert abs(w / 1e6 - G["bwd_bytes_written_MB"]["value"]) < G["bwd_bytes_written_MB"]["abs_tol_MB"]


def test_latency_to_tflops():
    g = G["bwd_v3_latency_to_tflops"]
    t = flops.tflops(flops.bwd_flops(8, 16, 4096, 128, True), g["latency_ms"])
    assert abs(t / g["tflops"] - 1) < g["rel_tol"]
    g = G["fwd_fp16v2_latency_to_tflops"]
    t = flops.tflops(flops.fwd_flops(1, g["BH"], g["N"], g["d"], False), g["latency_ms"])
    assert abs(t / g["tflops"] - 1) < g["rel_tol"]


def test_rescale_threshold_conversions():
    g = G["rescale_threshold_units"]
    nat = g["threshold_log2"] / math.log2(math.e)
    assert abs(nat - g["natural_gap"]) < 5e-4
    assert abs(nat * math.sqrt(128) - g["raw_score_gap_d128"]) < 0.05
    g = G["exp2_worked_value"]
    assert abs(2 ** g["x"] - g["approx"]) < g["abs_tol"]
    g = G["exp2_split_example"]
    ip = math.floor(g["x"])
    assert ip == g["integer_part"] and g["x"] - ip == g["fractional_part"]
