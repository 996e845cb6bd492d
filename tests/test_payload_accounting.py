"""The weight-streaming accounting the byte counts rest on, pinned to the
figures "Module 11. Speculative Decoding and Quantization" prints (§1, the
weight-streaming limit Q <= BW / W; §11, W_payload = N * b_eff / 8), and the
bench's per-step weight bytes pinned to the same formula for MX-FP4
(b_eff = 4 bits + one 8-bit scale per 32 elements = 4.25 bits)."""
import importlib.util
import json
import os

import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden", "payload_accounting.json")


def _bench():
    spec = importlib.util.spec_from_file_location("bench_acct", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def payload_bytes(params, bits_per_weight):
    return params * bits_per_weight / 8


def test_printed_weight_streaming_limits():
    g = json.load(open(GOLDEN))
    assert payload_bytes(g["params"], 16) == g["bf16_bytes"]
    assert payload_bytes(g["params"], 4.5) == g["b_eff_4p5_bytes"]
    # Q = BW / W, printed to one decimal
    assert round(g["bw_bytes_per_s"] / g["bf16_bytes"], g["printed_decimals"]) == g["bf16_tok_s"]
    assert round(g["bw_bytes_per_s"] / g["b_eff_4p5_bytes"], g["printed_decimals"]) == g["b_eff_4p5_tok_s"]
    # the same accounting for MX-FP4 (4-bit codes + an E8M0 byte per 32): 4.25 bits per weight
    assert payload_bytes(g["params"], 4 + 8 / 32) == 4.25e9
    assert abs(g["bw_bytes_per_s"] / 4.25e9 - 788.2) < 0.05


def test_stack_weight_bytes_follow_the_payload_formula():
    b = _bench()
    for model, expect in (("llama8b", 3_986_849_792), ("llama70b", None)):
        shapes = workloads.stack_shapes(model)
        params = sum(N * K for _, K, N in shapes)
        packed = sum(N * K // 2 + N * K // 32 for _, K, N in shapes)   # nibbles + E8M0 bytes
        assert packed == payload_bytes(params, 4.25)
        assert packed == b.config_block(model, model, 1, 4)["weight_bytes_per_step"]
        # the algorithmic bytes of a step are the weights plus bf16 X and fp32 Y
        M = 5
        alg = sum(b.gemm_bytes(M, N, K) for _, K, N in shapes)
        assert alg == packed + sum(2 * M * K + 4 * M * N for _, K, N in shapes)
        if expect is not None:
            assert packed == expect
