"""Host-side logic of bench.py (no GPU): the row passes and kernels the grouped
GEMM uses, the algorithmic byte counts, and the source keys of the recorded
DRAM-traffic ratios."""
import importlib.util
import os

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
bench = importlib.util.module_from_spec(spec)
spec.loader.exec_module(bench)


def test_gemm_passes_split_rows_and_pick_kernels():
    assert bench.gemm_passes(5) == [(5, "mma")]
    assert bench.gemm_passes(24) == [(24, "bs4")]
    assert bench.gemm_passes(8) == [(8, "mma")]
    assert bench.gemm_passes(70) == [(64, "bs8"), (6, "mma")]
    assert bench.gemm_passes(25) == [(25, "bs4")]
    assert bench.gemm_passes(64) == [(64, "bs8")]
    assert bench.gemm_passes(80) == [(64, "bs8"), (16, "bs4")]
    assert bench.gemm_passes(320) == [(64, "bs8")] * 5
    assert sum(r for r, _ in bench.gemm_passes(1000)) == 1000


def test_gemm_bytes_matches_the_stated_formula():
    # W nibbles + E8M0 scales + bf16 X + fp32 Y
    M, N, K = 5, 128256, 4096
    assert bench.gemm_bytes(M, N, K) == N * K // 2 + N * K // 32 + 2 * M * K + 4 * M * N
    # the 8B step at M=5 moves 4.026 GB of algorithmic bytes
    import workloads
    total = sum(bench.gemm_bytes(5, N, K) for _, K, N in workloads.stack_shapes("llama8b"))
    assert abs(total / 1e9 - 4.026) < 0.002


def test_accept_bytes_count_one_law_per_row():
    B, K, V = 3, 4, 1000
    n = np.array([5, 1, 3])  # all accepted (bonus law 4V) / rejections (residual pair 8V)
    b = bench.accept_bytes(B, K, V, n)
    laws = 4 * V + 8 * V + 8 * V
    # per row: gathers p, q (8K), uniforms (4(K+1)), draft ids (4K), tokens (4(K+1)), count (4)
    per_row = 8 * K + 4 * (K + 1) + 4 * K + 4 * (K + 1) + 4
    assert b == laws + B * per_row


def test_code_only_ignores_comments_and_blank_lines():
    a = "int x = 1;  // one\n/* block\n comment */\n\nint y = 2;\n"
    b = "int x = 1;\n// another comment\nint y = 2;   \n"
    assert bench.code_only(a) == bench.code_only(b)
    assert bench.code_only("int x = 1;") != bench.code_only("int x = 2;")


def test_recorded_traffic_keys_name_the_current_kernels():
    # a ratio is only reported for the kernel source it was measured on
    for kind, rec in bench.GEMM_TRAFFIC.items():
        if rec["ratio"] is not None:
            assert rec["sha"] == bench.src_sha(kind), kind


def test_tensor_pipe_table_covers_every_kernel():
    assert set(bench.GEMM_TENSOR_PCT) == set(bench.GEMM_TRAFFIC)
    for M in (5, 20, 64, 80, 320):
        pct = bench.tensor_pct(bench.gemm_passes(M))
        assert all(v is None or 0.0 < v < 100.0 for v in pct.values())


def test_w4a4_pass_plan():
    # as few passes as 256 rows allow, of equal size (to 16), covering M exactly
    for M in list(range(1, 1100, 7)) + [256, 257, 320, 512, 513]:
        passes = bench.w4a4_passes(M)
        assert sum(r for r, _ in passes) == M
        assert len(passes) == -(-M // 256)
        assert all(0 < r <= 256 for r, _ in passes)
    assert [r for r, _ in bench.w4a4_passes(320)] == [160, 160]
