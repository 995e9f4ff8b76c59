"""The bench's algorithmic byte and flop counts (the numerators of every roofline
figure it reports), pinned to hand-computed values for the workload's shapes."""
from __future__ import annotations

import pytest

import bench


def test_weight_bytes_by_hand():
    # 2048 x 2048 at 4 bits: codes 2048*2048/2, scales + biases 2 * 2048 * 32 bf16
    assert bench.weight_bytes(2048, 2048, 4) == 2_097_152 + 262_144
    # 8192 x 2048 at 6 bits: codes 8192*2048*6/8, scales + biases 2 * 8192 * 32 * 2
    assert bench.weight_bytes(8192, 2048, 6) == 12_582_912 + 1_048_576
    # 2048 x 8192 at 8 bits
    assert bench.weight_bytes(2048, 8192, 8) == 16_777_216 + 1_048_576


def test_layer_shapes_match_the_workload():
    shapes = bench.layer_shapes()
    assert len(shapes) == 16 * 3 + 6 * 5
    ffn = [(n, k) for name, n, k in shapes if name.endswith((".w1", ".w3"))]
    assert ffn == [(8192, 2048)] * 32
    assert all((n, k) == (2048, 8192) for name, n, k in shapes if name.endswith(".w2"))
    kv = [(n, k) for name, n, k in shapes if name.endswith((".k", ".v"))]
    assert kv == [(512, 2048)] * 12


def test_decode_bytes_by_hand():
    # weights of one pass: 16 x (w1 + w3 + w2) + 6 x (q + k + v + gate + o), 4-bit
    w = lambda n, k: n * k // 2 + 2 * n * (k // 64) * 2  # noqa: E731
    weights = 16 * (2 * w(8192, 2048) + w(2048, 8192)) + 6 * (3 * w(2048, 2048) + 2 * w(512, 2048))
    # activations read and outputs written per launch at R = 1
    attn = 6 * ((2048 * 2 + (2 * 2048 + 2 * 512) * 4) + (2048 * 2 + 2048 * 4))
    ffn = 16 * ((2048 * 2 + 8192 * 2) + (8192 * 2 + 2048 * 4))
    assert bench.decode_bytes(4, 1) == weights + attn + ffn
    assert weights == 502_530_048  # 502.5 MB of distinct weights per pass


def test_prefill_flops_by_hand():
    per_layer_ffn = 3 * 2 * 8192 * 8192 * 2048
    per_attn = 2 * 8192 * 2048 * (3 * 2048 + 2 * 512)
    assert bench.prefill_flops() == 16 * per_layer_ffn + 6 * per_attn


def test_job_throughput_is_units_over_time():
    assert bench.job_throughput(503_472_128, 10, 2.62, 1) == pytest.approx(503_472_128 * 10 / 2.62e-3, rel=1e-12)


def test_interp_cost_is_piecewise_linear():
    pts = [(1, 9.0), (2, 9.2), (4, 9.4), (8, 9.6), (16, 9.8)]
    # measured sizes come back exactly; in-between sizes sit on the segment
    for r, c in pts:
        assert bench.interp_cost(pts, r) == pytest.approx(c)
    assert bench.interp_cost(pts, 3) == pytest.approx(9.3)
    assert bench.interp_cost(pts, 12) == pytest.approx(9.7)
    # order of the points does not matter; missing costs are ignored
    assert bench.interp_cost(list(reversed(pts)) + [(32, None)], 6) == pytest.approx(9.5)
    # below the smallest size: its cost; above the largest: the last segment extended
    assert bench.interp_cost([(4, 5.0), (8, 7.0)], 1) == pytest.approx(5.0)
    assert bench.interp_cost([(4, 5.0), (8, 7.0)], 12) == pytest.approx(9.0)
    assert bench.interp_cost([(4, 5.0)], 100) == pytest.approx(5.0)
    assert bench.interp_cost([], 3) is None


def test_window_choice_runs():
    table = [{"rows": r, "mv_rows_us": mv, "pgemm_us": pg} for r, mv, pg in
             [(1, 9.0, 37.0), (2, 9.1, 37.0), (4, 9.2, 37.1), (8, 9.5, 37.1), (16, 9.8, 37.2),
              (32, None, 37.2), (64, None, 37.3)]]
    assert bench.window_choice(table, 64) == [{"rows": [1, 16], "call": "qlinear_mv_rows"},
                                              {"rows": [17, 64], "call": "qlinear_pgemm"}]
    # a matvec that grows past the GEMM's cost inside 1..16 hands over where the lines cross
    table2 = [{"rows": 1, "mv_rows_us": 10.0, "pgemm_us": 30.0},
              {"rows": 16, "mv_rows_us": 40.0, "pgemm_us": 30.0}]
    # crossing at 10 + 2 (R - 1) = 30  ->  R = 11 (ties go to the matvec)
    assert bench.window_choice(table2, 20) == [{"rows": [1, 11], "call": "qlinear_mv_rows"},
                                               {"rows": [12, 20], "call": "qlinear_pgemm"}]


def _run_bench(args, env_extra=None):
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {**os.environ, **(env_extra or {})}
    r = subprocess.run([sys.executable, "bench.py", *args], cwd=root, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    return [json.loads(ln) for ln in lines]


def test_reference_arm_prints_one_contract_line():
    (line,) = _run_bench(["--impl", "reference", "--steps", "1", "--warmup", "0"])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["higher_is_better"] is True
    assert line["metric"] == bench.METRIC and line["steps"] == 1 and line["value"] > 0
    assert line["dtype"] == "f64" and line["data"] == "synthetic" and line["vs_baseline"] is None
    # the same workload description as the CUDA arm's line, plus what one step samples
    cfg = dict(line["config"])
    assert cfg.pop("sample")
    assert cfg == bench.workload_config(4, 1)
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1 and cb["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_do_no_work():
    assert _run_bench(["--impl", "reference", "--steps", "1", "--warmup", "0"],
                      {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}) == []


def test_layer_bytes_add_up_to_the_pass():
    # the oracle baseline scales one FFN layer and one attention set to the pass: 16 + 6
    for bits in (4, 6, 8):
        for rows in (1, 16):
            assert 16 * bench.ffn_layer_bytes(bits, rows) + 6 * bench.attn_set_bytes(bits, rows) == \
                bench.decode_bytes(bits, rows)
    assert bench.sweep_weight_bytes(4) == 502_530_048
    # the windowed prefill streams every weight once per window
    assert bench.sweep_weight_bytes(8) == sum(bench.weight_bytes(n, k, 8) for _, n, k in bench.layer_shapes())
