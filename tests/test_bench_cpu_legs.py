"""The CPU legs of bench.py (the oracle baseline and the row-parallel C++ baseline) run on tiny
samples without a GPU, so a round-end benchmark cannot fail in them."""
import pytest

import bench


def test_oracle_leg_runs():
    rps, rounds, layers, w = bench.time_oracle("tiny", budget_s=0.2, max_rounds=2)
    assert rps > 0 and 1 <= rounds <= 2 and layers == 1 and w.name == "tiny"


def test_parallel_leg_runs_greedy_and_sampled():
    for name in ("tiny", "glm4_9b"):
        r = bench.time_cpu_parallel(name, budget_s=0.1, max_rounds=1, layers_sample=1)
        assert r["value"] > 0 and r["cores"] >= 1 and r["unit"] == "rounds/s"


def test_json_line_keys(monkeypatch, capsys):
    """The bench line carries every key of its contract (the GPU leg stubbed out)."""
    import json
    import sys
    fake = {"value": 10.0, "ms_per_step": 100.0, "launch": "graph+pdl",
            "clocks": {"sm_mhz": 1, "sm_max_mhz": 1, "reasons": []},
            "e2e": {"value": 9.0, "unit": "rounds/s", "h2d_bytes_per_step": 1,
                    "d2h_bytes_per_step": 1},
            "roofline": {"bound": "hbm", "achieved": 1.0, "peak": 2.0, "unit": "GB/s", "frac": 0.5,
                         "traffic": None},
            "verify": {}, "committed_slots_per_s": 1.0, "committed_per_round": 1.0,
            "cap_cols": 10, "bytes_per_round": 1e10}
    monkeypatch.setattr(bench, "run_specdec", lambda *a, **k: fake)
    monkeypatch.setattr(bench, "dist_setup", lambda gpus: (0, 1, 0))
    monkeypatch.setattr(bench, "time_oracle", lambda *a, **k: (2.0, 3, 1, None))
    monkeypatch.setattr(bench, "time_cpu_parallel", lambda *a, **k: {"value": 5.0})
    monkeypatch.setattr(bench, "run_all_configs", lambda *a, **k: {"tiny": {}})
    monkeypatch.setattr(bench, "specdec_summary", lambda *a, **k: {})
    monkeypatch.setattr(sys, "argv", ["bench.py", "--workload", "vicuna7b"])
    bench.main()
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "clocks",
              "e2e", "roofline", "gpu_launches", "cpu_baseline", "cpu_parallel", "run",
              "all_configs"):
        assert k in line, k
    assert line["config"]["workload"].startswith("vicuna7b")
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["gpu_launches"] == 2 * line["steps"]
    assert "launch" not in line["config"] and line["run"]["launch"] == "graph+pdl"


def test_default_workload_is_the_sampled_glm_shape(monkeypatch):
    import sys
    monkeypatch.setattr(sys, "argv", ["bench.py"])
    assert bench.parse().workload == "glm4_9b"


def test_reference_arm_times_whole_rounds_with_the_same_config(monkeypatch, capsys):
    """--impl reference times K whole oracle rounds (every layer) after W untimed ones, reports
    ms_per_step of those rounds, and prints the config dict the GPU arm prints."""
    import json
    import sys
    monkeypatch.setattr(bench, "dist_setup", lambda gpus: (0, 1, 0))
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--workload", "tiny",
                                      "--steps", "3", "--warmup", "1"])
    bench.main()
    ref = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert ref["impl"] == "reference" and ref["steps"] == 3 and ref["warmup"] == 1
    assert ref["value"] == pytest.approx(1e3 / ref["ms_per_step"], rel=1e-9)
    assert "extrapolated" not in ref and "all 1 layers" in ref["cpu_baseline"]["sample"]
    assert ref["e2e"]["h2d_bytes_per_step"] == 0
    args = bench.parse()
    assert ref["config"] == bench.workload_config(args, bench.workload(args), 1)


def test_accept_histogram():
    import numpy as np
    D = 3
    # rows' committed lengths at the start of rounds 0..3 (row r of the history)
    n = np.array([[5, 9], [6, 13], [10, 15], [11, 16]])
    h = bench.accept_histogram(n, 1, 3, D)     # rounds 1 and 2: a = [3, 1], [0, 0]
    assert h["accept_len_hist"] == [2, 1, 0, 1]
    assert h["mean_accept_len"] == 1.0
    assert bench.accept_histogram(n, 0, 1, D)["accept_len_hist"] == [1, 0, 0, 1]
    bad = n.copy()
    bad[2, 0] = 20
    try:
        bench.accept_histogram(bad, 1, 2, D)
    except RuntimeError:
        pass
    else:
        raise AssertionError("an accept length above D must raise")
