"""The CPU legs of bench.py (the oracle baseline and the row-parallel C++ baseline) run on tiny
samples without a GPU, so a round-end benchmark cannot fail in them."""
import bench


def test_oracle_leg_runs():
    rps, rounds, layers, w = bench.time_oracle("tiny", budget_s=0.2, max_rounds=2)
    assert rps > 0 and 1 <= rounds <= 2 and layers == 1 and w.name == "tiny"


def test_parallel_leg_runs_greedy_and_sampled():
    for name in ("tiny", "glm4_9b"):
        r = bench.time_cpu_parallel(name, budget_s=0.1, max_rounds=1, layers_sample=1)
        assert r["value"] > 0 and r["cores"] >= 1 and r["unit"] == "rounds/s"
