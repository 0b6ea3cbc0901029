"""The CPU legs of bench.py on a tiny workload: the single-threaded oracle sample
and the all-cores leg (spawned processes over disjoint (request, layer) units)
report consistent, positive throughput and say what they ran."""
import bench

TINY = dict(bench.CONFIGS["c1"], layers=2, batch=2, ntok=1000)


def _max_blocks(cfg, steps=80):
    return -(-(cfg["ntok"] + steps) // cfg["block_tokens"]) + 1


def test_single_thread_oracle_leg():
    import synth
    qs = synth.q_ar1(0, TINY["layers"], TINY["batch"], TINY["hq"], TINY["head_dim"], 4, TINY["rho"])
    r = bench.cpu_baseline(TINY, 0, qs, _max_blocks(TINY), None, budget_s=0.2, n_units=4)
    assert r["value"] > 0 and r["cores"] == 1 and r["kind"] == "oracle"
    assert "unit-steps" in r["sample"]


def test_all_cores_leg_splits_units_over_processes():
    r = bench.cpu_baseline_all_cores(TINY, 0, _max_blocks(TINY), budget_s=0.3, units_per_proc=1, procs=2)
    assert r["value"] > 0 and r["cores"] == 2 and r["kind"] == "oracle"
    assert "spawned processes" in r["sample"]
