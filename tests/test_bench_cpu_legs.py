"""The CPU legs of bench.py on a tiny workload: the single-threaded oracle sample
and the all-cores leg (spawned processes over disjoint (request, layer) units)
report consistent, positive throughput and say what they ran."""
import math

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


def test_variable_recall_oracle_sample_follows_the_workload():
    """The oracle sample of the variable-recall workload draws its budgets per
    (layer, step), its pool size per request and its preloaded residency the way
    the GPU run does: preloaded blocks sit in slots 0.. in ascending order with
    their bytes, and the budget stays in the workload's range."""
    import synth
    cfg = dict(bench.CONFIGS["c3"], layers=2, batch=2, ntok=2048, hq=8, hkv=2, head_dim=64, block_tokens=16,
               k=12, k_range=(4, 12))
    mb = _max_blocks(cfg, 8)
    samp = bench.OracleSample(cfg, 5, [(0, 0), (1, 1)], mb)
    nb0 = -(-cfg["ntok"] // cfg["block_tokens"])
    for (r, l), st in samp.state.items():
        f = synth.uniform_real(5, synth.KIND_FRAC, r, 0, 0, *cfg["frac_range"])
        res = synth.sample_sorted(5, synth.KIND_RESIDENT, l, r, nb0, int(round(f * nb0)))
        assert len(st["bos"]) == max(math.ceil(f * nb0), cfg["k"] + cfg["window"])
        assert list(st["bos"][: len(res)]) == list(res)
        for s_, b_ in enumerate(res):
            assert st["sob"][b_] == s_
            assert (st["pool"][s_] == st["region"][b_]).all()
    ks = {samp.budget(s, l) for s in range(20) for l in range(2)}
    assert min(ks) >= 4 and max(ks) <= 12 and len(ks) > 1
    qs = synth.q_ar1(5, cfg["layers"], cfg["batch"], cfg["hq"], cfg["head_dim"], 2, cfg["rho"])
    done, _ = samp.step(qs[0], 0)
    assert done == 2
