"""bench.py's workload tables and the oracle steps its CPU baseline and
reference arm time, on the CPU (no GPU)."""
import numpy as np

import bench
from workloads import CONFIGS, make_tokens, make_weights


def test_every_workload_names_a_layer_and_a_phase():
    for name, spec in bench.WORKLOADS.items():
        cfg_name, T, phase = spec[:3]
        assert cfg_name in CONFIGS and T > 0 and phase in ("decode", "prefill"), name
        if len(spec) > 3:
            assert 0.0 < spec[3] <= 1.0
    assert bench.DEFAULT_WORKLOAD in bench.WORKLOADS
    for table in (bench.CACHE_WORKLOADS, bench.LOOKAHEAD_WORKLOADS, bench.BITSLICE_WORKLOADS):
        for name in table:
            assert name in bench.WORKLOADS, name
    for J, tau, d_min in bench.LOOKAHEAD_WORKLOADS.values():
        assert 1 <= J <= 16 and d_min >= 0 and np.isfinite(tau)
    for bits in bench.BITSLICE_WORKLOADS.values():
        assert 1 <= bits <= 8


def test_oracle_steps_of_the_added_workloads_run():
    """The reference arm's step for a look-ahead workload runs the layer and
    the look-ahead depth; a bit-sliced workload's step gives a finite draft
    output that moves towards the dense layer's as the planes grow."""
    cfg = CONFIGS["tiny"]
    W = make_weights(cfg)
    x = make_tokens(cfg, T=2, batch=4)
    bench.LOOKAHEAD_WORKLOADS["tiny-lookahead-test"] = (3, 0.3, 1)
    try:
        bench.oracle_step(cfg, W, x, "tiny-lookahead-test")
    finally:
        del bench.LOOKAHEAD_WORKLOADS["tiny-lookahead-test"]
    ys = {b: bench.BitsliceOracle(cfg, W, b).token(x[0]) for b in (2, 4, 8)}
    for y in ys.values():
        assert y.shape == (cfg.d,) and np.isfinite(y).all()
    assert np.linalg.norm(ys[2] - ys[8]) > np.linalg.norm(ys[4] - ys[8]) > 0


def test_cpu_baseline_uses_every_core_and_reports_one_thread():
    """Decode: several T-token batches at once so that every core of the
    affinity mask has a token; prefill: tokens of one batch, one per core.
    Both carry a single-thread figure."""
    cfg = CONFIGS["tiny"]
    W = make_weights(cfg)
    r = bench.cpu_baseline(cfg, W, 2, 0.2)
    cores = bench.host_cores()
    assert r["kind"] == "oracle" and r["value"] > 0
    assert r["cores"] == 2 * max(1, cores // 2) or cores < 2
    assert r["single_thread"]["cores"] == 1 and r["single_thread"]["value"] > 0
    p = bench.cpu_baseline(cfg, W, 96, 0.2)
    assert p["cores"] == cores and p["value"] > 0 and p["single_thread"]["value"] > 0
    assert "of the 96 tokens" in p["sample"]


def test_fractions_and_nested_lines():
    f = bench.fractions(5000.0, 6694.5, bench.NOMINAL_HBM_GBS, "measured")
    assert f["frac"] == 5000.0 / 6694.5 and f["frac_of_nominal"] == 5000.0 / 8000.0
    line = {"metric": "m", "value": 1.0, "impl": "reference", "roofline": {}, "n_gpus": 1}
    assert bench.nested(line) == {"value": 1.0, "roofline": {}}
    assert bench.WORKLOADS[bench.PREFILL_WORKLOAD][2] == "prefill"
