"""The heterogeneous CPU-GPU path on the CPU (SPICE write-up, CPU-GPU
collaboration for prefetch misses, Fig. 6 and its cost model).

  - the oracle's per-miss decision is pinned to the page's cost formula by
    hand-worked numbers and by its limits;
  - the oracle's HETERO layer splits exactly the misses the formula says, per
    expert, by the rows of the batch that need it (recounted here), and its
    outputs equal the plain MoE layer's except on LoRE slots;
  - the library's threshold form of the decision (moe_hetero_fetch_min_rows)
    agrees with the oracle's decision on every row count;
  - the library's host expert FFN (moe_cpu_experts, pure host code) matches
    the oracle's expert FFN, and its result does not depend on the number of
    host threads.
"""
import math

import numpy as np
import pytest
import torch

import expert_routing_ffn_gb300 as moe
import oracle
from workloads import CONFIGS, make_tokens, make_weights

# DS-V2-Lite-shaped expert over a PCIe 4.0 x16 link (worked by hand):
# fetch = 17301504 / 32e9 + 5e-6 = 545.672 us; CPU(n) = n (200 us + 2*4096/32e9)
# = n * 200.256 us -> CPU for n = 1, 2 (200.3, 400.5 us), fetch from n = 3 (600.8 us)
PCIE = dict(link_bps=32e9, expert_bytes=17301504.0, gpu_expert_s=5e-6, cpu_row_s=200e-6, hidden_bytes=4096.0)


def test_cost_model_hand_worked():
    assert [oracle.hetero_fetch(n, PCIE)[0] for n in range(1, 6)] == [False, False, True, True, True]
    _, gap = oracle.hetero_fetch(2, PCIE)
    fetch, cpu2 = 17301504 / 32e9 + 5e-6, 2 * 200e-6 + 2 * 2 * 4096 / 32e9
    assert gap == pytest.approx(abs(fetch - cpu2) / fetch, rel=1e-12)


def test_cost_model_limits():
    # an infinitely fast link: fetch iff the GPU is faster than n rows on the host
    fast = dict(PCIE, link_bps=1e300)
    assert oracle.hetero_fetch(1, dict(fast, gpu_expert_s=1e-6, cpu_row_s=2e-6))[0]
    assert not oracle.hetero_fetch(1, dict(fast, gpu_expert_s=3e-6, cpu_row_s=2e-6))[0]
    # free host compute and no hidden state: never fetch
    assert not oracle.hetero_fetch(1000, dict(PCIE, cpu_row_s=0.0, hidden_bytes=0.0))[0]
    # equal costs go to the host
    tie = dict(link_bps=1.0, expert_bytes=2.0, gpu_expert_s=0.0, cpu_row_s=1.0, hidden_bytes=0.0)
    assert not oracle.hetero_fetch(2, tie)[0] and oracle.hetero_fetch(3, tie)[0]
    assert oracle.hetero_fetch(2, tie)[1] == 0.0


def _lib_cost(c):
    return moe.hetero_cost(c["link_bps"], c["expert_bytes"], c["gpu_expert_s"], c["cpu_row_s"], c["hidden_bytes"])


@pytest.mark.parametrize("c", [
    PCIE,
    dict(PCIE, link_bps=190e9),
    dict(PCIE, cpu_row_s=1e-9),
    dict(link_bps=1.0, expert_bytes=2.0, gpu_expert_s=0.0, cpu_row_s=1.0, hidden_bytes=0.0),
    dict(link_bps=3e9, expert_bytes=1e6, gpu_expert_s=1e-5, cpu_row_s=7e-5, hidden_bytes=3584 * 2),
    dict(link_bps=1e9, expert_bytes=1e6, gpu_expert_s=0.0, cpu_row_s=6e-4, hidden_bytes=0.0),
])
def test_library_threshold_agrees_with_the_oracle(c):
    n_min = moe.moe_hetero_fetch_min_rows(_lib_cost(c))
    for n in range(1, 200):
        assert oracle.hetero_fetch(n, c)[0] == (n >= n_min), (n, n_min)


def test_library_threshold_edges():
    assert moe.moe_hetero_fetch_min_rows(_lib_cost(dict(PCIE, cpu_row_s=0.0, hidden_bytes=0.0))) == 2**31 - 1
    assert moe.moe_hetero_fetch_min_rows(_lib_cost(dict(PCIE, expert_bytes=0.0, gpu_expert_s=0.0))) == 1
    for bad in (dict(PCIE, link_bps=0.0), dict(PCIE, cpu_row_s=-1.0), dict(PCIE, expert_bytes=math.nan)):
        with pytest.raises(ValueError):
            moe.moe_hetero_fetch_min_rows(_lib_cost(bad))


def _small_layer(**kw):
    cfg = CONFIGS["dsv2lite"].with_(d=256, I=64, I_shared=64, **kw)
    return cfg, make_weights(cfg)


# n_min = 2: an expert needed by one row of the batch goes to the host
SPLIT = dict(link_bps=1e9, expert_bytes=1e6, gpu_expert_s=0.0, cpu_row_s=6e-4, hidden_bytes=0.0)


def _median_missing_prob(cfg, W, x):
    """gamma at the median router probability of the routed experts outside
    the resident set, so that both LoRE and exact misses occur."""
    R = oracle.layer_forward(cfg, W, x, route_only=True)
    miss = [R.prob[t, e] for t in range(x.shape[0]) for e in R.topk_idx[t] if not (R.resident >> int(e)) & 1]
    return float(np.median(miss))


@pytest.mark.parametrize("T,lore", [(8, True), (32, True), (32, False)])
def test_oracle_hetero_layer_splits_misses_by_the_cost_model(T, lore):
    cfg, W = _small_layer()
    x = make_tokens(cfg, T=T, batch=2)
    gamma = _median_missing_prob(cfg, W, x) if lore else 0.0
    R = oracle.layer_forward(cfg, W, x, policy=oracle.POL_HETERO, gamma=gamma, cost=SPLIT)
    Re = oracle.layer_forward(cfg, W, x, policy=0, resident=R.resident)
    avail = R.resident
    rows = {}
    for t in range(T):
        for e, a in zip(R.topk_idx[t], R.prob[t, R.topk_idx[t]]):
            if not (avail >> int(e)) & 1 and a >= gamma:
                rows[int(e)] = rows.get(int(e), 0) + 1
    n_cpu = n_fetch = n_lore = 0
    for t in range(T):
        assert sorted(R.final_idx[t]) == sorted(R.topk_idx[t])      # exact or LoRE: never substituted
        for e, kd, a in zip(R.final_idx[t], R.final_kind[t], R.prob[t, R.final_idx[t]]):
            e = int(e)
            if (avail >> e) & 1:
                assert kd == 0
            elif a < gamma:
                assert kd == 2
                n_lore += 1
            else:
                want = 1 if oracle.hetero_fetch(rows[e], SPLIT)[0] else oracle.KIND_CPU
                assert kd == want
                n_cpu += kd == oracle.KIND_CPU
                n_fetch += kd == 1
    assert n_cpu > 0 and n_fetch > 0
    if gamma > 0:
        assert n_lore > 0
    else:
        # no LoRE: every miss is exact, so the output is the plain MoE layer's
        np.testing.assert_allclose(R.out, Re.out, rtol=0, atol=0)
    # the cost margin is set on tokens with an exact miss, and only there
    has_exact = np.array([any(k in (1, oracle.KIND_CPU) for k in R.final_kind[t]) for t in range(T)])
    assert np.isfinite(R.margin[has_exact, oracle.M_COST]).all()
    assert np.isinf(R.margin[~has_exact, oracle.M_COST]).all()


def _host_inputs(cfg, W, T, seed):
    rng = np.random.default_rng(seed)
    x = make_tokens(cfg, T=T, batch=seed)
    idx = np.stack([rng.choice(cfg.N, cfg.k, replace=False) for _ in range(T)]).astype(np.int32)
    kind = rng.choice([0, 1, 2, 3], size=(T, cfg.k), p=[0.3, 0.1, 0.1, 0.5]).astype(np.int32)
    return x, idx, kind


@pytest.mark.parametrize("name,T", [("tiny", 16), ("small_bf16", 12)])
def test_host_expert_ffn_matches_the_oracle(name, T):
    if name == "tiny":
        cfg = CONFIGS["tiny"]
        W = make_weights(cfg)
    else:
        cfg, W = _small_layer()
    D = moe.make_dims(T, cfg.d, cfg.N, cfg.k, cfg.I, cfg.n_shared, cfg.I_shared, cfg.r, wtype=cfg.wtype)
    x, idx, kind = _host_inputs(cfg, W, T, 7)
    dt = torch.bfloat16 if cfg.wtype == "bf16" else torch.float32
    hx = torch.from_numpy(x).to(dt).contiguous()
    hw = [[torch.from_numpy(M[e]).to(dt).contiguous() for e in range(cfg.N)] for M in (W.w_gate, W.w_up, W.w_down)]
    scratch = torch.empty(moe.moe_cpu_experts_scratch_size(D), dtype=torch.uint8)
    outs = []
    for threads in (1, 3, 0):
        y = torch.full((T * cfg.k, cfg.d), float("nan"), dtype=torch.float32)
        n, first = moe.moe_cpu_experts(D, hx, torch.from_numpy(idx), torch.from_numpy(kind), *hw, y, scratch,
                                       n_threads=threads)
        outs.append(y[:n].clone())
    assert all(torch.equal(outs[0], o) for o in outs[1:]), "result depends on the thread count"
    host = [(t, s) for t in range(T) for s in range(cfg.k) if kind[t, s] == 3]
    assert n == len(host) and first == int(((kind == 0) | (kind == 1)).sum())
    tol = 1e-5
    for j, (t, s) in enumerate(host):
        e = idx[t, s]
        want = oracle.expert_ffn(x[t], W.w_gate[e], W.w_up[e], W.w_down[e])
        got = outs[0][j].double().numpy()
        assert np.linalg.norm(got - want) <= tol * np.linalg.norm(want), (t, s)


def test_host_expert_ffn_rejects_bad_arguments():
    cfg, W = _small_layer()
    T = 4
    D = moe.make_dims(T, cfg.d, cfg.N, cfg.k, cfg.I, cfg.n_shared, cfg.I_shared, cfg.r, wtype="bf16")
    hx = torch.zeros((T, cfg.d), dtype=torch.bfloat16)
    idx = torch.zeros((T, cfg.k), dtype=torch.int32)
    kind = torch.full((T, cfg.k), 3, dtype=torch.int32)
    hw = [[torch.zeros((cfg.I, cfg.d), dtype=torch.bfloat16) for _ in range(cfg.N)] for _ in range(3)]
    y = torch.zeros((T * cfg.k, cfg.d), dtype=torch.float32)
    small = torch.empty(16, dtype=torch.uint8)
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_cpu_experts(D, hx, idx, kind, *hw, y, small)
    assert ei.value.status == moe.MOE_ERR_INVALID_ARG
    scratch = torch.empty(moe.moe_cpu_experts_scratch_size(D), dtype=torch.uint8)
    bad = idx.clone()
    bad[1, 2] = cfg.N
    with pytest.raises(moe.MoeError):
        moe.moe_cpu_experts(D, hx, bad, kind, *hw, y, scratch)
    # no host slot: nothing computed, the first row is the GPU slot count
    n, first = moe.moe_cpu_experts(D, hx, idx, torch.zeros_like(kind), *hw, y, scratch)
    assert (n, first) == (0, T * cfg.k)
