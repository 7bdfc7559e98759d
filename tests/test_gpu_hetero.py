"""Parity of the heterogeneous CPU-GPU path with the float64 oracle, through
the C ABI (SPICE write-up, CPU-GPU collaboration for prefetch misses, Fig. 6
and its cost model).

A routed expert outside the available set whose router probability is at
least gamma is computed exactly: fetched to the GPU, or run on the host cores
from the host copy of its weights, per expert by the cost model over the rows
of the batch that need it.  The cost model used here (1 MB over 1 GB/s
against 0.6 ms per host row) sends an expert needed by one row to the host
and one needed by two or more to the GPU.  On the resident-set layer the
device copies of every expert outside the resident set are overwritten with
NaN first: a fetched expert is restored by its copy from pinned host memory,
a host expert stays NaN on the device, so any GPU read of it would show.
GPU only.
"""
import numpy as np
import pytest
import torch

import expert_routing_ffn_gb300 as moe
import oracle
from expert_routing_ffn_gb300.layer import DeviceLayer, HeteroHost, LayerBuffers, as_u64, forward_hetero
from workloads import CONFIGS, make_tokens, make_weights

from parity import check_output, check_routing, check_selection, to_np, x_device

pytestmark = pytest.mark.gpu

SPLIT = dict(link_bps=1e9, expert_bytes=1e6, gpu_expert_s=0.0, cpu_row_s=6e-4, hidden_bytes=0.0)
ALL_HOST = dict(SPLIT, cpu_row_s=0.0)          # host rows cost nothing: never fetch
ALL_FETCH = dict(SPLIT, cpu_row_s=1.0)         # host rows cost a second: always fetch

_cache = {}


def _setup(name, T):
    if name not in _cache:
        _cache.clear()
        torch.cuda.empty_cache()
        cfg = CONFIGS[name]
        W = make_weights(cfg)
        layer = DeviceLayer(cfg, W, max(T, 128))
        host = HeteroHost(layer, max(T, 128))
        _cache[name] = (cfg, W, layer, host)
    return _cache[name]


def _lib_cost(c):
    return moe.hetero_cost(c["link_bps"], c["expert_bytes"], c["gpu_expert_s"], c["cpu_row_s"], c["hidden_bytes"])


FIXED = (1 << 24) - 1  # a predefined resident set: experts 0..23


def _run(name, T, cost, gamma, poison, fixed=False):
    """One hetero layer call; fixed: resident set = experts 0..23 instead of
    the batch's prefetch set (small batches then have exact misses too)."""
    cfg, W, layer, host = _setup(name, T)
    x = make_tokens(cfg, T=T, batch=11)
    if fixed:
        resident = FIXED
    else:
        resident = oracle.layer_forward(cfg, W, x, route_only=True).resident
    saved = []
    if poison:
        for e in range(cfg.N):
            if (resident >> e) & 1:
                continue
            saved.append((e, layer.w_gate[e].clone(), layer.w_up[e].clone(), layer.w_down[e].clone()))
            for m in (layer.w_gate, layer.w_up, layer.w_down):
                m[e].fill_(float("nan"))
    kw = {}
    if fixed:
        layer.set_resident(FIXED)
        kw["n_resident"] = 0
    try:
        bufs = LayerBuffers(layer, T)
        side = torch.cuda.Stream()
        ev = torch.cuda.Event()
        stats = forward_hetero(layer, bufs, x_device(x, layer.dt), host, _lib_cost(cost), side, ev, gamma=gamma,
                               **kw)
        st, det = moe.moe_check(layer.ws)
        assert st == moe.MOE_OK, (moe.status_string(st), det)
        R = oracle.layer_forward(cfg, W, x, policy=oracle.POL_HETERO, gamma=gamma, cost=cost,
                                 resident=FIXED if fixed else None)
    finally:
        for e, g, u, dn in saved:
            layer.w_gate[e].copy_(g); layer.w_up[e].copy_(u); layer.w_down[e].copy_(dn)
        layer.set_resident((1 << 64) - 1)
    return cfg, R, bufs, stats


@pytest.mark.parametrize("name,T,fixed,lore", [("dsv2lite", 1, True, False), ("dsv2lite", 3, True, False),
                                               ("dsv2lite", 8, False, True), ("dsv2lite", 64, False, True),
                                               ("dsv2lite", 96, False, True), ("granite", 200, False, False)])
def test_hetero_layer_matches_oracle(name, T, fixed, lore):
    """Routing, slot kinds (LoRE / fetch / host per the cost model) and the
    layer output against the oracle; the host slots' rows come from the
    library's host FFN."""
    poison = CONFIGS[name].n_resident > 0
    gamma = CONFIGS[name].gamma if lore else 0.0
    cfg, R, bufs, stats = _run(name, T, SPLIT, gamma, poison, fixed)
    check_routing(cfg, R, bufs)
    check_selection(cfg, R, bufs)
    check_output(cfg, R, bufs.out)
    kinds = np.bincount(R.final_kind.ravel(), minlength=4)
    assert stats.cpu_slots == kinds[oracle.KIND_CPU] == int(to_np(bufs.counters)[moe.MOE_CNT_CPU])
    assert stats.fetch_min_rows == 2
    assert kinds[oracle.KIND_CPU] > 0
    if T >= 64:
        assert kinds[1] > 0, "some experts are fetched"
    if lore:
        assert kinds[2] > 0
    gk = to_np(bufs.final_kind).ravel()
    assert stats.fetch_experts == len({int(e) for e, k in zip(to_np(bufs.final_idx).ravel(), gk) if k == 1})


@pytest.mark.parametrize("cost,kind", [(ALL_HOST, oracle.KIND_CPU), (ALL_FETCH, 1)])
def test_hetero_all_on_one_side(cost, kind):
    cfg, R, bufs, stats = _run("dsv2lite", 8, cost, CONFIGS["dsv2lite"].gamma, True)
    check_selection(cfg, R, bufs)
    check_output(cfg, R, bufs.out)
    gk = to_np(bufs.final_kind).ravel()
    other = oracle.KIND_CPU if kind == 1 else 1
    assert (gk == kind).sum() > 0 and (gk == other).sum() == 0


def test_select_hetero_places_host_slots_after_the_gpu_segments():
    """Stage-wise: moe_select_hetero gives the host slots the permuted
    positions after the GPU segments, in slot order; moe_permute fills the
    rest and leaves them; the masks and counters describe the kinds."""
    name, T = "dsv2lite", 64
    cfg, W, layer, host = _setup(name, T)
    x = make_tokens(cfg, T=T, batch=12)
    xd = x_device(x, layer.dt)
    D = layer.dims.with_T(T)
    b = LayerBuffers(layer, T)
    moe.moe_route(D, xd, layer.w_router, layer.router_bias, None, layer.w_prefetch, layer.w_ord, layer.theta,
                  cfg.tau, cfg.n_resident, b.topk_idx, b.topk_gate, b.router_prob, b.delta_hat, b.prefetch_mask,
                  b.delta_star, b.batch_resident, layer.ws)
    cpu_mask = torch.zeros(1, dtype=torch.int64, device="cuda")
    n_min = moe.moe_hetero_fetch_min_rows(_lib_cost(SPLIT))
    moe.moe_select_hetero(D, b.router_prob, b.topk_idx, None, b.batch_resident, cfg.gamma, n_min, b.delta_hat,
                          b.delta_star, b.final_idx, b.final_gate, b.final_kind, b.perm, b.inv_perm, b.fetch_mask,
                          cpu_mask, b.counters, layer.ws)
    moe.moe_permute(D, b.final_idx, b.final_kind, b.expert_offsets, b.perm, b.inv_perm, layer.ws)
    assert moe.moe_check(layer.ws)[0] == moe.MOE_OK
    fi, fk = to_np(b.final_idx).ravel(), to_np(b.final_kind).ravel()
    perm, inv, off = to_np(b.perm), to_np(b.inv_perm), to_np(b.expert_offsets)
    n_gpu = int(((fk == 0) | (fk == 1)).sum())
    assert off[-1] == n_gpu
    host = np.nonzero(fk == moe.MOE_KIND_CPU)[0]
    assert host.size > 0
    assert (inv[host] == n_gpu + np.arange(host.size)).all()
    assert (perm[n_gpu + np.arange(host.size)] == host).all()
    assert (inv[fk == moe.MOE_KIND_LORE] == -1).all()
    gpu = np.nonzero((fk == 0) | (fk == 1))[0]
    assert (perm[inv[gpu]] == gpu).all() and (inv[gpu] < n_gpu).all()
    fm, cm = as_u64(int(b.fetch_mask.item())), as_u64(int(cpu_mask.item()))
    assert fm == sum(1 << int(e) for e in set(fi[fk == 1].tolist()))
    assert cm == sum(1 << int(e) for e in set(fi[fk == moe.MOE_KIND_CPU].tolist()))
    assert fm & cm == 0
    c = to_np(b.counters)
    assert c[moe.MOE_CNT_CPU] == host.size and c[moe.MOE_CNT_FETCH] == (fk == 1).sum()
    # every expert on the host is needed by fewer rows than the threshold, every fetched one by at least that many
    for e in range(cfg.N):
        n = int(((fi == e) & ((fk == 1) | (fk == moe.MOE_KIND_CPU))).sum())
        if (cm >> e) & 1:
            assert 0 < n < n_min
        if (fm >> e) & 1:
            assert n >= n_min


def test_hetero_rejects_the_fused_layer_call():
    cfg, W, layer, host = _setup("dsv2lite", 8)
    from expert_routing_ffn_gb300.layer import forward
    bufs = LayerBuffers(layer, 8)
    with pytest.raises(moe.MoeError) as ei:
        forward(layer, bufs, x_device(make_tokens(cfg, T=8), layer.dt), policy=moe.MOE_MISS_HETERO)
    assert ei.value.status == moe.MOE_ERR_INVALID_ARG
