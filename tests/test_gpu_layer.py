"""Parity of the CUDA layer with the float64 oracle, through the C ABI.

Every layer shape at its full size (the prefill layer's expert outputs on a
seeded 512-token subset of the 4096-token batch, its routing on all tokens),
plus ragged and edge cases.  GPU only.
"""
from functools import lru_cache

import numpy as np
import pytest
import torch

import expert_routing_ffn_gb300 as moe
from expert_routing_ffn_gb300.layer import DeviceLayer, LayerBuffers, as_u64, forward
import oracle
from workloads import CONFIGS, make_tokens, make_weights

from parity import check_output, check_routing, check_selection, to_np, x_device

pytestmark = pytest.mark.gpu


@lru_cache(maxsize=2)
def _host(name):
    cfg = CONFIGS[name]
    return cfg, make_weights(cfg)


_dev_cache = {}


def _device(name, T):
    key = name
    if key in _dev_cache and _dev_cache[key].dims.T >= T:
        return _dev_cache[key]
    _dev_cache.clear()
    torch.cuda.empty_cache()
    cfg, W = _host(name)
    _dev_cache[key] = DeviceLayer(cfg, W, max(T, cfg.T))
    return _dev_cache[key]


def _run(name, T, batch=0, **kw):
    cfg, W = _host(name)
    layer = _device(name, T)
    x = make_tokens(cfg, T=T, batch=batch)
    bufs = LayerBuffers(layer, T)
    forward(layer, bufs, x_device(x, layer.dt), **kw)
    st, det = moe.moe_check(layer.ws)
    return cfg, W, layer, x, bufs, st, det


@pytest.mark.parametrize("name,T", [("tiny", 16), ("tiny", 1), ("tiny", 5), ("tiny", 64), ("tiny", 100),
                                    ("dsv2lite", 1), ("dsv2lite", 8), ("dsv2lite", 3),
                                    ("granite", 1), ("granite", 37), ("granite", 1024),
                                    ("granite", 65), ("granite", 200), ("dsv2lite", 96),
                                    ("mixtral", 1), ("mixtral", 8), ("mixtral", 32),
                                    ("mixtral", 100)])
def test_layer_matches_oracle(name, T):
    cfg, W, layer, x, bufs, st, det = _run(name, T)
    assert st == moe.MOE_OK, (moe.status_string(st), det)
    R = oracle.layer_forward(cfg, W, x)
    if cfg.n_resident > 0:
        assert R.resident_gap >= 1e-5
        assert as_u64(to_np(bufs.batch_resident)[0]) == R.resident
    check_routing(cfg, R, bufs)
    check_selection(cfg, R, bufs)
    check_output(cfg, R, bufs.out)


def test_prefill_layer_qwen2_shape():
    """4096-token prefill: routing on every token, outputs on a seeded subset."""
    name, T = "qwen2", 4096
    cfg, W, layer, x, bufs, st, det = _run(name, T)
    assert st == moe.MOE_OK, (moe.status_string(st), det)
    Rr = oracle.layer_forward(cfg, W, x, route_only=True)
    assert Rr.resident_gap >= 1e-5
    assert as_u64(to_np(bufs.batch_resident)[0]) == Rr.resident
    check_routing(cfg, Rr, bufs)
    check_selection(cfg, Rr, bufs)
    rows = np.sort(np.random.default_rng(0).choice(T, 512, replace=False))
    R = oracle.layer_forward(cfg, W, x[rows], resident=Rr.resident)
    check_output(cfg, R, bufs.out, tokens=rows)


@pytest.mark.parametrize("policy", [0, 1, 2, 3])
def test_policies_tiny(policy):
    cfg, W, layer, x, bufs, st, det = _run("tiny", 64, policy=policy)
    assert st == moe.MOE_OK
    R = oracle.layer_forward(cfg, W, x, policy=policy)
    check_selection(cfg, R, bufs)
    check_output(cfg, R, bufs.out)
    kinds = np.bincount(to_np(bufs.final_kind).ravel(), minlength=3)
    if policy == 0:
        assert kinds[1] > 0
    if policy in (2, 3):
        assert kinds[2] > 0


@pytest.mark.parametrize("name,T", [("tiny", 16),        # fp32 GEMV
                                    ("dsv2lite", 1),     # one-token GEMV, LoRE slots, shared experts
                                    ("granite", 1),      # one-token GEMV, d = 1536
                                    ("dsv2lite", 3),     # GEMV with rows per segment
                                    ("dsv2lite", 8),     # decode tensor-core path
                                    ("granite", 200)])   # prefill: chunked permutation, tensor-core GEMM
def test_stagewise_calls_equal_layer_forward(name, T):
    """The six stage calls in sequence give bitwise the same output as
    moe_layer_forward (whose epilogue fuses the partial-row sum, the LoRE B
    term and the combine)."""
    cfg, W, layer, x, bufs, st, _ = _run(name, T)
    assert st == moe.MOE_OK
    D = layer.dims.with_T(T)
    xd = x_device(x, layer.dt)
    b = LayerBuffers(layer, T)
    n_res = max(cfg.n_resident, 0)
    moe.moe_route(D, xd, layer.w_router, layer.router_bias, None, layer.w_prefetch, layer.w_ord,
                  layer.theta, cfg.tau, n_res, b.topk_idx, b.topk_gate, b.router_prob, b.delta_hat,
                  b.prefetch_mask, b.delta_star, b.batch_resident if n_res > 0 else None, layer.ws)
    moe.moe_select_resident(D, b.router_prob, b.topk_idx,
                            b.prefetch_mask if cfg.use_prefetch_mask else None,
                            b.batch_resident if n_res > 0 else layer.resident, cfg.policy,
                            cfg.gamma, b.delta_hat, b.delta_star, b.final_idx, b.final_gate,
                            b.final_kind, b.fetch_mask, b.counters, layer.ws)
    moe.moe_permute(D, b.final_idx, b.final_kind, b.expert_offsets, b.perm, b.inv_perm, layer.ws)
    moe.moe_expert_ffn(D, xd, layer.table, b.expert_offsets, b.perm, 1.0, b.y_perm, b.y_shared,
                       layer.ws)
    if cfg.r > 0:
        moe.moe_lore(D, xd, b.final_idx, b.final_kind, b.final_gate, layer.lore_a, layer.lore_b,
                     b.y_lore, layer.ws)
    moe.moe_combine(D, b.y_perm, b.inv_perm, b.final_gate, b.final_kind, b.y_shared,
                    b.y_lore if cfg.r > 0 else None, b.out)
    assert moe.moe_check(layer.ws)[0] == moe.MOE_OK
    assert torch.equal(b.final_idx, bufs.final_idx)
    assert torch.equal(b.out, bufs.out)


def test_permutation_invariants():
    cfg, W, layer, x, bufs, st, _ = _run("granite", 1024)
    off = to_np(bufs.expert_offsets)
    perm = to_np(bufs.perm)
    inv = to_np(bufs.inv_perm)
    fi = to_np(bufs.final_idx).ravel()
    fk = to_np(bufs.final_kind).ravel()
    valid = (fi >= 0) & (fk != moe.MOE_KIND_LORE)
    counts = np.bincount(fi[valid], minlength=cfg.N)
    assert off[0] == 0 and (np.diff(off) == counts).all()
    n = off[-1]
    assert n == valid.sum()
    assert (inv[perm[:n]] == np.arange(n)).all()
    assert (inv[~valid] == -1).all()
    for e in range(cfg.N):  # stable: slots of one expert in increasing slot order
        seg = perm[off[e]:off[e + 1]]
        assert (np.diff(seg) > 0).all() and (fi[seg] == e).all()


def test_deterministic():
    _, _, layer, x, b1, _, _ = _run("dsv2lite", 8)
    o1 = b1.out.clone()
    _, _, _, _, b2, _, _ = _run("dsv2lite", 8)
    assert torch.equal(o1, b2.out)


def test_empty_batch():
    cfg, W = _host("tiny")
    layer = _device("tiny", 16)
    bufs = LayerBuffers(layer, 1)
    x = torch.empty((0, cfg.d), dtype=layer.dt, device="cuda")
    forward(layer, bufs, x)
    assert moe.moe_check(layer.ws)[0] == moe.MOE_OK


def test_capacity_shortfall_reported_on_device():
    """An available set smaller than k under SUBSTITUTE is reported through
    the device error word (MOE_ERR_CAPACITY), without a fault."""
    cfg, W = _host("tiny")
    layer = _device("tiny", 16)
    x = make_tokens(cfg, T=4)
    bufs = LayerBuffers(layer, 4)
    layer.set_resident(0b1)
    try:
        forward(layer, bufs, x_device(x, layer.dt), policy=moe.MOE_MISS_SUBSTITUTE,
                use_prefetch_mask=0, n_resident=0)
        st, det = moe.moe_check(layer.ws)
        assert st == moe.MOE_ERR_CAPACITY
        assert to_np(bufs.counters)[7] == 4
    finally:
        layer.set_resident((1 << 64) - 1)
    # the error word was cleared by moe_check and the context is still usable
    forward(layer, bufs, x_device(x, layer.dt))
    assert moe.moe_check(layer.ws)[0] == moe.MOE_OK


def test_counters_match_oracle():
    cfg, W, layer, x, bufs, st, _ = _run("granite", 1024)
    R = oracle.layer_forward(cfg, W, x)
    c = to_np(bufs.counters)
    assert not R.excluded().any(), "near-tie tokens: counters are compared on exact inputs only"
    assert c[5] == R.delta_hat.sum()
    assert c[6] == R.delta_star.sum()
    overlap = sum(all((int(R.prefetch[t]) >> int(e)) & 1 for e in R.topk_idx[t]) for t in range(len(x)))
    assert c[4] == overlap
    routed_kept = sum(len(set(R.topk_idx[t]) & set(R.final_idx[t])) for t in range(len(x)))
    assert c[0] == routed_kept
    assert c[0] + c[1] == (R.final_idx >= 0).sum()


def test_all_tokens_on_the_same_experts():
    """Worst case for the FFN plan: a router bias sends every token to the same
    k experts (the most rows per expert, the most segments)."""
    cfg, W = _host("granite")
    Wb = type(W)(**{**W.__dict__})
    bias = np.zeros(cfg.N, np.float32)
    bias[:cfg.k] = 50.0
    Wb.router_bias = bias
    layer = DeviceLayer(cfg, Wb, 1024)
    x = make_tokens(cfg, T=1024)
    bufs = LayerBuffers(layer, 1024)
    forward(layer, bufs, x_device(x, layer.dt), use_prefetch_mask=0)
    st, det = moe.moe_check(layer.ws)
    assert st == moe.MOE_OK, (moe.status_string(st), det)
    off = to_np(bufs.expert_offsets)
    assert (np.diff(off)[:cfg.k] == 1024).all()
    R = oracle.layer_forward(cfg, Wb, x, use_prefetch=False)
    check_selection(cfg, R, bufs)
    check_output(cfg, R, bufs.out)


def test_exact_policy_with_staging_matches_plain_moe():
    """Correctness-preserving mode (APEX §4.3): experts outside the resident set
    are fetched from pinned host memory on a side stream (their device slots
    are first overwritten with NaN, so an unstaged or late copy would show)
    and the layer output equals the plain MoE layer."""
    cfg, W = _host("dsv2lite")
    T = 8
    layer = _device("dsv2lite", T)
    D = layer.dims.with_T(T)
    x = make_tokens(cfg, T=T, batch=3)
    xd = x_device(x, layer.dt)
    b = LayerBuffers(layer, T)
    moe.moe_route(D, xd, layer.w_router, layer.router_bias, None, layer.w_prefetch, layer.w_ord,
                  layer.theta, cfg.tau, cfg.n_resident, b.topk_idx, b.topk_gate, b.router_prob,
                  b.delta_hat, b.prefetch_mask, b.delta_star, b.batch_resident, layer.ws)
    moe.moe_select_resident(D, b.router_prob, b.topk_idx, None, b.batch_resident, moe.MOE_MISS_EXACT,
                            0.0, b.delta_hat, b.delta_star, b.final_idx, b.final_gate, b.final_kind,
                            b.fetch_mask, b.counters, layer.ws)
    fetch = as_u64(int(b.fetch_mask.item()))
    assert fetch != 0, "this batch fetches at least one expert"
    ids = [e for e in range(cfg.N) if (fetch >> e) & 1]
    host = [[t.cpu().pin_memory() for t in mats] for mats in (layer.w_gate, layer.w_up, layer.w_down)]
    saved = [(layer.w_gate[e].clone(), layer.w_up[e].clone(), layer.w_down[e].clone()) for e in ids]
    try:
        for e in ids:
            for m in (layer.w_gate, layer.w_up, layer.w_down):
                m[e].fill_(float("nan"))
        side = torch.cuda.Stream()
        done = torch.cuda.Event()
        nbytes = moe.moe_stage_experts(D, fetch, *host, list(layer.w_gate), list(layer.w_up),
                                       list(layer.w_down), side, done)
        assert nbytes == len(ids) * 3 * cfg.I * cfg.d * 2
        torch.cuda.current_stream().wait_event(done)
        moe.moe_permute(D, b.final_idx, b.final_kind, b.expert_offsets, b.perm, b.inv_perm, layer.ws)
        moe.moe_expert_ffn(D, xd, layer.table, b.expert_offsets, b.perm, 1.0, b.y_perm, b.y_shared,
                           layer.ws)
        moe.moe_combine(D, b.y_perm, b.inv_perm, b.final_gate, b.final_kind, b.y_shared, None, b.out)
        st, det = moe.moe_check(layer.ws)
        assert st == moe.MOE_OK, (moe.status_string(st), det)
        kinds = to_np(b.final_kind)
        assert (kinds == moe.MOE_KIND_FETCH).sum() == to_np(b.counters)[3] > 0
        R = oracle.layer_forward(cfg, W, x, policy=moe.MOE_MISS_EXACT)
        check_selection(cfg, R, b)
        check_output(cfg, R, b.out)
    finally:
        for e, (g, u, dn) in zip(ids, saved):
            layer.w_gate[e].copy_(g); layer.w_up[e].copy_(u); layer.w_down[e].copy_(dn)


@pytest.mark.parametrize("T", [1, 8, 32])
def test_floe_sparse_matches_oracle(T):
    """FloE contextual sparsity (method §1): each token keeps the m channels
    with the largest |x W_up| (m = ceil(0.1 I) = 1434 for I = 14336).  Kept
    sets are bit-exact on every slot whose |u| gap at the keep boundary is at
    least 1e-5 of max |u|; on the other slots (14336 channels make such gaps
    common) the GPU set must still be a valid top-m: m channels, none left
    out whose |u| exceeds a kept one's by more than that band.  Outputs on
    every token within the bf16 tolerance, those slots included."""
    cfg, W = _host("mixtral")
    layer = _device("mixtral", T)
    kf = np.float32(0.1)
    m = int(np.ceil(float(kf) * cfg.I - 1e-6))
    assert m == 1434
    x = make_tokens(cfg, T=T, batch=5)
    bufs = LayerBuffers(layer, T)
    forward(layer, bufs, x_device(x, layer.dt), keep_frac=float(kf))
    st, det = moe.moe_check(layer.ws)
    assert st == moe.MOE_OK, (moe.status_string(st), det)
    R = oracle.layer_forward(cfg, W, x, keep_m=m)
    check_selection(cfg, R, bufs, floe=False)
    check_output(cfg, R, bufs.out, floe=False)
    ptr, words = moe.moe_floe_kept_mask(layer.dims.with_T(T), layer.ws)
    rows = int(bufs.expert_offsets[-1])
    off = ptr - layer.ws.data_ptr()
    kept = layer.ws[off:off + rows * words * 4].view(torch.int32).cpu().numpy().view(np.uint32)
    kept = kept.reshape(rows, words)
    inv = to_np(bufs.inv_perm).reshape(T, cfg.k)
    fi = to_np(bufs.final_idx)
    n_exact = n_band = 0
    for t in range(T):
        for s in range(cfg.k):
            e = fi[t, s]
            pos = inv[t, s]
            so = list(R.final_idx[t]).index(e)
            bits = np.unpackbits(kept[pos].view(np.uint8), bitorder="little")[:cfg.I]
            got = np.nonzero(bits)[0]
            au = np.abs(W.w_up[e].astype(np.float64) @ x[t].astype(np.float64))
            band = 1e-5 * au.max()
            srt = np.sort(au)[::-1]
            if srt[m - 1] - srt[m] >= band:
                assert (got == R.kept[t, so]).all(), f"kept channels differ (token {t}, slot {s})"
                n_exact += 1
            else:
                assert got.size == m, f"token {t}, slot {s}: {got.size} channels kept"
                out = np.ones(cfg.I, bool)
                out[got] = False
                assert au[got].min() >= au[out].max() - band, f"token {t}, slot {s}: not a top-m set"
                n_band += 1
    assert n_exact > 0 and n_exact >= 4 * n_band


def test_expert_cache_over_decode_steps_matches_oracle():
    """Persistent expert cache (ELMoE-3D heat map with decay) over 48
    one-token decode steps of the DS-V2-Lite-shaped layer: each step runs the
    layer with resident = the cache, then moe_cache_update.  Every step is
    checked against the oracle's update from the same routed experts and the
    same incoming heat: heat within float32 rounding, the new cache bit-exact
    unless the oracle's heat gap at the capacity boundary is a near-tie, and
    the hit / slot / admit / evict counters exactly.  The layer's routing is
    checked against the oracle on every step too."""
    name, S, C, decay = "dsv2lite", 48, 24, 0.99
    cfg, W = _host(name)
    layer = _device(name, 1)
    bufs = LayerBuffers(layer, 1)
    dev = layer.ws.device
    heat = torch.zeros(cfg.N, dtype=torch.float32, device=dev)
    admit = torch.zeros(1, dtype=torch.int64, device=dev)
    stats = torch.zeros(4, dtype=torch.int32, device=dev)
    cache0 = (1 << C) - 1  # a predefined initial subset: experts 0 .. C-1
    layer.set_resident(cache0)
    h = np.zeros(cfg.N)
    cache = cache0
    want = np.zeros(4, np.int64)
    near = 0
    try:
        for s in range(S):
            x = make_tokens(cfg, T=1, batch=100 + s)
            forward(layer, bufs, x_device(x, layer.dt), n_resident=0)
            R = oracle.layer_forward(cfg, W, x, resident=cache, route_only=True)
            check_routing(cfg, R, bufs)
            check_selection(cfg, R, bufs)
            heat_in = heat.double().cpu().numpy()
            moe.moe_cache_update(layer.dims.with_T(1), bufs.topk_idx, decay, C, heat, layer.resident, admit, stats)
            torch.cuda.synchronize()
            routed = to_np(bufs.topk_idx).ravel()
            new, h, hits, gap = oracle.cache_update(routed, heat_in, decay, C, cache)
            np.testing.assert_allclose(heat.double().cpu().numpy(), h, rtol=2e-6, atol=1e-6)
            got = as_u64(to_np(layer.resident)[0])
            if gap >= 1e-5 * (1.0 + float(np.max(h))):
                assert got == new, (s, hex(got), hex(new))
            else:
                near += 1
            want += [hits, len(routed), bin(got & ~cache).count("1"), bin(cache & ~got).count("1")]
            assert as_u64(to_np(admit)[0]) == got & ~cache
            cache = got
        assert st_ok(layer)
        np.testing.assert_array_equal(to_np(stats).astype(np.int64), want)
        assert near < S // 4
        assert want[2] > 0  # the heat map moved experts in over these steps
    finally:
        layer.set_resident((1 << 64) - 1)


@pytest.mark.parametrize("tau", [0.6, 0.97])
@pytest.mark.parametrize("T", [1, 1024])
def test_granite_prefetch_thresholds_match_oracle(tau, T):
    """The Granite-shaped layer (SUBSTITUTE, available set = the prefetch set)
    at APEX's other two thresholds besides the default 0.9: delta_hat, the
    prefetch sets, the substitutes and the output against the oracle at the
    same tau; a lower threshold prefetches fewer experts on average."""
    cfg0, W = _host("granite")
    layer = _device("granite", T)
    x = make_tokens(cfg0, T=T, batch=5)
    bufs = LayerBuffers(layer, T)
    forward(layer, bufs, x_device(x, layer.dt), tau=tau)
    st, det = moe.moe_check(layer.ws)
    assert st == moe.MOE_OK, (moe.status_string(st), det)
    cfg = cfg0.with_(tau=tau)
    R = oracle.layer_forward(cfg, W, x)
    check_routing(cfg, R, bufs)
    check_selection(cfg, R, bufs)
    check_output(cfg, R, bufs.out)
    if T > 1:
        R9 = oracle.layer_forward(cfg0, W, x, route_only=True)
        dh, dh9 = R.delta_hat.mean(), R9.delta_hat.mean()
        assert (dh < dh9) if tau < cfg0.tau else (dh > dh9)


def st_ok(layer):
    st, _ = moe.moe_check(layer.ws)
    return st == moe.MOE_OK


def test_bounded_wait_times_out_and_the_context_stays_usable():
    """A device wait that can never finish (an mbarrier nothing arrives on)
    ends after its wall-clock bound with MOE_ERR_TIMEOUT in the error word, not
    with a hang or a trap; the next layer call on the same context is exact."""
    layer = _device("tiny", 16)
    moe.moe_testing_wait_timeout(layer.ws)
    st, det = moe.moe_check(layer.ws)
    assert (st, det) == (moe.MOE_ERR_TIMEOUT, -3)
    assert moe.moe_check(layer.ws) == (moe.MOE_OK, 0)  # moe_check cleared the word
    cfg, W, layer, x, bufs, st, det = _run("tiny", 16)
    assert st == moe.MOE_OK
    R = oracle.layer_forward(cfg, W, x)
    check_output(cfg, R, bufs.out)
