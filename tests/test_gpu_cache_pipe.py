"""The overlapped expert-cache pipeline against the oracle, through the C ABI
(ELMoE-3D heat map with decay; SPICE: copies land before the layer that
needs them).

Every expert outside the start set (experts 0..23) has its device copy
overwritten with NaN before the run: an expert enters a step's resident set
only after its copy from pinned host memory has landed, so a step that used
an expert too early would produce NaN.  Each step is checked against the
oracle run on the resident set that step actually used (read back from the
pipeline), so the comparison holds whatever the copies' timing.  GPU only.
"""
import numpy as np
import pytest
import torch

import expert_routing_ffn_gb300 as moe
import oracle
from expert_routing_ffn_gb300.layer import CachePipeline, DeviceLayer, LayerBuffers, as_u64
from workloads import CONFIGS, make_tokens, make_weights

from parity import check_output, check_routing, check_selection, to_np, x_device

pytestmark = pytest.mark.gpu

START = (1 << 24) - 1


@pytest.fixture(scope="module")
def setup():
    cfg = CONFIGS["dsv2lite"]
    W = make_weights(cfg)
    layer = DeviceLayer(cfg, W, 8)
    yield cfg, W, layer
    del layer
    torch.cuda.empty_cache()


def _poison(layer, cfg):
    saved = []
    for e in range(cfg.N):
        if (START >> e) & 1:
            continue
        saved.append((e, layer.w_gate[e].clone(), layer.w_up[e].clone(), layer.w_down[e].clone()))
        for m in (layer.w_gate, layer.w_up, layer.w_down):
            m[e].fill_(float("nan"))
    return saved


def _restore(layer, saved):
    for e, g, u, dn in saved:
        layer.w_gate[e].copy_(g); layer.w_up[e].copy_(u); layer.w_down[e].copy_(dn)


@pytest.mark.parametrize("policy,T,steps", [(moe.MOE_MISS_HYBRID, 1, 48), (moe.MOE_MISS_HYBRID, 8, 24),
                                            (moe.MOE_MISS_EXACT, 1, 32)])
def test_cache_pipeline_steps_match_the_oracle(setup, policy, T, steps):
    cfg, W, layer = setup
    stream = torch.cuda.current_stream()
    pipe = CachePipeline(layer, capacity=24, decay=0.99, max_flight_experts=4, stream=stream)
    saved = _poison(layer, cfg)
    bufs = LayerBuffers(layer, T)
    try:
        pipe.start(START)
        landed_ever = START
        for s in range(steps):
            x = make_tokens(cfg, T=T, batch=300 + s)
            pipe.step(bufs, x_device(x, layer.dt), policy=policy, n_resident=0)
            stream.synchronize()
            st, det = moe.moe_check(layer.ws)
            assert st == moe.MOE_OK, (moe.status_string(st), det)
            resident = START if s == 0 else pipe.resident_used(s)
            # the set a step runs on is inside the cache and holds only landed experts
            assert resident & ~pipe.pipe.landed & ~landed_ever == 0
            R = oracle.layer_forward(cfg, W, x, resident=resident, policy=policy)
            check_routing(cfg, R, bufs)
            check_selection(cfg, R, bufs)
            check_output(cfg, R, bufs.out)
            landed_ever |= pipe.pipe.landed
        pipe.drain()
        p = pipe.pipe
        assert p.staged_experts > 0, "the heat map admitted experts and they were copied"
        assert p.staged_bytes == p.staged_experts * 3 * cfg.I * cfg.d * 2
        assert p.in_flight == 0
        # the cache after the last step, and every member of it has landed
        last = as_u64(int(pipe.ring[((steps - 1) % moe.MOE_CACHE_RING) * 4].item()))
        assert bin(last).count("1") == 24 and last & ~p.landed == 0
        if policy == moe.MOE_MISS_EXACT:
            assert p.stall_experts + p.in_time_experts > 0
            assert to_np(bufs.final_kind).max() <= moe.MOE_KIND_FETCH
    finally:
        _restore(layer, saved)


@pytest.mark.parametrize("field,value", [("decay", 1.5), ("capacity", -1), ("host_ring", None)])
def test_cache_pipeline_start_rejects_bad_state(setup, field, value):
    cfg, W, layer = setup
    pipe = CachePipeline(layer, capacity=24, decay=0.99)
    setattr(pipe.pipe, field, value)
    with pytest.raises(moe.MoeError) as ei:
        pipe.start(START)
    assert ei.value.status == moe.MOE_ERR_INVALID_ARG
