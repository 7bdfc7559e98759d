"""The prefill FFN on CTA pairs (2-CTA MMA on 256-row tiles) against the
one-CTA kernel and the float64 oracle, through the C ABI.  Both kernels run
on the same inputs (the testing switch forces one or the other); each must
match the oracle, and the two outputs must agree closely (the same products
summed in the same K order per MMA).  GPU only.
"""
import pytest
import torch

import expert_routing_ffn_gb300 as moe
import oracle
from expert_routing_ffn_gb300.layer import DeviceLayer, LayerBuffers, forward
from workloads import CONFIGS, make_tokens, make_weights

from parity import check_output, check_routing, check_selection, x_device

pytestmark = pytest.mark.gpu

NOSHARED = CONFIGS["tiny"].with_(wtype="bf16", n_shared=0, I_shared=0, name="tiny-bf16-noshared")


@pytest.fixture(autouse=True)
def _restore_mode():
    yield
    moe.moe_testing_set_tc_pairs(-1)


@pytest.mark.parametrize("cfg,T,batch,policy", [(CONFIGS["dsv2lite"], 96, 0, None),
                                                (CONFIGS["dsv2lite"], 600, 1, None),
                                                (CONFIGS["granite"], 1024, 0, None),
                                                (CONFIGS["granite"], 333, 2, None),
                                                (NOSHARED, 200, 2, 2)])
def test_pairs_match_single_and_oracle(cfg, T, batch, policy):
    pol = cfg.policy if policy is None else policy
    W = make_weights(cfg)
    layer = DeviceLayer(cfg, W, T)
    assert moe.moe_expert_ffn_path(layer.dims.with_T(T)) == "tc-prefill"
    x = make_tokens(cfg, T=T, batch=batch)
    xd = x_device(x, layer.dt)
    outs = []
    for mode in (0, 1):
        moe.moe_testing_set_tc_pairs(mode)
        b = LayerBuffers(layer, T)
        b.y_perm.fill_(float("nan"))
        forward(layer, b, xd, policy=pol)
        st, det = moe.moe_check(layer.ws)
        assert st == moe.MOE_OK, (mode, moe.status_string(st), det)
        outs.append(b)
    R = oracle.layer_forward(cfg, W, x, policy=pol)
    for b in outs:
        check_routing(cfg, R, b)
        check_selection(cfg, R, b)
        check_output(cfg, R, b.out)
    a, p = outs[0].out, outs[1].out
    rel = float((a - p).norm() / a.norm())
    assert rel < 1e-5, rel


def test_pairs_qwen2_prefill():
    """The full Qwen2-57B-shaped prefill: pairs against the one-CTA kernel on
    every token (the oracle comparison of this layer runs in the layer
    tests, where the batch takes pairs by default)."""
    cfg = CONFIGS["qwen2"]
    W = make_weights(cfg)
    T = 4096
    layer = DeviceLayer(cfg, W, T)
    xd = x_device(make_tokens(cfg, T=T, batch=0), layer.dt)
    outs = []
    for mode in (0, 1):
        moe.moe_testing_set_tc_pairs(mode)
        b = LayerBuffers(layer, T)
        forward(layer, b, xd)
        st, det = moe.moe_check(layer.ws)
        assert st == moe.MOE_OK, (mode, moe.status_string(st), det)
        outs.append(b.out.clone())
        del b
    rel = float((outs[0] - outs[1]).norm() / outs[0].norm())
    assert rel < 1e-5, rel


def test_pairs_dsv2lite_prefill_4096_against_oracle():
    """The DeepSeek-V2-Lite-shaped 4096-token prefill (the default takes
    CTA pairs at this batch): routing on every token, outputs on a seeded
    512-token subset against the oracle on the batch's resident set."""
    import numpy as np
    from expert_routing_ffn_gb300.layer import as_u64
    from parity import to_np
    cfg = CONFIGS["dsv2lite"]
    W = make_weights(cfg)
    T = 4096
    layer = DeviceLayer(cfg, W, T)
    x = make_tokens(cfg, T=T, batch=0)
    b = LayerBuffers(layer, T)
    forward(layer, b, x_device(x, layer.dt))
    st, det = moe.moe_check(layer.ws)
    assert st == moe.MOE_OK, (moe.status_string(st), det)
    Rr = oracle.layer_forward(cfg, W, x, route_only=True)
    assert as_u64(to_np(b.batch_resident)[0]) == Rr.resident
    check_routing(cfg, Rr, b)
    check_selection(cfg, Rr, b)
    rows = np.sort(np.random.default_rng(1).choice(T, 512, replace=False))
    R = oracle.layer_forward(cfg, W, x[rows], resident=Rr.resident)
    check_output(cfg, R, b.out, tokens=rows)
