"""The tensor-core prefill path's epilogue launch.

On batches of more than 64 tokens moe_layer_forward runs the expert FFN, the
LoRE z rows grouped by expert, then one launch that forms each LoRE slot's
B_e z, sums them per token and combines (instead of the stage-wise LoRE B,
LoRE sum and combine kernels).  Checked here: the output is bitwise that of
the stage-wise calls (moe_expert_ffn, moe_lore, moe_combine), and matches the
oracle, including tokens with no computed slot (every slot LoRE, no shared
expert).  GPU only.
"""
import numpy as np
import pytest
import torch

import expert_routing_ffn_gb300 as moe
import oracle
from expert_routing_ffn_gb300.layer import DeviceLayer, LayerBuffers, forward
from workloads import CONFIGS, make_tokens, make_weights

from parity import check_output, check_selection, to_np, x_device

pytestmark = pytest.mark.gpu

MISS_LORE = 2
# the small layer in bf16 without a shared expert: with every miss a LoRE
# slot, some tokens have no computed slot (seed checked on the oracle)
NOSHARED = CONFIGS["tiny"].with_(wtype="bf16", n_shared=0, I_shared=0, name="tiny-bf16-noshared")


def _stagewise(cfg, layer, xd, T, policy):
    D = layer.dims.with_T(T)
    b = LayerBuffers(layer, T)
    n_res = max(cfg.n_resident, 0)
    moe.moe_route(D, xd, layer.w_router, layer.router_bias, None, layer.w_prefetch, layer.w_ord,
                  layer.theta, cfg.tau, n_res, b.topk_idx, b.topk_gate, b.router_prob, b.delta_hat,
                  b.prefetch_mask, b.delta_star, b.batch_resident if n_res > 0 else None, layer.ws)
    moe.moe_select_resident(D, b.router_prob, b.topk_idx,
                            b.prefetch_mask if cfg.use_prefetch_mask else None,
                            b.batch_resident if n_res > 0 else layer.resident, policy,
                            cfg.gamma, b.delta_hat, b.delta_star, b.final_idx, b.final_gate,
                            b.final_kind, b.fetch_mask, b.counters, layer.ws)
    moe.moe_permute(D, b.final_idx, b.final_kind, b.expert_offsets, b.perm, b.inv_perm, layer.ws)
    moe.moe_expert_ffn(D, xd, layer.table, b.expert_offsets, b.perm, 1.0, b.y_perm,
                       b.y_shared if cfg.n_shared > 0 else None, layer.ws)
    if cfg.r > 0:
        moe.moe_lore(D, xd, b.final_idx, b.final_kind, b.final_gate, layer.lore_a, layer.lore_b,
                     b.y_lore, layer.ws)
    moe.moe_combine(D, b.y_perm, b.inv_perm, b.final_gate, b.final_kind,
                    b.y_shared if cfg.n_shared > 0 else None, b.y_lore if cfg.r > 0 else None, b.out)
    return b


@pytest.mark.parametrize("cfg,T,batch,policy", [(CONFIGS["dsv2lite"], 96, 0, None),
                                                (CONFIGS["dsv2lite"], 256, 3, None),
                                                (CONFIGS["granite"], 1024, 0, None),
                                                (NOSHARED, 200, 2, MISS_LORE),
                                                (NOSHARED, 130, 1, MISS_LORE)])
def test_prefill_epilogue_equals_stagewise_and_oracle(cfg, T, batch, policy):
    pol = cfg.policy if policy is None else policy
    W = make_weights(cfg)
    layer = DeviceLayer(cfg, W, T)
    assert moe.moe_expert_ffn_path(layer.dims.with_T(T)) == "tc-prefill"
    x = make_tokens(cfg, T=T, batch=batch)
    xd = x_device(x, layer.dt)
    bufs = LayerBuffers(layer, T)
    bufs.out.fill_(float("nan"))  # every row must be written
    forward(layer, bufs, xd, policy=pol)
    st, det = moe.moe_check(layer.ws)
    assert st == moe.MOE_OK, (moe.status_string(st), det)
    ref = _stagewise(cfg, layer, xd, T, pol)
    assert moe.moe_check(layer.ws)[0] == moe.MOE_OK
    assert torch.equal(ref.final_idx, bufs.final_idx)
    assert torch.equal(ref.out, bufs.out)
    R = oracle.layer_forward(cfg, W, x, policy=pol)
    check_selection(cfg, R, bufs)
    check_output(cfg, R, bufs.out)
    fk = to_np(bufs.final_kind)
    if cfg.r > 0:
        assert (fk == moe.MOE_KIND_LORE).sum() > 0
    if cfg is NOSHARED:
        none = ((fk == moe.MOE_KIND_LORE) | (to_np(bufs.final_idx) < 0)).all(axis=1)
        assert none.sum() > 0, "tokens without a computed slot"
        assert torch.isfinite(bufs.out).all()


def test_prefill_epilogue_repeats_bitwise():
    """Three calls on the same buffers (captured once, then replayed) give
    the same output bitwise."""
    cfg = CONFIGS["dsv2lite"]
    W = make_weights(cfg)
    T = 200
    layer = DeviceLayer(cfg, W, T)
    xd = x_device(make_tokens(cfg, T=T, batch=5), layer.dt)
    bufs = LayerBuffers(layer, T)
    stream = torch.cuda.Stream()
    outs = []
    for _ in range(3):
        bufs.out.zero_()
        torch.cuda.synchronize()
        forward(layer, bufs, xd, stream=stream)
        stream.synchronize()
        outs.append(bufs.out.clone())
    assert moe.moe_check(layer.ws)[0] == moe.MOE_OK
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])


@pytest.mark.parametrize("r", [16, 32, 48, 64])
def test_grouped_lore_on_tensor_cores_matches_oracle(r):
    """Grouped LoRE products of a bf16 layer with r a multiple of 16 (up to
    64) and d a multiple of 256 run as warp-level MMAs (z from bf16 x and
    A_e, B_e z in tf32): the DeepSeek-V2-Lite shape at rank r, every miss a
    LoRE slot (experts with more than 16 LoRE slots, so several 16-position
    tiles), outputs against the oracle, and the stage-wise calls give the
    same bits."""
    cfg = CONFIGS["dsv2lite"].with_(r=r, name=f"dsv2lite-r{r}")
    T = 256
    W = make_weights(cfg)
    layer = DeviceLayer(cfg, W, T)
    x = make_tokens(cfg, T=T, batch=2)
    xd = x_device(x, layer.dt)
    b = LayerBuffers(layer, T)
    forward(layer, b, xd, policy=MISS_LORE)
    st, det = moe.moe_check(layer.ws)
    assert st == moe.MOE_OK, (moe.status_string(st), det)
    fi, fk = to_np(b.final_idx), to_np(b.final_kind)
    per_expert = np.bincount(fi[fk == moe.MOE_KIND_LORE], minlength=cfg.N)
    assert per_expert.max() > 16, per_expert
    R = oracle.layer_forward(cfg, W, x, policy=MISS_LORE)
    check_selection(cfg, R, b)
    check_output(cfg, R, b.out)
    s = _stagewise(cfg, layer, xd, T, MISS_LORE)
    assert torch.equal(s.out, b.out)
