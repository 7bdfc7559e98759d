"""moe_layer_forward's CUDA-graph replay: the first call with a set of
arguments on a non-default stream captures the launch sequence, later calls
replay it.  A replay reads the buffers at replay time, so new inputs in the
same buffers give the new outputs, bitwise equal to direct launches; the
launch counter counts a replay's kernels.  GPU only."""
import numpy as np
import pytest
import torch

import expert_routing_ffn_gb300 as moe
import oracle
from expert_routing_ffn_gb300.layer import DeviceLayer, LayerBuffers, forward
from workloads import CONFIGS, make_tokens, make_weights

from parity import check_output, x_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,T", [("tiny", 16), ("dsv2lite", 8), ("dsv2lite", 1), ("granite", 200)])
def test_replay_matches_direct_launches(name, T):
    cfg = CONFIGS[name]
    W = make_weights(cfg)
    layer = DeviceLayer(cfg, W, T)
    stream = torch.cuda.Stream()
    xs = [make_tokens(cfg, T=T, batch=40 + i) for i in range(3)]
    xd = torch.empty((T, cfg.d), dtype=layer.dt, device="cuda")
    direct, replayed = [], []
    try:
        moe.moe_set_graph_replay(False)
        b0 = LayerBuffers(layer, T)
        for x in xs:
            xd.copy_(torch.from_numpy(x).to(layer.dt))
            torch.cuda.synchronize()
            n0 = moe.moe_launch_total()
            forward(layer, b0, xd, stream=stream)
            stream.synchronize()
            n_direct = moe.moe_launch_total() - n0
            direct.append(b0.out.clone())
        moe.moe_set_graph_replay(True)
        b1 = LayerBuffers(layer, T)
        for i, x in enumerate(xs):
            xd.copy_(torch.from_numpy(x).to(layer.dt))
            torch.cuda.synchronize()
            n0 = moe.moe_launch_total()
            forward(layer, b1, xd, stream=stream)
            stream.synchronize()
            assert moe.moe_launch_total() - n0 == n_direct
            replayed.append(b1.out.clone())
        st, det = moe.moe_check(layer.ws)
        assert st == moe.MOE_OK, (moe.status_string(st), det)
    finally:
        moe.moe_set_graph_replay(True)
    for a, b in zip(direct, replayed):
        assert torch.equal(a, b)
    assert not torch.equal(replayed[0], replayed[1])  # the replays saw the new inputs
    R = oracle.layer_forward(cfg, W, xs[-1])
    check_output(cfg, R, replayed[-1])


def test_replay_on_another_stream_and_inside_a_caller_capture():
    cfg = CONFIGS["dsv2lite"]
    W = make_weights(cfg)
    T = 8
    layer = DeviceLayer(cfg, W, T)
    b = LayerBuffers(layer, T)
    x = x_device(make_tokens(cfg, T=T, batch=50), layer.dt)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    forward(layer, b, x, stream=s1)  # captured on s1
    s1.synchronize()
    ref = b.out.clone()
    b.out.zero_()
    torch.cuda.synchronize()
    forward(layer, b, x, stream=s2)  # replayed on s2
    s2.synchronize()
    assert torch.equal(ref, b.out)
    # inside the caller's own capture the kernels are captured directly
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s1):
        forward(layer, b, x, stream=s1)
    b.out.zero_()
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(ref, b.out)
    assert moe.moe_check(layer.ws)[0] == moe.MOE_OK


@pytest.mark.parametrize("name,T", [("dsv2lite", 8), ("granite", 200)])
def test_forward_with_host_buffers(name, T):
    """moe_layer_forward_host copies the pinned input in and the output out
    around the layer, replayed as one graph: new host inputs in the same
    buffer give the new outputs, bitwise those of the device-buffer call."""
    from expert_routing_ffn_gb300.layer import forward_host
    cfg = CONFIGS[name]
    W = make_weights(cfg)
    layer = DeviceLayer(cfg, W, T)
    stream = torch.cuda.Stream()
    xd = torch.empty((T, cfg.d), dtype=layer.dt, device="cuda")
    host_x = torch.empty((T, cfg.d), dtype=layer.dt).pin_memory()
    host_out = torch.empty((T, cfg.d), dtype=torch.float32).pin_memory()
    b = LayerBuffers(layer, T)
    ref_b = LayerBuffers(layer, T)
    for batch in (60, 61, 63):  # seeds without near-tie tokens (checked on the oracle)
        x = make_tokens(cfg, T=T, batch=batch)
        host_x.copy_(torch.from_numpy(x).to(layer.dt))
        forward_host(layer, b, xd, host_x, host_out, stream=stream)
        stream.synchronize()
        forward(layer, ref_b, x_device(x, layer.dt), stream=stream)
        stream.synchronize()
        assert torch.equal(host_out, ref_b.out.cpu())
    assert moe.moe_check(layer.ws)[0] == moe.MOE_OK
    R = oracle.layer_forward(cfg, W, x)
    check_output(cfg, R, host_out.cuda())
