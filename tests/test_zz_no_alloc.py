"""The allocation-free FFN entry point (moe_expert_ffn_noalloc).

Some callers cannot allocate device memory at the moment they run the layer
(an engine plugin that is handed only its inputs and outputs, a decode loop
that cannot pay cudaMalloc's device-wide synchronisation).  For them the
library keeps a fixed 16 MiB scratch array per GPU.  This file checks, through the C ABI, that the entry point gives the
same expert outputs as the workspace-based moe_expert_ffn on two calls in a
row (with different routing, so the second call runs over the first call's
leftovers in the shared array), and that a batch too large for the array is
refused before any work is queued.

It sits in its own file, collected last, and builds everything it needs, so
it passes alone in a fresh process as well as after the other GPU tests.
"""
import ctypes as C

import pytest
import torch

import expert_routing_ffn_gb300 as moe
from expert_routing_ffn_gb300.layer import DeviceLayer, LayerBuffers, forward
from workloads import CONFIGS, make_tokens, make_weights

from parity import rel_l2, tol_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def layer():
    cfg = CONFIGS["dsv2lite"]
    return DeviceLayer(cfg, make_weights(cfg), 8)


def test_noalloc_ffn_matches_workspace_ffn_on_two_calls(layer):
    cfg, T = layer.cfg, 8
    D = layer.dims.with_T(T)
    status = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    for batch in (0, 1):
        xd = torch.from_numpy(make_tokens(cfg, T=T, batch=batch)).cuda().to(layer.dt)
        b = LayerBuffers(layer, T)
        forward(layer, b, xd)  # routing, permutation, and the workspace-based FFN
        ref_perm, ref_shared = b.y_perm.clone(), b.y_shared.clone()
        y_perm = torch.full_like(b.y_perm, float("nan"))
        y_shared = torch.full_like(b.y_shared, float("nan"))
        moe.moe_expert_ffn_noalloc(D, xd, layer.table, b.expert_offsets, b.perm, y_perm, y_shared,
                                   status)
        torch.cuda.synchronize()
        assert status.tolist() == [moe.MOE_OK, 0]
        n = int(b.expert_offsets[-1])
        assert n > 0
        assert rel_l2(y_perm[:n].cpu().numpy(), ref_perm[:n].cpu().numpy()) <= tol_for(cfg)
        assert rel_l2(y_shared.cpu().numpy(), ref_shared.cpu().numpy()) <= tol_for(cfg)


def test_noalloc_ffn_refuses_batches_beyond_its_scratch(layer):
    cfg = layer.cfg
    D = layer.dims.with_T(4096)
    dummy = C.c_void_p(layer.table.data_ptr())  # never dereferenced: refused first
    st = moe.lib().moe_expert_ffn_noalloc(C.byref(D), dummy, dummy, dummy, dummy, dummy, dummy,
                                         None, None)
    assert st == moe.MOE_ERR_CAPACITY
