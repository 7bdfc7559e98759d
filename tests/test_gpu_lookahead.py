"""Parity of the confidence-aware look-ahead prefetch depth (SPICE,
confidence-aware adaptive prefetch) with the float64 oracle, through the C
ABI.  GPU only."""
import numpy as np
import pytest
import torch

import expert_routing_ffn_gb300 as moe
import oracle
from workloads import CONFIGS, make_lookahead_routers, make_tokens

pytestmark = pytest.mark.gpu


def _dev(a, dt):
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda").to(dt)


def _run(cfg, x, Ws, biases, tau, d_min):
    T, J = x.shape[0], len(Ws)
    dims = moe.make_dims(T, cfg.d, cfg.N, cfg.k, cfg.I, cfg.n_shared, cfg.I_shared, cfg.r, wtype=cfg.wtype)
    wt = moe.wdtype(dims)
    ws = torch.zeros(moe.moe_workspace_size(dims), dtype=torch.uint8, device="cuda")
    xd = _dev(x, wt)
    Wd = [_dev(W, wt) for W in Ws]
    bd = None if biases is None else [_dev(b, torch.float32) for b in biases]
    logits = torch.zeros((J, T, cfg.N), dtype=torch.float32, device="cuda")
    conf = torch.zeros((T, J), dtype=torch.float32, device="cuda")
    depth = torch.full((T,), -1, dtype=torch.int32, device="cuda")
    tok = torch.full((T, J), -1, dtype=torch.int64, device="cuda")
    lay = torch.full((J,), -1, dtype=torch.int64, device="cuda")
    moe.moe_prefetch_depth(dims, xd, Wd, bd, tau, d_min, logits, conf, depth, tok, lay, ws)
    torch.cuda.synchronize()
    st, _ = moe.moe_check(ws)
    assert st == moe.MOE_OK
    u64 = lambda t: t.cpu().numpy().view(np.uint64)
    return conf.double().cpu().numpy(), depth.cpu().numpy(), u64(tok), u64(lay), logits.cpu().numpy()


# (config, tokens, look-ahead layers, d_min, quantile of layer-1 confidence used as tau)
CASES = [("tiny", 16, 3, 0, 0.4), ("dsv2lite", 1, 4, 1, 0.5), ("dsv2lite", 8, 4, 0, 0.3),
         ("dsv2lite", 300, 4, 2, 0.5),   # more than 64 tokens: the tensor-core router GEMM
         ("granite", 1024, 2, 0, 0.5), ("qwen2", 200, 3, 1, 0.6), ("dsv2lite", 37, 16, 0, 0.2)]


@pytest.mark.parametrize("name,T,J,d_min,q", CASES)
def test_prefetch_depth_matches_oracle(name, T, J, d_min, q):
    """conf within float32 rounding; depth and the kept top-k sets bit-exact
    on every token whose decisive margins (|conf - tau| over the layers the
    scan reads, the logit gap at position k of the kept layers) are at least
    1e-4; the layer masks are the OR of the token masks and match the oracle's
    when no token is excluded."""
    cfg = CONFIGS[name]
    Ws, biases = make_lookahead_routers(cfg, J)
    x = make_tokens(cfg, T=T, batch=7)
    c0, _, _, _, _ = oracle.prefetch_depth(x, Ws, biases, cfg.k, 0.0, 0)
    tau = float(np.quantile(c0[:, min(1, J - 1)], q)) + 1e-3  # off every sampled value
    conf_o, depth_o, tok_o, lay_o, margin = oracle.prefetch_depth(x, Ws, biases, cfg.k, tau, d_min)
    conf, depth, tok, lay, logits = _run(cfg, x, Ws, biases, tau, d_min)
    for j in range(J):
        lo = (x.astype(np.float64) @ Ws[j].astype(np.float64).T)
        if biases is not None:
            lo += biases[j]
        np.testing.assert_allclose(logits[j], lo, rtol=1e-4, atol=1e-4)
    np.testing.assert_allclose(conf, conf_o, rtol=1e-5, atol=1e-5)
    keep = margin >= 1e-4
    assert keep.sum() >= 0.9 * T
    np.testing.assert_array_equal(depth[keep], depth_o[keep])
    np.testing.assert_array_equal(tok[keep], tok_o[keep])
    assert ((depth >= min(d_min, J)) & (depth <= J)).all()
    for j in range(J):
        acc = np.uint64(0)
        for t in range(T):
            acc |= tok[t, j]
        assert lay[j] == acc
        if keep.all():
            assert lay[j] == lay_o[j]
    if T >= 8:
        assert len(set(depth.tolist())) > 1  # the threshold splits the tokens


def test_prefetch_depth_extremes():
    """tau above 1: nothing passes, every token gets d_min; tau 0: every layer
    passes, every token gets J and its full top-k set in every layer."""
    cfg = CONFIGS["dsv2lite"]
    J = 3
    Ws, biases = make_lookahead_routers(cfg, J)
    x = make_tokens(cfg, T=8, batch=9)
    conf, depth, tok, lay, _ = _run(cfg, x, Ws, biases, 1.5, 2)
    assert (depth == 2).all() and (tok[:, 2] == 0).all() and lay[2] == 0
    conf, depth, tok, lay, _ = _run(cfg, x, Ws, biases, 0.0, 0)
    assert (depth == J).all()
    for t in range(8):
        for j in range(J):
            assert bin(int(tok[t, j])).count("1") == cfg.k
