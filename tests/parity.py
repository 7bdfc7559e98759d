"""Comparison of the CUDA path's outputs with the float64 oracle.

Bars (the agreement rule of the layer):
  - expert indices, delta_hat, prefetch sets, delta*, final experts and slot
    kinds: bit-exact, on every token whose decisive margins in the oracle are
    all >= 1e-5 (near-ties are excluded and counted);
  - the excluded tokens are at most 1 % of the batch (none below 100 tokens)
    unless a test states a larger budget, and at least one token is kept, so
    no comparison can pass on an empty or nearly empty kept set;
  - layer outputs: relative L2 error over the kept tokens <= 1e-2 for bf16
    weights (fp32 accumulation) and <= 1e-5 for the fp32 layer, and on every
    kept token on its own <= 3e-2 (bf16) / 1e-4 (fp32), so that one wrong row
    in a large batch cannot hide inside the batch norm.
Where several answers are correct (the order of slots whose logits differ by
less than the margin), sets are compared and the GPU order is checked for
validity (non-increasing router probability).
"""
from __future__ import annotations

import numpy as np
import torch

from expert_routing_ffn_gb300.layer import as_u64

EPS_MARGIN = 1e-5


def tol_for(cfg) -> float:
    return 1e-5 if cfg.wtype == "f32" else 1e-2


def token_tol_for(cfg) -> float:
    return 1e-4 if cfg.wtype == "f32" else 3e-2


def exclusion_budget(T: int) -> int:
    """Near-tie tokens a comparison of T tokens may leave out."""
    return int(0.01 * T)


def _check_excluded(excl, budget=None):
    T = int(excl.shape[0])
    n = int(excl.sum())
    lim = exclusion_budget(T) if budget is None else budget
    assert n <= lim, f"{n} of {T} tokens excluded as near-ties (budget {lim})"
    assert T == 0 or n < T, "every token excluded: nothing compared"
    return n


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))


def to_np(t):
    return None if t is None else t.detach().cpu().numpy()


def check_routing(cfg, R, bufs, tokens=None, check_prefetch=True, budget=None):
    """Bit-exact routing comparison.  tokens: GPU row index of each oracle row.
    Returns the number of excluded (near-tie) tokens."""
    T = R.topk_idx.shape[0]
    rows = np.arange(T) if tokens is None else np.asarray(tokens)
    excl = R.excluded(EPS_MARGIN)
    n_excl = _check_excluded(excl, budget)
    keep = ~excl
    g_topk = to_np(bufs.topk_idx)[rows]
    g_prob = to_np(bufs.router_prob)[rows]
    g_dh = to_np(bufs.delta_hat)[rows]
    g_pm = to_np(bufs.prefetch_mask)[rows]
    g_ds = to_np(bufs.delta_star)[rows]
    np.testing.assert_allclose(g_prob, R.prob, rtol=0, atol=2e-6, err_msg="router_prob")
    for t in np.nonzero(keep)[0]:
        assert sorted(g_topk[t]) == sorted(R.topk_idx[t]), f"top-k differs at token {t}"
        p = g_prob[t][g_topk[t]]
        assert (np.diff(p) <= 0).all(), f"top-k order not descending at token {t}"
        if check_prefetch:
            assert g_dh[t] == R.delta_hat[t], f"delta_hat differs at token {t}"
            assert as_u64(g_pm[t]) == int(R.prefetch[t]), f"prefetch set differs at token {t}"
            assert g_ds[t] == R.delta_star[t], f"delta* differs at token {t}"
    return n_excl


def check_selection(cfg, R, bufs, tokens=None, budget=None, floe=True):
    """Final experts, kinds and gates per kept token; returns the excluded count."""
    T = R.final_idx.shape[0]
    rows = np.arange(T) if tokens is None else np.asarray(tokens)
    excl = R.excluded(EPS_MARGIN, floe=floe)
    n_excl = _check_excluded(excl, budget)
    keep = ~excl
    gi = to_np(bufs.final_idx)[rows]
    gk = to_np(bufs.final_kind)[rows]
    gg = to_np(bufs.final_gate)[rows]
    for t in np.nonzero(keep)[0]:
        o_map = {int(e): (int(kd), g) for e, kd, g in zip(R.final_idx[t], R.final_kind[t], R.final_gate[t]) if e >= 0}
        g_map = {int(e): (int(kd), g) for e, kd, g in zip(gi[t], gk[t], gg[t]) if e >= 0}
        assert set(o_map) == set(g_map), f"final experts differ at token {t}: {o_map} vs {g_map}"
        for e in o_map:
            assert o_map[e][0] == g_map[e][0], f"slot kind of expert {e} differs at token {t}"
            assert abs(o_map[e][1] - g_map[e][1]) <= 2e-6 + 1e-5 * abs(o_map[e][1]), "gate"
        gp = [g for e, g in zip(gi[t], gg[t]) if e >= 0]
        assert all(gp[i] >= gp[i + 1] for i in range(len(gp) - 1)), "final slots not in gate order"
    return n_excl


def check_output(cfg, R, out_gpu, tokens=None, budget=None, floe=True):
    """Relative L2 over the kept tokens (the batch bar) and per kept token.
    floe=False keeps tokens whose only near-tie is a FloE channel at the
    keep boundary: either side of such a channel is a correct kept set, and
    the output moves by one channel's share.  Returns the batch error."""
    T = R.out.shape[0]
    rows = np.arange(T) if tokens is None else np.asarray(tokens)
    excl = R.excluded(EPS_MARGIN, floe=floe)
    _check_excluded(excl, budget)
    keep = ~excl
    g = to_np(out_gpu)[rows].astype(np.float64)
    err = rel_l2(g[keep], R.out[keep])
    assert err <= tol_for(cfg), f"relative L2 {err:.3e} > {tol_for(cfg)}"
    num = np.linalg.norm(g[keep] - R.out[keep], axis=1)
    den = np.linalg.norm(R.out[keep], axis=1)
    per = num / np.where(den > 0, den, 1.0)
    if per.size:
        worst = int(np.argmax(per))
        assert per[worst] <= token_tol_for(cfg), (
            f"token {int(rows[keep][worst])}: relative L2 {per[worst]:.3e} > {token_tol_for(cfg)}")
    return err


def x_device(x_np, dt):
    return torch.from_numpy(x_np).cuda().to(dt).contiguous()
