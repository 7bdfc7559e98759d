"""Pins of the oracle's decisive margins (the near-tie exclusion rule).

A token is left out of the bit-exact comparison when one of the decisions it
goes through is closer than 1e-5 to flipping.  The margins that measure this
come from the oracle, so they are pinned here to things other than the
oracle:
  - exact ties built by hand in a probe layer whose router logits, prefetch
    logits and ordinal score are the token's own coordinates (the router
    weights are an identity block), so every tie is exact in float32 and the
    margin must come out as exactly 0, or as a chosen power of two;
  - seeded layers of the five shapes, where every margin is recomputed in
    numpy from x and the weights (float64 matmul, stable library sorts) and
    must agree with the oracle's.

Margins (the decisions they guard):
  top-k     router logit gap between the k-th and (k+1)-th largest
            (APEX §1, the routed set);
  prefetch  prefetch-router logit gap at position k + delta_hat (APEX §4.2,
            the prefetch set);
  theta     |theta_delta - s - logit(tau)| at delta_hat and delta_hat - 1, the
            two tests of the ordinal CDF that fix delta_hat (APEX §4.2);
  delta*    prefetch logit gaps on both sides of the lowest-ranked routed
            expert (APEX §4.2, the oracle budget delta*);
  substitute logit gap among the replacement candidates at the number of
            replacements (APEX §4.3, stall-free selection);
  gamma     |alpha_e - gamma| over the misses that HYBRID classifies (SPICE
            write-up, LoRE section: low-confidence misses go to LoRE).
CPU only.
"""
import math

import numpy as np
import pytest

import oracle
from workloads import CONFIGS, LayerWeights, make_tokens, make_weights

M_TOPK, M_PREFETCH, M_THETA, M_DSTAR, M_SUBST, M_GAMMA = range(6)
POL_EXACT, POL_SUBSTITUTE, POL_LORE, POL_HYBRID = range(4)


# ---- probe layer: logits = the token's coordinates ---------------------------

def _probe(N=8, k=2, theta=None, policy=POL_HYBRID, gamma=0.5, use_prefetch=True):
    d = N + 1
    cfg = CONFIGS["tiny"].with_(d=d, N=N, k=k, I=4, n_shared=1, I_shared=4, r=2, policy=policy,
                                gamma=gamma, n_resident=0, use_prefetch_mask=use_prefetch)
    eye = np.zeros((N, d), np.float32)
    eye[:, :N] = np.eye(N, dtype=np.float32)
    w_ord = np.zeros(d, np.float32)
    w_ord[N] = 1.0
    if theta is None:
        theta = np.linspace(-3, 3, N - k + 1)
    z = lambda *s: np.zeros(s, np.float32)
    W = LayerWeights(w_router=eye, w_prefetch=eye.copy(), w_ord=w_ord,
                     theta=np.asarray(theta, np.float32), router_bias=None,
                     w_gate=z(N, 4, d), w_up=z(N, 4, d), w_down=z(N, 4, d),
                     sh_gate=z(1, 4, d), sh_up=z(1, 4, d), sh_down=z(1, 4, d),
                     lore_a=z(N, 2, d), lore_b=z(N, d, 2))
    return cfg, W


def _run_probe(cfg, W, l, lp, s, tau=0.5, resident=None, gamma=None):
    """One token with router logits l, prefetch logits lp, ordinal score s."""
    x = np.zeros((1, cfg.d), np.float32)
    x[0, :cfg.N] = l
    xp = np.zeros((1, cfg.d), np.float32)
    xp[0, :cfg.N] = lp
    xp[0, cfg.N] = s
    res = (1 << 64) - 1 if resident is None else resident
    return oracle.layer_forward(cfg, W, x, x_pre=xp, resident=res, tau=tau, gamma=gamma,
                                route_only=True)


def _mask(ids):
    m = 0
    for e in ids:
        m |= 1 << e
    return m


def test_probe_layer_reproduces_its_coordinates():
    cfg, W = _probe()
    l = [0.5, 2.0, -1.0, 0.25, 3.0, -2.0, 1.0, 0.0]
    lp = [1.0, 0.0, 2.0, -1.0, 0.5, 3.0, -0.5, 0.25]
    R = _run_probe(cfg, W, l, lp, s=0.75)
    np.testing.assert_array_equal(R.logits[0], l)
    np.testing.assert_array_equal(R.logits_p[0], lp)
    assert R.score[0] == 0.75


def test_topk_tie_at_the_boundary_gives_zero_margin():
    cfg, W = _probe()
    lp = [3.0, 2.0, 1.0, 0.0, -1.0, -2.0, -3.0, -4.0]
    R = _run_probe(cfg, W, [3.0, 2.0, 2.0, 1.0, 0.0, 0.0, -1.0, -2.0], lp, 0.0)
    assert R.margin[0, M_TOPK] == 0.0
    assert R.excluded()[0]
    assert sorted(R.topk_idx[0]) == [0, 1]         # the tie goes to the lower index
    # a tie inside the top-k decides nothing: the margin is the boundary gap
    R = _run_probe(cfg, W, [3.0, 3.0, 2.0, 1.0, 0.0, 0.0, -1.0, -2.0], lp, 0.0)
    assert R.margin[0, M_TOPK] == 1.0
    # a gap of 2^-20 (below 1e-5) is reported as such
    R = _run_probe(cfg, W, [3.0, 2.0, 2.0 - 2.0 ** -20, 1.0, 0.0, 0.0, -1.0, -2.0], lp, 0.0)
    assert R.margin[0, M_TOPK] == 2.0 ** -20
    assert R.excluded()[0]


def test_prefetch_tie_at_k_plus_delta_hat_gives_zero_margin():
    # tau = 0.5: delta_hat = first delta with theta_delta - s >= 0 -> 3
    theta = [-3.0, -2.0, -1.0, 0.5, 1.0, 2.0, 3.0]
    cfg, W = _probe(theta=theta)
    l = [3.0, 2.0, 1.0, 0.0, -1.0, -2.0, -3.0, -4.0]
    # prefetch set = top-5 of lp; positions 4 and 5 (0-based) tie at 1.0
    lp = [6.0, 5.0, 4.0, 3.0, 1.0, 1.0, 0.0, -1.0]
    R = _run_probe(cfg, W, l, lp, s=0.0)
    assert R.delta_hat[0] == 3
    assert R.margin[0, M_PREFETCH] == 0.0
    assert R.excluded()[0]
    assert int(R.prefetch[0]) == _mask([0, 1, 2, 3, 4])
    lp[5] = 0.5
    R = _run_probe(cfg, W, l, lp, s=0.0)
    assert R.margin[0, M_PREFETCH] == 0.5


def test_theta_boundary_at_delta_hat_and_below():
    l = [3.0, 2.0, 1.0, 0.0, -1.0, -2.0, -3.0, -4.0]
    lp = [7.0, 6.0, 5.0, 4.0, 3.0, 2.0, 1.0, 0.0]
    # theta_3 - s = 0 exactly: sigmoid = 0.5 >= tau, delta_hat = 3, margin 0
    cfg, W = _probe(theta=[-3.0, -2.0, -1.0, 0.5, 1.0, 2.0, 3.0])
    R = _run_probe(cfg, W, l, lp, s=0.5)
    assert R.delta_hat[0] == 3
    assert R.margin[0, M_THETA] == 0.0
    assert R.excluded()[0]
    # theta_2 falls 2^-20 short of the threshold: delta_hat stays 3, the
    # margin is set by delta_hat - 1
    cfg, W = _probe(theta=[-3.0, -2.0, 0.5 - 2.0 ** -20, 1.5, 2.0, 2.5, 3.0])
    R = _run_probe(cfg, W, l, lp, s=0.5)
    assert R.delta_hat[0] == 3
    assert R.margin[0, M_THETA] == 2.0 ** -20
    # clear of both: min(|1.5 - 0.5|, |-1 - 0.5|) = 1
    cfg, W = _probe(theta=[-3.0, -2.0, -1.0, 1.5, 2.0, 2.5, 3.0])
    R = _run_probe(cfg, W, l, lp, s=0.5)
    assert R.delta_hat[0] == 3
    assert R.margin[0, M_THETA] == 1.0
    # tau = 0.9 is measured in logit units: theta_delta - s - ln 9
    cfg, W = _probe(theta=[-3.0, -2.0, -1.0, 3.0, 4.0, 5.0, 6.0])
    R = _run_probe(cfg, W, l, lp, s=0.5, tau=0.9)
    assert R.delta_hat[0] == 3
    assert R.margin[0, M_THETA] == pytest.approx(min(abs(3.0 - 0.5 - math.log(9)), abs(-1.0 - 0.5 - math.log(9))),
                                                 abs=1e-15)


def test_delta_star_tie_next_to_the_lowest_routed_expert():
    cfg, W = _probe()
    l = [3.0, 2.0, 1.0, 0.0, -1.0, -2.0, -3.0, -4.0]          # routed {0, 1}
    # prefetch order 0 (5), 2 (4), 3 (3), 1 (1), 4 (1): expert 1 ranks 3rd
    # (0-based) and ties with expert 4 below it
    lp = [5.0, 1.0, 4.0, 3.0, 1.0, 0.0, -1.0, -2.0]
    R = _run_probe(cfg, W, l, lp, s=0.0)
    assert R.delta_star[0] == 2
    assert R.margin[0, M_DSTAR] == 0.0
    lp[4] = 0.5                                               # gaps now 2 above, 0.5 below
    R = _run_probe(cfg, W, l, lp, s=0.0)
    assert R.margin[0, M_DSTAR] == 0.5
    lp = [5.0, 4.0, 3.0, 2.0, 1.0, 0.0, -1.0, -2.0]           # routed are the top 2: delta* = 0
    R = _run_probe(cfg, W, l, lp, s=0.0)
    assert R.delta_star[0] == 0
    assert R.margin[0, M_DSTAR] == 1.0


def test_substitution_tie_among_candidates_gives_zero_margin():
    cfg, W = _probe(policy=POL_SUBSTITUTE, use_prefetch=False)
    lp = [3.0, 2.0, 1.0, 0.0, -1.0, -2.0, -3.0, -4.0]
    # routed {0, 1}; resident {0, 3, 4, 5}: expert 1 missing, candidates
    # 3, 4 (logit 1.0 each) and 5 (0.0), one replacement
    l = [3.0, 2.5, 2.0, 1.0, 1.0, 0.0, -1.0, -2.0]
    R = _run_probe(cfg, W, l, lp, s=0.0, resident=_mask([0, 3, 4, 5]))
    assert R.margin[0, M_SUBST] == 0.0
    assert R.excluded()[0]
    assert sorted(R.final_idx[0]) == [0, 3]
    l[4] = 0.75
    R = _run_probe(cfg, W, l, lp, s=0.0, resident=_mask([0, 3, 4, 5]))
    assert R.margin[0, M_SUBST] == 0.25
    # two replacements: the gap is between the 2nd and 3rd candidate
    R = _run_probe(cfg, W, l, lp, s=0.0, resident=_mask([3, 4, 5, 6]))
    assert sorted(R.final_idx[0]) == [3, 4]
    assert R.margin[0, M_SUBST] == 0.75
    # no miss: the margin does not apply
    R = _run_probe(cfg, W, l, lp, s=0.0, resident=_mask([0, 1, 5]))
    assert R.margin[0, M_SUBST] == math.inf and R.margin[0, M_GAMMA] == math.inf


def test_gamma_equal_to_a_missing_experts_probability():
    cfg, W = _probe(policy=POL_HYBRID, use_prefetch=False)
    lp = [3.0, 2.0, 1.0, 0.0, -1.0, -2.0, -3.0, -4.0]
    l = [3.0, 2.5, 2.0, 1.0, 0.5, 0.0, -1.0, -2.0]
    res = _mask([0, 3, 4, 5])                                   # expert 1 misses
    R0 = _run_probe(cfg, W, l, lp, s=0.0, resident=res)
    a1 = float(R0.prob[0, 1])
    R = _run_probe(cfg, W, l, lp, s=0.0, resident=res, gamma=a1)
    assert R.margin[0, M_GAMMA] == 0.0
    assert R.excluded()[0]
    assert sorted(R.final_idx[0]) == [0, 3]                     # alpha >= gamma: substituted
    g_up = float(np.nextafter(a1, 1.0))
    R = _run_probe(cfg, W, l, lp, s=0.0, resident=res, gamma=g_up)
    assert R.margin[0, M_GAMMA] == g_up - a1
    assert sorted(R.final_idx[0]) == [0, 1] and R.final_kind[0][list(R.final_idx[0]).index(1)] == 2
    R = _run_probe(cfg, W, l, lp, s=0.0, resident=res, gamma=a1 + 0.125)
    assert R.margin[0, M_GAMMA] == pytest.approx(0.125, abs=1e-16)


# ---- seeded layers: every margin recomputed in numpy --------------------------

def _desc_order(v):
    """Indices by descending value, equal values by ascending index."""
    return np.lexsort((np.arange(v.shape[0]), -v))


def _expected_margins(cfg, W, x, R, resident, use_prefetch, policy, gamma, tau):
    x64 = x.astype(np.float64)
    L = x64 @ W.w_router.astype(np.float64).T
    if W.router_bias is not None:
        L += W.router_bias.astype(np.float64)
    LP = x64 @ W.w_prefetch.astype(np.float64).T
    S = x64 @ W.w_ord.astype(np.float64)
    th = W.theta.astype(np.float64)
    lt = math.log(tau / (1.0 - tau))
    N, k = cfg.N, cfg.k
    out = np.full((x.shape[0], 6), np.inf)
    for t in range(x.shape[0]):
        l, lp, s = L[t], LP[t], S[t]
        o = _desc_order(l)
        routed = o[:k]
        if k < N:
            out[t, M_TOPK] = l[o[k - 1]] - l[o[k]]
        # delta_hat by the count form (theta sorted): #{delta : theta - s < logit tau}
        dh = min(int((th - s < lt).sum()), cfg.delta_max)
        assert dh == R.delta_hat[t]
        out[t, M_THETA] = min(abs(th[dd] - s - lt) for dd in (dh - 1, dh) if dd >= 0)
        op = _desc_order(lp)
        if k + dh < N:
            out[t, M_PREFETCH] = lp[op[k + dh - 1]] - lp[op[k + dh]]
        rank = np.empty(N, np.int64)
        rank[op] = np.arange(N)
        w = int(rank[routed].max())
        gaps = []
        if w > 0:
            gaps.append(lp[op[w - 1]] - lp[op[w]])
        if w + 1 < N:
            gaps.append(lp[op[w]] - lp[op[w + 1]])
        out[t, M_DSTAR] = min(gaps)
        pset = set(op[:k + dh].tolist())
        avail = {e for e in range(N) if (resident >> e) & 1}
        if use_prefetch:
            avail &= pset
        missing = [e for e in routed if e not in avail]
        alpha = np.exp(l - l.max())
        alpha /= alpha.sum()
        if policy == POL_HYBRID and missing:
            out[t, M_GAMMA] = min(abs(alpha[e] - gamma) for e in missing)
        n_sub = len(missing) if policy == POL_SUBSTITUTE else (
            sum(1 for e in missing if alpha[e] >= gamma) if policy == POL_HYBRID else 0)
        if n_sub:
            cand = np.sort(np.array([l[e] for e in avail if e not in set(routed.tolist())]))[::-1]
            if cand.shape[0] > n_sub:
                out[t, M_SUBST] = cand[n_sub - 1] - cand[n_sub]
    return out


@pytest.mark.parametrize("name,T,kw", [
    ("tiny", 64, {}),                                             # HYBRID over the prefetch set
    ("tiny", 64, {"policy": POL_SUBSTITUTE}),
    ("granite", 128, {}),                                         # SUBSTITUTE over the prefetch set
    ("granite", 128, {"tau": 0.6}),
    ("granite", 128, {"tau": 0.97}),
    ("dsv2lite", 48, {}),                                         # HYBRID over a resident set of 24
    ("dsv2lite", 48, {"policy": POL_SUBSTITUTE}),
    ("dsv2lite_zipf", 48, {}),                                    # router bias (the Zipf skew)
])
def test_margins_match_numpy_recomputation(name, T, kw):
    base = "dsv2lite" if name.startswith("dsv2lite") else name
    cfg = CONFIGS[base]
    if name == "dsv2lite_zipf":
        cfg = cfg.with_(zipf=1.1)
    W = make_weights(cfg, experts=[])
    x = make_tokens(cfg, T=T, batch=3)
    policy = kw.get("policy", cfg.policy)
    tau = kw.get("tau", cfg.tau)
    R = oracle.layer_forward(cfg, W, x, route_only=True, policy=policy, tau=tau)
    want = _expected_margins(cfg, W, x, R, R.resident, cfg.use_prefetch_mask, policy, cfg.gamma, tau)
    got = R.margin[:, :6]
    np.testing.assert_allclose(got, want, rtol=1e-9, atol=1e-12)
    # the margins are live: each applicable one is finite on some token
    live = [M_TOPK, M_THETA, M_DSTAR]
    if policy in (POL_SUBSTITUTE, POL_HYBRID):
        live.append(M_SUBST)
    if policy == POL_HYBRID:
        live.append(M_GAMMA)
    if cfg.delta_max > 0:
        live.append(M_PREFETCH)
    for m in live:
        assert np.isfinite(got[:, m]).any(), f"margin {m} never applies"


def test_excluded_is_any_margin_below_the_bound():
    cfg = CONFIGS["granite"]
    W = make_weights(cfg, experts=[])
    x = make_tokens(cfg, T=256, batch=5)
    R = oracle.layer_forward(cfg, W, x, route_only=True)
    want = (R.margin[:, :7] < 1e-5).any(axis=1)
    np.testing.assert_array_equal(R.excluded(), want)
    # with a larger bound more tokens drop out, never fewer
    assert R.excluded(1e-2).sum() >= R.excluded().sum()
    assert R.excluded(1e-2).sum() > 0
