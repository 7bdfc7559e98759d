"""Pins of the float64 oracle to things other than itself.

Each test checks an oracle step against a hand-worked case (tests/golden/),
a closed form, an invariant of the method, a reduction to a library routine,
or brute force on tiny inputs.  They are chosen so that a plausible slip
(a wrong tie rule, '>' for '>=', ranking substitutes by the prefetch router,
a dropped shared term, a transposed LoRE factor, a wrong SiLU) fails at least
one of them.  CPU only.
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch

import oracle
from workloads import CONFIGS, make_tokens, make_weights

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _cases(name):
    rows = []
    with open(os.path.join(GOLD, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append([fld.strip() for fld in line.split(";")])
    return rows


def _nums(s, typ=float):
    return [typ(v) for v in s.split(",")] if s else []


def _mask(ids):
    m = 0
    for e in ids:
        m |= 1 << int(e)
    return m


def _ids(mask, N):
    return [e for e in range(N) if (mask >> e) & 1]


# ---- hand-worked cases ----------------------------------------------------

@pytest.mark.parametrize("row", _cases("delta_hat_cases.txt"))
def test_delta_hat_golden(row):
    theta = np.array(_nums(row[0]), np.float32)
    s, tau, want = float(row[1]), float(row[2]), int(row[3])
    dh, s_out = oracle.delta_hat(np.array([s], np.float32), np.array([1.0], np.float32), theta, tau)
    assert s_out == s
    assert dh == want


@pytest.mark.parametrize("row", _cases("delta_star_cases.txt"))
def test_delta_star_golden(row):
    lp = np.array(_nums(row[0]))
    routed = np.array(_nums(row[1], int), np.int32)
    assert oracle.delta_star(routed, lp) == int(row[2])


@pytest.mark.parametrize("row", _cases("stall_free_cases.txt"))
def test_stall_free_golden(row):
    routed, alpha, pref, want = _nums(row[0], int), _nums(row[1]), _nums(row[2], int), _nums(row[3], int)
    got = oracle.stall_free_select(6, _mask(routed), np.array(alpha), _mask(pref))
    assert _ids(got, 6) == sorted(want)


@pytest.mark.parametrize("row", _cases("topk_cases.txt"))
def test_topk_golden(row):
    v, k, want = np.array(_nums(row[0])), int(row[1]), _nums(row[2], int)
    assert list(oracle.topk(v, k)) == want


@pytest.mark.parametrize("row", _cases("ffn_cases.txt"))
def test_ffn_golden(row):
    x, wg, wu, wd, want = (float(v) for v in row)
    y = oracle.expert_ffn(np.array([x]), np.array([[wg]]), np.array([[wu]]), np.array([[wd]]))
    assert y[0] == pytest.approx(want, rel=1e-12)


@pytest.mark.parametrize("row", _cases("lore_cases.txt"))
def test_lore_golden(row):
    r = int(row[3])
    x = np.array(_nums(row[2]))
    d = x.size
    A = np.array(_nums(row[0])).reshape(r, d)
    B = np.array(_nums(row[1])).reshape(d, r)
    assert list(oracle.lore(x, A, B)) == _nums(row[4])


# ---- router steps ---------------------------------------------------------

def test_logits_match_matmul():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((5, 33)).astype(np.float32)
    W = rng.standard_normal((7, 33)).astype(np.float32)
    b = rng.standard_normal(7).astype(np.float32)
    want = x.astype(np.float64) @ W.astype(np.float64).T + b
    np.testing.assert_allclose(oracle.logits(x, W, b), want, rtol=1e-13, atol=1e-13)


def test_softmax_matches_library():
    from scipy.special import softmax
    rng = np.random.default_rng(2)
    l = rng.standard_normal(40) * 3
    np.testing.assert_allclose(oracle.softmax(l), softmax(l), rtol=1e-13)


@pytest.mark.parametrize("N,k", [(5, 2), (6, 3), (8, 2), (10, 4)])
def test_topk_brute_force(N, k):
    """The defining property over every k-subset, on values with many ties."""
    rng = np.random.default_rng(N * 10 + k)
    for _ in range(40):
        v = rng.integers(0, 4, N).astype(np.float64)
        got = list(oracle.topk(v, k))
        best = None
        for S in itertools.combinations(range(N), k):
            rest = [j for j in range(N) if j not in S]
            ok = all(v[i] > v[j] or (v[i] == v[j] and i < j) for i in S for j in rest)
            if ok:
                assert best is None, "defining property picks a unique set"
                best = set(S)
        assert set(got) == best
        # order: descending value, lower index first (a stable library sort)
        assert got == list(np.lexsort((np.arange(N), -v)))[:k]


def test_delta_hat_count_form_and_monotone():
    """Sorted thresholds make delta_hat = #{delta : theta_delta - s < logit(tau)}
    (clipped to delta_max), non-decreasing in tau, 0 as tau -> 0 and delta_max
    as tau -> 1."""
    cfg = CONFIGS["granite"]
    W = make_weights(cfg, experts=[])
    x = make_tokens(cfg, T=64)
    dm = cfg.delta_max
    for t in range(x.shape[0]):
        prev = -1
        for tau in (1e-9, 0.3, 0.6, 0.9, 0.97, 0.999, 1 - 1e-12):
            dh, s = oracle.delta_hat(W.w_ord, x[t], W.theta, tau)
            count = int(np.sum(W.theta.astype(np.float64) - s < math.log(tau / (1 - tau))))
            assert dh == min(count, dm)
            assert dh >= prev
            prev = dh
        assert oracle.delta_hat(W.w_ord, x[t], W.theta, 1e-9)[0] == 0
        assert oracle.delta_hat(W.w_ord, x[t], W.theta, 1 - 1e-12)[0] == dm


def test_delta_star_closed_form_and_zero_when_routers_agree():
    rng = np.random.default_rng(3)
    for N, k in [(8, 2), (16, 4), (64, 6)]:
        for _ in range(50):
            lp = rng.integers(0, 6, N).astype(np.float64) if N <= 8 else rng.standard_normal(N)
            l = rng.standard_normal(N)
            routed = oracle.topk(l, k)
            order = list(np.lexsort((np.arange(N), -lp)))
            rank = {e: order.index(e) for e in range(N)}
            closed = max(0, max(rank[int(e)] for e in routed) + 1 - k)
            assert oracle.delta_star(routed, lp) == closed
            # prefetch router equal to the router: delta* = 0
            assert oracle.delta_star(routed, l) == 0


def test_prefetch_set_is_top_k_plus_delta():
    rng = np.random.default_rng(4)
    for _ in range(50):
        lp = rng.integers(0, 5, 12).astype(np.float64)
        for dh in range(0, 7):
            m = oracle.prefetch_set(3, dh, lp)
            assert bin(m).count("1") == 3 + dh
            assert _ids(m, 12) == sorted(np.lexsort((np.arange(12), -lp))[:3 + dh])


# ---- stall-free substitution ------------------------------------------------

def _closed_form(N, k, alpha, avail):
    """Top-k of alpha restricted to the available set (equal alpha: lower index)."""
    cand = [e for e in range(N) if (avail >> e) & 1]
    cand.sort(key=lambda e: (-alpha[e], e))
    return set(cand[:k])


def _best_total_alpha(N, routed, alpha, avail):
    """Brute force over every way of filling the missing slots: among the
    supersets of (routed & available) inside the available set with as many
    members as routed, the largest total alpha; equal totals: the
    lexicographically smallest sorted index list."""
    keep = [e for e in range(N) if (routed >> e) & 1 and (avail >> e) & 1]
    pool = [e for e in range(N) if (avail >> e) & 1 and not (routed >> e) & 1]
    m = bin(routed).count("1") - len(keep)
    best = None
    for sub in itertools.combinations(pool, m):
        key = (-sum(alpha[e] for e in sub), sorted(keep + list(sub)))
        if best is None or key < best:
            best = key
    return set(best[1])


@pytest.mark.parametrize("N,k", [(6, 2), (6, 3)])
def test_stall_free_exhaustive(N, k):
    """Every ordering of alpha x every available set with |A| >= k: the
    selection equals the filling of the missing slots with the largest total
    alpha (brute force), equals the top-k of alpha over A, has k members, lies
    inside A and keeps every routed expert that was available."""
    for perm in itertools.permutations(range(N)):
        alpha = np.array(perm, np.float64) + 1.0
        alpha /= alpha.sum()
        routed = set(np.argsort(-alpha, kind="stable")[:k].tolist())
        rmask = _mask(routed)
        for avail in range(1 << N):
            if bin(avail).count("1") < k:
                continue
            got = oracle.stall_free_select(N, rmask, alpha, avail)
            gs = set(_ids(got, N))
            assert gs == _closed_form(N, k, alpha, avail)
            if avail & ~rmask and perm[0] % 2 == 0:
                assert gs == _best_total_alpha(N, rmask, alpha, avail)
            assert len(gs) == k and got & ~avail == 0
            assert (rmask & avail) & ~got == 0


def test_stall_free_brute_force_with_ties_and_short_pool():
    """Integer-valued alpha (many ties) on N = 7: brute force over every
    filling; a pool smaller than the number of missing experts is refused."""
    rng = np.random.default_rng(17)
    N = 7
    for _ in range(60):
        alpha = rng.integers(1, 4, N).astype(np.float64)
        alpha /= alpha.sum()
        for k in (2, 3):
            order = sorted(range(N), key=lambda e: (-alpha[e], e))
            rmask = _mask(order[:k])
            for avail in range(1 << N):
                got = oracle.stall_free_select(N, rmask, alpha, avail)
                missing = bin(rmask & ~avail).count("1")
                if bin(avail & ~rmask).count("1") < missing:
                    assert got == (1 << 64) - 1
                    continue
                assert set(_ids(got, N)) == _best_total_alpha(N, rmask, alpha, avail)


def test_stall_free_sampled_n8_ignores_prefetch_scores():
    """N = 8, k = 2 on random orderings (with ties) and every available set."""
    rng = np.random.default_rng(5)
    N, k = 8, 2
    for _ in range(150):
        alpha = rng.integers(1, 5, N).astype(np.float64)
        alpha /= alpha.sum()
        order = sorted(range(N), key=lambda e: (-alpha[e], e))
        rmask = _mask(order[:k])
        for avail in range(1 << N):
            if bin(avail).count("1") < k:
                continue
            got = oracle.stall_free_select(N, rmask, alpha, avail)
            assert set(_ids(got, N)) == _closed_form(N, k, alpha, avail)


# ---- expert FFN, FloE, LoRE ------------------------------------------------

def _torch_ffn(x, Wg, Wu, Wd):
    x = torch.tensor(x, dtype=torch.float64)
    Wg, Wu, Wd = (torch.tensor(a, dtype=torch.float64) for a in (Wg, Wu, Wd))
    h = torch.nn.functional.silu(x @ Wg.T) * (x @ Wu.T)
    return (h @ Wd).numpy()


def test_expert_ffn_matches_torch():
    rng = np.random.default_rng(6)
    d, I = 48, 40
    x = rng.standard_normal(d).astype(np.float32)
    Wg, Wu, Wd = (rng.standard_normal((I, d)).astype(np.float32) * 0.1 for _ in range(3))
    np.testing.assert_allclose(oracle.expert_ffn(x, Wg, Wu, Wd), _torch_ffn(x, Wg, Wu, Wd),
                               rtol=1e-12, atol=1e-12)


def test_floe_keep_all_is_dense_and_mask_is_top_abs_u():
    rng = np.random.default_rng(7)
    d, I = 32, 64
    x = rng.standard_normal(d).astype(np.float32)
    Wg, Wu, Wd = (rng.standard_normal((I, d)).astype(np.float32) * 0.2 for _ in range(3))
    dense = oracle.expert_ffn(x, Wg, Wu, Wd)
    y, kept, _ = oracle.expert_ffn_floe(x, Wg, Wu, Wd, I)
    np.testing.assert_allclose(y, dense, rtol=1e-12, atol=1e-12)
    assert list(kept) == list(range(I))
    m = 7
    y, kept, gap = oracle.expert_ffn_floe(x, Wg, Wu, Wd, m)
    u = x.astype(np.float64) @ Wu.astype(np.float64).T
    want = sorted(np.lexsort((np.arange(I), -np.abs(u)))[:m])
    assert list(kept) == want
    # zeroing the up rows of dropped channels reproduces the sparse forward
    Wu_m = np.zeros_like(Wu)
    Wu_m[want] = Wu[want]
    np.testing.assert_allclose(y, _torch_ffn(x, Wg, Wu_m, Wd), rtol=1e-12, atol=1e-12)
    au = np.sort(np.abs(u))[::-1]
    assert gap == pytest.approx((au[m - 1] - au[m]) / au[0])


def test_lore_identity_reproduces_linear_map():
    """r = d with A = identity: B A x = B x."""
    rng = np.random.default_rng(8)
    d = 16
    x = rng.standard_normal(d).astype(np.float32)
    B = rng.standard_normal((d, d)).astype(np.float32)
    v = oracle.lore(x, np.eye(d, dtype=np.float32), B)
    np.testing.assert_allclose(v, B.astype(np.float64) @ x.astype(np.float64), rtol=1e-12)


# ---- whole layer ------------------------------------------------------------

def _small(name="tiny", **kw):
    cfg = CONFIGS[name].with_(**kw)
    return cfg, make_weights(cfg), make_tokens(cfg)


def _dense_moe(cfg, W, x, R):
    """Independent dense formula: sum over ALL experts of 1[e routed] g_e FFN_e(x)
    plus the shared experts, in torch float64."""
    T = x.shape[0]
    X = torch.tensor(x, dtype=torch.float64)
    out = torch.zeros((T, cfg.d), dtype=torch.float64)
    gates = torch.zeros((T, cfg.N), dtype=torch.float64)
    for t in range(T):
        for s in range(cfg.k):
            gates[t, R.topk_idx[t, s]] = R.prob[t, R.topk_idx[t, s]]
    for e in range(cfg.N):
        y = torch.tensor(_torch_ffn(x, W.w_gate[e], W.w_up[e], W.w_down[e]))
        out += gates[:, e:e + 1] * y
    for s in range(cfg.n_shared):
        out += torch.tensor(_torch_ffn(x, W.sh_gate[s], W.sh_up[s], W.sh_down[s]))
    return out.numpy()


def test_layer_router_matches_softmax_topk():
    cfg, W, x = _small()
    R = oracle.layer_forward(cfg, W, x)
    l = x.astype(np.float64) @ W.w_router.astype(np.float64).T
    np.testing.assert_allclose(R.logits, l, rtol=1e-12, atol=1e-12)
    from scipy.special import softmax
    np.testing.assert_allclose(R.prob, softmax(l, axis=1), rtol=1e-12)
    for t in range(x.shape[0]):
        assert list(R.topk_idx[t]) == list(np.lexsort((np.arange(cfg.N), -l[t]))[:cfg.k])


@pytest.mark.parametrize("policy", [0, 1, 2, 3])
def test_all_resident_is_plain_moe(policy):
    """With every expert available no miss occurs: all policies give the plain
    MoE layer (APEX §4.3: prefetching never changes what is computed)."""
    cfg, W, x = _small()
    R = oracle.layer_forward(cfg, W, x, resident=(1 << 64) - 1, use_prefetch=False, policy=policy)
    np.testing.assert_allclose(R.out, _dense_moe(cfg, W, x, R), rtol=1e-10, atol=1e-12)
    assert (R.final_kind == 0).all()


def test_exact_policy_is_plain_moe_with_fetches():
    """Correctness-preserving mode (APEX §4.3): missing experts are fetched and
    the output equals the plain MoE layer."""
    cfg, W, x = _small(policy=0)
    R = oracle.layer_forward(cfg, W, x)
    assert (R.final_kind == 1).sum() > 0
    np.testing.assert_allclose(R.out, _dense_moe(cfg, W, x, R), rtol=1e-10, atol=1e-12)
    assert (np.sort(R.final_idx, axis=1) == np.sort(R.topk_idx, axis=1)).all()


def test_lore_zero_factors_give_shared_output():
    """A = B = 0: each LoRE slot contributes exactly g * y_shared."""
    cfg, W, x = _small(policy=2)
    W.lore_a[:] = 0
    W.lore_b[:] = 0
    R = oracle.layer_forward(cfg, W, x)
    lore = R.final_kind == 2
    assert lore.sum() > 0
    want = np.zeros_like(R.out)
    for t in range(x.shape[0]):
        want[t] = R.y_shared[t] * (1.0 + R.final_gate[t][lore[t]].sum())
        for s in range(cfg.k):
            if not lore[t, s]:
                e = R.final_idx[t, s]
                want[t] += R.final_gate[t, s] * _torch_ffn(x[t], W.w_gate[e], W.w_up[e], W.w_down[e])
    np.testing.assert_allclose(R.out, want, rtol=1e-10, atol=1e-12)
    shared = sum(_torch_ffn(x, W.sh_gate[s], W.sh_up[s], W.sh_down[s]) for s in range(cfg.n_shared))
    np.testing.assert_allclose(R.y_shared, shared, rtol=1e-10, atol=1e-12)


def test_lore_slot_adds_low_rank_term():
    """LoRE slot output minus the A = B = 0 output is g * B_e A_e x."""
    cfg, W, x = _small(policy=2)
    R1 = oracle.layer_forward(cfg, W, x)
    A, B = W.lore_a.copy(), W.lore_b.copy()
    W.lore_a[:] = 0
    W.lore_b[:] = 0
    R0 = oracle.layer_forward(cfg, W, x)
    for t in range(x.shape[0]):
        want = np.zeros(cfg.d)
        for s in range(cfg.k):
            if R1.final_kind[t, s] == 2:
                e = R1.final_idx[t, s]
                want += R1.final_gate[t, s] * (B[e].astype(np.float64) @ (A[e].astype(np.float64) @ x[t]))
        np.testing.assert_allclose(R1.out[t] - R0.out[t], want, rtol=1e-9, atol=1e-12)


def test_substitute_policy_is_top_k_over_available():
    cfg, W, x = _small("granite", I=16, T=96)
    R = oracle.layer_forward(cfg, W, x)
    n_sub = 0
    for t in range(x.shape[0]):
        avail = int(R.prefetch[t])
        want = _closed_form(cfg.N, cfg.k, R.logits[t], avail)
        assert set(R.final_idx[t].tolist()) == want
        n_sub += len(want - set(R.topk_idx[t].tolist()))
        # gates: each final expert carries its own router probability
        np.testing.assert_allclose(R.final_gate[t], R.prob[t, R.final_idx[t]], rtol=0)
        # canonical slot order: descending logit
        assert list(R.final_idx[t]) == sorted(want, key=lambda e: (-R.logits[t, e], e))
    assert n_sub > 0


def test_hybrid_extremes():
    """gamma = 0 sends every miss to substitution, gamma = 1 sends every miss to LoRE."""
    cfg, W, x = _small(T=64)
    Rh0 = oracle.layer_forward(cfg, W, x, gamma=0.0)
    Rs = oracle.layer_forward(cfg, W, x, policy=1)
    np.testing.assert_array_equal(Rh0.final_idx, Rs.final_idx)
    np.testing.assert_allclose(Rh0.out, Rs.out, rtol=0, atol=0)
    Rh1 = oracle.layer_forward(cfg, W, x, gamma=1.0)
    Rl = oracle.layer_forward(cfg, W, x, policy=2)
    np.testing.assert_array_equal(Rh1.final_kind, Rl.final_kind)
    np.testing.assert_allclose(Rh1.out, Rl.out, rtol=0, atol=0)
    Rh = oracle.layer_forward(cfg, W, x)
    kinds = np.bincount(Rh.final_kind.ravel(), minlength=3)
    subs = sum(len(set(Rh.final_idx[t]) - set(Rh.topk_idx[t])) for t in range(64))
    assert kinds[2] > 0 and subs > 0, "both HYBRID branches occur at the config's gamma"


def test_floe_keep_all_equals_dense_layer():
    cfg, W, x = _small("mixtral", d=64, I=96, T=6)
    Rd = oracle.layer_forward(cfg, W, x)
    Rf = oracle.layer_forward(cfg, W, x, keep_m=cfg.I - 1)
    Rf_all = oracle.layer_forward(cfg, W, x, keep_m=cfg.I)
    np.testing.assert_allclose(Rf_all.out, Rd.out, rtol=0, atol=0)
    assert not np.allclose(Rf.out, Rd.out, rtol=1e-14, atol=0)


def test_token_permutation_invariance():
    cfg, W, x = _small(T=16)
    R = oracle.layer_forward(cfg, W, x)
    p = np.random.default_rng(9).permutation(x.shape[0])
    Rp = oracle.layer_forward(cfg, W, x[p])
    np.testing.assert_allclose(Rp.out, R.out[p], rtol=1e-13, atol=1e-15)
    np.testing.assert_array_equal(Rp.final_idx, R.final_idx[p])


def test_batch_resident_matches_summed_softmax():
    from scipy.special import softmax
    rng = np.random.default_rng(10)
    lp = rng.standard_normal((20, 16))
    m, gap = oracle.batch_resident(lp, 5)
    s = softmax(lp, axis=1).sum(0)
    order = np.lexsort((np.arange(16), -s))
    assert _ids(m, 16) == sorted(order[:5].tolist())
    assert gap == pytest.approx(s[order[4]] - s[order[5]])


def test_capacity_shortfall_flagged():
    cfg, W, x = _small(policy=1, use_prefetch_mask=False)
    R = oracle.layer_forward(cfg, W, x, resident=0b1)  # one expert available, k = 2
    assert (R.status == 1).all()


# ---- persistent expert cache (ELMoE-3D heat map with decay) ----------------

def test_cache_heat_closed_form_and_extremes():
    """The same routed slots every step: heat is the geometric series
    count * (1 - decay^S) / (1 - decay); decay 1 is plain counting, decay 0
    keeps this step's counts only."""
    rng = np.random.default_rng(7)
    N, C, S = 12, 4, 9
    routed = rng.integers(0, N, size=10)
    counts = np.bincount(routed, minlength=N).astype(np.float64)
    for decay in (0.0, 0.5, 0.99, 1.0):
        heat, cache = np.zeros(N), 0
        for _ in range(S):
            cache, heat, _, _ = oracle.cache_update(routed, heat, decay, C, cache)
        series = S if decay == 1.0 else (1.0 - decay ** S) / (1.0 - decay)
        np.testing.assert_allclose(heat, counts * series, rtol=1e-12, atol=0)


def test_cache_is_top_c_by_heat_with_low_index_ties():
    """Brute force over random histories: every cached expert has at least
    the heat of every other, equal heat goes to the lower index, the cache
    has exactly min(C, N) members and hits count routed slots in the old
    cache."""
    rng = np.random.default_rng(11)
    for trial in range(200):
        N = int(rng.integers(2, 16))
        C = int(rng.integers(1, N + 2))
        heat = rng.integers(0, 4, size=N).astype(np.float64)  # integers: many ties
        old = int(rng.integers(0, 1 << N))
        routed = rng.integers(-1, N, size=int(rng.integers(0, 12)))
        cache, new_heat, hits, gap = oracle.cache_update(routed, heat, 0.5, C, old)
        expect = 0.5 * heat + np.bincount(routed[routed >= 0], minlength=N)
        np.testing.assert_array_equal(new_heat, expect)
        members = [e for e in range(N) if (cache >> e) & 1]
        assert len(members) == min(C, N)
        for e in members:
            for o in range(N):
                if (cache >> o) & 1:
                    continue
                assert expect[e] > expect[o] or (expect[e] == expect[o] and e < o)
        assert hits == sum(1 for e in routed if e >= 0 and (old >> int(e)) & 1)
        if C < N:
            order = sorted(range(N), key=lambda e: (-expect[e], e))
            assert gap == expect[order[C - 1]] - expect[order[C]]


def test_cache_hand_worked_step():
    """Routed {0, 1, 1, 3} from zero heat, C = 2: heat (1, 2, 0, 1, 0); the
    tie between experts 0 and 3 goes to 0."""
    cache, heat, hits, gap = oracle.cache_update([0, 1, 1, 3], np.zeros(5), 0.9, 2, 0b01000)
    assert cache == 0b00011
    np.testing.assert_array_equal(heat, [1, 2, 0, 1, 0])
    assert hits == 1 and gap == 0.0


# ---- look-ahead prefetch depth (SPICE, confidence-aware adaptive prefetch) --

def test_lookahead_confidence_is_largest_k_subset_mass():
    """The confidence of a look-ahead layer is the probability mass on its
    top-K experts: brute force over every K-subset, the largest subset mass
    equals it; K = N gives the whole distribution (1)."""
    rng = np.random.default_rng(21)
    for trial in range(40):
        N = int(rng.integers(2, 9))
        K = int(rng.integers(1, N + 1))
        d, T, J = 16, 3, 2
        x = rng.standard_normal((T, d)).astype(np.float32)
        Ws = [rng.standard_normal((N, d)).astype(np.float32) * 0.3 for _ in range(J)]
        conf, _, tok, _, _ = oracle.prefetch_depth(x, Ws, None, K, 0.5, 0)
        for t in range(T):
            for j in range(J):
                lg = Ws[j].astype(np.float64) @ x[t].astype(np.float64)
                p = torch.softmax(torch.from_numpy(lg), 0).numpy()
                best = max(sum(p[list(c)]) for c in itertools.combinations(range(N), K))
                assert abs(conf[t, j] - best) < 1e-12
                if K == N:
                    assert abs(conf[t, j] - 1.0) < 1e-12


def test_lookahead_uniform_prediction_and_ties():
    """Zero router weights: every expert has probability 1/N, so the
    confidence is exactly K/N and the predicted set is the K lowest indices.
    A threshold at or below K/N keeps all J layers; above it only d_min."""
    N, K, d, T, J = 8, 2, 32, 4, 3
    x = np.random.default_rng(3).standard_normal((T, d)).astype(np.float32)
    Ws = [np.zeros((N, d), np.float32) for _ in range(J)]
    conf, depth, tok, lay, _ = oracle.prefetch_depth(x, Ws, None, K, 0.25, 0)
    np.testing.assert_array_equal(conf, np.full((T, J), 0.25))
    np.testing.assert_array_equal(depth, np.full(T, J))
    np.testing.assert_array_equal(tok, np.full((T, J), 0b11, np.uint64))
    for d_min, expect in ((0, 0), (2, 2), (5, J)):
        conf, depth, tok, lay, _ = oracle.prefetch_depth(x, Ws, None, K, 0.2500001, d_min)
        np.testing.assert_array_equal(depth, np.full(T, expect))
        for j in range(J):
            assert lay[j] == (0b11 if j < expect else 0)


def test_lookahead_hand_worked_stop_at_first_low_layer():
    """N = 4, K = 1, zero weights, the bias sets each look-ahead layer's top
    probability: 0.95, 0.92, 0.50, 0.99.  At tau = 0.9 the scan keeps layers
    0 and 1 and stops at layer 2, so layer 3 (0.99) is not reached: depth 2.
    d_min raises the depth (3), J caps it (4)."""
    N, d, J = 4, 8, 4
    tops = [0.95, 0.92, 0.50, 0.99]
    biases = []
    for p in tops:
        b = np.zeros(N, np.float32)
        b[1] = math.log(3 * p / (1 - p))  # p = a / (a + 3) for expert 1
        biases.append(b)
    x = np.ones((1, d), np.float32)
    Ws = [np.zeros((N, d), np.float32) for _ in range(J)]
    for d_min, expect in ((0, 2), (2, 2), (3, 3), (9, 4)):
        conf, depth, tok, lay, margin = oracle.prefetch_depth(x, Ws, biases, 1, 0.9, d_min)
        np.testing.assert_allclose(conf[0], tops, rtol=1e-6)
        assert depth[0] == expect
        np.testing.assert_array_equal(tok[0], [0b10 if j < expect else 0 for j in range(J)])
        np.testing.assert_array_equal(lay, tok[0])
        # the scan read layers 0..2: the nearest to tau is 0.92
        assert abs(margin[0] - 0.02) < 1e-6


def test_lookahead_depth_monotone_in_tau_and_masks_are_top_k():
    """A higher threshold never deepens the prefetch; a kept layer's token
    mask is the top-K of its logits; the layer mask is the OR over tokens."""
    rng = np.random.default_rng(5)
    N, K, d, T, J = 16, 4, 64, 12, 4
    x = rng.standard_normal((T, d)).astype(np.float32)
    Ws = [(rng.standard_normal((N, d)) * 0.25).astype(np.float32) for _ in range(J)]
    prev = None
    for tau in (0.0, 0.3, 0.5, 0.7, 0.9, 1.01):
        conf, depth, tok, lay, _ = oracle.prefetch_depth(x, Ws, None, K, tau, 1)
        if prev is not None:
            assert (depth <= prev).all()
        prev = depth
        for t in range(T):
            for j in range(J):
                if j < depth[t]:
                    lg = Ws[j].astype(np.float64) @ x[t].astype(np.float64)
                    top = sorted(range(N), key=lambda e: (-lg[e], e))[:K]
                    assert tok[t, j] == sum(1 << e for e in top)
                else:
                    assert tok[t, j] == 0
        for j in range(J):
            acc = 0
            for t in range(T):
                acc |= int(tok[t, j])
            assert int(lay[j]) == acc
    assert (prev == 1).all()  # tau above 1: nothing passes, d_min = 1 remains


# ---- bit-sliced expert weights (ELMoE-3D, bit slicing) ----------------------

def test_bitslice_top_planes_are_floor_truncation():
    """Every INT8 value and every precision: recombining the top b bit planes
    (plane 7 weighted -128) equals flooring the value to a multiple of
    2^(8-b) (an arithmetic right shift then a left shift); b = 8 gives the
    value itself."""
    for q in range(-128, 128):
        assert oracle.bitslice_value(q, 8) == q
        for b in range(1, 9):
            assert oracle.bitslice_value(q, b) == (q >> (8 - b)) << (8 - b), (q, b)


def test_bitslice_quantisation_bound_and_layout():
    """Per output row: the largest |q| is 127 on a nonzero row, every weight is
    within half a step of s*q, a zero row gives s = 0 and q = 0, and the
    transposed quantisation is the quantisation of W^T."""
    rng = np.random.default_rng(8)
    W = (rng.standard_normal((24, 96)) * 0.02).astype(np.float32)
    W[5] = 0.0
    q, s = oracle.bitslice_quantize(W)
    assert q.shape == (24, 96) and s.shape == (24,)
    for r in range(24):
        if r == 5:
            assert s[r] == 0.0 and (q[r] == 0).all()
            continue
        assert np.abs(q[r].astype(int)).max() == 127
        err = np.abs(W[r].astype(np.float64) - float(s[r]) * q[r].astype(np.float64))
        assert err.max() <= 0.5 * float(s[r]) * (1 + 1e-5)
    qt, st = oracle.bitslice_quantize(W, transpose=True)
    q2, s2 = oracle.bitslice_quantize(np.ascontiguousarray(W.T))
    np.testing.assert_array_equal(qt, q2)
    np.testing.assert_array_equal(st, s2)


def test_bitslice_ffn_full_precision_is_the_dense_expert():
    """With all 8 planes the bit-sliced expert is the dense SwiGLU expert on
    the dequantised weights s*q (the dense expert oracle is pinned against
    torch); fewer planes move the output further from it."""
    rng = np.random.default_rng(12)
    d, I = 64, 96
    x = rng.standard_normal(d).astype(np.float32)
    Wg, Wu, Wd = [(rng.standard_normal((I, d)) * 0.05).astype(np.float32) for _ in range(3)]
    qg, sg = oracle.bitslice_quantize(Wg)
    qu, su = oracle.bitslice_quantize(Wu)
    qdT, sd = oracle.bitslice_quantize(Wd, transpose=True)   # [d, I]
    y8 = oracle.bitslice_ffn(x, qg, sg, qu, su, qdT, sd, 8)
    deq = lambda q, s: (q.astype(np.float64) * s.astype(np.float64)[:, None])
    Wg8, Wu8 = deq(qg, sg), deq(qu, su)
    Wd8 = deq(qdT, sd).T                                      # back to [I, d]
    g, u = Wg8 @ x.astype(np.float64), Wu8 @ x.astype(np.float64)
    h = g / (1 + np.exp(-g)) * u
    np.testing.assert_allclose(y8, h @ Wd8, rtol=1e-12, atol=1e-14)
    dense = oracle.expert_ffn(x, Wg8.astype(np.float32), Wu8.astype(np.float32), Wd8.astype(np.float32))
    np.testing.assert_allclose(y8, dense, rtol=1e-5, atol=1e-7)
    errs = [np.linalg.norm(oracle.bitslice_ffn(x, qg, sg, qu, su, qdT, sd, b) - y8) for b in (2, 4, 6)]
    assert errs[0] > errs[1] > errs[2] > 0


def test_bitslice_quantiser_rounds_half_steps_to_even():
    """A row whose largest magnitude is 127 has scale exactly 1, so its other
    entries land on exact half-steps: round half to even (0.5 -> 0, 1.5 -> 2,
    2.5 -> 2, -0.5 -> 0, -1.5 -> -2), not half away from zero; -127 stays the
    symmetric minimum."""
    W = np.array([[127.0, 0.5, 1.5, 2.5, -0.5, -1.5, -127.0, 3.0] * 4], np.float32)
    q, s = oracle.bitslice_quantize(W)
    assert s[0] == 1.0
    np.testing.assert_array_equal(q[0, :8], [127, 0, 2, 2, 0, -2, -127, 3])
