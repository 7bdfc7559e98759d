"""Float64 CPU oracle for the offloading-aware MoE layer — TEST INFRASTRUCTURE.

Only the tests, the smoke check and the benchmark's CPU-baseline leg use this
package.  The CUDA library never imports, links or calls it, and it shares no
code with the CUDA path; the two meet only in the seeded inputs of
`workloads`.

The arithmetic lives in `moe_oracle.c` (plain C, double precision, one token
at a time, OpenMP over tokens).  This module compiles it with gcc and wraps
it with ctypes.  Each C function cites the page and section it follows.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

# decisive-margin columns (match the M_* enum in moe_oracle.c)
M_TOPK, M_PREFETCH, M_THETA, M_DSTAR, M_SUBST, M_GAMMA, M_FLOE, M_COST = range(8)
M_COUNT = 8
MARGIN_NAMES = ["topk", "prefetch", "theta", "delta_star", "substitute", "gamma", "floe", "cost"]
POL_HETERO = 4
KIND_CPU = 3
COST_FIELDS = ("link_bps", "expert_bytes", "gpu_expert_s", "cpu_row_s", "hidden_bytes")


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into liboracle.so next to it (OpenMP if available)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", _LIB_PATH + ".tmp", _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


class _Cfg(C.Structure):
    _fields_ = [(n, C.c_int) for n in ("T", "d", "N", "k", "I", "n_shared", "I_shared", "r",
                                       "delta_max", "renorm", "policy", "use_prefetch",
                                       "m_keep", "has_prefetch", "route_only")] + [
        ("tau", C.c_double), ("gamma", C.c_double), ("resident", C.c_uint64)] + [
        (n, C.c_double) for n in ("link_bps", "expert_bytes", "gpu_expert_s", "cpu_row_s", "hidden_bytes")]


_FP = C.POINTER(C.c_float)
_DP = C.POINTER(C.c_double)
_IP = C.POINTER(C.c_int)
_UP = C.POINTER(C.c_uint64)


class _Inputs(C.Structure):
    _fields_ = [(n, _FP) for n in ("x", "x_pre", "w_router", "router_bias", "w_prefetch", "w_ord",
                                   "theta", "w_gate", "w_up", "w_down", "sh_gate", "sh_up",
                                   "sh_down", "lore_a", "lore_b")]


class _Outputs(C.Structure):
    _fields_ = [("logits", _DP), ("prob", _DP), ("logits_p", _DP), ("topk_idx", _IP),
                ("topk_gate", _DP), ("delta_hat", _IP), ("score", _DP), ("prefetch", _UP),
                ("delta_star", _IP), ("final_idx", _IP), ("final_gate", _DP),
                ("final_kind", _IP), ("y_shared", _DP), ("out", _DP), ("margin", _DP),
                ("kept", _IP), ("status", _IP)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = C.CDLL(build())
            L.orc_num_threads.restype = C.c_int
            L.orc_set_num_threads.argtypes = [C.c_int]
            L.orc_set_num_threads.restype = None
            L.orc_logits.argtypes = [C.c_int, C.c_int, C.c_int, _FP, _FP, _FP, _DP]
            L.orc_softmax.argtypes = [C.c_int, _DP, _DP]
            L.orc_topk.argtypes = [C.c_int, C.c_int, _DP, _IP]
            L.orc_delta_hat.argtypes = [C.c_int, C.c_int, _FP, _FP, _FP, C.c_double, _DP]
            L.orc_delta_hat.restype = C.c_int
            L.orc_prefetch_set.argtypes = [C.c_int, C.c_int, C.c_int, _DP]
            L.orc_prefetch_set.restype = C.c_uint64
            L.orc_delta_star.argtypes = [C.c_int, C.c_int, _IP, _DP]
            L.orc_delta_star.restype = C.c_int
            L.orc_stall_free_select.argtypes = [C.c_int, C.c_uint64, _DP, C.c_uint64]
            L.orc_stall_free_select.restype = C.c_uint64
            L.orc_expert_ffn.argtypes = [C.c_int, C.c_int, _FP, _FP, _FP, _FP, _DP]
            L.orc_expert_ffn_floe.argtypes = [C.c_int, C.c_int, C.c_int, _FP, _FP, _FP, _FP, _DP,
                                              _IP, _DP]
            L.orc_lore.argtypes = [C.c_int, C.c_int, _FP, _FP, _FP, _DP]
            L.orc_batch_resident.argtypes = [C.c_int, C.c_int, _DP, C.c_int, _DP]
            L.orc_batch_resident.restype = C.c_uint64
            L.orc_cache_update.argtypes = [C.c_int, C.c_int, _IP, C.c_double, C.c_int, _DP, C.c_uint64,
                                           C.POINTER(C.c_int), _DP]
            L.orc_cache_update.restype = C.c_uint64
            L.orc_prefetch_depth.argtypes = [C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, _FP,
                                             C.POINTER(_FP), C.POINTER(_FP), C.c_double, C.c_int, _DP, _IP,
                                             C.POINTER(C.c_uint64), C.POINTER(C.c_uint64), _DP]
            L.orc_prefetch_depth.restype = None
            _BP = C.POINTER(C.c_byte)
            L.orc_bitslice_quantize.argtypes = [C.c_int, C.c_int, _FP, C.c_int, _BP, _FP]
            L.orc_bitslice_quantize.restype = None
            L.orc_bitslice_value.argtypes = [C.c_int, C.c_int]
            L.orc_bitslice_value.restype = C.c_int
            L.orc_bitslice_ffn.argtypes = [C.c_int, C.c_int, C.c_int, _FP, _BP, _FP, _BP, _FP, _BP, _FP, _DP]
            L.orc_bitslice_ffn.restype = None
            L.orc_layer_forward.argtypes = [C.POINTER(_Cfg), C.POINTER(_Inputs), C.POINTER(_Outputs)]
            L.orc_hetero_fetch.argtypes = [C.c_int] + [C.c_double] * 5 + [_DP]
            L.orc_hetero_fetch.restype = C.c_int
            _lib = L
    return _lib


def _f(a):
    if a is None:
        return None
    assert a.dtype == np.float32 and a.flags.c_contiguous
    return a.ctypes.data_as(_FP)


def _d(a):
    assert a.dtype == np.float64 and a.flags.c_contiguous
    return a.ctypes.data_as(_DP)


def _i(a):
    assert a.dtype == np.int32 and a.flags.c_contiguous
    return a.ctypes.data_as(_IP)


def f32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32)


def num_threads() -> int:
    return lib().orc_num_threads()


def set_num_threads(n: int) -> None:
    """OpenMP threads of the calling Python thread's later oracle calls."""
    lib().orc_set_num_threads(int(n))


# ---- single steps (used by the pins) -------------------------------------

def logits(x, W, bias=None) -> np.ndarray:
    x, W = f32(x), f32(W)
    T, d = x.shape
    N = W.shape[0]
    out = np.zeros((T, N), np.float64)
    lib().orc_logits(T, d, N, _f(x), _f(W), _f(None if bias is None else f32(bias)), _d(out))
    return out


def softmax(l) -> np.ndarray:
    l = np.ascontiguousarray(l, np.float64)
    out = np.zeros_like(l)
    lib().orc_softmax(l.shape[-1], _d(l), _d(out))
    return out


def topk(v, k) -> np.ndarray:
    v = np.ascontiguousarray(v, np.float64)
    idx = np.zeros(k, np.int32)
    lib().orc_topk(v.shape[0], k, _d(v), _i(idx))
    return idx


def delta_hat(w, x_pre, theta, tau):
    w, x_pre, theta = f32(w), f32(x_pre), f32(theta)
    s = C.c_double()
    dh = lib().orc_delta_hat(w.shape[0], theta.shape[0] - 1, _f(w), _f(x_pre), _f(theta), tau, C.byref(s))
    return dh, s.value


def prefetch_set(k, dh, lp) -> int:
    lp = np.ascontiguousarray(lp, np.float64)
    return int(lib().orc_prefetch_set(lp.shape[0], k, dh, _d(lp)))


def delta_star(routed, lp) -> int:
    routed = np.ascontiguousarray(routed, np.int32)
    lp = np.ascontiguousarray(lp, np.float64)
    return lib().orc_delta_star(lp.shape[0], routed.shape[0], _i(routed), _d(lp))


def stall_free_select(N, routed_mask, alpha, prefetched_mask) -> int:
    alpha = np.ascontiguousarray(alpha, np.float64)
    return int(lib().orc_stall_free_select(N, routed_mask, _d(alpha), prefetched_mask))


def expert_ffn(x, Wg, Wu, Wd) -> np.ndarray:
    x, Wg, Wu, Wd = f32(x), f32(Wg), f32(Wu), f32(Wd)
    I, d = Wg.shape
    y = np.zeros(d, np.float64)
    lib().orc_expert_ffn(d, I, _f(x), _f(Wg), _f(Wu), _f(Wd), _d(y))
    return y


def expert_ffn_floe(x, Wg, Wu, Wd, m):
    x, Wg, Wu, Wd = f32(x), f32(Wg), f32(Wu), f32(Wd)
    I, d = Wg.shape
    y = np.zeros(d, np.float64)
    kept = np.zeros(m, np.int32)
    gap = C.c_double()
    lib().orc_expert_ffn_floe(d, I, m, _f(x), _f(Wg), _f(Wu), _f(Wd), _d(y), _i(kept), C.byref(gap))
    return y, kept, gap.value


def lore(x, A, B) -> np.ndarray:
    x, A, B = f32(x), f32(A), f32(B)
    r, d = A.shape
    v = np.zeros(d, np.float64)
    lib().orc_lore(d, r, _f(x), _f(A), _f(B), _d(v))
    return v


def hetero_fetch(n: int, cost: dict) -> tuple[bool, float]:
    """SPICE's per-miss cost model for an expert needed by n token rows:
    (fetch wins, relative cost gap).  cost: the COST_FIELDS."""
    m = C.c_double()
    f = lib().orc_hetero_fetch(int(n), *[float(cost[k]) for k in COST_FIELDS], C.byref(m))
    return bool(f), m.value


def batch_resident(lp, n_res):
    lp = np.ascontiguousarray(lp, np.float64)
    T, N = lp.shape
    gap = C.c_double()
    m = lib().orc_batch_resident(T, N, _d(lp), n_res, C.byref(gap))
    return int(m), gap.value


def cache_update(routed, heat, decay, capacity, old_cache):
    """One decode step of the persistent expert cache (ELMoE-3D heat map with
    decay): returns (new cache mask, updated heat [float64], hits, boundary gap)."""
    routed = np.ascontiguousarray(np.asarray(routed).ravel(), np.int32)
    heat = np.array(heat, np.float64, copy=True)
    hits, gap = C.c_int(), C.c_double()
    m = lib().orc_cache_update(len(heat), len(routed), routed.ctypes.data_as(_IP), float(decay), int(capacity),
                               _d(heat), C.c_uint64(old_cache), C.byref(hits), C.byref(gap))
    return int(m), heat, hits.value, gap.value


def prefetch_depth(x, Ws, biases, K, tau, d_min):
    """Confidence-aware prefetch depth over J look-ahead routers (SPICE
    write-up, confidence-aware adaptive prefetch).  Ws: J arrays [N, d];
    biases: None or J arrays [N] (entries may be None).  Returns
    (conf [T,J] float64, depth [T] int, tok_masks [T,J] uint64,
    layer_masks [J] uint64, margin [T] float64)."""
    xs = f32(x)
    T, d = xs.shape
    J = len(Ws)
    Wf = [f32(W) for W in Ws]
    N = Wf[0].shape[0]
    if not (1 <= J <= 64 and 1 <= K <= N <= 64):
        raise ValueError("prefetch_depth: 1 <= J <= 64 look-ahead layers and 1 <= K <= N <= 64 experts")
    Wp = (_FP * J)(*[_f(W) for W in Wf])
    if biases is None:
        bp = None
        keep = []
    else:
        keep = [None if b is None else f32(b) for b in biases]
        bp = (_FP * J)(*[C.cast(None, _FP) if b is None else _f(b) for b in keep])
    conf = np.zeros((T, J), np.float64)
    depth = np.zeros(T, np.int32)
    tok = np.zeros((T, J), np.uint64)
    lay = np.zeros(J, np.uint64)
    margin = np.zeros(T, np.float64)
    lib().orc_prefetch_depth(T, d, N, int(K), J, _f(xs), Wp, bp, float(tau), int(d_min), _d(conf),
                             depth.ctypes.data_as(_IP), tok.ctypes.data_as(C.POINTER(C.c_uint64)),
                             lay.ctypes.data_as(C.POINTER(C.c_uint64)), _d(margin))
    del keep
    return conf, depth.astype(np.int64), tok, lay, margin


def bitslice_quantize(W, transpose=False):
    """Symmetric per-row INT8 quantisation of W (or W^T) in float32
    arithmetic, for the bit-sliced weights (ELMoE-3D).  Returns (q int8
    [R, C], scale float32 [R])."""
    Wf = f32(W)
    rows, cols = Wf.shape
    R, Cc = (cols, rows) if transpose else (rows, cols)
    q = np.zeros((R, Cc), np.int8)
    sc = np.zeros(R, np.float32)
    lib().orc_bitslice_quantize(rows, cols, _f(Wf), int(bool(transpose)), q.ctypes.data_as(C.POINTER(C.c_byte)),
                                sc.ctypes.data_as(_FP))
    return q, sc


def bitslice_value(q: int, b: int) -> int:
    """The b-bit value of INT8 weight q: its top b bit planes recombined."""
    return int(lib().orc_bitslice_value(int(q), int(b)))


def bitslice_ffn(x, qg, sg, qu, su, qdT, sd, b):
    """One expert on one token with b-bit weights: y [d] float64."""
    x = f32(np.asarray(x).ravel())
    I, d = qg.shape
    y = np.zeros(d, np.float64)
    bp = C.POINTER(C.c_byte)
    cont = lambda a: np.ascontiguousarray(a, np.int8)
    qg, qu, qdT = cont(qg), cont(qu), cont(qdT)
    lib().orc_bitslice_ffn(d, I, int(b), _f(x), qg.ctypes.data_as(bp), _f(f32(sg)), qu.ctypes.data_as(bp),
                           _f(f32(su)), qdT.ctypes.data_as(bp), _f(f32(sd)), _d(y))
    return y


# ---- whole layer ---------------------------------------------------------

@dataclass
class LayerResult:
    logits: np.ndarray
    prob: np.ndarray
    logits_p: np.ndarray
    topk_idx: np.ndarray
    topk_gate: np.ndarray
    delta_hat: np.ndarray
    score: np.ndarray
    prefetch: np.ndarray
    delta_star: np.ndarray
    final_idx: np.ndarray
    final_gate: np.ndarray
    final_kind: np.ndarray
    y_shared: np.ndarray
    out: np.ndarray
    margin: np.ndarray
    kept: np.ndarray | None
    status: np.ndarray
    resident: int
    resident_gap: float

    def excluded(self, eps: float = 1e-5, floe: bool = True) -> np.ndarray:
        """Tokens with any decisive margin below eps (near ties).  floe=False
        leaves the FloE channel-gap margin out (for comparisons that accept
        either side of a near-tied channel instead of dropping the token)."""
        m = self.margin if floe else np.delete(self.margin, M_FLOE, axis=1)
        return (m < eps).any(axis=1)


def resident_mask(cfg, W, x_batch) -> tuple[int, float]:
    """Batch resident set for a layer config (or every expert)."""
    if cfg.n_resident < 0:
        return (1 << 64) - 1, float("inf")
    if cfg.n_resident == 0:
        return (1 << 64) - 1, float("inf")
    lp = logits(x_batch, W.w_prefetch)
    return batch_resident(lp, cfg.n_resident)


def layer_forward(cfg, W, x, resident: int | None = None, x_pre=None, keep_m: int | None = None,
                  policy: int | None = None, gamma: float | None = None, tau: float | None = None,
                  renorm: int = 0, use_prefetch: bool | None = None,
                  route_only: bool = False, cost: dict | None = None) -> LayerResult:
    """Run the whole layer for the tokens x [T, d].

    resident: batch-level resident mask (default: computed from x itself with
    the config's n_resident).  keep_m: FloE channels kept (default: dense).
    route_only: stop after the routing decisions (outputs stay zero).
    cost: the HETERO policy's cost model (COST_FIELDS), required with it.
    """
    x = f32(x)
    T, d = x.shape
    N, k = cfg.N, cfg.k
    res_gap = float("inf")
    if resident is None:
        resident, res_gap = resident_mask(cfg, W, x)
    c = _Cfg()
    c.T, c.d, c.N, c.k, c.I = T, d, N, k, cfg.I
    c.n_shared, c.I_shared, c.r, c.delta_max = cfg.n_shared, cfg.I_shared, cfg.r, cfg.delta_max
    c.renorm = renorm
    c.policy = cfg.policy if policy is None else policy
    c.use_prefetch = int(cfg.use_prefetch_mask if use_prefetch is None else use_prefetch)
    c.m_keep = cfg.I if keep_m is None else keep_m
    c.has_prefetch = 1
    c.route_only = int(route_only)
    c.tau = cfg.tau if tau is None else tau
    c.gamma = cfg.gamma if gamma is None else gamma
    c.resident = resident
    if c.policy == POL_HETERO:
        if cost is None:
            raise ValueError("the HETERO policy needs its cost model")
        for k_ in COST_FIELDS:
            setattr(c, k_, float(cost[k_]))
    keep = [x]  # keep arrays alive
    inp = _Inputs()
    inp.x = _f(x)
    if x_pre is not None:
        xp = f32(x_pre); keep.append(xp); inp.x_pre = _f(xp)
    for name in ("w_router", "w_prefetch", "w_ord", "theta", "w_gate", "w_up", "w_down",
                 "sh_gate", "sh_up", "sh_down", "lore_a", "lore_b"):
        a = f32(getattr(W, name)); keep.append(a); setattr(inp, name, _f(a))
    if W.router_bias is not None:
        b = f32(W.router_bias); keep.append(b); inp.router_bias = _f(b)
    R = LayerResult(
        logits=np.zeros((T, N)), prob=np.zeros((T, N)), logits_p=np.zeros((T, N)),
        topk_idx=np.zeros((T, k), np.int32), topk_gate=np.zeros((T, k)),
        delta_hat=np.zeros(T, np.int32), score=np.zeros(T), prefetch=np.zeros(T, np.uint64),
        delta_star=np.zeros(T, np.int32), final_idx=np.zeros((T, k), np.int32),
        final_gate=np.zeros((T, k)), final_kind=np.zeros((T, k), np.int32),
        y_shared=np.zeros((T, 0 if route_only else d)), out=np.zeros((T, 0 if route_only else d)),
        margin=np.zeros((T, M_COUNT)),
        kept=np.zeros((T, k, c.m_keep), np.int32) if c.m_keep < cfg.I else None,
        status=np.zeros(T, np.int32), resident=resident, resident_gap=res_gap)
    o = _Outputs()
    for name in ("logits", "prob", "logits_p", "topk_gate", "score", "final_gate", "y_shared",
                 "out", "margin"):
        setattr(o, name, _d(getattr(R, name)))
    for name in ("topk_idx", "delta_hat", "delta_star", "final_idx", "final_kind", "status"):
        setattr(o, name, _i(getattr(R, name)))
    o.prefetch = R.prefetch.ctypes.data_as(_UP)
    if R.kept is not None:
        o.kept = _i(R.kept)
    lib().orc_layer_forward(C.byref(c), C.byref(inp), C.byref(o))
    return R
