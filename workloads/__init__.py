"""Seeded synthetic inputs for the offloading-aware MoE layer.

This module only draws random numbers and fixes shapes.  It holds none of the
layer's arithmetic (no router, no top-k, no FFN): both the CUDA path and the
float64 oracle take their inputs from here, and nothing else is shared
between them.

Shapes follow the models the four source pages evaluate on (DeepSeek-V2-Lite,
Qwen2-57B-A14B, Mixtral-8x7B, Granite-3B-A800M, plus a tiny fp32 case).  No
checkpoint or dataset is used: weights are N(0, 0.02^2), activations N(0, 1),
LoRE factors N(0, 0.02^2), every draw from its own PCG64 stream keyed by
(seed, stream id, expert, matrix), so any single matrix can be regenerated
without the others and matrices can be filled in parallel.

Values for bf16 layers are rounded to bfloat16 (round to nearest even) once,
here, and returned as float32 arrays whose values are exactly representable
in bf16.  The CUDA side converts them to bf16 (exact); the oracle converts
them to float64 (exact).
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field, replace
from functools import lru_cache

import numpy as np

# Miss policies and slot kinds use the same integer codes as the C ABI.
MISS_EXACT, MISS_SUBSTITUTE, MISS_LORE, MISS_HYBRID = 0, 1, 2, 3
KIND_COMPUTE, KIND_FETCH, KIND_LORE = 0, 1, 2
ALL_RESIDENT = (1 << 64) - 1

# Stream ids for the per-matrix generators.
_S_ROUTER, _S_PREF_NOISE, _S_WORD, _S_THETA, _S_GATE, _S_UP, _S_DOWN = 1, 2, 3, 4, 5, 6, 7
_S_SH_GATE, _S_SH_UP, _S_SH_DOWN, _S_LORE_A, _S_LORE_B, _S_BIAS, _S_X = 8, 9, 10, 11, 12, 13, 14
_S_AHEAD = 15


@dataclass(frozen=True)
class LayerConfig:
    """Shape and policy of one synthetic MoE layer.

    d: hidden size; N: routed experts; k: top-k; I: routed expert
    intermediate size; n_shared / I_shared: shared experts and their
    intermediate size; r: LoRE rank (0 = no LoRE factors); delta_max = N - k.
    wtype: "bf16" or "f32" (weights and activations).
    policy: miss policy code; gamma: HYBRID threshold on the router
    probability; n_resident: size of the batch-level resident set (0 = use
    the per-token prefetch set as the available set, -1 = every expert
    resident); use_prefetch_mask: whether the per-token prefetch set enters
    the available set.
    zipf: exponent of the per-expert router bias that skews expert load
    (0 = no bias).  keep_frac: FloE channel keep fraction (1.0 = dense).
    theta_centre / theta_spread: the synthetic ordinal-CDF thresholds put the
    tau=0.9 budget at about theta_centre, moving by about theta_spread per
    standard deviation of w.x.
    """

    name: str
    d: int
    N: int
    k: int
    I: int
    n_shared: int
    I_shared: int
    r: int
    wtype: str
    tau: float
    policy: int
    gamma: float
    n_resident: int
    use_prefetch_mask: bool
    T: int
    zipf: float = 0.0
    keep_frac: float = 1.0
    prefetch_rho: float = 0.2
    theta_centre: float = 3.5
    theta_spread: float = 2.0
    seed: int = 0
    decode_T: tuple = field(default=())

    @property
    def delta_max(self) -> int:
        return self.N - self.k

    def with_(self, **kw) -> "LayerConfig":
        return replace(self, **kw)


# The five layers.  gamma values for the HYBRID layers are the median router
# probability of the routed (token, expert) pairs that miss the available set
# in the seed-0 inputs, rounded to three decimals, so that both HYBRID
# branches (LoRE and substitution) occur (tests/golden/make_gamma.py).
CONFIGS = {
    "tiny": LayerConfig(
        name="tiny", d=256, N=8, k=2, I=512, n_shared=1, I_shared=512, r=8,
        wtype="f32", tau=0.9, policy=MISS_HYBRID, gamma=0.149, n_resident=0,
        use_prefetch_mask=True, T=16, prefetch_rho=0.5, theta_centre=1.0),
    "dsv2lite": LayerConfig(
        name="dsv2lite", d=2048, N=64, k=6, I=1408, n_shared=2, I_shared=1408,
        r=16, wtype="bf16", tau=0.9, policy=MISS_HYBRID, gamma=0.05,
        n_resident=24, use_prefetch_mask=False, T=8, decode_T=(1, 8)),
    "qwen2": LayerConfig(
        name="qwen2", d=3584, N=64, k=8, I=2560, n_shared=1, I_shared=20480,
        r=32, wtype="bf16", tau=0.9, policy=MISS_HYBRID, gamma=0.072,
        n_resident=48, use_prefetch_mask=False, T=4096, zipf=1.1),
    "mixtral": LayerConfig(
        name="mixtral", d=4096, N=8, k=2, I=14336, n_shared=0, I_shared=0,
        r=0, wtype="bf16", tau=0.9, policy=MISS_EXACT, gamma=0.0,
        n_resident=-1, use_prefetch_mask=False, T=32,
        decode_T=(1, 2, 4, 8, 16, 32)),
    "granite": LayerConfig(
        name="granite", d=1536, N=40, k=8, I=512, n_shared=0, I_shared=0,
        r=0, wtype="bf16", tau=0.9, policy=MISS_SUBSTITUTE, gamma=0.0,
        n_resident=0, use_prefetch_mask=True, T=1024),
}


def _rng(seed: int, *key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=key)))


def _normal(seed: int, key: tuple, shape, std: float) -> np.ndarray:
    a = _rng(seed, *key).standard_normal(int(np.prod(shape)), dtype=np.float32)
    a *= np.float32(std)
    return a.reshape(shape)


def round_bf16(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even), in place.

    Returns float32 values that bf16 represents exactly.  Inputs are finite.
    """
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    step = 1 << 22
    for s in range(0, u.size, step):
        v = u.reshape(-1)[s:s + step]
        lsb = (v >> np.uint32(16)) & np.uint32(1)
        lsb += np.uint32(0x7FFF)
        v += lsb
        v &= np.uint32(0xFFFF0000)
    return a


def _weights(cfg: LayerConfig, seed: int, key: tuple, shape, std: float) -> np.ndarray:
    a = _normal(seed, key, shape, std)
    return round_bf16(a) if cfg.wtype == "bf16" else a


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


@dataclass
class LayerWeights:
    """All parameters of one layer, as float32 arrays (bf16-exact for bf16)."""

    w_router: np.ndarray      # [N, d]
    w_prefetch: np.ndarray    # [N, d]
    w_ord: np.ndarray         # [d]   ordinal-CDF scorer w
    theta: np.ndarray         # [delta_max + 1], non-decreasing
    router_bias: np.ndarray | None   # [N] or None
    w_gate: np.ndarray        # [N, I, d]  channel-major rows
    w_up: np.ndarray          # [N, I, d]
    w_down: np.ndarray        # [N, I, d]  row i = down-projection of channel i
    sh_gate: np.ndarray       # [n_shared, I_shared, d]
    sh_up: np.ndarray
    sh_down: np.ndarray
    lore_a: np.ndarray        # [N, r, d]
    lore_b: np.ndarray        # [N, d, r]


def make_weights(cfg: LayerConfig, seed: int | None = None, experts=None) -> LayerWeights:
    """Draw every weight of the layer.

    experts: optional iterable of routed expert ids to fill; the others are
    left as zeros (used by tests that only need a few experts at full size).
    """
    seed = cfg.seed if seed is None else seed
    d, N, I, r = cfg.d, cfg.N, cfg.I, cfg.r
    std = 0.02
    w_router = _weights(cfg, seed, (_S_ROUTER,), (N, d), std)
    noise = _weights(cfg, seed, (_S_PREF_NOISE,), (N, d), std * cfg.prefetch_rho)
    w_prefetch = w_router + noise
    if cfg.wtype == "bf16":
        w_prefetch = round_bf16(w_prefetch)
    # w is drawn at bf16 precision so that w_j * x_j is exact in fp32.
    w_ord = round_bf16(_normal(seed, (_S_WORD,), (d,), std))
    # Synthetic ordinal thresholds: evenly spaced around logit(0.9) so that the
    # tau=0.9 budget lands near theta_centre, with a small seeded jitter, then
    # sorted so that theta_0 <= ... <= theta_{N-k} as the model requires.
    dm = cfg.delta_max
    sigma_s = std * math.sqrt(d)
    slope = sigma_s / cfg.theta_spread
    jitter = _rng(seed, _S_THETA).standard_normal(dm + 1) * (0.05 * slope)
    theta = math.log(0.9 / 0.1) + slope * (np.arange(dm + 1) - cfg.theta_centre) + jitter
    theta = np.sort(theta).astype(np.float32)
    bias = None
    if cfg.zipf > 0:
        perm = _rng(seed, _S_BIAS).permutation(N)
        bias = (-cfg.zipf * np.log(perm.astype(np.float64) + 1.0)).astype(np.float32)

    shp = (N, I, d)
    w_gate = np.zeros(shp, np.float32)
    w_up = np.zeros(shp, np.float32)
    w_down = np.zeros(shp, np.float32)
    ns, Is = cfg.n_shared, cfg.I_shared
    sh_gate = np.zeros((ns, Is, d), np.float32)
    sh_up = np.zeros((ns, Is, d), np.float32)
    sh_down = np.zeros((ns, Is, d), np.float32)
    lore_a = np.zeros((N, r, d), np.float32)
    lore_b = np.zeros((N, d, r), np.float32)
    ids = range(N) if experts is None else sorted(set(int(e) for e in experts))
    jobs = []
    for e in ids:
        jobs += [(w_gate, e, (_S_GATE, e)), (w_up, e, (_S_UP, e)), (w_down, e, (_S_DOWN, e))]
    for s in range(ns):
        jobs += [(sh_gate, s, (_S_SH_GATE, s)), (sh_up, s, (_S_SH_UP, s)), (sh_down, s, (_S_SH_DOWN, s))]
    if r > 0:
        for e in ids:
            jobs += [(lore_a, e, (_S_LORE_A, e)), (lore_b, e, (_S_LORE_B, e))]

    def fill(job):
        dst, i, key = job
        dst[i] = _weights(cfg, seed, key, dst.shape[1:], std)

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(fill, jobs))
    return LayerWeights(w_router, w_prefetch, w_ord, theta, bias, w_gate, w_up, w_down,
                        sh_gate, sh_up, sh_down, lore_a, lore_b)


def make_tokens(cfg: LayerConfig, T: int | None = None, seed: int | None = None, batch: int = 0) -> np.ndarray:
    """Activations x [T, d] ~ N(0, 1); `batch` selects an independent draw."""
    seed = cfg.seed if seed is None else seed
    T = cfg.T if T is None else T
    x = _normal(seed, (_S_X, batch), (T, cfg.d), 1.0)
    return round_bf16(x) if cfg.wtype == "bf16" else x


def make_lookahead_routers(cfg: LayerConfig, J: int, seed: int | None = None):
    """Routers of the next J layers of a synthetic layer stack, for the
    look-ahead prefetch depth: look-ahead layer j's router mixes this layer's
    router with seeded N(0, 0.02^2) noise at constant norm, the noise share
    a_j = min(0.9, 0.3 (j + 1)), and is scaled by 1.5 / (1 + j / 2), so the
    predicted distributions drift and flatten with depth (bf16-exact for bf16
    layers).  A Zipf router bias, when the layer has one, is shared by every
    layer.  Returns (routers [J] of [N, d], biases [J] of [N] or None)."""
    seed = cfg.seed if seed is None else seed
    base = _normal(seed, (_S_ROUTER,), (cfg.N, cfg.d), 0.02)
    Ws = []
    for j in range(J):
        a = min(0.9, 0.3 * (j + 1))
        noise = _normal(seed, (_S_AHEAD, j), (cfg.N, cfg.d), 0.02)
        w = (np.float32(math.sqrt(1.0 - a * a)) * base + np.float32(a) * noise) * np.float32(1.5 / (1.0 + 0.5 * j))
        Ws.append(round_bf16(w) if cfg.wtype == "bf16" else np.ascontiguousarray(w, np.float32))
    biases = None
    if cfg.zipf > 0:
        perm = _rng(seed, _S_BIAS).permutation(cfg.N)
        b = (-cfg.zipf * np.log(perm.astype(np.float64) + 1.0)).astype(np.float32)
        biases = [b] * J
    return Ws, biases


@lru_cache(maxsize=4)
def cached_weights(name: str, seed: int = 0) -> LayerWeights:
    return make_weights(CONFIGS[name], seed)


def n_keep(cfg: LayerConfig) -> int:
    """FloE keep count m = ceil(keep_frac * I)."""
    return int(math.ceil(cfg.keep_frac * cfg.I - 1e-9))
