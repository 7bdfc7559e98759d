"""Parity of the bit-sliced expert weights (ELMoE-3D, bit slicing) with the
float64 oracle, through the C ABI: the packed planes and scales bit-exact, the
b-bit draft FFN within float32 accumulation.  GPU only."""
import numpy as np
import pytest
import torch

import expert_routing_ffn_gb300 as moe
import oracle
from workloads import round_bf16

pytestmark = pytest.mark.gpu


def _weights(rng, n, rows, cols, bf16=True):
    w = (rng.standard_normal((n, rows, cols)) * 0.02).astype(np.float32)
    return round_bf16(w) if bf16 else w


def _planes_of(q):
    """The plane words the layout puts for an INT8 matrix q [R, C]."""
    R, Cc = q.shape
    u = q.astype(np.int16) & 0xFF
    out = np.zeros((8, R, Cc // 32), np.uint32)
    for p in range(8):
        bits = ((u >> p) & 1).astype(np.uint32).reshape(R, Cc // 32, 32)
        out[7 - p] = (bits << np.arange(32, dtype=np.uint32)).sum(axis=2).astype(np.uint32)
    return out


def _pack(Ws, transpose, dt):
    n, rows, cols = Ws.shape
    R, Cc = (cols, rows) if transpose else (rows, cols)
    planes = torch.zeros(n * 8 * R * Cc // 32, dtype=torch.int32, device="cuda")
    scales = torch.zeros(n * R, dtype=torch.float32, device="cuda")
    for e in range(n):
        w = torch.from_numpy(Ws[e]).to("cuda").to(dt).contiguous()
        moe.moe_bitslice_pack(w, transpose, planes[e * 8 * R * Cc // 32:(e + 1) * 8 * R * Cc // 32],
                              scales[e * R:(e + 1) * R])
    torch.cuda.synchronize()
    return planes, scales


@pytest.mark.parametrize("rows,cols,transpose", [(96, 256, False), (512, 1536, True), (1408, 2048, False),
                                                 (1408, 2048, True)])
def test_pack_matches_oracle_quantisation(rows, cols, transpose):
    rng = np.random.default_rng(rows + cols)
    W = _weights(rng, 1, rows, cols)
    W[0, 3] = 0.0  # a zero row (a zero column when transposed)
    planes, scales = _pack(W, transpose, torch.bfloat16)
    q, s = oracle.bitslice_quantize(W[0], transpose=transpose)
    np.testing.assert_array_equal(scales.cpu().numpy(), s)
    got = planes.cpu().numpy().view(np.uint32).reshape(8, q.shape[0], q.shape[1] // 32)
    np.testing.assert_array_equal(got, _planes_of(q))


# (d, I, routed experts, shared experts, tokens, slots, bits, x dtype)
CASES = [(2048, 1408, 8, 2, 2, 6, 4, "bf16"), (2048, 1408, 8, 0, 1, 6, 8, "bf16"),
         (2048, 1408, 8, 2, 1, 6, 1, "bf16"), (256, 512, 3, 1, 5, 2, 3, "f32"), (1536, 512, 40, 0, 3, 8, 4, "bf16"),
         (3584, 2560, 4, 1, 1, 8, 2, "bf16")]


@pytest.mark.parametrize("d,I,N,ns,T,k,bits,xt", CASES)
def test_bitslice_ffn_matches_oracle(d, I, N, ns, T, k, bits, xt):
    """y[t] = sum_s gate * FFN_b(idx[t,s], x_t) + the shared experts' FFN_b,
    every expert from the oracle's quantisation; one routed slot names no
    expert and one names a shared expert's index (both contribute 0); the
    second call accumulates onto the first.  Relative L2 <= 1e-4: float32
    table sums and accumulation over d and I terms, no intermediate rounding
    to bf16."""
    rng = np.random.default_rng(d + I + bits)
    bf16 = xt == "bf16"
    dt = torch.bfloat16 if bf16 else torch.float32
    NS = N + ns
    Wg, Wu, Wd = _weights(rng, NS, I, d, bf16), _weights(rng, NS, I, d, bf16), _weights(rng, NS, I, d, bf16)
    pg, sg = _pack(Wg, False, dt)
    pu, su = _pack(Wu, False, dt)
    pd, sd = _pack(Wd, True, dt)
    x = rng.standard_normal((T, d)).astype(np.float32)
    x = round_bf16(x) if bf16 else x
    idx = rng.integers(0, N, size=(T, k)).astype(np.int32)
    idx[0, -1] = -1
    if ns:
        idx[0, 0] = N  # a shared expert's index is not a routed expert
    gate = rng.random((T, k)).astype(np.float32)
    q = {}
    for e in (set(idx.ravel().tolist()) - {-1, N}) | set(range(N, NS)):
        q[e] = (oracle.bitslice_quantize(Wg[e]) + oracle.bitslice_quantize(Wu[e]) +
                oracle.bitslice_quantize(Wd[e], transpose=True))
    ffn = np.zeros((T, k + ns, d))
    for t in range(T):
        for s in range(k + ns):
            e = int(idx[t, s]) if s < k else N + (s - k)
            if 0 <= e < N or s >= k:
                qg, sgo, qu, suo, qd, sdo = q[e]
                ffn[t, s] = oracle.bitslice_ffn(x[t], qg, sgo, qu, suo, qd, sdo, bits)
    want = np.zeros((T, d))
    for t in range(T):
        for s in range(k + ns):
            want[t] += (float(gate[t, s]) if s < k else 1.0) * ffn[t, s]
    xd = torch.from_numpy(x).to("cuda").to(dt)
    idx_d = torch.from_numpy(idx).to("cuda")
    gate_d = torch.from_numpy(gate).to("cuda")
    y = torch.zeros((T, d), dtype=torch.float32, device="cuda")
    scratch = torch.zeros(moe.moe_bitslice_scratch_size(d, I, T, k + ns), dtype=torch.uint8, device="cuda")
    moe.moe_bitslice_ffn(d, I, N, bits, xd, idx_d, gate_d, pg, sg, pu, su, pd, sd, y, scratch, n_shared=ns)
    torch.cuda.synchronize()
    got = y.double().cpu().numpy()
    rel = np.linalg.norm(got - want) / np.linalg.norm(want)
    assert rel <= 1e-4, rel
    moe.moe_bitslice_ffn(d, I, N, bits, xd, idx_d, None, pg, sg, pu, su, pd, sd, y, scratch, accumulate=True,
                         n_shared=ns)
    torch.cuda.synchronize()
    want2 = want + ffn.sum(axis=1)
    got2 = y.double().cpu().numpy()
    assert np.linalg.norm(got2 - want2) / np.linalg.norm(want2) <= 1e-4
