"""The C-ABI library on a machine without a GPU: it loads, exports every
function the headers declare, and rejects bad arguments on the host before
any CUDA call.  No compute call is made here."""
import ctypes as C
import glob
import os
import re

import pytest

import expert_routing_ffn_gb300 as moe
from workloads import CONFIGS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        txt = open(h).read()
        txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
        names |= set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", txt))
    return names


def test_library_loads_and_exports_every_declared_symbol():
    L = moe.lib()
    names = _declared()
    assert len(names) >= 15
    for n in sorted(names):
        assert hasattr(L, n), f"{n} declared in include/ but not exported"


def test_status_strings():
    for s in range(8):
        assert moe.status_string(s) and "unknown" not in moe.status_string(s)
    assert "unknown" in moe.status_string(99)


@pytest.mark.parametrize("name", sorted(CONFIGS))
def test_workspace_size_grows_with_T(name):
    cfg = CONFIGS[name]
    sizes = [moe.moe_workspace_size(moe.make_dims(T, cfg.d, cfg.N, cfg.k, cfg.I, cfg.n_shared,
                                                  cfg.I_shared, cfg.r, wtype=cfg.wtype))
             for T in (1, 8, 64, 1024)]
    assert all(a < b for a, b in zip(sizes, sizes[1:]))
    assert moe.moe_expert_table_size(moe.make_dims(1, cfg.d, cfg.N, cfg.k, cfg.I, cfg.n_shared,
                                                   cfg.I_shared, cfg.r, wtype=cfg.wtype)) > 0


@pytest.mark.parametrize("kw,status", [
    (dict(N=65), moe.MOE_ERR_UNSUPPORTED),
    (dict(k=9, N=16), moe.MOE_ERR_UNSUPPORTED),
    (dict(d=300), moe.MOE_ERR_UNSUPPORTED),
    (dict(d=8192), moe.MOE_ERR_UNSUPPORTED),
    (dict(wtype="f32", d=2048), moe.MOE_ERR_UNSUPPORTED),
    (dict(k=0), moe.MOE_ERR_INVALID_ARG),
    (dict(T=-1), moe.MOE_ERR_INVALID_ARG),
    (dict(delta_max=60, N=8, k=2), moe.MOE_ERR_INVALID_ARG),
    (dict(n_shared=1, I_shared=0), moe.MOE_ERR_INVALID_ARG),
])
def test_bad_dims_rejected(kw, status):
    base = dict(T=4, d=256, N=8, k=2, I=64, n_shared=0, I_shared=0, r=0, wtype="bf16")
    base.update(kw)
    D = moe.make_dims(**base)
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_workspace_size(D)
    assert ei.value.status == status


def _raw_dims(**kw):
    base = dict(T=4, d=256, N=8, k=2, I=64, n_shared=0, I_shared=0, r=0, wtype="bf16")
    base.update(kw)
    return moe.make_dims(**base)


def test_null_buffers_rejected_before_cuda():
    L = moe.lib()
    D = _raw_dims()
    # no workspace
    st = L.moe_route(C.byref(D), None, None, None, None, None, None, None, 0.9, 0, None, None, None,
                     None, None, None, None, None, 0, None)
    assert st == moe.MOE_ERR_INVALID_ARG
    # workspace present but too small
    fake_ws = C.c_void_p(1 << 20)  # aligned, never dereferenced on this path
    st = L.moe_permute(C.byref(D), None, None, None, None, None, fake_ws, 16, None)
    assert st == moe.MOE_ERR_CAPACITY
    st = L.moe_combine(C.byref(D), None, None, None, None, None, None, None, None)
    assert st == moe.MOE_ERR_INVALID_ARG
    # LoRE needs a rank
    st = L.moe_lore(C.byref(D), None, None, None, None, None, None, None, None, 0, None)
    assert st == moe.MOE_ERR_INVALID_ARG
    # a bad miss policy
    n = moe.moe_workspace_size(D)
    st = L.moe_select_resident(C.byref(D), None, None, None, None, 7, 0.1, None, None, None, None,
                               None, None, None, fake_ws, n, None)
    assert st == moe.MOE_ERR_INVALID_ARG


def test_prefill_ffn_rejects_misaligned_outputs_before_cuda():
    """The prefill tensor-core FFN writes y_perm and y_shared with TMA stores:
    an output that is not 16-byte aligned is an argument error, found before
    any CUDA call."""
    L = moe.lib()
    D = _raw_dims(T=100, d=256, N=8, k=2, I=128)
    n = moe.moe_workspace_size(D)
    fake_ws = C.c_void_p(1 << 20)
    x, table, offs, perm = C.c_void_p(0x1000), C.c_void_p(0x2000), C.c_void_p(0x3000), C.c_void_p(0x4000)
    fn = L.moe_expert_ffn
    st = fn(C.byref(D), x, table, offs, perm, C.c_float(1.0), C.c_void_p(0x5004), None, fake_ws, n, None)
    assert st == moe.MOE_ERR_INVALID_ARG


def test_staging_failure_is_reported_on_the_host():
    """An injected copy failure makes moe_stage_experts return
    MOE_ERR_STAGING before anything is queued (no GPU fault involved)."""
    L = moe.lib()
    D = _raw_dims(N=4, k=2)
    ptrs = (C.c_void_p * 4)(*[0x1000 * (i + 1) for i in range(4)])
    n = C.c_size_t(123)
    moe.moe_testing_fail_copies_after(0)
    try:
        st = L.moe_stage_experts(C.byref(D), 0b0101, ptrs, ptrs, ptrs, ptrs, ptrs, ptrs, None,
                                 C.c_void_p(0x10), C.byref(n))
    finally:
        moe.moe_testing_fail_copies_after(-1)
    assert st == moe.MOE_ERR_STAGING
    assert n.value == 0
    # a mask naming an expert beyond N is an argument error
    st = L.moe_stage_experts(C.byref(D), 1 << 5, ptrs, ptrs, ptrs, ptrs, ptrs, ptrs, None,
                             C.c_void_p(0x10), C.byref(n))
    assert st == moe.MOE_ERR_INVALID_ARG


def test_empty_mask_stages_nothing_without_gpu_calls_failing():
    L = moe.lib()
    D = _raw_dims(N=4, k=2)
    ptrs = (C.c_void_p * 4)(*[0x1000 * (i + 1) for i in range(4)])
    n = C.c_size_t(7)
    st = L.moe_stage_experts(C.byref(D), 0, ptrs, ptrs, ptrs, ptrs, ptrs, ptrs, None,
                             C.c_void_p(0x10), C.byref(n))
    # with nothing to copy only the event record remains; without a GPU it fails as STAGING
    assert st in (moe.MOE_OK, moe.MOE_ERR_STAGING)
    assert n.value == 0


def _dims(name, T):
    c = CONFIGS[name]
    return moe.make_dims(T, c.d, c.N, c.k, c.I, c.n_shared, c.I_shared, c.r, c.delta_max, c.wtype)


@pytest.mark.parametrize("name,T,keep,path", [
    ("tiny", 16, 1.0, "gemv"),               # fp32 layer: CUDA-core GEMV
    ("dsv2lite", 1, 1.0, "gemv-1tok"),       # one token, d 1536 / 2048: a channel per warp
    ("granite", 1, 1.0, "gemv-1tok"),
    ("mixtral", 1, 1.0, "gemv"),             # 1..3 tokens: CUDA-core GEMV
    ("dsv2lite", 2, 1.0, "gemv"),
    ("dsv2lite", 3, 1.0, "gemv"),
    ("dsv2lite", 4, 1.0, "tc-decode"),       # 4..64 tokens: tensor-core decode GEMM
    ("dsv2lite", 8, 1.0, "tc-decode"),
    ("mixtral", 32, 1.0, "tc-decode"),
    ("granite", 64, 1.0, "tc-decode"),
    ("granite", 65, 1.0, "tc-prefill"),      # > 64 tokens: grouped tensor-core GEMM
    ("qwen2", 4096, 1.0, "tc-prefill"),
    ("mixtral", 8, 0.1, "gemv-floe"),        # FloE sparsity on the GEMV
    ("mixtral", 128, 0.1, "unsupported"),    # FloE is decode-only
    ("tiny", 16, 0.5, "unsupported"),        # ... and bf16-only
    ("dsv2lite", 8, 0.0, "unsupported"),     # keep_frac outside (0, 1]
])
def test_expert_ffn_path_choice(name, T, keep, path):
    assert moe.moe_expert_ffn_path(_dims(name, T), keep) == path


def test_prefetch_min_depth_closed_form():
    """SPICE's minimum prefetch depth ceil(W_e / (B * T_layer)), on values
    whose quotients are exact in binary floating point."""
    f = moe.moe_prefetch_min_depth
    assert f(2.0 ** 31, 2.0 ** 30, 0.5) == 4          # exactly 4
    assert f(2.0 ** 31 + 2.0 ** 12, 2.0 ** 30, 0.5) == 5  # 4 + 2^-17: above 4
    assert f(0.0, 1e9, 1e-3) == 0
    assert f(3 * 17_301_504 * 2 / 2, 32e9, 1e-3) == 2  # 51.9 MB over 32 GB/s in 1 ms: 1.62 -> 2
    # a quotient one rounding away from an integer counts as that integer
    assert f(64e6, 32e9, 2e-3) == 1
    for bad in ((-1.0, 1e9, 1e-3), (1.0, 0.0, 1e-3), (1.0, 1e9, 0.0), (1e30, 1.0, 1e-9)):
        with pytest.raises(ValueError):
            f(*bad)


def test_prefetch_depth_rejects_bad_arguments_before_cuda():
    """n_ahead outside 1..MOE_MAX_AHEAD, a negative d_min, a non-finite tau or
    a missing router are argument errors found before any CUDA call."""
    L = moe.lib()
    D = _raw_dims(T=4, d=256, N=8, k=2, I=64)
    n = moe.moe_workspace_size(D)
    fake_ws = C.c_void_p(1 << 20)
    x = C.c_void_p(0x1000)
    w = (C.c_void_p * 17)(*([0x2000] * 17))
    out = C.c_void_p(0x3000)
    call = lambda J, tau, d_min, warr=w, xx=x: L.moe_prefetch_depth(
        C.byref(D), J, xx, warr, None, C.c_float(tau), d_min, out, out, out, out, out, fake_ws, n, None)
    assert call(0, 0.9, 0) == moe.MOE_ERR_INVALID_ARG
    assert call(17, 0.9, 0) == moe.MOE_ERR_INVALID_ARG
    assert call(2, 0.9, -1) == moe.MOE_ERR_INVALID_ARG
    assert call(2, float("nan"), 0) == moe.MOE_ERR_INVALID_ARG
    assert call(2, 0.9, 0, warr=(C.c_void_p * 2)(0x2000, None)) == moe.MOE_ERR_INVALID_ARG
    assert call(2, 0.9, 0, warr=(C.c_void_p * 2)(0x2000, 0x2004)) == moe.MOE_ERR_INVALID_ARG
    assert call(2, 0.9, 0, xx=None) == moe.MOE_ERR_INVALID_ARG
    D64 = _raw_dims(T=4, d=256, N=65, k=2, I=64)
    assert L.moe_prefetch_depth(C.byref(D64), 2, x, w, None, C.c_float(0.9), 0, out, out, out, out, out,
                                fake_ws, n, None) == moe.MOE_ERR_UNSUPPORTED


def test_bitslice_rejects_bad_arguments_before_cuda():
    """Bit-sliced weights: bits outside 1..8, widths that are not multiples of
    32, a too-small scratch, an unsupported width and a NULL buffer are
    reported before any CUDA call; an empty batch is a no-op."""
    L = moe.lib()
    p = C.c_void_p(0x1000)
    bf16 = moe.MOE_DTYPE_BF16
    ok_scratch = moe.moe_bitslice_scratch_size(256, 512, 2, 3)
    assert ok_scratch == 2 * 3 * (512 + 256) * 4 + 2 * (256 // 16) * 4
    assert moe.moe_bitslice_scratch_size(256, 512, 2, 0) == 0

    def ffn(d=256, I=512, N=4, ns=1, bits=4, T=2, k=2, scratch=ok_scratch, x=p):
        return L.moe_bitslice_ffn(d, I, N, ns, bits, bf16, x, T, k, p, None, p, p, p, p, p, p, 0, p, p, scratch, None)

    assert ffn(bits=0) == moe.MOE_ERR_INVALID_ARG
    assert ffn(bits=9) == moe.MOE_ERR_INVALID_ARG
    assert ffn(d=250) == moe.MOE_ERR_INVALID_ARG
    assert ffn(I=500) == moe.MOE_ERR_INVALID_ARG
    assert ffn(d=4128) == moe.MOE_ERR_UNSUPPORTED
    assert ffn(I=4128) == moe.MOE_ERR_UNSUPPORTED
    assert ffn(T=30000, k=2, ns=1, scratch=1 << 40) == moe.MOE_ERR_UNSUPPORTED  # 90000 (token, slot) pairs
    assert ffn(scratch=ok_scratch - 4) == moe.MOE_ERR_CAPACITY
    assert ffn(x=None) == moe.MOE_ERR_INVALID_ARG
    assert ffn(x=C.c_void_p(0x1004)) == moe.MOE_ERR_INVALID_ARG  # misaligned
    assert ffn(T=0, x=None) == moe.MOE_OK
    # packing: the packed width must be a multiple of 32
    assert L.moe_bitslice_pack(64, 100, bf16, p, 0, p, p, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_bitslice_pack(100, 64, bf16, p, 1, p, p, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_bitslice_pack(64, 96, 7, p, 0, p, p, None) == moe.MOE_ERR_UNSUPPORTED
    assert L.moe_bitslice_pack(64, 96, bf16, None, 0, p, p, None) == moe.MOE_ERR_INVALID_ARG
