"""Python binding of the GB300 MoE-layer C ABI (include/moe.h).

Argument marshalling only: every function below checks tensor dtype, device,
contiguity and size, then calls the C function of the same name in
libmoe_gb300.so, where every step of the layer runs as a CUDA kernel.  There
is no Python or CPU implementation of any step: if the library is missing the
calls raise.

Tensors are torch tensors on the current CUDA device.  uint64 expert masks
are carried in int64 tensors (same bits).  `stream` defaults to torch's
current stream.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_gb300.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CAPACITY = 0, 1, 2, 3
MOE_ERR_CUDA, MOE_ERR_STAGING, MOE_ERR_TIMEOUT, MOE_ERR_DEVICE_INDEX = 4, 5, 6, 7
MOE_DTYPE_F32, MOE_DTYPE_BF16 = 0, 1
MOE_MISS_EXACT, MOE_MISS_SUBSTITUTE, MOE_MISS_LORE, MOE_MISS_HYBRID, MOE_MISS_HETERO = 0, 1, 2, 3, 4
MOE_KIND_COMPUTE, MOE_KIND_FETCH, MOE_KIND_LORE, MOE_KIND_CPU = 0, 1, 2, 3
(MOE_CNT_HIT, MOE_CNT_SUBSTITUTE, MOE_CNT_LORE, MOE_CNT_FETCH, MOE_CNT_OVERLAP, MOE_CNT_DELTA_HAT,
 MOE_CNT_DELTA_STAR, MOE_CNT_SHORTFALL, MOE_CNT_CPU) = range(9)
MOE_NUM_COUNTERS = 9
COUNTER_NAMES = ["hit", "substitute", "lore", "fetch", "overlap", "delta_hat_sum",
                 "delta_star_sum", "shortfall", "cpu"]


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        extra = ""
        if status == MOE_ERR_CUDA:
            extra = " — " + lib().moe_last_error_detail().decode()
        super().__init__(f"{where}: {status_string(status)} (status {status}){extra}")


class moe_dims(C.Structure):
    _fields_ = [(n, C.c_int) for n in ("T", "d", "N", "k", "I", "n_shared", "I_shared", "r",
                                       "delta_max", "wtype", "renorm_topk")]

    def with_T(self, T: int) -> "moe_dims":
        d = moe_dims()
        C.pointer(d)[0] = self
        d.T = T
        return d


_VP = C.c_void_p


class moe_layer_args(C.Structure):
    _fields_ = [("x", _VP), ("x_pre", _VP), ("w_router", _VP), ("router_bias", _VP),
                ("w_prefetch", _VP), ("w_ord", _VP), ("theta", _VP), ("tau", C.c_float),
                ("n_resident", C.c_int), ("resident", _VP), ("use_prefetch_mask", C.c_int),
                ("policy", C.c_int), ("gamma", C.c_float), ("keep_frac", C.c_float),
                ("table", _VP), ("lore_a", _VP), ("lore_b", _VP)]


class moe_layer_outputs(C.Structure):
    _fields_ = [(n, _VP) for n in (
        "topk_idx", "topk_gate", "router_prob", "delta_hat", "prefetch_mask", "delta_star",
        "batch_resident", "final_idx", "final_gate", "final_kind", "fetch_mask", "counters",
        "expert_offsets", "perm", "inv_perm", "y_perm", "y_shared", "y_lore", "out")]


class moe_hetero_cost(C.Structure):
    """SPICE's per-miss cost model: link bytes/s, expert bytes, GPU seconds of
    one expert, host seconds per token row of one expert, hidden-state bytes."""
    _fields_ = [(n, C.c_double) for n in ("link_bytes_per_s", "expert_bytes", "gpu_expert_s", "cpu_row_s",
                                          "hidden_bytes")]


class moe_hetero_host(C.Structure):
    _fields_ = [("x", _VP), ("final_idx", _VP), ("final_kind", _VP), ("masks", _VP), ("y_rows", _VP),
                ("scratch", _VP), ("scratch_bytes", C.c_size_t)]


class moe_hetero_stats(C.Structure):
    _fields_ = [("cpu_slots", C.c_int32), ("fetch_experts", C.c_int32), ("fetch_min_rows", C.c_int32),
                ("lore_slots", C.c_int32), ("fetch_bytes", C.c_double), ("cpu_link_bytes", C.c_double),
                ("host_ms", C.c_double), ("wait_ms", C.c_double)]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


MOE_CACHE_RING, MOE_CACHE_FLIGHTS = 16, 8


class moe_cache_pipe(C.Structure):
    """State of the overlapped expert-cache pipeline (include/moe.h)."""
    _fields_ = [("capacity", C.c_int), ("decay", C.c_float), ("max_flight_experts", C.c_int),
                ("host_ring", _VP), ("step_events", _VP * MOE_CACHE_RING), ("copy_events", _VP * MOE_CACHE_FLIGHTS),
                ("dev_masks", _VP), ("dev_heat", _VP), ("dev_stats", _VP),
                ("step", C.c_longlong), ("consumed", C.c_longlong), ("landed", C.c_uint64), ("in_flight", C.c_uint64),
                ("flight_mask", C.c_uint64 * MOE_CACHE_FLIGHTS),
                ("staged_experts", C.c_longlong), ("staged_bytes", C.c_longlong), ("in_time_experts", C.c_longlong),
                ("stall_experts", C.c_longlong), ("stall_steps", C.c_longlong), ("dev_ring", _VP)]


_lib = None
_lock = threading.Lock()

# argument type codes for the C prototypes
_P, _I, _F, _U64, _SZ = _VP, C.c_int, C.c_float, C.c_uint64, C.c_size_t
_DIMS = C.POINTER(moe_dims)
_PROTOS = {
    "moe_status_string": ([C.c_int], C.c_char_p),
    "moe_launch_total": ([], C.c_uint64),
    "moe_expert_ffn_path": ([C.POINTER(moe_dims), C.c_float], C.c_char_p),
    "moe_last_error_detail": ([], C.c_char_p),
    "moe_workspace_size": ([_DIMS, C.POINTER(C.c_size_t)], C.c_int),
    "moe_expert_table_size": ([_DIMS, C.POINTER(C.c_size_t)], C.c_int),
    "moe_expert_table_init": ([_DIMS, _P, _P, _P, _P, _P, _P, _P, _SZ, _P], C.c_int),
    "moe_route": ([_DIMS, _P, _P, _P, _P, _P, _P, _P, _F, _I, _P, _P, _P, _P, _P, _P, _P, _P, _SZ,
                   _P], C.c_int),
    "moe_select_resident": ([_DIMS, _P, _P, _P, _P, _I, _F, _P, _P, _P, _P, _P, _P, _P, _P, _SZ,
                             _P], C.c_int),
    "moe_stage_experts": ([_DIMS, _U64, _P, _P, _P, _P, _P, _P, _P, _P, C.POINTER(C.c_size_t)],
                          C.c_int),
    "moe_permute": ([_DIMS, _P, _P, _P, _P, _P, _P, _SZ, _P], C.c_int),
    "moe_expert_ffn": ([_DIMS, _P, _P, _P, _P, _F, _P, _P, _P, _SZ, _P], C.c_int),
    "moe_floe_kept_mask": ([_DIMS, _P, _SZ, C.POINTER(C.c_void_p), C.POINTER(C.c_int32)], C.c_int),
    "moe_expert_ffn_noalloc": ([_DIMS, _P, _P, _P, _P, _P, _P, _P, _P], C.c_int),
    "moe_lore": ([_DIMS, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P], C.c_int),
    "moe_combine": ([_DIMS, _P, _P, _P, _P, _P, _P, _P, _P], C.c_int),
    "moe_bitslice_pack": ([C.c_int, C.c_int, C.c_int, _P, C.c_int, _P, _P, _P], C.c_int),
    "moe_bitslice_scratch_size": ([C.c_int, C.c_int, C.c_int, C.c_int], C.c_size_t),
    "moe_bitslice_ffn": ([C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, _P, C.c_int, C.c_int, _P, _P, _P, _P,
                          _P, _P,
                          _P, _P, C.c_int, _P, _P, _SZ, _P], C.c_int),
    "moe_prefetch_depth": ([_DIMS, C.c_int, _P, C.POINTER(C.c_void_p), C.POINTER(C.c_void_p), C.c_float, C.c_int,
                            _P, _P, _P, _P, _P, _P, _SZ, _P], C.c_int),
    "moe_prefetch_min_depth": ([C.c_double, C.c_double, C.c_double], C.c_int),
    "moe_cache_update": ([_DIMS, _P, C.c_float, C.c_int, _P, _P, _P, _P, _P], C.c_int),
    "moe_layer_forward": ([_DIMS, C.POINTER(moe_layer_args), C.POINTER(moe_layer_outputs), _P, _SZ,
                           _P], C.c_int),
    "moe_check": ([_P, _P, C.POINTER(C.c_int), C.POINTER(C.c_int32)], C.c_int),
    "moe_hetero_fetch_min_rows": ([C.POINTER(moe_hetero_cost)], C.c_int),
    "moe_set_graph_replay": ([C.c_int], None),
    "moe_layer_forward_host": ([_DIMS, C.POINTER(moe_layer_args), C.POINTER(moe_layer_outputs), _P, _P, _P, _SZ, _P],
                               C.c_int),
    "moe_cache_start": ([_DIMS, C.POINTER(moe_cache_pipe), _U64, _P], C.c_int),
    "moe_cache_step": ([_DIMS, C.POINTER(moe_layer_args), C.POINTER(moe_layer_outputs), C.POINTER(moe_cache_pipe),
                        _P, _P, _P, _P, _P, _P, _P, _SZ, _P, _P], C.c_int),
    "moe_cache_drain": ([_DIMS, C.POINTER(moe_cache_pipe), _P, _P, _P, _P, _P, _P, _P], C.c_int),
    "moe_select_hetero": ([_DIMS, _P, _P, _P, _P, _F, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P],
                          C.c_int),
    "moe_cpu_experts_scratch_size": ([_DIMS], C.c_size_t),
    "moe_cpu_experts": ([_DIMS, _P, _P, _P, _P, _P, _P, _I, _P, _P, _SZ, C.POINTER(C.c_int32),
                         C.POINTER(C.c_int32)], C.c_int),
    "moe_layer_forward_hetero": ([_DIMS, C.POINTER(moe_layer_args), C.POINTER(moe_layer_outputs),
                                  C.POINTER(moe_hetero_cost), _P, _P, _P, _P, _P, _P, C.POINTER(moe_hetero_host),
                                  _I, _P, _SZ, _P, _P, _P, C.POINTER(moe_hetero_stats)], C.c_int),
    "moe_testing_fail_copies_after": ([C.c_int], None),
    "moe_testing_wait_timeout": ([C.c_void_p, C.c_size_t, C.c_void_p], C.c_int),
    "moe_testing_set_tc_pairs": ([C.c_int], None),
}


def lib():
    """Load libmoe_gb300.so (built by build.py / __graft_entry__.build())."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build the CUDA library first "
                                   "(python -m expert_routing_ffn_gb300.build)")
            L = C.CDLL(LIB_PATH)
            for name, (args, res) in _PROTOS.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = res
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().moe_status_string(status).decode()


def _check(status: int, where: str):
    if status != MOE_OK:
        raise MoeError(status, where)


def _stream(stream):
    if stream is None:
        return C.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return C.c_void_p(stream.cuda_stream)
    return C.c_void_p(int(stream))


def _ptr(t, dtype=None, numel=None, name="tensor", optional=False):
    """Device pointer of a contiguous CUDA tensor (None -> NULL if optional)."""
    if t is None:
        if optional:
            return None
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{name} has {t.numel()} elements, needs {numel}")
    return C.c_void_p(t.data_ptr())


def wdtype(dims: moe_dims):
    return torch.bfloat16 if dims.wtype == MOE_DTYPE_BF16 else torch.float32


def make_dims(T, d, N, k, I, n_shared=0, I_shared=0, r=0, delta_max=None, wtype="bf16",
              renorm_topk=0) -> moe_dims:
    D = moe_dims()
    D.T, D.d, D.N, D.k, D.I = T, d, N, k, I
    D.n_shared, D.I_shared, D.r = n_shared, I_shared, r
    D.delta_max = N - k if delta_max is None else delta_max
    D.wtype = MOE_DTYPE_BF16 if wtype in ("bf16", MOE_DTYPE_BF16) else MOE_DTYPE_F32
    D.renorm_topk = renorm_topk
    return D


def moe_launch_total() -> int:
    return int(lib().moe_launch_total())


def moe_expert_ffn_path(dims: moe_dims, keep_frac: float = 1.0) -> str:
    """Which kernels moe_expert_ffn runs for these dimensions (no device work)."""
    return lib().moe_expert_ffn_path(C.byref(dims), float(keep_frac)).decode()


def moe_workspace_size(dims: moe_dims) -> int:
    n = C.c_size_t()
    _check(lib().moe_workspace_size(C.byref(dims), C.byref(n)), "moe_workspace_size")
    return n.value


def moe_expert_table_size(dims: moe_dims) -> int:
    n = C.c_size_t()
    _check(lib().moe_expert_table_size(C.byref(dims), C.byref(n)), "moe_expert_table_size")
    return n.value


def _ptr_array(tensors, name):
    arr = (C.c_void_p * len(tensors))()
    for i, t in enumerate(tensors):
        arr[i] = _ptr(t, name=f"{name}[{i}]").value
    return arr


def moe_expert_table_init(dims, w_gate, w_up, w_down, sh_gate, sh_up, sh_down, table, stream=None):
    """w_*: sequences of N device tensors [I, d]; sh_*: n_shared tensors [I_shared, d]."""
    keep = [_ptr_array(w_gate, "w_gate"), _ptr_array(w_up, "w_up"), _ptr_array(w_down, "w_down")]
    sh = [_ptr_array(s, n) if dims.n_shared else None for s, n in
          ((sh_gate, "sh_gate"), (sh_up, "sh_up"), (sh_down, "sh_down"))]
    _check(lib().moe_expert_table_init(
        C.byref(dims), *[C.cast(a, C.c_void_p) for a in keep],
        *[C.cast(a, C.c_void_p) if a is not None else None for a in sh],
        _ptr(table, torch.uint8, name="table"), table.numel(), _stream(stream)),
        "moe_expert_table_init")


def moe_route(dims, x, w_router, router_bias, x_pre, w_prefetch, w_ord, theta, tau, n_resident,
              topk_idx, topk_gate, router_prob, delta_hat, prefetch_mask, delta_star,
              batch_resident, ws, stream=None):
    T, d, N, k = dims.T, dims.d, dims.N, dims.k
    wt = wdtype(dims)
    _check(lib().moe_route(
        C.byref(dims), _ptr(x, wt, T * d, "x"), _ptr(w_router, wt, N * d, "w_router"),
        _ptr(router_bias, torch.float32, N, "router_bias", True),
        _ptr(x_pre, wt, T * d, "x_pre", True), _ptr(w_prefetch, wt, N * d, "w_prefetch", True),
        _ptr(w_ord, torch.float32, d, "w_ord", True),
        _ptr(theta, torch.float32, dims.delta_max + 1, "theta", True), float(tau), int(n_resident),
        _ptr(topk_idx, torch.int32, T * k, "topk_idx"), _ptr(topk_gate, torch.float32, T * k, "topk_gate"),
        _ptr(router_prob, torch.float32, T * N, "router_prob"), _ptr(delta_hat, torch.int32, T, "delta_hat"),
        _ptr(prefetch_mask, torch.int64, T, "prefetch_mask"),
        _ptr(delta_star, torch.int32, T, "delta_star", True),
        _ptr(batch_resident, torch.int64, 1, "batch_resident", True),
        _ptr(ws, torch.uint8, name="ws"), ws.numel(), _stream(stream)), "moe_route")


def moe_select_resident(dims, router_prob, topk_idx, prefetch_mask, resident, policy, gamma,
                        delta_hat, delta_star, final_idx, final_gate, final_kind, fetch_mask,
                        counters, ws, stream=None):
    T, N, k = dims.T, dims.N, dims.k
    _check(lib().moe_select_resident(
        C.byref(dims), _ptr(router_prob, torch.float32, T * N, "router_prob"),
        _ptr(topk_idx, torch.int32, T * k, "topk_idx"),
        _ptr(prefetch_mask, torch.int64, T, "prefetch_mask", True),
        _ptr(resident, torch.int64, 1, "resident", True), int(policy), float(gamma),
        _ptr(delta_hat, torch.int32, T, "delta_hat", True),
        _ptr(delta_star, torch.int32, T, "delta_star", True),
        _ptr(final_idx, torch.int32, T * k, "final_idx"), _ptr(final_gate, torch.float32, T * k, "final_gate"),
        _ptr(final_kind, torch.int32, T * k, "final_kind"),
        _ptr(fetch_mask, torch.int64, 1, "fetch_mask", True),
        _ptr(counters, torch.int32, MOE_NUM_COUNTERS, "counters", True),
        _ptr(ws, torch.uint8, name="ws"), ws.numel(), _stream(stream)), "moe_select_resident")


def moe_prefetch_depth(dims, x, w_routers, biases, tau, d_min, logits, conf, depth, token_masks, layer_masks,
                       ws, stream=None):
    """Confidence-aware prefetch depth over len(w_routers) look-ahead layers
    (SPICE, confidence-aware adaptive prefetch).  w_routers: device tensors
    [N, d] in the layer's weight type; biases: None or a sequence of [N]
    float32 tensors / None.  Outputs: logits [J, T, N] float32, conf [T, J]
    float32, depth [T] int32, token_masks [T, J] and layer_masks [J] int64
    (uint64 bit patterns)."""
    T, d, N = dims.T, dims.d, dims.N
    J = len(w_routers)
    wt = wdtype(dims)
    warr = (C.c_void_p * J)(*[_ptr(w, wt, N * d, f"w_routers[{j}]").value for j, w in enumerate(w_routers)])
    barr = None
    if biases is not None:
        barr = (C.c_void_p * J)(*[(_ptr(b, torch.float32, N, f"biases[{j}]", True) or C.c_void_p()).value
                                  for j, b in enumerate(biases)])
    _check(lib().moe_prefetch_depth(
        C.byref(dims), J, _ptr(x, wt, T * d, "x", T == 0), warr, barr, float(tau), int(d_min),
        _ptr(logits, torch.float32, J * T * N, "logits", T == 0), _ptr(conf, torch.float32, T * J, "conf", T == 0),
        _ptr(depth, torch.int32, T, "depth", T == 0), _ptr(token_masks, torch.int64, T * J, "token_masks", T == 0),
        _ptr(layer_masks, torch.int64, J, "layer_masks"), _ptr(ws, torch.uint8, name="ws"), ws.numel(),
        _stream(stream)), "moe_prefetch_depth")


def moe_bitslice_pack(w, transpose, planes, scales, stream=None):
    """Pack one weight matrix w [rows, cols] (bf16 or float32 CUDA tensor), or
    its transpose, into 8 bit planes: planes int32 [8 * R * C / 32] (uint32
    bit patterns), scales float32 [R]."""
    rows, cols = w.shape
    R, Cc = (cols, rows) if transpose else (rows, cols)
    wt = MOE_DTYPE_BF16 if w.dtype == torch.bfloat16 else MOE_DTYPE_F32
    _check(lib().moe_bitslice_pack(rows, cols, wt, _ptr(w, (torch.bfloat16, torch.float32), rows * cols, "w"),
                                   int(bool(transpose)), _ptr(planes, torch.int32, 8 * R * Cc // 32, "planes"),
                                   _ptr(scales, torch.float32, R, "scales"), _stream(stream)), "moe_bitslice_pack")


def moe_bitslice_scratch_size(d, I, T, slots) -> int:
    return int(lib().moe_bitslice_scratch_size(int(d), int(I), int(T), int(slots)))


def moe_bitslice_ffn(d, I, N, bits, x, idx, gate, planes_gate, scales_gate, planes_up, scales_up, planes_down,
                     scales_down, y, scratch, accumulate=False, n_shared=0, stream=None):
    """Draft FFN with b-bit weights: y[t] (+)= sum_s gate[t,s] FFN_b(idx[t,s], x_t)
    + sum_i FFN_b(N + i, x_t) over the n_shared shared experts.  x [T, d] bf16
    or float32; idx [T, k] int32; gate [T, k] float32 or None; planes / scales
    as written by moe_bitslice_pack for the N routed then the n_shared shared
    experts back to back (down projection packed transposed); y [T, d]
    float32; scratch uint8."""
    T, k = idx.shape
    xt = MOE_DTYPE_BF16 if x.dtype == torch.bfloat16 else MOE_DTYPE_F32
    w8 = lambda R, Cc: 8 * (N + n_shared) * R * Cc // 32
    NS = N + n_shared
    _check(lib().moe_bitslice_ffn(
        int(d), int(I), int(N), int(n_shared), int(bits), xt, _ptr(x, (torch.bfloat16, torch.float32), T * d, "x", T == 0), T, k,
        _ptr(idx, torch.int32, T * k, "idx", T == 0), _ptr(gate, torch.float32, T * k, "gate", True),
        _ptr(planes_gate, torch.int32, w8(I, d), "planes_gate"), _ptr(scales_gate, torch.float32, NS * I, "scales_gate"),
        _ptr(planes_up, torch.int32, w8(I, d), "planes_up"), _ptr(scales_up, torch.float32, NS * I, "scales_up"),
        _ptr(planes_down, torch.int32, w8(d, I), "planes_down"),
        _ptr(scales_down, torch.float32, NS * d, "scales_down"), int(bool(accumulate)),
        _ptr(y, torch.float32, T * d, "y", T == 0), _ptr(scratch, torch.uint8, name="scratch"), scratch.numel(),
        _stream(stream)), "moe_bitslice_ffn")


def moe_prefetch_min_depth(expert_bytes: float, link_bytes_per_s: float, layer_seconds: float) -> int:
    """ceil(expert_bytes / (link bandwidth * layer time)) (SPICE's minimum
    prefetch depth); host only."""
    v = lib().moe_prefetch_min_depth(float(expert_bytes), float(link_bytes_per_s), float(layer_seconds))
    if v < 0:
        raise ValueError("moe_prefetch_min_depth: bad size, bandwidth or layer time")
    return int(v)


def moe_stage_experts(dims, host_fetch_mask: int, host_w_gate, host_w_up, host_w_down,
                      dev_w_gate, dev_w_up, dev_w_down, stage_stream, done_event) -> int:
    """host_w_*: sequences of N pinned CPU tensors; dev_w_*: N device tensors."""
    def arr(ts, name, pinned):
        a = (C.c_void_p * len(ts))()
        for i, t in enumerate(ts):
            if pinned and not t.is_pinned():
                raise ValueError(f"{name}[{i}] must be pinned host memory")
            a[i] = t.data_ptr()
        return a
    a = [arr(host_w_gate, "host_w_gate", True), arr(host_w_up, "host_w_up", True),
         arr(host_w_down, "host_w_down", True), arr(dev_w_gate, "dev_w_gate", False),
         arr(dev_w_up, "dev_w_up", False), arr(dev_w_down, "dev_w_down", False)]
    if done_event.cuda_event == 0:  # torch creates the CUDA event on its first record
        done_event.record(stage_stream)
    n = C.c_size_t()
    _check(lib().moe_stage_experts(C.byref(dims), C.c_uint64(host_fetch_mask & (2**64 - 1)),
                                   *[C.cast(x, C.c_void_p) for x in a], _stream(stage_stream),
                                   C.c_void_p(done_event.cuda_event), C.byref(n)),
           "moe_stage_experts")
    return n.value


def moe_permute(dims, final_idx, final_kind, expert_offsets, perm, inv_perm, ws, stream=None):
    T, N, k = dims.T, dims.N, dims.k
    _check(lib().moe_permute(
        C.byref(dims), _ptr(final_idx, torch.int32, T * k, "final_idx"),
        _ptr(final_kind, torch.int32, T * k, "final_kind"),
        _ptr(expert_offsets, torch.int32, N + 1, "expert_offsets"), _ptr(perm, torch.int32, T * k, "perm"),
        _ptr(inv_perm, torch.int32, T * k, "inv_perm"), _ptr(ws, torch.uint8, name="ws"), ws.numel(),
        _stream(stream)), "moe_permute")


def moe_expert_ffn(dims, x, table, expert_offsets, perm, keep_frac, y_perm, y_shared, ws,
                   stream=None):
    T, d, N, k = dims.T, dims.d, dims.N, dims.k
    _check(lib().moe_expert_ffn(
        C.byref(dims), _ptr(x, wdtype(dims), T * d, "x"), _ptr(table, torch.uint8, name="table"),
        _ptr(expert_offsets, torch.int32, N + 1, "expert_offsets"), _ptr(perm, torch.int32, T * k, "perm"),
        float(keep_frac), _ptr(y_perm, torch.float32, T * k * d, "y_perm"),
        _ptr(y_shared, torch.float32, T * d, "y_shared", True), _ptr(ws, torch.uint8, name="ws"),
        ws.numel(), _stream(stream)), "moe_expert_ffn")


def moe_floe_kept_mask(dims, ws):
    """Device pointer and words per row of the FloE kept-channel bitsets left
    in `ws` by the last moe_expert_ffn call with keep_frac < 1."""
    ptr = C.c_void_p()
    words = C.c_int32()
    _check(lib().moe_floe_kept_mask(C.byref(dims), _ptr(ws, torch.uint8, name="ws"), ws.numel(),
                                    C.byref(ptr), C.byref(words)), "moe_floe_kept_mask")
    return ptr.value, words.value


def moe_expert_ffn_noalloc(dims, x, table, expert_offsets, perm, y_perm, y_shared,
                           device_status=None, stream=None):
    """moe_expert_ffn with the library's fixed device scratch instead of a
    workspace, for callers that cannot allocate device memory at run time."""
    T, d, N, k = dims.T, dims.d, dims.N, dims.k
    _check(lib().moe_expert_ffn_noalloc(
        C.byref(dims), _ptr(x, wdtype(dims), T * d, "x"), _ptr(table, torch.uint8, name="table"),
        _ptr(expert_offsets, torch.int32, N + 1, "expert_offsets"), _ptr(perm, torch.int32, T * k, "perm"),
        _ptr(y_perm, torch.float32, T * k * d, "y_perm"),
        _ptr(y_shared, torch.float32, T * d, "y_shared", True),
        _ptr(device_status, torch.int32, 2, "device_status", True), _stream(stream)),
        "moe_expert_ffn_noalloc")


def moe_lore(dims, x, final_idx, final_kind, final_gate, lore_a, lore_b, y_lore, ws, stream=None):
    T, d, N, k, r = dims.T, dims.d, dims.N, dims.k, dims.r
    wt = wdtype(dims)
    _check(lib().moe_lore(
        C.byref(dims), _ptr(x, wt, T * d, "x"), _ptr(final_idx, torch.int32, T * k, "final_idx"),
        _ptr(final_kind, torch.int32, T * k, "final_kind"), _ptr(final_gate, torch.float32, T * k, "final_gate"),
        _ptr(lore_a, wt, N * r * d, "lore_a"), _ptr(lore_b, wt, N * d * r, "lore_b"),
        _ptr(y_lore, torch.float32, T * d, "y_lore"), _ptr(ws, torch.uint8, name="ws"), ws.numel(),
        _stream(stream)), "moe_lore")


def moe_combine(dims, y_perm, inv_perm, final_gate, final_kind, y_shared, y_lore, out, stream=None):
    T, d, k = dims.T, dims.d, dims.k
    _check(lib().moe_combine(
        C.byref(dims), _ptr(y_perm, torch.float32, T * k * d, "y_perm"),
        _ptr(inv_perm, torch.int32, T * k, "inv_perm"), _ptr(final_gate, torch.float32, T * k, "final_gate"),
        _ptr(final_kind, torch.int32, T * k, "final_kind"),
        _ptr(y_shared, torch.float32, T * d, "y_shared", True),
        _ptr(y_lore, torch.float32, T * d, "y_lore", True), _ptr(out, torch.float32, T * d, "out"),
        _stream(stream)), "moe_combine")


def moe_cache_update(dims, topk_idx, decay, capacity, heat, cache_mask, admit_mask=None, stats=None,
                     stream=None):
    T, N, k = dims.T, dims.N, dims.k
    _check(lib().moe_cache_update(
        C.byref(dims), _ptr(topk_idx, torch.int32, T * k, "topk_idx"), float(decay), int(capacity),
        _ptr(heat, torch.float32, N, "heat"), _ptr(cache_mask, torch.int64, 1, "cache_mask"),
        _ptr(admit_mask, torch.int64, 1, "admit_mask", True), _ptr(stats, torch.int32, 4, "stats", True),
        _stream(stream)), "moe_cache_update")


def moe_layer_forward(dims, args: moe_layer_args, outs: moe_layer_outputs, ws, stream=None):
    _check(lib().moe_layer_forward(C.byref(dims), C.byref(args), C.byref(outs),
                                   _ptr(ws, torch.uint8, name="ws"), ws.numel(), _stream(stream)),
           "moe_layer_forward")


def hetero_cost(link_bytes_per_s, expert_bytes, gpu_expert_s, cpu_row_s, hidden_bytes) -> moe_hetero_cost:
    c = moe_hetero_cost()
    c.link_bytes_per_s, c.expert_bytes, c.gpu_expert_s = link_bytes_per_s, expert_bytes, gpu_expert_s
    c.cpu_row_s, c.hidden_bytes = cpu_row_s, hidden_bytes
    return c


def moe_hetero_fetch_min_rows(cost: moe_hetero_cost) -> int:
    """The smallest number of a missing expert's token rows for which
    fetching it beats computing it on the host (SPICE's cost model)."""
    v = lib().moe_hetero_fetch_min_rows(C.byref(cost))
    if v < 0:
        raise ValueError("moe_hetero_fetch_min_rows: bad cost model")
    return int(v)


def moe_select_hetero(dims, router_prob, topk_idx, prefetch_mask, resident, gamma, fetch_min_rows, delta_hat,
                      delta_star, final_idx, final_gate, final_kind, perm, inv_perm, fetch_mask, cpu_mask,
                      counters, ws, stream=None):
    T, N, k = dims.T, dims.N, dims.k
    _check(lib().moe_select_hetero(
        C.byref(dims), _ptr(router_prob, torch.float32, T * N, "router_prob"),
        _ptr(topk_idx, torch.int32, T * k, "topk_idx"),
        _ptr(prefetch_mask, torch.int64, T, "prefetch_mask", True),
        _ptr(resident, torch.int64, 1, "resident", True), float(gamma), int(fetch_min_rows),
        _ptr(delta_hat, torch.int32, T, "delta_hat", True), _ptr(delta_star, torch.int32, T, "delta_star", True),
        _ptr(final_idx, torch.int32, T * k, "final_idx"), _ptr(final_gate, torch.float32, T * k, "final_gate"),
        _ptr(final_kind, torch.int32, T * k, "final_kind"), _ptr(perm, torch.int32, T * k, "perm"),
        _ptr(inv_perm, torch.int32, T * k, "inv_perm"), _ptr(fetch_mask, torch.int64, 1, "fetch_mask", True),
        _ptr(cpu_mask, torch.int64, 1, "cpu_mask", True),
        _ptr(counters, torch.int32, MOE_NUM_COUNTERS, "counters", True),
        _ptr(ws, torch.uint8, name="ws"), ws.numel(), _stream(stream)), "moe_select_hetero")


def moe_cpu_experts_scratch_size(dims) -> int:
    return int(lib().moe_cpu_experts_scratch_size(C.byref(dims)))


def _host_ptr(t, dtype, numel, name):
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise TypeError(f"{name} must be a host (CPU) tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if t.numel() < numel:
        raise ValueError(f"{name} has {t.numel()} elements, needs {numel}")
    return C.c_void_p(t.data_ptr())


def _host_array(ts, name):
    a = (C.c_void_p * len(ts))()
    for i, t in enumerate(ts):
        if t is None:
            continue
        if t.is_cuda:
            raise TypeError(f"{name}[{i}] must be host memory")
        a[i] = t.data_ptr()
    return a


def moe_cpu_experts(dims, host_x, host_final_idx, host_final_kind, host_w_gate, host_w_up, host_w_down, host_y_rows,
                    scratch, n_threads=0):
    """The host slots' expert FFN on the host cores (all host tensors):
    returns (rows computed, y_perm row of the first)."""
    T, d, k = dims.T, dims.d, dims.k
    n_rows, first = C.c_int32(), C.c_int32()
    arrs = [_host_array(w, n) for w, n in ((host_w_gate, "host_w_gate"), (host_w_up, "host_w_up"),
                                            (host_w_down, "host_w_down"))]
    _check(lib().moe_cpu_experts(
        C.byref(dims), _host_ptr(host_x, wdtype(dims), T * d, "host_x"),
        _host_ptr(host_final_idx, torch.int32, T * k, "host_final_idx"),
        _host_ptr(host_final_kind, torch.int32, T * k, "host_final_kind"),
        *[C.cast(a, C.c_void_p) for a in arrs], int(n_threads),
        _host_ptr(host_y_rows, torch.float32, T * k * d, "host_y_rows"),
        _host_ptr(scratch, torch.uint8, 0, "scratch"), scratch.numel(), C.byref(n_rows), C.byref(first)),
        "moe_cpu_experts")
    return n_rows.value, first.value


def moe_layer_forward_hetero(dims, args: moe_layer_args, outs: moe_layer_outputs, cost: moe_hetero_cost,
                             host_w_gate, host_w_up, host_w_down, dev_w_gate, dev_w_up, dev_w_down,
                             host: moe_hetero_host, ws, stage_stream, stage_event, n_threads=0, stream=None):
    """One layer forward on the heterogeneous CPU-GPU path; returns its stats."""
    st = moe_hetero_stats()
    hw = [_host_array(w, n) for w, n in ((host_w_gate, "host_w_gate"), (host_w_up, "host_w_up"),
                                          (host_w_down, "host_w_down"))]
    dw = [_ptr_array(w, n) for w, n in ((dev_w_gate, "dev_w_gate"), (dev_w_up, "dev_w_up"),
                                         (dev_w_down, "dev_w_down"))]
    if stage_event.cuda_event == 0:  # torch creates the CUDA event on its first record
        stage_event.record(stage_stream)
    _check(lib().moe_layer_forward_hetero(
        C.byref(dims), C.byref(args), C.byref(outs), C.byref(cost), *[C.cast(a, C.c_void_p) for a in hw],
        *[C.cast(a, C.c_void_p) for a in dw], C.byref(host), int(n_threads), _ptr(ws, torch.uint8, name="ws"),
        ws.numel(), _stream(stream), _stream(stage_stream), C.c_void_p(stage_event.cuda_event), C.byref(st)),
        "moe_layer_forward_hetero")
    return st


def moe_cache_start(dims, pipe: moe_cache_pipe, start_set: int, stream=None):
    _check(lib().moe_cache_start(C.byref(dims), C.byref(pipe), C.c_uint64(start_set & (2**64 - 1)), _stream(stream)),
           "moe_cache_start")


def moe_cache_step(dims, args: moe_layer_args, outs: moe_layer_outputs, pipe: moe_cache_pipe, host_w, dev_w, ws,
                   stage_stream, stream=None):
    """host_w / dev_w: three C arrays of the N experts' host (pinned) and
    device pointers each (gate, up, down), built once by the caller."""
    _check(lib().moe_cache_step(C.byref(dims), C.byref(args), C.byref(outs), C.byref(pipe),
                                *[C.cast(a, C.c_void_p) for a in host_w], *[C.cast(a, C.c_void_p) for a in dev_w],
                                C.c_void_p(ws.data_ptr()), ws.numel(), _stream(stream), _stream(stage_stream)),
           "moe_cache_step")


def moe_cache_step_prepared(call_args):
    """moe_cache_step with its ctypes arguments built once (a decode loop's
    fast path): call_args = the tuple moe_cache_step would pass."""
    _check(lib().moe_cache_step(*call_args), "moe_cache_step")


def moe_cache_drain(dims, pipe: moe_cache_pipe, host_w, dev_w, stage_stream):
    _check(lib().moe_cache_drain(C.byref(dims), C.byref(pipe), *[C.cast(a, C.c_void_p) for a in host_w],
                                 *[C.cast(a, C.c_void_p) for a in dev_w], _stream(stage_stream)), "moe_cache_drain")


def moe_set_graph_replay(enabled: bool):
    """moe_layer_forward's graph replay on (default) or off."""
    lib().moe_set_graph_replay(int(bool(enabled)))


def moe_check(ws, stream=None):
    """Synchronise and return (device_status, detail); clears the error word."""
    st = C.c_int()
    det = C.c_int32()
    _check(lib().moe_check(_ptr(ws, torch.uint8, name="ws"), _stream(stream), C.byref(st), C.byref(det)),
           "moe_check")
    return st.value, det.value


def moe_testing_fail_copies_after(n: int):
    lib().moe_testing_fail_copies_after(int(n))


def moe_testing_set_tc_pairs(mode: int):
    """-1: the prefill FFN chooses single CTAs or CTA pairs; 0 / 1: force."""
    lib().moe_testing_set_tc_pairs(int(mode))


def moe_testing_wait_timeout(ws, stream=None):
    """Queue a kernel whose device wait cannot finish; it times out (about 1 s)
    and records MOE_ERR_TIMEOUT in ws's error word (read it with moe_check)."""
    _check(lib().moe_testing_wait_timeout(C.c_void_p(ws.data_ptr()), ws.numel() * ws.element_size(),
                                          _stream(stream)), "moe_testing_wait_timeout")


from .layer import DeviceLayer, LayerBuffers  # noqa: E402,F401
