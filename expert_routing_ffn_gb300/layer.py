"""Device-side holders for one MoE layer: weights, expert table, workspace and
output buffers, wired to the C ABI.  Marshalling only — all arithmetic runs
in the library's CUDA kernels."""
from __future__ import annotations

import ctypes as C

import torch

from . import (MOE_NUM_COUNTERS, _check, _stream, lib, make_dims, moe_expert_table_init,
               moe_expert_table_size, moe_layer_args, moe_layer_forward, moe_layer_outputs,
               moe_workspace_size)


def as_i64(mask: int) -> int:
    """uint64 bit pattern as a signed int64 value."""
    mask &= (1 << 64) - 1
    return mask - (1 << 64) if mask >= (1 << 63) else mask


def as_u64(v: int) -> int:
    return int(v) & ((1 << 64) - 1)


class DeviceLayer:
    """Weights of one layer on the GPU plus its expert table and workspace.

    cfg: a workloads.LayerConfig; W: a workloads.LayerWeights (float32 arrays
    holding the exact parameter values).  T_max: the largest token count the
    workspace is sized for.
    """

    def __init__(self, cfg, W, T_max: int, device: str = "cuda"):
        self.cfg = cfg
        self.dims = make_dims(T_max, cfg.d, cfg.N, cfg.k, cfg.I, cfg.n_shared, cfg.I_shared, cfg.r,
                              cfg.delta_max, cfg.wtype)
        self.dt = torch.bfloat16 if cfg.wtype == "bf16" else torch.float32
        dev = torch.device(device)
        self.device = dev

        def t(a, dt=None):
            return torch.from_numpy(a).to(dev).to(dt or self.dt).contiguous()

        self.w_router = t(W.w_router)
        self.w_prefetch = t(W.w_prefetch)
        self.w_ord = t(W.w_ord, torch.float32)
        self.theta = t(W.theta, torch.float32)
        self.router_bias = None if W.router_bias is None else t(W.router_bias, torch.float32)
        self.w_gate = torch.empty((cfg.N, cfg.I, cfg.d), dtype=self.dt, device=dev)
        self.w_up = torch.empty_like(self.w_gate)
        self.w_down = torch.empty_like(self.w_gate)
        for e in range(cfg.N):  # one expert at a time keeps host->device staging small
            self.w_gate[e].copy_(torch.from_numpy(W.w_gate[e]))
            self.w_up[e].copy_(torch.from_numpy(W.w_up[e]))
            self.w_down[e].copy_(torch.from_numpy(W.w_down[e]))
        ns = max(cfg.n_shared, 0)
        self.sh_gate = t(W.sh_gate) if ns else None
        self.sh_up = t(W.sh_up) if ns else None
        self.sh_down = t(W.sh_down) if ns else None
        self.lore_a = t(W.lore_a) if cfg.r > 0 else None
        self.lore_b = t(W.lore_b) if cfg.r > 0 else None
        self.table = torch.empty(moe_expert_table_size(self.dims), dtype=torch.uint8, device=dev)
        self.ws = torch.zeros(moe_workspace_size(self.dims), dtype=torch.uint8, device=dev)
        self.resident = torch.full((1,), as_i64((1 << 64) - 1), dtype=torch.int64, device=dev)
        self.bind_table()

    def bind_table(self):
        sh = [list(self.sh_gate), list(self.sh_up), list(self.sh_down)] if self.cfg.n_shared else [None] * 3
        moe_expert_table_init(self.dims, list(self.w_gate), list(self.w_up), list(self.w_down),
                              *sh, self.table)

    def set_resident(self, mask: int):
        self.resident.fill_(as_i64(mask))

    def clone(self) -> "DeviceLayer":
        """Another copy of the layer: expert weights in new device buffers (same
        values), its own expert table and workspace; router and LoRE tensors are
        shared."""
        other = object.__new__(DeviceLayer)
        other.__dict__.update(self.__dict__)
        other.__dict__.pop("_call_cache", None)  # cached ABI structs point at this layer's tensors
        for name in ("w_gate", "w_up", "w_down", "sh_gate", "sh_up", "sh_down"):
            t = getattr(self, name)
            setattr(other, name, None if t is None else t.clone())
        other.table = torch.empty_like(self.table)
        other.ws = torch.zeros_like(self.ws)
        other.resident = self.resident.clone()
        other.bind_table()
        return other


class LayerBuffers:
    """Outputs of moe_layer_forward for up to T tokens."""

    def __init__(self, layer: DeviceLayer, T: int):
        cfg, dev = layer.cfg, layer.device
        k, N, d = cfg.k, cfg.N, cfg.d
        i32 = dict(dtype=torch.int32, device=dev)
        f32 = dict(dtype=torch.float32, device=dev)
        i64 = dict(dtype=torch.int64, device=dev)
        self.T = T
        self.topk_idx = torch.empty((T, k), **i32)
        self.topk_gate = torch.empty((T, k), **f32)
        self.router_prob = torch.empty((T, N), **f32)
        self.delta_hat = torch.empty((T,), **i32)
        self.prefetch_mask = torch.empty((T,), **i64)
        self.delta_star = torch.empty((T,), **i32)
        self.batch_resident = torch.zeros((1,), **i64)
        self.final_idx = torch.empty((T, k), **i32)
        self.final_gate = torch.empty((T, k), **f32)
        self.final_kind = torch.empty((T, k), **i32)
        self.fetch_mask = torch.zeros((1,), **i64)
        self.counters = torch.zeros((MOE_NUM_COUNTERS,), **i32)
        self.expert_offsets = torch.empty((N + 1,), **i32)
        self.perm = torch.empty((T * k,), **i32)
        self.inv_perm = torch.empty((T * k,), **i32)
        self.y_perm = torch.empty((T * k, d), **f32)
        self.y_shared = torch.empty((T, d), **f32) if cfg.n_shared else None
        self.y_lore = torch.empty((T, d), **f32) if cfg.r > 0 else None
        self.out = torch.empty((T, d), **f32)

    def outputs_struct(self) -> moe_layer_outputs:
        """The output pointers for the ABI (built once: the buffers never move)."""
        o = getattr(self, "_outs", None)
        if o is None:
            o = moe_layer_outputs()
            for name, _ in moe_layer_outputs._fields_:
                tns = getattr(self, name)
                setattr(o, name, None if tns is None else tns.data_ptr())
            self._outs = o
        return o


def layer_args(layer: DeviceLayer, x, x_pre=None, policy=None, gamma=None, tau=None,
               keep_frac=None, n_resident=None, use_prefetch_mask=None) -> moe_layer_args:
    cfg = layer.cfg
    a = moe_layer_args()
    a.x = x.data_ptr()
    a.x_pre = None if x_pre is None else x_pre.data_ptr()
    a.w_router = layer.w_router.data_ptr()
    a.router_bias = None if layer.router_bias is None else layer.router_bias.data_ptr()
    a.w_prefetch = layer.w_prefetch.data_ptr()
    a.w_ord = layer.w_ord.data_ptr()
    a.theta = layer.theta.data_ptr()
    a.tau = cfg.tau if tau is None else tau
    a.n_resident = max(cfg.n_resident, 0) if n_resident is None else n_resident
    a.resident = layer.resident.data_ptr()
    a.use_prefetch_mask = int(cfg.use_prefetch_mask if use_prefetch_mask is None else use_prefetch_mask)
    a.policy = cfg.policy if policy is None else policy
    a.gamma = cfg.gamma if gamma is None else gamma
    a.keep_frac = cfg.keep_frac if keep_frac is None else keep_frac
    a.table = layer.table.data_ptr()
    a.lore_a = None if layer.lore_a is None else layer.lore_a.data_ptr()
    a.lore_b = None if layer.lore_b is None else layer.lore_b.data_ptr()
    return a


def forward(layer: DeviceLayer, bufs: LayerBuffers, x, stream=None, **kw):
    """One layer forward through moe_layer_forward for x [T, d] (T <= bufs.T).

    The ABI structs of a call (dims for T, the layer arguments for this x and
    these options, the output pointers) are built once and reused while the
    tensors stay where they are, so a decode loop pays only the ABI call."""
    T = x.shape[0]
    assert T <= bufs.T and x.is_contiguous() and x.dtype == layer.dt
    cache = layer.__dict__.setdefault("_call_cache", {})
    key = (T, x.data_ptr(), tuple(sorted(kw.items())), layer.ws.data_ptr())
    hit = cache.get(key)
    if hit is None:
        if len(cache) > 64:
            cache.clear()
        hit = (layer.dims.with_T(T), layer_args(layer, x, **kw), C.c_void_p(layer.ws.data_ptr()),
               layer.ws.numel())
        cache[key] = hit
    dims, args, ws_ptr, ws_bytes = hit
    outs = bufs.outputs_struct()
    _check(lib().moe_layer_forward(C.byref(dims), C.byref(args), C.byref(outs), ws_ptr, ws_bytes,
                                   _stream(stream)), "moe_layer_forward")
    return bufs


def forward_host(layer: DeviceLayer, bufs: LayerBuffers, x, host_x, host_out, stream=None, **kw):
    """One layer forward with the input and the output in (pinned) host
    memory, through moe_layer_forward_host: host_x [T, d] is copied into the
    device buffer x, the layer runs, bufs.out is copied to host_out [T, d]
    float32; all on `stream`, replayed as one CUDA graph per argument set.
    Synchronise the stream before reading host_out."""
    T = x.shape[0]
    assert T <= bufs.T and x.is_contiguous() and x.dtype == layer.dt and x.is_cuda
    assert not host_x.is_cuda and host_x.dtype == layer.dt and host_x.is_contiguous() and host_x.numel() >= x.numel()
    assert not host_out.is_cuda and host_out.dtype == torch.float32 and host_out.numel() >= T * layer.cfg.d
    cache = layer.__dict__.setdefault("_call_cache", {})
    key = (T, x.data_ptr(), tuple(sorted(kw.items())), layer.ws.data_ptr())
    hit = cache.get(key)
    if hit is None:
        if len(cache) > 64:
            cache.clear()
        hit = (layer.dims.with_T(T), layer_args(layer, x, **kw), C.c_void_p(layer.ws.data_ptr()),
               layer.ws.numel())
        cache[key] = hit
    dims, args, ws_ptr, ws_bytes = hit
    outs = bufs.outputs_struct()
    _check(lib().moe_layer_forward_host(C.byref(dims), C.byref(args), C.byref(outs), C.c_void_p(host_x.data_ptr()),
                                        C.c_void_p(host_out.data_ptr()), ws_ptr, ws_bytes, _stream(stream)),
           "moe_layer_forward_host")
    return bufs


class HeteroHost:
    """Pinned host buffers and the host copy of the routed experts for the
    heterogeneous CPU-GPU path (moe_layer_forward_hetero), sized for T tokens.
    The host weights are the layer's own device values copied down once."""

    def __init__(self, layer: DeviceLayer, T: int):
        from . import moe_cpu_experts_scratch_size, moe_hetero_host
        cfg = layer.cfg
        k, d = cfg.k, cfg.d
        pin = dict(pin_memory=True)
        self.T = T
        self.x = torch.empty((T, d), dtype=layer.dt, **pin)
        self.final_idx = torch.empty((T, k), dtype=torch.int32, **pin)
        self.final_kind = torch.empty((T, k), dtype=torch.int32, **pin)
        self.masks = torch.zeros(2, dtype=torch.int64, **pin)
        self.y_rows = torch.empty((T * k, d), dtype=torch.float32, **pin)
        self.scratch = torch.empty(moe_cpu_experts_scratch_size(layer.dims.with_T(T)), dtype=torch.uint8)
        self.w_gate = [layer.w_gate[e].cpu().pin_memory() for e in range(cfg.N)]
        self.w_up = [layer.w_up[e].cpu().pin_memory() for e in range(cfg.N)]
        self.w_down = [layer.w_down[e].cpu().pin_memory() for e in range(cfg.N)]
        h = moe_hetero_host()
        h.x, h.final_idx, h.final_kind = self.x.data_ptr(), self.final_idx.data_ptr(), self.final_kind.data_ptr()
        h.masks, h.y_rows = self.masks.data_ptr(), self.y_rows.data_ptr()
        h.scratch, h.scratch_bytes = self.scratch.data_ptr(), self.scratch.numel()
        self.struct = h


def forward_hetero(layer: DeviceLayer, bufs: LayerBuffers, x, host: HeteroHost, cost, stage_stream, stage_event,
                   n_threads=0, stream=None, **kw):
    """One layer forward on the heterogeneous path (moe_layer_forward_hetero):
    high-confidence misses fetched or run on the host cores by the cost model.
    Returns the call's moe_hetero_stats."""
    from . import moe_layer_forward_hetero
    T = x.shape[0]
    assert T <= bufs.T and T <= host.T and x.is_contiguous() and x.dtype == layer.dt
    args = layer_args(layer, x, **kw)
    return moe_layer_forward_hetero(layer.dims.with_T(T), args, bufs.outputs_struct(), cost, host.w_gate, host.w_up,
                                    host.w_down, list(layer.w_gate), list(layer.w_up), list(layer.w_down),
                                    host.struct, layer.ws, stage_stream, stage_event, n_threads, stream)


class CachePipeline:
    """The overlapped expert-cache pipeline of one layer (moe_cache_start /
    moe_cache_step): heat-decayed cache of `capacity` experts, admissions
    copied from pinned host memory on a staging stream while later steps run
    on the experts already landed.  The host copies are the layer's own
    device values copied down once."""

    def __init__(self, layer: DeviceLayer, capacity: int, decay: float, max_flight_experts: int = 0,
                 stream=None):
        from . import MOE_CACHE_FLIGHTS, MOE_CACHE_RING, moe_cache_pipe
        cfg, dev = layer.cfg, layer.device
        self.layer = layer
        self.stream = stream if stream is not None else torch.cuda.current_stream(dev)
        self.stage_stream = torch.cuda.Stream(device=dev)
        self.ring = torch.zeros(MOE_CACHE_RING * 4, dtype=torch.int64).pin_memory()
        self.masks = torch.zeros(4, dtype=torch.int64, device=dev)
        self.heat = torch.zeros(cfg.N, dtype=torch.float32, device=dev)
        self.stats = torch.zeros(4, dtype=torch.int32, device=dev)
        self.events = [torch.cuda.Event() for _ in range(MOE_CACHE_RING + MOE_CACHE_FLIGHTS)]
        for ev in self.events:  # torch creates the CUDA event on its first record
            ev.record(self.stream)
        self.host_w = [[layer.w_gate[e].cpu().pin_memory() for e in range(cfg.N)],
                       [layer.w_up[e].cpu().pin_memory() for e in range(cfg.N)],
                       [layer.w_down[e].cpu().pin_memory() for e in range(cfg.N)]]
        self._host_arr = [(C.c_void_p * cfg.N)(*[t.data_ptr() for t in m]) for m in self.host_w]
        self._dev_arr = [(C.c_void_p * cfg.N)(*[t.data_ptr() for t in m])
                         for m in (list(layer.w_gate), list(layer.w_up), list(layer.w_down))]
        p = moe_cache_pipe()
        p.capacity, p.decay, p.max_flight_experts = capacity, decay, max_flight_experts
        p.host_ring = self.ring.data_ptr()
        for i in range(MOE_CACHE_RING):
            p.step_events[i] = self.events[i].cuda_event
        for i in range(MOE_CACHE_FLIGHTS):
            p.copy_events[i] = self.events[MOE_CACHE_RING + i].cuda_event
        p.dev_masks, p.dev_heat, p.dev_stats = self.masks.data_ptr(), self.heat.data_ptr(), self.stats.data_ptr()
        self.pipe = p
        self._args = {}

    def start(self, start_set: int):
        from . import moe_cache_start
        self.stream.synchronize()
        moe_cache_start(self.layer.dims.with_T(1), self.pipe, start_set, self.stream)

    def step(self, bufs: LayerBuffers, x, **kw):
        """One pipeline step; the ctypes arguments of a (tokens, x, options,
        buffers) combination are built once and reused."""
        from . import moe_cache_step_prepared
        T = x.shape[0]
        key = (T, x.data_ptr(), tuple(sorted(kw.items())), id(bufs))
        hit = self._args.get(key)
        if hit is None:
            if len(self._args) > 64:
                self._args.clear()
            dims, args, outs = self.layer.dims.with_T(T), layer_args(self.layer, x, **kw), bufs.outputs_struct()
            hit = (C.byref(dims), C.byref(args), C.byref(outs), C.byref(self.pipe),
                   *[C.cast(a, C.c_void_p) for a in self._host_arr], *[C.cast(a, C.c_void_p) for a in self._dev_arr],
                   C.c_void_p(self.layer.ws.data_ptr()), self.layer.ws.numel(), _stream(self.stream),
                   _stream(self.stage_stream), dims, args, outs)
            self._args[key] = hit
        moe_cache_step_prepared(hit[:14])

    def drain(self):
        from . import moe_cache_drain
        moe_cache_drain(self.layer.dims.with_T(1), self.pipe, self._host_arr, self._dev_arr, self.stage_stream)

    def resident_used(self, step: int) -> int:
        """The resident set step `step` ran on (its read-back must have completed)."""
        from . import MOE_CACHE_RING
        if step == 0:
            return as_u64(int(self.ring[2].item())) if self.pipe.step == 0 else None
        return as_u64(int(self.ring[((step - 1) % MOE_CACHE_RING) * 4 + 2].item()))
