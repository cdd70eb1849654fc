"""ctypes binding of the kvs C ABI (include/kvs.h).

Argument marshalling only: every step of the attention path runs in the CUDA
library ``_build/libkvs.so``.  The functions named ``kvs_*`` mirror the C entry
points one to one; :class:`KVStream` owns the torch-allocated arena,
workspace, host history and streams that a context needs.  If the library is
missing, :func:`load` raises -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
import math
import os

import numpy as np

from . import build as _build

KVS_OK = 0
KVS_ERR_INVALID = -1
KVS_ERR_UNSUPPORTED = -2
KVS_ERR_ARENA = -3
KVS_ERR_HOST = -4
KVS_ERR_CUDA = -5
KVS_ERR_COVERAGE = -6
KVS_ERR_CAPACITY = -7
KVS_ERR_TIMEOUT = -8
KVS_ERR_INJECTED = -9
KVS_ERR_STATE = -10

KVS_TYPE_Q4_0 = 2
KVS_TYPE_Q8_0 = 8
KVS_F32 = 0
KVS_F16 = 1
KVS_FLAG_PLAN_ONLY = 1
KVS_FLAG_DMA_FILL = 2
KVS_FLAG_F16_OPERANDS = 4

KVS_OP_RECORD, KVS_OP_WAIT, KVS_OP_FILL, KVS_OP_READ, KVS_OP_POOL_LOAD = 1, 2, 3, 4, 5
KVS_OP_PUBLISH, KVS_OP_WRITE, KVS_OP_LAUNCH, KVS_OP_MOVE = 6, 7, 8, 9
KVS_FAULT_NONE, KVS_FAULT_FILL_ENQUEUE, KVS_FAULT_SYNC_STALL, KVS_FAULT_DEVICE_WAIT = 0, 1, 2, 3


class kvs_config(ctypes.Structure):
    _fields_ = [
        ("page_tokens", ctypes.c_uint32),
        ("n_layers", ctypes.c_uint32),
        ("n_kv_head", ctypes.c_uint32),
        ("head_dim", ctypes.c_uint32),
        ("max_q_head", ctypes.c_uint32),
        ("max_rows", ctypes.c_uint32),
        ("max_tokens", ctypes.c_uint64),
        ("k_type", ctypes.c_int32),
        ("v_type", ctypes.c_int32),
        ("arena", ctypes.c_void_p),
        ("arena_bytes", ctypes.c_uint64),
        ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_uint64),
        ("host", ctypes.c_void_p),
        ("host_bytes", ctypes.c_uint64),
        ("ring_slots", ctypes.c_uint32),
        ("chunk_pages", ctypes.c_uint32),
        ("attn_stream", ctypes.c_void_p),
        ("copy_stream", ctypes.c_void_p),
        ("flags", ctypes.c_uint32),
        ("n_lanes", ctypes.c_uint32),
        ("lane_attn_streams", ctypes.c_void_p * 7),
        ("lane_copy_streams", ctypes.c_void_p * 7),
        ("prefill_split_pages", ctypes.c_uint32),
        ("max_verify_rows", ctypes.c_uint32),
    ]


class kvs_stats_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in (
        "h2d_bytes", "h2d_pages", "h2d_launches", "pool_load_bytes", "d2h_bytes", "d2h_pages",
        "ring_chunks", "ring_recycles", "resident_pages_read", "ring_pages_read", "attend_calls",
        "kernel_launches", "decode_launches")] + [("decode_ms", ctypes.c_double)] + [
        (n, ctypes.c_uint64) for n in ("decode_timed", "decode_bytes", "ring_slots", "pool_slots",
                                       "pool_used", "graph_launches", "graph_kernels",
                                       "chunk_pages", "observed_reads", "ready_misses")] + [
        (n, ctypes.c_double) for n in ("ring_occupancy", "copy_busy")]


class kvs_trace_op(ctypes.Structure):
    _fields_ = [("op", ctypes.c_uint32), ("stream", ctypes.c_uint32), ("layer", ctypes.c_uint32),
                ("event", ctypes.c_uint32), ("a", ctypes.c_int64), ("b", ctypes.c_int64),
                ("c", ctypes.c_int64), ("d", ctypes.c_int64)]


class kvs_timeline_record(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_uint32), ("layer", ctypes.c_uint32), ("stream", ctypes.c_int32),
                ("pages", ctypes.c_uint32), ("start_ns", ctypes.c_uint64), ("end_ns", ctypes.c_uint64)]


KVS_TL_KINDS = {1: "append", 2: "clear", 3: "qprep", 4: "read_resident", 5: "read_ring", 6: "combine",
                7: "fill", 8: "pool_load", 9: "prefill"}


class kvs_policy_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint32) for n in (
        "page_tokens", "n_layers", "budget_slots", "min_ring_slots", "max_ring_slots", "step_slots",
        "hold_steps")] + [(n, ctypes.c_float) for n in ("miss_grow", "copy_busy_max", "occupancy_shrink",
                                                      "link_gbs")]


class kvs_policy_state(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint32) for n in ("ring_slots", "grow_run", "shrink_run", "steps")]


class kvs_policy_observation(ctypes.Structure):
    _fields_ = [("context_tokens", ctypes.c_uint64), ("streamed_reads", ctypes.c_uint64),
                ("ready_misses", ctypes.c_uint64), ("ring_occupancy", ctypes.c_float),
                ("copy_busy", ctypes.c_float), ("copy_bytes", ctypes.c_uint64), ("interval_ns", ctypes.c_uint64)]


class kvs_policy_decision(ctypes.Structure):
    _fields_ = [("ring_slots", ctypes.c_uint32), ("resident_slots", ctypes.c_uint32),
                ("resident_pages_per_layer", ctypes.c_uint64), ("pages_per_layer", ctypes.c_uint64),
                ("reason", ctypes.c_uint32), ("changed", ctypes.c_int32)]


KVS_POLICY_INIT, KVS_POLICY_FITS, KVS_POLICY_HOLD, KVS_POLICY_GROW, KVS_POLICY_SHRINK, KVS_POLICY_CLAMP = range(1, 7)


# every symbol include/kvs.h declares, with its ctypes signature
_P, _U32, _U64, _I32, _I64, _F32 = (ctypes.c_void_p, ctypes.c_uint32, ctypes.c_uint64,
                                    ctypes.c_int32, ctypes.c_int64, ctypes.c_float)
SIGNATURES = {
    "kvs_query_sizes": ([_P, _P, _P, _P, _P], _I32),
    "kvs_create": ([_P, _P], _I32),
    "kvs_destroy": ([_P], _I32),
    "kvs_append": ([_P, _U32, _P, _P, _U32], _I32),
    "kvs_truncate": ([_P, _U32, _U64], _I32),
    "kvs_length": ([_P, _U32, _P], _I32),
    "kvs_load_host_pages": ([_P, _U32, _U64, _U64, _P], _I32),
    "kvs_set_residency": ([_P, _U32, _P, _U64], _I32),
    "kvs_set_ring_slots": ([_P, _U32, _U32], _I32),
    "kvs_prefetch": ([_P, _U32], _I32),
    "kvs_observe": ([_P, _P, ctypes.c_int], _I32),
    "kvs_lease_acquire": ([_P, _U32, _U32], _I32),
    "kvs_lease_release": ([_P], _I32),
    "kvs_lease_info": ([_P, _P, _P, _P], _I32),
    "kvs_attend": ([_P, _U32, _P, _I32, _U32, _U32, _U64, _F32, _P, _P], _I32),
    "kvs_sync": ([_P, _U32], _I32),
    "kvs_flush": ([_P, _U32], _I32),
    "kvs_page_location": ([_P, _U32, _U64, _P, _P], _I32),
    "kvs_read_slot": ([_P, _I64, _P], _I32),
    "kvs_read_host_page": ([_P, _U32, _U64, _P], _I32),
    "kvs_ring_info": ([_P, _P, _P], _I32),
    "kvs_stats": ([_P, _P, ctypes.c_int], _I32),
    "kvs_set_timing": ([_P, ctypes.c_int], _I32),
    "kvs_timeline_begin": ([_P, _P, _U32], _I32),
    "kvs_timeline_end": ([_P], _I32),
    "kvs_timeline_read": ([_P, _P, _U32, _P, _P], _I32),
    "kvs_last_error": ([_P], ctypes.c_char_p),
    "kvs_debug_inject": ([_P, _U32, _U64], _I32),
    "kvs_trace_read": ([_P, _U64, _U64, _P, _P, _P], _I32),
    "kvs_version": ([], _I32),
    "kvs_graph_begin": ([_P], _I32),
    "kvs_graph_end": ([_P], _I32),
    "kvs_graph_launch": ([_P], _I32),
    "kvs_graph_destroy": ([_P], _I32),
    "kvs_attend_pages_noalloc": ([_P, _U64, _P, _U64, _U32, _U32, _U32, _P, _I32, _U32, _U32, _U64, _F32,
                                  _P, _P, _P], _I32),
    "kvs_policy_step": ([_P, _P, _P, _P, _P], _I32),
}
KVS_TIME_RESIDENT = 1
KVS_TIME_RING = 2

_lib = None


class KVSError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"kvs status {status}: {msg}")
        self.status = status


def load(build_if_stale: bool = True):
    """Load ``libkvs.so`` (building it first if its sources are newer)."""
    global _lib
    if _lib is not None:
        return _lib
    if build_if_stale:
        _build.build()
    if not os.path.exists(_build.LIB):
        raise ImportError(f"kvs CUDA library not built: {_build.LIB} is missing")
    lib = ctypes.CDLL(_build.LIB)
    for name, (args, res) in SIGNATURES.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    _lib = lib
    return lib


def _ptr(t) -> int:
    """Address of a torch tensor / numpy array / int (None -> 0)."""
    if t is None:
        return 0
    if isinstance(t, int):
        return t
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


def _check(ctx, status: int):
    if status != KVS_OK:
        msg = load().kvs_last_error(ctx)
        raise KVSError(status, msg.decode() if msg else "")
    return status


# ------------------------------------------------------------ C ABI mirror

def kvs_version() -> int:
    return load().kvs_version()


def kvs_query_sizes(cfg: kvs_config):
    out = [ctypes.c_uint64() for _ in range(4)]
    _check(None, load().kvs_query_sizes(ctypes.byref(cfg), *[ctypes.byref(o) for o in out]))
    return tuple(o.value for o in out)  # page_bytes, host_bytes, arena_min, workspace_min


def kvs_create(cfg: kvs_config) -> int:
    h = ctypes.c_void_p()
    _check(None, load().kvs_create(ctypes.byref(cfg), ctypes.byref(h)))
    return h.value


def kvs_destroy(ctx: int) -> int:
    return _check(ctx, load().kvs_destroy(ctx))


def kvs_append(ctx, layer, k, v, n_tokens) -> int:
    return _check(ctx, load().kvs_append(ctx, layer, _ptr(k), _ptr(v), n_tokens))


def kvs_truncate(ctx, layer, n_tokens) -> int:
    return _check(ctx, load().kvs_truncate(ctx, layer, n_tokens))


def kvs_length(ctx, layer) -> int:
    n = ctypes.c_uint64()
    _check(ctx, load().kvs_length(ctx, layer, ctypes.byref(n)))
    return n.value


def kvs_load_host_pages(ctx, layer, first_page, n_pages, src) -> int:
    """Install n_pages encoded pages (host memory at src) into the host history of layer."""
    return _check(ctx, load().kvs_load_host_pages(ctx, layer, first_page, n_pages, _ptr(src)))


def kvs_set_residency(ctx, layer, mask) -> int:
    m = np.ascontiguousarray(mask, dtype=np.uint8)
    return _check(ctx, load().kvs_set_residency(ctx, layer, m.ctypes.data, m.size))


def kvs_set_ring_slots(ctx, n_slots, chunk_pages=0) -> int:
    return _check(ctx, load().kvs_set_ring_slots(ctx, n_slots, chunk_pages))


def kvs_policy_step(config: kvs_policy_config, previous: kvs_policy_state,
                    observation: kvs_policy_observation):
    """One residency-policy decision: returns (next state, decision).  Pure host call."""
    nxt, dec = kvs_policy_state(), kvs_policy_decision()
    st = load().kvs_policy_step(ctypes.byref(config), ctypes.byref(previous), ctypes.byref(observation),
                                ctypes.byref(nxt), ctypes.byref(dec))
    if st != KVS_OK:
        raise KVSError(st, "kvs_policy_step: invalid config, state or observation")
    return nxt, dec


def kvs_observe(ctx, reset=False) -> "kvs_policy_observation":
    """The policy's feedback measured on the device since the last reset."""
    obs = kvs_policy_observation()
    _check(ctx, load().kvs_observe(ctx, ctypes.byref(obs), 1 if reset else 0))
    return obs


def kvs_lease_acquire(ctx, layer, extra_slots=0) -> int:
    return _check(ctx, load().kvs_lease_acquire(ctx, layer, extra_slots))


def kvs_lease_release(ctx) -> int:
    return _check(ctx, load().kvs_lease_release(ctx))


def kvs_lease_info(ctx):
    """(leased layer or -1, leased slots, spare slots)"""
    layer, held, spare = ctypes.c_int64(), ctypes.c_uint32(), ctypes.c_uint32()
    _check(ctx, load().kvs_lease_info(ctx, ctypes.byref(layer), ctypes.byref(held), ctypes.byref(spare)))
    return layer.value, held.value, spare.value


def kvs_prefetch(ctx, layer) -> int:
    return _check(ctx, load().kvs_prefetch(ctx, layer))


def kvs_attend(ctx, layer, q, q_dtype, n_rows, n_q_head, pos0, scale, out, lse=None) -> int:
    return _check(ctx, load().kvs_attend(ctx, layer, _ptr(q), q_dtype, n_rows, n_q_head, pos0,
                                         float(scale), _ptr(out), _ptr(lse)))


def kvs_sync(ctx, timeout_ms=0) -> int:
    return _check(ctx, load().kvs_sync(ctx, timeout_ms))


def kvs_flush(ctx, layer=0xFFFFFFFF) -> int:
    return _check(ctx, load().kvs_flush(ctx, layer))


def kvs_page_location(ctx, layer, page):
    kind, slot = ctypes.c_int32(), ctypes.c_int64()
    _check(ctx, load().kvs_page_location(ctx, layer, page, ctypes.byref(kind), ctypes.byref(slot)))
    return kind.value, slot.value


def kvs_read_slot(ctx, slot, dst: np.ndarray) -> int:
    return _check(ctx, load().kvs_read_slot(ctx, slot, dst.ctypes.data))


def kvs_read_host_page(ctx, layer, page, dst: np.ndarray) -> int:
    return _check(ctx, load().kvs_read_host_page(ctx, layer, page, dst.ctypes.data))


def kvs_ring_info(ctx):
    first, n = ctypes.c_int64(), ctypes.c_uint32()
    _check(ctx, load().kvs_ring_info(ctx, ctypes.byref(first), ctypes.byref(n)))
    return first.value, n.value


def kvs_stats(ctx, reset=False) -> dict:
    st = kvs_stats_t()
    _check(ctx, load().kvs_stats(ctx, ctypes.byref(st), 1 if reset else 0))
    return {name: getattr(st, name) for name, _ in kvs_stats_t._fields_}


def kvs_set_timing(ctx, mask=KVS_TIME_RESIDENT | KVS_TIME_RING) -> int:
    return _check(ctx, load().kvs_set_timing(ctx, int(mask)))


def kvs_timeline_begin(ctx, records, max_records) -> int:
    return _check(ctx, load().kvs_timeline_begin(ctx, _ptr(records), int(max_records)))


def kvs_timeline_end(ctx) -> int:
    return _check(ctx, load().kvs_timeline_end(ctx))


def kvs_timeline_read(ctx, max_out):
    """(list of per-launch dicts with kind names, dropped launches)."""
    buf = (kvs_timeline_record * max(int(max_out), 1))()
    n, dropped = ctypes.c_uint32(), ctypes.c_uint32()
    _check(ctx, load().kvs_timeline_read(ctx, buf, int(max_out), ctypes.byref(n), ctypes.byref(dropped)))
    out = []
    for i in range(n.value):
        r = {f: getattr(buf[i], f) for f, _ in kvs_timeline_record._fields_}
        r["kind"] = KVS_TL_KINDS.get(r["kind"], str(r["kind"]))
        out.append(r)
    return out, dropped.value


def kvs_attend_pages_noalloc(pages, pages_bytes, page_slots, page_tokens, n_kv_head, head_dim, q, q_dtype,
                             n_rows, n_q_head, pos0, scale, out, lse=None, stream=0) -> int:
    """Attention over caller pages with no workspace (fixed in-library scratch)."""
    slots = np.ascontiguousarray(page_slots, dtype=np.uint32)
    return _check(None, load().kvs_attend_pages_noalloc(_ptr(pages), pages_bytes, slots.ctypes.data, slots.size,
                                                        page_tokens, n_kv_head, head_dim, _ptr(q), q_dtype,
                                                        n_rows, n_q_head, pos0, float(scale), _ptr(out),
                                                        _ptr(lse), stream))


def kvs_graph_begin(ctx) -> int:
    return _check(ctx, load().kvs_graph_begin(ctx))


def kvs_graph_end(ctx) -> int:
    return _check(ctx, load().kvs_graph_end(ctx))


def kvs_graph_launch(ctx) -> int:
    return _check(ctx, load().kvs_graph_launch(ctx))


def kvs_graph_destroy(ctx) -> int:
    return _check(ctx, load().kvs_graph_destroy(ctx))




def kvs_last_error(ctx) -> str:
    m = load().kvs_last_error(ctx)
    return m.decode() if m else ""


def kvs_debug_inject(ctx, fault, nth) -> int:
    return _check(ctx, load().kvs_debug_inject(ctx, fault, nth))


def kvs_trace_read(ctx):
    """All logged operations of a plan-only context as a list of dicts."""
    total = ctypes.c_uint64()
    _check(ctx, load().kvs_trace_read(ctx, 0, 0, None, None, ctypes.byref(total)))
    n = total.value
    buf = (kvs_trace_op * max(n, 1))()
    got = ctypes.c_uint64()
    _check(ctx, load().kvs_trace_read(ctx, 0, n, buf, ctypes.byref(got), None))
    return [{f: getattr(buf[i], f) for f, _ in kvs_trace_op._fields_} for i in range(got.value)]


# ------------------------------------------------------------ owner class

def _alloc_host(nbytes, how):
    """Host history buffer.  "pinned" (default): CUDA-allocated pinned memory
    (torch); "pageable": numpy memory that kvs_create registers with CUDA;
    "hugepage": an anonymous mapping advised for transparent huge pages, then
    registered.  Measured on GB300 with 64 layers x 262144 tokens (27 GB): ring
    refills from CUDA-allocated memory ran at 89 % of the host-link ceiling,
    from registered pageable memory at 7.5 % (the GPU maps it with small pages),
    from huge-page advised memory at 57 %."""
    if how == "pageable":
        return np.empty(nbytes, dtype=np.uint8)
    if how == "pinned":
        import torch
        return torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    if how == "hugepage":
        import mmap
        m = mmap.mmap(-1, nbytes, flags=mmap.MAP_PRIVATE | mmap.MAP_ANONYMOUS)
        if hasattr(m, "madvise") and hasattr(mmap, "MADV_HUGEPAGE"):
            m.madvise(mmap.MADV_HUGEPAGE)
        return np.frombuffer(m, dtype=np.uint8)
    raise ValueError(f"unknown host allocation {how!r}")



class KVStream:
    """A kvs context with its torch-owned arena, workspace, streams and host history.

    ``arena_slots`` counts page slots (tails + pool + ring); default = tails +
    ring + one layer's pages of pool.  ``host`` may be given (numpy uint8 or a
    pinned torch tensor); otherwise ``host_alloc`` chooses the buffer:
    "pinned" (the default, CUDA-allocated pinned memory), "pageable" (numpy
    memory that kvs_create registers with CUDA) or "hugepage".  A plan-only
    context keeps ``host`` (if given) as a plain host buffer.
    """

    def __init__(self, *, page_tokens, n_layers, n_kv_head, head_dim, max_q_head, max_rows,
                 max_tokens, ring_slots=8, chunk_pages=0, arena_slots=None, arena_bytes=None,
                 plan_only=False, host=None, device="cuda", lanes=1, copy_priority=None,
                 prefill_split_pages=0, dma_fill=False, host_alloc="pinned", max_verify_rows=0,
                 f16_operands=False):
        cfg = kvs_config()
        cfg.page_tokens, cfg.n_layers, cfg.n_kv_head, cfg.head_dim = page_tokens, n_layers, n_kv_head, head_dim
        cfg.max_q_head, cfg.max_rows, cfg.max_tokens = max_q_head, max_rows, max_tokens
        cfg.k_type, cfg.v_type = KVS_TYPE_Q8_0, KVS_TYPE_Q4_0
        cfg.ring_slots, cfg.chunk_pages = ring_slots, chunk_pages
        cfg.n_lanes = lanes
        cfg.prefill_split_pages = prefill_split_pages
        cfg.max_verify_rows = max_verify_rows
        cfg.flags = (KVS_FLAG_DMA_FILL if dma_fill else 0) | (KVS_FLAG_F16_OPERANDS if f16_operands else 0)
        self.page_bytes, host_bytes, arena_min, ws_bytes = kvs_query_sizes(cfg)
        self.max_pages = math.ceil(max_tokens / page_tokens)
        if arena_bytes is None:
            if arena_slots is None:
                arena_slots = 2 * n_layers + ring_slots + self.max_pages
            arena_bytes = arena_slots * self.page_bytes
        self.plan_only = plan_only
        self.geom = dict(P=page_tokens, L=n_layers, Hk=n_kv_head, D=head_dim)
        if plan_only:
            cfg.flags |= KVS_FLAG_PLAN_ONLY
            cfg.arena, cfg.workspace = 1 << 20, 1 << 21  # never dereferenced
            # host memory is plain memory: a plan-only context may keep a history
            self.host = host
            cfg.host = _ptr(host)
            self.arena = self.workspace = None
        else:
            import torch
            # ring refills are the critical path of a streamed step: their copy
            # streams get the higher scheduling priority, so fill kernels take
            # SMs ahead of queued attention blocks
            try:
                hi = torch.cuda.Stream.priority_range()[1]
            except Exception:
                hi = -1
            self.attn_stream = torch.cuda.Stream(device=device)
            self.copy_stream = torch.cuda.Stream(device=device, priority=copy_priority if copy_priority is not None else hi)
            self.arena = torch.empty(arena_bytes, dtype=torch.uint8, device=device)
            self.workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=device)
            if host is None:
                host = _alloc_host(host_bytes, host_alloc)
            self.host = host
            cfg.arena, cfg.workspace = self.arena.data_ptr(), self.workspace.data_ptr()
            cfg.host = _ptr(host)
            cfg.attn_stream = self.attn_stream.cuda_stream
            cfg.copy_stream = self.copy_stream.cuda_stream
            self.lane_streams = []
            for i in range(lanes - 1):
                a = torch.cuda.Stream(device=device)
                c = torch.cuda.Stream(device=device, priority=copy_priority if copy_priority is not None else hi)
                self.lane_streams += [a, c]
                cfg.lane_attn_streams[i] = a.cuda_stream
                cfg.lane_copy_streams[i] = c.cuda_stream
        cfg.arena_bytes, cfg.workspace_bytes, cfg.host_bytes = arena_bytes, ws_bytes, host_bytes
        self.cfg = cfg
        self.ctx = kvs_create(cfg)

    # -- lifecycle
    def close(self):
        if getattr(self, "ctx", None):
            kvs_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- calls (device tensors in, device tensors out)
    def append(self, layer, k, v):
        assert k.is_contiguous() and v.is_contiguous() and k.shape == v.shape
        return kvs_append(self.ctx, layer, k, v, k.shape[0])

    def attend(self, layer, q, pos0, scale=None, out=None, lse=None):
        import torch
        R, Hq, D = q.shape
        scale = 1.0 / math.sqrt(D) if scale is None else scale
        if out is None and not self.plan_only:
            out = torch.empty((R, Hq, D), dtype=torch.float32, device=q.device)
        if lse is None and not self.plan_only:
            lse = torch.empty((R, Hq), dtype=torch.float32, device=q.device)
        dt = KVS_F16 if q.dtype == torch.float16 else KVS_F32
        kvs_attend(self.ctx, layer, None if self.plan_only else q, dt, R, Hq, pos0, scale, out, lse)
        return out, lse

    def attend_plan(self, layer, n_rows, n_q_head, pos0):
        """Plan-only attend (no tensors)."""
        return kvs_attend(self.ctx, layer, None, KVS_F32, n_rows, n_q_head, pos0, 1.0, None, None)

    def truncate(self, layer, n):
        return kvs_truncate(self.ctx, layer, n)

    def length(self, layer):
        return kvs_length(self.ctx, layer)

    def load_host_pages(self, layer, first_page, pages):
        """pages: host uint8 array of whole pages (n_pages * page_bytes) in the library layout."""
        src = np.ascontiguousarray(pages, dtype=np.uint8).reshape(-1)
        if src.size % self.page_bytes:
            raise ValueError("pages must hold a whole number of page_bytes")
        return kvs_load_host_pages(self.ctx, layer, first_page, src.size // self.page_bytes, src)

    def set_residency(self, layer, mask):
        return kvs_set_residency(self.ctx, layer, mask)

    def set_ring_slots(self, n, chunk_pages=0):
        return kvs_set_ring_slots(self.ctx, n, chunk_pages)

    def prefetch(self, layer):
        return kvs_prefetch(self.ctx, layer)

    def observe(self, reset=False):
        return kvs_observe(self.ctx, reset)

    def lease_acquire(self, layer, extra_slots=0):
        return kvs_lease_acquire(self.ctx, layer, extra_slots)

    def lease_release(self):
        return kvs_lease_release(self.ctx)

    def lease_info(self):
        return kvs_lease_info(self.ctx)

    def sync(self, timeout_ms=0):
        return kvs_sync(self.ctx, timeout_ms)

    def flush(self, layer=0xFFFFFFFF):
        return kvs_flush(self.ctx, layer)

    def page_location(self, layer, page):
        return kvs_page_location(self.ctx, layer, page)

    def read_slot(self, slot):
        buf = np.empty(self.page_bytes, dtype=np.uint8)
        kvs_read_slot(self.ctx, slot, buf)
        return buf

    def read_host_page(self, layer, page):
        buf = np.empty(self.page_bytes, dtype=np.uint8)
        kvs_read_host_page(self.ctx, layer, page, buf)
        return buf

    def ring_info(self):
        return kvs_ring_info(self.ctx)

    def stats(self, reset=False):
        return kvs_stats(self.ctx, reset)

    def set_timing(self, mask=KVS_TIME_RESIDENT | KVS_TIME_RING):
        return kvs_set_timing(self.ctx, mask)

    def timeline_begin(self, max_records=1 << 16):
        """Stamp every following launch (until timeline_end) into a device buffer of max_records."""
        import torch
        self._tl = torch.zeros(2 * max_records, dtype=torch.int64, device=self.arena.device)
        return kvs_timeline_begin(self.ctx, self._tl, max_records)

    def timeline_zero(self):
        """Zero the records on the attention stream (before the stamped launches run again)."""
        import torch
        with torch.cuda.stream(self.attn_stream):
            self._tl.zero_()

    def timeline_end(self):
        return kvs_timeline_end(self.ctx)

    def timeline_read(self):
        return kvs_timeline_read(self.ctx, self._tl.numel() // 2)

    def graph_begin(self):
        return kvs_graph_begin(self.ctx)

    def graph_end(self):
        return kvs_graph_end(self.ctx)

    def graph_launch(self):
        return kvs_graph_launch(self.ctx)

    def graph_destroy(self):
        return kvs_graph_destroy(self.ctx)

    def inject(self, fault, nth):
        return kvs_debug_inject(self.ctx, fault, nth)

    def trace(self):
        return kvs_trace_read(self.ctx)

    def last_error(self):
        return kvs_last_error(self.ctx)
