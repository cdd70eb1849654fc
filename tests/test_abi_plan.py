"""C-ABI checks that need no GPU: exports, sizes, refusals, and the host-side
scheduler, exercised through a plan-only context (which logs every stream
operation instead of issuing it).

The scheduler tests replay the logged operations through a two-stream
happens-before model (vector clocks; a WAIT orders everything after it on its
stream behind everything before the latest RECORD of that event), then check
the fences the design requires: a ring slot is read only after the copy of
that page into it completed (ready fence), and no copy overwrites a slot
before its last reader finished (consumed fence).
"""
import math
import os
import re

import numpy as np
import pytest

from host_streamed_paged_gb300 import kvs
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_library_exports_every_declared_symbol():
    lib = kvs.load()
    header = open(os.path.join(ROOT, "include", "kvs.h")).read()
    declared = set(re.findall(r"^\S.*?\b(kvs_[a-z_]+)\s*\(", header, flags=re.M))
    assert len(declared) >= 20
    for name in sorted(declared):
        assert hasattr(lib, name), name
    assert declared <= set(kvs.SIGNATURES), declared - set(kvs.SIGNATURES)
    assert kvs.kvs_version() == 4


def _cfg(**kw):
    c = kvs.kvs_config()
    c.page_tokens, c.n_layers, c.n_kv_head, c.head_dim = 256, 4, 4, 256
    c.max_q_head, c.max_rows, c.max_tokens = 24, 6, 32768
    c.k_type, c.v_type = kvs.KVS_TYPE_Q8_0, kvs.KVS_TYPE_Q4_0
    c.ring_slots = 8
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def test_query_sizes_formulas():
    pb, hb, amin, wmin = kvs.kvs_query_sizes(_cfg())
    assert pb == 4 * 256 * 256 * 13 // 8 == 425984  # 416 KiB per page
    assert hb == 4 * 128 * pb
    assert amin == (2 * 4 + 8) * pb
    qfrag = 4 * 8 * 16 * 32 * 16  # query fragments of 4 kv heads (already 256-aligned)
    obs = 1024 * 16  # observation records (one per ring chunk id modulo 1024)
    assert wmin == 256 + obs + qfrag + 128 * 24 * 6 * (256 + 2) * 4  # status, records, fragments, one partial per page
    pb2, *_ = kvs.kvs_query_sizes(_cfg(page_tokens=256, n_kv_head=2, head_dim=128, max_q_head=8))
    assert pb2 == 2 * 256 * 128 * 13 // 8 == 106496  # 104 KiB


@pytest.mark.parametrize("kw", [dict(page_tokens=48), dict(head_dim=96), dict(k_type=kvs.KVS_TYPE_Q4_0),
                                dict(v_type=kvs.KVS_TYPE_Q8_0), dict(max_q_head=6), dict(max_rows=257),
                                dict(max_q_head=0)])
def test_unsupported_configs_refused(kw):
    with pytest.raises(kvs.KVSError) as e:
        kvs.kvs_query_sizes(_cfg(**kw))
    assert e.value.status == kvs.KVS_ERR_UNSUPPORTED


def _plan_cfg(arena_slots, host_bytes=None, ws=None, **kw):
    c = _cfg(**kw)
    pb, hb, amin, wmin = kvs.kvs_query_sizes(c)
    c.flags = kvs.KVS_FLAG_PLAN_ONLY
    c.arena, c.workspace = 1 << 20, 1 << 30
    c.arena_bytes = arena_slots * pb
    c.workspace_bytes = wmin if ws is None else ws
    c.host_bytes = hb if host_bytes is None else host_bytes
    return c


@pytest.mark.parametrize("kw", [dict(max_rows=11, head_dim=128), dict(max_rows=11, page_tokens=32),
                                dict(max_rows=49, max_verify_rows=49)])
def test_wide_split_k_calls_size_the_workspace_for_every_row(kw):
    """More than 64 rows x heads per kv head without the tensor-core path (another
    head dim or page size, or fp32 queries): row groups on the split-K kernel, with
    one partial per (page, row, head) and one query-fragment area per row group."""
    cfg = _cfg(**kw)
    pb, hb, amin, wmin = kvs.kvs_query_sizes(cfg)
    D, Hk, Hq = cfg.head_dim, cfg.n_kv_head, cfg.max_q_head
    pages = -(-cfg.max_tokens // cfg.page_tokens)
    rows = cfg.max_verify_rows or cfg.max_rows
    groups = -(-rows // (64 // (Hq // Hk)))
    qfrag = Hk * 8 * (D // 16) * 32 * 16
    assert wmin >= 256 + groups * qfrag + pages * Hq * rows * (D + 2) * 4


def test_create_refusals():
    with pytest.raises(kvs.KVSError) as e:
        kvs.kvs_create(_plan_cfg(2 * 4 + 7))  # below tails + ring
    assert e.value.status == kvs.KVS_ERR_ARENA
    with pytest.raises(kvs.KVSError) as e:
        kvs.kvs_create(_plan_cfg(64, ws=1024))
    assert e.value.status == kvs.KVS_ERR_ARENA
    with pytest.raises(kvs.KVSError) as e:
        kvs.kvs_create(_plan_cfg(64, host_bytes=1024))
    assert e.value.status == kvs.KVS_ERR_HOST
    c = _plan_cfg(64)
    c.arena = (1 << 20) + 16
    with pytest.raises(kvs.KVSError) as e:
        kvs.kvs_create(c)
    assert e.value.status == kvs.KVS_ERR_INVALID
    ctx = kvs.kvs_create(_plan_cfg(64))
    kvs.kvs_destroy(ctx)


# ------------------------------------------------------------ trace model

class HB:
    """Happens-before over a logged two-stream trace (vector clocks)."""

    def __init__(self, trace, n_streams=None):
        self.ops = []
        if n_streams is None:
            n_streams = 1 + max([t["stream"] for t in trace] + [0])
        vc = [[0] * n_streams for _ in range(n_streams)]
        ev = {}
        for t in trace:
            s = t["stream"]
            vc[s][s] += 1
            if t["op"] == kvs.KVS_OP_WAIT:
                if t["event"] in ev:
                    e = ev[t["event"]]
                    vc[s] = [max(a, b) for a, b in zip(vc[s], e)]
            mine = list(vc[s])
            if t["op"] == kvs.KVS_OP_RECORD:
                ev[t["event"]] = mine
            self.ops.append(dict(t, vc=mine))

    @staticmethod
    def before(a, b):
        s = a["stream"]
        return a is not b and a["vc"][s] <= b["vc"][s]


def check_trace(st, n_q_head, fixed_ring=True):
    """Validate fences and coverage of every READ in a plan-only trace.  With fixed_ring, the
    trace must not span a ring resize: reads from the final ring's slots must come from fills."""
    hb = HB(st.trace())
    ops = hb.ops
    first_ring, n_ring = st.ring_info()
    P, Hk = st.geom["P"], st.geom["Hk"]
    writers = {}   # slot -> list of (op index, page) that put a page in that slot
    for i, o in enumerate(ops):
        if o["op"] in (kvs.KVS_OP_FILL, kvs.KVS_OP_POOL_LOAD, kvs.KVS_OP_MOVE, kvs.KVS_OP_WRITE):
            writers.setdefault(o["b"], []).append(i)
    n_reads = 0
    for i, o in enumerate(ops):
        if o["op"] != kvs.KVS_OP_READ:
            continue
        n_reads += 1
        slot, page, layer = o["b"], o["a"], o["layer"]
        ws = [j for j in writers.get(slot, []) if ops[j]["a"] == page and ops[j]["layer"] == layer
              and HB.before(ops[j], o)]
        assert ws, f"read of page {page} layer {layer} from slot {slot} with no prior write of it"
        src = ws[-1]
        # every other write into the slot is ordered before src or after this read
        for j in writers[slot]:
            if j == src:
                continue
            wj = ops[j]
            if wj["op"] == kvs.KVS_OP_WRITE and wj["a"] == page and wj["layer"] == layer:
                continue  # appending rows to the same page (same stream, ordered)
            assert HB.before(wj, ops[src]) or HB.before(o, wj), (
                f"slot {slot} overwritten (op {j}) between its fill (op {src}) and read (op {i})")
        if fixed_ring and first_ring <= slot < first_ring + n_ring:
            assert ops[src]["op"] == kvs.KVS_OP_FILL
    # every ring fill of a published page is ordered after that publish
    pubs = {}
    for i, o in enumerate(ops):
        if o["op"] == kvs.KVS_OP_PUBLISH:
            pubs.setdefault((o["layer"], o["a"]), []).append(i)
        if o["op"] in (kvs.KVS_OP_FILL, kvs.KVS_OP_POOL_LOAD) and (o["layer"], o["a"]) in pubs:
            assert HB.before(ops[pubs[(o["layer"], o["a"])][-1]], o)
    return ops, n_reads


def _reads_of_attend(ops, layer):
    return [(o["a"], o["c"]) for o in ops if o["op"] == kvs.KVS_OP_READ and o["layer"] == layer]


def _plan_stream(L, Hk, P, max_tokens, ring, chunk, arena_slots, G=6, R=6, lanes=1):
    return kvs.KVStream(page_tokens=P, n_layers=L, n_kv_head=Hk, head_dim=128, max_q_head=G * Hk,
                        max_rows=R, max_tokens=max_tokens, ring_slots=ring, chunk_pages=chunk,
                        arena_slots=arena_slots, plan_only=True, lanes=lanes)


@pytest.mark.parametrize("seed", range(16))
def test_scheduler_random_residency_fences_and_coverage(seed):
    rng = np.random.default_rng(seed)
    P = int(rng.choice([32, 64, 128, 256]))
    L = int(rng.integers(1, 5))
    Hk = int(rng.integers(1, 3))
    ring = int(rng.integers(1, 17))
    chunk = int(rng.integers(0, ring + 1))
    lanes = int(rng.integers(1, 9))
    T0 = int(rng.integers(1, 40 * P))
    max_tokens = T0 + 4 * P
    npages_max = math.ceil(max_tokens / P)
    st = _plan_stream(L, Hk, P, max_tokens, ring, chunk, 2 * L + ring + L * npages_max, lanes=lanes)
    for l in range(L):
        kvs.kvs_append(st.ctx, l, None, None, T0)
        n = math.ceil(T0 / P)
        st.set_residency(l, (rng.random(n) < rng.random()).astype(np.uint8))
    # decode-like loop: per step append one row to every layer and attend it,
    # prefetching the next layer at random points
    T = T0
    for step in range(int(rng.integers(1, 4))):
        order = list(range(L))
        if rng.random() < 0.5:
            st.prefetch(0)
        for l in order:
            kvs.kvs_append(st.ctx, l, None, None, 1)
            if l + 1 < L and rng.random() < 0.7:
                st.prefetch(l)  # announce l first: layers are attended in announcement order
                st.prefetch(l + 1)
            R = int(rng.integers(1, 4))
            st.attend_plan(l, R, 6 * Hk, T + 1 - R)
        T += 1
    ops, n_reads = check_trace(st, 6 * Hk)
    assert n_reads > 0
    # coverage: each attend reads every page 0..last exactly once per kv head
    # (checked on the last attend of each layer)
    st.close()


def test_scheduler_coverage_exact_and_streamed_pages():
    P, L, Hk, T = 64, 3, 2, 64 * 20 + 7
    st = _plan_stream(L, Hk, P, T + P, 3, 1, 2 * L + 3 + 200)
    for l in range(L):
        kvs.kvs_append(st.ctx, l, None, None, T)
        mask = np.zeros(21, np.uint8)
        mask[l::3] = 1
        st.set_residency(l, mask)
    n_before = len(st.trace())
    st.prefetch(0)
    for l in range(L):
        if l + 1 < L:
            st.prefetch(l + 1)
        st.attend_plan(l, 1, 6 * Hk, T - 1)
    ops, _ = check_trace(st, 6 * Hk)
    new = ops[n_before:]
    for l in range(L):
        reads = sorted(_reads_of_attend(new, l))
        expect = sorted((p, g) for p in range(21) for g in range(Hk))
        assert reads == expect
    s = st.stats()
    tails = 2
    streamed = sum(21 - tails - len(range(l, 19, 3)) for l in range(L))
    assert s["h2d_pages"] == streamed
    assert s["ring_recycles"] == streamed - 3
    st.close()


def test_prefetch_order_enforced_and_state_errors():
    st = _plan_stream(3, 1, 64, 64 * 10, 4, 1, 6 + 4 + 30)
    for l in range(3):
        kvs.kvs_append(st.ctx, l, None, None, 64 * 8)
    st.prefetch(1)
    with pytest.raises(kvs.KVSError) as e:
        st.attend_plan(0, 1, 6, 64 * 8 - 1)
    assert e.value.status == kvs.KVS_ERR_STATE
    with pytest.raises(kvs.KVSError) as e:
        st.set_residency(0, np.ones(8, np.uint8))
    assert e.value.status == kvs.KVS_ERR_STATE
    with pytest.raises(kvs.KVSError) as e:
        st.truncate(1, 10)
    assert e.value.status == kvs.KVS_ERR_STATE
    with pytest.raises(kvs.KVSError) as e:
        st.set_ring_slots(2)
    assert e.value.status == kvs.KVS_ERR_STATE
    st.attend_plan(1, 1, 6, 64 * 8 - 1)
    st.attend_plan(0, 1, 6, 64 * 8 - 1)
    with pytest.raises(kvs.KVSError) as e:
        st.attend_plan(0, 2, 6, 64 * 8 - 1)  # row beyond the appended length
    assert e.value.status == kvs.KVS_ERR_CAPACITY
    with pytest.raises(kvs.KVSError) as e:
        st.attend_plan(0, 7, 6, 0)
    assert e.value.status == kvs.KVS_ERR_UNSUPPORTED
    with pytest.raises(kvs.KVSError) as e:
        st.attend_plan(0, 1, 7, 0)  # more query heads than max_q_head
    assert e.value.status == kvs.KVS_ERR_INVALID
    with pytest.raises(kvs.KVSError) as e:
        st.attend_plan(0, 0, 6, 0)  # empty span
    assert e.value.status == kvs.KVS_ERR_INVALID
    with pytest.raises(kvs.KVSError) as e:
        st.attend_plan(3, 1, 6, 0)  # layer out of range
    assert e.value.status == kvs.KVS_ERR_INVALID
    n_ops = len(st.trace())
    for bad in ((0, 0, 6, 0), (3, 1, 6, 0), (0, 2, 6, 64 * 8 - 1)):
        with pytest.raises(kvs.KVSError):
            st.attend_plan(*bad)
    assert len(st.trace()) == n_ops  # a refused call enqueues nothing
    check_trace(st, 6)
    st.close()


def test_pool_capacity_refusal_changes_nothing():
    st = _plan_stream(2, 1, 64, 64 * 10, 2, 1, 4 + 2 + 5)  # pool of 5 slots
    for l in range(2):
        kvs.kvs_append(st.ctx, l, None, None, 64 * 9)
    st.set_residency(0, np.ones(4, np.uint8))
    with pytest.raises(kvs.KVSError) as e:
        st.set_residency(1, np.ones(7, np.uint8))
    assert e.value.status == kvs.KVS_ERR_CAPACITY
    assert st.stats()["pool_used"] == 4
    assert st.page_location(1, 0) == (0, -1)


def test_set_ring_slots_compacts_pool():
    st = _plan_stream(1, 1, 64, 64 * 40, 2, 1, 2 + 2 + 30)
    kvs.kvs_append(st.ctx, 0, None, None, 64 * 30)
    mask = np.zeros(30, np.uint8)
    mask[:20] = 1
    st.set_residency(0, mask)
    st.set_residency(0, np.r_[np.zeros(10, np.uint8), np.ones(10, np.uint8)])
    st.set_ring_slots(18, 3)
    first, n = st.ring_info()
    assert n == 18
    for p in range(10, 20):
        kind, slot = st.page_location(0, p)
        assert kind == 2 and 2 <= slot < first
    with pytest.raises(kvs.KVSError) as e:
        st.set_ring_slots(25)
    assert e.value.status == kvs.KVS_ERR_CAPACITY
    st.attend_plan(0, 1, 6, 64 * 30 - 1)
    check_trace(st, 6)


def test_injected_fill_fault_is_reported_and_recoverable():
    st = _plan_stream(1, 1, 64, 64 * 20, 2, 1, 2 + 2 + 20)
    kvs.kvs_append(st.ctx, 0, None, None, 64 * 12)
    st.inject(kvs.KVS_FAULT_FILL_ENQUEUE, 2)
    with pytest.raises(kvs.KVSError) as e:
        st.prefetch(0)
    assert e.value.status == kvs.KVS_ERR_INJECTED
    st.inject(kvs.KVS_FAULT_NONE, 0)
    st.attend_plan(0, 1, 6, 64 * 12 - 1)
    ops, _ = check_trace(st, 6)
    reads = sorted(_reads_of_attend(ops, 0))
    assert reads == [(p, 0) for p in range(12)]


def test_sync_timeout_is_reported():
    import time
    st = _plan_stream(1, 1, 64, 640, 2, 1, 2 + 2 + 4)
    st.inject(kvs.KVS_FAULT_SYNC_STALL, 1)
    t0 = time.monotonic()
    with pytest.raises(kvs.KVSError) as e:
        st.sync(60)
    assert e.value.status == kvs.KVS_ERR_TIMEOUT
    assert time.monotonic() - t0 >= 0.055
    st.inject(kvs.KVS_FAULT_NONE, 0)
    st.sync(60)


def test_page_boundary_append_with_pending_prefetch_keeps_plan():
    """A tail page pushed out while its layer has a pending plan goes to the pool."""
    P = 32
    st = _plan_stream(2, 1, P, P * 12, 2, 1, 4 + 2 + 12)
    for l in range(2):
        kvs.kvs_append(st.ctx, l, None, None, P * 6)  # pages 4, 5 in tail slots
    st.prefetch(0)
    st.prefetch(1)
    kvs.kvs_append(st.ctx, 0, None, None, 1)  # page 6 starts: page 4 leaves its tail slot
    assert st.page_location(0, 4)[0] == 2
    st.attend_plan(0, 1, 6, P * 6)
    kvs.kvs_append(st.ctx, 1, None, None, 1)
    st.attend_plan(1, 1, 6, P * 6)
    ops, _ = check_trace(st, 6)
    for l in range(2):
        reads = sorted(p for p, g in _reads_of_attend(ops, l))
        assert reads == list(range(7))


@pytest.mark.parametrize("seed", range(6))
def test_prefill_scheduling_fences_and_split_coverage(seed):
    """Prefill attends (more than 64 query rows per kv head) read every page of
    every split once, with each split's ring chunks ready before its launch."""
    rng = np.random.default_rng(100 + seed)
    P, L, Hk, R = 64, 2, 1, 40
    ring = int(rng.integers(4, 12))
    split = int(rng.integers(1, ring + 1))
    T0 = int(rng.integers(R + 1, 30 * P))
    st = kvs.KVStream(page_tokens=P, n_layers=L, n_kv_head=Hk, head_dim=256, max_q_head=6 * Hk, max_rows=R,
                      max_tokens=T0 + R, ring_slots=ring, chunk_pages=int(rng.integers(1, ring + 1)),
                      arena_slots=2 * L + ring + 64, plan_only=True, lanes=int(rng.integers(1, 4)),
                      prefill_split_pages=split)
    for l in range(L):
        kvs.kvs_append(st.ctx, l, None, None, T0 + R)
        st.set_residency(l, (rng.random(math.ceil((T0 + R) / P)) < 0.4).astype(np.uint8))
    st.prefetch(0)
    st.prefetch(1)
    for l in range(L):
        n0 = len(st.trace())
        kvs.kvs_attend(st.ctx, l, None, kvs.KVS_F16, R, 6 * Hk, T0, 1.0, None, None)
        reads = sorted(p for p, g in _reads_of_attend(st.trace()[n0:], l))
        assert reads == list(range(math.ceil((T0 + R) / P)))
    check_trace(st, 6 * Hk)


@pytest.mark.parametrize("ring,chunk", [(8, 2), (24, 2), (32, 5)])
def test_prefill_default_split_scheduling_and_coverage(ring, chunk):
    """The default prefill split (24 pages, at most the ring) over a 60-page
    context with a random 40% resident: every page of every split is read once
    and each split's ring chunks are ready before its launch."""
    rng = np.random.default_rng(ring)
    P, L, Hk, R = 64, 1, 1, 40
    T0 = 60 * P - R
    st = kvs.KVStream(page_tokens=P, n_layers=L, n_kv_head=Hk, head_dim=256, max_q_head=6 * Hk, max_rows=R,
                      max_tokens=T0 + R, ring_slots=ring, chunk_pages=chunk, arena_slots=2 * L + ring + 64,
                      plan_only=True, lanes=2)
    kvs.kvs_append(st.ctx, 0, None, None, T0 + R)
    st.set_residency(0, (rng.random(60) < 0.4).astype(np.uint8))
    st.prefetch(0)
    n0 = len(st.trace())
    kvs.kvs_attend(st.ctx, 0, None, kvs.KVS_F16, R, 6 * Hk, T0, 1.0, None, None)
    reads = sorted(p for p, g in _reads_of_attend(st.trace()[n0:], 0))
    assert reads == list(range(60))
    check_trace(st, 6 * Hk)


def test_load_host_pages_installs_pages_and_streams_them():
    """Encoded pages written into the host history are attended like any streamed page."""
    P, Hk, D, maxp = 64, 1, 128, 12
    pb = Hk * P * D * 13 // 8
    host = np.zeros(2 * maxp * pb, np.uint8)
    st = kvs.KVStream(page_tokens=P, n_layers=2, n_kv_head=Hk, head_dim=D, max_q_head=6, max_rows=6,
                      max_tokens=P * maxp, ring_slots=2, chunk_pages=1, arena_slots=4 + 2 + 12,
                      plan_only=True, host=host)
    assert st.page_bytes == pb
    kvs.kvs_append(st.ctx, 0, None, None, 2 * P)  # pages 0, 1 sit in the tail slots
    st.set_residency(0, np.array([1, 0], np.uint8))  # page 0 wanted resident
    rng = np.random.default_rng(5)
    pages = rng.integers(0, 256, size=3 * pb, dtype=np.uint8)
    st.load_host_pages(0, 2, pages)
    assert st.length(0) == 5 * P
    for i in range(3):
        assert np.array_equal(st.read_host_page(0, 2 + i), pages[i * pb:(i + 1) * pb])
    # the tail slots gave up their pages: page 0 to the pool (mask), page 1 to the host
    assert st.page_location(0, 0)[0] == 2
    assert st.page_location(0, 1) == (0, -1)
    for p in range(2, 5):
        assert st.page_location(0, p) == (0, -1)
    # refusals change nothing
    for bad_first in (4, 6):
        with pytest.raises(kvs.KVSError) as e:
            st.load_host_pages(0, bad_first, pages[:pb])
        assert e.value.status == kvs.KVS_ERR_INVALID
    with pytest.raises(kvs.KVSError) as e:
        st.load_host_pages(0, 5, np.zeros(8 * pb, np.uint8))  # 13 pages > 12
    assert e.value.status == kvs.KVS_ERR_CAPACITY
    st.prefetch(0)
    with pytest.raises(kvs.KVSError) as e:
        st.load_host_pages(1, 0, pages[:pb])
    assert e.value.status == kvs.KVS_ERR_STATE
    assert st.length(0) == 5 * P and st.length(1) == 0
    # one new row starts page 5 in a tail slot; every page is read once, loaded ones through the ring
    st.attend_plan(0, 1, 6, 5 * P - 1)
    kvs.kvs_append(st.ctx, 0, None, None, 1)
    st.attend_plan(0, 1, 6, 5 * P)
    ops, _ = check_trace(st, 6)
    fills = {o["a"] for o in ops if o["op"] == kvs.KVS_OP_FILL and o["layer"] == 0}
    assert {1, 2, 3, 4} <= fills and 0 not in fills
    reads = [o["a"] for o in ops if o["op"] == kvs.KVS_OP_READ]
    assert sorted(reads) == sorted(list(range(5)) + list(range(6)))
    # a history that is not page-aligned refuses a load
    kvs.kvs_append(st.ctx, 1, None, None, 10)
    with pytest.raises(kvs.KVSError) as e:
        st.load_host_pages(1, 0, pages[:pb])
    assert e.value.status == kvs.KVS_ERR_INVALID
    st.close()


def test_noalloc_refusals_come_before_any_device_work():
    """Every refusal of kvs_attend_pages_noalloc is decided on the host from its
    arguments (the pointers below are never dereferenced)."""
    fake = 1 << 20
    pb = 4 * 256 * 256 * 13 // 8
    base = dict(pages=fake, pages_bytes=8 * pb, page_slots=np.arange(8, dtype=np.uint32), page_tokens=256,
                n_kv_head=4, head_dim=256, q=fake, q_dtype=kvs.KVS_F32, n_rows=6, n_q_head=24,
                pos0=256 * 8 - 6, scale=0.1, out=fake, lse=None, stream=0)
    cases = [
        (dict(page_tokens=48), kvs.KVS_ERR_UNSUPPORTED),
        (dict(head_dim=96), kvs.KVS_ERR_UNSUPPORTED),
        (dict(q_dtype=7), kvs.KVS_ERR_INVALID),
        (dict(n_q_head=26), kvs.KVS_ERR_INVALID),
        (dict(n_rows=0), kvs.KVS_ERR_INVALID),
        (dict(n_rows=11, pos0=0), kvs.KVS_ERR_UNSUPPORTED),  # 6 heads x 11 rows > 64
        (dict(q=None), kvs.KVS_ERR_INVALID),
        (dict(out=None), kvs.KVS_ERR_INVALID),
        (dict(pos0=2**63 - 3), kvs.KVS_ERR_INVALID),  # pos0 + n_rows wraps
        (dict(pos0=2**64 - 6), kvs.KVS_ERR_INVALID),
        (dict(pos0=256 * 8 - 5), kvs.KVS_ERR_CAPACITY),  # the last row reaches a ninth page
        (dict(page_slots=np.r_[np.arange(7), 8].astype(np.uint32)), kvs.KVS_ERR_INVALID),  # slot 8 outside
        (dict(page_slots=np.zeros(300, np.uint32), pos0=300 * 256 - 6), kvs.KVS_ERR_CAPACITY),  # > 32 MiB
    ]
    for over, want in cases:
        a = dict(base, **over)
        with pytest.raises(kvs.KVSError) as e:
            kvs.kvs_attend_pages_noalloc(a["pages"], a["pages_bytes"], a["page_slots"], a["page_tokens"],
                                         a["n_kv_head"], a["head_dim"], a["q"], a["q_dtype"], a["n_rows"],
                                         a["n_q_head"], a["pos0"], a["scale"], a["out"], a["lse"], a["stream"])
        assert e.value.status == want, (over, e.value)
        assert kvs.kvs_last_error(None)


@pytest.mark.parametrize("R,G,lanes", [(20, 6, 1), (49, 6, 2), (9, 8, 1)])
def test_wide_split_k_row_groups_read_every_chunk_before_release(R, G, lanes):
    """A call wider than 64 rows x heads per kv head on the split-K kernel: every
    row group reads each ring chunk after its fill and before any refill of its
    slots (the fence model), and each (page, kv head) is read once per group."""
    P, Hk, T = 64, 2, 64 * 11 + 30
    st = kvs.KVStream(page_tokens=P, n_layers=2, n_kv_head=Hk, head_dim=128, max_q_head=G * Hk, max_rows=R,
                      max_tokens=T, ring_slots=2, chunk_pages=1, arena_slots=4 + 2 + 24, plan_only=True,
                      lanes=lanes, max_verify_rows=R)
    for l in range(2):
        kvs.kvs_append(st.ctx, l, None, None, T)
        mask = np.zeros(12, np.uint8)
        mask[l::2] = 1
        st.set_residency(l, mask)
    st.prefetch(0)
    st.prefetch(1)
    for l in range(2):
        st.attend_plan(l, R, G * Hk, T - R)
    ops, _ = check_trace(st, G * Hk)
    groups = -(-R // (64 // G))
    for l in range(2):
        reads = _reads_of_attend(ops, l)
        assert sorted(set(reads)) == [(p, g) for p in range(12) for g in range(Hk)]
        assert all(reads.count(x) == groups for x in set(reads)), l
    # the split-K kernel is not used beyond max_verify_rows
    with pytest.raises(kvs.KVSError) as e:
        small = kvs.KVStream(page_tokens=P, n_layers=1, n_kv_head=Hk, head_dim=128, max_q_head=G * Hk, max_rows=R,
                             max_tokens=T, ring_slots=2, chunk_pages=1, arena_slots=2 + 2 + 12, plan_only=True,
                             max_verify_rows=max(1, R // 2))
        kvs.kvs_append(small.ctx, 0, None, None, T)
        small.attend_plan(0, R, G * Hk, T - R)
    assert e.value.status == kvs.KVS_ERR_UNSUPPORTED


def test_lease_holds_a_layers_pages_and_guards_the_ring():
    """A complete-layer lease: the layer's nonresident pages are loaded once into
    slots taken off the ring, its attends read no ring chunk, the other layers'
    refills never write a leased slot, a page leaving its tail fills a spare
    leased slot, and release gives the whole ring back."""
    P = 64
    st = _plan_stream(3, 1, P, P * 14, 8, 2, 6 + 8 + 6)  # 6 tail slots, pool of 6, ring of 8
    for l in range(3):
        kvs.kvs_append(st.ctx, l, None, None, P * 10 + 5)  # pages 0..10, tail pages 9, 10
    st.set_residency(2, np.array([1, 1, 1], np.uint8))
    first, n = st.ring_info()
    with pytest.raises(kvs.KVSError) as e:
        st.lease_acquire(2, 2)  # 6 nonresident pages + 2 spares = the whole ring
    assert e.value.status == kvs.KVS_ERR_CAPACITY
    st.lease_acquire(2, 1)  # pages 3..8 + one spare: 7 slots, the ring keeps 1
    assert st.lease_info() == (2, 7, 1) and st.ring_info() == (first, 1)
    leased = set(range(first + 1, first + 8))
    for p in range(3, 9):
        kind, slot = st.page_location(2, p)
        assert kind == 3 and slot in leased
    for call in (lambda: st.lease_acquire(0), lambda: st.set_residency(0, np.ones(2, np.uint8)),
                 lambda: st.set_ring_slots(4)):
        with pytest.raises(kvs.KVSError) as e:
            call()
        assert e.value.status == kvs.KVS_ERR_STATE
    n0 = len(st.trace())
    for _ in range(2):  # a catch-up / draft phase of the leased layer, the others streaming
        for l in (2, 0, 1):
            st.attend_plan(l, 1, 6, P * 10 + 4)
    # page 11 starts: page 9 leaves its tail slot into the spare; page 12: page 10 goes to the host
    kvs.kvs_append(st.ctx, 2, None, None, 2 * P)
    assert st.page_location(2, 9)[0] == 3 and st.page_location(2, 10) == (0, -1)
    assert st.lease_info() == (2, 7, 0)
    st.attend_plan(2, 1, 6, P * 12 + 4)
    ops = st.trace()[n0:]
    fills = [o for o in ops if o["op"] == kvs.KVS_OP_FILL]
    assert fills and not any(o["b"] in leased for o in fills)
    assert {o["a"] for o in fills if o["layer"] == 2} == {10}  # only the page the lease could not hold
    st.lease_release()
    assert st.lease_info() == (-1, 0, 0) and st.ring_info() == (first, 8)
    assert st.page_location(2, 5) == (0, -1)
    with pytest.raises(kvs.KVSError) as e:
        st.lease_release()
    assert e.value.status == kvs.KVS_ERR_STATE
    st.attend_plan(2, 1, 6, P * 12 + 4)
    ops, n_reads = check_trace(st, 6, fixed_ring=False)
    late = [o["a"] for o in st.trace()[n0:] if o["op"] == kvs.KVS_OP_FILL and o["layer"] == 2]
    assert set(range(3, 11)) <= set(late)  # after release the layer streams again
    st.close()


def test_observe_on_a_plan_only_context_reports_only_the_context_length():
    st = _plan_stream(2, 1, 64, 64 * 10, 2, 1, 4 + 2 + 4)
    kvs.kvs_append(st.ctx, 0, None, None, 200)
    kvs.kvs_append(st.ctx, 1, None, None, 333)
    st.attend_plan(1, 1, 6, 332)
    o = st.observe(reset=True)
    assert (o.context_tokens, o.streamed_reads, o.ready_misses, o.ring_occupancy, o.copy_busy) == (333, 0, 0, 0.0, 0.0)
    s = st.stats()
    assert s["observed_reads"] == 0 and s["copy_busy"] == 0.0


def test_timeline_in_a_plan_only_context_stamps_nothing():
    st = _plan_stream(2, 2, 64, 64 * 6, 2, 1, 2 * 2 + 2 + 12)
    for l in range(2):
        kvs.kvs_append(st.ctx, l, None, None, 64 * 6)
    assert kvs.kvs_timeline_begin(st.ctx, None, 16) == kvs.KVS_OK
    st.prefetch(0)
    st.attend_plan(0, 1, 12, 64 * 6 - 1)
    assert kvs.kvs_timeline_end(st.ctx) == kvs.KVS_OK
    recs, dropped = kvs.kvs_timeline_read(st.ctx, 16)
    assert recs == [] and dropped == 0
    st.close()
