"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Bit-exact: page bytes written by the KV writer (host history, tail slots,
resident pool, ring slots) against the oracle's page encoder.
Within tolerance (max over (row, head) of max_d |gpu - oracle| / max_d |oracle|
<= 1e-3, lse absolute error <= 1e-4): attention outputs for decode (1 row) and
span verify (2..6 causal rows) over every page size and head dim served.
Bitwise: streamed output equals all-resident output for any residency, ring
size and chunk size (the split-K partition never depends on them).
"""
import math

import numpy as np
import pytest

import oracle
import synth
from host_streamed_paged_gb300 import kvs
from kvs_testutil import (SEED, append_rows, attend, check_parity, history, make_stream,
                          oracle_ref, queries, rel_err)

pytestmark = pytest.mark.gpu


def _fill(st, L, T, Hk, D, pieces=None, seed=SEED):
    hist = []
    for l in range(L):
        k, v = history(seed, l, T, Hk, D)
        append_rows(st, l, k, v, pieces)
        hist.append((k, v))
    return hist


# ------------------------------------------------------------ bit-exact layout

@pytest.mark.parametrize("P,Hk,D,T", [(64, 2, 64, 64 * 3 + 29), (256, 4, 256, 256 * 3 + 100),
                                      (128, 1, 128, 128 * 4), (32, 3, 128, 32 * 7 + 1)])
def test_append_pages_bit_exact(P, Hk, D, T):
    st = make_stream(P, 1, Hk, D, Hk, 1, T + P, ring=2, chunk=1)
    k, v = history(SEED, 0, T, Hk, D)
    pieces = [1, 2, 37, P // 2 + 3, 3 * P // 2]  # irregular sizes crossing page boundaries
    assert sum(pieces) < T
    pieces.append(T - sum(pieces))
    append_rows(st, 0, k, v, pieces)
    st.flush()
    st.sync()
    ref = oracle.QuantKV(k, v)
    npages = math.ceil(T / P)
    for p in range(npages):
        want = ref.encode_page(P, p)
        assert np.array_equal(st.read_host_page(0, p), want), f"host page {p}"
        kind, slot = st.page_location(0, p)
        if kind:
            assert np.array_equal(st.read_slot(slot), want), f"device page {p} (kind {kind})"
    # resident pool copies
    st.set_residency(0, np.ones(npages, np.uint8))
    st.sync()
    for p in range(npages):
        kind, slot = st.page_location(0, p)
        assert kind in (1, 2)
        assert np.array_equal(st.read_slot(slot), ref.encode_page(P, p))


def test_ring_slots_bit_exact():
    P, Hk, D, T, ring = 64, 2, 128, 64 * 12 + 5, 5
    st = make_stream(P, 1, Hk, D, Hk, 1, T + P, ring=ring, chunk=1)
    k, v = history(SEED, 0, T, Hk, D)
    append_rows(st, 0, k, v)
    mask = np.zeros(12, np.uint8)
    mask[[0, 3, 4, 9]] = 1
    st.set_residency(0, mask)
    st.prefetch(0)
    st.sync()
    first, n = st.ring_info()
    streamed = [p for p in range(13) if st.page_location(0, p)[0] == 0]
    ref = oracle.QuantKV(k, v)
    for i, p in enumerate(streamed[:ring]):
        assert np.array_equal(st.read_slot(first + i), ref.encode_page(P, p)), f"ring slot {i} page {p}"
    # consume the plan
    q = queries(SEED, 0, 1, Hk, D)
    attend(st, 0, q, T - 1, 0.1)


# ------------------------------------------------------------ attention parity

def test_decode_small_config_all_resident():
    """1 row at context 4096, 8 q / 2 kv heads, D 128, page 256, all 16 pages resident."""
    P, L, Hk, Hq, D, T = 256, 1, 2, 8, 128, 4096
    st = make_stream(P, L, Hk, D, Hq, 1, T, ring=2)
    (k, v), = _fill(st, L, T, Hk, D)
    st.set_residency(0, np.ones(16, np.uint8))
    q = queries(SEED, 0, 1, Hq, D)
    scale = 1.0 / math.sqrt(D)
    out, lse = attend(st, 0, q, T - 1, scale)
    ro, rl = oracle_ref(k, v, q, T - 1, scale)
    check_parity(out, lse, ro, rl)


@pytest.mark.parametrize("P,D,Hk,G,R,T", [
    (256, 256, 4, 6, 1, 256 * 5 + 77),
    (256, 256, 4, 6, 2, 256 * 4 + 1),
    (256, 256, 4, 6, 4, 256 * 6),
    (256, 256, 4, 6, 6, 256 * 3 + 250),
    (256, 128, 2, 4, 3, 256 * 4 + 9),
    (128, 128, 2, 8, 8, 128 * 9 + 3),
    (64, 64, 3, 2, 5, 64 * 11 + 60),
    (32, 256, 1, 6, 6, 32 * 20 + 7),
    (64, 256, 2, 1, 1, 64 * 3 + 2),
    (256, 64, 1, 16, 4, 256 * 2 + 255),
])
def test_attention_parity_geometries(P, D, Hk, G, R, T):
    Hq = G * Hk
    st = make_stream(P, 1, Hk, D, Hq, R, T, ring=3, chunk=1)
    (k, v), = _fill(st, 1, T, Hk, D)
    npages = math.ceil(T / P)
    mask = (synth.u64(SEED + 1, synth.tag("mask", P, D), npages) % 2).astype(np.uint8)
    st.set_residency(0, mask)
    q = queries(SEED, 0, R, Hq, D)
    scale = 1.0 / math.sqrt(D)
    out, lse = attend(st, 0, q, T - R, scale)
    ro, rl = oracle_ref(k, v, q, T - R, scale)
    check_parity(out, lse, ro, rl)
    s = st.stats()
    assert s["h2d_pages"] > 0 or mask.sum() + 2 >= npages


def test_rows_inside_history_and_across_page_boundary():
    """Rows whose positions straddle a page boundary, not at the end of the history."""
    P, D, Hk, G, R = 64, 128, 2, 6, 5
    T = 64 * 6
    st = make_stream(P, 1, Hk, D, G * Hk, R, T, ring=2, chunk=1)
    (k, v), = _fill(st, 1, T, Hk, D)
    q = queries(SEED, 3, R, G * Hk, D)
    for pos0 in (62, 127, 0, 200):
        out, lse = attend(st, 0, q, pos0, 0.07)
        ro, rl = oracle_ref(k, v, q, pos0, 0.07)
        check_parity(out, lse, ro, rl)


def test_single_token_history():
    P, D, Hk, G = 256, 256, 4, 6
    st = make_stream(P, 1, Hk, D, G * Hk, 1, 512, ring=1)
    (k, v), = _fill(st, 1, 1, Hk, D)
    q = queries(SEED, 0, 1, G * Hk, D)
    out, lse = attend(st, 0, q, 0, 1 / 16)
    ro, rl = oracle_ref(k, v, q, 0, 1 / 16)
    check_parity(out, lse, ro, rl)


def test_constant_values_weights_sum_to_one():
    P, D, Hk, G, R, T = 128, 256, 2, 6, 3, 128 * 5 + 17
    st = make_stream(P, 1, Hk, D, G * Hk, R, T, ring=2, chunk=1)
    k = synth.normal(SEED, synth.tag("K1"), (T, Hk, D))
    v = np.ones((T, Hk, D), np.float32)
    append_rows(st, 0, k, v)
    q = queries(SEED, 0, R, G * Hk, D) * np.float32(4.0)
    out, _ = attend(st, 0, q, T - R, 0.0625)
    # o and l are summed along different fp32 paths (tensor-core MMA for o, warp
    # shuffles for l) from f16 hi/lo parts (2^-22 relative per product); over
    # ~700 keys that leaves a few 1e-6, far below any misweighted key (>= 1e-3)
    assert np.abs(out - 1.0).max() <= 1e-5


def test_f16_queries():
    P, D, Hk, G, R, T = 256, 256, 4, 6, 2, 256 * 3 + 5
    import torch
    st = make_stream(P, 1, Hk, D, G * Hk, R, T, ring=2)
    (k, v), = _fill(st, 1, T, Hk, D)
    q = queries(SEED, 0, R, G * Hk, D).astype(np.float16).astype(np.float32)  # the f16 values exactly
    out, lse = attend(st, 0, q, T - R, 1 / 16, dtype=torch.float16)
    ro, rl = oracle_ref(k, v, q, T - R, 1 / 16)
    check_parity(out, lse, ro, rl)


# ------------------------------------------------------------ invariants

# Resident pages go through the multi-tile attention launch, ring chunks
# through the one-tile-per-CTA launch: the output must not depend on which.
@pytest.mark.parametrize("lanes,R,D,P,dma", [(1, 3, 256, 64, False), (3, 3, 256, 64, False), (8, 1, 256, 64, False),
                                             (4, 6, 256, 128, False), (2, 5, 128, 64, False),
                                             (5, 2, 64, 256, False), (4, 6, 256, 64, True), (1, 1, 128, 64, True)])
def test_streamed_equals_resident_bitwise(lanes, R, D, P, dma):
    L, Hk, G = 2, 2, 6
    T = P * (640 // P) + 33
    Hq = G * Hk
    st = make_stream(P, L, Hk, D, Hq, R, T, ring=8, chunk=2, lanes=lanes, dma=dma)
    hist = _fill(st, L, T, Hk, D)
    npages = math.ceil(T / P)
    qs = [queries(SEED, l, R, Hq, D) for l in range(L)]
    for l in range(L):
        st.set_residency(l, np.ones(npages, np.uint8))
    base = [attend(st, l, qs[l], T - R, 0.0625) for l in range(L)]
    for l in range(L):
        ro, rl = oracle_ref(*hist[l], qs[l], T - R, 0.0625)
        check_parity(*base[l], ro, rl)
    rng = np.random.default_rng(5)
    for ring, chunk in [(1, 1), (2, 1), (3, 2), (8, 4), (5, 5)]:
        for l in range(L):
            st.set_residency(l, (rng.random(npages) < 0.4).astype(np.uint8))
        st.set_ring_slots(ring, chunk)
        st.stats(reset=True)
        st.prefetch(0)
        for l in range(L):
            if l + 1 < L:
                st.prefetch(l + 1)
            out, lse = attend(st, l, qs[l], T - R, 0.0625)
            assert np.array_equal(out, base[l][0]), f"ring {ring} chunk {chunk} layer {l}"
            assert np.array_equal(lse, base[l][1])
        s = st.stats()
        assert s["h2d_pages"] > 0 and (s["h2d_pages"] <= ring or s["ring_recycles"] > 0)


def test_page_size_changes_result_only_within_tolerance():
    D, Hk, G, R, T = 128, 2, 4, 2, 1500
    k, v = history(SEED, 0, T, Hk, D)
    q = queries(SEED, 0, R, G * Hk, D)
    outs = []
    for P in (64, 128, 256):
        st = make_stream(P, 1, Hk, D, G * Hk, R, T, ring=2, chunk=1)
        append_rows(st, 0, k, v)
        outs.append(attend(st, 0, q, T - R, 0.09))
        st.close()
    ro, rl = oracle_ref(k, v, q, T - R, 0.09)
    for o, l in outs:
        check_parity(o, l, ro, rl)
    assert rel_err(outs[0][0], outs[2][0].astype(np.float64)) <= 1e-5


def test_decode_loop_with_appends_and_page_starts():
    """Decode steps that append a row per layer, cross page boundaries and prefetch ahead."""
    P, L, Hk, G, D = 32, 3, 2, 6, 128
    T0, steps = 32 * 4 + 30, 6
    Hq = G * Hk
    st = make_stream(P, L, Hk, D, Hq, 1, T0 + steps, ring=2, chunk=1, pool_pages=8)
    full = [history(SEED, l, T0 + steps, Hk, D) for l in range(L)]
    for l in range(L):
        append_rows(st, l, full[l][0][:T0], full[l][1][:T0])
        st.set_residency(l, np.array([1, 0, 1, 0, 0], np.uint8))
    for s in range(steps):
        T = T0 + s + 1
        st.prefetch(0)
        for l in range(L):
            append_rows(st, l, full[l][0][T - 1:T], full[l][1][T - 1:T])
            if l + 1 < L:
                st.prefetch(l + 1)
            q = queries(SEED, 100 * s + l, 1, Hq, D)
            out, lse = attend(st, l, q, T - 1, 0.088)
            ro, rl = oracle_ref(full[l][0][:T], full[l][1][:T], q, T - 1, 0.088)
            check_parity(out, lse, ro, rl)


def test_truncate_then_reappend():
    P, D, Hk, G = 64, 128, 2, 6
    T = 64 * 3 + 10
    st = make_stream(P, 1, Hk, D, G * Hk, 1, T + 64, ring=2)
    k, v = history(SEED, 0, T, Hk, D)
    append_rows(st, 0, k, v)
    st.truncate(0, T - 20)
    k2, v2 = history(SEED + 7, 0, 20, Hk, D)
    append_rows(st, 0, k2, v2)
    kk = np.concatenate([k[:T - 20], k2])
    vv = np.concatenate([v[:T - 20], v2])
    q = queries(SEED, 0, 1, G * Hk, D)
    out, lse = attend(st, 0, q, T - 1, 0.1)
    ro, rl = oracle_ref(kk, vv, q, T - 1, 0.1)
    check_parity(out, lse, ro, rl)
    st.flush()
    st.sync()
    ref = oracle.QuantKV(kk, vv)
    for p in range(4):
        assert np.array_equal(st.read_host_page(0, p), ref.encode_page(P, p))


def test_sync_timeout_injection_on_gpu_context():
    st = make_stream(64, 1, 1, 64, 1, 1, 640, ring=1)
    st.inject(kvs.KVS_FAULT_SYNC_STALL, 1)
    with pytest.raises(kvs.KVSError) as e:
        st.sync(30)
    assert e.value.status == kvs.KVS_ERR_TIMEOUT
    st.inject(kvs.KVS_FAULT_NONE, 0)
    st.sync(1000)


def test_device_wait_that_gives_up_is_reported_and_recovered():
    """A bounded pipeline wait in the attention kernel that gives up (made to
    give up at once by the test hook) leaves NaN outputs, kvs_sync reports
    KVS_ERR_CUDA, and the next attend is correct again."""
    import torch
    P, D, Hk, G, T = 64, 128, 2, 6, 64 * 9 + 13
    st = make_stream(P, 1, Hk, D, G * Hk, 1, T, ring=2, chunk=1)
    k, v = history(SEED, 0, T, Hk, D)
    append_rows(st, 0, k, v)
    mask = np.zeros(math.ceil(T / P), np.uint8)
    mask[::2] = 1
    st.set_residency(0, mask)
    st.sync()
    q = queries(SEED, 0, 1, G * Hk, D)
    st.inject(kvs.KVS_FAULT_DEVICE_WAIT, 1)
    qt = torch.from_numpy(q).cuda()
    torch.cuda.synchronize()
    out, lse = st.attend(0, qt, T - 1, 0.1)
    with pytest.raises(kvs.KVSError) as e:
        st.sync()
    assert e.value.status == kvs.KVS_ERR_CUDA and "timed out" in str(e.value)
    torch.cuda.synchronize()
    assert np.isnan(out.cpu().numpy()).all() and np.isnan(lse.cpu().numpy()).all()
    st.inject(kvs.KVS_FAULT_NONE, 0)
    out, lse = attend(st, 0, q, T - 1, 0.1)
    ro, rl = oracle_ref(k, v, q, T - 1, 0.1)
    check_parity(out, lse, ro, rl)


def test_loaded_host_pages_stream_and_match_the_oracle():
    """Pages encoded elsewhere (here by the oracle, following the documented
    layout) installed with kvs_load_host_pages, half of them made resident,
    the rest streamed through a 2-slot ring."""
    P, D, Hk, G = 256, 256, 4, 6
    full, extra = 12, 70
    T = full * P + extra
    st = make_stream(P, 1, Hk, D, G * Hk, 2, T, ring=2, chunk=1)
    k, v = history(SEED, 3, T, Hk, D)
    ref = oracle.QuantKV(k[:full * P], v[:full * P])
    pages = np.concatenate([ref.encode_page(P, i) for i in range(full)])
    st.load_host_pages(0, 0, pages)
    append_rows(st, 0, k[full * P:], v[full * P:])
    for i in (0, 5, 11):
        assert np.array_equal(st.read_host_page(0, i), pages[i * st.page_bytes:(i + 1) * st.page_bytes])
    mask = np.zeros(full + 1, np.uint8)
    mask[1::2] = 1
    st.set_residency(0, mask)
    q = queries(SEED, 3, 2, G * Hk, D)
    out, lse = attend(st, 0, q, T - 2, 1.0 / math.sqrt(D))
    ro, rl = oracle_ref(k, v, q, T - 2, 1.0 / math.sqrt(D))
    check_parity(out, lse, ro, rl)
    assert st.stats()["h2d_pages"] >= full // 2


def _wide_case(R, T, mask_fn, ring=8, chunk=2, lanes=1, seed=SEED, P=256, D=256, Hk=4, G=6):
    st = kvs.KVStream(page_tokens=P, n_layers=1, n_kv_head=Hk, head_dim=D, max_q_head=G * Hk, max_rows=R,
                      max_tokens=T, ring_slots=ring, chunk_pages=chunk, lanes=lanes,
                      arena_slots=2 + ring + math.ceil(T / P), max_verify_rows=R)
    (k, v), = _fill(st, 1, T, Hk, D, seed=seed)
    st.set_residency(0, mask_fn(math.ceil(T / P)))
    q = queries(seed, 0, R, G * Hk, D)
    out, lse = attend(st, 0, q, T - R, 1.0 / math.sqrt(D))
    return st, k, v, q, out, lse


@pytest.mark.parametrize("R,T,P,D", [(49, 256 * 12 + 70, 256, 256), (20, 128 * 9 + 5, 128, 128)])
def test_wide_fp32_verify_row_groups_match_the_oracle(R, T, P, D):
    """An fp32 span of R causal rows (49 at 6 query heads per kv head: 294 rows x
    heads) runs on the split-K kernel as row groups of 10 rows; half the pages
    stream through the ring, every group reading each chunk before its release."""
    st, k, v, q, out, lse = _wide_case(R, T, lambda n: (np.arange(n) % 2 == 1).astype(np.uint8), P=P, D=D)
    ro, rl = oracle_ref(k, v, q, T - R, 1.0 / math.sqrt(D))
    check_parity(out, lse, ro, rl)
    assert st.stats()["h2d_pages"] > 0


@pytest.mark.parametrize("R,T,P,D", [(32, 128 * 9 + 5, 128, 128), (32, 64 * 20 + 3, 64, 64)])
def test_wide_fp32_verify_warp_per_pair_combine(R, T, P, D):
    """32 rows x 24 query heads = 768 (row, head) pairs over at most 21 one-page
    splits: the log-sum-exp combine runs one warp per pair (its D 256 form is
    reached by the 49-row case above); a third of the pages stream."""
    st, k, v, q, out, lse = _wide_case(R, T, lambda n: (np.arange(n) % 3 == 1).astype(np.uint8), P=P, D=D)
    ro, rl = oracle_ref(k, v, q, T - R, 1.0 / math.sqrt(D))
    check_parity(out, lse, ro, rl)
    assert st.stats()["h2d_pages"] > 0


def test_wide_fp32_verify_streamed_equals_resident_bitwise():
    R, T = 49, 256 * 16 + 3
    base = _wide_case(R, T, lambda n: np.ones(n, np.uint8))
    rng = np.random.default_rng(11)
    for ring, chunk, lanes in [(8, 2, 1), (6, 3, 2)]:
        st, _, _, _, out, lse = _wide_case(R, T, lambda n: (rng.random(n) < 0.5).astype(np.uint8),
                                           ring=ring, chunk=chunk, lanes=lanes)
        assert st.stats()["h2d_pages"] > 0
        assert np.array_equal(out, base[4]) and np.array_equal(lse, base[5]), (ring, chunk, lanes)
        st.close()


def test_wide_fp32_verify_full_size_sampled_rows():
    """49 fp32 rows at context 163840 (the span-verify stack's geometry), 400
    resident pages, the rest through an 8-slot ring; six sampled rows."""
    R, P = 49, 256
    T = 163840 + R
    st, k, v, q, out, lse = _wide_case(R, T, lambda n: (np.arange(n) < 400).astype(np.uint8), chunk=1, lanes=4)
    qkv = oracle.QuantKV(k, v)
    for r in (0, 9, 10, 30, 47, 48):
        ro, rl = qkv.attend(q[r:r + 1], T - R + r, 1.0 / 16)
        check_parity(out[r:r + 1], lse[r:r + 1], ro, rl)
    assert st.stats()["h2d_pages"] > 0


def test_lease_draft_phase_matches_the_oracle_and_resident_bitwise():
    """Layer 1 is a second history (an attached draft layer) leased into the ring:
    it appends and attends three draft rows while layer 0 keeps streaming through
    the rest of the ring; every output matches the oracle, and matches the same
    calls on an all-resident context bitwise."""
    import torch
    P, D, Hk, G = 64, 128, 2, 6
    Hq = G * Hk
    T0, T1 = 64 * 20 + 7, 64 * 6 + 10
    k0, v0 = history(SEED, 0, T0, Hk, D)
    k1, v1 = history(SEED, 1, T1 + 3, Hk, D)
    kinds = []

    def run(leased):
        st = make_stream(P, 2, Hk, D, Hq, 1, T0 + 64, ring=8, chunk=1, pool_pages=None if not leased else 4)
        append_rows(st, 0, k0, v0)
        append_rows(st, 1, k1[:T1], v1[:T1])
        if not leased:
            st.set_residency(0, np.ones(21, np.uint8))
            st.set_residency(1, np.ones(8, np.uint8))
        else:
            st.lease_acquire(1, 1)  # pages 0..4 of layer 1 + one spare
            kinds.append([st.page_location(1, p)[0] for p in range(7)])
        outs = []
        for i in range(3):
            kn = torch.from_numpy(np.ascontiguousarray(k1[T1 + i:T1 + i + 1])).cuda()
            vn = torch.from_numpy(np.ascontiguousarray(v1[T1 + i:T1 + i + 1])).cuda()
            torch.cuda.synchronize()
            st.append(1, kn, vn)
            q = queries(SEED, 10 + i, 1, Hq, D)
            outs.append(attend(st, 1, q, T1 + i, 0.1))
            q0 = queries(SEED, 20 + i, 1, Hq, D)
            outs.append(attend(st, 0, q0, T0 - 1, 0.1))
        stats = st.stats()
        if leased:
            st.lease_release()
            outs.append(attend(st, 1, queries(SEED, 30, 1, Hq, D), T1 + 2, 0.1))
        st.close()
        return outs, stats

    base, _ = run(False)
    got, stats = run(True)
    assert kinds[0][:5] == [3] * 5 and kinds[0][5:] == [1, 1]
    assert stats["h2d_pages"] > 0  # layer 0 streamed through the smaller ring
    for i in range(3):
        ro, rl = oracle_ref(k1[:T1 + i + 1], v1[:T1 + i + 1], queries(SEED, 10 + i, 1, Hq, D), T1 + i, 0.1)
        check_parity(*got[2 * i], ro, rl)
        ro, rl = oracle_ref(k0, v0, queries(SEED, 20 + i, 1, Hq, D), T0 - 1, 0.1)
        check_parity(*got[2 * i + 1], ro, rl)
    for g, b in zip(got, base):
        assert np.array_equal(g[0], b[0]) and np.array_equal(g[1], b[1])
    ro, rl = oracle_ref(k1[:T1 + 3], v1[:T1 + 3], queries(SEED, 30, 1, Hq, D), T1 + 2, 0.1)
    check_parity(*got[6], ro, rl)


def test_observation_counts_every_streamed_read_and_stays_in_range():
    P, D, Hk, G, T = 256, 256, 4, 6, 256 * 24 + 9
    st = make_stream(P, 2, Hk, D, G * Hk, 1, T, ring=8, chunk=2, pool_pages=8)
    for l in range(2):
        k, v = history(SEED, l, T, Hk, D)
        append_rows(st, l, k, v)
    st.set_residency(0, (np.arange(25) < 4).astype(np.uint8))
    st.sync()
    st.observe(reset=True)
    st.stats(reset=True)
    q = queries(SEED, 0, 1, G * Hk, D)
    for l in range(2):
        attend(st, l, q, T - 1, 1 / 16)
    o = st.observe(reset=False)
    chunks = st.stats()["ring_chunks"]
    assert o.streamed_reads == chunks > 0 and o.ready_misses <= o.streamed_reads
    assert 0.0 <= o.ring_occupancy <= 1.0 and 0.0 < o.copy_busy <= 1.0
    assert o.context_tokens == T
    s = st.stats()
    assert s["observed_reads"] == chunks and s["copy_busy"] == o.copy_busy
    # counters accumulate until a reset, also over a step graph's replays
    import torch
    q_t = torch.from_numpy(q).cuda()
    bufs = [(torch.empty((1, G * Hk, D), device="cuda"), torch.empty((1, G * Hk), device="cuda")) for _ in range(2)]
    torch.cuda.synchronize()
    st.graph_begin()
    st.prefetch(0)
    st.prefetch(1)
    for l in range(2):
        st.attend(l, q_t, T - 1, 1 / 16, out=bufs[l][0], lse=bufs[l][1])
    st.graph_end()
    st.graph_launch()
    st.graph_launch()
    o2 = st.observe(reset=True)
    assert o2.streamed_reads == 3 * chunks
    assert st.observe().streamed_reads == 0


@pytest.mark.parametrize("link_gbs", [0.0, 1e4])
def test_residency_policy_drives_a_streamed_stack_in_closed_loop(link_gbs):
    """kvs_policy_step chooses the resident/ring split of a fixed 96-slot budget
    from the library's own observations (kvs_observe), step after step, and the
    decisions are applied with kvs_set_ring_slots / kvs_set_residency; the
    outputs match the oracle on sampled layers after every change.  With a link
    ceiling (link_gbs, here far above any refill rate) the observation's refill
    bytes and interval are measured and the link always has room."""
    import torch
    P, D, Hk, G, L, T = 256, 256, 4, 6, 4, 256 * 64
    Hq = G * Hk
    budget = 96
    npages = T // P
    st = kvs.KVStream(page_tokens=P, n_layers=L, n_kv_head=Hk, head_dim=D, max_q_head=Hq, max_rows=1,
                      max_tokens=T, ring_slots=8, chunk_pages=2, lanes=2, arena_slots=2 * L + budget)
    hist = _fill(st, L, T, Hk, D)
    cfg = kvs.kvs_policy_config(page_tokens=P, n_layers=L, budget_slots=budget, min_ring_slots=8,
                                max_ring_slots=64, step_slots=8, hold_steps=2, miss_grow=0.25,
                                copy_busy_max=0.98, occupancy_shrink=0.05, link_gbs=link_gbs)
    state = kvs.kvs_policy_state()
    qs = [queries(SEED, 50 + l, 1, Hq, D) for l in range(L)]
    q_dev = [torch.from_numpy(q).cuda() for q in qs]
    torch.cuda.synchronize()
    applied = []
    for step in range(6):
        st.prefetch(0)
        outs = []
        for l in range(L):
            if l + 1 < L:
                st.prefetch(l + 1)
            outs.append(st.attend(l, q_dev[l], T - 1, 1 / 16))
        st.sync()
        obs = st.observe(reset=True)
        assert obs.streamed_reads > 0 and obs.ready_misses <= obs.streamed_reads
        # every accounted read's chunk moved whole pages, within a measured interval
        assert obs.interval_ns > 0 and obs.copy_bytes > 0 and obs.copy_bytes % st.page_bytes == 0
        if step in (0, 5) or applied and applied[-1][0] == step - 1:
            for l in (0, L - 1):
                ro, rl = oracle_ref(*hist[l], qs[l], T - 1, 1 / 16)
                check_parity(outs[l][0].cpu().numpy(), outs[l][1].cpu().numpy(), ro, rl)
        state, dec = kvs.kvs_policy_step(cfg, state, obs)
        assert 8 <= dec.ring_slots <= 64 and dec.resident_slots == budget - dec.ring_slots
        if dec.changed or step == 0:
            per = min(npages - 2, dec.resident_pages_per_layer)
            for l in range(L):
                st.set_residency(l, np.zeros(npages, np.uint8))
            st.set_ring_slots(dec.ring_slots, max(1, dec.ring_slots // 4))
            for l in range(L):
                m = np.zeros(npages, np.uint8)
                m[:per] = 1
                st.set_residency(l, m)
            st.sync()
            applied.append((step, dec.ring_slots, dec.reason))
            assert st.stats()["ring_slots"] == dec.ring_slots
    assert applied and applied[0][2] == kvs.KVS_POLICY_INIT


# ------------------------------------------------------------ full-size samples

@pytest.mark.parametrize("chunk,lanes", [(2, 1), (4, 2), (2, 3)])
def test_decode_stack_sampled_layers_full_size(chunk, lanes):
    """Context 32768, 24 q / 4 kv heads, D 256, page 256, half the pages resident
    (seeded), 8-slot ring: the launch configurations of the decode benchmark,
    checked on three layers against the oracle."""
    P, Hk, Hq, D, T, L = 256, 4, 24, 256, 32768, 3
    st = make_stream(P, L, Hk, D, Hq, 1, T, ring=8, chunk=chunk, pool_pages=L * 64, lanes=lanes)
    hist = _fill(st, L, T, Hk, D)
    for l in range(L):
        # 62 seeded pages + the two tail pages = half of the 128 pages resident
        res = synth.choose(SEED + 1, synth.tag("resident", l), 126, 62)
        mask = np.zeros(128, np.uint8)
        mask[res] = 1
        st.set_residency(l, mask)
    st.prefetch(0)
    for l in range(L):
        if l + 1 < L:
            st.prefetch(l + 1)
        q = queries(SEED, l, 1, Hq, D)
        out, lse = attend(st, l, q, T - 1, 1 / 16)
        ro, rl = oracle_ref(*hist[l], q, T - 1, 1 / 16)
        check_parity(out, lse, ro, rl)
    s = st.stats()
    assert s["h2d_pages"] == L * 64 and s["ring_recycles"] > 0


def test_span_verify_full_size_one_layer():
    """6 causal rows at 163840..163845, 24 q / 4 kv heads, D 256, 400 resident
    pages (prefix), the rest through an 8-slot ring."""
    P, Hk, Hq, D, R = 256, 4, 24, 256, 6
    T = 163840 + R
    st = make_stream(P, 1, Hk, D, Hq, R, T, ring=8, chunk=2, pool_pages=400)
    (k, v), = _fill(st, 1, T, Hk, D)
    mask = np.zeros(641, np.uint8)
    mask[:400] = 1
    st.set_residency(0, mask)
    q = queries(SEED, 0, R, Hq, D)
    out, lse = attend(st, 0, q, T - R, 1 / 16)
    ro, rl = oracle_ref(k, v, q, T - R, 1 / 16)
    check_parity(out, lse, ro, rl)
    assert st.stats()["h2d_pages"] == 641 - 400 - 2  # the last two pages sit in tail slots


@pytest.mark.parametrize("R,resident", [(1, 0.5), (4, 0.0)])
def test_long_context_full_size_one_layer(R, resident):
    """Context 262144 (1024 pages of 256), 24 q / 4 kv heads, D 256: a resident
    prefix, the rest through a large ring in 32-page chunks on 4 lanes, as the
    long-context benchmark runs it; every row against the oracle."""
    P, Hk, Hq, D = 256, 4, 24, 256
    T = 262144 + R - 1
    npages = -(-T // P)
    n_res = int(resident * npages)
    st = make_stream(P, 1, Hk, D, Hq, R, T, ring=1009, chunk=32, pool_pages=max(n_res, 1), lanes=4)
    (k, v), = _fill(st, 1, T, Hk, D)
    mask = np.zeros(npages, np.uint8)
    mask[:n_res] = 1
    st.set_residency(0, mask)
    q = queries(SEED, 0, R, Hq, D)
    out, lse = attend(st, 0, q, T - R, 1 / 16)
    ro, rl = oracle_ref(k, v, q, T - R, 1 / 16)
    check_parity(out, lse, ro, rl)
    assert st.stats()["h2d_pages"] == npages - n_res - 2


def test_prefill_full_size_sampled_rows():
    """A 256-row fp16 prefill chunk at context 131072 (tensor-core path), half
    the pages resident as a prefix and the rest through the 8-slot ring;
    eight sampled rows against the oracle (each row at its own position)."""
    import torch
    P, Hk, G, D, R = 256, 4, 6, 256, 256
    Hq = G * Hk
    T = 131072 + R
    npages = -(-T // P)
    st = kvs.KVStream(page_tokens=P, n_layers=1, n_kv_head=Hk, head_dim=D, max_q_head=Hq, max_rows=R,
                      max_tokens=T, ring_slots=8, chunk_pages=2, lanes=2, arena_slots=2 + 8 + npages)
    (k, v), = _fill(st, 1, T, Hk, D)
    mask = np.zeros(npages, np.uint8)
    mask[:npages // 2] = 1
    st.set_residency(0, mask)
    q = queries(SEED, 0, R, Hq, D).astype(np.float16).astype(np.float32)  # the f16 values exactly
    out, lse = attend(st, 0, q, T - R, 1 / 16, dtype=torch.float16)
    qkv = oracle.QuantKV(k, v)
    for r in (0, 1, 63, 64, 127, 128, 200, 255):
        ro, rl = qkv.attend(q[r:r + 1], T - R + r, 1 / 16)
        check_parity(out[r:r + 1], lse[r:r + 1], ro, rl)
    assert st.stats()["h2d_pages"] > 0


def test_step_graph_replay_matches_eager_bitwise():
    """A decode step captured with kvs_graph_* replays to the eager step's exact outputs."""
    import torch
    P, L, Hk, G, D = 64, 3, 2, 6, 128
    Hq, T0 = G * Hk, 64 * 8 - 1  # the appended row completes a page: the step publishes it
    st = make_stream(P, L, Hk, D, Hq, 1, T0 + 1, ring=4, chunk=2, pool_pages=3 * 8)
    for l in range(L):
        k, v = history(SEED, l, T0, Hk, D)
        append_rows(st, l, k, v)
        st.set_residency(l, np.array([1, 0, 0, 1, 0, 1, 0, 0], np.uint8))
    kn = torch.from_numpy(np.stack([history(SEED + 9, l, 1, Hk, D)[0] for l in range(L)])).cuda()
    vn = torch.from_numpy(np.stack([history(SEED + 9, l, 1, Hk, D)[1] for l in range(L)])).cuda()
    q = torch.from_numpy(np.stack([queries(SEED, l, 1, Hq, D) for l in range(L)])).cuda()
    out = torch.zeros((L, 1, Hq, D), device="cuda")
    lse = torch.zeros((L, 1, Hq), device="cuda")
    torch.cuda.synchronize()

    def step():
        st.prefetch(0)
        for l in range(L):
            kvs.kvs_append(st.ctx, l, kn[l], vn[l], 1)
            if l + 1 < L:
                st.prefetch(l + 1)
            kvs.kvs_attend(st.ctx, l, q[l], kvs.KVS_F32, 1, Hq, T0, 0.088, out[l], lse[l])
            st.truncate(l, T0)

    step()
    st.sync()
    eager = (out.cpu().numpy().copy(), lse.cpu().numpy().copy())
    out.zero_()
    lse.zero_()
    torch.cuda.synchronize()
    st.graph_begin()
    step()
    st.graph_end()
    assert st.stats()["graph_kernels"] > 0
    for _ in range(3):
        out.zero_()
        torch.cuda.synchronize()
        st.graph_launch()
        st.sync()
        assert np.array_equal(out.cpu().numpy(), eager[0])
        assert np.array_equal(lse.cpu().numpy(), eager[1])
    st.graph_destroy()
    # host-issued work after the replays still sees consistent events and ring
    step()
    st.sync()
    assert np.array_equal(out.cpu().numpy(), eager[0])
    assert st.stats()["d2h_pages"] >= 2 * L


# ------------------------------------------------------------ tensor-core prefill

def _prefill_case(R, T, mask_fn=None, ring=8, chunk=2, lanes=1, split=8, seed=SEED, P=256):
    import torch
    Hk, G, D = 4, 6, 256
    Hq = G * Hk
    st = kvs.KVStream(page_tokens=P, n_layers=1, n_kv_head=Hk, head_dim=D, max_q_head=Hq, max_rows=R,
                      max_tokens=T, ring_slots=ring, chunk_pages=chunk, lanes=lanes,
                      arena_slots=2 + ring + math.ceil(T / P), prefill_split_pages=split)
    (k, v), = _fill(st, 1, T, Hk, D, seed=seed)
    npages = math.ceil(T / P)
    if mask_fn is not None:
        st.set_residency(0, mask_fn(npages))
    q = queries(seed, 0, R, Hq, D).astype(np.float16).astype(np.float32)  # the f16 values exactly
    out, lse = attend(st, 0, q, T - R, 1 / 16, dtype=torch.float16)
    return st, k, v, q, out, lse


@pytest.mark.parametrize("R,T", [(256, 256 * 6 + 37), (256, 256 * 4), (100, 256 * 3 + 200), (11, 256 * 2 + 5)])
def test_prefill_tensor_core_parity(R, T):
    st, k, v, q, out, lse = _prefill_case(R, T, mask_fn=lambda n: np.ones(n, np.uint8))
    ro, rl = oracle_ref(k, v, q, T - R, 1 / 16)
    check_parity(out, lse, ro, rl)
    assert st.stats()["h2d_pages"] == 0


@pytest.mark.parametrize("P,R,T,split,ring", [(64, 256, 64 * 13 + 17, 3, 4), (64, 200, 64 * 9, 2, 2),
                                               (128, 130, 128 * 7 + 50, 2, 4)])
def test_prefill_small_pages_and_ragged_splits(P, R, T, split, ring):
    """Pages of 64 and 128 tokens: a 128-key block of the tensor-core kernel
    spans two pages, and with an odd number of 64-token pages per split it
    runs past the split's end (those keys are masked); half the pages stream."""
    st, k, v, q, out, lse = _prefill_case(R, T, mask_fn=lambda n: (np.arange(n) % 2 == 0).astype(np.uint8),
                                          ring=ring, chunk=1, split=split, P=P)
    ro, rl = oracle_ref(k, v, q, T - R, 1 / 16)
    check_parity(out, lse, ro, rl)
    assert st.stats()["h2d_pages"] > 0


def test_prefill_streamed_equals_resident_bitwise():
    R, T = 256, 256 * 20 + 100
    base = _prefill_case(R, T, mask_fn=lambda n: np.ones(n, np.uint8))
    ro, rl = oracle_ref(base[1], base[2], base[3], T - R, 1 / 16)
    check_parity(base[4], base[5], ro, rl)
    rng = np.random.default_rng(3)
    for ring, chunk, lanes in [(8, 2, 1), (8, 3, 2), (12, 4, 1)]:
        st, _, _, _, out, lse = _prefill_case(
            R, T, mask_fn=lambda n: (rng.random(n) < 0.5).astype(np.uint8), ring=ring, chunk=chunk, lanes=lanes)
        assert st.stats()["h2d_pages"] > 0
        assert np.array_equal(out, base[4]) and np.array_equal(lse, base[5]), (ring, chunk, lanes)
        st.close()


def test_timeline_records_every_launch_and_reads_follow_their_copies():
    """The launch timeline of a streamed decode step: every stamped launch ran
    (start <= end), the kinds match the step's work, and the k-th ring-chunk
    read starts only after the k-th ring refill has ended (the ready fence,
    observed on the device clock)."""
    P, Hk, G, D, L = 64, 2, 6, 128, 2
    T = 64 * 12 + 5
    Hq = G * Hk
    st = make_stream(P, L, Hk, D, Hq, 1, T + 1, ring=4, chunk=1, pool_pages=L * 4, lanes=2)
    hist = _fill(st, L, T, Hk, D)
    npages = math.ceil(T / P)
    for l in range(L):
        mask = np.zeros(npages, np.uint8)
        mask[[1, 4, 7]] = 1
        st.set_residency(l, mask)
    st.sync()
    st.timeline_begin(4096)
    st.prefetch(0)
    outs = []
    for l in range(L):
        if l + 1 < L:
            st.prefetch(l + 1)
        q = queries(SEED, l, 1, Hq, D)
        outs.append((q, attend(st, l, q, T - 1, 0.09)))
    st.timeline_end()
    recs, dropped = st.timeline_read()
    assert dropped == 0 and recs
    for r in recs:
        assert 0 < r["start_ns"] <= r["end_ns"], r
    kinds = [r["kind"] for r in recs]
    assert kinds.count("combine") == L and kinds.count("qprep") == L
    fills = [r for r in recs if r["kind"] == "fill"]
    reads = [r for r in recs if r["kind"] == "read_ring"]
    assert len(fills) == len(reads) == st.stats()["ring_chunks"] > 0
    for f, r in zip(fills, reads):
        assert (f["layer"], f["pages"]) == (r["layer"], r["pages"])
        assert r["start_ns"] >= f["end_ns"], (f, r)
    for l, (q, (o, lse)) in enumerate(outs):
        check_parity(o, lse, *oracle_ref(*hist[l], q, T - 1, 0.09))
