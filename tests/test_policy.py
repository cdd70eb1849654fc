"""Adaptive residency policy (kvs_policy_step): a pure host function, tested on CPU.

The pages (Adaptive KV Streaming for llama.cpp V2, "KV data movement and attention" and "Logical
KV layout, policy, and physical execution"; Adaptive KV Streaming for llama.cpp, "Adaptive KV
streaming") fix what the policy reads and what it may do: it proposes a resident/ring split of a
fixed budget from the context length and from feedback (reads that waited on copies, ring fill,
copy-stream load), changes it only on consistent evidence, and keeps resident space as large as
the budget allows.  They give no thresholds, so the
tests check the rules the C header states, not particular numbers.
"""
import numpy as np
import pytest

from host_streamed_paged_gb300 import kvs

P, L = 256, 64


def cfg(**kw):
    base = dict(page_tokens=P, n_layers=L, budget_slots=5041, min_ring_slots=8, max_ring_slots=0,
                step_slots=8, hold_steps=3, miss_grow=0.05, copy_busy_max=0.9, occupancy_shrink=0.5)
    base.update(kw)
    return kvs.kvs_policy_config(**base)


def obs(ctx=262144, reads=100, misses=0, occ=0.9, busy=0.5):
    return kvs.kvs_policy_observation(context_tokens=ctx, streamed_reads=reads, ready_misses=misses,
                                      ring_occupancy=occ, copy_busy=busy)


def state(ring=0, grow=0, shrink=0, steps=0):
    return kvs.kvs_policy_state(ring_slots=ring, grow_run=grow, shrink_run=shrink, steps=steps)


def run(c, s, observations):
    out = []
    for o in observations:
        s, d = kvs.kvs_policy_step(c, s, o)
        out.append((s, d))
    return out


def test_whole_history_fits_keeps_smallest_ring():
    # 64 layers x 64 pages = 4096 <= 5041 - 8: everything resident, even right after a larger ring
    s, d = kvs.kvs_policy_step(cfg(), state(ring=200), obs(ctx=64 * P, misses=50))
    assert (d.ring_slots, d.reason, d.changed) == (8, kvs.KVS_POLICY_FITS, 1)
    assert d.pages_per_layer == 64 and d.resident_pages_per_layer == 64
    assert s.grow_run == 0 and s.shrink_run == 0 and s.steps == 1


def test_fit_boundary_is_exact():
    # need == budget - min_ring fits; one page more does not
    c = cfg(n_layers=1, budget_slots=100, min_ring_slots=4)
    _, d = kvs.kvs_policy_step(c, state(ring=4), obs(ctx=96 * P))
    assert d.reason == kvs.KVS_POLICY_FITS
    _, d = kvs.kvs_policy_step(c, state(ring=4), obs(ctx=96 * P + 1))
    assert d.reason == kvs.KVS_POLICY_HOLD and d.pages_per_layer == 97


def test_first_decision_when_streaming_is_smallest_ring():
    s, d = kvs.kvs_policy_step(cfg(), state(), obs(misses=90))
    assert (d.ring_slots, d.reason, d.changed) == (8, kvs.KVS_POLICY_INIT, 1)
    assert d.resident_slots == 5041 - 8
    assert d.resident_pages_per_layer == (5041 - 8) // L


def test_growth_needs_hold_steps_consecutive_misses():
    c = cfg(hold_steps=3)
    steps = run(c, state(ring=8), [obs(misses=10)] * 3)
    assert [d.ring_slots for _, d in steps] == [8, 8, 16]
    assert [d.reason for _, d in steps] == [kvs.KVS_POLICY_HOLD] * 2 + [kvs.KVS_POLICY_GROW]
    assert steps[-1][0].grow_run == 0  # a change restarts the count


def test_an_interruption_restarts_the_count():
    seq = [obs(misses=10), obs(misses=10), obs(misses=0), obs(misses=10), obs(misses=10)]
    steps = run(cfg(hold_steps=3), state(ring=8), seq)
    assert all(d.ring_slots == 8 for _, d in steps)
    assert steps[-1][0].grow_run == 2


def test_alternating_feedback_never_moves_the_split():
    grow, shrink = obs(misses=20, occ=0.9), obs(misses=0, occ=0.1)
    steps = run(cfg(hold_steps=2), state(ring=64), [grow, shrink] * 20)
    assert all(d.ring_slots == 64 and not d.changed for _, d in steps)


def test_saturated_copy_stream_blocks_growth():
    steps = run(cfg(hold_steps=1), state(ring=8), [obs(misses=50, busy=0.95)] * 5)
    assert all(d.ring_slots == 8 and d.reason == kvs.KVS_POLICY_HOLD for _, d in steps)


def test_miss_rate_threshold_is_strict():
    c = cfg(hold_steps=1, miss_grow=0.05)
    _, d = kvs.kvs_policy_step(c, state(ring=8), obs(reads=100, misses=5))  # 0.05: not above
    assert d.ring_slots == 8
    _, d = kvs.kvs_policy_step(c, state(ring=8), obs(reads=100, misses=6))
    assert d.ring_slots == 16


def test_idle_ring_shrinks_to_the_lower_bound():
    steps = run(cfg(hold_steps=2, step_slots=8), state(ring=24), [obs(misses=0, occ=0.2)] * 12)
    rings = [d.ring_slots for _, d in steps]
    assert rings[:6] == [24, 16, 16, 8, 8, 8]
    assert min(rings) == 8
    # at the bound nothing changes and the reason says so
    assert steps[-1][1].reason == kvs.KVS_POLICY_HOLD and not steps[-1][1].changed


def test_a_missed_read_blocks_shrinking():
    steps = run(cfg(hold_steps=1), state(ring=24), [obs(misses=1, occ=0.1)] * 4)
    assert all(d.ring_slots == 24 for _, d in steps)


def test_growth_stops_at_max_ring_and_budget():
    steps = run(cfg(hold_steps=1, step_slots=8, max_ring_slots=20), state(ring=8), [obs(misses=50)] * 5)
    assert [d.ring_slots for _, d in steps] == [16, 20, 20, 20, 20]
    c = cfg(n_layers=1, budget_slots=30, min_ring_slots=2, max_ring_slots=1000, hold_steps=1, step_slots=16)
    steps = run(c, state(ring=2), [obs(ctx=10000 * P, misses=50)] * 3)
    assert [d.ring_slots for _, d in steps] == [18, 30, 30]
    assert steps[-1][1].resident_slots == 0 and steps[-1][1].resident_pages_per_layer == 0


def test_split_outside_bounds_is_clamped():
    _, d = kvs.kvs_policy_step(cfg(max_ring_slots=32), state(ring=100), obs())
    assert (d.ring_slots, d.reason, d.changed) == (32, kvs.KVS_POLICY_CLAMP, 1)


def test_context_growth_hands_resident_space_to_the_ring_gradually():
    # misses appear once the streamed share outgrows the ring; each change is one step
    c = cfg(hold_steps=2, step_slots=8, max_ring_slots=256)
    s, rings = state(), []
    for t in range(0, 600):
        ctx = 16384 + 512 * t
        ppl = -(-ctx // P)
        streamed = max(0, ppl * L - (5041 - s.ring_slots))
        misses = 10 if streamed > 40 * max(s.ring_slots, 8) else 0
        s, d = kvs.kvs_policy_step(c, s, obs(ctx=ctx, misses=misses, occ=0.9, busy=0.6))
        rings.append(d.ring_slots)
    diffs = np.diff(rings)
    assert rings[0] == 8 and rings[-1] > rings[0]
    assert np.all(diffs >= 0) and np.all(diffs <= 8)


@pytest.mark.parametrize("bad", [
    dict(page_tokens=0), dict(n_layers=0), dict(budget_slots=0), dict(step_slots=0),
    dict(hold_steps=0), dict(min_ring_slots=0), dict(min_ring_slots=50, max_ring_slots=40),
    dict(min_ring_slots=6000), dict(miss_grow=1.5), dict(copy_busy_max=-0.1),
    dict(occupancy_shrink=float("nan")),
])
def test_invalid_config_is_refused(bad):
    with pytest.raises(kvs.KVSError) as e:
        kvs.kvs_policy_step(cfg(**bad), state(ring=8), obs())
    assert e.value.status == kvs.KVS_ERR_INVALID


@pytest.mark.parametrize("bad", [dict(occ=1.2), dict(busy=-0.5), dict(reads=3, misses=4)])
def test_invalid_observation_is_refused(bad):
    with pytest.raises(kvs.KVSError):
        kvs.kvs_policy_step(cfg(), state(ring=8), obs(**bad))


def test_null_pointers_are_refused():
    lib = kvs.load()
    assert lib.kvs_policy_step(None, None, None, None, None) == kvs.KVS_ERR_INVALID


def test_random_feedback_keeps_every_invariant():
    rng = np.random.default_rng(1234)
    for trial in range(20):
        c = cfg(budget_slots=int(rng.integers(64, 6000)), min_ring_slots=int(rng.integers(1, 16)),
                max_ring_slots=int(rng.integers(0, 400)), step_slots=int(rng.integers(1, 32)),
                hold_steps=int(rng.integers(1, 5)), n_layers=int(rng.integers(1, 80)))
        hi = min(c.max_ring_slots or c.budget_slots, c.budget_slots)
        if c.min_ring_slots > hi:
            continue
        s = state()
        for _ in range(300):
            reads = int(rng.integers(0, 200))
            o = obs(ctx=int(rng.integers(1, 400000)), reads=reads,
                    misses=int(rng.integers(0, reads + 1)) if rng.random() < 0.5 else 0,
                    occ=float(rng.random()), busy=float(rng.random()))
            prev = s.ring_slots
            s, d = kvs.kvs_policy_step(c, s, o)
            assert c.min_ring_slots <= d.ring_slots <= hi
            assert d.resident_slots == c.budget_slots - d.ring_slots
            assert d.ring_slots + d.resident_pages_per_layer * c.n_layers <= c.budget_slots
            assert d.resident_pages_per_layer <= d.pages_per_layer
            assert d.changed == int(d.ring_slots != prev)
            assert s.ring_slots == d.ring_slots
            if d.reason in (kvs.KVS_POLICY_GROW, kvs.KVS_POLICY_SHRINK):
                assert 0 < abs(d.ring_slots - prev) <= c.step_slots
            if d.reason == kvs.KVS_POLICY_HOLD:
                assert d.ring_slots == prev


def test_huge_context_does_not_overflow():
    _, d = kvs.kvs_policy_step(cfg(), state(ring=8), obs(ctx=2**64 - 1))
    assert d.pages_per_layer == (2**64 - 1) // P + 1 and d.reason == kvs.KVS_POLICY_HOLD


def test_policy_drives_a_plan_only_context():
    """Closed loop on the host scheduler: as the context grows, each decision is applied with
    kvs_set_residency / kvs_set_ring_slots; every read stays fenced and every attend covers its
    whole history."""
    from test_abi_plan import _plan_stream, _reads_of_attend, check_trace

    Pg, Ln, Hk, budget = 64, 2, 1, 40
    st = _plan_stream(Ln, Hk, Pg, Pg * 80, 2, 1, 2 * Ln + budget)
    c = cfg(page_tokens=Pg, n_layers=Ln, budget_slots=budget, min_ring_slots=2, max_ring_slots=16,
            step_slots=2, hold_steps=2)
    s, T, rings = state(), 0, []
    for l in range(Ln):
        kvs.kvs_append(st.ctx, l, None, None, 10 * Pg)
    T = 10 * Pg
    for step in range(50):
        for l in range(Ln):
            kvs.kvs_append(st.ctx, l, None, None, Pg)
        T += Pg
        ring_now = st.stats()["ring_slots"]
        ppl = -(-T // Pg)
        streamed = max(0, ppl - (budget - ring_now) // Ln)
        miss = 5 if streamed > 4 * ring_now else 0
        s, d = kvs.kvs_policy_step(c, s, obs(ctx=T, reads=20, misses=miss, occ=0.9 if miss else 0.3,
                                             busy=0.5))
        rings.append(d.ring_slots)
        n_mask = ppl - 2  # the two tail pages are device-readable without a pool slot
        mask = np.zeros(n_mask, np.uint8)
        mask[:min(d.resident_pages_per_layer, n_mask)] = 1
        if d.ring_slots > ring_now:  # shrink residency first, then hand slots to the ring
            for l in range(Ln):
                st.set_residency(l, mask)
            st.set_ring_slots(d.ring_slots)
        else:
            if d.ring_slots < ring_now:
                st.set_ring_slots(d.ring_slots)
            for l in range(Ln):
                st.set_residency(l, mask)
        n0 = len(st.trace())
        st.prefetch(0)
        for l in range(Ln):
            if l + 1 < Ln:
                st.prefetch(l + 1)
            st.attend_plan(l, 1, 6 * Hk, T - 1)
        new = st.trace()[n0:]
        for l in range(Ln):
            assert sorted(_reads_of_attend(new, l)) == [(p, 0) for p in range(ppl)]
    check_trace(st, 6 * Hk, fixed_ring=False)  # the ring boundary moves during the trace
    assert rings[0] == 2 and max(rings) > 2 and st.stats()["ring_slots"] == rings[-1]
    st.close()


def test_link_rate_decides_room_when_the_ceiling_is_given():
    """With link_gbs set, room on the link is the observed refill rate against
    copy_busy_max x link_gbs; copy_busy (which saturates at 1 when refills of
    several lanes overlap) is then not consulted."""
    c = cfg(hold_steps=1, copy_busy_max=0.9, link_gbs=200.0)
    miss = dict(reads=100, misses=90, occ=0.9, busy=1.0)
    slow = kvs.kvs_policy_observation(context_tokens=262144, streamed_reads=100, ready_misses=90,
                                      ring_occupancy=0.9, copy_busy=1.0,
                                      copy_bytes=120 * 10**6, interval_ns=10**6)   # 120 GB/s
    fast = kvs.kvs_policy_observation(context_tokens=262144, streamed_reads=100, ready_misses=90,
                                      ring_occupancy=0.9, copy_busy=1.0,
                                      copy_bytes=185 * 10**6, interval_ns=10**6)   # 185 GB/s >= 0.9 x 200
    _, d = kvs.kvs_policy_step(c, state(ring=64), slow)
    assert (d.ring_slots, d.reason) == (72, kvs.KVS_POLICY_GROW)
    _, d = kvs.kvs_policy_step(c, state(ring=64), fast)
    assert (d.ring_slots, d.reason) == (64, kvs.KVS_POLICY_HOLD)
    # without the ceiling the busy fraction decides: 1.0 is never below 0.9
    _, d = kvs.kvs_policy_step(cfg(hold_steps=1, copy_busy_max=0.9), state(ring=64), slow)
    assert d.reason == kvs.KVS_POLICY_HOLD
    # with the ceiling but no measured interval, the busy fraction decides too
    _, d = kvs.kvs_policy_step(c, state(ring=64), obs(**miss))
    assert d.reason == kvs.KVS_POLICY_HOLD


@pytest.mark.parametrize("bad", [-1.0, float("nan"), float("inf")])
def test_link_rate_must_be_a_finite_nonnegative_number(bad):
    o = obs()
    with pytest.raises(kvs.KVSError):
        kvs.kvs_policy_step(cfg(link_gbs=bad), state(ring=64), o)
