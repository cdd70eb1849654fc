"""GPU parity of the single-f16 operand mode of the split-K attention kernel.

With KVS_FLAG_F16_OPERANDS the query and the softmax weights times the Q4_0
scale enter the tensor cores as single f16 values instead of f16 hi + lo
pairs; the K and V codes are exact either way and accumulation stays fp32.
The output bar is unchanged (per (row, head) vector, max_d |gpu - oracle| /
max_d |oracle| <= 1e-3).  The log-sum-exp bar is 1e-3 here: a score carries
the query's f16 rounding (about 2^-12 relative per element, ~3e-4 on a score
of unit size), and with a single visible key lse is that score.
Streamed output still equals all-resident output bit for bit.
"""
import math

import numpy as np
import pytest

import oracle
import synth
from kvs_testutil import (SEED, append_rows, attend, check_parity, history, make_stream, oracle_ref,
                          queries)

pytestmark = pytest.mark.gpu

LSE_TOL_F16 = 1e-3


def _stream(*a, **kw):
    return make_stream(*a, f16_operands=True, **kw)


def _fill(st, L, T, Hk, D, seed=SEED):
    hist = []
    for l in range(L):
        k, v = history(seed, l, T, Hk, D)
        append_rows(st, l, k, v)
        hist.append((k, v))
    return hist


def _check(out, lse, ro, rl):
    return check_parity(out, lse, ro, rl, lse_tol=LSE_TOL_F16)


@pytest.mark.parametrize("P,D,Hk,G,R,T", [
    (256, 256, 4, 6, 1, 256 * 5 + 77),
    (256, 256, 4, 6, 6, 256 * 3 + 250),
    (256, 128, 2, 4, 3, 256 * 4 + 9),
    (128, 128, 2, 8, 8, 128 * 9 + 3),
    (64, 64, 3, 2, 5, 64 * 11 + 60),
    (32, 256, 1, 6, 6, 32 * 20 + 7),
    (256, 64, 1, 16, 4, 256 * 2 + 255),
    (256, 128, 2, 4, 1, 4096),
])
def test_f16_operands_parity_geometries(P, D, Hk, G, R, T):
    Hq = G * Hk
    st = _stream(P, 1, Hk, D, Hq, R, T, ring=3, chunk=1)
    (k, v), = _fill(st, 1, T, Hk, D)
    npages = math.ceil(T / P)
    mask = (synth.u64(SEED + 1, synth.tag("mask", P, D), npages) % 2).astype(np.uint8)
    st.set_residency(0, mask)
    q = queries(SEED, 0, R, Hq, D)
    scale = 1.0 / math.sqrt(D)
    out, lse = attend(st, 0, q, T - R, scale)
    ro, rl = oracle_ref(k, v, q, T - R, scale)
    _check(out, lse, ro, rl)


def test_f16_operands_single_key_and_rows_across_pages():
    P, D, Hk, G = 64, 256, 2, 6
    st = _stream(P, 1, Hk, D, G * Hk, 5, 64 * 6, ring=2, chunk=1)
    (k, v), = _fill(st, 1, 64 * 6, Hk, D)
    for R, pos0 in ((1, 0), (5, 62), (5, 127), (3, 200)):
        q = queries(SEED, pos0, R, G * Hk, D)
        out, lse = attend(st, 0, q, pos0, 0.07)
        ro, rl = oracle_ref(k, v, q, pos0, 0.07)
        _check(out, lse, ro, rl)


def test_f16_operands_constant_values_and_large_scores():
    """V = 1 everywhere: every output is 1 up to the weights' f16 rounding; a
    query scaled by 4 makes the softmax peaked (a few keys dominate)."""
    P, D, Hk, G, R, T = 128, 256, 2, 6, 3, 128 * 5 + 17
    st = _stream(P, 1, Hk, D, G * Hk, R, T, ring=2, chunk=1)
    k = synth.normal(SEED, synth.tag("K1"), (T, Hk, D))
    v = np.ones((T, Hk, D), np.float32)
    append_rows(st, 0, k, v)
    q = queries(SEED, 0, R, G * Hk, D) * np.float32(4.0)
    out, _ = attend(st, 0, q, T - R, 0.0625)
    assert np.abs(out - 1.0).max() <= 1e-3


def test_f16_operands_f16_queries():
    import torch
    P, D, Hk, G, R, T = 256, 256, 4, 6, 2, 256 * 3 + 5
    st = _stream(P, 1, Hk, D, G * Hk, R, T, ring=2)
    (k, v), = _fill(st, 1, T, Hk, D)
    q = queries(SEED, 0, R, G * Hk, D).astype(np.float16).astype(np.float32)
    out, lse = attend(st, 0, q, T - R, 1 / 16, dtype=torch.float16)
    ro, rl = oracle_ref(k, v, q, T - R, 1 / 16)
    _check(out, lse, ro, rl)


@pytest.mark.parametrize("lanes,R,D,P", [(1, 3, 256, 64), (8, 1, 256, 64), (4, 6, 256, 128), (2, 5, 128, 64)])
def test_f16_operands_streamed_equals_resident_bitwise(lanes, R, D, P):
    L, Hk, G = 2, 2, 6
    T = P * (640 // P) + 33
    Hq = G * Hk
    st = _stream(P, L, Hk, D, Hq, R, T, ring=8, chunk=2, lanes=lanes)
    hist = _fill(st, L, T, Hk, D)
    npages = math.ceil(T / P)
    qs = [queries(SEED, l, R, Hq, D) for l in range(L)]
    for l in range(L):
        st.set_residency(l, np.ones(npages, np.uint8))
    base = [attend(st, l, qs[l], T - R, 0.0625) for l in range(L)]
    for l in range(L):
        _check(*base[l], *oracle_ref(*hist[l], qs[l], T - R, 0.0625))
    rng = np.random.default_rng(9)
    for ring, chunk in [(1, 1), (3, 2), (8, 4)]:
        for l in range(L):
            st.set_residency(l, (rng.random(npages) < 0.4).astype(np.uint8))
        st.set_ring_slots(ring, chunk)
        st.prefetch(0)
        for l in range(L):
            if l + 1 < L:
                st.prefetch(l + 1)
            out, lse = attend(st, l, qs[l], T - R, 0.0625)
            assert np.array_equal(out, base[l][0]) and np.array_equal(lse, base[l][1]), (ring, chunk, l)


def test_f16_operands_wide_verify_row_groups():
    """49 causal fp32 rows at 6 query heads per kv head: row groups of the split-K kernel."""
    R, P, D, Hk, G = 49, 256, 256, 4, 6
    T = 256 * 12 + 70
    st = _stream(P, 1, Hk, D, G * Hk, R, T, ring=8, chunk=2, max_verify_rows=R)
    (k, v), = _fill(st, 1, T, Hk, D)
    st.set_residency(0, (np.arange(math.ceil(T / P)) % 2 == 1).astype(np.uint8))
    q = queries(SEED, 0, R, G * Hk, D)
    out, lse = attend(st, 0, q, T - R, 1 / 16)
    _check(out, lse, *oracle_ref(k, v, q, T - R, 1 / 16))


# ------------------------------------------------------------ full size, benchmark launch shapes

def test_f16_operands_decode_stack_full_size():
    """Context 32768, 24 q / 4 kv heads, D 256, half the pages resident (seeded),
    8-slot ring in 4-page chunks on 2 lanes: three layers against the oracle."""
    P, Hk, Hq, D, T, L = 256, 4, 24, 256, 32768, 3
    st = _stream(P, L, Hk, D, Hq, 1, T, ring=8, chunk=4, pool_pages=L * 64, lanes=2)
    hist = _fill(st, L, T, Hk, D)
    for l in range(L):
        mask = np.zeros(128, np.uint8)
        mask[synth.choose(SEED + 1, synth.tag("resident", l), 126, 62)] = 1
        st.set_residency(l, mask)
    st.prefetch(0)
    for l in range(L):
        if l + 1 < L:
            st.prefetch(l + 1)
        q = queries(SEED, l, 1, Hq, D)
        out, lse = attend(st, l, q, T - 1, 1 / 16)
        _check(out, lse, *oracle_ref(*hist[l], q, T - 1, 1 / 16))


def test_f16_operands_span_verify_full_size():
    """6 causal rows at 163840..163845, 400 resident pages, 8-slot ring in 1-page chunks on 8 lanes."""
    P, Hk, Hq, D, R = 256, 4, 24, 256, 6
    T = 163840 + R
    st = _stream(P, 1, Hk, D, Hq, R, T, ring=8, chunk=1, pool_pages=400, lanes=8)
    (k, v), = _fill(st, 1, T, Hk, D)
    mask = np.zeros(641, np.uint8)
    mask[:400] = 1
    st.set_residency(0, mask)
    q = queries(SEED, 0, R, Hq, D)
    out, lse = attend(st, 0, q, T - R, 1 / 16)
    _check(out, lse, *oracle_ref(k, v, q, T - R, 1 / 16))


@pytest.mark.parametrize("R,resident", [(1, 0.5), (4, 0.1), (1, 1.0)])
def test_f16_operands_long_context_full_size(R, resident):
    """Context 262144 (1024 pages): a resident prefix, the rest through a large ring
    in 32-page chunks on 4 lanes; every row against the oracle."""
    P, Hk, Hq, D = 256, 4, 24, 256
    T = 262144 + R - 1
    npages = -(-T // P)
    n_res = int(resident * npages)
    st = _stream(P, 1, Hk, D, Hq, R, T, ring=1009, chunk=32, pool_pages=max(n_res, 1), lanes=4)
    (k, v), = _fill(st, 1, T, Hk, D)
    mask = np.zeros(npages, np.uint8)
    mask[:n_res] = 1
    st.set_residency(0, mask)
    q = queries(SEED, 0, R, Hq, D)
    out, lse = attend(st, 0, q, T - R, 1 / 16)
    _check(out, lse, *oracle_ref(k, v, q, T - R, 1 / 16))
