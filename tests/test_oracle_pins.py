"""Pins for the oracle: each check ties it to something other than itself.

- fp16 conversion against numpy's IEEE binary16 conversion (a library routine);
- quantisers against hand-worked blocks (tests/golden) and closed-form bounds;
- the page encoder against byte positions worked out from the stated layout;
- attention against torch's scaled_dot_product_attention in float64 on the
  dequantised cache (brute force, a library routine), against closed forms
  (one key, zero query, constant V) and against causality;
- the log-sum-exp combine against a hand-worked two-split example, the
  empty-split guard, and against whole attention split at arbitrary points.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_cases(name, fill_code):
    cases = []
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        nm, xs, qs, d = [f.strip() for f in line.split(";")]
        x = np.zeros(32, np.float32)
        vals = [float(t) for t in xs.split()]
        x[: len(vals)] = vals
        q = np.full(32, fill_code, np.int64)
        cv = [int(t) for t in qs.split()]
        q[: len(cv)] = cv
        cases.append((nm, x, q, int(d, 16)))
    return cases


# ---------------------------------------------------------------- fp16

def test_f16_to_f32_exhaustive_matches_numpy():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.f16_bits_to_f32(h)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_f32_to_f16_rne_matches_numpy():
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 2**32, size=400000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    # values near the binary16 range, ties, subnormals and overflow edges
    edge = np.array([0.0, -0.0, 1.0, 65504.0, 65519.0, 65519.996, 65520.0, 1e6, 2.0**-14,
                     2.0**-24, 2.0**-25, 3 * 2.0**-26, 2.0**-26, 1 + 2.0**-11, 1 + 3 * 2.0**-11,
                     1 + 2.0**-11 + 2.0**-20, -(1 + 2.0**-11)], np.float32)
    near = (rng.standard_normal(200000) * np.exp2(rng.integers(-26, 17, 200000))).astype(np.float32)
    x = np.concatenate([x, edge, near])
    ours = oracle.f32_to_f16_bits(x)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)


# ---------------------------------------------------------- quantisers

@pytest.mark.parametrize("case", _read_cases("q8_0_blocks.txt", 0), ids=lambda c: c[0])
def test_q8_0_golden(case):
    _, x, q_exp, d_exp = case
    q, d = oracle.q8_0_block(x)
    assert d == d_exp
    assert np.array_equal(q.astype(np.int64), q_exp)


@pytest.mark.parametrize("case", _read_cases("q4_0_blocks.txt", 8), ids=lambda c: c[0])
def test_q4_0_golden(case):
    _, x, q_exp, d_exp = case
    q, d = oracle.q4_0_block(x)
    assert d == d_exp
    assert np.array_equal(q.astype(np.int64), q_exp)


def test_q8_0_bounds_random():
    x = synth.normal(11, synth.tag("q8pin"), (4000, 32)) * np.float32(3.0)
    for row in x:
        q, d16 = oracle.q8_0_block(row)
        amax = np.abs(row).max()
        d = np.float32(amax) / np.float32(127.0)
        i = int(np.argmax(np.abs(row)))
        assert abs(int(q[i])) == 127
        err = np.abs(row.astype(np.float64) - q.astype(np.float64) * float(d))
        assert err.max() <= float(d) * 0.5 * (1 + 1e-5)
        # stored scale is fp16(d): within half a binary16 ulp (relative 2^-11)
        ds = float(np.uint16(d16).view(np.float16))
        assert abs(ds - float(d)) <= abs(float(d)) * 2.0**-11


def test_q4_0_bounds_random():
    x = synth.normal(12, synth.tag("q4pin"), (4000, 32)) * np.float32(2.0)
    for row in x:
        q, d16 = oracle.q4_0_block(row)
        i = int(np.argmax(np.abs(row)))  # first index of the largest magnitude
        d = np.float32(row[i]) / np.float32(-8.0)
        assert q[i] == 0  # the extreme element always codes to 0 (value -8 d = m)
        assert q.max() <= 15
        xh = (q.astype(np.float64) - 8.0) * float(d)
        err = np.abs(row.astype(np.float64) - xh)
        clamped = q == 15
        assert err[~clamped].max(initial=0) <= abs(float(d)) * 0.5 * (1 + 1e-5)
        assert err[clamped].max(initial=0) <= abs(float(d)) * (1 + 1e-5)


# ---------------------------------------------------------- page layout

def _kq_at(t, d, NB):
    # K byte of (token t, dim d): 16-token groups, one 32-byte line per (block, token)
    return ((t // 16 * NB + d // 32) * 16 + t % 16) * 32 + d % 32


def _vq_at(t, row, NB):
    # V nibble byte of (byte row b*16+c, token t): 32-token chunks, one 32-byte line per (block, byte row)
    return ((t // 32 * NB + row // 16) * 16 + row % 16) * 32 + t % 32


def test_page_layout_bytes():
    """Byte positions of the page layout, worked out from its stated definition."""
    P, Hk, D = 32, 2, 64
    NB = D // 32
    T = 45  # page 1 holds tokens 32..44, slots 13..31 are empty
    k = np.zeros((T, Hk, D), np.float32)
    v = np.zeros((T, Hk, D), np.float32)
    for t in range(T):
        for g in range(Hk):
            for d in range(D):
                k[t, g, d] = ((t * 7 + g * 13 + d) % 100) - 50
                v[t, g, d] = ((t + 3 * g + d) % 16) - 8
            for b in range(D // 32):
                k[t, g, 32 * b] = 127.0  # max|x| = 127 -> d = 1 -> codes = x
                v[t, g, 32 * b] = -8.0   # extreme -8 -> d = 1 -> codes = x + 8
    qkv = oracle.QuantKV(k, v)
    pg = qkv.encode_page(P, 1)
    HS = P * D * 13 // 8
    assert pg.size == Hk * HS
    # hand-placed examples: token 0 dim 5 -> line (group 0, block 0, token 0) byte 5 = 5;
    # token 12 dim 63 -> ((0*2+1)*16+12)*32+31 = 927; token 3 dim 33 -> (16+3)*32+1 = 609
    assert [_kq_at(0, 5, NB), _kq_at(12, 63, NB), _kq_at(3, 33, NB), _kq_at(7, 32, NB)] == [5, 927, 609, 736]
    for (t, g, d) in [(0, 0, 5), (12, 1, 63), (3, 1, 33), (7, 0, 32)]:
        tok = 32 + t
        assert pg[g * HS + _kq_at(t, d, NB)].view(np.int8) == k[tok, g, d]
    # K scales: fp16(1.0) = 0x3c00, little-endian, token-major [P][D/32]
    off = 1 * HS + P * D + (5 * 2 + 1) * 2
    assert pg[off] == 0x00 and pg[off + 1] == 0x3C
    # V nibbles: byte row b*16 + c holds dims b*32+c (low) and b*32+c+16 (high)
    vq0 = P * D + P * D // 16
    assert [_vq_at(0, 3, NB), _vq_at(12, 31, NB), _vq_at(5, 0, NB), _vq_at(9, 23, NB)] == [96, 1004, 5, 745]
    for (t, g, b, c) in [(0, 0, 0, 3), (12, 1, 1, 15), (5, 1, 0, 0), (9, 0, 1, 7)]:
        tok = 32 + t
        lo = int(v[tok, g, 32 * b + c]) + 8
        hi = int(v[tok, g, 32 * b + c + 16]) + 8
        assert pg[g * HS + vq0 + _vq_at(t, b * 16 + c, NB)] == lo | (hi << 4)
    # V scales: dim-major [D/32][P]
    vs0 = vq0 + P * D // 2
    off = 1 * HS + vs0 + (1 * P + 12) * 2
    assert pg[off] == 0x00 and pg[off + 1] == 0x3C
    # empty token slots are zero bytes in every section
    for g in range(Hk):
        sec = pg[g * HS:(g + 1) * HS]
        for t in range(13, P):
            assert not any(sec[_kq_at(t, d, NB)] for d in range(D))
            assert not any(sec[vq0 + _vq_at(t, r, NB)] for r in range(D // 2))
            assert not sec[P * D + t * NB * 2: P * D + (t + 1) * NB * 2].any()


def test_page_roundtrip_parse():
    """Parsing the page bytes per the layout recovers every code and scale."""
    P, Hk, D, T = 64, 3, 128, 150
    NB = D // 32
    k = synth.normal(5, synth.tag("pk"), (T, Hk, D))
    v = synth.normal(5, synth.tag("pv"), (T, Hk, D))
    qkv = oracle.QuantKV(k, v)
    HS = P * D * 13 // 8
    for page in range(3):
        pg = qkv.encode_page(P, page)
        n = min(P, T - page * P)
        for g in range(Hk):
            sec = pg[g * HS:(g + 1) * HS]
            # Kq: [P/16][NB][16][32] -> [P][D]
            kq = sec[:P * D].view(np.int8).reshape(P // 16, NB, 16, 32).transpose(0, 2, 1, 3).reshape(P, D)
            ks = sec[P * D:P * D + P * D // 16].view(np.uint16).reshape(P, NB)
            # Vq: [P/32][NB][16][32] -> [NB*16][P]
            vq = sec[P * D + P * D // 16: P * D + P * D // 16 + P * D // 2].reshape(P // 32, NB, 16, 32)
            vq = vq.transpose(1, 2, 0, 3).reshape(NB * 16, P)
            vs = sec[P * D + P * D // 16 + P * D // 2:].view(np.uint16).reshape(NB, P)
            toks = slice(page * P, page * P + n)
            assert np.array_equal(kq[:n], qkv.kq[toks, g])
            assert np.array_equal(ks[:n], qkv.kd[toks, g])
            assert np.array_equal(vs[:, :n].T, qkv.vd[toks, g])
            codes = np.empty((n, D), np.uint8)
            for b in range(NB):
                rows = vq[b * 16:(b + 1) * 16, :n]  # [16][n]
                codes[:, b * 32:b * 32 + 16] = (rows & 0xF).T
                codes[:, b * 32 + 16:b * 32 + 32] = (rows >> 4).T
            assert np.array_equal(codes, qkv.vq[toks, g])


# ---------------------------------------------------------- attention

def _dequant(qkv):
    ks = qkv.kd.view(np.float16).astype(np.float64)
    vs = qkv.vd.view(np.float16).astype(np.float64)
    kh = qkv.kq.astype(np.float64) * np.repeat(ks, 32, axis=2)
    vh = (qkv.vq.astype(np.float64) - 8.0) * np.repeat(vs, 32, axis=2)
    return kh, vh


def _sdpa(qkv, q, pos0, scale):
    kh, vh = _dequant(qkv)
    R, Hq, D = q.shape
    G = Hq // qkv.Hk
    K = torch.from_numpy(kh).permute(1, 0, 2).repeat_interleave(G, dim=0)  # [Hq][T][D]
    V = torch.from_numpy(vh).permute(1, 0, 2).repeat_interleave(G, dim=0)
    Q = torch.from_numpy(q.astype(np.float64)).permute(1, 0, 2)  # [Hq][R][D]
    T = qkv.T
    mask = torch.arange(T)[None, :] <= (pos0 + torch.arange(R))[:, None]
    o = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask, scale=scale)
    return o.permute(1, 0, 2).numpy()


@pytest.mark.parametrize("T,Hk,Hq,D,R", [(70, 2, 6, 64, 3), (300, 1, 4, 32, 1), (129, 4, 8, 128, 6)])
def test_attend_matches_torch_sdpa_fp64(T, Hk, Hq, D, R):
    k = synth.normal(21, synth.tag("ak", T), (T, Hk, D))
    v = synth.normal(21, synth.tag("av", T), (T, Hk, D))
    q = synth.normal(21, synth.tag("aq", T), (R, Hq, D))
    qkv = oracle.QuantKV(k, v)
    pos0 = T - R
    scale = 1.0 / math.sqrt(D)
    o, _ = qkv.attend(q, pos0, scale)
    ref = _sdpa(qkv, q, pos0, scale)
    assert np.abs(o - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max())


def test_attend_single_key_returns_that_value():
    T, Hk, Hq, D = 1, 2, 4, 64
    k = synth.normal(3, synth.tag("s1k"), (T, Hk, D))
    v = synth.normal(3, synth.tag("s1v"), (T, Hk, D))
    q = synth.normal(3, synth.tag("s1q"), (1, Hq, D))
    qkv = oracle.QuantKV(k, v)
    o, lse = qkv.attend(q, 0, 0.125)
    _, vh = _dequant(qkv)
    kh, _ = _dequant(qkv)
    for h in range(Hq):
        g = h // 2
        assert np.array_equal(o[0, h], vh[0, g])
        s = 0.125 * float(np.dot(q[0, h].astype(np.float64), kh[0, g]))
        assert abs(lse[0, h] - s) <= 1e-12 * max(1.0, abs(s))


def test_attend_zero_query_is_mean_and_log_n():
    T, Hk, Hq, D, R = 97, 2, 2, 32, 4
    k = synth.normal(4, synth.tag("zk"), (T, Hk, D))
    v = synth.normal(4, synth.tag("zv"), (T, Hk, D))
    q = np.zeros((R, Hq, D), np.float32)
    qkv = oracle.QuantKV(k, v)
    pos0 = 50
    o, lse = qkv.attend(q, pos0, 0.3)
    _, vh = _dequant(qkv)
    for r in range(R):
        n = pos0 + r + 1
        for h in range(Hq):
            assert np.allclose(o[r, h], vh[:n, h].mean(axis=0), rtol=0, atol=1e-13)
            assert abs(lse[r, h] - math.log(n)) <= 1e-12


def test_attend_constant_v_gives_one():
    """Softmax weights sum to one: with every decoded V element equal to 1, o == 1."""
    T, Hk, Hq, D, R = 200, 2, 6, 64, 2
    k = synth.normal(6, synth.tag("ck"), (T, Hk, D))
    v = np.ones((T, Hk, D), np.float32)  # Q4_0: m = 1, d = -1/8, code 0 -> (0-8)*(-1/8) = 1
    q = synth.normal(6, synth.tag("cq"), (R, Hq, D)) * np.float32(3.0)
    qkv = oracle.QuantKV(k, v)
    o, _ = qkv.attend(q, T - R, 0.125)
    assert np.abs(o - 1.0).max() <= 1e-13


def test_attend_is_causal():
    T, Hk, Hq, D, R = 120, 1, 2, 32, 5
    k = synth.normal(8, synth.tag("ck2"), (T, Hk, D))
    v = synth.normal(8, synth.tag("cv2"), (T, Hk, D))
    q = synth.normal(8, synth.tag("cq2"), (R, Hq, D))
    pos0 = T - R
    o1, l1 = oracle.QuantKV(k, v).attend(q, pos0, 0.2)
    k2, v2 = k.copy(), v.copy()
    k2[pos0 + 2:] += 5.0
    v2[pos0 + 2:] -= 3.0
    o2, l2 = oracle.QuantKV(k2, v2).attend(q, pos0, 0.2)
    assert np.array_equal(o1[:2], o2[:2]) and np.array_equal(l1[:2], l2[:2])
    assert not np.array_equal(o1[2:], o2[2:])


# ---------------------------------------------------------- combine

def test_combine_hand_worked():
    # split A: m=0, l=1, o=[1,2];  split B: m=ln3, l=2, o=[3,0]
    # M = ln3, L = 1/3 + 2 = 7/3, o = ([1/3 + 3, 2/3]) / (7/3) = [10/7, 2/7], lse = ln7
    m = [0.0, -math.inf, math.log(3.0)]
    l = [1.0, 0.0, 2.0]
    op = [[1.0, 2.0], [0.0, 0.0], [3.0, 0.0]]
    o, lse = oracle.combine(m, l, op)
    assert np.allclose(o, [10 / 7, 2 / 7], rtol=0, atol=1e-15)
    assert abs(lse - math.log(7.0)) <= 1e-15


def test_combine_all_empty_guard():
    o, lse = oracle.combine([-math.inf, -math.inf], [0.0, 0.0], np.zeros((2, 4)))
    assert np.array_equal(o, np.zeros(4)) and lse == -math.inf


@pytest.mark.parametrize("cuts", [[0, 256, 512, 700], [0, 1, 333, 334, 700], [0, 700]])
def test_combine_of_partials_equals_whole(cuts):
    T, Hk, Hq, D, R = 700, 2, 6, 64, 3
    k = synth.normal(9, synth.tag("pk9"), (T, Hk, D))
    v = synth.normal(9, synth.tag("pv9"), (T, Hk, D))
    q = synth.normal(9, synth.tag("pq9"), (R, Hq, D))
    qkv = oracle.QuantKV(k, v)
    pos0 = T - R
    o_ref, lse_ref = qkv.attend(q, pos0, 0.0625)
    parts = [qkv.attend_partial(q, pos0, 0.0625, a, b) for a, b in zip(cuts[:-1], cuts[1:])]
    for r in range(R):
        for h in range(Hq):
            m = [p[0][r, h] for p in parts]
            l = [p[1][r, h] for p in parts]
            op = np.stack([p[2][r, h] for p in parts])
            o, lse = oracle.combine(m, l, op)
            assert np.abs(o - o_ref[r, h]).max() <= 1e-12 * np.abs(o_ref[r, h]).max()
            assert abs(lse - lse_ref[r, h]) <= 1e-12
