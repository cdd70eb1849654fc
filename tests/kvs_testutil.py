"""Shared helpers for the GPU parity tests: seeded inputs, stream setup, error metrics."""
from __future__ import annotations

import math

import numpy as np

import oracle
import synth
from host_streamed_paged_gb300 import kvs

SEED = 1234

# parity bar: per (row, head) vector, max_d |gpu - oracle| / max_d |oracle|
REL_TOL = 1e-3
LSE_TOL = 1e-4


def history(seed, layer, T, Hk, D):
    k = synth.normal(seed, synth.tag("K", layer), (T, Hk, D))
    v = synth.normal(seed, synth.tag("V", layer), (T, Hk, D))
    return k, v


def queries(seed, layer, R, Hq, D, tag="Q"):
    return synth.normal(seed, synth.tag(tag, layer), (R, Hq, D))


def make_stream(P, L, Hk, D, Hq, R, max_tokens, ring=8, chunk=0, pool_pages=None, lanes=1, dma=False,
                f16_operands=False, max_verify_rows=0):
    pool = pool_pages if pool_pages is not None else L * math.ceil(max_tokens / P)
    return kvs.KVStream(page_tokens=P, n_layers=L, n_kv_head=Hk, head_dim=D, max_q_head=Hq,
                        max_rows=R, max_tokens=max_tokens, ring_slots=ring, chunk_pages=chunk,
                        arena_slots=2 * L + ring + pool, lanes=lanes, dma_fill=dma,
                        f16_operands=f16_operands, max_verify_rows=max_verify_rows)


def append_rows(st, layer, k, v, pieces=None):
    """Append host rows k, v [n][Hk][D] to `layer`, optionally in irregular pieces."""
    import torch
    n = k.shape[0]
    pieces = pieces or [n]
    assert sum(pieces) == n
    kt = torch.from_numpy(np.ascontiguousarray(k)).cuda()
    vt = torch.from_numpy(np.ascontiguousarray(v)).cuda()
    torch.cuda.synchronize()
    i = 0
    for m in pieces:
        st.append(layer, kt[i:i + m], vt[i:i + m])
        i += m
    st.sync()
    del kt, vt


def attend(st, layer, q, pos0, scale, dtype=None):
    import torch
    qt = torch.from_numpy(np.ascontiguousarray(q)).cuda()
    if dtype is not None:
        qt = qt.to(dtype)
    torch.cuda.synchronize()
    out, lse = st.attend(layer, qt, pos0, scale)
    st.sync()
    torch.cuda.synchronize()
    return out.cpu().numpy(), lse.cpu().numpy()


def rel_err(g, r):
    """max over (row, head) of max_d |g - r| / max_d |r|."""
    num = np.abs(g.astype(np.float64) - r).max(axis=-1)
    den = np.abs(r).max(axis=-1)
    return float((num / den).max())


def check_parity(out, lse, ref_o, ref_lse, lse_tol=LSE_TOL):
    e = rel_err(out, ref_o)
    el = float(np.abs(lse.astype(np.float64) - ref_lse).max())
    assert e <= REL_TOL, f"relative error {e:.3e} > {REL_TOL}"
    assert el <= lse_tol, f"lse error {el:.3e} > {lse_tol}"
    return e, el


def oracle_ref(k, v, q, pos0, scale, threads=0):
    return oracle.QuantKV(k, v).attend(q, pos0, scale, threads=threads)
