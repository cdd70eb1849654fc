"""kvs_attend_pages_noalloc: the attention entry point for callers that cannot
allocate device memory (allocator callbacks, plug-ins on a fixed device
budget, services that must not grow their footprint).  Its split partials
live in a fixed array inside the library instead of a caller workspace.

The pages handed to it are built on the host by the oracle's page encoder
(the layout include/kvs.h states) and placed in shuffled slots of one device
buffer.  Two calls in a row (the second reuses the array the first left
behind) are checked, within the parity tolerance the other GPU tests use,
against the oracle's attention and against kvs_attend, the entry point that
takes a workspace, run over the same pages installed in a context with
kvs_load_host_pages.
This file sorts last so that a run stopping at the first failure has
already run every other test.
"""
import math

import numpy as np
import pytest

import oracle
from host_streamed_paged_gb300 import kvs
from kvs_testutil import LSE_TOL, REL_TOL, SEED, history, make_stream, queries, rel_err

pytestmark = pytest.mark.gpu


def test_noalloc_matches_the_oracle_on_two_calls_in_a_row():
    import torch
    P, Hk, G, D, T = 256, 4, 6, 256, 256 * 9 + 100
    Hq = G * Hk
    k, v = history(SEED, 0, T, Hk, D)
    qkv = oracle.QuantKV(k, v)
    npages = math.ceil(T / P)
    page_bytes = Hk * P * D * 13 // 8
    # logical page i sits in slot order[i] of a buffer with two spare slots
    order = np.random.default_rng(3).permutation(npages + 2)[:npages].astype(np.uint32)
    host = np.zeros((npages + 2) * page_bytes, np.uint8)
    for i in range(npages):
        host[order[i] * page_bytes:(order[i] + 1) * page_bytes] = qkv.encode_page(P, i)
    pages = torch.from_numpy(host).cuda()
    stream = torch.cuda.Stream()
    scale = 1.0 / math.sqrt(D)
    # the same pages through kvs_attend: installed in a context's host history, all resident
    st = make_stream(P, 1, Hk, D, Hq, 6, T, ring=2)
    full = (npages - 1) * P  # complete pages go in as encoded bytes, the partial last one by the KV writer
    st.load_host_pages(0, 0, np.concatenate([qkv.encode_page(P, i) for i in range(npages - 1)]))
    kt = torch.from_numpy(np.ascontiguousarray(k[full:])).cuda()
    vt = torch.from_numpy(np.ascontiguousarray(v[full:])).cuda()
    torch.cuda.synchronize()
    st.append(0, kt, vt)
    st.set_residency(0, np.ones(npages, np.uint8))
    st.sync()

    for call, R in enumerate((6, 1)):
        q = queries(SEED, 40 + call, R, Hq, D)
        qt = torch.from_numpy(q).cuda()
        out = torch.full((R, Hq, D), float("nan"), device="cuda")
        lse = torch.full((R, Hq), float("nan"), device="cuda")
        torch.cuda.synchronize()
        kvs.kvs_attend_pages_noalloc(pages, pages.numel(), order, P, Hk, D, qt, kvs.KVS_F32, R, Hq,
                                     T - R, scale, out, lse, stream.cuda_stream)
        stream.synchronize()
        ro, rl = qkv.attend(q, T - R, scale)
        g, gl = out.cpu().numpy(), lse.cpu().numpy().astype(np.float64)
        assert np.isfinite(g).all(), f"call {call}"
        assert rel_err(g, ro) <= REL_TOL, f"call {call}"
        assert np.abs(gl - rl).max() <= LSE_TOL, f"call {call}"
        wo, wl = st.attend(0, qt, T - R, scale)
        st.sync()
        w, wl = wo.cpu().numpy().astype(np.float64), wl.cpu().numpy().astype(np.float64)
        assert rel_err(g, w) <= REL_TOL, f"call {call}: noalloc vs kvs_attend"
        assert np.abs(gl - wl).max() <= LSE_TOL, f"call {call}: noalloc vs kvs_attend"
    st.close()


def test_noalloc_refuses_beyond_its_fixed_scratch():
    import torch
    q = torch.zeros((6, 24, 256), device="cuda")
    out = torch.zeros((6, 24, 256), device="cuda")
    pages = torch.zeros(425984, dtype=torch.uint8, device="cuda")  # one 416 KiB page
    # 300 pages x 24 heads x 6 rows x 258 floats x 4 B = 44.6 MB > 32 MiB: refused before any work
    slots = np.zeros(300, np.uint32)
    with pytest.raises(kvs.KVSError) as e:
        kvs.kvs_attend_pages_noalloc(pages, pages.numel(), slots, 256, 4, 256, q, kvs.KVS_F32, 6, 24,
                                     300 * 256 - 6, 0.1, out, None, 0)
    assert e.value.status == kvs.KVS_ERR_CAPACITY
    assert "scratch" in kvs.kvs_last_error(None)
