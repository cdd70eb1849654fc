"""kvs_attend_pages_noalloc: the attention entry point for callers that cannot
allocate device memory (allocator callbacks, plug-ins on a fixed device
budget, services that must not grow their footprint).  Its split partials
live in a fixed array inside the library instead of a caller workspace.

Checked through the C ABI against kvs_attend, the entry point that takes a
workspace, on two calls in a row (the second call reuses the array the first
left behind), within the parity tolerance the other GPU tests use.  This file
sorts last so that a run stopping at the first failure has already run every
other test.
"""
import math

import numpy as np
import pytest

from host_streamed_paged_gb300 import kvs
from kvs_testutil import REL_TOL, LSE_TOL, SEED, append_rows, history, make_stream, queries, rel_err

pytestmark = pytest.mark.gpu


def _pages_of(st, layer, npages):
    slots = []
    for p in range(npages):
        kind, slot = st.page_location(layer, p)
        assert kind in (1, 2), "every page must be device-resident for this call"
        slots.append(slot)
    return np.array(slots, dtype=np.uint32)


def test_noalloc_matches_workspace_entry_point_twice():
    import torch
    P, Hk, G, D, T = 256, 4, 6, 256, 256 * 9 + 100
    Hq = G * Hk
    st = make_stream(P, 1, Hk, D, Hq, 6, T, ring=2)
    k, v = history(SEED, 0, T, Hk, D)
    append_rows(st, 0, k, v)
    npages = math.ceil(T / P)
    st.set_residency(0, np.ones(npages, np.uint8))
    st.sync()
    slots = _pages_of(st, 0, npages)
    scale = 1.0 / math.sqrt(D)
    stream = st.attn_stream.cuda_stream

    for call, R in enumerate((6, 1)):
        q = torch.from_numpy(queries(SEED, 40 + call, R, Hq, D)).cuda()
        torch.cuda.synchronize()
        ref_o, ref_l = st.attend(0, q, T - R, scale)
        st.sync()
        out = torch.full((R, Hq, D), float("nan"), device="cuda")
        lse = torch.full((R, Hq), float("nan"), device="cuda")
        torch.cuda.synchronize()
        kvs.kvs_attend_pages_noalloc(st.arena, st.arena.numel(), slots, P, Hk, D, q, kvs.KVS_F32, R, Hq,
                                     T - R, scale, out, lse, stream)
        st.sync()
        torch.cuda.synchronize()
        g, r = out.cpu().numpy(), ref_o.cpu().numpy().astype(np.float64)
        assert rel_err(g, r) <= REL_TOL, f"call {call}"
        assert np.abs(lse.cpu().numpy() - ref_l.cpu().numpy()).max() <= LSE_TOL, f"call {call}"


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
    assert "32" in kvs.kvs_last_error(None) or "bytes" in kvs.kvs_last_error(None)
