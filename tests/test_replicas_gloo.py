"""The N > 1 path on CPU: two gloo ranks, each an independent replica.

Each rank drives its own plan-only context through the same decode steps (the
host scheduler with no GPU), and the ranks check with collectives that their
plans agree, that the step time reduction takes the slowest rank and that the
throughput aggregates over ranks.
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from host_streamed_paged_gb300 import kvs, replicas


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _replica_plan(lanes):
    P, L, Hk, G, R, T = 64, 3, 2, 6, 1, 64 * 9 + 5
    st = kvs.KVStream(page_tokens=P, n_layers=L, n_kv_head=Hk, head_dim=128, max_q_head=G * Hk, max_rows=R,
                      max_tokens=T + 4, ring_slots=4, chunk_pages=2, arena_slots=2 * L + 4 + L * 10,
                      plan_only=True, lanes=lanes)
    npages = -(-T // P)
    rng = np.random.default_rng(7)  # the same residency on every replica
    for layer in range(L):
        kvs.kvs_append(st.ctx, layer, None, None, T)
        st.set_residency(layer, (rng.random(npages) < 0.5).astype(np.uint8))
    for step in range(2):
        st.prefetch(0)
        for layer in range(L):
            if layer + 1 < L:
                st.prefetch(layer + 1)
            st.attend_plan(layer, R, G * Hk, T - R)
    sig = replicas.plan_signature(st.trace())
    st.close()
    return sig


def _worker(rank, world, port, lanes, out):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        sig = _replica_plan(lanes)
        sigs = [None] * world
        dist.all_gather_object(sigs, sig)
        ms = 10.0 + 2.5 * rank  # the replicas' own step times
        slowest = replicas.max_over_ranks(ms, dist)
        value = replicas.aggregate_rows_per_s(1, slowest, world)
        out[rank] = (sigs, slowest, value)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("lanes", [1, 3])
def test_two_gloo_replicas_agree_and_aggregate(lanes):
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, world, port, lanes, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    assert set(res) == {0, 1}
    sigs0, slow0, val0 = res[0]
    sigs1, slow1, val1 = res[1]
    assert sigs0 == sigs1 and sigs0[0] == sigs0[1]  # identical plans on both replicas
    assert slow0 == slow1 == 12.5                   # the slowest rank bounds the step
    assert val0 == val1 == pytest.approx(2 / 12.5e-3)



def test_aggregate_and_max_without_process_group():
    assert replicas.max_over_ranks(3.0) == 3.0
    assert replicas.aggregate_rows_per_s(6, 10.0, 1) == pytest.approx(600.0)
    with pytest.raises(ValueError):
        replicas.aggregate_rows_per_s(1, 0.0, 1)
