"""Benchmark: streamed paged Q8_0-K / Q4_0-V decode attention on GB300.

Workload (default, "decode32k"): a 64-layer decode step with one query row
at context 32768, 24 query / 4 kv heads, head dim 256, 256-token pages, K as
Q8_0 and V as Q4_0 from seeded N(0,1) data; half of every layer's pages
resident (62 seeded pages + the two tail pages), the other 64 streamed from
host memory through an 8-slot ring with next-layer prefetch.  One step = for
every layer: append the new row (quantise into the tail page, publish the
completed page to host), announce the next layer, attend over all 32768 keys,
truncate back so every step attends the same context.  The step is captured
once as a CUDA graph (kvs_graph_*) and replayed.

Prints one JSON line.  ``--impl reference`` times the oracle (fp64 CPU) on the
same workload instead.  Under torchrun each rank runs an independent replica
(the path has no exchange between GPUs); rank 0 prints the aggregate.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

SEED, RES_SEED = 1234, 1235

WORKLOADS = {
    "decode32k": dict(
        desc=("decode stack: 64 layers x 1 row, context 32768, 24 q / 4 kv heads, D 256, page 256, "
              "Q8_0 K / Q4_0 V, 50% of pages resident (seeded), rest streamed via an 8-slot ring "
              "with next-layer prefetch (2-page chunks on 4 copy/attention lanes)"),
        L=64, T=32768, R=1, Hq=24, Hk=4, D=256, P=256, ring=8, chunk=2, lanes=4, resident_frac=0.5),
    "decode32k_small": dict(  # a reduced copy for quick checks and profiling captures
        desc="decode stack, 8 layers, otherwise as decode32k",
        L=8, T=32768, R=1, Hq=24, Hk=4, D=256, P=256, ring=8, chunk=2, lanes=4, resident_frac=0.5),
    "resident131k": dict(  # the attention kernel over resident pages, launches far larger than L2
        desc=("all-resident decode: 4 layers x 1 row, context 131072, 24 q / 4 kv heads, D 256, page 256, "
              "Q8_0 K / Q4_0 V, every page resident (218 MB of pages per layer)"),
        L=4, T=131072, R=1, Hq=24, Hk=4, D=256, P=256, ring=8, chunk=2, resident_frac=1.0),
}


def _rank_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def _measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    return 6800.0, "fallback 6.8 TB/s"


def _resident_mask(wl, layer):
    """Seeded residency: resident_frac of the pages, counting the two tail pages."""
    n = math.ceil(wl["T"] / wl["P"])
    want = int(round(wl["resident_frac"] * n)) - 2
    mask = np.zeros(n, np.uint8)
    if want > 0:
        mask[synth.choose(RES_SEED, synth.tag("resident", layer), n - 2, want)] = 1
    return mask


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.out = tempfile.NamedTemporaryFile(mode="w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        self.proc.wait()
        self.out.seek(0)
        rows = [r.split(",") for r in self.out.read().strip().splitlines() if r.strip()]
        os.unlink(self.out.name)
        sm = [float(r[1]) for r in rows if len(r) >= 9 and r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if len(r) >= 9 and r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            if len(r) < 9:
                continue
            for i, nm in enumerate(names):
                if r[5 + i].strip().lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows)}


def h2d_ceiling(torch, dev):
    """Best pinned host -> device copy rate (GB/s) over 1 GiB, best of 5."""
    n = 1 << 30
    h = torch.empty(n, dtype=torch.uint8, pin_memory=True)
    h.fill_(1)
    d = torch.empty(n, dtype=torch.uint8, device=dev)
    s = torch.cuda.Stream(device=dev)
    best = 1e30
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            e0.record(s)
            d.copy_(h, non_blocking=True)
            e1.record(s)
        e1.synchronize()
        best = min(best, e0.elapsed_time(e1))
    del h, d
    return n / (best * 1e-3) / 1e9


def oracle_layer_sample(wl, layer, k_hist, v_hist, k_new, v_new, q, threads=0):
    """The oracle's decode of one layer: returns (seconds, o, lse)."""
    import oracle
    k = np.concatenate([k_hist, k_new])
    v = np.concatenate([v_hist, v_new])
    qkv = oracle.QuantKV(k, v)
    t0 = time.perf_counter()
    o, lse = qkv.attend(q, wl["T"] - 1, 1.0 / math.sqrt(wl["D"]), threads=threads)
    return time.perf_counter() - t0, o, lse


def run_reference(args, wl):
    """Reference arm: the oracle, timed on the host cores, one sampled layer per step."""
    import oracle
    rank, world, _ = _rank_env()
    if rank != 0:
        return
    T, Hk, D, Hq = wl["T"], wl["Hk"], wl["D"], wl["Hq"]
    times = []
    for step in range(args.warmup + args.steps):
        layer = step % wl["L"]
        k = synth.normal(SEED, synth.tag("K", layer), (T - 1, Hk, D))
        v = synth.normal(SEED, synth.tag("V", layer), (T - 1, Hk, D))
        kn = synth.normal(SEED, synth.tag("Knew", layer), (1, Hk, D))
        vn = synth.normal(SEED, synth.tag("Vnew", layer), (1, Hk, D))
        q = synth.normal(SEED, synth.tag("Q", layer), (1, Hq, D))
        t, _, _ = oracle_layer_sample(wl, layer, k, v, kn, vn, q)
        if step >= args.warmup:
            times.append(t)
    step_s = statistics.mean(times) * wl["L"]
    value = wl["R"] / step_s
    cores = oracle.threads()
    sample = f"oracle fp64 decode of 1 of {wl['L']} layers per step (24 heads x {T} keys), time x {wl['L']}"
    line = {
        "impl": "reference", "metric": "streamed-attention tokens/s", "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl["desc"], "layers": wl["L"], "context": T},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, wl):
    import torch
    from host_streamed_paged_gb300 import kvs

    rank, world, local = _rank_env()
    dist = None
    if world > 1:
        import torch.distributed as dist_mod
        dist = dist_mod
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    kvs.load()

    L, T, R, Hq, Hk, D, P = (wl[k] for k in ("L", "T", "R", "Hq", "Hk", "D", "P"))
    T0 = T - 1  # history before the step's appended row
    npages = math.ceil(T / P)
    masks = [_resident_mask(wl, l) for l in range(L)]
    pool = int(sum(int(m.sum()) for m in masks))
    st = kvs.KVStream(page_tokens=P, n_layers=L, n_kv_head=Hk, head_dim=D, max_q_head=Hq, max_rows=max(R, 1),
                      max_tokens=T, ring_slots=wl["ring"], chunk_pages=wl["chunk"],
                      arena_slots=2 * L + wl["ring"] + pool, device=dev, lanes=wl.get("lanes", 1))

    ceiling = h2d_ceiling(torch, dev)

    # history: seeded rows appended through the KV writer, then residency
    keep = {}  # oracle sample layers
    n_cpu_layers = max(1, min(L, args.cpu_layers))
    cpu_layers = list(range(0, L, max(1, L // n_cpu_layers)))[:n_cpu_layers] if rank == 0 else []
    for l in range(L):
        k = synth.normal(SEED, synth.tag("K", l), (T0, Hk, D))
        v = synth.normal(SEED, synth.tag("V", l), (T0, Hk, D))
        kt = torch.from_numpy(k).to(dev)
        vt = torch.from_numpy(v).to(dev)
        torch.cuda.synchronize(dev)
        st.append(l, kt, vt)
        st.sync()
        del kt, vt
        st.set_residency(l, masks[l])
        if l in cpu_layers:
            keep[l] = (k, v)
    st.sync()

    # per-step inputs (device) and their pinned host copies for the e2e leg
    q_h = torch.from_numpy(np.stack([synth.normal(SEED, synth.tag("Q", l), (R, Hq, D)) for l in range(L)])).pin_memory()
    kn_h = torch.from_numpy(np.stack([synth.normal(SEED, synth.tag("Knew", l), (R, Hk, D)) for l in range(L)])).pin_memory()
    vn_h = torch.from_numpy(np.stack([synth.normal(SEED, synth.tag("Vnew", l), (R, Hk, D)) for l in range(L)])).pin_memory()
    q_d, kn_d, vn_d = q_h.to(dev), kn_h.to(dev), vn_h.to(dev)
    out_d = torch.empty((L, R, Hq, D), dtype=torch.float32, device=dev)
    lse_d = torch.empty((L, R, Hq), dtype=torch.float32, device=dev)
    out_h = torch.empty_like(out_d, device="cpu").pin_memory()
    torch.cuda.synchronize(dev)
    scale = 1.0 / math.sqrt(D)

    def step():
        st.prefetch(0)
        for l in range(L):
            kvs.kvs_append(st.ctx, l, kn_d[l], vn_d[l], R)
            if l + 1 < L:
                st.prefetch(l + 1)
            kvs.kvs_attend(st.ctx, l, q_d[l], kvs.KVS_F32, R, Hq, T - R, scale, out_d[l], lse_d[l])
            st.truncate(l, T0)

    # one eager step (host-issued), timed for context
    st.sync()
    t0 = time.perf_counter()
    step()
    st.sync()
    eager_ms = (time.perf_counter() - t0) * 1e3
    s_eager = st.stats(reset=True)

    # capture the step once; replays re-execute every kernel and copy in it
    st.set_timing(0)
    st.graph_begin()
    step()
    st.graph_end()
    gstats = st.stats(reset=True)
    kernels_per_step = gstats["graph_kernels"]
    h2d_bytes_step = gstats["h2d_bytes"]

    attn = st.attn_stream

    def timed(n, e2e=False):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if dist:
            dist.barrier()
        torch.cuda.synchronize(dev)
        e0.record(attn)
        for _ in range(n):
            if e2e:
                with torch.cuda.stream(attn):
                    q_d.copy_(q_h, non_blocking=True)
                    kn_d.copy_(kn_h, non_blocking=True)
                    vn_d.copy_(vn_h, non_blocking=True)
            st.graph_launch()
            if e2e:
                with torch.cuda.stream(attn):
                    out_h.copy_(out_d, non_blocking=True)
        e1.record(attn)
        torch.cuda.synchronize(dev)
        st.sync()
        ms = e0.elapsed_time(e1) / n
        if dist:
            t = torch.tensor([ms], device=dev)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            ms = float(t.item())
        return ms

    for _ in range(args.warmup):
        st.graph_launch()
    st.sync()
    clocks = ClockSampler(local)
    clocks.start()
    ms_step = timed(args.steps)
    clk = clocks.stop()
    st.sync()
    out_ref = out_d.detach().cpu().numpy()

    # e2e: the same step with host inputs copied in and outputs copied out
    for _ in range(args.warmup):
        st.graph_launch()
    e2e_ms = timed(args.steps, e2e=True)
    h2d_in = q_h.numel() * 4 + kn_h.numel() * 4 + vn_h.numel() * 4
    d2h_out = out_h.numel() * 4

    # roofline leg: host-issued steps with CUDA events around each resident-page
    # attention launch (the HBM-bound part; the ring-chunk launches wait on
    # copies), timed in their own region; graph-recorded events carry no timing
    st.graph_destroy()
    for _ in range(2):
        step()
    st.sync()
    st.stats(reset=True)
    st.set_timing(kvs.KVS_TIME_RESIDENT)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    n_eager = max(3, min(args.steps, 10))
    for _ in range(n_eager):
        step()
    st.sync()
    ms_timed_eager = (time.perf_counter() - t0) * 1e3 / n_eager
    st.set_timing(0)
    rs = st.stats(reset=True)
    r_ms, r_n, r_bytes = rs["decode_ms"], rs["decode_timed"], rs["decode_bytes"]

    hbm_peak, peak_src = _measured_peaks()
    achieved = (r_bytes / (r_ms * 1e-3) / 1e9) if r_ms > 0 else 0.0

    # CPU baseline (rank 0): the oracle on sampled layers, scaled to the step
    cpu = None
    parity = None
    if rank == 0 and cpu_layers and not args.no_cpu:
        import oracle
        tsum, errs = 0.0, []
        for l in cpu_layers:
            k, v = keep[l]
            t, o, lse = oracle_layer_sample(wl, l, k, v, kn_h[l].numpy(), vn_h[l].numpy(), q_h[l].numpy())
            tsum += t
            g = out_ref[l].astype(np.float64)
            errs.append(float((np.abs(g - o).max(axis=-1) / np.abs(o).max(axis=-1)).max()))
        step_s = tsum / len(cpu_layers) * L
        cpu = {"value": R / step_s, "unit": "tokens/s", "cores": oracle.threads(), "kind": "oracle",
               "sample": (f"oracle fp64 decode of {len(cpu_layers)} of the {L} layers of one step "
                          f"({Hq} heads x {T} keys each), time scaled x {L}/{len(cpu_layers)}")}
        parity = {"layers_checked": cpu_layers, "max_rel_err": max(errs), "tol": 1e-3}

    value = world * R / (ms_step * 1e-3)
    kv_bytes_step = L * npages * st.page_bytes
    line = {
        "metric": "streamed-attention tokens/s", "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": wl["desc"], "layers": L, "context": T, "rows": R, "q_heads": Hq, "kv_heads": Hk,
                   "head_dim": D, "page_tokens": P, "resident_fraction": wl["resident_frac"],
                   "ring_slots": wl["ring"], "chunk_pages": wl["chunk"], "lanes": wl.get("lanes", 1),
                   "parallelism": f"replicas x{world}",
                   "l2": f"inputs larger than L2: {kv_bytes_step / 1e9:.2f} GB of KV pages read per step",
                   "step": "per layer: append row, prefetch next layer, attend, truncate; one CUDA graph replay"},
        "kv_gbs": kv_bytes_step / (ms_step * 1e-3) / 1e9,
        "h2d": {"achieved_gbs": h2d_bytes_step / (ms_step * 1e-3) / 1e9, "ceiling_gbs": ceiling,
                "frac": h2d_bytes_step / (ms_step * 1e-3) / 1e9 / ceiling, "bytes_per_step": h2d_bytes_step,
                "ceiling_how": "pinned cudaMemcpyAsync 1 GiB, best of 5"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "traffic": None,
                     "kernel": f"decode_kernel<{D},1> launches over resident + tail pages",
                     "launches_timed": r_n, "bytes_per_launch": r_bytes / max(r_n, 1),
                     "ms_per_launch": r_ms / max(r_n, 1), "peak_source": peak_src,
                     "timed_region": f"{n_eager} host-issued steps ({ms_timed_eager:.2f} ms/step)"},
        "cpu_baseline": cpu,
        "e2e": {"value": world * R / (e2e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d_in,
                "d2h_bytes_per_step": d2h_out},
        "gpu_launches": kernels_per_step * args.steps,
        "clocks": clk,
        "eager_ms_per_step": eager_ms,
        "parity": parity,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    st.close()
    if dist:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="decode32k")
    ap.add_argument("--cpu-layers", type=int, default=8, help="layers the oracle baseline samples")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--ring", type=int, default=0, help="override the workload's ring slots")
    ap.add_argument("--chunk", type=int, default=0, help="override the workload's pages per ring chunk")
    ap.add_argument("--layers", type=int, default=0, help="override the workload's layer count")
    ap.add_argument("--lanes", type=int, default=0, help="override the workload's ring lanes")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    wl = dict(WORKLOADS[args.workload])
    for key in ("ring", "chunk", "layers", "lanes"):
        v = getattr(args, key)
        if v:
            wl["L" if key == "layers" else key] = v
            wl["desc"] += f" [{key} override: {v}]"
    if args.impl == "reference":
        run_reference(args, wl)
    else:
        run_ours(args, wl)


if __name__ == "__main__":
    main()
