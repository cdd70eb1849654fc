"""Benchmark: streamed paged Q8_0-K / Q4_0-V attention on one GB300.

Default workload ("decode32k"): a 64-layer decode step with one query row at
context 32768, 24 query / 4 kv heads, head dim 256, 256-token pages, K as
Q8_0 and V as Q4_0 from seeded N(0,1) data; half of every layer's pages
resident (62 seeded pages + the two tail pages), the other 64 streamed from
host memory through an 8-slot ring with next-layer prefetch.  One step = for
every layer: append the step's rows (quantise into the tail page, publish a
completed page to host), announce the next layer, attend over the whole
history, truncate back so every step sees the same context.  The step is
captured once as a CUDA graph (kvs_graph_*) and replayed.

Other workloads (``--workload``): ``verify163k`` (6 causal rows at 163840,
400 resident pages per layer), ``prefill131k`` (a 256-row fp16 prefill chunk
at 131072 on the tensor-core path; ``--layers 1`` for the one-layer case and
``--resident`` for its residency), ``long262k`` (1 or 4 rows at 262144 in a
fixed 2048 MiB arena, ``--sweep`` over the resident fraction 0..100 % prints
one line per point), ``resident131k`` (the attention kernel over resident
pages only).

Prints one JSON line per measured configuration.  ``--impl reference`` times
the oracle (fp64, host cores) on a bounded sample of the same workload.
Under torchrun each rank runs an independent replica (the path has no
exchange between GPUs); rank 0 prints the aggregate.
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
ARENA_PAGE_SLOTS_2GIB = (2048 << 20) // 425984  # 5041 page slots of 416 KiB

WORKLOADS = {
    "decode32k": dict(
        desc=("decode stack: 64 layers x 1 row, context 32768, 24 q / 4 kv heads, D 256, page 256, "
              "Q8_0 K / Q4_0 V, 50% of pages resident (seeded), rest streamed via an 8-slot ring "
              "with next-layer prefetch (4-page chunks on 2 lanes)"),
        L=64, T=32768, R=1, ring=8, chunk=4, lanes=2, residency=("random", 0.5)),
    "single4k": dict(
        desc=("single layer decode: 1 query row, context 4096, 8 q / 2 kv heads (GQA), head_dim 128, page 256, "
              "all 16 pages resident, Q8_0 K / Q4_0 V from seeded N(0,1)"),
        L=1, T=4096, R=1, ring=2, chunk=1, lanes=1, residency=("prefix_frac", 1.0),
        geom=dict(Hq=8, Hk=2, D=128, P=256)),
    "decode32k_small": dict(  # a reduced copy for quick checks and profiling captures
        desc="decode stack, 8 layers, otherwise as decode32k",
        L=8, T=32768, R=1, ring=8, chunk=4, lanes=2, residency=("random", 0.5)),
    "verify163k": dict(
        desc=("span verify: 6 causal rows at positions 163840..163845, 64 layers, 24 q / 4 kv heads, D 256, "
              "page 256, Q8_0 K / Q4_0 V; 400 resident pages per layer (prefix), the rest via an 8-slot ring "
              "(1-page chunks on 8 lanes)"),
        L=64, T=163840 + 6, R=6, ring=8, chunk=1, lanes=8, residency=("prefix_pages", 400)),
    "prefill131k": dict(
        desc=("prefill chunk: 256 fp16 query rows appended at context 131072, causal, 24 q / 4 kv heads, D 256, "
              "page 256, Q8_0 K / Q4_0 V, tcgen05 tensor-core path"),
        L=64, T=131072 + 256, R=256, ring=24, chunk=2, lanes=2, residency=("prefix_frac", 1.0), q_f16=True),
    "long262k": dict(
        desc=("long-context decode: 64 layers, context 262144, 24 q / 4 kv heads, D 256, page 256, Q8_0 K / "
              "Q4_0 V, fixed 2048 MiB arena split between resident pages (per-layer prefixes) and the ring "
              "(chunks of a quarter of the ring, at most 32 pages)"),
        L=64, T=262144, R=1, ring=8, chunk=0, lanes=4, residency=("arena_frac", 0.5),
        arena_slots=ARENA_PAGE_SLOTS_2GIB),
    "resident131k": dict(  # the attention kernel over resident pages, launches far larger than L2
        desc=("all-resident decode: 4 layers x 1 row, context 131072, 24 q / 4 kv heads, D 256, page 256, "
              "Q8_0 K / Q4_0 V, every page resident (218 MB of pages per layer)"),
        L=4, T=131072, R=1, ring=8, chunk=2, lanes=1, residency=("prefix_frac", 1.0)),
}
GEOM = dict(Hq=24, Hk=4, D=256, P=256)

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of the roofline kernel,
# from one ncu capture of that launch on a GB300 (a workload missing here, or a kernel changed since
# its capture, reports traffic as null).
# resident131k, single-f16 operand mode: 218.19 MB read + 8.63 MB written, captured with
#   ncu --metrics gpu__time_duration.sum,dram__bytes_read.sum,dram__bytes_write.sum,launch__grid_size \
#       --clock-control none -k regex:decode_kernel -s 4 -c 1 --csv \
#       python bench.py --workload resident131k --layers 1 --steps 1 --warmup 3 --no-cpu --no-timeline --no-extras
# decode32k: the resident-page launch of a layer (64 pages x 4 kv heads, 27.26 MB algorithmic):
# 27.33 MB read, 0 written (the 1.5 MB of partials stay in L2), the same in every layer, captured on
# a 2-layer copy of the workload with
#   ncu --metrics gpu__time_duration.sum,dram__bytes_read.sum,dram__bytes_write.sum,launch__grid_size \
#       --clock-control none -k regex:decode_kernel -c 60 --csv \
#       python bench.py --no-cpu --no-extras --no-timeline --layers 2 --steps 1 --warmup 3
# prefill131k, default 24-page splits: 223.76 MB read + 103.55 MB written (split partials), captured with
#   ncu --set full --clock-control none -k regex:prefill_kernel -s 1 -c 1 -o <report> \
#       python bench.py --workload prefill131k --layers 1 --steps 1 --warmup 3 --no-cpu --no-timeline --no-extras
TRAFFIC = {
    "resident131k": (226.82e6, "ncu capture of one decode_kernel launch (resident131k, 1 layer)"),
    "decode32k": (27.33e6, "ncu capture of the resident decode_kernel launches (decode32k, 2 layers)"),
    "prefill131k": (327.30e6, "ncu capture of one prefill_kernel launch (prefill131k, 1 layer, 24-page splits)"),
}


def _rank_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def _measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return (float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "measured (MEASURED_PEAKS.json)")
    return 6800.0, 1900.0, 1700.0, "fallback (6.8 TB/s, 1.9 PFLOP/s)"


def _masks(wl, pool_pages=None):
    """Per-layer residency masks (the two tail pages are device-readable besides)."""
    n = math.ceil(wl["T"] / wl["P"])
    kind, x = wl["residency"]
    out = []
    for layer in range(wl["L"]):
        mask = np.zeros(n, np.uint8)
        if kind == "random":  # x of all pages, counting the two tail pages
            want = int(round(x * n)) - 2
            if want > 0:
                mask[synth.choose(RES_SEED, synth.tag("resident", layer), n - 2, want)] = 1
        elif kind == "prefix_pages":
            mask[:min(int(x), n)] = 1
        elif kind == "prefix_frac":
            mask[:int(round(x * n))] = 1
        elif kind == "arena_frac":  # x of the arena's pool slots, spread evenly as prefixes
            mask[:min(n, pool_pages // wl["L"])] = 1
        out.append(mask)
    return out


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
        num = lambda t: t.strip().replace(".", "", 1).isdigit()  # noqa: E731
        sm = [float(r[1]) for r in rows if len(r) >= 9 and num(r[1])]
        mx = [float(r[2]) for r in rows if len(r) >= 9 and num(r[2])]
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


def _union(iv):
    """Total length of the union of intervals [(a, b)]."""
    tot, cur_a, cur_b = 0, None, None
    for a, b in sorted(iv):
        if cur_b is None or a > cur_b:
            if cur_b is not None:
                tot += cur_b - cur_a
            cur_a, cur_b = a, b
        else:
            cur_b = max(cur_b, b)
    return tot + ((cur_b - cur_a) if cur_b is not None else 0)


def _clip(iv, lo, hi):
    return [(max(a, lo), min(b, hi)) for a, b in iv if b > lo and a < hi]


def timeline_summary(recs, L):
    """Per-step summary of one replayed step's launch timeline (device %globaltimer stamps).

    Link: the union of ring-refill launches is the time the host link is being
    read.  Layer boundary: from the end of layer l's last page read to the start
    of layer l+1's first page read; the kernels on that chain (combine of l,
    truncate clear of l, append of l+1, query fragments of l+1) are listed with
    their median durations, and the refill time inside the boundary shows
    whether the link idles there."""
    ran = [r for r in recs if r["start_ns"] and r["end_ns"]]
    if not ran:
        return None
    t0 = min(r["start_ns"] for r in ran)
    t1 = max(r["end_ns"] for r in ran)
    fills = [(r["start_ns"], r["end_ns"]) for r in ran if r["kind"] == "fill"]
    reads = {}
    for r in ran:
        if r["kind"] in ("read_resident", "read_ring", "prefill"):
            reads.setdefault(r["layer"], []).append((r["start_ns"], r["end_ns"]))
    bounds, fill_in, chain = [], [], {}
    for l in range(L - 1):
        if l not in reads or l + 1 not in reads:
            continue
        a = max(b for _, b in reads[l])
        b = min(x for x, _ in reads[l + 1])
        bounds.append(max(0, b - a))
        fill_in.append(_union(_clip(fills, a, b)) if b > a else 0)
        for r in ran:
            key = None
            if r["layer"] == l and r["kind"] in ("combine", "clear"):
                key = r["kind"] + " (layer l)"
            elif r["layer"] == l + 1 and r["kind"] in ("append", "qprep", "clear"):
                key = r["kind"] + " (layer l+1)"
            if key and a - 5000 <= r["start_ns"] <= b + 5000:
                chain.setdefault(key, []).append(r["end_ns"] - r["start_ns"])
    med = lambda v: statistics.median(v) / 1e3 if v else None  # noqa: E731
    span = t1 - t0
    busy = _union(fills)
    return {
        "step_us": span / 1e3,
        "refill_busy_us": busy / 1e3,
        "refill_busy_frac": busy / span if span else None,
        "refill_launches": len(fills),
        "boundary_us_median": med(bounds),
        "boundary_us_total": sum(bounds) / 1e3,
        "refill_busy_in_boundaries_frac": (sum(fill_in) / sum(bounds)) if sum(bounds) else None,
        "boundary_kernels_us_median": {k: med(v) for k, v in sorted(chain.items())},
        "how": ("one replay of the captured step with every launch stamped (first CTA start, last CTA end, "
                "%globaltimer); refill = SM fill kernels reading pinned host memory"),
    }


def alg_flops_per_layer(wl):
    """QK^T and PV multiply-adds, 2 flops each, over the keys each row sees."""
    T, R, Hq, D = wl["T"], wl["R"], wl["Hq"], wl["D"]
    keys = sum(T - R + r + 1 for r in range(R))
    return 4.0 * D * Hq * keys


def oracle_sample(wl, k_hist, v_hist, k_new, v_new, q, rows=None, threads=0):
    """The oracle on one layer (optionally a subset of its rows): (seconds, o, lse)."""
    import oracle
    k = np.concatenate([k_hist, k_new])
    v = np.concatenate([v_hist, v_new])
    qkv = oracle.QuantKV(k, v)
    T, R = wl["T"], wl["R"]
    rows = rows if rows is not None else list(range(R))
    t0 = time.perf_counter()
    outs = [qkv.attend(q[r:r + 1], T - R + r, 1.0 / math.sqrt(wl["D"]), threads=threads) for r in rows]
    dt = time.perf_counter() - t0
    return dt, np.concatenate([o for o, _ in outs]), np.concatenate([l for _, l in outs])


def layer_inputs(wl, layer):
    T, R, Hk, D = wl["T"], wl["R"], wl["Hk"], wl["D"]
    k = synth.normal(SEED, synth.tag("K", layer), (T - R, Hk, D))
    v = synth.normal(SEED, synth.tag("V", layer), (T - R, Hk, D))
    return k, v


def step_inputs(wl, layer):
    R, Hq, Hk, D = wl["R"], wl["Hq"], wl["Hk"], wl["D"]
    q = synth.normal(SEED, synth.tag("Q", layer), (R, Hq, D))
    if wl.get("q_f16"):
        q = q.astype(np.float16).astype(np.float32)
    kn = synth.normal(SEED, synth.tag("Knew", layer), (R, Hk, D))
    vn = synth.normal(SEED, synth.tag("Vnew", layer), (R, Hk, D))
    return q, kn, vn


def cpu_rows_sample(wl):
    # rows of one layer the oracle baseline times: all rows for decode/verify,
    # 8 rows spread over the chunk for prefill
    R = wl["R"]
    return list(range(R)) if R <= 8 else list(range(0, R, R // 8))[:8]


def run_reference(args, wl):
    """Reference arm: the oracle, timed on the host cores, one sampled layer per step."""
    import oracle
    rank, world, _ = _rank_env()
    if rank != 0:
        return
    rows = cpu_rows_sample(wl)
    times = []
    for step in range(args.warmup + args.steps):
        layer = step % wl["L"]
        k, v = layer_inputs(wl, layer)
        q, kn, vn = step_inputs(wl, layer)
        t, _, _ = oracle_sample(wl, k, v, kn, vn, q, rows)
        if step >= args.warmup:
            times.append(t)
    step_s = statistics.mean(times) * wl["L"] * wl["R"] / len(rows)
    value = wl["R"] / step_s
    cores = oracle.threads()
    sample = (f"oracle fp64 attention of {len(rows)} of {wl['R']} rows of 1 of {wl['L']} layers per step "
              f"({wl['Hq']} heads x {wl['T']} keys), time scaled to the whole step")
    line = {
        "impl": "reference", "metric": "streamed-attention tokens/s", "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl["desc"], "layers": wl["L"], "context": wl["T"]},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# The other configurations' headline numbers, carried on the default line: each
# runs as its own process (its history is built from scratch and freed after),
# with a short timed region and the oracle on one sampled layer for parity.
EXTRAS = [
    ("single4k", []),
    ("verify163k", []),
    ("prefill131k_1layer", ["--workload", "prefill131k", "--layers", "1"]),
    ("prefill131k", []),
    ("long262k_1row", ["--workload", "long262k"]),
    ("long262k_4rows", ["--workload", "long262k", "--rows", "4"]),
    ("long262k_policy", ["--workload", "long262k", "--policy", "6"]),
    ("resident131k", []),
]


def run_extras(args):
    out = {}
    for name, extra in EXTRAS:
        cmd = [sys.executable, os.path.abspath(__file__), "--steps", "5", "--warmup", "3", "--cpu-layers", "1",
               "--no-extras", "--operands", args.operands]
        cmd += extra if extra else ["--workload", name]
        t0 = time.perf_counter()
        try:
            r = subprocess.run(cmd, capture_output=True, text=True, timeout=600)
            d = json.loads([x for x in r.stdout.strip().splitlines() if x.startswith("{")][-1])
        except Exception as e:  # noqa: BLE001 - reported, never fatal to the main line
            out[name] = {"error": f"{type(e).__name__}: {str(e)[:200]}"}
            continue
        roof = d.get("roofline") or {}
        out[name] = {
            "config": d["config"]["workload"], "layers": d["config"]["layers"], "rows": d["config"]["rows"],
            "tokens_per_s": d["value"], "ms_per_step": d["ms_per_step"], "e2e_tokens_per_s": d["e2e"]["value"],
            "kv_gbs": d["kv_gbs"], "h2d_frac": d["h2d"]["frac"] if d["h2d"]["bytes_per_step"] else None,
            "roofline": {k: roof.get(k) for k in ("bound", "achieved", "peak", "unit", "frac", "ms_per_launch")},
            "tflops": d.get("tflops"),
            "policy": d.get("policy"),
            "parity_max_rel_err": (d.get("parity") or {}).get("max_rel_err"),
            "clocks_sm_mhz": (d.get("clocks") or {}).get("sm_mhz"),
            "throttle_reasons": (d.get("clocks") or {}).get("reasons"),
            "steps": d["steps"], "wall_s": time.perf_counter() - t0,
        }
    return out


def run_ours(args, wl):
    import torch
    from host_streamed_paged_gb300 import kvs, replicas

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
    T0 = T - R  # history before the step's appended rows
    npages = math.ceil(T / P)
    fixed_arena = wl.get("arena_slots")
    free = (fixed_arena - 2 * L) if fixed_arena else 0  # pool + ring slots of a fixed arena
    masks0 = _masks(wl, pool_pages=(free - wl["ring"]) if fixed_arena else None)
    pool = int(sum(int(m.sum()) for m in masks0))
    arena_slots = fixed_arena if fixed_arena else 2 * L + wl["ring"] + pool
    st = kvs.KVStream(page_tokens=P, n_layers=L, n_kv_head=Hk, head_dim=D, max_q_head=Hq, max_rows=R,
                      max_tokens=T, ring_slots=wl["ring"], chunk_pages=wl["chunk"], arena_slots=arena_slots,
                      device=dev, lanes=wl.get("lanes", 1), dma_fill=wl.get("dma", False),
                      host_alloc=args.host_alloc, f16_operands=args.operands == "f16",
                      prefill_split_pages=wl.get("split", 0))
    ceiling = h2d_ceiling(torch, dev)

    # history: seeded rows appended through the KV writer
    rows_cpu = cpu_rows_sample(wl)
    n_cpu_layers = max(1, min(L, args.cpu_layers))
    cpu_layers = list(range(0, L, max(1, L // n_cpu_layers)))[:n_cpu_layers] if (rank == 0 and not args.no_cpu) else []
    keep = {}
    t_prep = time.perf_counter()
    for l in range(L):
        k, v = layer_inputs(wl, l)
        kt = torch.from_numpy(k).to(dev)
        vt = torch.from_numpy(v).to(dev)
        torch.cuda.synchronize(dev)
        st.append(l, kt, vt)
        st.sync()
        del kt, vt
        if l in cpu_layers:
            keep[l] = (k, v)
    prep_s = time.perf_counter() - t_prep

    # per-step inputs (device) and their pinned host copies for the e2e leg
    qs, kns, vns = zip(*[step_inputs(wl, l) for l in range(L)])
    qdt = torch.float16 if wl.get("q_f16") else torch.float32
    q_h = torch.from_numpy(np.stack(qs)).to(qdt).pin_memory()
    kn_h = torch.from_numpy(np.stack(kns)).pin_memory()
    vn_h = torch.from_numpy(np.stack(vns)).pin_memory()
    q_d, kn_d, vn_d = q_h.to(dev), kn_h.to(dev), vn_h.to(dev)
    out_d = torch.empty((L, R, Hq, D), dtype=torch.float32, device=dev)
    lse_d = torch.empty((L, R, Hq), dtype=torch.float32, device=dev)
    out_h = torch.empty_like(out_d, device="cpu").pin_memory()
    torch.cuda.synchronize(dev)
    scale = 1.0 / math.sqrt(D)
    q_type = kvs.KVS_F16 if wl.get("q_f16") else kvs.KVS_F32
    prefill = R * Hq // Hk > 64

    def step():
        st.prefetch(0)
        for l in range(L):
            kvs.kvs_append(st.ctx, l, kn_d[l], vn_d[l], R)
            if l + 1 < L:
                st.prefetch(l + 1)
            kvs.kvs_attend(st.ctx, l, q_d[l], q_type, R, Hq, T0, scale, out_d[l], lse_d[l])
            st.truncate(l, T0)

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
        return replicas.max_over_ranks(e0.elapsed_time(e1) / n, dist, dev)

    hbm_peak, tc_peak, _, peak_src = _measured_peaks()
    fracs = [None]
    if args.sweep and wl["residency"][0] == "arena_frac":
        fracs = [i / 10 for i in range(11)]

    def set_split(ring_slots, per_layer):
        # a fixed arena: resident prefixes of per_layer pages, the ring gets the rest
        for l in range(L):
            st.set_residency(l, np.zeros(npages, np.uint8))
        st.set_ring_slots(ring_slots, wl["chunk"])
        m = np.zeros(npages, np.uint8)
        m[:per_layer] = 1
        for l in range(L):
            st.set_residency(l, m)
        st.sync()

    # Closed loop (fixed arena): the residency policy chooses the resident / ring
    # split from the device-measured observation of the steps run at the split in
    # force (readiness misses, ring occupancy, copy-busy fraction); the line is
    # then measured at its last decision
    policy_trace, forced = None, None
    if args.policy and fixed_arena:
        # the link has room while refills run below 90% of the pinned-copy ceiling
        # measured in this run
        pcfg = kvs.kvs_policy_config(page_tokens=P, n_layers=L, budget_slots=free, min_ring_slots=8,
                                     max_ring_slots=free - L, step_slots=max(8, free // 16), hold_steps=1,
                                     miss_grow=0.25, copy_busy_max=0.9, occupancy_shrink=0.05,
                                     link_gbs=ceiling)
        # first decision from the context length alone
        pstate, dec = kvs.kvs_policy_step(pcfg, kvs.kvs_policy_state(),
                                          kvs.kvs_policy_observation(context_tokens=T))
        ring_now, per_now = dec.ring_slots, min(npages, int(dec.resident_pages_per_layer))
        policy_trace = []
        for k in range(args.policy):
            set_split(ring_now, per_now)
            st.graph_begin()
            step()
            st.graph_end()
            st.graph_launch()
            st.sync()
            st.observe(reset=True)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st.attn_stream)
            for _ in range(2):
                st.graph_launch()
            e1.record(st.attn_stream)
            st.sync()
            ms = e0.elapsed_time(e1) / 2
            obs = st.observe(reset=True)
            st.graph_destroy()
            pstate, dec = kvs.kvs_policy_step(pcfg, pstate, obs)
            policy_trace.append({
                "ring_slots": ring_now, "resident_pages_per_layer": per_now, "tokens_per_s": R / (ms * 1e-3),
                "streamed_reads": obs.streamed_reads, "ready_misses": obs.ready_misses,
                "ring_occupancy": obs.ring_occupancy, "copy_busy": obs.copy_busy,
                "refill_gbs": obs.copy_bytes / obs.interval_ns if obs.interval_ns else None,
                "decision": {"ring_slots": dec.ring_slots, "resident_pages_per_layer": dec.resident_pages_per_layer,
                             "reason": ["", "init", "fits", "hold", "grow", "shrink", "clamp"][dec.reason]}})
            ring_now = dec.ring_slots
            per_now = min(npages, int(dec.resident_pages_per_layer))
        forced = (ring_now, per_now)

    for frac in fracs:
        # residency (and, in a fixed arena, the ring gets every slot the pool does not)
        if fixed_arena:
            f = wl["residency"][1] if frac is None else frac
            pool_slots = int(round(f * (free - 8)))
            per_layer = min(npages, pool_slots // L)
            ring = free - per_layer * L
            if forced is not None:
                ring, per_layer = forced
            masks = []
            for _ in range(L):
                m = np.zeros(npages, np.uint8)
                m[:per_layer] = 1
                masks.append(m)
            for l in range(L):
                st.set_residency(l, np.zeros(npages, np.uint8))
            st.set_ring_slots(ring, wl["chunk"])
        else:
            masks = masks0
            ring = wl["ring"]
        for l in range(L):
            st.set_residency(l, masks[l])
        st.sync()

        # one eager (host-issued) step, timed for context
        t0 = time.perf_counter()
        step()
        st.sync()
        eager_ms = (time.perf_counter() - t0) * 1e3
        st.stats(reset=True)

        # capture the step once; replays re-execute every kernel and copy in it
        st.set_timing(0)
        st.graph_begin()
        step()
        st.graph_end()
        gstats = st.stats(reset=True)
        kernels_per_step = gstats["graph_kernels"]
        chunk_eff = int(gstats["chunk_pages"])
        h2d_bytes_step = gstats["h2d_bytes"]

        for _ in range(args.warmup):
            st.graph_launch()
        st.sync()
        clocks = ClockSampler(local)
        clocks.start()
        ms_step = timed(args.steps)
        clk = clocks.stop()
        st.sync()
        out_ref = out_d.detach().cpu().numpy()

        for _ in range(args.warmup):
            st.graph_launch()
        e2e_ms = timed(args.steps, e2e=True)
        h2d_in = q_h.numel() * q_h.element_size() + kn_h.numel() * 4 + vn_h.numel() * 4
        d2h_out = out_h.numel() * 4

        # roofline leg: host-issued steps with CUDA events around each attention
        # launch over device-resident pages (for prefill, every launch), timed in
        # their own region; graph-recorded events carry no timing
        st.graph_destroy()
        step()
        st.sync()
        st.stats(reset=True)
        st.set_timing(kvs.KVS_TIME_RESIDENT | (kvs.KVS_TIME_RING if prefill else 0))
        n_eager = max(3, min(args.steps, 10))
        t0 = time.perf_counter()
        for _ in range(n_eager):
            step()
        st.sync()
        ms_timed_eager = (time.perf_counter() - t0) * 1e3 / n_eager
        st.set_timing(0)
        rs = st.stats(reset=True)
        r_ms, r_n, r_bytes = rs["decode_ms"], rs["decode_timed"], rs["decode_bytes"]
        if prefill:  # tensor-core prefill: algorithmic flops over the timed launches
            flops_step = alg_flops_per_layer(wl) * L
            achieved = flops_step * n_eager / (r_ms * 1e-3) / 1e12 if r_ms > 0 else 0.0
            tr = TRAFFIC.get(args.workload) if args.split in (0, 24) and args.ring in (0, 24) else None
            roof = {"bound": "tensor", "achieved": achieved, "peak": tc_peak, "unit": "TFLOP/s",
                    "frac": achieved / tc_peak, "traffic": tr[0] if tr else None,
                    "traffic_source": tr[1] if tr else None,
                    "kernel": "prefill_kernel (tcgen05 kind::f16, M128 x N64/N256, TMEM accumulators)",
                    "flops_per_step_algorithmic": flops_step, "launches_timed": r_n,
                    "ms_per_launch": r_ms / max(r_n, 1),
                    "peak_source": peak_src + " bf16 burst (f16 runs at the same rate)",
                    "timed_region": f"{n_eager} host-issued steps ({ms_timed_eager:.2f} ms/step)"}
        else:
            achieved = (r_bytes / (r_ms * 1e-3) / 1e9) if r_ms > 0 else 0.0
            tr = TRAFFIC.get(args.workload)
            roof = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                    "frac": achieved / hbm_peak, "traffic": tr[0] if tr and L == WORKLOADS[args.workload]["L"] else None,
                    "traffic_source": tr[1] if tr else None,
                    "kernel": f"decode_kernel<{D},{math.ceil(R * Hq / Hk / 8)},8> launches over resident + tail pages",
                    "launches_timed": r_n, "bytes_per_launch": r_bytes / max(r_n, 1),
                    "ms_per_launch": r_ms / max(r_n, 1), "peak_source": peak_src + " hbm_gbs",
                    "timed_region": f"{n_eager} host-issued steps ({ms_timed_eager:.2f} ms/step)"}

        # timeline leg: the same step captured with every launch stamped, one replay read back
        st.graph_destroy()
        timeline = None
        if not args.no_timeline:
            st.timeline_begin(1 << 16)
            st.graph_begin()
            step()
            st.graph_end()
            st.timeline_end()
            for _ in range(args.warmup):
                st.timeline_zero()
                st.graph_launch()
            st.timeline_zero()
            st.graph_launch()
            st.sync()
            recs, dropped = st.timeline_read()
            st.graph_destroy()
            timeline = timeline_summary(recs, L)
            if timeline is not None:
                timeline["launches"] = len(recs)
                timeline["dropped"] = dropped
            # the roofline kernel timed inside the replayed step: its launches' device-clock
            # durations (first CTA start to last CTA end), not the host-issued timing leg
            kind = "prefill" if prefill else "read_resident"
            kl = [r for r in recs if r["kind"] == kind and r["start_ns"] and r["end_ns"]]
            if kl:
                dur_s = sum(r["end_ns"] - r["start_ns"] for r in kl) * 1e-9
                eager = {k: roof[k] for k in ("achieved", "frac", "ms_per_launch", "timed_region")}
                if prefill:
                    achieved = alg_flops_per_layer(wl) * L / dur_s / 1e12
                    roof.update(achieved=achieved, frac=achieved / tc_peak)
                else:
                    nbytes = sum(r["pages"] for r in kl) * st.page_bytes
                    achieved = nbytes / dur_s / 1e9
                    roof.update(achieved=achieved, frac=achieved / hbm_peak, bytes_per_launch=nbytes / len(kl))
                roof.update(ms_per_launch=dur_s * 1e3 / len(kl), launches_timed=len(kl),
                            timed_region=("one replay of the captured step, every launch stamped with the "
                                          "device clock (%globaltimer: first CTA start, last CTA end)"),
                            host_issued_events=eager)
            if args.timeline_out and rank == 0:
                with open(args.timeline_out, "w") as f:
                    f.write("kind,layer,stream,pages,start_us,end_us\n")
                    base = min((r["start_ns"] for r in recs if r["start_ns"]), default=0)
                    for r in recs:
                        f.write(f"{r['kind']},{r['layer']},{r['stream']},{r['pages']},"
                                f"{(r['start_ns'] - base) / 1e3 if r['start_ns'] else ''},"
                                f"{(r['end_ns'] - base) / 1e3 if r['end_ns'] else ''}\n")

        # CPU baseline (rank 0): the oracle on sampled layers/rows, scaled to the step
        cpu = parity = None
        if rank == 0 and cpu_layers and frac in (None, fracs[0]):
            import oracle
            tsum, errs = 0.0, []
            for l in cpu_layers:
                k, v = keep[l]
                t, o, lse = oracle_sample(wl, k, v, kn_h[l].numpy(), vn_h[l].numpy(),
                                          q_h[l].float().numpy(), rows_cpu)
                tsum += t
                g = out_ref[l][rows_cpu].astype(np.float64)
                errs.append(float((np.abs(g - o).max(axis=-1) / np.abs(o).max(axis=-1)).max()))
            step_s = tsum / len(cpu_layers) * L * R / len(rows_cpu)
            cpu = {"value": R / step_s, "unit": "tokens/s", "cores": oracle.threads(), "kind": "oracle",
                   "sample": (f"oracle fp64 attention of {len(rows_cpu)} of {R} rows on {len(cpu_layers)} of the "
                              f"{L} layers of one step ({Hq} heads x {T} keys), time scaled to the whole step")}
            parity = {"layers_checked": cpu_layers, "rows_checked": rows_cpu, "max_rel_err": max(errs), "tol": 1e-3}

        value = replicas.aggregate_rows_per_s(R, ms_step, world)
        kv_bytes_step = L * npages * st.page_bytes
        res_pages = int(sum(int(m.sum()) for m in masks))
        line = {
            "metric": "streamed-attention tokens/s", "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
            "config": {"workload": wl["desc"], "layers": L, "context": T, "rows": R, "q_heads": Hq, "kv_heads": Hk,
                       "head_dim": D, "page_tokens": P, "resident_pages_per_step": res_pages,
                       "resident_fraction": res_pages / (L * npages), "ring_slots": ring,
                       "chunk_pages": chunk_eff, "lanes": wl.get("lanes", 1),
                       "fill": "copy engines" if wl.get("dma") else "SM fill kernel",
                       "host_alloc": args.host_alloc,
                       "operands": ("single f16 (query and softmax weight x V scale rounded to f16; K/V codes exact; "
                                    "fp32 accumulation)" if args.operands == "f16" else
                                    "f16 hi + lo pairs (query and softmax weight x V scale); fp32 accumulation"),
                       "parallelism": f"replicas x{world}",
                       "l2": f"inputs larger than L2: {kv_bytes_step / 1e9:.2f} GB of KV pages read per step",
                       "step": "per layer: append rows, prefetch next layer, attend, truncate; one CUDA graph replay"},
            "kv_gbs": kv_bytes_step / (ms_step * 1e-3) / 1e9,
            "h2d": {"achieved_gbs": h2d_bytes_step / (ms_step * 1e-3) / 1e9, "ceiling_gbs": ceiling,
                    "frac": h2d_bytes_step / (ms_step * 1e-3) / 1e9 / ceiling, "bytes_per_step": h2d_bytes_step,
                    "ceiling_how": "pinned cudaMemcpyAsync 1 GiB, best of 5"},
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": {"value": replicas.aggregate_rows_per_s(R, e2e_ms, world), "unit": "tokens/s",
                    "h2d_bytes_per_step": h2d_in,
                    "d2h_bytes_per_step": d2h_out,
                    "how": ("every step: three pinned host -> device copies (all layers' Q, new K and new V "
                            "rows), one replay of the captured step graph (kvs_graph_launch), one device -> "
                            "pinned host copy of all layers' outputs, on the attention stream")},
            "gpu_launches": kernels_per_step * args.steps,
            "clocks": clk,
            "timeline": timeline,
            "policy": policy_trace,
            "eager_ms_per_step": eager_ms,
            "parity": parity,
            "prep_s": prep_s,
        }
        if prefill:
            line["tflops"] = alg_flops_per_layer(wl) * L / (ms_step * 1e-3) / 1e12
        if rank == 0:
            if args.extras and world == 1 and frac is None and args.workload == "decode32k" and not args.overridden:
                st.close()
                torch.cuda.synchronize(dev)
                torch.cuda.empty_cache()
                line["workloads"] = run_extras(args)
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
    ap.add_argument("--rows", type=int, default=0, help="override the workload's query rows")
    ap.add_argument("--resident", type=float, default=-1.0,
                    help="override the resident fraction (prefix of each layer; for long262k of the arena)")
    ap.add_argument("--sweep", action="store_true", help="long262k: sweep the resident fraction 0..100%%")
    ap.add_argument("--policy", type=int, default=0,
                    help="long262k: this many closed-loop steps of the residency policy choose the split first")
    ap.add_argument("--host-alloc", choices=["pageable", "pinned", "hugepage"], default="pinned",
                    help="host history buffer: registered numpy memory, CUDA pinned, or huge-page advised")
    ap.add_argument("--operands", choices=["split", "f16"], default="f16",
                    help="split-K attention operands: single f16 values (Q and P' rounded once), or f16 "
                         "hi + lo pairs (about 22 significant bits)")
    ap.add_argument("--no-timeline", action="store_true", help="skip the stamped-timeline replay")
    ap.add_argument("--no-extras", dest="extras", action="store_false",
                    help="do not run the other configurations after the default one")
    ap.add_argument("--timeline-out", default="", help="write the stamped launches of one step as CSV")
    ap.add_argument("--split", type=int, default=0, help="override the tensor-core prefill split (pages)")
    ap.add_argument("--fill", choices=["default", "sm", "dma"], default="default",
                    help="ring refills by the SM fill kernel or the copy engines (default: the workload's)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    wl = dict(WORKLOADS[args.workload])
    wl.update(wl.pop("geom", GEOM))
    for key, name in (("ring", "ring"), ("chunk", "chunk"), ("layers", "L"), ("lanes", "lanes"), ("split", "split")):
        v = getattr(args, key)
        if v:
            wl[name] = v
            wl["desc"] += f" [{key} override: {v}]"
    if args.fill != "default":
        wl["dma"] = args.fill == "dma"
        wl["desc"] += f" [fill override: {args.fill}]"
    if args.rows:
        wl["T"] = wl["T"] - wl["R"] + args.rows
        wl["R"] = args.rows
        wl["desc"] += f" [rows override: {args.rows}]"
    if args.resident >= 0:
        kind = "arena_frac" if wl["residency"][0] == "arena_frac" else "prefix_frac"
        wl["residency"] = (kind, args.resident)
        wl["desc"] += f" [resident override: {args.resident}]"
    args.overridden = any((args.ring, args.chunk, args.layers, args.lanes, args.rows, args.split, args.policy,
                           args.resident >= 0,
                           args.fill != "default", args.sweep))
    if args.impl == "reference":
        run_reference(args, wl)
    else:
        run_ours(args, wl)


if __name__ == "__main__":
    main()
