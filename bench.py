#!/usr/bin/env python
"""Benchmark: ring / context-parallel attention forward on GB300.

One step = one ring_attn_fwd call over the whole workload (all N virtual
ranks, all ring steps, in one launch).  Default workload: B=1, H=8,
S=131072, D=128, N=16 virtual ranks, zigzag, causal, bf16.  The metric is
TFLOP/s on masked-in FLOPs (4*D per visible (query, key) pair).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With N > 1 (torchrun, one process per GPU) the GPUs form a real ring: the
same sequence is sharded over the N ranks (zigzag, 2N chunks), each rank runs
N flash_block_step launches while the K/V blocks travel rank -> rank + 1 over
NCCL point-to-point (ring.P2PTransport), and the line reports the whole
sequence's masked-in FLOPs over the slowest rank's time ("scaling": "strong",
the total work is fixed).  ``--impl reference`` times the fp64 CPU oracle on
the host cores on a bounded sample of the same workload (rank 0 only).

Prints one JSON line.
"""
from __future__ import annotations

import argparse
import datetime
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "ring-attn fwd TFLOP/s (masked-in FLOPs) and % of GB300 BF16 dense peak"
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK), "fallback"


def workload(name):
    import torch
    from context_parallelism_02_gb300 import inputs
    table = {
        "long128k_zigzag": inputs.LONG128K,
        "long128k_contiguous": inputs.LONG128K.with_(layout=inputs.CONTIGUOUS),
        "long128k_striped": inputs.LONG128K.with_(layout=inputs.STRIPED),
        "s8192": inputs.S8K,
        "gqa32k": inputs.GQA32K,
    }
    w = table[name]
    assert w.dtype == torch.bfloat16
    return w


def masked_pairs(w):
    return w.S * (w.S + 1) // 2 if w.causal else w.S * w.S


def fwd_flops(w):
    return 4 * w.D * w.B * w.Hq * masked_pairs(w)


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,timestamp")

    def __init__(self, dev_index, uuid=None, period_ms=200):
        self.dev = uuid or str(dev_index)
        self.period_ms = period_ms
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.dev, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)

    def stop(self, windows=None):
        """Summary of the samples.  windows: {name: [(t0, t1), ...]} in
        time.time() seconds; adds each window set's median SM clock and mean
        power (samples whose timestamp falls inside)."""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        rows = []
        if self.path and os.path.exists(self.path):
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) >= 9 and parts[1].isdigit():
                        rows.append(parts)
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        sm = [int(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        power = [float(r[3]) for r in rows if r[3].replace(".", "", 1).isdigit()]
        out = {"sm_mhz": statistics.median(sm), "sm_max_mhz": int(rows[0][2]),
               "reasons": reasons, "samples": len(rows),
               "power_w_max": max(power) if power else None}
        for name, spans in (windows or {}).items():
            inside = []
            for r in rows:
                try:
                    t = datetime.datetime.strptime(r[9], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                except (ValueError, IndexError):
                    continue
                if any(a <= t <= b for a, b in spans):
                    inside.append(r)
            pw = [float(r[3]) for r in inside if r[3].replace(".", "", 1).isdigit()]
            out[name] = {"sm_mhz": statistics.median(int(r[1]) for r in inside) if inside else None,
                         "power_w_mean": round(sum(pw) / len(pw), 1) if pw else None, "samples": len(inside)}
        return out


def clocks_rejected(c):
    bad = {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}
    if bad & set(c.get("reasons", [])):
        return True
    if c.get("sm_mhz") and c.get("sm_max_mhz") and not c["reasons"]:
        return c["sm_mhz"] < 0.5 * c["sm_max_mhz"]
    return False


# ----------------------------------------------------------------------------- oracle timing

_QKV_CACHE = {}


def oracle_per_config():
    """The fp64 oracle on the other forward workloads: the tiny one and S=8192
    in full, the GQA S=32768 one on a row sample (seconds each)."""
    import oracle
    from context_parallelism_02_gb300 import inputs
    oracle.build()
    res = {}
    for w in (inputs.TINY, inputs.S8K):
        q, k, v = inputs.make_qkv(w)
        t0 = time.perf_counter()
        oracle.attn_fwd(q, k, v, w.causal)
        dt = time.perf_counter() - t0
        res[w.name] = {"s": dt, "TFLOP/s": fwd_flops(w) / dt / 1e12, "rows": "all"}
    w = inputs.GQA32K
    tf, dt, n, _ = oracle_sample_rows(w, target_s=3.0)
    res[w.name] = {"s": dt, "TFLOP/s": tf, "rows": f"{n} random query rows x {w.Hq} heads"}
    return res


def oracle_sample_rows(w, target_s, seed=0):
    """Time the fp64 oracle on a bounded sample of query rows of the workload.

    Rows are drawn uniformly over positions (all heads of batch 0); the
    sample's masked-in FLOPs are counted exactly.  Returns (tflops, seconds,
    rows, threads)."""
    import numpy as np
    import oracle
    from context_parallelism_02_gb300 import inputs
    oracle.build()
    key = (w.name, w.seed)
    if key not in _QKV_CACHE:
        q, k, v = inputs.make_qkv(w)
        _QKV_CACHE[key] = (q[:1], k[:1], v[:1])
    q, k, v = _QKV_CACHE[key]
    rng = np.random.default_rng(seed)

    def run(nrows):
        rows = np.sort(rng.integers(0, w.S, nrows))
        t0 = time.perf_counter()
        oracle.attn_fwd(q, k, v, w.causal, rows=rows)
        dt = time.perf_counter() - t0
        keys = (rows + 1).sum() if w.causal else nrows * w.S
        return 4.0 * w.D * w.Hq * keys / dt / 1e12, dt, nrows

    tf, dt, n = run(16)                                  # calibration
    n = int(max(16, min(50000, 16 * target_s / max(dt, 1e-3))))
    tf, dt, n = run(n)
    return tf, dt, n, oracle.num_threads()


def run_reference(args, w, rank):
    if rank != 0:
        return
    steps = []
    sample_desc = None
    for i in range(args.warmup + args.steps):
        tf, dt, n, cores = oracle_sample_rows(w, target_s=args.ref_seconds, seed=i)
        if i >= args.warmup:
            steps.append((tf, dt))
        sample_desc = (f"{n} random query rows x {w.Hq} heads of the workload per step "
                       f"(~{dt:.1f} s of fp64 CPU work), masked-in FLOPs counted exactly")
    value = statistics.median(t for t, _ in steps)
    ms = statistics.median(d for _, d in steps) * 1e3
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "strong", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_of(w, args.workload),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample_desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_of(w, name):
    from context_parallelism_02_gb300.inputs import LAYOUT_NAMES
    return {"workload": name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "S": w.S, "D": w.D,
            "N_virtual_ranks": w.N, "layout": LAYOUT_NAMES[w.layout], "causal": w.causal,
            "seed": w.seed, "masked_in_flops_per_step": fwd_flops(w),
            "l2": "inputs larger than L2 (q,k,v %.0f MB vs 129 MB); no flush"
                  % (3 * w.B * w.S * w.Hq * w.D * 2 / 1e6)}


# ----------------------------------------------------------------------------- extras

def time_events(fn, reps, stream):
    import torch
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        fn()
    e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) / reps


def extras(dev, stream, peaks):
    """lse_merge and Ulysses relayout bandwidth, per-rank work/time of the long
    workload for contiguous vs zigzag vs striped, and the backward."""
    import torch
    from context_parallelism_02_gb300 import api, inputs
    hbm = peaks["hbm_gbs"]
    out = {}
    # the other forward workloads of the scope table: tiny fp32 (S=512, D=64,
    # N=4), S=8192 (H=8, N=8) and GQA S=32768 (Hq=32, Hkv=8, N=8), zigzag, causal
    cfgs = {}
    for w in (inputs.TINY, inputs.S8K, inputs.GQA32K):
        g = torch.Generator(device=dev).manual_seed(w.seed)
        q = torch.randn(w.B, w.S, w.Hq, w.D, device=dev, generator=g).to(w.dtype)
        k, v = (torch.randn(w.B, w.S, w.Hkv, w.D, device=dev, generator=g).to(w.dtype) for _ in range(2))
        o = torch.empty_like(q)
        lo = torch.empty(w.B, w.Hq, w.S, device=dev)
        f = lambda: api.ring_attn_fwd(q, k, v, w.N, w.layout, w.causal, out=o, lse=lo, stream=stream)
        for _ in range(3):
            f()
        ms = time_events(f, 20, stream)
        tf = fwd_flops(w) / ms / 1e9
        entry = {"dtype": str(w.dtype).replace("torch.", ""), "ms": ms, "TFLOP/s": tf,
                 "masked_in_flops": fwd_flops(w)}
        if w.dtype == torch.bfloat16:
            entry["frac_bf16_burst"] = tf / peaks["bf16_tflops"]
        cfgs[w.name] = entry
        del q, k, v, o, lo
    out["configs_fwd"] = cfgs
    # lse_merge: rows = 1x8x131072, D = 128, fp32 partials
    a, la, b, lb = (t.to(dev) for t in inputs.make_merge_inputs())
    o = torch.empty_like(a)
    lo = torch.empty_like(la)
    rows, D = la.numel(), a.shape[1]
    nbytes = 3 * rows * D * 4 + 3 * rows * 4
    f = lambda: api.lse_merge(a, la, b, lb, out=o, lse=lo, stream=stream)
    for _ in range(3):
        f()
    ms = time_events(f, 20, stream)
    out["lse_merge"] = {"rows": rows, "D": D, "bytes": nbytes, "ms": ms,
                        "GB/s": nbytes / ms / 1e6, "frac_hbm": nbytes / ms / 1e6 / hbm}
    del a, la, b, lb, o, lo
    # lse_merge_n: n = 4 partials of the same rows (one pass, (n+1)(D+1)*4 B per row)
    n_parts = 4
    xs, ls = (t.to(dev) for t in inputs.make_merge_n_inputs(n_parts))
    o = torch.empty(rows, D, device=dev)
    lo = torch.empty(rows, device=dev)
    nbytes = (n_parts + 1) * rows * (D + 1) * 4
    f = lambda: api.lse_merge_n(xs, ls, out=o, lse=lo, stream=stream)
    for _ in range(3):
        f()
    ms = time_events(f, 20, stream)
    out["lse_merge_n4"] = {"rows": rows, "D": D, "n": n_parts, "bytes": nbytes, "ms": ms,
                           "GB/s": nbytes / ms / 1e6, "frac_hbm": nbytes / ms / 1e6 / hbm}
    del xs, ls, o, lo
    # Ulysses relayout of the GQA workload's q (N=8, S=32768, H=32, D=128, bf16, zigzag)
    N, B, S, H, D = 8, 1, 32768, 32, 128
    x = torch.randn(N, B, S // N, H, D, device=dev).to(torch.bfloat16)
    y = torch.empty(N, B, S, H // N, D, device=dev, dtype=torch.bfloat16)
    x2 = torch.empty_like(x)
    nb = 2 * x.numel() * 2
    res = {}
    for name, fn in (("seq_to_head", lambda: api.ulysses_seq_to_head(x, N, 1, y=y, stream=stream)),
                     ("head_to_seq", lambda: api.ulysses_head_to_seq(y, N, 1, x=x2, stream=stream))):
        for _ in range(3):
            fn()
        ms = time_events(fn, 20, stream)
        res[name] = {"ms": ms, "GB/s": nb / ms / 1e6, "frac_hbm": nb / ms / 1e6 / hbm}
    torch.cuda.synchronize()
    res["bit_exact_roundtrip"] = bool(torch.equal(x, x2))
    res["bytes"] = nb
    out["ulysses_q_gqa32k"] = res
    del x, y, x2
    # USP on the GQA workload: n_ulysses x n_ring = 8 virtual ranks, each grid
    # against the plain ring over 8 ranks (relayouts included in the time)
    w = inputs.GQA32K
    g = torch.Generator(device=dev).manual_seed(w.seed)
    q = torch.randn(w.B, w.S, w.Hq, w.D, device=dev, generator=g).to(torch.bfloat16)
    k, v = (torch.randn(w.B, w.S, w.Hkv, w.D, device=dev, generator=g).to(torch.bfloat16) for _ in range(2))
    o = torch.empty_like(q)
    lo = torch.empty(w.B, w.Hq, w.S, device=dev)
    usp = {}
    for nu in (1, 2, 4, 8):
        nr = 8 // nu
        if nu == 1:
            f = lambda: api.ring_attn_fwd(q, k, v, nr, w.layout, True, out=o, lse=lo, stream=stream)
        else:
            ws = torch.empty(api._lib.load().usp_attn_fwd_workspace(w.Hq, w.Hkv, w.S, w.D, 1),
                             dtype=torch.uint8, device=dev)
            f = lambda: api.usp_attn_fwd(q, k, v, nu, nr, w.layout, True, out=o, lse=lo,
                                         workspace=ws, stream=stream)
        for _ in range(3):
            f()
        ms = time_events(f, 10, stream)
        usp[f"{nu}x{nr}"] = {"ms": ms, "TFLOP/s": fwd_flops(w) / ms / 1e9}
    out["usp_gqa32k"] = {"grid": "n_ulysses x n_ring (1 x 8 is the plain ring)", **usp}
    del q, k, v, o, lo
    # per-rank work and time, long workload, contiguous vs zigzag vs striped
    w = inputs.LONG128K
    g = torch.Generator(device=dev).manual_seed(w.seed)
    q = torch.randn(w.B, w.S, w.Hq, w.D, device=dev, generator=g).to(torch.bfloat16)
    k = torch.randn(w.B, w.S, w.Hkv, w.D, device=dev, generator=g).to(torch.bfloat16)
    v = torch.randn(w.B, w.S, w.Hkv, w.D, device=dev, generator=g).to(torch.bfloat16)
    ob = torch.empty_like(q)
    lb_ = torch.empty(w.B, w.Hq, w.S, device=dev)
    per = {}
    for layout in (inputs.CONTIGUOUS, inputs.ZIGZAG, inputs.STRIPED):
        pairs, tiles = api.cp_schedule_pairs(w.S, w.N, layout, True)
        whole = lambda: api.ring_attn_fwd(q, k, v, w.N, layout, True, out=ob, lse=lb_, stream=stream)
        whole()
        ms_all = time_events(whole, 3, stream)
        times = []
        for r in range(w.N):
            fn = lambda: api.ring_attn_fwd(q, k, v, w.N, layout, True, out=ob, lse=lb_,
                                           stream=stream, rank_range=(r, r + 1))
            fn()
            times.append(time_events(fn, 3, stream))
        work = (pairs.sum(1) * w.B * w.Hq).tolist()
        # the same per-rank launches split-KV (ring_attn_fwd_split) at the count
        # cp_fwd_split_count picks for each rank
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        nsp = [api.cp_fwd_split_count(w.B, w.Hq, w.S, w.D, w.N, layout, True, (r, r + 1), sms)
               for r in range(w.N)]
        ws = torch.empty(max(16, api.ring_attn_fwd_split_workspace(w.B, w.Hq, w.S, w.D, max(nsp))),
                         dtype=torch.uint8, device=dev)
        times_split = []
        for r in range(w.N):
            fn = lambda: api.ring_attn_fwd_split(q, k, v, w.N, layout, True, n_split=nsp[r], out=ob,
                                                 lse=lb_, workspace=ws, stream=stream,
                                                 rank_range=(r, r + 1))
            fn()
            times_split.append(time_events(fn, 3, stream))
        del ws
        per[inputs.LAYOUT_NAMES[layout]] = {
            "n_split_per_rank": nsp,
            "ms_per_rank_split": times_split,
            "split_max_rank_ms_vs_unsplit": [max(times_split), max(times)],
            "masked_in_pairs_per_rank": work,
            "work_max_over_mean": max(work) / (sum(work) / len(work)),
            "ms_per_rank": times,
            "time_max_over_mean": max(times) / (sum(times) / len(times)),
            "ms_all_ranks": ms_all,
            "TFLOP/s_all_ranks": fwd_flops(w) / ms_all / 1e9,
            "executed_tiles_128x256": int(tiles.sum()) * w.B * w.Hq,
        }
    out["per_rank_long128k"] = per
    # the real ring's per-step launches: every (rank, step) of the long
    # workload as flash_block_step on shard-local buffers (the launches one
    # device of a 16-GPU ring makes), ranks run one after another; and the
    # link rate at which a K/V hop would hide under one step's compute
    from context_parallelism_02_gb300 import ring
    lay = inputs.ZIGZAG
    C = w.S // w.N
    qs = [ring.shard(q, r, w.N, lay) for r in range(w.N)]
    ks = [ring.shard(k, r, w.N, lay) for r in range(w.N)]
    vs = [ring.shard(v, r, w.N, lay) for r in range(w.N)]
    oacc = torch.empty(w.B, C, w.Hq, w.D, device=dev)
    lacc = torch.empty(w.B, w.Hq, C, device=dev)
    ofin = torch.empty_like(qs[0])

    def ring_rank(r):
        for s_ in range(w.N):
            src = (r - s_) % w.N
            api.flash_block_step(qs[r], ks[src], vs[src], r, src, w.N, w.S, lay, True,
                                 out_acc=oacc, lse_acc=lacc,
                                 out_final=ofin if s_ == w.N - 1 else None, accumulate=s_ > 0,
                                 stream=stream)

    rank_ms = []
    for r in range(w.N):
        ring_rank(r)
        rank_ms.append(time_events(lambda: ring_rank(r), 3, stream))
    hop = 2 * w.B * C * w.Hkv * w.D * 2
    step_ms = sum(rank_ms) / len(rank_ms) / w.N
    out["ring_steps_long128k"] = {
        "ms_all_ranks_one_after_another": sum(rank_ms),
        "ms_fused_ring_attn_fwd": per["zigzag"]["ms_all_ranks"],
        "slowest_rank_ms": max(rank_ms), "rank_time_max_over_mean": max(rank_ms) / (sum(rank_ms) / len(rank_ms)),
        "step_ms_mean": step_ms, "hop_bytes": hop,
        "link_GBs_to_hide_hop": hop / (step_ms * 1e6),
        "slowest_rank_TFLOPs": fwd_flops(w) / w.N / max(rank_ms) / 1e9}
    del qs, ks, vs, oacc, lacc, ofin
    del q, k, v, ob, lb_
    # split-KV forward where it pays: one head of the long workload, one rank
    # per launch (64 query tiles of up to 512 KV tiles for 152 SMs), zigzag;
    # each rank unsplit and at the count cp_fwd_split_count picks
    w = inputs.LONG128K.with_(Hq=1, Hkv=1)
    g = torch.Generator(device=dev).manual_seed(w.seed)
    q, k, v = (torch.randn(w.B, w.S, 1, w.D, device=dev, generator=g).to(torch.bfloat16)
               for _ in range(3))
    ob = torch.empty_like(q)
    lb_ = torch.empty(w.B, 1, w.S, device=dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    nsp = [api.cp_fwd_split_count(w.B, 1, w.S, w.D, w.N, w.layout, True, (r, r + 1), sms)
           for r in range(w.N)]
    ws = torch.empty(api.ring_attn_fwd_split_workspace(w.B, 1, w.S, w.D, max(nsp)),
                     dtype=torch.uint8, device=dev)
    t_un, t_sp = [], []
    for r in range(w.N):
        fu = lambda: api.ring_attn_fwd(q, k, v, w.N, w.layout, True, out=ob, lse=lb_, stream=stream,
                                       rank_range=(r, r + 1))
        fs = lambda: api.ring_attn_fwd_split(q, k, v, w.N, w.layout, True, n_split=nsp[r], out=ob,
                                             lse=lb_, workspace=ws, stream=stream,
                                             rank_range=(r, r + 1))
        for f in (fu, fs):
            f()
        t_un.append(time_events(fu, 5, stream))
        t_sp.append(time_events(fs, 5, stream))
    out["split_kv_one_head_long128k"] = {
        "workload": "B=1, H=1, S=131072, D=128, N=16, zigzag, causal; one launch per rank",
        "n_split_per_rank": nsp, "ms_per_rank_unsplit": t_un, "ms_per_rank_split": t_sp,
        "max_rank_ms_unsplit": max(t_un), "max_rank_ms_split": max(t_sp),
        "speedup_max_rank": max(t_un) / max(t_sp)}
    del q, k, v, ob, lb_, ws
    # backward: B=2, H=16, S=32768, D=128, N=8, zigzag, causal
    w = inputs.BWD32K
    g = torch.Generator(device=dev).manual_seed(w.seed)
    q, k, v, do = (torch.randn(w.B, w.S, w.Hq, w.D, device=dev, generator=g).to(torch.bfloat16)
                   for _ in range(4))
    o, l = api.ring_attn_fwd(q, k, v, w.N, w.layout, True, stream=stream)
    ws = torch.empty(api.ring_attn_bwd_workspace(w.B, w.Hq, w.S), dtype=torch.uint8, device=dev)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    fn = lambda: api.ring_attn_bwd(q, k, v, o, l, do, w.N, w.layout, True, dq=dq, dk=dk, dv=dv,
                                   workspace=ws, stream=stream)
    for _ in range(3):
        fn()
    ms = time_events(fn, 5, stream)
    pairs = masked_pairs(w)
    alg = 10 * w.D * w.B * w.Hq * pairs
    out["ring_attn_bwd_bwd32k"] = {
        "ms": ms, "flops_algorithmic": alg, "TFLOP/s": alg / ms / 1e9,
        "frac_bf16_burst": alg / ms / 1e9 / peaks["bf16_tflops"],
        "executed_TFLOP/s": 14 * w.D * w.B * w.Hq * pairs / ms / 1e9,
        "note": "algorithmic 10*D FLOPs per masked-in pair; the kernels execute 14*D "
                "(dQ recomputes S and dP instead of using atomics)"}
    return out


def _r(x, sig=4):
    return float(f"{x:.{sig}g}") if isinstance(x, float) and math.isfinite(x) else x


def rounded(obj):
    """Floats to 4 significant digits (keeps the JSON line short)."""
    if isinstance(obj, dict):
        return {k: rounded(v) for k, v in obj.items()}
    if isinstance(obj, (list, tuple)):
        return [rounded(v) for v in obj]
    return _r(obj)


def compact_extras(full):
    """Scalar summaries of the extras: per-rank arrays become max/mean ratios."""
    c = {}
    for name, e in full.get("configs_fwd", {}).items():
        c[f"fwd_{name.split('_')[0]}_ms"] = e["ms"]
        c[f"fwd_{name.split('_')[0]}_TFLOPs"] = e["TFLOP/s"]
    b = full.get("ring_attn_bwd_bwd32k")
    if b:
        c["bwd32k_ms"] = b["ms"]
        c["bwd32k_TFLOPs_alg"] = b["TFLOP/s"]
        c["bwd32k_frac_burst"] = b["frac_bf16_burst"]
    for lay, e in full.get("per_rank_long128k", {}).items():
        c[f"long128k_{lay}_ms"] = e["ms_all_ranks"]
        c[f"long128k_{lay}_rank_time_max_over_mean"] = e["time_max_over_mean"]
        c[f"long128k_{lay}_rank_work_max_over_mean"] = e["work_max_over_mean"]
        c[f"long128k_{lay}_slowest_rank_ms_unsplit_split"] = e["split_max_rank_ms_vs_unsplit"][::-1]
    sk = full.get("split_kv_one_head_long128k")
    if sk:
        c["split_1head_slowest_rank_ms_unsplit_split"] = [sk["max_rank_ms_unsplit"],
                                                          sk["max_rank_ms_split"]]
    u = full.get("usp_gqa32k")
    if u:
        c["usp_gqa32k_ms"] = {k: v["ms"] for k, v in u.items() if isinstance(v, dict)}
    for key in ("ring_steps_long128k",):
        if key in full:
            c[key] = full[key]
    return c


def hbm_summary(full, peaks):
    out = {"peak_GBs": peaks["hbm_gbs"]}
    for key, name in (("lse_merge", "lse_merge"), ("lse_merge_n4", "lse_merge_n4")):
        if key in full:
            out[name] = {"GB/s": full[key]["GB/s"], "frac_hbm": full[key]["frac_hbm"]}
    u = full.get("ulysses_q_gqa32k")
    if u:
        for d in ("seq_to_head", "head_to_seq"):
            out[f"ulysses_{d}"] = {"GB/s": u[d]["GB/s"], "frac_hbm": u[d]["frac_hbm"]}
        out["ulysses_roundtrip_bit_exact"] = u["bit_exact_roundtrip"]
    return out


# ----------------------------------------------------------------------------- real ring (N > 1)

def _timed(run, steps, warmup, world, device):
    """ms per call of run() on this rank (CUDA events on the current stream, or
    the host clock for CPU tensors), bracketed by a barrier and a device sync;
    returns (max over ranks, this rank's)."""
    import torch
    import torch.distributed as dist
    for _ in range(warmup):
        run()
    cuda = device.type == "cuda"
    if cuda:
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    if cuda:
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
    t0 = time.perf_counter()
    for _ in range(steps):
        run()
    if cuda:
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / steps
    else:
        ms = (time.perf_counter() - t0) * 1e3 / steps
    if world > 1:
        dist.barrier()
    return max_over_ranks(ms, world, device if cuda else "cpu"), ms


def ring_measure(q, k, v, *, rank, world, S, layout, causal, steps, warmup, transport,
                 blocks, step=None, state_dtype=None):
    """Time one rank's part of a real ring three ways: the whole ring (compute
    with the transfers overlapped), its N compute steps alone (the other
    ranks' blocks taken from ``blocks``, as if already received), and its
    N - 1 transfers alone.  q, k, v: this rank's shards; blocks[src] = (k, v)
    of every rank.  Returns a dict of ms (max over ranks) and the fraction of
    the transfer time hidden under compute."""
    import torch
    from context_parallelism_02_gb300 import ring
    kw = dict(rank=rank, N=world, S=S, layout=layout, causal=causal)
    step = step or ring.cuda_step
    sdt = state_dtype or torch.float32
    run_ring = lambda: ring.ring_attention(q, k, v, transport=transport, step=step,
                                           state_dtype=sdt, **kw)
    B, C, Hq, D = q.shape
    oacc = torch.empty((B, C, Hq, D), dtype=sdt, device=q.device)
    lacc = torch.empty((B, Hq, C), dtype=sdt, device=q.device)

    def run_compute():
        for s in range(world):
            src = (rank - s) % world
            step(q, blocks[src][0], blocks[src][1], oacc, lacc, None, source=src, scale=None,
                 accumulate=s > 0, **kw)

    bufs = [(torch.empty_like(k), torch.empty_like(v)) for _ in range(2)]

    def run_comm():
        cur = (k, v)
        for s in range(world - 1):
            h = transport.start(cur, bufs[s % 2])
            transport.wait(h)
            cur = bufs[s % 2]

    dev = q.device
    ms_ring, ms_ring_local = _timed(run_ring, steps, warmup, world, dev)
    ms_comp, _ = _timed(run_compute, steps, warmup, world, dev)
    ms_comm, _ = _timed(run_comm, steps, warmup, world, dev)
    hidden = (ms_comp + ms_comm - ms_ring) / ms_comm if ms_comm > 0 else None
    hop_bytes = 2 * k.numel() * k.element_size()
    return {"ms_ring": ms_ring, "ms_ring_local": ms_ring_local, "ms_compute": ms_comp,
            "ms_transfers": ms_comm, "transfer_hidden_frac": hidden, "hop_bytes": hop_bytes,
            "hop_GBs": hop_bytes * (world - 1) / (ms_comm * 1e6) if ms_comm > 0 else None}


def main_ring(args, w, world, rank, local, dev, stream, peaks):
    """N > 1: the GPUs of the job form one ring over the workload's sequence."""
    import torch
    import torch.distributed as dist
    from context_parallelism_02_gb300 import api, inputs, ring
    wl = w.with_(N=world)
    q, k, v = inputs.make_qkv(wl)
    pos_layout = wl.layout
    qs, ks, vs = (ring.shard(x, rank, world, pos_layout).to(dev) for x in (q, k, v))
    blocks = [tuple(ring.shard(x, r, world, pos_layout).to(dev) for x in (k, v)) for r in range(world)]
    del q, k, v
    # NCCL moves the blocks GPU to GPU; over a gloo group (CP_BENCH_BACKEND=gloo,
    # e.g. several ranks sharing one GPU in a test) they go through pinned host
    # memory
    transport = (ring.P2PTransport() if dist.get_backend() == "nccl"
                 else ring.HostStagedTransport())
    sampler = ClockSampler(dev.index)
    sampler.start()
    m = ring_measure(qs, ks, vs, rank=rank, world=world, S=wl.S, layout=wl.layout,
                     causal=wl.causal, steps=args.steps, warmup=args.warmup,
                     transport=transport, blocks=blocks)
    clocks = sampler.stop()
    assert api.cp_get_error() == 0
    flops = fwd_flops(wl)
    value = flops / (m["ms_ring"] * 1e-3) / 1e12
    achieved_local = flops / world / (m["ms_compute"] * 1e-3) / 1e12
    # end to end: this rank's shards uploaded from pinned host memory, the
    # ring, and this rank's out and lse read back, every step
    qh, kh, vh = (t.cpu().pin_memory() for t in (qs, ks, vs))
    dq, dk, dv = (torch.empty_like(t) for t in (qs, ks, vs))
    outs_h = {}

    def e2e():
        for d_, h_ in zip((dq, dk, dv), (qh, kh, vh)):
            d_.copy_(h_, non_blocking=True)
        o, l = ring.ring_attention(dq, dk, dv, rank=rank, N=world, S=wl.S, layout=wl.layout,
                                   causal=wl.causal, transport=transport)
        if not outs_h:
            outs_h["o"] = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
            outs_h["l"] = torch.empty(l.shape, dtype=l.dtype, pin_memory=True)
        outs_h["o"].copy_(o, non_blocking=True)
        outs_h["l"].copy_(l, non_blocking=True)

    e2e_ms, _ = _timed(e2e, max(3, min(args.steps, 10)), 2, world, dev)
    h2d = sum(t.numel() * t.element_size() for t in (qh, kh, vh))
    d2h = outs_h["o"].numel() * outs_h["o"].element_size() + outs_h["l"].numel() * 4
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": m["ms_ring"],
        "higher_is_better": True, "scaling": "strong", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) q, k, v drawn on the host)",
        "config": {**config_of(wl, args.workload), "parallelism": f"ring over {world} GPUs (NCCL P2P)"},
        "roofline": {"bound": "tensor", "achieved": achieved_local,
                     "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": achieved_local / peaks["bf16_tflops"], "traffic": None,
                     "kernel": "fwd_bf16_kernel<128, 2> (flash_block_step), per GPU",
                     "note": "one GPU's masked-in FLOPs over its compute-only steps"},
        "clocks": clocks,
        "e2e": {"value": flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "note": "per rank: its shards uploaded from pinned memory, the ring, out and lse "
                        "read back; h2d/d2h bytes are one rank's"},
        "gpu_launches": args.steps * world,
        "ring": rounded(m),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- ranks

def max_over_ranks(x, world, device):
    """Max of a per-rank float over all ranks (identity with one rank)."""
    import torch
    import torch.distributed as dist
    if world > 1 and dist.get_backend() == "gloo":
        device = "cpu"   # gloo reduces host tensors
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(flops_per_rank, world, ms_max):
    """Whole-job TFLOP/s: every rank's work over the slowest rank's time."""
    return world * flops_per_rank / (ms_max * 1e-3) / 1e12


# ----------------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="long128k_zigzag")
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-seconds", type=float, default=6.0)
    ap.add_argument("--extras-full", action="store_true",
                    help="print every per-rank array of the extras (a long line)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    w = workload(args.workload)

    if args.impl == "reference":
        run_reference(args, w, rank)
        return

    import torch
    import torch.distributed as dist
    from context_parallelism_02_gb300 import api, build, inputs

    build.build()
    # one GPU per rank; ranks beyond the visible GPUs share them (tests only)
    dev = torch.device("cuda", local % max(1, torch.cuda.device_count()))
    torch.cuda.set_device(dev)
    if world > 1:
        backend = os.environ.get("CP_BENCH_BACKEND", "nccl")
        if backend == "nccl":
            dist.init_process_group("nccl", device_id=dev)
        else:
            dist.init_process_group(backend)
    peaks, peak_src = load_peaks()
    # one ordinary stream for all work of this process (the legacy default
    # stream would order itself against the end-to-end copy streams)
    stream = torch.cuda.Stream(dev)
    torch.cuda.set_stream(stream)
    if world > 1:
        main_ring(args, w, world, rank, local, dev, stream, peaks)
        dist.destroy_process_group()
        return

    # inputs: drawn on the host (seeded), pinned, copied once to HBM
    qh, kh, vh = (t.pin_memory() for t in inputs.make_qkv(w))
    q, k, v = (t.to(dev, non_blocking=True) for t in (qh, kh, vh))
    out = torch.empty_like(q)
    lse = torch.empty(w.B, w.Hq, w.S, device=dev)
    step = lambda: api.ring_attn_fwd(q, k, v, w.N, w.layout, w.causal, out=out, lse=lse,
                                     stream=stream)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert api.cp_get_error() == 0

    def timed():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        sampler = ClockSampler(local, getattr(torch.cuda.get_device_properties(dev), "uuid", None)
                               and "GPU-" + str(torch.cuda.get_device_properties(dev).uuid))
        sampler.start()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        clocks = sampler.stop()
        if world > 1:
            dist.barrier()
        ms = e0.elapsed_time(e1) / args.steps
        return max_over_ranks(ms, world, dev), ms, clocks

    ms_max, ms_local, clocks = timed()
    remeasured = False
    if clocks_rejected(clocks):
        ms_max, ms_local, clocks = timed()
        remeasured = True
    assert api.cp_get_error() == 0

    flops = fwd_flops(w)
    value = job_value(flops, world, ms_max)
    achieved = flops / (ms_local * 1e-3) / 1e12
    long_run = args.steps * ms_local >= 1000.0
    peak = peaks["bf16_tflops_sustained"] if long_run else peaks["bf16_tflops"]
    peak_kind = "sustained" if long_run else "burst"

    # end to end through the public call with host buffers: every step uploads
    # its q, k, v from pinned host memory, runs the forward and reads out and
    # lse back.  Steps are pipelined the way a streaming caller would run them:
    # two device buffer sets, uploads on one copy stream and read-backs on
    # another (the host link is full duplex), ordered by events, so that the
    # copies of step i+1 and i-1 overlap the forward of step i.  All copies of
    # the timed steps lie inside the timed region.
    # as many pipelined steps as the timed region (at least 3): the first
    # upload and the last read-back of a repetition cannot overlap a forward,
    # and more steps spread them thinner
    e2e_steps = max(3, min(args.steps, 50))
    ins = [(q, k, v), tuple(torch.empty_like(t) for t in (q, k, v))]
    outs = [(out, lse), (torch.empty_like(out), torch.empty_like(lse))]
    outs_h = [tuple(torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in o) for o in outs]
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = {key: [torch.cuda.Event() for _ in range(2)] for key in ("in", "done", "out")}

    def upload(b):
        for d_, h_ in zip(ins[b], (qh, kh, vh)):
            d_.copy_(h_, non_blocking=True)
        ev["in"][b].record(up)

    def e2e_run(n):
        """n pipelined steps; returns after the last read-back is queued."""
        with torch.cuda.stream(up):
            upload(0)
        for i in range(n):
            b = i & 1
            stream.wait_event(ev["in"][b])
            if i >= 2:
                stream.wait_event(ev["out"][b])        # step i-2's outputs are read back
            api.ring_attn_fwd(*ins[b], w.N, w.layout, w.causal, out=outs[b][0], lse=outs[b][1],
                              stream=stream)
            ev["done"][b].record(stream)
            if i + 1 < n:
                with torch.cuda.stream(up):
                    if i >= 1:
                        up.wait_event(ev["done"][b ^ 1])   # step i-1 no longer reads set b^1
                    upload(b ^ 1)
            with torch.cuda.stream(down):
                down.wait_event(ev["done"][b])
                for h_, d_ in zip(outs_h[b], outs[b]):
                    h_.copy_(d_, non_blocking=True)
                ev["out"][b].record(down)
        stream.wait_stream(down)

    e2e_run(2)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    # clocks during the end-to-end steps too: the copies share the board's
    # power budget with the SMs
    e2e_sampler = ClockSampler(local, getattr(torch.cuda.get_device_properties(dev), "uuid", None)
                               and "GPU-" + str(torch.cuda.get_device_properties(dev).uuid), 50)
    e2e_sampler.start()
    # three repetitions of the pipelined steps, each with all its copies inside
    # its own timed region; the median is reported (the host link of these
    # boxes drops for a while now and then from ~208 GB/s to ~15 GB/s, and a
    # repetition that catches such a drop is copy-bound)
    e2e_all, fwd_only_all = [], []
    spans = {"fwd_only_phase": [], "e2e_phase": []}   # host wall-clock windows of each phase
    for _ in range(3):
        # the same forward with inputs already in HBM, timed right before the
        # end-to-end steps, so both see the same clocks and power state
        h0 = time.time()
        t0.record(stream)
        for _ in range(e2e_steps):
            step()
        t1.record(stream)
        torch.cuda.synchronize()
        spans["fwd_only_phase"].append((h0, time.time()))
        fwd_only_all.append(t0.elapsed_time(t1) / e2e_steps)
        h0 = time.time()
        t0.record(stream)
        up.wait_event(t0)
        e2e_run(e2e_steps)
        t1.record(stream)
        torch.cuda.synchronize()
        spans["e2e_phase"].append((h0, time.time()))
        e2e_all.append(t0.elapsed_time(t1) / e2e_steps)
    e2e_clocks = e2e_sampler.stop(spans)
    # what the copies do to the forward: one forward with the next step's whole
    # upload running beside it on the copy stream, with the upload and a
    # read-back of the previous outputs beside it (both directions, as in the
    # pipelined steps), against the same forward and the upload alone (CUDA
    # events; medians of three)
    conc = {"fwd_alone": [], "fwd_with_upload": [], "upload_alone": [], "fwd_with_upload_and_readback": []}
    for _ in range(3):
        for key in conc:
            torch.cuda.synchronize()
            a0 = torch.cuda.Event(enable_timing=True)
            a1 = torch.cuda.Event(enable_timing=True)
            a0.record(stream)
            up.wait_event(a0)
            down.wait_event(a0)
            if key != "upload_alone":
                step()
            if key != "fwd_alone":
                with torch.cuda.stream(up):
                    upload(1)
            if key == "fwd_with_upload_and_readback":
                with torch.cuda.stream(down):
                    for h_, d_ in zip(outs_h[1], outs[1]):
                        h_.copy_(d_, non_blocking=True)
            stream.wait_stream(up)
            stream.wait_stream(down)
            a1.record(stream)
            torch.cuda.synchronize()
            conc[key].append(a0.elapsed_time(a1))
    assert api.cp_get_error() == 0
    e2e_ms = max_over_ranks(statistics.median(e2e_all), world, dev)
    fwd_only_ms = max_over_ranks(statistics.median(fwd_only_all), world, dev)
    h2d = sum(x.numel() * x.element_size() for x in (qh, kh, vh))
    d2h = out.numel() * out.element_size() + lse.numel() * lse.element_size()
    # the host link alone (one upload, one read-back, nothing else running): the
    # pipelined steps are copy-bound when (h2d + d2h) / link rate exceeds the
    # forward's time
    link = {}
    for name, st_, fn in (("h2d", up, lambda: upload(0)),
                          ("d2h", down, lambda: [h_.copy_(d_, non_blocking=True)
                                                 for h_, d_ in zip(outs_h[0], outs[0])])):
        rates = []
        for _ in range(3):
            torch.cuda.synchronize()
            a0 = torch.cuda.Event(enable_timing=True)
            a1 = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(st_):
                a0.record(st_)
                fn()
                a1.record(st_)
            torch.cuda.synchronize()
            rates.append((h2d if name == "h2d" else d2h) / a0.elapsed_time(a1) / 1e6)
        link[name] = statistics.median(rates)
        link[name + "_min"] = min(rates)

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
        "higher_is_better": True, "scaling": "strong", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) q, k, v drawn on the host)",
        "config": config_of(w, args.workload),
        "pct_of_bf16_peak": 100.0 * achieved / peak,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak,
                     "unit": "TFLOP/s", "frac": achieved / peak, "traffic": None,
                     "peak_source": f"{peak_src} bf16 dense ({peak_kind}; timed region "
                                    f"{args.steps * ms_local / 1e3:.2f} s)",
                     "frac_of_burst": achieved / peaks["bf16_tflops"],
                     "kernel": "fwd_bf16_kernel<128, 0> (ring mode)",
                     "flops_per_launch": flops},
        "clocks": clocks,
        "e2e": {"value": job_value(flops, world, e2e_ms), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "steps": e2e_steps,
                "fwd_only_ms_per_step": fwd_only_ms,
                "e2e_over_fwd_only": e2e_ms / fwd_only_ms,
                "rep_ms_min": min(e2e_all), "rep_ms_max": max(e2e_all),
                "link_h2d_gbs": link["h2d"], "link_d2h_gbs": link["d2h"],
                "link_h2d_gbs_min": link["h2d_min"], "link_d2h_gbs_min": link["d2h_min"],
                "copy_ms_per_step": h2d / link["h2d"] / 1e6 + d2h / link["d2h"] / 1e6,
                "fwd_alone_ms": statistics.median(conc["fwd_alone"]),
                "fwd_with_concurrent_upload_ms": statistics.median(conc["fwd_with_upload"]),
                "fwd_with_upload_and_readback_ms": statistics.median(conc["fwd_with_upload_and_readback"]),
                "upload_alone_ms": statistics.median(conc["upload_alone"]),
                "sm_mhz": e2e_clocks.get("sm_mhz"),
                "power_w_max": e2e_clocks.get("power_w_max"),
                "reasons": ",".join(e2e_clocks.get("reasons", [])),
                # the same samples split by phase (host wall-clock windows): the
                # copies draw on the board's power budget beside the SMs
                "sm_mhz_fwd_only_phase": (e2e_clocks.get("fwd_only_phase") or {}).get("sm_mhz"),
                "sm_mhz_e2e_phase": (e2e_clocks.get("e2e_phase") or {}).get("sm_mhz"),
                "power_w_fwd_only_phase": (e2e_clocks.get("fwd_only_phase") or {}).get("power_w_mean"),
                "power_w_e2e_phase": (e2e_clocks.get("e2e_phase") or {}).get("power_w_mean"),
                "phase_samples": [(e2e_clocks.get(k) or {}).get("samples") for k in ("fwd_only_phase", "e2e_phase")],
                "note": "pinned host buffers; uploads and read-backs of neighbouring steps "
                        "overlap the forward on two copy streams; fwd_only_ms_per_step is the "
                        "device-only forward timed just before each repetition (same clocks)"},
        "gpu_launches": args.steps,
    }
    if remeasured:
        line["clocks"]["remeasured"] = True
    traffic = os.path.join(ROOT, "profiles", "fwd_bf16_traffic.json")
    if os.path.exists(traffic):
        with open(traffic) as f:
            tr = json.load(f)
        if tr.get("workload") == args.workload and tr.get("kernel_source_sha") == kernel_sha():
            line["roofline"]["traffic"] = tr["bytes_per_launch"]

    full = None
    if rank == 0 and world == 1 and not args.no_extras:
        full = extras(dev, stream, peaks)
        line["extras"] = full if args.extras_full else compact_extras(full)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tf, dt, n, cores = oracle_sample_rows(w, target_s=12.0)
        line["cpu_baseline"] = {
            "value": tf, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} random query rows x {w.Hq} heads of the workload ({dt:.1f} s, "
                      f"fp64, OpenMP); masked-in FLOPs of the sample counted exactly"}
        if args.extras_full:
            line["cpu_baseline"]["per_config"] = oracle_per_config()
    if full is not None:
        # the HBM-bound kernels last, so that they survive any truncation of the
        # line from the front
        line["hbm_kernels"] = rounded(hbm_summary(full, peaks))
    if "extras" in line:
        line["extras"] = rounded(line["extras"])
    keep = {k: line["e2e"][k] for k in ("value", "ms_per_step")}
    line["e2e"] = {**rounded(line["e2e"]), **keep}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def kernel_sha():
    """Hash of the forward kernel's code (comments and whitespace removed): the
    recorded DRAM traffic stays valid while this is unchanged."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in ("fwd_bf16_sm103.cu", "cp_common.cuh", "tmem_io.cuh", "tc_helpers.cuh"):
        with open(os.path.join(ROOT, "context_parallelism_02_gb300", "csrc", f)) as fh:
            src = fh.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


if __name__ == "__main__":
    main()
