#!/usr/bin/env python
"""Benchmark of the dense attention backward on GB300 (one JSON line).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one call of attn_bwd_dense (C ABI) on the workload
``dense_bf16_s2048``: bf16 Q, K, V, dY [B=4, S=2048, H=16, D=128] ~ N(0,1)*0.5,
causal (bottom-right) + custom per-key mask (10% zeros, < 0.5 -> -1e9) +
additive bias [B,H,Sq,Sk] ~ N(0,1), self-contained mode (the row statistics
are recomputed from Q, K, V, dY).  The call runs the whole hot path: the
row-statistics prologue, the dK/dV kernel (which also stores every dS tile,
ATTN_OPT_STORE_DS) and the dQ kernel (dQ = scale * dS K over those tiles);
--recompute-dq times the default dQ kernel, which recomputes S and dP.

Metric: attention-backward TFLOP/s counted as 10 * D * (visible query/key
pairs) per head (five products of 2*D flops each), visible = allowed by the
causal mask; custom-masked keys are computed and counted.  Inputs stay resident
in HBM; the per-step working set (bias 512 MiB + Q, K, V, dY 128 MiB) is larger
than the 129 MB L2, so no flush is needed between steps.

Under torchrun (N > 1) every rank runs the same workload on its own GPU (weak
scaling, no data-path collective); the time is the max over ranks.  The
reference arm (--impl reference) times the CPU oracle on the host cores on a
bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attn-bwd TFLOP/s (dQ+dK+dV) on 1 GB300; % of tensor-core dense peak"
WORKLOAD = "dense_bf16_s2048"
WORKLOAD_DESC = ("dense SDPA backward, bf16 in / fp32 accumulate, B=4 H=16 Sq=Sk=2048 D=128, [B,S,H,D], "
                 "N(0,1)*0.5 inputs, causal + custom per-key mask (10% zeros, thr 0.5 -> -1e9) + additive "
                 "bias [B,H,Sq,Sk] ~ N(0,1) bf16, self-contained (row statistics recomputed)")


def visible_pairs(sq: int, sk: int, causal: bool, window) -> int:
    """Structurally visible (query, key) pairs, bottom-right aligned."""
    q_off = max(sk - sq, 0)
    tot = 0
    for q in range(sq):
        aq = q + q_off
        hi = sk - 1
        lo = 0
        if causal or window is not None:
            hi = min(hi, aq)
        if window is not None:
            lo = max(0, aq - window)
        tot += max(0, hi - lo + 1)
    return tot


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples taken while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        # raw samples: $BENCH_CLOCKS_DIR/clocks_rank<i>.csv if set, else a temporary file
        import tempfile
        d = os.environ.get("BENCH_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(d, f"clocks_rank{index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as fh:
            for line in fh:
                f = [x.strip() for x in line.split(",")]
                if len(f) < 9:
                    continue
                try:
                    rows.append(dict(sm=float(f[1]), smax=float(f[2]), power=float(f[3]), hw=f[5], hwt=f[6],
                                     swt=f[7], pcap=f[8]))
                except ValueError:
                    continue
        if not rows:
            return None
        # samples under load: the highest-power half
        pw = sorted(r["power"] for r in rows)
        cut = pw[len(pw) // 2]
        load = [r for r in rows if r["power"] >= cut] or rows
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in load), "sm_max_mhz": max(r["smax"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows), "power_w_max": max(r["power"] for r in rows)}


# DRAM bytes per launch of the dominant kernel, from the committed ncu summary,
# scaled from the captured case to this launch by the number of (batch, head)
# pairs; None when the kernel sources changed since the capture.
TRAFFIC_PROFILES = {
    "dkdv": ("profiles/dkdv2_kernel_dense_bf16_b2h8.md",
             ["dense_dkdv2.cu", "sm103.cuh", "dense_common.cuh", "dense_launch.h"]),
}


def recorded_traffic(kernel: str, units: int):
    import hashlib
    import re
    if kernel not in TRAFFIC_PROFILES:
        return None
    prof, files = TRAFFIC_PROFILES[kernel]
    try:
        text = open(os.path.join(ROOT, prof)).read()
        h = hashlib.sha256()
        for f in files:
            with open(os.path.join(ROOT, "attention_backward_recompute_gb300", "csrc", f), "rb") as fh:
                h.update(fh.read())
    except OSError:
        return None
    fields = dict(re.findall(r"^\s*(dram_bytes_per_launch|units_per_launch|sources_sha256):\s*(\S+)", text, re.M))
    if len(fields) != 3 or fields["sources_sha256"] != h.hexdigest():
        return None
    return float(fields["dram_bytes_per_launch"]) * units / float(fields["units_per_launch"])


def cpu_baseline(case, budget_s: float):
    """The oracle as it stands, on the host cores, on a bounded sample of heads."""
    import numpy as np  # noqa: F401
    from oracle import attn_bwd_dense
    B, H = case.batch, case.heads
    vp = visible_pairs(case.seq_q, case.seq_k, case.causal, case.window)
    per_head = 10.0 * case.head_dim * vp
    order = [(b, h) for b in range(B) for h in range(H)]
    done = 0
    t0 = time.perf_counter()
    while done < len(order):
        attn_bwd_dense(case.q, case.k, case.v, case.dy, layout=case.layout, causal=case.causal,
                       window=case.window, key_mask=case.key_mask, bias=case.bias, heads_subset=[order[done]])
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"value": per_head * done / dt / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{done} of {B * H} (batch, head) pairs of {WORKLOAD}, float64 numpy, {dt:.1f} s"}


def rank_max(x: float, dist, device) -> float:
    """The largest x over the ranks (x itself without a process group): the
    timing rule of the multi-GPU line is the slowest rank's time."""
    if not dist:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_reference(args, rank, world):
    """--impl reference: the CPU oracle timed on the host, K steps of one head each."""
    if rank != 0:
        return 0
    from attention_backward_recompute_gb300 import inputs
    from oracle import attn_bwd_dense
    case = inputs.dense_config(WORKLOAD)
    vp = visible_pairs(case.seq_q, case.seq_k, case.causal, case.window)
    per_head = 10.0 * case.head_dim * vp
    order = [(b, h) for b in range(case.batch) for h in range(case.heads)]

    def step(i):
        attn_bwd_dense(case.q, case.k, case.v, case.dy, layout=case.layout, causal=case.causal,
                       window=case.window, key_mask=case.key_mask, bias=case.bias,
                       heads_subset=[order[i % len(order)]])

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    dt = time.perf_counter() - t0
    value = per_head * args.steps / dt / 1e12
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "description": WORKLOAD_DESC,
                       "step": "oracle backward of one (batch, head) pair of the workload"},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": "one (batch, head) pair per step, float64 numpy"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def sweep(args) -> int:
    """Every configuration once (not the bench contract line): GPU time (CUDA
    events, median of reps), counted TFLOP/s or GB/s, % of the measured peak,
    max error against the oracle on a sample, and the oracle's own time on that
    sample with the extrapolation to the whole configuration labelled as such.
    One JSON line per configuration."""
    import numpy as np
    import torch
    from attention_backward_recompute_gb300 import binding as bd
    from attention_backward_recompute_gb300 import build, inputs
    from oracle import attn_bwd_dense, attn_bwd_paged, attn_fwd_dense, paged_query_backward
    build.build()
    bd.lib()
    peaks, src = load_peaks()
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()

    def timed(fn, reps):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        bd.check_device_error()
        return statistics.median(ts), min(ts)

    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")

    def timed_flushed(fn, reps):
        # a 256 MiB write (twice L2) between repetitions, outside the timed region
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            flush_buf.fill_(1)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        return statistics.median(ts)

    def oracle_one_thread(name, heads, over):
        # the oracle with its BLAS held to one thread, in a child process (the
        # thread count of a loaded BLAS cannot be changed in place)
        import subprocess
        code = ("import json, sys, time; sys.path.insert(0, %r)\n"
                "from attention_backward_recompute_gb300 import inputs\n"
                "from oracle import attn_bwd_dense\n"
                "c = inputs.dense_config(%r)\n"
                "over = %r\n"
                "km = None if over.get('no_mask_bias') else c.key_mask\n"
                "bias = None if over.get('no_mask_bias') else c.bias\n"
                "t0 = time.perf_counter()\n"
                "attn_bwd_dense(c.q, c.k, c.v, c.dy, layout=c.layout, causal=c.causal, window=c.window, "
                "key_mask=km, bias=bias, heads_subset=%r)\n"
                "print(json.dumps(time.perf_counter() - t0))\n") % (ROOT, name, over, heads)
        env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
        r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
        return float(r.stdout.strip().splitlines()[-1]) if r.returncode == 0 else None

    def rel(got, want, mask=None):
        g = got.float().cpu().numpy().astype(np.float64)
        if mask is not None:
            g, want = g[mask], want[mask]
        return float(np.max(np.abs(g - want)) / max(np.max(np.abs(want)), 1e-30))

    def emit(d):
        print(json.dumps(d), flush=True)

    only = re.compile(args.only) if args.only else None

    def want(tag):
        return only is None or only.search(tag) is not None

    dense = [("C1", "dense_small_f32", {}), ("C2c", "dense_f32_causal", {}), ("C2w", "dense_f32_window", {}),
             ("C3", "dense_bf16_s2048", {}), ("C3 causal only", "dense_bf16_s2048", {"no_mask_bias": True}),
             ("C3 O+LSE supplied", "dense_bf16_s2048", {"supplied": True}),
             ("C4", "dense_bf16_cross", {}),
             ("C3 stored dS", "dense_bf16_s2048", {"store_ds": True}),
             ("C3 O+LSE supplied, stored dS", "dense_bf16_s2048", {"supplied": True, "store_ds": True}),
             ("C4 stored dS", "dense_bf16_cross", {"store_ds": True})]
    for tag, name, opt in dense:
        if not want(tag):
            continue
        c = inputs.dense_config(name)
        dt = torch.float32 if c.dtype == "f32" else torch.bfloat16
        t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda().to(dt)
        q, k, v, dy = t(c.q), t(c.k), t(c.v), t(c.dy)
        if opt.get("no_mask_bias"):  # the same shape without key mask and bias: what the bias reads cost
            c.key_mask = c.bias = None
        km = None if c.key_mask is None else torch.from_numpy(c.key_mask).cuda()
        bias = None if c.bias is None else t(c.bias)
        o = lse = None
        if opt.get("supplied"):
            o_np, lse_np = attn_fwd_dense(c.q, c.k, c.v, layout=c.layout, causal=c.causal, window=c.window,
                                          key_mask=c.key_mask, bias=c.bias)
            o = t(o_np)
            lse = torch.from_numpy(lse_np.astype(np.float32)).cuda()
        outs = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
        call = lambda: bd.dense_backward(q, k, v, dy, layout=c.layout, causal=c.causal, window=c.window,
                                         key_mask=km, bias=bias, o=o, lse=lse, outputs=outs,
                                         store_ds=bool(opt.get("store_ds")))
        reps = 20 if c.seq_q * c.seq_k * c.batch * c.heads > 1e7 else 50
        ms, ms_min = timed(call, reps)
        ms_flushed = timed_flushed(call, reps)
        # per-kernel split of one call (fp32 storage first splits its inputs)
        names = (["split"] if c.dtype == "f32" else []) + ["prologue", "dkdv", "dq"]
        kev = [torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)]
        for e in kev:  # CUDA events are created on first record
            e.record()
        torch.cuda.synchronize()
        bd.attn_set_timing_events([e.cuda_event for e in kev])
        call()
        torch.cuda.synchronize()
        kernel_ms = {n: kev[i].elapsed_time(kev[i + 1]) for i, n in enumerate(names)}
        vp = visible_pairs(c.seq_q, c.seq_k, c.causal, c.window)
        flops = 10.0 * c.head_dim * vp * c.batch * c.heads
        heads = [(b, h) for b in range(c.batch) for h in range(c.heads)]
        sample = heads if len(heads) <= 16 else [heads[0], heads[len(heads) // 2], heads[-1]]
        t0 = time.perf_counter()
        ref = attn_bwd_dense(c.q, c.k, c.v, c.dy, layout=c.layout, causal=c.causal, window=c.window,
                             key_mask=c.key_mask, bias=c.bias, heads_subset=sample)
        t_or = time.perf_counter() - t0
        res = call()
        torch.cuda.synchronize()
        errs = []
        for g, w in zip(res, ref):
            gh = g.float().cpu().numpy().astype(np.float64)
            if c.layout == "bshd":
                gs = np.stack([gh[b, :, h] for b, h in sample]); ws = np.stack([w[b, :, h] for b, h in sample])
            else:
                gs = np.stack([gh[b, h] for b, h in sample]); ws = np.stack([w[b, h] for b, h in sample])
            errs.append(float(np.max(np.abs(gs - ws)) / max(np.max(np.abs(ws)), 1e-30)))
        tflops = flops / (ms * 1e-3) / 1e12
        # algorithmic bytes: q, dy, dq and k, v, dk, dv once, the visible bias once, the key mask
        es = 4 if c.dtype == "f32" else 2
        alg_bytes = (es * c.head_dim * c.batch * c.heads * (3 * c.seq_q + 4 * c.seq_k) +
                     (2 * vp * c.batch * c.heads if c.bias is not None else 0) +
                     (4 * c.batch * c.seq_k if c.key_mask is not None else 0))
        one = None
        if tag in ("C1", "C2c", "C2w", "C3"):
            h1 = heads[:1] if tag == "C3" else heads
            t1 = oracle_one_thread(name, h1, dict(opt))
            if t1 is not None:
                one = {"s": t1, "sample": f"{len(h1)} of {len(heads)} (batch, head) pairs",
                       "s_extrapolated": t1 * len(heads) / len(h1)}
        emit({"config": tag, "workload": name, "gpu_ms_median": ms, "gpu_ms_min": ms_min, "kernel_ms": kernel_ms,
              "gpu_ms_median_l2_flushed": ms_flushed, "l2_flush": "256 MiB write between repetitions",
              "algorithmic_gbs": alg_bytes / (ms * 1e-3) / 1e9,
              "pct_of_hbm_peak": 100.0 * alg_bytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
              "oracle_one_thread": one,
              "counted_tflops": tflops, "pct_of_bf16_peak": 100.0 * tflops / peaks["bf16_tflops"],
              "max_err_rel": max(errs), "tolerance": 2e-4 if c.dtype == "f32" else 2e-2,
              "oracle_s_sample": t_or, "oracle_sample": f"{len(sample)} of {len(heads)} (batch, head) pairs",
              "oracle_s_extrapolated": t_or * len(heads) / len(sample), "host_cores": cores,
              "peak_source": src})

    # forward export (O and LSE) on the headline shape
    if want("C3 forward export"):
        c = inputs.dense_config("dense_bf16_s2048")
        t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda().to(torch.bfloat16)
        q, k, v = t(c.q), t(c.k), t(c.v)
        km = torch.from_numpy(c.key_mask).cuda()
        bias = t(c.bias)
        fo = (torch.empty_like(q), torch.empty((c.batch, c.heads, c.seq_q), dtype=torch.float32, device="cuda"))
        fcall = lambda: bd.dense_forward(q, k, v, layout=c.layout, causal=c.causal, window=c.window, key_mask=km,
                                         bias=bias, outputs=fo)
        fms, fms_min = timed(fcall, 20)
        vp = visible_pairs(c.seq_q, c.seq_k, c.causal, c.window)
        fflops = 4.0 * c.head_dim * vp * c.batch * c.heads
        sample = [(0, 0), (3, 15)]
        from oracle import attn_fwd_dense as fwd_oracle
        t0 = time.perf_counter()
        o_ref, lse_ref = fwd_oracle(c.q, c.k, c.v, layout=c.layout, causal=c.causal, window=c.window,
                                    key_mask=c.key_mask, bias=c.bias)
        ft_or = time.perf_counter() - t0
        g = fo[0].float().cpu().numpy()
        ferr = max(float(np.max(np.abs(g[b_, :, h_] - o_ref[b_, :, h_])) / np.max(np.abs(o_ref[b_, :, h_])))
                   for b_, h_ in sample)
        emit({"config": "C3 forward export (O, LSE)", "workload": "dense_bf16_s2048", "gpu_ms_median": fms,
              "gpu_ms_min": fms_min, "counted_tflops": fflops / (fms * 1e-3) / 1e12,
              "pct_of_bf16_peak": 100.0 * fflops / (fms * 1e-3) / 1e12 / peaks["bf16_tflops"],
              "flops_counted": "4*D per visible pair (S = Q K^T, O = P V)", "max_err_rel_o": ferr, "tolerance": 2e-2,
              "oracle_s": ft_or, "oracle_sample": "all 64 (batch, head) pairs, error on 2", "host_cores": cores,
              "peak_source": src})

    # the two paged workloads, then the same with a 1024-token prefix (64
    # pages) shared by every sequence
    for tag, name, ov in (("C5g", "paged_gqa", {}), ("C5m", "paged_mla", {}),
                          ("C5g prefix1024", "paged_gqa", {"shared_prefix_pages": 64}),
                          ("C5m prefix1024", "paged_mla", {"shared_prefix_pages": 64})):
        if not want(tag):
            continue
        if args.seqs is not None:
            ov = dict(ov, num_seqs=args.seqs)
        c = inputs.paged_config(name, **ov)
        tb = lambda x: None if x is None else torch.from_numpy(np.ascontiguousarray(x)).cuda().to(torch.bfloat16)
        dv = dict(q=tb(c.q), dy=tb(c.dy), k=tb(c.k_pool), v=tb(c.v_pool), qp=tb(c.qp), kp=tb(c.kp_pool))
        table = torch.from_numpy(c.page_table).cuda().contiguous()
        meta = bd.seq_meta_tensor(c.seq_len, c.q_start, c.q_pos, "cuda")
        lse, delta = bd.paged_row_stats(dv["q"], dv["k"], dv["v"], dv["dy"], table, meta, heads=c.heads,
                                        kv_heads=c.kv_heads, page_size=c.page_size, causal=c.causal,
                                        qp=dv["qp"], kp_pool=dv["kp"])
        first = bd.paged_backward(dv["q"], dv["k"], dv["v"], dv["dy"], table, meta, lse, delta, heads=c.heads,
                                  kv_heads=c.kv_heads, page_size=c.page_size, causal=c.causal, qp=dv["qp"],
                                  kp_pool=dv["kp"])
        buf = tuple(torch.empty_like(x) for x in first)
        outs = (buf[0], None, buf[1]) if c.position_dim else (buf[0], buf[1], None)
        call = lambda: bd.paged_backward(dv["q"], dv["k"], dv["v"], dv["dy"], table, meta, lse, delta,
                                         heads=c.heads, kv_heads=c.kv_heads, page_size=c.page_size,
                                         causal=c.causal, outputs=outs, qp=dv["qp"], kp_pool=dv["kp"])
        ms, ms_min = timed(call, 20)
        # per-kernel split of one call: links, zero store, history (MLA: plan, the cluster-split kernel,
        # then the history kernel; the recorded events keep these two from overlapping in this one call)
        names = (["links", "zero_unlinked", "plan", "history_split", "history"] if c.position_dim
                 else ["links", "zero_unlinked", "history"])
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)]
        for e in evs:  # CUDA events are created on first record
            e.record()
        torch.cuda.synchronize()
        bd.attn_set_timing_events([e.cuda_event for e in evs])
        call()
        torch.cuda.synchronize()
        kernel_ms = {n: evs[i].elapsed_time(evs[i + 1]) for i, n in enumerate(names)}
        compact = None
        if "shared_prefix_pages" not in ov:
            # compact history listing the referenced pages only: the zero store
            # of the unreferenced pool pages is skipped
            ref_pages = np.unique(np.concatenate([c.page_table[s_, :(int(c.seq_len[s_]) + c.page_size - 1) // c.page_size]
                                                  for s_ in range(c.num_seqs)])).astype(np.int32)
            hist = torch.from_numpy(ref_pages).cuda()
            ccall = lambda: bd.paged_backward(dv["q"], dv["k"], dv["v"], dv["dy"], table, meta, lse, delta,
                                              heads=c.heads, kv_heads=c.kv_heads, page_size=c.page_size,
                                              causal=c.causal, outputs=outs, qp=dv["qp"], kp_pool=dv["kp"],
                                              history_pages=hist)
            cms, _ = timed(ccall, 20)
            compact = {"gpu_ms_median": cms, "listed_pages": int(ref_pages.size), "pool_pages": int(c.num_pages)}
        stats_call = lambda: bd.paged_row_stats(dv["q"], dv["k"], dv["v"], dv["dy"], table, meta, heads=c.heads,
                                                kv_heads=c.kv_heads, page_size=c.page_size, causal=c.causal,
                                                qp=dv["qp"], kp_pool=dv["kp"])
        stats_ms, _ = timed(stats_call, 10)
        stable = all(torch.equal(a, b) for a, b in zip(first, call()))
        for _ in range(3):
            stable = stable and all(torch.equal(a, b) for a, b in zip(first, call()))
        triples = int(sum(int(p) + 1 for p in c.q_pos)) * c.heads if c.causal else None
        kvh, dk_, dvv = c.kv_heads, c.key_dim, c.value_dim
        valid = int(np.sum(c.seq_len))
        slots = c.num_pages * c.page_size
        if c.position_dim:
            flops = (2 * (dk_ + c.position_dim) + 2 * dvv + 4 * dvv + 2 * c.position_dim) * triples
            alg_bytes = (valid * kvh * (dk_ + c.position_dim) * 2 + slots * kvh * (dk_ + c.position_dim) * 2 +
                         c.q.shape[0] * c.heads * (dk_ + c.position_dim + dvv) * 2)
        else:
            flops = 1024 * triples * dk_ // 128
            alg_bytes = (valid * kvh * (dk_ + dvv) * 2 + slots * kvh * (dk_ + dvv) * 2 +
                         c.q.shape[0] * c.heads * (dk_ + dvv) * 2)
        pick = [0, c.num_seqs // 2]
        qs = [np.arange(c.q_start[s], c.q_start[s + 1]) for s in pick]
        rows = np.concatenate(qs)
        sub = np.concatenate([[0], np.cumsum([len(x) for x in qs])]).astype(np.int32)
        t0 = time.perf_counter()
        ref = attn_bwd_paged(c.q[rows], c.dy[rows], c.k_pool, c.page_table[pick], c.seq_len[pick], sub,
                             c.q_pos[rows], page_size=c.page_size, kv_heads=c.kv_heads, v_pool=c.v_pool,
                             qp=None if c.qp is None else c.qp[rows], kp_pool=c.kp_pool, causal=c.causal)
        t_or = time.perf_counter() - t0
        # compare the slots of pages that only the sampled sequences map
        owned = np.zeros(slots, bool)
        for s_ in pick:
            for tok in range(int(c.seq_len[s_])):
                owned[int(c.page_table[s_, tok // c.page_size]) * c.page_size + tok % c.page_size] = True
        for s_ in set(range(c.num_seqs)) - set(pick):
            for lp in range((int(c.seq_len[s_]) + c.page_size - 1) // c.page_size):
                ph = int(c.page_table[s_, lp])
                owned[ph * c.page_size:(ph + 1) * c.page_size] = False
        err = max(rel(g, w, owned) for g, w in zip(first, ref))
        emit({"config": tag, "workload": name, **({"shared_prefix_pages": ov["shared_prefix_pages"]} if "shared_prefix_pages" in ov else {}),
              "gpu_ms_median": ms, "gpu_ms_min": ms_min,
              "counted_tflops": flops / (ms * 1e-3) / 1e12,
              "pct_of_bf16_peak": 100.0 * flops / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"],
              "algorithmic_gbs": alg_bytes / (ms * 1e-3) / 1e9,
              "pct_of_hbm_peak": 100.0 * alg_bytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
              "row_stats_ms": stats_ms, "kernel_ms": kernel_ms, "compact_history_referenced_pages": compact,
              "max_err_rel": err, "tolerance": 2e-2, "bit_stable_5_runs": bool(stable),
              "oracle_s_sample": t_or, "oracle_sample": f"{len(pick)} of {c.num_seqs} sequences",
              "oracle_s_extrapolated": t_or * c.num_seqs / len(pick), "host_cores": cores,
              "peak_source": src})
        # query side (row statistics and dQ, dQp for MLA, in one call)
        mla = bool(c.position_dim)
        qouts = (torch.empty((c.q.shape[0], c.heads), dtype=torch.float32, device="cuda"),
                 torch.empty((c.q.shape[0], c.heads), dtype=torch.float32, device="cuda"), torch.empty_like(dv["q"]))
        if mla:
            qouts = qouts + (torch.empty_like(dv["qp"]),)
        qcall = lambda: bd.paged_query_backward(dv["q"], dv["k"], dv["v"], dv["dy"], table, meta, heads=c.heads,
                                                kv_heads=c.kv_heads, page_size=c.page_size, causal=c.causal,
                                                qp=dv["qp"], kp_pool=dv["kp"], outputs=qouts)
        qcall()
        qfirst = tuple(x.clone() for x in qouts)
        qms, qms_min = timed(qcall, 20)
        qstable = all(torch.equal(a, b) for a, b in zip(qfirst, qouts))
        if mla:  # statistics: S (576), dP (512); query: S, dP again, dQ and dQp (576)
            qflops = (2 * (dk_ + c.position_dim) + 2 * dvv) * 2 * triples + 2 * (dk_ + c.position_dim) * triples
            qbytes = valid * kvh * (dk_ + c.position_dim) * 2 + c.q.shape[0] * c.heads * (
                2 * (dk_ + c.position_dim) + dvv) * 2
            qdesc = "per visible (row, head, token): S and dP twice (576 + 512), dQ and dQp (576)"
        else:
            qflops = (6 * dk_ + 4 * dvv) * triples  # S twice, O += P V, dP, dQ += dS K
            qbytes = valid * kvh * (dk_ + dvv) * 2 + c.q.shape[0] * c.heads * (2 * dk_ + dvv) * 2
            qdesc = "10*D per visible (row, head, token): S twice, O += P V, dP, dQ += dS K"
        t0 = time.perf_counter()
        qref = paged_query_backward(c.q[rows], c.dy[rows], c.k_pool, c.page_table[pick], c.seq_len[pick], sub,
                                    c.q_pos[rows], page_size=c.page_size, kv_heads=c.kv_heads, v_pool=c.v_pool,
                                    qp=None if c.qp is None else c.qp[rows], kp_pool=c.kp_pool, causal=c.causal)
        qt_or = time.perf_counter() - t0
        rsel = torch.from_numpy(rows).cuda()
        qerr = rel(qouts[2].index_select(0, rsel), qref[2])
        if mla:
            qerr = max(qerr, rel(qouts[3].index_select(0, rsel), qref[3]))
        emit({"config": tag + " query side", "workload": name, "gpu_ms_median": qms, "gpu_ms_min": qms_min,
              "executed_tflops": qflops / (qms * 1e-3) / 1e12,
              "pct_of_bf16_peak": 100.0 * qflops / (qms * 1e-3) / 1e12 / peaks["bf16_tflops"],
              "algorithmic_gbs": qbytes / (qms * 1e-3) / 1e9,
              "pct_of_hbm_peak": 100.0 * qbytes / (qms * 1e-3) / 1e9 / peaks["hbm_gbs"],
              "flops_counted": qdesc,
              "max_err_rel_dq": qerr, "tolerance": 2e-2, "bit_stable": bool(qstable),
              "oracle_s_sample": qt_or, "oracle_sample": f"{len(pick)} of {c.num_seqs} sequences",
              "host_cores": cores, "peak_source": src})
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--batch", type=int, default=None, help="override B (profiling runs on a smaller case)")
    ap.add_argument("--heads", type=int, default=None, help="override H (profiling runs on a smaller case)")
    ap.add_argument("--seqs", type=int, default=None,
                    help="--sweep: override the number of sequences of the paged workloads (profiling runs on a "
                         "smaller case)")
    ap.add_argument("--sweep", action="store_true",
                    help="time every configuration once against its oracle sample (one JSON line each)")
    ap.add_argument("--recompute-dq", action="store_true",
                    help="time the default dQ path (S and dP recomputed) instead of ATTN_OPT_STORE_DS")
    ap.add_argument("--only", default=None, help="--sweep: only the configurations whose tag matches this regex")
    args = ap.parse_args()
    if args.sweep:
        return sweep(args)
    args.warmup = max(args.warmup, 3)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)

    import numpy as np
    import torch
    from attention_backward_recompute_gb300 import binding as bd
    from attention_backward_recompute_gb300 import build, inputs

    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build.build()
    bd.lib()

    over = {k: v for k, v in (("batch", args.batch), ("heads", args.heads)) if v is not None}
    case = inputs.dense_config(WORKLOAD, **over)
    B, H, S, D = case.batch, case.heads, case.seq_q, case.head_dim
    vp = visible_pairs(case.seq_q, case.seq_k, case.causal, case.window)
    flops = 10.0 * D * vp * B * H
    # dQ from the dS tiles the dK/dV kernel stores (ATTN_OPT_STORE_DS, one
    # product: 2*D per pair) unless --recompute-dq (S, dP and dS K: 6*D)
    store_ds = not args.recompute_dq
    alg = {"prologue": 4.0 * D * vp * B * H, "dkdv": 8.0 * D * vp * B * H,
           "dq": (2.0 if store_ds else 6.0) * D * vp * B * H}

    host = {"q": case.q, "k": case.k, "v": case.v, "dy": case.dy, "bias": case.bias}
    pinned = {n: torch.from_numpy(x).to(torch.bfloat16).pin_memory() for n, x in host.items()}
    km_host = torch.from_numpy(case.key_mask).pin_memory()
    dvc = {n: t.to(dev) for n, t in pinned.items()}
    km = km_host.to(dev)
    dq, dk, dv = (torch.empty_like(dvc[n]) for n in ("q", "k", "v"))
    desc = bd.make_dense_desc(batch=B, heads=H, seq_q=S, seq_k=S, head_dim=D, causal=True, key_mask=True,
                              bias=True, store_ds=store_ds)
    ws_bytes = bd.attn_bwd_dense_workspace_bytes(desc)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    sh = bd.ctypes.c_void_p(stream.cuda_stream)
    P = bd._ptr

    def call(qq, kk, vv, dyy, kmm, bb, oq, ok_, ov):
        st = bd.attn_bwd_dense(desc, P(qq), P(kk), P(vv), P(dyy), P(kmm), P(bb), None, None, P(oq), P(ok_), P(ov),
                               7, P(ws), ws_bytes, sh)
        if st != bd.ATTN_OK:
            raise bd.AttnError(st, bd.last_error())

    def step():
        call(dvc["q"], dvc["k"], dvc["v"], dvc["dy"], km, dvc["bias"], dq, dk, dv)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    bd.check_device_error()

    # per-kernel events for every timed step
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    for row in evs:  # CUDA events are created on first record; create them before the timed region
        for e in row:
            e.record(stream)
    torch.cuda.synchronize(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    sampler.start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    start.record(stream)
    for i in range(args.steps):
        bd.attn_set_timing_events([e.cuda_event for e in evs[i]])
        step()
    end.record(stream)
    torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()
    clocks = sampler.stop()
    bd.check_device_error()
    ms = start.elapsed_time(end) / args.steps
    ms = rank_max(ms, dist, dev)
    kt = {"prologue": [], "dkdv": [], "dq": []}
    for e in evs:
        kt["prologue"].append(e[0].elapsed_time(e[1]))
        kt["dkdv"].append(e[1].elapsed_time(e[2]))
        kt["dq"].append(e[2].elapsed_time(e[3]))
    kmean = {k: sum(v) / len(v) for k, v in kt.items()}
    dom = max(kmean, key=kmean.get)
    peaks, peak_src = load_peaks()
    peak = float(peaks["bf16_tflops"])
    achieved = alg[dom] / (kmean[dom] * 1e-3) / 1e12
    value = world * flops / (ms * 1e-3) / 1e12

    # end to end through the C ABI with host buffers: H2D of every input and
    # D2H of every gradient inside the timed region, pipelined over two device
    # buffer sets: the inputs of step i+1 go up on one copy stream and the
    # gradients of step i-1 come down on another while step i's kernels run
    # (each copy waits only for the kernels that use its buffers)
    h2d = sum(t.numel() * t.element_size() for t in pinned.values()) + km_host.numel() * 4
    sets = [(dvc, km, (dq, dk, dv)),
            ({n: torch.empty_like(t) for n, t in dvc.items()}, torch.empty_like(km),
             tuple(torch.empty_like(t) for t in (dq, dk, dv)))]
    outs_host = [[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (dq, dk, dv)] for _ in sets]
    d2h = sum(t.numel() * t.element_size() for t in outs_host[0])
    e2e_steps = max(3, args.e2e_steps)
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = {k: [torch.cuda.Event() for _ in sets] for k in ("in_ready", "in_free", "out_ready", "out_free")}

    def e2e_run(nsteps, t_start=None):
        if t_start is not None:
            up.wait_event(t_start)
        for i in range(nsteps):
            b = i % 2
            ins, kmb, outs = sets[b]
            with torch.cuda.stream(up):
                up.wait_event(ev["in_free"][b])
                for n in pinned:
                    ins[n].copy_(pinned[n], non_blocking=True)
                kmb.copy_(km_host, non_blocking=True)
                ev["in_ready"][b].record(up)
            stream.wait_event(ev["in_ready"][b])
            stream.wait_event(ev["out_free"][b])
            call(ins["q"], ins["k"], ins["v"], ins["dy"], kmb, ins["bias"], *outs)
            ev["in_free"][b].record(stream)
            ev["out_ready"][b].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(ev["out_ready"][b])
                for h_, d_ in zip(outs_host[b], outs):
                    h_.copy_(d_, non_blocking=True)
                ev["out_free"][b].record(down)
        stream.wait_stream(down)

    e2e_run(2)
    torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    e2e_run(e2e_steps, t0)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = t0.elapsed_time(t1) / e2e_steps
    e2e_ms = rank_max(e2e_ms, dist, dev)
    bd.check_device_error()

    if rank == 0:
        cpu = cpu_baseline(case, args.cpu_budget) if world == 1 and args.cpu_budget > 0 else None
        traffic = recorded_traffic(dom, B * H)
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD if not over else f"{WORKLOAD} with {over}", "description": WORKLOAD_DESC,
                       "counted_flops_per_step": flops,
                       "visible_pairs_per_head": vp, "l2": "inputs larger than L2 (640 MiB read per step), no flush",
                       "parallelism": f"replicas x{world} (weak)" if world > 1 else "1 GPU",
                       "pct_of_peak": 100.0 * value / world / peak,
                       "dq_path": "stored dS (ATTN_OPT_STORE_DS)" if store_ds else "recomputed S, dP",
                       "kernel_ms": kmean},
            "roofline": {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak,
                         "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic,
                         "peak_source": f"{peak_src} bf16 (burst)",
                         "algorithmic": f"{int(alg[dom] / (D * vp * B * H))}*D flops per visible pair"},
            "cpu_baseline": cpu,
            "clocks": clocks,
            "e2e": {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                    "copies": "two buffer sets: step i+1's host->device and step i-1's device->host copies "
                              "run on their own streams beside step i's kernels"},
            "gpu_launches": 3 * args.steps,
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
