#!/usr/bin/env python
"""Benchmark of the chunked gated delta rule on one or more GB300 GPUs.

One step = one full pass of the hot path over one synthetic batch: gdn_chunk_fwd for the
forward workloads, gdn_chunk_fwd + gdn_chunk_bwd for the training-step workload.  Prints ONE
JSON line on rank 0; for the default forward workload (1 x 32768 tokens, 2 / 8 heads) the
line also carries the training step at 1 x 32768 tokens, 16 / 16 heads ("fwdbwd"), the
metric's other half.  "roofline" is the whole step's: the method's compulsory bytes (each
input read once, each output written once) over the step time, with each kernel's share.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Multi-GPU (torchrun, one rank per GPU): every rank runs its own copy of the workload (the
(sequence, head) problems are independent, so there is no data-path collective; scaling is
weak); value = tokens of all ranks / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import gc
import json
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from chunked_prefill_gb300 import roofline as rl  # noqa: E402
from chunked_prefill_gb300.inputs import WORKLOADS, workload_inputs  # noqa: E402

METRIC = "GDN chunked fwd & fwd+bwd ms at T=32768 (tokens/s), % of roofline"
DEFAULT_WORKLOAD = "fwd_t32k_hqk2_hv8"
# FlashQLA's published H200 forward latency for 1 x 32768 tokens, h_qk = 2, h_v = 8
# (agentlenshq page, benchmark table, TP8 row): context only, another machine.
PUBLISHED_MS = {"fwd_t32k_hqk2_hv8": 0.310, "fwd_t32k_hqk8_hv24": 0.659}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def lengths_of(inp):
    if inp.cu_seqlens is None:
        return [inp.meta["T"]] * inp.meta["B"]
    cu = inp.cu_seqlens.tolist()
    return [b - a for a, b in zip(cu[:-1], cu[1:])]


def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, dev):
        self.dev = dev
        self.proc = None

    def __enter__(self):
        if self.dev is None:
            return self
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.rows = []
        if self.proc is None:
            return
        time.sleep(0.25)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) == 7:
                self.rows.append(f)

    def summary(self):
        rows = getattr(self, "rows", [])
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[3 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def make_step(inp, dev, backward, save_states=False, d=None, stream=None, fwd_kw=None):
    """One step on device inputs (copied from inp, or the given dict d), with its own outputs
    and workspace; every library call is enqueued on ``stream`` (None = current stream).
    fwd_kw: extra problem fields of the forward (context-parallel mode, warm-up chunks)."""
    fwd_kw = dict(fwd_kw or {})
    from chunked_prefill_gb300 import gdn
    if d is None:
        d = {n: (None if getattr(inp, n) is None else getattr(inp, n).to(dev).contiguous())
             for n in ("q", "k", "v", "g", "beta", "h0", "dO", "dht")}
    else:
        d = {n: d.get(n) for n in ("q", "k", "v", "g", "beta", "h0", "dO", "dht")}
    cu = None if inp.cu_seqlens is None else inp.cu_seqlens.to(dev)
    cu_host = inp.cu_seqlens
    o = torch.empty_like(d["v"])
    prob = gdn.Problem(d["q"], d["v"], inp.scale, cu, cu_host, **fwd_kw)
    ht = torch.empty(prob.num_seqs, d["v"].shape[2], 128, 128, device=dev)
    ws_f = torch.empty(max(gdn.gdn_chunk_fwd_workspace_size(prob), 16), dtype=torch.uint8, device=dev)
    bufs = None
    ws_b = None
    if backward:
        ws_b = torch.empty(max(gdn.gdn_chunk_bwd_workspace_size(prob), 16), dtype=torch.uint8,
                           device=dev)
        bufs = (torch.empty_like(d["q"]), torch.empty_like(d["k"]), torch.empty_like(d["v"]),
                torch.empty_like(d["g"]), torch.empty_like(d["beta"]),
                torch.empty_like(ht))

    if backward and save_states:
        # the forward keeps the state entering every chunk and the chunk records in ws_b; the
        # backward reads them back instead of recomputing the forward
        C, nchunks = gdn.gdn_chunk_layout(prob)
        hbuf = torch.empty(nchunks, d["v"].shape[2], 128, 128, dtype=d["v"].dtype, device=dev)

        def step():
            gdn.gdn_chunk_fwd_saved(d["q"], d["k"], d["v"], d["g"], d["beta"], inp.scale,
                                    h0=d["h0"], cu_seqlens=cu, cu_seqlens_host=cu_host,
                                    want_g_cum=False, want_A=False, workspace=ws_b, o=o, ht=ht,
                                    h=hbuf, stream=stream)
            gdn.gdn_chunk_bwd_saved(d["q"], d["k"], d["v"], d["g"], d["beta"], inp.scale, hbuf,
                                    ws_b, d["dO"], dht=d["dht"], cu_seqlens=cu,
                                    cu_seqlens_host=cu_host, out=bufs, stream=stream)
        return step, d, o, ht, cu, cu_host, ws_f, ws_b, bufs

    def step():
        gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], inp.scale, h0=d["h0"],
                          cu_seqlens=cu, cu_seqlens_host=cu_host, o=o, ht=ht, workspace=ws_f,
                          stream=stream, **fwd_kw)
        if backward:
            gdn.gdn_chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], inp.scale, d["dO"],
                              h0=d["h0"], dht=d["dht"], cu_seqlens=cu, cu_seqlens_host=cu_host,
                              workspace=ws_b, out=bufs, stream=stream)
    return step, d, o, ht, cu, cu_host, ws_f, ws_b, bufs


def time_steps(step, K, flush):
    evs = []
    for _ in range(K):
        flush.zero_()  # overwrite a buffer larger than L2 between timed steps
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        step()
        b.record()
        evs.append((a, b))
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in evs)


def e2e_run(inp, dev, K, W, backward, save_states=False):
    """The same step through the public API with HOST buffers: every step copies its inputs
    from pinned host memory, runs the call and copies its results back to pinned host memory,
    all inside the timed region.  Steps are pipelined the way a host-fed loop would run them:
    host-to-device copies on one stream, the calls on a second, device-to-host copies on a
    third, two device buffer sets alternating between steps, with events ordering each
    buffer's reuse; the clock runs from the first copy in to the last copy out."""
    names = ["q", "k", "v", "g", "beta", "h0"] + (["dO", "dht"] if backward else [])
    host = {n: getattr(inp, n).pin_memory() for n in names if getattr(inp, n) is not None}
    NB = 2
    s_in, s_run, s_out = (torch.cuda.Stream(device=dev) for _ in range(3))
    sets = []
    for _ in range(NB):
        devb = {n: torch.empty_like(t, device=dev) for n, t in host.items()}
        step, d, o, ht, cu, cu_host, ws_f, ws_b, bufs = make_step(inp, dev, backward, save_states,
                                                                  d=devb, stream=s_run)
        outs = [o, ht] if not backward else [o, ht] + [x for x in bufs if x is not None]
        host_out = [torch.empty_like(t, device="cpu").pin_memory() for t in outs]
        ev = {k: torch.cuda.Event() for k in ("in", "run", "out")}
        sets.append((devb, step, outs, host_out, ev))
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in sets[0][3])

    def run(i):
        devb, step, outs, host_out, ev = sets[i % NB]
        if i >= NB:
            s_in.wait_event(ev["run"])     # the call of step i - NB has read these inputs
            s_run.wait_event(ev["out"])    # and its results have left
        with torch.cuda.stream(s_in):
            for n, t in host.items():
                devb[n].copy_(t, non_blocking=True)
        ev["in"].record(s_in)
        s_run.wait_event(ev["in"])
        step()
        ev["run"].record(s_run)
        s_out.wait_event(ev["run"])
        with torch.cuda.stream(s_out):
            for src, dst in zip(outs, host_out):
                dst.copy_(src, non_blocking=True)
        ev["out"].record(s_out)

    for i in range(W):
        run(i)
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    for i in range(K):
        run(i)
    s_out.wait_event(sets[(K - 1) % NB][4]["out"])
    b.record(s_out)
    torch.cuda.synchronize(dev)
    return a.elapsed_time(b) / K, h2d, d2h


def oracle_sample(inp, budget_s, backward, max_steps=1):
    """Time the fp64 oracle on the first n tokens of every sequence, n sized so that one
    call takes about budget_s seconds.  Returns (tokens/s, tokens, seconds, threads)."""
    from oracle import oracle as orc
    lens = lengths_of(inp)
    cu = [0]
    for L in lens:
        cu.append(cu[-1] + L)

    def sub(n):
        idx = []
        new_cu = [0]
        for a, L in zip(cu[:-1], lens):
            m = min(n, L)
            idx.extend(range(a, a + m))
            new_cu.append(new_cu[-1] + m)
        it = torch.tensor(idx, dtype=torch.long)
        f = lambda t: None if t is None else t.reshape((-1,) + tuple(t.shape[2:]))[it].unsqueeze(0)
        return [f(inp.q), f(inp.k), f(inp.v), f(inp.g), f(inp.beta), f(inp.dO)], new_cu

    def run(n):
        (q, k, v, g, b, dO), c = sub(n)
        t0 = time.perf_counter()
        orc.fwd(q, k, v, g, b, inp.scale, h0=inp.h0, cu_seqlens=c)
        if backward:
            orc.bwd(q, k, v, g, b, inp.scale, dO, h0=inp.h0, dht=inp.dht, cu_seqlens=c)
        return time.perf_counter() - t0, c[-1]

    dt, toks = run(64)
    n = 64
    while dt < budget_s / 4 and n < max(lens):
        n = min(max(lens), n * 4)
        dt, toks = run(n)
    if dt < budget_s and n < max(lens):
        n = min(max(lens), int(n * budget_s / max(dt, 1e-3)))
        dt, toks = run(n)
    return toks / dt, toks, dt, orc.max_threads(), n


def reference_arm(args, world, rank):
    """The oracle as it stands, on the host cores: W untimed + K timed steps, each one call
    on a fixed bounded sample of the workload (rank 0 only)."""
    if rank != 0:
        return
    inp = workload_inputs(args.workload)
    w = WORKLOADS[args.workload]
    per_step = max(1.0, min(8.0, 150.0 / max(1, args.steps + args.warmup)))
    _, _, _, thr, n = oracle_sample(inp, per_step, w.backward)
    lens = lengths_of(inp)
    timed = []
    for i in range(args.warmup + args.steps):
        _, tk, d, thr, _ = oracle_sample_fixed(inp, n, w.backward)
        if i >= args.warmup:
            timed.append((tk, d))
    tot_t = sum(d for _, d in timed)
    value = sum(tk for tk, _ in timed) / tot_t
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000 * tot_t / len(timed), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(args.workload),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": thr, "kind": "oracle",
                         "sample": f"first {n} tokens of each of {len(lens)} sequence(s), all "
                                   f"{w.Hv} v-heads, per step ({'fwd+bwd' if w.backward else 'fwd'})"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def oracle_sample_fixed(inp, n, backward):
    from oracle import oracle as orc
    lens = lengths_of(inp)
    cu = [0]
    for L in lens:
        cu.append(cu[-1] + L)
    idx, new_cu = [], [0]
    for a, L in zip(cu[:-1], lens):
        m = min(n, L)
        idx.extend(range(a, a + m))
        new_cu.append(new_cu[-1] + m)
    it = torch.tensor(idx, dtype=torch.long)
    f = lambda t: None if t is None else t.reshape((-1,) + tuple(t.shape[2:]))[it].unsqueeze(0)
    q, k, v, g, b, dO = (f(x) for x in (inp.q, inp.k, inp.v, inp.g, inp.beta, inp.dO))
    t0 = time.perf_counter()
    orc.fwd(q, k, v, g, b, inp.scale, h0=inp.h0, cu_seqlens=new_cu)
    if backward:
        orc.bwd(q, k, v, g, b, inp.scale, dO, h0=inp.h0, dht=inp.dht, cu_seqlens=new_cu)
    dt = time.perf_counter() - t0
    return new_cu[-1] / dt, new_cu[-1], dt, orc.max_threads(), n


# DRAM bytes (read + write) of one whole step, from an ncu capture of the step's kernels,
# keyed by workload and by the set of kernels the step launches: a key that no longer
# matches the kernels this build launches gives no figure (null), so a capture of an older
# kernel set is never reported against a newer one.
NCU_STEP_TRAFFIC = {
    # 1 x 32768 tokens, 2 / 8 heads: k_prep 111.0 MB + first output pass 298.9 MB (section
    # captures of this kernel set); the three gated launches (transitions, fix-up, correction:
    # they read a few flags here) are not captured
    ("fwd_t32k_hqk2_hv8", ("fwd_correction", "fwd_fixup", "fwd_pass1", "fwd_prep",
                           "fwd_transitions")): 409.9e6,
}


def method_bytes(tokens, lens, w):
    """Compulsory HBM bytes of the method per tensor (bf16 activations, fp32 gates and
    states): what the step must read or write once, whatever the kernels in between."""
    nseq = len(lens)
    st = nseq * w.Hv * 128 * 128 * 4
    return {"q": tokens * w.Hqk * 128 * 2, "k": tokens * w.Hqk * 128 * 2,
            "v": tokens * w.Hv * 128 * 2, "g": tokens * w.Hv * 4, "beta": tokens * w.Hv * 4,
            "h0": st if w.h0_std > 0 else 0, "o": tokens * w.Hv * 128 * 2, "ht": st,
            "dO": tokens * w.Hv * 128 * 2, "dht": st, "dq": tokens * w.Hqk * 128 * 2,
            "dk": tokens * w.Hqk * 128 * 2, "dv": tokens * w.Hv * 128 * 2,
            "dg": tokens * w.Hv * 4, "dbeta": tokens * w.Hv * 4, "dh0": st}


# the method tensors each kernel reads or writes (intermediate records and partial states
# handed between this library's own kernels are not method bytes and are not counted)
KERNEL_TENSORS = {
    "fwd_prep": ("q", "k", "g", "beta"),
    "fwd_pass1": ("q", "k", "v", "g", "beta", "h0", "o", "ht"),
    "fwd_phase_c": ("q", "k", "v", "g", "beta", "h0", "o", "ht"),
    "fwd_phase_a": ("k", "v", "g", "beta", "h0"),
    "fwd_recompute_states": ("k", "v", "g", "beta", "h0"),
    "fwd_recompute_pass1": ("k", "v", "g", "beta", "h0"),
    "bwd_phase_a": ("q", "k", "dO", "g", "beta", "dht"),
    "bwd_dh_pass1": ("q", "k", "dO", "g", "beta", "dht", "dh0"),
    "bwd_dh_scan": ("q", "k", "dO", "g", "beta", "dht", "dh0"),
    "bwd_local": ("q", "k", "v", "dO", "g", "beta", "dq", "dk", "dv", "dg", "dbeta"),
}


def kernel_bytes(name, mb):
    names = KERNEL_TENSORS.get(name)
    if not names:
        return 0.0, "no method tensors"
    return float(sum(mb[n] for n in names)), ",".join(names)


def step_tensors(backward):
    f = ("q", "k", "v", "g", "beta", "h0", "o", "ht")
    b = ("dO", "dht", "dq", "dk", "dv", "dg", "dbeta", "dh0")
    return f + b if backward else f


def config_of(name):
    w = WORKLOADS[name]
    c = {"workload": name, "B": w.B, "T": w.T, "Hqk": w.Hqk, "Hv": w.Hv, "K": w.K, "V": w.V,
         "chunk": 64, "pass": "fwd+bwd" if w.backward else "fwd",
         "h0": w.h0_std > 0, "final_state": True,
         "l2": "flushed between timed steps (256 MiB write)", "cp": "auto (exact)"}
    if w.varlen_seqs:
        c["varlen_seqs"] = w.varlen_seqs
    return c


def sweep(args, local):
    """Forward tokens/s and roofline fraction over the head / length sweep (inputs.SWEEP)."""
    from chunked_prefill_gb300 import build, gdn
    from chunked_prefill_gb300.inputs import SWEEP
    build.build()
    dev = torch.device("cuda", local)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    pk, pk_kind = peaks()
    for name, w in SWEEP.items():
        inp = workload_inputs(name)
        lens = lengths_of(inp)
        tokens = sum(lens)
        step = make_step(inp, dev, False)[0]
        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
        ms = time_steps(step, args.steps, flush) / args.steps
        gdn.gdn_timing_enable(True)
        time_steps(step, args.steps, flush)
        gdn.gdn_timing_enable(False)
        kt = gdn.gdn_timing_collect()
        fl = rl.fwd_flops(lens, w.Hqk, w.Hv)
        by = rl.fwd_bytes(tokens, len(lens), w.Hqk, w.Hv, h0=w.h0_std > 0)
        t_roof = max(fl / (pk["bf16_tflops"] * 1e12), by / (pk["hbm_gbs"] * 1e9))
        print(json.dumps({
            "sweep": True, "workload": name, "B": w.B, "T": w.T, "Hqk": w.Hqk, "Hv": w.Hv,
            "ms_per_step": ms, "tokens_per_s": tokens / (ms / 1000.0),
            "roofline_ms": t_roof * 1000.0, "frac": t_roof * 1000.0 / ms, "peak_kind": pk_kind,
            "kernels_ms_per_step": {k: v[1] / args.steps for k, v in kt.items()}}), flush=True)
        del inp, step
        torch.cuda.empty_cache()


def prologue_bench(args, local):
    """Fused prologue forward and reverse on the q/k/gate shapes of two workloads: HBM bytes
    each launch must move, CUDA-event time, fraction of the measured copy bandwidth."""
    from chunked_prefill_gb300 import build, gdn
    from chunked_prefill_gb300.inputs import make_prologue_inputs
    build.build()
    dev = torch.device("cuda", local)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    pk, pk_kind = peaks()
    names = ("q_raw", "k_raw", "a", "b", "A_log", "dt_bias")
    for wl in ("fwd_t32k_hqk2_hv8", "fwdbwd_t32k_hqk16_hv16"):
        w = WORKLOADS[wl]
        d = {n: t.to(dev) for n, t in make_prologue_inputs(w.B, w.T, w.Hqk, w.Hv,
                                                           backward=True).items()}
        tok = w.B * w.T
        qk = 2 * tok * w.Hqk * 128 * 2
        gt = tok * w.Hv * 4
        legs = {
            # read q_raw, k_raw, a, b; write q, k, g, beta
            "prologue_fwd": (lambda: gdn.gdn_prologue_fwd(*(d[n] for n in names)),
                             2 * qk + 4 * gt),
            # read q_raw, k_raw, dq, dk, a, b, dg, dbeta; write dq_raw, dk_raw, da, db;
            # the per-head sums re-read a, dg, da
            "prologue_bwd": (lambda: gdn.gdn_prologue_bwd(*(d[n] for n in names), d["dq"], d["dk"],
                                                          d["dg"], d["dbeta"]),
                             3 * qk + 8 * gt + 3 * gt),
        }
        for leg, (fn, by) in legs.items():
            for _ in range(args.warmup):
                fn()
            torch.cuda.synchronize()
            ms = time_steps(fn, args.steps, flush) / args.steps
            gdn.gdn_timing_enable(True)
            time_steps(fn, args.steps, flush)
            gdn.gdn_timing_enable(False)
            kt = gdn.gdn_timing_collect()
            kms = {k: v[1] / args.steps for k, v in kt.items()}
            main_ms = sum(kms.values())  # kernel time (event pairs around each launch)
            print(json.dumps({
                "prologue": True, "workload": wl, "leg": leg, "ms_per_call": ms,
                "kernels_ms_per_call": kms, "algorithmic_bytes": by,
                "achieved_gbs": by / (main_ms / 1000.0) / 1e9,
                "frac": by / (main_ms / 1000.0) / 1e9 / pk["hbm_gbs"], "peak_kind": pk_kind}),
                flush=True)
        del d
        torch.cuda.empty_cache()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile", action="store_true",
                    help="for ncu: warm-up and timed steps only (no clock sampling, e2e or "
                         "CPU baseline)")
    ap.add_argument("--save-states", action="store_true",
                    help="training workloads: the forward keeps the state entering every chunk "
                         "for the backward (low-level saved pair) instead of the backward "
                         "recomputing it")
    ap.add_argument("--prologue", action="store_true",
                    help="fused prologue forward / reverse: one JSON line per leg and shape "
                         "(an auxiliary report, not the benchmark line)")
    ap.add_argument("--no-fwdbwd", action="store_true",
                    help="forward workloads: skip the fwd+bwd training-step sub-record")
    ap.add_argument("--warmup-report", action="store_true",
                    help="opt-in warm-up mode vs the exact mode: step time and error against "
                         "the oracle (an auxiliary report, not the benchmark line)")
    ap.add_argument("--sweep", action="store_true",
                    help="head / length sweep of the forward: one JSON line per point "
                         "(an auxiliary report, not the benchmark line)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    world, rank, local = dist_setup(args.gpus)
    if args.sweep:
        sweep(args, local)
        return
    if args.prologue:
        prologue_bench(args, local)
        return
    if args.warmup_report:
        warmup_report(args, local)
        return

    if args.impl == "reference":
        reference_arm(args, world, rank)
        return

    from chunked_prefill_gb300 import build
    build.build()
    dev = torch.device("cuda", local)
    if args.profile:
        args.no_e2e = args.no_cpu_baseline = True
    res = measure(args.workload, args, dev, world, local, clocks=not args.profile,
                  save=args.save_states)
    w = WORKLOADS[args.workload]
    tokens = res["tokens"]
    value = world * tokens / (res["ms_per_step"] / 1000.0)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["ms_per_step"],
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": (value / (tokens / (PUBLISHED_MS[args.workload] / 1000.0))
                        if args.workload in PUBLISHED_MS and world == 1 else None),
        "vs_baseline_note": ("ratio to the FlashQLA pages' H200 forward latency for this "
                             "shape (another machine: context, not the target)"
                             if args.workload in PUBLISHED_MS else None),
        "dtype": "bf16", "data": "synthetic",
        "config": dict(config_of(args.workload),
                       **({"save_states": True} if args.save_states and w.backward else {})),
        "roofline": res["roofline"],
        "gpu_launches": res["launches"],
        "clocks": res["clocks"],
    }
    if "e2e" in res:
        line["e2e"] = res["e2e"]
    # the metric's other half: the fwd+bwd training step at T = 32768 (16 / 16 heads), as a
    # sub-record of the same line
    if not w.backward and not args.no_fwdbwd and not args.profile:
        sub = sub_measure(FWDBWD_WORKLOAD, args, dev, world, local, save=False)
        line["fwdbwd"] = {
            "workload": FWDBWD_WORKLOAD, "config": config_of(FWDBWD_WORKLOAD),
            "ms_per_step": sub["ms_per_step"],
            "value": world * sub["tokens"] / (sub["ms_per_step"] / 1000.0), "unit": "tokens/s",
            "roofline": sub["roofline"], "gpu_launches": sub["launches"], "clocks": sub["clocks"],
            "process": sub["process"],
        }
        if "e2e" in sub:
            line["fwdbwd"]["e2e"] = sub["e2e"]
        # the same training step with the low-level saved pair: the forward keeps the state
        # entering every chunk (and its chunk records) and the backward reads them instead of
        # recomputing the forward (more memory, less work)
        sv = sub_measure(FWDBWD_WORKLOAD, args, dev, world, local, save=True)
        line["fwdbwd_saved_states"] = {
            "ms_per_step": sv["ms_per_step"],
            "value": world * sv["tokens"] / (sv["ms_per_step"] / 1000.0), "unit": "tokens/s",
            "roofline_frac": sv["roofline"]["frac"], "gpu_launches": sv["launches"],
            "kernels_ms_per_step": {k: v["ms_per_step"] for k, v in sv["roofline"]["kernels"].items()},
            "clocks": sv["clocks"], "process": sv["process"]}
        if "e2e" in sv:
            line["fwdbwd_saved_states"]["e2e"] = sv["e2e"]
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        inp = workload_inputs(args.workload)
        lens = lengths_of(inp)
        tps, toks, dt, thr, n = oracle_sample(inp, 10.0, w.backward)
        reps = 1
        if n >= max(lens):  # the whole workload fits the budget: repeat it up to ~10 s
            while dt < 10.0 and reps < 50:
                _, tk, d, thr, _ = oracle_sample_fixed(inp, n, w.backward)
                toks, dt, reps = toks + tk, dt + d, reps + 1
            tps = toks / dt
        line["cpu_baseline"] = {"value": tps, "unit": "tokens/s", "cores": thr, "kind": "oracle",
                                "sample": f"first {n} tokens of each of {len(lens)} sequence(s), "
                                          f"all {w.Hv} v-heads, {reps} call(s) ({toks} tokens, "
                                          f"{dt:.1f} s)"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


FWDBWD_WORKLOAD = "fwdbwd_t32k_hqk16_hv16"


def sub_measure(name, args, dev, world, local, save):
    """A sub-record of the line, measured as if alone.  Kernels load on first use, so where a
    kernel's code lands in device memory depends on what the process ran before; the training
    step's local gradients once ran ~6 % slower after another workload in the same process (an
    instruction-fetch effect, gone since that kernel's code was compacted).  On one GPU each
    sub-record therefore still runs in a fresh child process (the same bench.py, its JSON line
    parsed back), loading and allocating as it would alone.  Several ranks measure it
    in-process, as the ranks must."""
    if world > 1:
        r = measure(name, args, dev, world, local, clocks=True, save=save)
        r["process"] = "in-process (ranks)"
        return r
    gc.collect()
    torch.cuda.empty_cache()
    cmd = [sys.executable, os.path.abspath(__file__), "--workload", name, "--steps", str(args.steps),
           "--warmup", str(args.warmup), "--no-cpu-baseline", "--no-fwdbwd"]
    if save:
        cmd.append("--save-states")
    if args.no_e2e:
        cmd.append("--no-e2e")
    env = dict(os.environ, CUDA_VISIBLE_DEVICES=os.environ.get("CUDA_VISIBLE_DEVICES", str(local)))
    out = subprocess.run(cmd, env=env, capture_output=True, text=True, check=True).stdout
    d = json.loads([l for l in out.splitlines() if l.startswith("{")][-1])
    r = {"tokens": d["value"] * d["ms_per_step"] / 1000.0, "ms_per_step": d["ms_per_step"],
         "roofline": d["roofline"], "launches": d["gpu_launches"], "clocks": d["clocks"],
         "process": "fresh child process"}
    if "e2e" in d:
        r["e2e"] = d["e2e"]
    return r


def measure(name, args, dev, world, local, clocks=True, save=False, fwd_kw=None):
    """Warm-up, then K timed steps (L2 flushed between them, CUDA events, max over ranks),
    a second instrumented pass for the per-kernel split, the step roofline and (unless
    disabled) the end-to-end leg of one workload."""
    from chunked_prefill_gb300 import gdn
    w = WORKLOADS[name]
    inp = workload_inputs(name)
    lens = lengths_of(inp)
    tokens = sum(lens)
    save = save and w.backward
    step = make_step(inp, dev, w.backward, save, fwd_kw=fwd_kw)[0]
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local if clocks else None) as clk:
        # keep the GPU busy (untimed) while nvidia-smi starts, so the sampled clocks are
        # those under load and its start-up does not overlap the timed steps
        t_busy = time.time() + (1.0 if clocks else 0.0)
        while time.time() < t_busy:
            step()
            torch.cuda.synchronize()
        ms_total = time_steps(step, args.steps, flush)
    # per-kernel split from a second, instrumented pass (the event records between kernels
    # would otherwise sit inside the headline's timed region)
    gdn.gdn_timing_enable(True)
    time_steps(step, args.steps, flush)
    gdn.gdn_timing_enable(False)
    kt = gdn.gdn_timing_collect()
    torch.cuda.synchronize()
    barrier(world)
    ms_total = max_over_ranks(ms_total, world)
    ms_per_step = ms_total / args.steps

    pk, pk_kind = peaks()
    fl = rl.fwd_flops(lens, w.Hqk, w.Hv) + (rl.bwd_flops(lens, w.Hqk, w.Hv) if w.backward else 0)
    by = rl.fwd_bytes(tokens, len(lens), w.Hqk, w.Hv, h0=w.h0_std > 0)
    if w.backward:
        by += rl.bwd_bytes(tokens, len(lens), w.Hqk, w.Hv, h0=w.h0_std > 0)
    t_tc = fl / (pk["bf16_tflops"] * 1e12)
    t_hbm = by / (pk["hbm_gbs"] * 1e9)
    mb = method_bytes(tokens, lens, w)
    kernels = {}
    for k, (n, ms) in kt.items():
        kb, names = kernel_bytes(k, mb)
        avg_s = ms / max(n, 1) / 1000.0
        kernels[k] = {"launches_per_step": n / args.steps, "ms_per_step": ms / args.steps,
                      "share": ms / max(sum(v[1] for v in kt.values()), 1e-30),
                      "method_bytes_per_launch": kb, "method_tensors": names,
                      "achieved_gbs": kb / avg_s / 1e9 if kb else None,
                      "frac": kb / avg_s / 1e9 / pk["hbm_gbs"] if kb else None}
    dom = max(kt.items(), key=lambda kv: kv[1][1])[0] if kt else None
    achieved = by / (ms_per_step / 1000.0) / 1e9
    key = (name, tuple(sorted(kt)))
    roof = {"bound": "hbm" if t_hbm >= t_tc else "tensor", "scope": "whole step",
            "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / pk["hbm_gbs"], "peak_kind": pk_kind,
            "traffic": NCU_STEP_TRAFFIC.get(key),
            "algorithmic_bytes_per_step": by,
            "bytes_counted": ("forward call: q+k+v+g+beta+h0 read, o+ht written; backward call: "
                              "q+k+v+dO+g+beta+h0+dht read, dq+dk+dv+dg+dbeta+dh0 written "
                              "(each once per call)") if w.backward else
                             "+".join(step_tensors(False)) + " (each read or written once)",
            "algorithmic_flops_per_step": fl,
            "roofline_ms": max(t_tc, t_hbm) * 1000.0,
            "dominant_kernel": dom, "kernels": kernels}
    res = {"tokens": tokens, "ms_per_step": ms_per_step, "roofline": roof,
           "launches": sum(v[0] for v in kt.values()),  # this library's kernels in K steps
           "clocks": clk.summary() if clocks else None}
    if not args.no_e2e:
        e2e_ms, h2d, d2h = e2e_run(inp, dev, args.steps, args.warmup, w.backward, save)
        e2e_ms = max_over_ranks(e2e_ms, world)
        res["e2e"] = {"value": world * tokens / (e2e_ms / 1000.0), "unit": "tokens/s",
                      "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                      "mode": "pinned host buffers; copies in, calls and copies out on three "
                              "streams, two device buffer sets alternating between steps"}
    del inp, step, flush
    torch.cuda.empty_cache()
    return res


def warmup_report(args, local):
    """The opt-in warm-up mode against the exact mode on one workload: step time, and the
    error of o and of the final state against the fp64 oracle, for warm-up windows of 6 and
    8 chunks (one JSON line per mode)."""
    import numpy as np
    from chunked_prefill_gb300 import build, gdn
    from oracle import oracle as orc
    build.build()
    dev = torch.device("cuda", local)
    inp = workload_inputs(args.workload)
    w = WORKLOADS[args.workload]
    ro, rht = orc.fwd(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.scale, h0=inp.h0,
                      cu_seqlens=None if inp.cu_seqlens is None else inp.cu_seqlens.numpy())
    args.no_e2e = True
    modes = [("exact", dict(cp_mode=gdn.CP_AUTO))]
    modes += [(f"warmup{wc}", dict(cp_mode=gdn.CP_WARMUP, warmup_chunks=wc)) for wc in (6, 8)]
    for label, kw in modes:
        res = measure(args.workload, args, dev, 1, local, clocks=False, fwd_kw=kw)
        step, d, o, ht = make_step(inp, dev, False, fwd_kw=kw)[:4]
        step()
        torch.cuda.synchronize()
        oo, hh = o.float().cpu().numpy(), ht.cpu().numpy()
        rel = lambda a, b: float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-30))
        print(json.dumps({"warmup_report": True, "workload": args.workload, "mode": label,
                          "cp": kw, "ms_per_step": res["ms_per_step"],
                          "tokens_per_s": res["tokens"] / (res["ms_per_step"] / 1000.0),
                          "o_rel_err": rel(oo, ro), "ht_rel_err": rel(hh, rht),
                          "kernels_ms_per_step": {k: v["ms_per_step"] for k, v in
                                                  res["roofline"]["kernels"].items()}}),
              flush=True)
        del step, d, o, ht
        torch.cuda.empty_cache()


if __name__ == "__main__":
    main()
