#!/usr/bin/env python
"""Benchmark of the block-diagonal causal attention hot path on GB300.

One step = the whole path on one synthetic packed batch, every call through
the C ABI's single-call entry points: bd_attn_fwd (the plan -- mask bounds
and ordered tile lists -- from cu_seqlens, the fp16 copy of v, the forward
kernel) then bd_attn_bwd (the per-row terms with the forward's plan reused,
the main kernel, the dq conversion), for every query interval.  Default
workload: 1 row x 8192 tokens, Hq=32, Hkv=8, D=128, lognormal(1024, 1.0)
document lengths (seed 0).

Metric: useful TFLOP/s = 14 * D * (unmasked query/key pairs) * Hq per step
(4*D forward + 10*D backward per pair and query head) over the step time;
tokens/s (non-padding query tokens) is reported beside it.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
For N > 1 run under torch.distributed.run: every rank runs its own replica of
the workload (weak scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import tempfile
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from packed_sequence_block_gb300.workloads import make_qkv_do, make_workload  # noqa: E402

CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,"
                "utilization.gpu")
# seconds of back-to-back step replays right before the timed steps, with the
# clock sampler running, so that it records the clocks under this load
SOAK_S = 1.5


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="lognormal8k")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of oracle work for the CPU baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=None,
                    help="steps of the end-to-end timing (default: --steps)")
    ap.add_argument("--dropout-p", type=float, default=0.1,
                    help="also time the step with attention dropout at this p (0: skip)")
    ap.add_argument("--soak", type=float, default=SOAK_S,
                    help="seconds of step replays before the timed steps, under the clock sampler")
    args = ap.parse_args()
    if args.e2e_steps is None:
        args.e2e_steps = args.steps
    return args


def useful_pairs(wl):
    total = 0
    for cu in wl.cu:
        cu = [int(x) for x in cu]
        for s0 in wl.seq_starts:
            for a, b in zip(cu[:-1], cu[1:]):
                lo, hi = max(a, s0), min(b, s0 + wl.L)
                if lo < hi:
                    n1, n2 = lo - a + 1, hi - a
                    total += (n1 + n2) * (n2 - n1 + 1) // 2
    return total


def describe(wl):
    docs = sum(len(c) - 1 for c in wl.cu)
    pad = sum(wl.S - int(c[-1]) for c in wl.cu)
    return (f"{wl.name}: {wl.B} row(s) x {wl.S} tokens, Hq={wl.Hq}, Hkv={wl.Hkv}, D={wl.D}, "
            f"{docs} docs, {pad} padding tokens, {len(wl.seq_starts)} query interval(s) of "
            f"{wl.L}, seed {wl.seed}")


def doc_boundaries(wl):
    """The workload's document boundaries per row, or their SHA-256 when there are many."""
    rows = [[int(x) for x in c] for c in wl.cu]
    if sum(len(r) for r in rows) <= 64:
        return rows
    return "sha256:" + hashlib.sha256(json.dumps(rows).encode()).hexdigest()


def profiled_traffic(workload, seed):
    """DRAM bytes per launch of the backward main kernel from the committed ncu
    figures (profiles/bd_bwd_kernel_lognormal8k.json), or None when the kernel
    sources differ from the profiled ones or the workload is not the profiled one."""
    path = os.path.join(ROOT, "profiles", "bd_bwd_kernel_lognormal8k.json")
    try:
        with open(path) as f:
            fig = json.load(f)
    except (OSError, ValueError):
        return None, "no capture"
    if workload != fig.get("workload") or seed != fig.get("seed"):
        return None, "no capture for this workload"
    traffic, shas = fig.get("traffic_bytes_per_launch"), fig.get("source_sha256") or {}
    if not isinstance(traffic, int) or not shas:
        return None, "no capture"
    csrc = os.path.join(ROOT, "packed_sequence_block_gb300", "csrc")
    for name, digest in shas.items():
        try:
            with open(os.path.join(csrc, name), "rb") as f:
                if hashlib.sha256(f.read()).hexdigest() != digest:
                    return None, f"{name} changed since the ncu capture"
        except OSError:
            return None, f"{name} changed since the ncu capture"
    return traffic, "ncu dram__bytes_read.sum + dram__bytes_write.sum, one launch"


def read_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, \
            "fallback"


class ClockSampler:
    """nvidia-smi samples every 200 ms while the timed region runs."""

    def __init__(self, path, soak=SOAK_S):
        self.path = path
        self.proc = None
        self.soak = soak

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self, gpu_index):
        """Median SM clock over the samples taken under load (GPU utilisation >= 50%),
        the maximum clock, and every throttle reason seen while under load."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm_all, sm_load, mx, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    if int(parts[0]) != gpu_index:
                        continue
                    mhz, top, util = float(parts[1]), float(parts[2]), float(parts[9])
                except ValueError:
                    continue
                sm_all.append(mhz)
                mx.append(top)
                if util >= 50.0:
                    sm_load.append(mhz)
                    for n, val in zip(names, parts[5:9]):
                        if val.lower() == "active":
                            reasons.add(n)
        return {"sm_mhz": statistics.median(sm_load) if sm_load else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm_all), "samples_under_load": len(sm_load),
                "window": f"{self.soak} s of back-to-back step replays, then the timed steps"}


class HotPath:
    """Device buffers and the per-step call sequence through the C ABI."""

    def __init__(self, wl, device):
        from packed_sequence_block_gb300 import _native as N
        from packed_sequence_block_gb300.attention import device_status_word
        self.N, self.wl, self.dev = N, wl, device
        B, S, L, Hq, Hkv, D = wl.B, wl.S, wl.L, wl.Hq, wl.Hkv, wl.D
        flat, rp = wl.cu_csr()
        self.cu_h = torch.from_numpy(flat).pin_memory()
        self.rp_h = torch.from_numpy(rp).pin_memory()
        self.cu = self.cu_h.to(device)
        self.rp = self.rp_h.to(device)
        q, k, v, do = make_qkv_do(wl, device=device, generator_device=device)
        self.k, self.v = k, v
        self.q_iv = [q[:, :, s:s + L].contiguous() for s in wl.seq_starts]
        self.do_iv = [do[:, :, s:s + L].contiguous() for s in wl.seq_starts]
        del q, do
        self.out = [torch.empty_like(x) for x in self.q_iv]
        self.lse = [torch.empty((B, Hq, L), dtype=torch.float32, device=device)
                    for _ in wl.seq_starts]
        self.dq = [torch.empty_like(x) for x in self.q_iv]
        self.dk = torch.empty_like(k)
        self.dv = torch.empty_like(v)
        # one workspace serves every interval: each interval's forward and
        # backward run back to back on the stream
        self.ws = torch.empty(N.bd_attn_workspace_size(B, Hq, Hkv, L, S, D), dtype=torch.uint8,
                              device=device)
        self.status = device_status_word(device)
        self.scale = D ** -0.5
        self.gqa = Hq != Hkv
        self.main_events = []
        self.drop = None  # (p, seed, offset) to run the dropout entry points

    def launches_per_step(self):
        # per interval: plan + fp16 v, forward, plan + row terms, backward main, dq conversion
        return len(self.wl.seq_starts) * 5

    def _io(self):
        """This object's own per-step inputs and outputs."""
        return {"cu": self.cu, "rp": self.rp, "k": self.k, "v": self.v, "q": self.q_iv,
                "do": self.do_iv, "out": self.out, "lse": self.lse, "dq": self.dq,
                "dk": self.dk, "dv": self.dv}

    def step(self, time_main=False, io=None):
        """One pass of the hot path: every query interval's forward and backward
        through the single-call entry points (boundaries in, gradients out)."""
        N, wl = self.N, self.wl
        io = io if io is not None else self._io()
        B, S, L, Hq, Hkv, D = wl.B, wl.S, wl.L, wl.Hq, wl.Hkv, wl.D
        cu, rp, st = io["cu"], io["rp"], self.status
        for i, s0 in enumerate(wl.seq_starts):
            if self.drop is not None:
                p, seed, off = self.drop
                N.bd_attn_fwd_dropout(io["q"][i], io["k"], io["v"], B, Hq, Hkv, L, S, D, cu, rp,
                                      s0, self.scale, self.gqa, io["out"][i], io["lse"][i],
                                      self.ws, p, seed, off, st)
                N.bd_attn_bwd_dropout(io["q"][i], io["k"], io["v"], io["out"][i], io["lse"][i],
                                      io["do"][i], B, Hq, Hkv, L, S, D, cu, rp, s0, self.scale,
                                      self.gqa, io["dq"][i], io["dk"], io["dv"], self.ws, p,
                                      seed, off, st)
                continue
            N.bd_attn_fwd(io["q"][i], io["k"], io["v"], B, Hq, Hkv, L, S, D, cu, rp, s0,
                          self.scale, self.gqa, io["out"][i], io["lse"][i], self.ws, st)
            args = (io["q"][i], io["k"], io["v"], io["out"][i], io["lse"][i], io["do"][i], B, Hq,
                    Hkv, L, S, D, cu, rp, s0, self.scale, self.gqa, io["dq"][i], io["dk"],
                    io["dv"], self.ws)
            if not time_main:
                N.bd_attn_bwd(*args, dev_status=st)
                continue
            N.bd_attn_bwd_stages(*args, dev_status=st, stages=1)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            N.bd_attn_bwd_stages(*args, dev_status=st, stages=2)
            e1.record()
            self.main_events.append((e0, e1))
            N.bd_attn_bwd_stages(*args, dev_status=st, stages=4)

    def e2e_setup(self):
        """Pinned host copies of the inputs, and two device/host buffer sets, so that a
        step's copies in and out overlap the neighbouring steps' compute."""
        pin = lambda t: torch.empty(t.shape, dtype=t.dtype, pin_memory=True)  # noqa: E731
        own = self._io()
        in_keys, out_keys = ("cu", "rp", "k", "v", "q", "do"), ("out", "lse", "dq", "dk", "dv")

        def flat(io, keys):
            ts = []
            for key in keys:
                ts.extend(io[key] if isinstance(io[key], list) else [io[key]])
            return ts

        self.h_in = []
        for t in flat(own, in_keys):
            h = pin(t)
            h.copy_(t)
            self.h_in.append(h)
        clone = {k: ([torch.empty_like(x) for x in t] if isinstance(t, list)
                     else torch.empty_like(t)) for k, t in own.items()}
        self.sets = []
        for io in (own, clone):
            self.sets.append({"io": io, "d_in": flat(io, in_keys), "d_out": flat(io, out_keys),
                              "h_out": [pin(t) for t in flat(io, out_keys)],
                              "ev": {n: torch.cuda.Event() for n in ("in", "done", "out")}})
        self.s_in, self.s_out = torch.cuda.Stream(), torch.cuda.Stream()
        h2d = sum(h.numel() * h.element_size() for h in self.h_in)
        d2h = sum(t.numel() * t.element_size() for t in self.sets[0]["d_out"])
        return h2d, d2h

    def e2e_run(self, n_steps):
        """n_steps steps through the library with each step's inputs copied in from
        pinned host memory and its results copied out; returns elapsed ms."""
        cur = torch.cuda.current_stream()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(cur)
        self.s_in.wait_event(t0)
        self.s_out.wait_event(t0)
        for i in range(n_steps):
            st = self.sets[i % 2]
            ev = st["ev"]
            if i >= 2:
                self.s_in.wait_event(ev["done"])  # step i-2 no longer reads this set
            with torch.cuda.stream(self.s_in):
                for h, d in zip(self.h_in, st["d_in"]):
                    d.copy_(h, non_blocking=True)
                ev["in"].record(self.s_in)
            cur.wait_event(ev["in"])
            if i >= 2:
                cur.wait_event(ev["out"])  # step i-2's results have left this set
            self.step(io=st["io"])
            ev["done"].record(cur)
            self.s_out.wait_event(ev["done"])
            with torch.cuda.stream(self.s_out):
                for h, d in zip(st["h_out"], st["d_out"]):
                    h.copy_(d, non_blocking=True)
                ev["out"].record(self.s_out)
        for st in self.sets[:min(2, n_steps)]:
            cur.wait_event(st["ev"]["out"])
        t1.record(cur)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1)


def time_layout_kernels(device, hbm_gbs, reps=20):
    """Device times of the row-layout kernels at the 8192- and 131072-token rows.

    Bytes are the algorithmic ones (each input read once, each output written
    once); at these sizes the kernels are bound by launch latency, not HBM.
    """
    from packed_sequence_block_gb300 import _native as N
    from packed_sequence_block_gb300.attention import device_status_word, segment_cu_seqlens
    out = {}
    for name in ("lognormal8k", "interval131k"):
        wl = make_workload(name)
        B, S, L = wl.B, wl.S, wl.L
        lens_rows = [np.diff(np.asarray(c, np.int64)) for c in wl.cu]
        nd = max(len(x) for x in lens_rows)
        lens = np.full((B, nd), -1000, np.int32)
        for b, x in enumerate(lens_rows):
            lens[b, :len(x)] = x
        lens_d = torch.from_numpy(lens).to(device)
        ids = torch.empty((B, S), dtype=torch.int32, device=device)
        pos = torch.empty((B, S), dtype=torch.int32, device=device)
        keep = torch.empty((B, S), dtype=torch.bool, device=device)
        bad = torch.empty((B,), dtype=torch.int32, device=device)
        st = device_status_word(device)
        N.bd_doc_ids_from_seq_lens(lens_d, B, nd, S, -1000, ids, st)
        seg, sid, nseg = segment_cu_seqlens(ids)
        rng_ = torch.empty((B, 2), dtype=torch.int32, device=device)
        rows = torch.empty((B, -(-S // L)), dtype=torch.int32, device=device)
        calls = {
            "doc_ids_from_seq_lens": (lambda: N.bd_doc_ids_from_seq_lens(
                lens_d, B, nd, S, -1000, ids, st), 4 * B * nd + 4 * B * S),
            "position_ids_from_doc_ids": (lambda: N.bd_position_ids_from_doc_ids(
                ids, B, S, pos, keep), 4 * B * S + 5 * B * S),
            "validate_document_positions": (lambda: N.bd_validate_document_positions(
                keep, pos, B, S, bad, st), 5 * B * S + 4 * B),
            "kv_needed_range": (lambda: N.bd_kv_needed_range(
                seg, sid, nseg, B, S, L, wl.seq_starts[-1], rng_, rows),
                8 * B * nd + 8 * B + 4 * B * rows.shape[1]),
        }
        res = {}
        for key, (fn, nbytes) in calls.items():
            # ten back-to-back calls captured as one graph, so that host-side
            # launch time stays out of the device time measured
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for _ in range(10):
                    fn()
            g.replay()
            ts = []
            for _ in range(reps):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record()
                g.replay()
                e1.record()
                ts.append((e0, e1))
            torch.cuda.synchronize()
            us = statistics.median(a.elapsed_time(b) for a, b in ts) * 1e3 / 10
            gbs = nbytes / (us * 1e-6) / 1e9
            res[key] = {"us": round(us, 2), "bytes": nbytes, "GB/s": round(gbs, 1),
                        "frac_of_hbm": round(gbs / hbm_gbs, 4)}
        out[f"{name}: B={B}, S={S}"] = res
    return out


def flush_l2(buf):
    buf.add_(1)


def oracle_inputs(wl, seed):
    from oracle import blockdiag as orc
    q, k, v, do = make_qkv_do(wl, seed=seed, device="cpu")
    ids = np.stack([orc.doc_ids_from_cu_seqlens(c, wl.S) for c in wl.cu])
    return q, k, v, do, ids


def cpu_oracle_sample(wl, budget_s, inputs):
    """Time the fp64 oracle (fwd + bwd) on whole kv-head groups until the budget is used."""
    from oracle import blockdiag as orc
    q, k, v, do, ids = inputs
    G = wl.G
    s0 = wl.seq_starts[0]
    pairs_all = useful_pairs_interval(wl, s0)
    done_heads, elapsed = 0, 0.0
    t_start = time.perf_counter()
    for g in range(wl.Hkv):
        hs = slice(g * G, (g + 1) * G)
        qi = q[:, hs, s0:s0 + wl.L]
        di = do[:, hs, s0:s0 + wl.L]
        kg, vg = k[:, g:g + 1], v[:, g:g + 1]
        o, l = orc.blockdiag_sdpa_forward(qi, kg, vg, ids, s0, None, G > 1)
        orc.blockdiag_sdpa_backward(qi, kg, vg, di, ids, s0, None, G > 1, out=o, lse=l)
        done_heads += G
        elapsed = time.perf_counter() - t_start
        if elapsed >= budget_s:
            break
    flops = 14.0 * wl.D * pairs_all * done_heads
    return {
        "value": flops / elapsed / 1e12, "unit": "TFLOP/s", "kind": "oracle",
        "cores": len(os.sched_getaffinity(0)),
        "sample": (f"{done_heads} of {wl.Hq} query heads ({done_heads // G} kv-head groups), "
                   f"query interval at {s0}, forward+backward in numpy fp64, "
                   f"{elapsed:.1f} s"),
        "seconds": elapsed,
    }


def useful_pairs_interval(wl, s0):
    total = 0
    for cu in wl.cu:
        cu = [int(x) for x in cu]
        for a, b in zip(cu[:-1], cu[1:]):
            lo, hi = max(a, s0), min(b, s0 + wl.L)
            if lo < hi:
                n1, n2 = lo - a + 1, hi - a
                total += (n1 + n2) * (n2 - n1 + 1) // 2
    return total


def max_over_ranks(values, world, device):
    """Each value's maximum over the ranks (the slowest rank's time); one
    collective on the timing numbers only, never on the data path."""
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def job_rate(units_per_rank_step, steps, slowest_ms, world):
    """Whole-job throughput: every rank's units over the slowest rank's time."""
    return world * units_per_rank_step * steps / (slowest_ms * 1e-3)


def run_reference(args, wl, rank, world):
    if rank != 0:
        return
    pairs = useful_pairs(wl)
    inputs = oracle_inputs(wl, args.seed)
    for _ in range(args.warmup):
        cpu_oracle_sample(wl, 0.0, inputs)
    vals, secs = [], []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        r = cpu_oracle_sample(wl, 0.0, inputs)
        vals.append(r["value"])
        secs.append(r["seconds"])
    total = time.perf_counter() - t0
    value = statistics.mean(vals)
    line = {
        "impl": "reference", "metric": "useful TFLOP/s, block-causal varlen attention fwd+bwd",
        "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": describe(wl), "useful_pairs": pairs},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "kind": "oracle",
                         "cores": len(os.sched_getaffinity(0)),
                         "sample": f"one kv-head group ({wl.G} of {wl.Hq} query heads) per "
                                   f"step, forward+backward in numpy fp64"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    wl = make_workload(args.workload, args.seed)
    if args.impl == "reference":
        run_reference(args, wl, rank, world)
        return

    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    from packed_sequence_block_gb300.attention import check_device_status

    hp = HotPath(wl, device)
    pairs = useful_pairs(wl)
    D, Hq = wl.D, wl.Hq
    flops_step = 14.0 * D * pairs * Hq
    flops_bwd_main_step = 10.0 * D * pairs * Hq  # all intervals of one step
    tokens_step = wl.non_pad_tokens()
    l2_buf = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=device)

    for _ in range(max(3, args.warmup)):
        hp.step()
    torch.cuda.synchronize()
    check_device_status(device)

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    # One step is a fixed sequence of stream-ordered library calls; it is
    # captured once as a CUDA graph and replayed, so the timed steps carry no
    # host-side launch gaps.
    step_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(step_graph):
        hp.step()
    step_graph.replay()
    torch.cuda.synchronize()
    check_device_status(device)

    peaks, peak_src = read_peaks()
    # the raw samples go to BD_CLOCKS_DIR when it is set (the JSON line carries the summary)
    clocks_dir = os.environ.get("BD_CLOCKS_DIR")
    sampler = ClockSampler(os.path.join(clocks_dir, f"clocks_rank{rank}.csv") if clocks_dir
                           else os.path.join(tempfile.gettempdir(),
                                             f"bd_clocks_{os.getpid()}_{rank}.csv"),
                           args.soak)
    step_ms = []
    barrier()
    with sampler:
        t_end = time.perf_counter() + args.soak
        while time.perf_counter() < t_end:
            for _ in range(50):
                step_graph.replay()
            torch.cuda.synchronize()
        for _ in range(args.steps):
            flush_l2(l2_buf)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            step_graph.replay()
            e1.record()
            step_ms.append((e0, e1))
        barrier()
    check_device_status(device)
    times = [a.elapsed_time(b) for a, b in step_ms]
    total_ms = sum(times)

    # the backward main kernel alone, for the roofline: the same calls issued
    # directly, with events on the launching stream around that launch
    for _ in range(args.steps):
        flush_l2(l2_buf)
        hp.step(time_main=True)
    barrier()
    check_device_status(device)
    main_ms = [a.elapsed_time(b) for a, b in hp.main_events]

    # end to end through the public API with host buffers: every step copies its
    # inputs in from pinned host memory and its results out inside the timed
    # region, on two copy streams, double-buffered so that they overlap the
    # neighbouring steps' compute
    h2d, d2h = hp.e2e_setup()
    hp.e2e_run(2)
    barrier()
    e2e_total = hp.e2e_run(args.e2e_steps)
    barrier()
    check_device_status(device)

    # the same step with attention dropout (counter-based mask regenerated in
    # the backward), graph-replayed like the timed steps above
    drop_ms = 0.0
    if args.dropout_p > 0.0:
        hp.drop = (args.dropout_p, 0x9E3779B97F4A7C15, 0)
        for _ in range(3):
            hp.step()
        drop_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(drop_graph):
            hp.step()
        drop_graph.replay()
        barrier()
        check_device_status(device)
        ev = []
        for _ in range(args.steps):
            flush_l2(l2_buf)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            drop_graph.replay()
            e1.record()
            ev.append((e0, e1))
        barrier()
        check_device_status(device)
        drop_ms = sum(a.elapsed_time(b) for a, b in ev)
        hp.drop = None

    total_ms, e2e_total, drop_ms = max_over_ranks([total_ms, e2e_total, drop_ms], world, device)
    value = job_rate(flops_step, args.steps, total_ms, world) / 1e12
    e2e_value = job_rate(flops_step, args.e2e_steps, e2e_total, world) / 1e12
    tok_s = job_rate(tokens_step, args.steps, total_ms, world)

    main_avg = statistics.mean(main_ms)
    achieved = flops_bwd_main_step * args.steps / (sum(main_ms) * 1e-3) / 1e12
    peak = float(peaks["bf16_tflops"])
    clocks = sampler.summary(local)
    traffic, traffic_src = profiled_traffic(args.workload, args.seed)
    layout_times = time_layout_kernels(device, float(peaks["hbm_gbs"])) if rank == 0 else None

    if rank == 0:
        line = {
            "metric": "useful TFLOP/s, block-causal varlen attention fwd+bwd",
            "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": describe(wl), "B": wl.B, "S": wl.S, "L": wl.L, "Hq": Hq,
                       "Hkv": wl.Hkv, "D": D, "useful_pairs": pairs,
                       "cu_seqlens": doc_boundaries(wl),
                       "useful_tflop_per_step": flops_step / 1e12,
                       "strict_12D_tflops": value * 12.0 / 14.0,
                       "l2": "flushed between timed steps (256 MiB write, outside the events)",
                       "timing": "CUDA graph replay of one step's library calls, CUDA events",
                       "parallelism": f"{world} independent replica(s)"},
            "tokens_per_s": tok_s,
            "frac_of_bf16_peak": value / peak,
            "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": args.e2e_steps,
                    "ms_per_step": e2e_total / args.e2e_steps,
                    "schedule": "each step's inputs copied in from pinned host memory and its "
                                "results copied out inside the timed region, on two copy "
                                "streams, double-buffered to overlap the neighbouring steps' "
                                "compute"},
            "gpu_launches": hp.launches_per_step() * args.steps,
            "roofline": {"kernel": "bd_bwd_kernel (backward main)", "bound": "tensor",
                         "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "traffic_source": traffic_src,
                         "peak_source": f"{peak_src} bf16_tflops (burst)",
                         "avg_launch_ms": main_avg},
            "clocks": clocks,
            "layout_kernels": {"bound": "launch latency (KB-scale rows); HBM peak "
                                        f"{float(peaks['hbm_gbs']):.0f} GB/s ({peak_src})",
                               "timings": layout_times},
        }
        if args.dropout_p > 0.0:
            dv_ = job_rate(flops_step, args.steps, drop_ms, world) / 1e12
            line["dropout"] = {"p": args.dropout_p, "value": dv_, "unit": "TFLOP/s",
                               "ms_per_step": drop_ms / args.steps,
                               "frac_of_bf16_peak": dv_ / peak,
                               "relative_to_no_dropout": dv_ / value}
        if not args.no_cpu_baseline and world == 1:
            line["cpu_baseline"] = cpu_oracle_sample(wl, args.cpu_budget,
                                                     oracle_inputs(wl, args.seed))
            line["cpu_baseline"].pop("seconds", None)
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
