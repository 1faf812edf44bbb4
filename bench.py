#!/usr/bin/env python
"""Throughput of the speculative-sampling verify step on GB300.

One step = one spec_verify_ex call over one synthetic batch of the workload (default: B=64 sequences,
gamma=5, V=128256, bf16 logits, T=1; 704 logit rows = 180,584,448 bytes read at least once). Inputs are
resident in HBM; device copies of the batch are rotated so that the batch a step reads is never the one
left in the 126 MB L2 (more than 3x L2 in all). Steps are replayed from a CUDA graph (launch overhead off
the host). The line printed by rank 0 reports verified logit rows/s, the roofline of the dominant kernel
against the measured HBM copy bandwidth, the end-to-end figure through the C ABI with host buffers, the
CPU oracle timed on a bounded sample as a reported baseline, a parity sample (GPU against the oracle on
many steps: band and mismatch counts), and one block per synthetic workload with the timing protocol of
the scope table (median and p10/p90 over repeats, graph replay against per-call launches, the oracle on
all host cores and on one).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

For N > 1 (torchrun) every rank verifies its own batch (sequences are independent: weak scaling, no
collective on the data path); the barrier and max-over-ranks timing use NCCL.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from speculative_decoding_verification_35_gb300 import synth  # noqa: E402

METRIC = "verified logit rows/s and achieved HBM GB/s (% of ~8 TB/s) at V=128256, B=64, γ=5"
UNIT = "rows/s"


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


_TOKENS = re.compile(r'"(?:\\.|[^"\\\n])*"|//[^\n]*|/\*.*?\*/', re.S)


def code_only(src: str) -> str:
    """C/C++ source without its comments and with whitespace runs collapsed (string literals kept)."""
    src = _TOKENS.sub(lambda m: m.group(0) if m.group(0).startswith('"') else " ", src)
    return " ".join(src.split())


# the sources a profiled kernel's launch is built from: its kernel file, the device helpers, the shared
# declarations, the host code that fills its parameters and picks its launch, and the public header
KERNEL_SOURCES = {
    "k_verify": ("speculative_decoding_verification_35_gb300/csrc/sv_api.cu",
                 "speculative_decoding_verification_35_gb300/csrc/sv_kernels.cu",
                 "speculative_decoding_verification_35_gb300/csrc/sv_device.cuh",
                 "speculative_decoding_verification_35_gb300/csrc/sv_internal.h",
                 "include/specverify.h"),
}


def kernel_source_hash(kernel: str = "k_verify") -> str:
    """Hash of the code (comments and layout excluded) of the sources a kernel is built from, keying
    profiled figures to the code they were measured on."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        h.update(f.encode() + b"\0" + code_only(open(os.path.join(ROOT, f), encoding="utf-8").read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per launch of the dominant kernel from the committed ncu summary, if it was taken on
    the current kernel sources; else None."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    e = d.get(workload)
    if not e or e.get("source_hash") != kernel_source_hash():
        return None
    return e.get("bytes_per_launch")


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons, from the warm-up under load through the timed
    region (a timed region of a few milliseconds is shorter than any sampling period, so the samples of the
    warm-up steps just before it, under the same load, are kept with it)."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 20):
        self.proc = None
        self.period_ms = period_ms
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", str(period_ms)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = []
        for line in out.splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) != 7:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), float(parts[2]), parts[3:]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for *_, r in rows for i, v in enumerate(r) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "power_w_max": max(r[2] for r in rows), "reasons": reasons, "samples": len(rows),
                "period_ms": self.period_ms, "window": "warm-up under load and the timed region"}


def cpu_oracle_rate(b, budget_s: float, threads: int | None = None):
    """The oracle as it stands, on `threads` host threads (all cores by default), over whole batches until
    ~budget_s of wall time (at least one batch)."""
    import oracle
    cores = threads or len(os.sched_getaffinity(0))
    rows = 0
    t0 = time.perf_counter()
    step = 0
    while True:
        r = oracle.verify(b.target, b.draft, b.draft_tokens, b.seq_offsets, b.gammas, b.V, b.temperature,
                          1234, step, nthreads=cores)
        assert r.status == 0
        rows += b.verified_rows()
        step += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return rows / dt, cores, f"{step} full batches of the workload ({b.verified_rows()} rows each) in {dt:.1f} s"


def workload_config(w, b):
    return {"workload": w.name, "B": b.B, "gamma": int(w.gamma) if w.gamma else "U{1..8}", "V": b.V,
            "temperature": w.temperature, "dtype": w.dtype, "rows_per_step": b.verified_rows(),
            "algorithmic_bytes_per_step": b.algorithmic_bytes()}


def reference_arm(args):
    """The oracle as the reference implementation, on the full batch of the workload: each step verifies
    every sequence on the host cores (same workload, metric and unit as the GPU arm)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    w = synth.WORKLOADS[args.workload]
    b = synth.make_batch(args.workload)
    cores = len(os.sched_getaffinity(0))
    for s in range(args.warmup):
        oracle.verify(b.target, b.draft, b.draft_tokens, b.seq_offsets, b.gammas, b.V, b.temperature, 1234, s,
                      nthreads=cores)
    t0 = time.perf_counter()
    for s in range(args.steps):
        r = oracle.verify(b.target, b.draft, b.draft_tokens, b.seq_offsets, b.gammas, b.V, b.temperature, 1234,
                          args.warmup + s, nthreads=cores)
        assert r.status == 0
    dt = time.perf_counter() - t0
    rate = b.verified_rows() * args.steps / dt
    sample = f"the full batch ({b.B} sequences, {b.verified_rows()} rows) per step, {args.steps} steps"
    line = {"impl": "reference", "metric": METRIC, "value": rate, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(w, b),
            "cpu_baseline": {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": rate, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def pct(v, q):
    return float(np.percentile(np.asarray(v, dtype=np.float64), q))


class Rig:
    """Device copies of one batch (rotated so that a step never reads the batch left in L2), one verify
    call's buffers and its stream; one(i) enqueues step i on copy i mod ncopy."""

    def __init__(self, b, dev, L2, seed, stream=None, debug=False):
        import torch
        from speculative_decoding_verification_35_gb300 import specverify as sv
        self.sv, self.torch, self.b, self.dev, self.seed = sv, torch, b, dev, seed
        w = b.workload
        self.in_bytes = b.target.nbytes + (b.draft.nbytes if b.draft is not None and not w.greedy else 0)
        self.ncopy = min(16, max(2, int(np.ceil(3 * L2 / self.in_bytes)) + 1))
        # a batch too small for 16 copies to exceed 3x L2 is L2-resident in graph replays; its cold-L2 figure
        # comes from single steps with L2 flushed before each (flushed_repeats)
        self.l2_resident = self.ncopy * self.in_bytes < 3 * L2
        self.L2 = L2

        def logits(a):
            if a is None:
                return None
            if a.dtype == np.uint16:
                return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
            return torch.from_numpy(a)

        self.host = dict(target=logits(b.target).pin_memory(),
                         draft=logits(b.draft).pin_memory() if b.draft is not None else None,
                         draft_tokens=torch.from_numpy(b.draft_tokens).pin_memory(),
                         seq_offsets=torch.from_numpy(b.seq_offsets).pin_memory(),
                         gammas=torch.from_numpy(b.gammas).pin_memory())
        self.copies = [{k: (v.to(dev) if v is not None else None) for k, v in self.host.items()}
                       for _ in range(self.ncopy)]
        self.mg = int(b.gammas.max())
        self.call = sv.Call(b.B, b.V, self.mg, b.R_t, b.R_d, device=dev, debug=debug)
        self.stream = stream or torch.cuda.Stream(device=dev)
        self.G = self.ncopy * max(1, 20 // self.ncopy)  # steps per captured graph: whole rotations

    def one(self, i, out_tokens=None, out_n=None):
        c = self.copies[i % self.ncopy]
        w = self.b.workload
        if out_tokens is None:
            rc = self.call.run(c["target"], c["draft"], c["draft_tokens"], c["seq_offsets"], c["gammas"],
                               w.temperature, self.seed, i, stream=self.stream, clear_status=False)
        else:  # outputs of this step into the caller's buffers (parity samples)
            sv, call = self.sv, self.call
            rc = sv.spec_verify_ex(c["target"].data_ptr(), c["draft"].data_ptr() if c["draft"] is not None else None,
                                   sv.dtype_code(c["target"]), c["draft_tokens"].data_ptr(),
                                   c["seq_offsets"].data_ptr(), c["gammas"].data_ptr(), call.B, call.V, call.max_gamma,
                                   w.temperature, self.seed, i, out_tokens, out_n, call.status.data_ptr(),
                                   call.workspace.data_ptr(), call.ws_bytes, None, self.stream.cuda_stream)
        if rc != self.sv.SV_OK:
            raise RuntimeError(self.sv.spec_verify_status_string(rc))

    def capture(self, first):
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.stream):
            for i in range(self.G):
                self.one(first + i)
        return g

    def check_status(self, what):
        bits = self.call.status_bits()
        if bits:
            raise RuntimeError(f"device status {bits:#x} after {what}")

    def event(self):
        return self.torch.cuda.Event(enable_timing=True)

    def replay(self, graph, n=1):
        """n replays of a captured graph on the rig's stream (a replay goes to the current stream: outside this
        context it would run on the default stream, beside and unordered with the rig's work)."""
        with self.torch.cuda.stream(self.stream):
            for _ in range(n):
                graph.replay()

    def graph_repeats(self, graph, reps):
        """Per-step ms of `reps` replays of a G-step graph, each replay timed on the stream."""
        out = []
        for _ in range(reps):
            e0, e1 = self.event(), self.event()
            e0.record(self.stream)
            self.replay(graph)
            e1.record(self.stream)
            self.stream.synchronize()
            out.append(e0.elapsed_time(e1) / self.G)
        return out

    def direct_repeats(self, first, reps):
        """Per-step ms of `reps` runs of G per-call launches (host enqueue of every call included)."""
        out = []
        with self.torch.cuda.stream(self.stream):
            for r in range(reps):
                e0, e1 = self.event(), self.event()
                e0.record(self.stream)
                for i in range(self.G):
                    self.one(first + r * self.G + i)
                e1.record(self.stream)
                self.stream.synchronize()
                out.append(e0.elapsed_time(e1) / self.G)
        return out

    def flushed_repeats(self, first, n):
        """Device ms of `n` single steps, each preceded (outside its events) by a write of 2x L2 bytes, so
        that the step finds none of its inputs in L2; the flush also covers the host's launch of the step."""
        torch = self.torch
        flush = torch.empty(2 * self.L2, dtype=torch.uint8, device=self.dev)
        ev = [(self.event(), self.event()) for _ in range(n)]
        with torch.cuda.stream(self.stream):
            for i, (e0, e1) in enumerate(ev):
                flush.zero_()
                e0.record(self.stream)
                self.one(first + i)
                e1.record(self.stream)
        self.stream.synchronize()
        del flush
        return [e0.elapsed_time(e1) for e0, e1 in ev]

    def l2_policy(self):
        tot = self.ncopy * self.in_bytes
        if not self.l2_resident:
            return (f"{self.ncopy} rotating input copies ({tot / 1e6:.0f} MB > 3x L2 {self.L2 / 1e6:.0f} MB): a step "
                    f"never reads the batch a previous step left in L2")
        return (f"batch of {self.in_bytes / 1e6:.3f} MB: {self.ncopy} rotating copies fit in L2, so graph replays "
                f"read L2-resident inputs; cold-L2 steps are timed one by one with a 2x L2 write before each")

    def release(self):
        self.copies = None
        self.host = None
        self.call = None
        self.torch.cuda.synchronize(self.dev)
        self.torch.cuda.empty_cache()


def parity_sample(rig, steps, first):
    """`steps` consecutive verify calls on one copy of the batch, each with its own outputs, compared with
    the oracle's multi-step entry: token draws, uniform draws (accept tests and draws), band and mismatch
    counts of the contract (mismatch outside the 1e-6 band: none allowed; band: below 1e-5 of draws)."""
    import oracle
    from tests import parity
    torch, b = rig.torch, rig.b
    out_t = torch.full((steps, b.R_t), -9, dtype=torch.int32, device=rig.dev)
    out_n = torch.full((steps, b.B), -9, dtype=torch.int32, device=rig.dev)
    rig.call.status.zero_()
    with torch.cuda.stream(rig.stream):
        for s in range(steps):
            rig.one(first + s, out_t[s].data_ptr(), out_n[s].data_ptr())
    rig.stream.synchronize()
    rig.check_status("the parity sample")
    # every step above ran on copy (first + s) mod ncopy; all copies hold the same batch
    T = float(np.float32(b.temperature))
    r_t, r_n, st = oracle.verify_steps(b.target, b.draft, b.draft_tokens, b.seq_offsets, b.gammas, b.V, T,
                                       rig.seed, first, steps)
    r0 = oracle.verify(b.target, b.draft, b.draft_tokens, b.seq_offsets, b.gammas, b.V, T, rig.seed, first)
    rep = parity.compare_steps(b, out_t.cpu().numpy(), out_n.cpu().numpy(), r_t, r_n, r0, rig.seed, first)
    return {"steps": steps, "seed": rig.seed, "first_step": first, "token_draws": rep["token_draws"],
            "uniform_draws": rep["draws"], "band": len(rep["band"]), "mismatch": len(rep["bad"]),
            "rule": "tokens and counts equal the fp64 oracle's except draws whose uniform lies within 1e-6 of "
                    "an oracle boundary (band, allowed below 1e-5 of draws); mismatch: any other difference",
            "oracle_status": st}, out_n.cpu().numpy(), r0


def beta_groups(rig, n_sample):
    """Realised beta per draft-noise group of the headline workload (sigma_b cycles over the sequences):
    mean beta_i = sum_x min(p_i, q_i) of the group's draft slots from the debug output, and the share of
    slot-0 accept tests passed in the parity sample (an estimate of beta_0)."""
    torch, b, sv = rig.torch, rig.b, rig.sv
    w = b.workload
    dbg_call = sv.Call(b.B, b.V, rig.mg, b.R_t, b.R_d, device=rig.dev, debug=True)
    c = rig.copies[0]
    rc = dbg_call.run(c["target"], c["draft"], c["draft_tokens"], c["seq_offsets"], c["gammas"], w.temperature,
                      rig.seed, 0, stream=rig.stream)
    if rc != sv.SV_OK:
        raise RuntimeError(sv.spec_verify_status_string(rc))
    rig.stream.synchronize()
    beta = dbg_call.dbg["beta"].cpu().numpy()
    sig = np.array([w.draft_sigmas[q % len(w.draft_sigmas)] for q in range(b.B)])
    slot_seq = np.repeat(np.arange(b.B), b.gammas)
    out = {}
    for sg in w.draft_sigmas:
        seqs = np.nonzero(sig == sg)[0]
        acc0 = (n_sample[:, seqs] >= 1).mean() if len(seqs) and b.gammas[seqs].min() > 0 else None
        out[f"sigma_{sg}"] = {"sequences": int(len(seqs)), "beta_mean": float(beta[np.isin(slot_seq, seqs)].mean()),
                              "slot0_accept_rate": None if acc0 is None else float(acc0)}
    return out


def measure_workload(name, dev, L2, peak, peak_src, reps, oracle_budget):
    """One workload with the scope table's timing protocol: a CUDA graph of G steps over rotating copies,
    `reps` timed replays (median, p10, p90 of the per-step time), the same steps as per-call launches, and
    the oracle on all host cores and on one (bounded samples of whole batches)."""
    b = synth.make_batch(name)
    rig = Rig(b, dev, L2, seed=1234)
    with rig.torch.cuda.stream(rig.stream):
        for i in range(3):
            rig.one(i)
    graph = rig.capture(3)
    rig.replay(graph)
    rig.stream.synchronize()
    g_ms = rig.graph_repeats(graph, reps)
    d_ms = rig.direct_repeats(3 + rig.G, reps)
    f_ms = rig.flushed_repeats(3 + rig.G * (reps + 1), 8 * reps) if rig.l2_resident else None
    rig.check_status(name)
    med = statistics.median(f_ms if f_ms else g_ms)
    alg = b.algorithmic_bytes()
    cores = len(os.sched_getaffinity(0))
    o_all, _, s_all = cpu_oracle_rate(b, oracle_budget)
    o_one, _, s_one = cpu_oracle_rate(b, oracle_budget, threads=1)
    rows = b.verified_rows()
    out = {"config": workload_config(b.workload, b),
           "rows_per_s": rows / (med * 1e-3), "achieved_gbs": alg / (med * 1e-3) / 1e9,
           "frac": alg / (med * 1e-3) / 1e9 / peak, "peak_gbs": peak, "peak_source": peak_src,
           "graph_ms_per_step": {"median": statistics.median(g_ms), "p10": pct(g_ms, 10), "p90": pct(g_ms, 90),
                                 "repeats": reps,
                                 "steps_per_repeat": rig.G},
           "launch_ms_per_step": {"median": statistics.median(d_ms), "p10": pct(d_ms, 10), "p90": pct(d_ms, 90),
                                  "repeats": reps, "steps_per_repeat": rig.G},
           "cold_l2_ms_per_step": None if f_ms is None else {"median": statistics.median(f_ms), "p10": pct(f_ms, 10),
                                                             "p90": pct(f_ms, 90), "steps": len(f_ms)},
           "rate_basis": "median cold-L2 single step" if f_ms else "median graph-replayed step (inputs beyond L2)",
           "l2_policy": rig.l2_policy(),
           "oracle": {"all_cores": {"rows_per_s": o_all, "threads": cores, "sample": s_all},
                      "one_thread": {"rows_per_s": o_one, "threads": 1, "sample": s_one}}}
    rig.release()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--workload", default=synth.HEADLINE, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU oracle budget (0: skip)")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--parity-steps", type=int, default=1000, help="steps of the parity sample (0: skip)")
    ap.add_argument("--workloads", default="all",
                    help="comma-separated workloads to measure with the full protocol ('all', or 'none')")
    ap.add_argument("--repeats", type=int, default=25, help="timed repeats per workload")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.impl == "reference":
        return reference_arm(args)

    import torch
    from speculative_decoding_verification_35_gb300 import specverify as sv

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)

    b = synth.make_batch(args.workload)
    w = b.workload
    L2 = torch.cuda.get_device_properties(dev).L2_cache_size
    peak, peak_src = peaks()
    rig = Rig(b, dev, L2, seed=1234 + rank)
    stream, G = rig.stream, rig.G
    kernels_per_step = 1  # the verify kernel (the call also enqueues one memset of the zeroed handoff regions)

    # warm-up: W direct steps, then graph replays until the GPU has run under load for >= 0.3 s (clocks up),
    # with the clock sampler running from here through the timed region
    sampler = ClockSampler(local)
    with torch.cuda.stream(stream):
        rig.call.status.zero_()
        for i in range(args.warmup):
            rig.one(i)
    stream.synchronize()
    rig.check_status("warm-up")
    graph = rig.capture(args.warmup)
    warm_steps, t_warm = args.warmup, time.perf_counter()
    while warm_steps < 100_000:  # each replay waited for: 0.3 s of steps actually run
        rig.replay(graph)
        stream.synchronize()
        warm_steps += G
        if time.perf_counter() - t_warm >= 0.3:
            break

    # the timed region: exactly K steps (graph replays of G steps, then the remainder as direct launches)
    reps, rem = divmod(args.steps, G)
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    e0, e1 = rig.event(), rig.event()
    e0.record(stream)
    rig.replay(graph, reps)
    with torch.cuda.stream(stream):
        for i in range(rem):
            rig.one(args.warmup + G + i)
    e1.record(stream)
    stream.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    ms = e0.elapsed_time(e1) / args.steps
    if dist:
        t = torch.tensor([ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    rig.check_status("the timed region")

    # repeats of the same graph (timing spread of the headline) and the same steps as per-call launches
    rep_ms = rig.graph_repeats(graph, args.repeats)
    launch_ms = rig.direct_repeats(args.warmup + G, args.repeats)
    rig.check_status("the repeats")

    # end to end through the C ABI with host buffers (spec_verify_host): H2D of the inputs into staging
    # buffers, the step, D2H of the results, all enqueued by the one call
    call, host = rig.call, rig.host
    dev_buf = rig.copies[0]
    out_t_host = torch.empty(b.R_t, dtype=torch.int32).pin_memory()
    out_n_host = torch.empty(b.B, dtype=torch.int32).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in host.values() if v is not None)
    d2h = out_t_host.numel() * 4 + out_n_host.numel() * 4
    n_e2e = max(1, args.e2e_steps)  # its own step count: a few ms of copies, independent of --steps
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    x0, x1 = rig.event(), rig.event()
    x0.record(stream)
    with torch.cuda.stream(stream):
        for i in range(n_e2e):
            rc = call.run_host(host["target"], host["draft"], host["draft_tokens"], host["seq_offsets"],
                               host["gammas"], w.temperature, rig.seed, i, out_t_host, out_n_host, dev_buf,
                               stream=stream, clear_status=False)
            if rc != sv.SV_OK:
                raise RuntimeError(sv.spec_verify_status_string(rc))
    x1.record(stream)
    stream.synchronize()
    ms_e2e = x0.elapsed_time(x1) / n_e2e
    if dist:
        t = torch.tensor([ms_e2e], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_e2e = float(t.item())

    # parity sample (rank 0 of a single-GPU run): GPU steps against the oracle, band and mismatch counts
    psample, betas = None, None
    if world == 1 and args.parity_steps > 0 and not w.greedy:
        psample, n_sample, _ = parity_sample(rig, args.parity_steps, 100_000)
        if len(w.draft_sigmas) > 1:
            betas = beta_groups(rig, n_sample)

    # post-verify update (spec_verify_commit) on the last call's outputs: the device-side append of the
    # emitted tokens and the next input token, stream-ordered launches, no host sync between them
    n_commit = 200
    cap = 8 * n_commit
    hist = torch.zeros((b.B, cap), dtype=torch.int32, device=dev)
    lens = torch.zeros(b.B, dtype=torch.int32, device=dev)
    nxt = torch.zeros(b.B, dtype=torch.int32, device=dev)
    c0, c1 = rig.event(), rig.event()
    with torch.cuda.stream(stream):
        call.commit(dev_buf["seq_offsets"], hist, cap, lens, nxt, stream=stream)  # warm
        lens.zero_()
        c0.record(stream)
        for _ in range(n_commit):
            if call.commit(dev_buf["seq_offsets"], hist, cap, lens, nxt, stream=stream) != sv.SV_OK:
                raise RuntimeError("spec_verify_commit failed")
        c1.record(stream)
    stream.synchronize()
    us_commit = c0.elapsed_time(c1) / n_commit * 1e3
    rig.check_status("the post-verify update")

    # the same steps with the update fused into the verify launch (spec_verify_fused), from a CUDA graph of G
    # steps like the timed region above; warmed up under load like the headline, then timed over a fixed
    # number of steps (independent of --steps)
    n_fused_warm, n_fused = 10 * G, G * max(1, 1000 // G)
    fcap = (rig.mg + 1) * (n_fused + n_fused_warm + G + 1)
    fhist = torch.zeros((b.B, fcap), dtype=torch.int32, device=dev)
    flens = torch.zeros(b.B, dtype=torch.int32, device=dev)
    fnext = torch.zeros(b.B, dtype=torch.int32, device=dev)

    def one_fused(i):
        c = rig.copies[i % rig.ncopy]
        rc = call.run_fused(c["target"], c["draft"], c["draft_tokens"], c["seq_offsets"], c["gammas"], w.temperature,
                            rig.seed, i, fhist, fcap, flens, fnext, stream=stream, clear_status=False)
        if rc != sv.SV_OK:
            raise RuntimeError(sv.spec_verify_status_string(rc))

    fgraph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(fgraph, stream=stream):
        for i in range(G):
            one_fused(i)
    rig.replay(fgraph, n_fused_warm // G)
    stream.synchronize()
    f0, f1 = rig.event(), rig.event()
    f0.record(stream)
    rig.replay(fgraph, n_fused // G)
    f1.record(stream)
    stream.synchronize()
    ms_fused = f0.elapsed_time(f1) / n_fused
    # the unfused steps timed the same way right after, for the difference
    u0, u1 = rig.event(), rig.event()
    u0.record(stream)
    rig.replay(graph, n_fused // G)
    u1.record(stream)
    stream.synchronize()
    ms_unfused = u0.elapsed_time(u1) / n_fused
    rig.check_status("the fused steps")

    # n-gram drafter (spec_draft_ngram) on synthetic histories of 2000 tokens with repeats, B sequences
    ng_cap, ng_len, ng_g = 4096, 2000, max(rig.mg, 1)
    ng_rng = np.random.default_rng(77)
    ng_hist = ng_rng.integers(0, 500, size=(b.B, ng_cap)).astype(np.int32)
    for r in range(b.B):  # plant a repeat of the last 4 tokens 300 tokens earlier
        ng_hist[r, ng_len - 300:ng_len - 296] = ng_hist[r, ng_len - 4:ng_len]
    ng_h = torch.from_numpy(ng_hist).to(dev)
    ng_L = torch.full((b.B,), ng_len, dtype=torch.int32, device=dev)
    ng_t = torch.zeros(b.B * ng_g, dtype=torch.int32, device=dev)
    ng_gam = torch.zeros(b.B, dtype=torch.int32, device=dev)
    ng_off = torch.zeros(b.B + 1, dtype=torch.int32, device=dev)
    ng_pos = torch.zeros(b.B, dtype=torch.int32, device=dev)

    def ngram_call():
        if sv.spec_draft_ngram(ng_h.data_ptr(), ng_cap, ng_L.data_ptr(), b.B, 1, 4, ng_g, ng_t.data_ptr(),
                               ng_gam.data_ptr(), ng_off.data_ptr(), ng_pos.data_ptr(), call.status.data_ptr(),
                               stream.cuda_stream) != sv.SV_OK:
            raise RuntimeError("spec_draft_ngram failed")

    ngram_call()
    n0, n1 = rig.event(), rig.event()
    n_ng = 100
    n0.record(stream)
    for _ in range(n_ng):
        ngram_call()
    n1.record(stream)
    stream.synchronize()
    us_ngram = n0.elapsed_time(n1) / n_ng * 1e3

    # token-tree verification (spec_verify_tree): 64 trees of up to 15 candidate nodes, V of the workload,
    # rotating input copies like the headline (the tree read is never the one left in L2)
    tb = synth.make_tree_batch(64, b.V, 15, seed=1)
    tmg = int(tb.gammas.max())
    t_host = torch.from_numpy(tb.target.view(np.int16)).view(torch.bfloat16)
    t_ncopy = max(2, int(np.ceil(3 * L2 / tb.target.nbytes)) + 1)
    t_tg = [t_host.to(dev) for _ in range(t_ncopy)]
    t_d = {k: torch.from_numpy(v).to(dev) for k, v in dict(t=tb.draft_tokens, p=tb.parents, o=tb.seq_offsets,
                                                         g=tb.gammas).items()}
    t_ws_bytes = sv.spec_verify_workspace_size(tb.B, tb.V, tmg)
    t_ws = torch.empty(t_ws_bytes, dtype=torch.uint8, device=dev)
    t_out = torch.empty(tb.R_t, dtype=torch.int32, device=dev)
    t_n = torch.empty(tb.B, dtype=torch.int32, device=dev)
    t_path = torch.empty(max(int(tb.seq_offsets[-1]), 1), dtype=torch.int32, device=dev)

    def tree_call(i):
        if sv.spec_verify_tree(t_tg[i % t_ncopy].data_ptr(), sv.SV_BF16, t_d["t"].data_ptr(), t_d["p"].data_ptr(),
                               t_d["o"].data_ptr(), t_d["g"].data_ptr(), tb.B, tb.V, tmg, 1.0, rig.seed, i,
                               t_out.data_ptr(), t_n.data_ptr(), t_path.data_ptr(), call.status.data_ptr(),
                               t_ws.data_ptr(), t_ws_bytes, stream.cuda_stream) != sv.SV_OK:
            raise RuntimeError("spec_verify_tree failed")

    with torch.cuda.stream(stream):
        for i in range(3):
            tree_call(i)
    n_tree = 20 * t_ncopy
    v0, v1 = rig.event(), rig.event()
    with torch.cuda.stream(stream):
        v0.record(stream)
        for i in range(n_tree):
            tree_call(i)
        v1.record(stream)
    stream.synchronize()
    ms_tree = v0.elapsed_time(v1) / n_tree
    rig.check_status("the tree steps")
    del t_tg

    # vocabulary-sharded verify (spec_shard_*): the headline batch split over S shards held by this process
    # on this one GPU, each shard's four calls in turn and the exchanges as stacks of the shards' records
    # (the protocol a tensor-parallel group runs over NCCL); a single-GPU figure, not a multi-GPU one
    sharded = None
    if world == 1:
        from speculative_decoding_verification_35_gb300.shard import CudaShard, local_steps
        sharded = {}
        c0d = rig.copies[0]
        for S in (2, 4):
            bounds = [b.V * j // S for j in range(S + 1)]
            shards = [CudaShard(j, bounds, c0d["target"][:, bounds[j]:bounds[j + 1]].contiguous(),
                                c0d["draft"][:, bounds[j]:bounds[j + 1]].contiguous() if c0d["draft"] is not None else None,
                                c0d["draft_tokens"], c0d["seq_offsets"], c0d["gammas"], b.B, b.V, rig.mg, b.R_t, b.R_d,
                                w.temperature) for j in range(S)]
            with torch.cuda.stream(stream):
                for i in range(3):
                    local_steps(shards, rig.seed, i)
            stream.synchronize()
            n_sh = 20  # steps per graph (the calls and the exchanges' stacks, captured once)
            sgraph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(sgraph, stream=stream):
                for i in range(n_sh):
                    local_steps(shards, rig.seed, 3 + i)
            rig.replay(sgraph)
            stream.synchronize()
            s0, s1 = rig.event(), rig.event()
            s0.record(stream)
            rig.replay(sgraph, 5)
            s1.record(stream)
            stream.synchronize()
            n_sh *= 5
            if any(int(sh.status.item()) for sh in shards):
                raise RuntimeError("device status bits set by the sharded steps")
            sharded[f"S{S}"] = {"ms_per_step": s0.elapsed_time(s1) / n_sh, "steps": n_sh, "shards": S}
            del shards
        sharded["launch"] = ("per step and shard: statistics, decisions, sums, finish (4 launches), the records "
                             "stacked between them; shards run in turn on one GPU, inputs resident (one copy); "
                             "replayed from a CUDA graph of 20 steps")

    rows = b.verified_rows()
    value = rows * world / (ms * 1e-3)
    e2e_value = rows * world / (ms_e2e * 1e-3)
    alg = b.algorithmic_bytes()
    achieved = alg / (ms * 1e-3) / 1e9
    traffic = profiled_traffic(args.workload)
    cfg = workload_config(w, b)
    cfg.update({"l2_policy": rig.l2_policy(),
                "launch": f"CUDA graph of {G} steps; per step one memset node (handoff regions) and "
                          f"{kernels_per_step} verify kernel",
                "parallelism": f"{world} independent replica(s): each rank verifies its own batch"})
    line = None
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": warm_steps, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16" if w.dtype == synth.BF16 else "f32",
            "data": "synthetic (seeded Gaussian + Zipf log-prior logits, Gumbel-max draft tokens)",
            "config": cfg,
            "achieved_hbm_gbs": achieved,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
                         else "fallback 6.8 TB/s",
                         "timed": "whole verify step (memset + kernel) per step, CUDA events on the launch "
                                  "stream; the kernel's share of the step is in profiles/"},
            "timing_spread": {"graph_ms_per_step": {"median": statistics.median(rep_ms), "p10": pct(rep_ms, 10),
                                                    "p90": pct(rep_ms, 90), "repeats": args.repeats,
                                                    "steps_per_repeat": G},
                              "launch_ms_per_step": {"median": statistics.median(launch_ms),
                                                     "p10": pct(launch_ms, 10), "p90": pct(launch_ms, 90),
                                                     "repeats": args.repeats, "steps_per_repeat": G,
                                                     "launch": "per-call spec_verify_ex from Python, "
                                                               "stream-ordered, no graph"}},
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "call": "spec_verify_host per step: page-locked host buffers in and out, copies inside",
                    "steps": n_e2e, "ms_per_step": ms_e2e},
            "gpu_launches": args.steps * kernels_per_step,
            "clocks": clocks,
            "parity_sample": psample,
            "beta_by_draft_sigma": betas,
            "post_verify_update": {"us_per_call": us_commit, "calls": n_commit, "B": b.B,
                                   "launch": "spec_verify_commit, stream-ordered after the verify steps, "
                                             "one kernel per call, no host sync",
                                   "fused_ms_per_step": ms_fused, "unfused_ms_per_step": ms_unfused,
                                   "fused_steps": n_fused, "fused_warmup_steps": n_fused_warm,
                                   "fused_extra_us_per_step": (ms_fused - ms_unfused) * 1e3,
                                   "fused_launch": f"spec_verify_fused from a CUDA graph of {G} steps; the "
                                                   f"unfused graph timed right after over as many steps"},
            "tree_verify": {"ms_per_call": ms_tree, "calls": n_tree, "B": tb.B, "nodes": tb.R_t, "V": tb.V,
                            "rows_per_s": tb.R_t / (ms_tree * 1e-3),
                            "launch": f"spec_verify_tree, stream-ordered, {t_ncopy} rotating input copies"},
            "vocab_sharded_verify": sharded,
            "ngram_drafter": {"us_per_call": us_ngram, "calls": n_ng, "B": b.B, "history_tokens": ng_len,
                              "n": "4..1", "gamma_max": ng_g,
                              "launch": "spec_draft_ngram: search (one CTA per sequence) + pack (one CTA)"},
        }
    rig.release()
    if rank == 0 and world == 1:
        names = [] if args.workloads == "none" else (
            [n for n in synth.WORKLOADS] if args.workloads == "all" else args.workloads.split(","))
        line["workloads"] = {n: measure_workload(n, dev, L2, peak, peak_src, args.repeats, 1.0) for n in names}
        if args.cpu_seconds > 0:
            rate, cores, sample = cpu_oracle_rate(b, args.cpu_seconds)
            line["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
