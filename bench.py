#!/usr/bin/env python
"""Throughput of the speculative-sampling verify step on GB300.

One step = one spec_verify_ex call over one synthetic batch of the workload (default: B=64 sequences,
gamma=5, V=128256, bf16 logits, T=1; 704 logit rows = 180,584,448 bytes read at least once). Inputs are
resident in HBM; four device copies are rotated so that the batch a step reads (180 MB each, 722 MB in
all) is never the one left in the 126 MB L2. Steps are replayed from a CUDA graph (launch overhead off
the host). The line printed by rank 0 reports verified logit rows/s, the roofline of the dominant kernel
against the measured HBM copy bandwidth, the end-to-end figure through the C ABI with host buffers, and
the CPU oracle timed on a bounded sample as a reported baseline.

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


def kernel_source_hash() -> str:
    """Hash of the CUDA sources' code (comments and layout excluded), keying profiled figures to the
    code they were measured on."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_decoding_verification_35_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h")):
            h.update(f.encode() + b"\0" + code_only(open(os.path.join(csrc, f), encoding="utf-8").read()).encode())
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
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
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
                rows.append((float(parts[0]), float(parts[1]), parts[3:]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


def cpu_oracle_rate(b, budget_s: float):
    """The oracle as it stands, on the host cores, over whole batches until ~budget_s of CPU time."""
    import oracle
    cores = len(os.sched_getaffinity(0))
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


def reference_arm(args):
    """The oracle as the reference implementation: each step verifies a bounded sample (the first
    `sample_b` sequences of the batch) on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    w = synth.WORKLOADS[args.workload]
    sample_b = min(w.B, 8)
    b = synth.make_batch(args.workload, B=sample_b)
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
    sample = f"first {sample_b} of {w.B} sequences ({b.verified_rows()} rows) per step"
    line = {"impl": "reference", "metric": METRIC, "value": rate, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": args.workload, "B": w.B, "gamma": int(w.gamma) if w.gamma else "U{1..8}",
                       "V": w.V, "temperature": w.temperature, "sample_B": sample_b},
            "cpu_baseline": {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": rate, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--workload", default=synth.HEADLINE, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU oracle budget (0: skip)")
    ap.add_argument("--e2e-steps", type=int, default=200)
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
    mg = int(b.gammas.max())
    L2 = torch.cuda.get_device_properties(dev).L2_cache_size
    in_bytes = b.target.nbytes + (b.draft.nbytes if b.draft is not None and not w.greedy else 0)
    ncopy = max(2, int(np.ceil(3 * L2 / in_bytes)) + 1)

    def logits(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
        return torch.from_numpy(a)

    host = dict(target=logits(b.target).pin_memory(),
                draft=logits(b.draft).pin_memory() if b.draft is not None else None,
                draft_tokens=torch.from_numpy(b.draft_tokens).pin_memory(),
                seq_offsets=torch.from_numpy(b.seq_offsets).pin_memory(),
                gammas=torch.from_numpy(b.gammas).pin_memory())
    copies = [{k: (v.to(dev) if v is not None else None) for k, v in host.items()} for _ in range(ncopy)]
    call = sv.Call(b.B, b.V, mg, b.R_t, b.R_d, device=dev)
    seed = 1234 + rank
    stream = torch.cuda.Stream(device=dev)
    kernels_per_step = 1  # the verify kernel (the call also enqueues one memset of the zeroed handoff regions)

    def one(i, c=None):
        c = copies[i % ncopy] if c is None else c
        rc = call.run(c["target"], c["draft"], c["draft_tokens"], c["seq_offsets"], c["gammas"], w.temperature,
                      seed, i, stream=stream, clear_status=False)
        if rc != sv.SV_OK:
            raise RuntimeError(sv.spec_verify_status_string(rc))

    # warm-up (direct launches), then one CUDA graph of G consecutive steps over the rotating copies
    with torch.cuda.stream(stream):
        call.status.zero_()
        for i in range(args.warmup):
            one(i)
    stream.synchronize()
    if call.status_bits():
        raise RuntimeError("device status " + sv.spec_verify_status_string(sv.spec_verify_status_from_bits(call.status_bits())))
    G = ncopy * 5
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(G):
            one(args.warmup + i)
    graph.replay()
    stream.synchronize()

    reps, rem = divmod(args.steps, G)
    sampler = ClockSampler(local)
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(reps):
            graph.replay()
        for i in range(rem):
            one(args.warmup + G + i)
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
    if call.status_bits():
        raise RuntimeError("device status bits set during the timed region")

    # end to end through the C ABI with host buffers (spec_verify_host): H2D of the inputs into staging
    # buffers, the step, D2H of the results, all enqueued by the one call
    dev_buf = copies[0]
    out_t_host = torch.empty(b.R_t, dtype=torch.int32).pin_memory()
    out_n_host = torch.empty(b.B, dtype=torch.int32).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in host.values() if v is not None)
    d2h = out_t_host.numel() * 4 + out_n_host.numel() * 4
    n_e2e = max(1, min(args.e2e_steps, args.steps))
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    x0 = torch.cuda.Event(enable_timing=True)
    x1 = torch.cuda.Event(enable_timing=True)
    x0.record(stream)
    with torch.cuda.stream(stream):
        for i in range(n_e2e):
            rc = call.run_host(host["target"], host["draft"], host["draft_tokens"], host["seq_offsets"],
                               host["gammas"], w.temperature, seed, i, out_t_host, out_n_host, dev_buf,
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

    # post-verify update (spec_verify_commit) on the last call's outputs: the device-side append of the
    # emitted tokens and the next input token, stream-ordered launches, no host sync between them
    n_commit = 200
    cap = 8 * n_commit
    hist = torch.zeros((b.B, cap), dtype=torch.int32, device=dev)
    lens = torch.zeros(b.B, dtype=torch.int32, device=dev)
    nxt = torch.zeros(b.B, dtype=torch.int32, device=dev)
    c0 = torch.cuda.Event(enable_timing=True)
    c1 = torch.cuda.Event(enable_timing=True)
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
    if call.status_bits():
        raise RuntimeError("device status bits set by the post-verify update")

    # the same steps with the update fused into the verify launch (spec_verify_fused), from a CUDA graph of
    # G steps like the timed region above; the history grows by at most max_gamma + 1 tokens per step
    n_fused = G * max(1, min(args.steps, 1000) // G)
    fcap = (mg + 1) * (n_fused + G + 1)
    fhist = torch.zeros((b.B, fcap), dtype=torch.int32, device=dev)
    flens = torch.zeros(b.B, dtype=torch.int32, device=dev)
    fnext = torch.zeros(b.B, dtype=torch.int32, device=dev)

    def one_fused(i):
        c = copies[i % ncopy]
        rc = call.run_fused(c["target"], c["draft"], c["draft_tokens"], c["seq_offsets"], c["gammas"], w.temperature,
                            seed, i, fhist, fcap, flens, fnext, stream=stream, clear_status=False)
        if rc != sv.SV_OK:
            raise RuntimeError(sv.spec_verify_status_string(rc))

    fgraph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(fgraph, stream=stream):
        for i in range(G):
            one_fused(i)
    fgraph.replay()  # warm (G steps of history)
    stream.synchronize()
    f0 = torch.cuda.Event(enable_timing=True)
    f1 = torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(n_fused // G):
            fgraph.replay()
    f1.record(stream)
    stream.synchronize()
    ms_fused = f0.elapsed_time(f1) / n_fused
    if call.status_bits():
        raise RuntimeError("device status bits set by the fused steps")

    # n-gram drafter (spec_draft_ngram) on synthetic histories of 2000 tokens with repeats, B sequences
    ng_cap, ng_len, ng_g = 4096, 2000, max(mg, 1)
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
    n0 = torch.cuda.Event(enable_timing=True)
    n1 = torch.cuda.Event(enable_timing=True)
    n_ng = 100
    n0.record(stream)
    for _ in range(n_ng):
        ngram_call()
    n1.record(stream)
    stream.synchronize()
    us_ngram = n0.elapsed_time(n1) / n_ng * 1e3

    # token-tree verification (spec_verify_tree): 64 trees of up to 15 candidate nodes, V of the workload
    tb = synth.make_tree_batch(64, b.V, 15, seed=1)
    tmg = int(tb.gammas.max())
    t_tg = torch.from_numpy(tb.target.view(np.int16)).view(torch.bfloat16).to(dev)
    t_d = {k: torch.from_numpy(v).to(dev) for k, v in dict(t=tb.draft_tokens, p=tb.parents, o=tb.seq_offsets,
                                                         g=tb.gammas).items()}
    t_ws_bytes = sv.spec_verify_workspace_size(tb.B, tb.V, tmg)
    t_ws = torch.empty(t_ws_bytes, dtype=torch.uint8, device=dev)
    t_out = torch.empty(tb.R_t, dtype=torch.int32, device=dev)
    t_n = torch.empty(tb.B, dtype=torch.int32, device=dev)
    t_path = torch.empty(max(int(tb.seq_offsets[-1]), 1), dtype=torch.int32, device=dev)

    def tree_call(i):
        if sv.spec_verify_tree(t_tg.data_ptr(), sv.SV_BF16, t_d["t"].data_ptr(), t_d["p"].data_ptr(),
                               t_d["o"].data_ptr(), t_d["g"].data_ptr(), tb.B, tb.V, tmg, 1.0, seed, i,
                               t_out.data_ptr(), t_n.data_ptr(), t_path.data_ptr(), call.status.data_ptr(),
                               t_ws.data_ptr(), t_ws_bytes, stream.cuda_stream) != sv.SV_OK:
            raise RuntimeError("spec_verify_tree failed")

    for i in range(3):
        tree_call(i)
    n_tree = 50
    v0 = torch.cuda.Event(enable_timing=True)
    v1 = torch.cuda.Event(enable_timing=True)
    v0.record(stream)
    for i in range(n_tree):
        tree_call(i)
    v1.record(stream)
    stream.synchronize()
    ms_tree = v0.elapsed_time(v1) / n_tree
    if call.status_bits():
        raise RuntimeError("device status bits set by the tree steps")

    rows = b.verified_rows()
    value = rows * world / (ms * 1e-3)
    e2e_value = rows * world / (ms_e2e * 1e-3)
    alg = b.algorithmic_bytes()
    peak, peak_src = peaks()
    achieved = alg / (ms * 1e-3) / 1e9
    traffic = profiled_traffic(args.workload)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16" if w.dtype == synth.BF16 else "f32",
            "data": "synthetic (seeded Gaussian + Zipf log-prior logits, Gumbel-max draft tokens)",
            "config": {"workload": args.workload, "B": b.B, "gamma": int(w.gamma) if w.gamma else "U{1..8}",
                       "V": b.V, "temperature": w.temperature, "rows_per_step": rows,
                       "algorithmic_bytes_per_step": alg, "l2_policy": f"{ncopy} rotating input copies "
                       f"({ncopy * in_bytes / 1e6:.0f} MB > 3x L2 {L2 / 1e6:.0f} MB)",
                       "launch": f"CUDA graph of {G} steps; per step one memset node (handoff regions) and "
                                 f"{kernels_per_step} verify kernel",
                       "parallelism": f"{world} independent replica(s), sequences sharded by rank"},
            "achieved_hbm_gbs": achieved,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
                         else "fallback 6.8 TB/s",
                         "timed": "whole verify step (memset + kernel) per step, CUDA events on the launch "
                                  "stream; the kernel's share of the step is in profiles/"},
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "call": "spec_verify_host per step: page-locked host buffers in and out, copies inside",
                    "steps": n_e2e, "ms_per_step": ms_e2e},
            "gpu_launches": args.steps * kernels_per_step,
            "clocks": clocks,
            "post_verify_update": {"us_per_call": us_commit, "calls": n_commit, "B": b.B,
                                   "launch": "spec_verify_commit, stream-ordered after the verify steps, "
                                             "one kernel per call, no host sync",
                                   "fused_ms_per_step": ms_fused, "fused_steps": n_fused,
                                   "fused_extra_us_per_step": (ms_fused - ms) * 1e3,
                                   "fused_launch": f"spec_verify_fused from a CUDA graph of {G} steps"},
            "tree_verify": {"ms_per_call": ms_tree, "calls": n_tree, "B": tb.B, "nodes": tb.R_t, "V": tb.V,
                            "rows_per_s": tb.R_t / (ms_tree * 1e-3),
                            "launch": "spec_verify_tree, stream-ordered, inputs resident (L2 may hold part)"},
            "ngram_drafter": {"us_per_call": us_ngram, "calls": n_ng, "B": b.B, "history_tokens": ng_len,
                              "n": "4..1", "gamma_max": ng_g,
                              "launch": "spec_draft_ngram: search (one CTA per sequence) + pack (one CTA)"},
        }
        if world == 1 and args.cpu_seconds > 0:
            rate, cores, sample = cpu_oracle_rate(b, args.cpu_seconds)
            line["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample}
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
