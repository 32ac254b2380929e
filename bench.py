#!/usr/bin/env python3
"""Benchmark of the batched speculative-verification step on GB300.

One step = one spec_verify_dense call over the dense workload of B = 64 rows,
gamma = 7 drafts, V = 128,256 (bf16 logits): every row of the hot path runs
in it (softmax statistics, gather, ratio test, first-reject scan, residual /
bonus inverse CDF, emit).  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

value      verified positions/s (B * gamma per step) over all ranks, inputs
           resident in HBM (two rotating input copies, 2 x 246 MB > L2)
e2e        the same metric through the C ABI with host buffers: per step the
           pinned-host -> device copy of the inputs, the call, and the
           device -> host copy of n_accepted and out_tokens
roofline   the fused dense kernel: algorithmic bytes per launch / mean launch
           time (CUDA events on the launching stream) against the measured
           HBM copy bandwidth
cpu_baseline  the fp64 CPU oracle on the host's cores, bounded sample
variants   the other workloads, each timed the same way
Multi-GPU: one process per GPU (torchrun); each rank verifies its own batch
(weak scaling, no collective on the data path); barrier + max over ranks.
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORKLOAD = "dense_b64_g7_v128256"
METRIC = "verified positions/sec and achieved HBM GB/s (fraction of GB300 peak)"
UNIT = "positions/s"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0
KERNEL_SOURCES = ("rejection_sampling_gb300/csrc/sv_dense.cu",
                  "rejection_sampling_gb300/csrc/sv_common.cuh",
                  "rejection_sampling_gb300/csrc/sv_internal.h")
PATH_ENV = "SPEC_VERIFY_DENSE_KERNELS"  # split | fused: force one large-vocabulary dense path
TRAFFIC_PROFILE = os.path.join(ROOT, "profiles", "dense_b64_g7_v128256_ncu.txt")


# ---------------------------------------------------------------------------
# helpers shared by both arms
# ---------------------------------------------------------------------------
def dense_bytes(B, G, V, es):
    """Algorithmic bytes of one dense call: every logit read once."""
    return B * ((G + 1) * V + G * V) * es


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """Per-launch DRAM bytes from the committed ncu summary, if it was taken on
    the current kernel source; else None."""
    try:
        txt = open(TRAFFIC_PROFILE).read()
    except OSError:
        return None
    m_h = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]{16})", txt)
    m_t = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    if not (m_h and m_t) or m_h.group(1) != kernel_source_hash():
        return None
    return float(m_t.group(1))


def measured_peak():
    try:
        d = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def bench_config(B, G, V, ws):
    """The workload description both arms print (identical dicts)."""
    return {"workload": WORKLOAD, "B": B, "gamma": G, "V": V, "logits": "bf16",
            "global_batch_rows": B * ws, "parallelism": f"rows sharded over {ws} GPU(s)",
            "l2": "inputs larger than L2: two resident copies (2 x 246 MB) alternated"}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_timing(elapsed_s: float, units: float, group=None):
    """(max elapsed over ranks, sum of units over ranks); identity without a
    process group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return elapsed_s, units
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend(group) == "nccl" \
        else torch.device("cpu")
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    dist.all_reduce(u, op=dist.ReduceOp.SUM, group=group)
    return float(t.item()), float(u.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None, interval_ms: int = 100):
        self.samples = []
        self.proc = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               f"-lms={interval_ms}"]
        if gpu_id:
            cmd.insert(1, f"--id={gpu_id}")
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0: float, t1: float, timed0: float):
        win = [p for (t, p) in self.samples if t0 <= t <= t1]
        in_timed = sum(1 for (t, _) in self.samples if timed0 <= t <= t1)
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "samples_in_timed": 0}
        sm = [float(p[1]) for p in win if p[1].replace(".", "").isdigit()]
        smax = [float(p[2]) for p in win if p[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in win for i in range(4) if p[5 + i].lower() == "active"})
        pw = [float(p[3]) for p in win if re.match(r"^[0-9.]+$", p[3])]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "power_w_max": max(pw) if pw else None, "samples": len(win),
                "samples_in_timed": in_timed}


def gpu_uuid(dev_index: int):
    import torch
    try:
        u = str(torch.cuda.get_device_properties(dev_index).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def to_dev(a, dev):
    import numpy as np
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    if a.dtype == np.uint16:
        t = t.view(torch.bfloat16)
    return t.to(dev)


def time_prepared(calls, stream, iters):
    """Mean time per call (ms) of a rotating list of prepared calls, CUDA events
    on the launching stream, L2 defeated by rotating inputs larger than L2."""
    import torch
    for c in calls:
        c()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(iters):
        calls[i % len(calls)]()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / iters


def variant_lines(dev, stream, only=None):
    """Kernel time of the other workloads (each call timed back to back);
    `only`: the line names to run (all when None)."""
    import numpy as np
    import torch
    import rejection_sampling_gb300 as rs
    from rejection_sampling_gb300 import workloads as wl
    out = {}
    # (line name, workload, forced dense path or None)
    runs = [("dense_v32_g4", "dense_v32_g4", None), ("dense_v151936_g15", "dense_v151936_g15", None),
            ("dense_v151936_g15_two_kernel", "dense_v151936_g15", "split"),
            ("dense_b64_g7_v128256_single_pass", "dense_b64_g7_v128256", "fused"),
            ("sparse_b256_g15_k64", "sparse_b256_g15_k64", None),
            ("anyorder_b4096_w32_v33", "anyorder_b4096_w32_v33", None),
            ("greedy_b64_g7_v128256", "greedy_b64_g7_v128256", None),
            ("commit_b64_w4_v151936", "commit_b64_w4_v151936", None),
            ("support_b64_g7_v128256", "support_b64_g7_v128256", None),
            ("rounds_b4096_r4_d256_v27", "rounds_b4096_r4_d256_v27", None)]
    for name, wname, forced in runs:
        if only is not None and name not in only:
            continue
        d = wl.make(wname, seed=0)
        if forced:
            os.environ[PATH_ENV] = forced
        else:
            os.environ.pop(PATH_ENV, None)
        copies = 8  # rotate over copies so the inputs exceed L2 where they are small
        calls = []
        if d["kind"] == "dense":
            B, G, V = d["B"], d["gamma"], d["V"]
            es = 2 if d["dtype"] == "bf16" else 4
            nbytes = dense_bytes(B, G, V, es)
            positions = B * G
            copies = max(2, min(64, -(-300_000_000 // nbytes)))  # rotating copies > 2 x L2
            base = [to_dev(d[k], dev) for k in ("target", "draft", "draft_ids", "u_accept", "u_sample")]
            for c in range(copies):
                args = [t.clone() for t in base]
                o = rs.VerifyResult(torch.empty(B, dtype=torch.int32, device=dev),
                                    torch.empty(B, G + 1, dtype=torch.int32, device=dev), None, None)
                torch.cuda.synchronize()  # inputs built on the default stream; calls run on `stream`
                calls.append(rs.prepare_dense(*args, out=o, stream=stream))
        elif d["kind"] == "greedy":
            B, G, V = d["B"], d["gamma"], d["V"]
            nbytes = B * (G + 1) * V * (2 if d["dtype"] == "bf16" else 4)  # target logits only
            positions = B * G
            copies = 2  # 2 x 131 MB > L2
            base = [to_dev(d[k], dev) for k in ("target", "draft_ids")]
            for c in range(copies):
                args = [t.clone() for t in base]
                o = rs.VerifyResult(torch.empty(B, dtype=torch.int32, device=dev),
                                    torch.empty(B, G + 1, dtype=torch.int32, device=dev), None, None)
                torch.cuda.synchronize()  # inputs built on the default stream; calls run on `stream`
                calls.append(rs.prepare_greedy(*args, out=o, stream=stream))
        elif d["kind"] == "commit":
            B, W, V = d["B"], d["W"], d["V"]
            nmask = int(np.count_nonzero(d["masked"]))
            nbytes = nmask * V * (2 if d["dtype"] == "bf16" else 4)  # masked positions' logits
            positions = nmask
            copies = 4  # 4 x 78 MB > L2
            base = [to_dev(d[k], dev) for k in ("logits", "masked")]
            for c in range(copies):
                args = [t.clone() for t in base]
                o = rs.CommitResult(torch.empty(B, W, dtype=torch.int32, device=dev),
                                    torch.empty(B, W, dtype=torch.int32, device=dev), None)
                torch.cuda.synchronize()  # inputs built on the default stream; calls run on `stream`
                calls.append(rs.prepare_commit(*args, d["tau"], out=o, stream=stream))
        elif d["kind"] == "support":
            N, V, K = d["N"], d["V"], d["K"]
            nbytes = N * V * (2 if d["dtype"] == "bf16" else 4)
            positions = N
            copies = 2  # 2 x 246 MB > L2
            base = to_dev(d["logits"], dev)
            for c in range(copies):
                lg = base.clone()
                o = rs.SupportResult(torch.empty(N, K, dtype=torch.int32, device=dev),
                                     torch.empty(N, K, dtype=torch.float32, device=dev))
                torch.cuda.synchronize()  # inputs built on the default stream; calls run on `stream`
                calls.append(rs.prepare_support(lg, d["T"], K, d["top_p"], out=o, stream=stream))
        elif d["kind"] == "rounds":
            B, R, D, V = d["B"], d["R"], d["D"], d["V"]
            window = np.array([rs.spec_anyorder_window(D, int(i), d["dtau"]) for i in d["revealed"]],
                              np.int32)
            base = [to_dev(x, dev) for x in (d["target"], d["draft"], d["order"], d["revealed"], window,
                                             d["draft_tokens"], d["u_accept"], d["u_sample"])]
            copies = 2  # the rows a call reads are scattered; two copies alternate anyway
            for c in range(copies):
                args = [t.clone() for t in base]
                o = rs.RoundsResult(torch.full((B, D), -1, dtype=torch.int32, device=dev),
                                    torch.empty(B, dtype=torch.int32, device=dev),
                                    torch.empty(B, R, dtype=torch.int32, device=dev))
                torch.cuda.synchronize()  # inputs built on the default stream; calls run on `stream`
                calls.append(rs.prepare_rounds(*args, out=o, stream=stream))
            torch.cuda.synchronize()
            revealed = int((o.n_revealed - base[3]).sum())
            # every revealed position's target row (its round) and draft row is read once
            nbytes = 2 * revealed * V * (2 if d["dtype"] == "bf16" else 4)
            positions = revealed
        elif d["kind"] == "sparse":
            B, G, k = d["B"], d["gamma"], d["kt"]
            nbytes = B * ((G + 1) * k + G * k) * 8 + B * G * 8 + B * 4
            positions = B * G
            copies = max(2, min(64, -(-300_000_000 // nbytes)))  # rotating copies > 2 x L2
            base = [to_dev(d[x], dev) for x in ("tgt_ids", "tgt_probs", "drf_ids", "drf_probs",
                                                "draft_tokens", "u_accept", "u_sample")]
            for c in range(copies):
                args = [t.clone() for t in base]
                o = rs.VerifyResult(torch.empty(B, dtype=torch.int32, device=dev),
                                    torch.empty(B, G + 1, dtype=torch.int32, device=dev), None, None)
                torch.cuda.synchronize()  # inputs built on the default stream; calls run on `stream`
                calls.append(rs.prepare_sparse(*args, d["V"], out=o, stream=stream))
        else:
            B, D, W, V = d["B"], d["D"], d["W"], d["V"]
            nbytes = 2 * B * D * V * 4 + B * W * 8 + B * D * 4 + B * 4
            positions = B * W
            base = [to_dev(d[x], dev) for x in ("target", "draft", "order", "draft_tokens",
                                                "u_accept", "u_sample")]
            for c in range(copies):
                args = [t.clone() for t in base]
                tok = torch.full((B, D), -1, dtype=torch.int32, device=dev)
                torch.cuda.synchronize()  # inputs built on the default stream; calls run on `stream`
                calls.append(rs.prepare_anyorder(*args, tok, stream=stream))
        with torch.cuda.stream(stream):
            ms = time_prepared(calls, stream, 400)
        out[name] = {"us_per_call": round(ms * 1e3, 2),
                     "positions_per_s": positions / (ms * 1e-3),
                     "GBps": nbytes / (ms * 1e-3) / 1e9,
                     "bytes_per_call": nbytes}
        if d["kind"] in ("greedy", "commit", "support", "dense", "anyorder"):  # reads every logit once
            peak, _ = measured_peak()
            out[name]["frac_of_measured_hbm"] = out[name]["GBps"] / peak
        if forced:
            out[name]["dense_path"] = forced
        del calls
    os.environ.pop(PATH_ENV, None)
    torch.cuda.synchronize()
    return out


def cpu_baseline_leg(d, budget_s=10.0):
    """The oracle as it stands, threaded over rows on all host cores, on
    repeated full batches of the workload for about budget_s seconds."""
    import oracle
    oracle.build()
    cores = oracle.default_threads()
    B, G = d["B"], d["gamma"]
    t0 = time.perf_counter()
    reps = 0
    while True:
        oracle.verify_dense(d["target"], d["draft"], d["draft_ids"], d["u_accept"], d["u_sample"],
                            residual=False, nthreads=cores)
        reps += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": reps * B * G / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{reps} full batches of {WORKLOAD} ({B} rows x {G} drafts), "
                      f"{dt:.1f} s, rows split over {cores} threads"}


def run_ours(args):
    import numpy as np
    import torch
    import rejection_sampling_gb300 as rs
    from rejection_sampling_gb300 import workloads as wl

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    rs.build()
    rs.load()
    stream = torch.cuda.Stream(dev)

    d = wl.make(WORKLOAD, seed=args.seed + rank)
    B, G, V = d["B"], d["gamma"], d["V"]
    es = 2
    host = {k: d[k] for k in ("target", "draft", "draft_ids", "u_accept", "u_sample")}
    sets, outs = [], []
    base = [to_dev(host[k], dev) for k in ("target", "draft", "draft_ids", "u_accept", "u_sample")]
    for c in range(2):  # two resident copies: 2 x 246 MB > L2 (the reuse distance defeats it)
        sets.append([t.clone() for t in base] if c else base)
        outs.append(rs.VerifyResult(torch.empty(B, dtype=torch.int32, device=dev),
                                    torch.empty(B, G + 1, dtype=torch.int32, device=dev), None, None))
    torch.cuda.synchronize()  # the copies are built on the default stream; the calls run on `stream`
    calls = [rs.prepare_dense(*sets[c], out=outs[c], stream=stream) for c in range(2)]
    torch.cuda.synchronize()

    # warm-up, then a preheat window so the clock samples see the GPU under load
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            calls[i % 2]()
    torch.cuda.synchronize()
    sampler = ClockSampler(gpu_uuid(local)) if rank == 0 else None
    t_pre0 = time.time()
    with torch.cuda.stream(stream):
        while time.time() - t_pre0 < args.preheat_s:
            for i in range(50):
                calls[i % 2]()
            torch.cuda.synchronize()

    # timed region: exactly K steps, barrier + synchronize on both sides.  The
    # calls run back to back on one stream with events only at the two ends:
    # an event recorded between calls would sit between one call's row kernel
    # and the next call's statistics kernel and stop the latter from being
    # scheduled early (programmatic dependent launch), which a caller issuing
    # calls back to back does not pay.
    t_all0, t_all1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    t_timed0 = time.time()
    with torch.cuda.stream(stream):
        t_all0.record(stream)
        for i in range(args.steps):
            calls[i % 2]()
        t_all1.record(stream)
    torch.cuda.synchronize()
    barrier()
    t_timed1 = time.time()
    if sampler:
        time.sleep(0.15)
        sampler.stop()
    elapsed = t_all0.elapsed_time(t_all1) / 1e3
    kernel_ms = elapsed * 1e3 / args.steps  # mean duration of one call (both kernels)
    max_elapsed, total_pos = reduce_timing(elapsed, float(B * G * args.steps))
    value = total_pos / max_elapsed
    nbytes = dense_bytes(B, G, V, es)
    peak, peak_kind = measured_peak()
    achieved = nbytes / (kernel_ms * 1e-3) / 1e9
    rc = rs.check(dev, stream)
    if rc != rs.SV_OK:
        raise SystemExit(f"device status after timing: {rs.status_string(rc)}")

    # end to end through the C ABI with host buffers (pinned), rank-local
    e2e = None
    if not args.no_e2e:
        pin = {k: torch.from_numpy(np.ascontiguousarray(v)).pin_memory() for k, v in host.items()}
        pin["target"] = pin["target"].view(torch.bfloat16)
        pin["draft"] = pin["draft"].view(torch.bfloat16)
        dst = [pin[k].to(dev) for k in ("target", "draft", "draft_ids", "u_accept", "u_sample")]
        torch.cuda.synchronize()  # the validating call below runs on `stream`
        o = outs[0]
        call = rs.prepare_dense(*dst, out=o, stream=stream)
        h_n = torch.empty(B, dtype=torch.int32).pin_memory()
        h_tok = torch.empty(B, G + 1, dtype=torch.int32).pin_memory()
        keys = ("target", "draft", "draft_ids", "u_accept", "u_sample")
        h2d = sum(pin[k].numel() * pin[k].element_size() for k in keys)
        d2h = h_n.numel() * 4 + h_tok.numel() * 4
        n_e2e = max(3, min(args.steps, 50))

        def e2e_step():
            for k, t in zip(keys, dst):
                t.copy_(pin[k], non_blocking=True)
            call()
            h_n.copy_(o.n_accepted, non_blocking=True)
            h_tok.copy_(o.out_tokens, non_blocking=True)

        with torch.cuda.stream(stream):
            for _ in range(3):
                e2e_step()
            torch.cuda.synchronize()
            barrier()
            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            w0 = time.perf_counter()
            a0.record(stream)
            for _ in range(n_e2e):
                e2e_step()
            a1.record(stream)
            torch.cuda.synchronize()
            w1 = time.perf_counter()
        e_el, e_pos = reduce_timing(max(a0.elapsed_time(a1) / 1e3, w1 - w0),
                                    float(B * G * n_e2e))
        e2e = {"value": e_pos / e_el, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "steps": n_e2e}

    variants = None
    if rank == 0 and ws == 1 and not args.no_variants:
        variants = variant_lines(dev, stream)

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_leg(d, args.cpu_budget_s)

    if rank == 0:
        clocks = sampler.summary(t_pre0, t_timed1, t_timed0) if sampler else None
        traffic = profiled_traffic()
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": max_elapsed * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded; bf16 logits, fp32 arithmetic)",
            "config": bench_config(B, G, V, ws),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_kind": peak_kind,
                         "frac_of_nominal_8TBps": achieved / NOMINAL_HBM_GBS,
                         "traffic": traffic, "algorithmic_bytes_per_launch": nbytes,
                         "kernel": "dense_stats_kernel + dense_row_kernel (one call)", "mean_launch_us": kernel_ms * 1e3},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": 2 * args.steps,  # dense_stats_kernel + dense_row_kernel per call
            "clocks": clocks,
            "variants": variants,
            "kernel_source_sha256_16": kernel_source_hash(),
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# reference arm: the CPU oracle on the same workload
# ---------------------------------------------------------------------------
def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    from rejection_sampling_gb300 import workloads as wl
    oracle.build()
    d = wl.make(WORKLOAD, seed=args.seed)
    B, G = d["B"], d["gamma"]
    cores = oracle.default_threads()

    rows = B

    def step():
        oracle.verify_dense(d["target"][:rows], d["draft"][:rows], d["draft_ids"][:rows],
                            d["u_accept"][:rows], d["u_sample"][:rows], residual=False,
                            nthreads=cores)

    # bound the whole run to about two minutes: a step is the first `rows`
    # rows of the batch, fewer than B only when K full batches would not fit
    t0 = time.perf_counter()
    step()
    t_full = time.perf_counter() - t0
    budget_s = 120.0
    if t_full * (args.steps + args.warmup) > budget_s:
        rows = max(1, int(B * budget_s / (t_full * (args.steps + args.warmup))))
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    value = rows * G * args.steps / dt
    sample = (f"each step: the first {rows} of the {B} rows of {WORKLOAD} ({G} drafts each), "
              f"rows over {cores} threads")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)", "config": bench_config(B, G, d["V"], ws),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def run_calls_only(args):
    """Profiling driver: args.calls_only untimed calls of one workload (the
    headline by default; ``--workload NAME`` for any other named workload), no
    output beyond one status line (ncu's launch filters pick the kernels
    out)."""
    import torch
    import rejection_sampling_gb300 as rs
    from rejection_sampling_gb300 import workloads as wl
    rs.build()
    rs.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    name = args.workload or WORKLOAD
    d = wl.make(name, seed=args.seed)
    if d["kind"] == "greedy":
        t = [to_dev(d[k], dev) for k in ("target", "draft_ids")]
        fn = rs.spec_verify_greedy
    elif d["kind"] == "dense":
        t = [to_dev(d[k], dev) for k in ("target", "draft", "draft_ids", "u_accept", "u_sample")]
        fn = rs.spec_verify_dense
    elif d["kind"] == "commit":
        t = [to_dev(d[k], dev) for k in ("logits", "masked")] + [d["tau"]]
        fn = rs.spec_commit_confident
    elif d["kind"] == "support":
        t = [to_dev(d["logits"], dev), d["T"], d["K"], d["top_p"]]
        fn = rs.spec_support_topk
    elif d["kind"] == "rounds":
        import numpy as np
        window = np.array([rs.spec_anyorder_window(d["D"], int(i), d["dtau"]) for i in d["revealed"]],
                          np.int32)
        t = [to_dev(x, dev) for x in (d["target"], d["draft"], d["order"], d["revealed"], window,
                                      d["draft_tokens"], d["u_accept"], d["u_sample"])]
        fn = rs.spec_verify_anyorder_rounds
    elif d["kind"] == "sparse":
        t = [to_dev(d[x], dev) for x in ("tgt_ids", "tgt_probs", "drf_ids", "drf_probs",
                                         "draft_tokens", "u_accept", "u_sample")] + [d["V"]]
        fn = rs.spec_verify_sparse
    elif d["kind"] == "anyorder":
        t = [to_dev(d[x], dev) for x in ("target", "draft", "order", "draft_tokens", "u_accept",
                                         "u_sample")]
        fn = rs.spec_verify_anyorder
    else:
        raise SystemExit(f"--calls-only cannot drive workload {name}")
    for _ in range(args.calls_only):
        fn(*t)
    torch.cuda.synchronize()
    rc = rs.check(dev, torch.cuda.current_stream(dev))
    print(f"{args.calls_only} calls of {name}: {rs.status_string(rc)}")
    if rc != rs.SV_OK:
        raise SystemExit(1)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--preheat-s", dest="preheat_s", type=float, default=1.0)
    ap.add_argument("--cpu-budget-s", dest="cpu_budget_s", type=float, default=10.0)
    ap.add_argument("--no-e2e", dest="no_e2e", action="store_true")
    ap.add_argument("--no-variants", dest="no_variants", action="store_true")
    ap.add_argument("--no-cpu-baseline", dest="no_cpu_baseline", action="store_true")
    ap.add_argument("--calls-only", dest="calls_only", type=int, default=0,
                    help="profiling driver: N untimed calls on the headline workload")
    ap.add_argument("--workload", default=None,
                    help="with --calls-only: the workload to drive (default: the headline)")
    args = ap.parse_args(argv)
    if args.calls_only > 0:
        run_calls_only(args)
        return
    if args.impl == "reference":
        args.steps = 5 if args.steps is None else args.steps
        args.warmup = 1 if args.warmup is None else args.warmup
        run_reference(args)
    else:
        args.steps = 20000 if args.steps is None else args.steps  # about 1 s timed: several clock samples inside it
        args.warmup = 20 if args.warmup is None else max(3, args.warmup)
        run_ours(args)


if __name__ == "__main__":
    main()
