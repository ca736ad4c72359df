#!/usr/bin/env python
"""Benchmark of batched speculative-decoding verification on GB300.

One step = one spec_verify call over one batch of the workload: every verified position of every
row gets its temperature softmaxes, accept test, residual or bonus draw and the row's emit.

Default workload: B=1024 rows, ragged draft lengths 1..8 (gamma_max 8), V=256000 bf16 logits, 10% of
rows greedy -- the largest of the workloads, and the one that exercises every step of the path. The
logits (4.9 GB read per step) are far larger than the 129 MB L2, so no flush is needed between steps.

Prints one JSON line (rank 0). Under torchrun every rank verifies its own replica of the batch on
its own GPU (rows are independent: weak scaling, no data-path collective); the step time is the max
over ranks.

  python bench.py [--steps K] [--warmup W] [--workload N] [--impl {gb300,reference}]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time
from pathlib import Path

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

METRIC = "verified positions/sec (B·(γ+1)) and logits HBM GB/s vs 8 TB/s roofline"
UNIT = "positions/s"
NOMINAL_HBM_GBS = 8000.0
DEFAULT_WORKLOAD = 5
TRAFFIC_FILE = ROOT / "profiles" / "sv_stream_kernel_traffic.json"
KERNEL_SOURCES = ["sv_stream.cu", "sv_common.cuh", "sv_api.cu"]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", type=int, default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--rows", type=int, default=0, help="use only the first N rows (profiling runs)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="single-core oracle seconds the CPU baseline's row sample is sized for")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the kernel timings of workloads 3 and 4 after the headline")
    ap.add_argument("--onehot", action="store_true",
                    help="one-hot drafts (greedy drafter): time spec_verify_onehot, no draft logits")
    ap.add_argument("--filter", action="store_true",
                    help="per-row top-k / top-p filtering of p and q before the test: time "
                         "spec_verify_filtered on the workload with seeded top_k in {off, 20, 50, 100} "
                         "and top_p in {off, 0.9, 0.95}")
    ap.add_argument("--rollback", action="store_true",
                    help="KV-cache rollback after a round: B=1024 rows of the default workload's draft "
                         "lengths, 320 KB cache entries (80 layers of K and V, 8 heads x 128, bf16)")
    ap.add_argument("--tree", action="store_true",
                    help="greedy tree verification: Medusa-shaped trees (top 2 of 4 heads, 31 nodes), "
                         "B=256, V=128256 bf16, timed through spec_verify_tree_greedy")
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def rank_seed(base_seed, rank):
    """The workload seed of one rank: every rank verifies its own independent batch (weak scaling,
    the rows shard across GPUs with no exchange)."""
    return base_seed + 1000 * rank


def job_totals(ms, units, device=None):
    """Whole-job figures of a run over every rank of the process group: the slowest rank's
    milliseconds (each timed region ends at a barrier that waits for it) and the units all ranks
    processed (ragged batches give each rank its own count). One rank: the inputs themselves."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(ms), float(units)
    slowest = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    done = torch.tensor([float(units)], dtype=torch.float64, device=device)
    dist.all_reduce(slowest, op=dist.ReduceOp.MAX)
    dist.all_reduce(done, op=dist.ReduceOp.SUM)
    return float(slowest.item()), float(done.item())


def kernel_source_hash():
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        h.update((ROOT / "speculative_decoding_verification_55_gb300" / "csrc" / name).read_bytes())
    return h.hexdigest()[:16]


def measured_peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clocks and throttle reasons while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def workload_for(args, rank):
    from workloads import get_config, make_workload
    import dataclasses
    cfg = get_config(args.workload)
    seed = rank_seed(cfg.seed, rank)
    if args.rows:
        cfg = dataclasses.replace(cfg, B=min(args.rows, cfg.B))
    return cfg, make_workload(cfg, seed=seed, backend="torch", device="cuda")


# ------------------------------------------------------------------------------------------------
# CPU baseline: the fp64 oracle, as it stands, on a bounded sample of the same workload
# ------------------------------------------------------------------------------------------------

def _oracle(w, onehot, filt=None):
    from oracle.spec_verify_oracle import oracle_verify, oracle_verify_onehot
    if onehot:
        return oracle_verify_onehot(w.target_logits, w.draft_tokens, w.draft_len, w.temperature,
                                    w.uniforms)
    top_k, top_p = filt if filt is not None else (None, None)
    return oracle_verify(w.target_logits, w.draft_logits, w.draft_tokens, w.draft_len,
                         w.temperature, w.uniforms, top_k=top_k, top_p=top_p)


def oracle_pool(cfg_key, seconds, seed=12345, onehot=False, filt=False):
    """Rows of the workload drawn on the host (numpy backend), as many as the oracle verifies in
    about `seconds` of single-thread CPU time (calibrated on 8 rows). Input generation is untimed."""
    import dataclasses

    import numpy as np

    from workloads import get_config, make_workload
    cfg = get_config(cfg_key)
    from workloads import filter_params
    probe = make_workload(dataclasses.replace(cfg, B=8), seed=seed, backend="numpy")
    t0 = time.perf_counter()
    _oracle(probe, onehot, filter_params(8, seed) if filt else None)
    t8 = time.perf_counter() - t0
    rows = int(max(8, min(cfg.B, round(seconds / max(t8, 1e-6) * 8 / 8) * 8)))
    w = make_workload(dataclasses.replace(cfg, B=rows), seed=seed + 1, backend="numpy")
    if filt:
        w.filters = filter_params(rows, seed + 1)
    return w, int(np.sum(w.draft_len.astype(np.int64) + 1))


def oracle_run(w, onehot=False, threads=1):
    """Wall seconds of one oracle pass over the pool's rows (the plain spec_verify rule with
    threads > 1: rows in parallel threads)."""
    t0 = time.perf_counter()
    if threads > 1 and not onehot and getattr(w, "filters", None) is None:
        from oracle.spec_verify_oracle import oracle_verify_rows
        oracle_verify_rows(lambda b: (w.target_logits[b], w.draft_logits[b]), w.draft_tokens,
                           w.draft_len, w.temperature, w.uniforms, w.G, w.V, range(w.B),
                           threads=threads)
    else:
        _oracle(w, onehot, getattr(w, "filters", None))
    return time.perf_counter() - t0


def oracle_sample_rate(cfg_key, seconds, onehot=False, filt=False):
    """Oracle throughput (positions/s) on a bounded host-drawn sample of the workload."""
    w, pos = oracle_pool(cfg_key, seconds, onehot=onehot, filt=filt)
    secs = oracle_run(w, onehot)
    return pos / secs, w.B, pos, secs


def oracle_threads():
    """Host cores this process may run on (the all-cores oracle figure uses that many threads)."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def cpu_leg(w, gpu_out, seconds, seed=4242):
    """The oracle, as it stands, on a bounded sample of the timed batch's own rows: timed on one
    core and on all cores (a thread per core, rows in parallel), then compared with the GPU's
    outputs for those rows under the margin rule (outside every timed region).

    gpu_out: (out_tokens, out_num, out_alpha) numpy arrays of the timed batch. Returns
    (cpu_baseline dict, parity dict)."""
    import numpy as np

    sys.path.insert(0, str(ROOT / "tests"))
    from _parity import compare
    from oracle.spec_verify_oracle import oracle_verify_rows
    rng = np.random.default_rng(seed)
    order = rng.permutation(w.B)
    host = {}

    def source(b):
        return host[b]

    def run(rows, threads, diagnostics=False):
        return oracle_verify_rows(source, w.draft_tokens, w.draft_len, w.temperature, w.uniforms,
                                  w.G, w.V, rows, threads=threads, diagnostics=diagnostics)

    probe = [int(b) for b in order[:4]]
    for b in probe:
        host[b] = w.host_rows(b)
    t0 = time.perf_counter()
    run(probe, 1)
    per_row = (time.perf_counter() - t0) / len(probe)
    n = int(max(4, min(w.B, round(seconds / max(per_row, 1e-6)))))
    rows = [int(b) for b in order[:n]]
    for b in rows:
        if b not in host:
            host[b] = w.host_rows(b)
    pos = int(np.sum(w.draft_len[rows].astype(np.int64) + 1))
    t0 = time.perf_counter()
    run(rows, 1)
    t1 = time.perf_counter() - t0
    cores = oracle_threads()
    t0 = time.perf_counter()
    run(rows, cores)
    tn = time.perf_counter() - t0
    o = run(rows, cores, diagnostics=True)
    tok, num, alpha = gpu_out
    rep = compare(o, tok, num, alpha, None, None, w.draft_tokens, w.draft_len, rows=rows)
    sample = (f"{n} rows ({pos} positions) of the timed batch, seeded sample, copied back from the "
              f"device; fp64 oracle, rows in parallel threads")
    cpu = {"value": pos / tn, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample,
           "seconds": tn,
           "single_core": {"value": pos / t1, "unit": UNIT, "cores": 1, "seconds": t1}}
    parity = dict(rep.as_dict(), sample=f"the same {n} rows", rule="tokens and accept counts "
                  "bit-exact outside the 1e-5 margin; alpha within 1e-5")
    return cpu, parity


def time_workload(sv, key, steps, warmup, dev, flush_bytes=0):
    """Kernel time of one spec_verify call on workload `key` (inputs resident in HBM), CUDA events
    on the launching stream. With flush_bytes, a buffer that large is written between steps (L2
    flushed) and each step is timed on its own; the mean step time is returned."""
    import torch
    from workloads import get_config, make_workload
    cfg = get_config(key)
    w = make_workload(cfg, backend="torch", device=dev)
    t = w.device_tensors(dev)
    B, G, V = w.B, w.G, w.V
    dcode = sv.SV_DTYPE_BF16 if cfg.dtype == "bf16" else sv.SV_DTYPE_F32
    stream = torch.cuda.current_stream(dev)
    ws = sv.workspace_for(B, G, V, dcode, dev, stream)
    out = (torch.empty((B, G + 1), dtype=torch.int32, device=dev),
           torch.empty((B,), dtype=torch.int32, device=dev),
           torch.empty((B, G), dtype=torch.float32, device=dev))

    def step():
        sv.spec_verify(t["target_logits"], t["draft_logits"], t["draft_tokens"], t["draft_len"],
                       t["temperature"], t["uniforms"], *out, ws, stream)

    flush = torch.empty(flush_bytes, dtype=torch.uint8, device=dev) if flush_bytes else None
    for _ in range(max(warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    times = []
    if flush is not None:
        for _ in range(steps):
            flush.fill_(1)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            step()
            b.record(stream)
            torch.cuda.synchronize(dev)
            times.append(a.elapsed_time(b))
        ms = sum(times) / len(times)
    else:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            step()
        b.record(stream)
        torch.cuda.synchronize(dev)
        ms = a.elapsed_time(b) / steps
    algo = w.algorithmic_bytes()
    gbs = algo / (ms * 1e-3) / 1e9
    peak, peak_kind = measured_peaks()
    res = {"workload": cfg.name, "ms_per_step": ms, "steps": steps,
           "positions_per_s": w.positions() / (ms * 1e-3), "algorithmic_bytes_per_step": algo,
           "achieved_gbs": gbs, "frac": gbs / peak, "peak": peak, "peak_kind": peak_kind,
           "frac_of_8tbs": gbs / NOMINAL_HBM_GBS,
           "l2": (f"{flush_bytes >> 20} MB written between steps" if flush_bytes
                  else "inputs larger than L2 (no flush)")}
    del t, w, out, flush
    torch.cuda.empty_cache()
    return res


def workload_name(cfg, args):
    return cfg.name + ("_onehot_drafts" if args.onehot else "") + ("_topk_topp" if args.filter else "")


def run_reference_tree(args):
    """The oracle arm of --tree: oracle_tree_greedy on 16 host-drawn trees per step."""
    from oracle.spec_verify_oracle import oracle_tree_greedy
    hz, ht, hp = tree_inputs(16, 99, "numpy")
    N = hz.shape[1]
    for _ in range(args.warmup):
        oracle_tree_greedy(hz, ht, hp)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_tree_greedy(hz, ht, hp)
    total = time.perf_counter() - t0
    value = 16 * N * args.steps / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"tree_greedy_b{TREE_B}_n{N}_v{TREE_V}_bf16", "sample_trees_per_step": 16},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": "16 trees of the workload drawn on the host per step, single-thread "
                                   "fp64 oracle"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ.setdefault(v, "1")
    if args.tree:
        return run_reference_tree(args)
    from workloads import get_config
    cfg = get_config(args.workload)
    per_step = 1.5      # seconds of single-thread oracle work per step
    w, pos = oracle_pool(args.workload, per_step, onehot=args.onehot, filt=args.filter)
    threads = 1 if (args.onehot or args.filter) else oracle_threads()
    for _ in range(args.warmup):
        oracle_run(w, args.onehot, threads)
    total = 0.0
    for _ in range(args.steps):
        total += oracle_run(w, args.onehot, threads)
    value = pos * args.steps / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": workload_name(cfg, args), "B": cfg.B,
                   "gamma_max": cfg.gamma_max, "V": cfg.V,
                   "logits": cfg.dtype, "sample_rows_per_step": w.B,
                   "sample_positions_per_step": pos},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"{w.B} rows ({pos} positions) of the workload drawn on the host "
                                   f"per step, fp64 oracle on {threads} thread(s), rows in "
                                   f"parallel"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------------------------------------
# GPU arm
# ------------------------------------------------------------------------------------------------

def run_gpu(args):
    import torch
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    import speculative_decoding_verification_55_gb300 as sv
    sv.build_library()

    cfg, w = workload_for(args, rank)
    t = w.device_tensors(dev)
    B, G, V = w.B, w.G, w.V
    dcode = sv.SV_DTYPE_BF16 if cfg.dtype == "bf16" else sv.SV_DTYPE_F32
    stream = torch.cuda.current_stream(dev)
    # --filter: the workspace with room for the kept lists (spec_verify_filtered_workspace_size)
    ws = sv.workspace_for(B, G, V, dcode, dev, stream, filtered=args.filter)
    out_tokens = torch.empty((B, G + 1), dtype=torch.int32, device=dev)
    out_num = torch.empty((B,), dtype=torch.int32, device=dev)
    out_alpha = torch.empty((B, G), dtype=torch.float32, device=dev)

    if args.onehot:                  # one-hot drafts: no draft logits exist
        del t["draft_logits"]
    if args.filter:                  # per-row top-k / top-p, part of the step's inputs
        from workloads import filter_params
        fk, fp = filter_params(B, rank_seed(cfg.seed, rank))
        t["top_k"] = torch.from_numpy(fk).to(dev)
        t["top_p"] = torch.from_numpy(fp).to(dev)

    def call(inp):
        if args.filter:
            sv.spec_verify_filtered(inp["target_logits"], inp["draft_logits"], inp["draft_tokens"],
                                    inp["draft_len"], inp["temperature"], inp["top_k"],
                                    inp["top_p"], inp["uniforms"], out_tokens, out_num, out_alpha,
                                    None, None, ws, stream)
        elif args.onehot:
            sv.spec_verify_onehot(inp["target_logits"], inp["draft_tokens"], inp["draft_len"],
                                  inp["temperature"], inp["uniforms"], out_tokens, out_num,
                                  out_alpha, None, None, ws, stream)
        else:
            sv.spec_verify(inp["target_logits"], inp["draft_logits"], inp["draft_tokens"],
                           inp["draft_len"], inp["temperature"], inp["uniforms"], out_tokens,
                           out_num, out_alpha, ws, stream)

    def step():
        call(t)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    barrier()
    ms_total = ev0.elapsed_time(ev1)
    clock_info = clocks.stop()
    positions = w.positions()
    ms_step, positions_all = job_totals(ms_total / args.steps, positions, dev)
    value = positions_all / (ms_step * 1e-3)
    algo_bytes = w.algorithmic_bytes(onehot=args.onehot)
    achieved_gbs = algo_bytes / (ms_step * 1e-3) / 1e9
    peak, peak_kind = measured_peaks()

    traffic = None
    if TRAFFIC_FILE.exists():
        tr = json.loads(TRAFFIC_FILE.read_text())
        if tr.get("kernel_source_hash") == kernel_source_hash() and tr.get("workload") == cfg.name \
                and not args.onehot and not args.filter:
            traffic = tr["bytes_per_full_launch"]

    # ---- end to end: pinned host inputs -> device, the call, outputs -> pinned host ----
    e2e = None
    if not args.no_e2e:
        host = {k: v.cpu().pin_memory() for k, v in t.items()}
        h_tok = torch.empty((B, G + 1), dtype=torch.int32).pin_memory()
        h_num = torch.empty((B,), dtype=torch.int32).pin_memory()
        h_alpha = torch.empty((B, G), dtype=torch.float32).pin_memory()
        bo = sum(v.numel() * v.element_size() for v in (h_tok, h_num, h_alpha))
        if args.filter or args.onehot:
            # every input tensor copied in whole, then the device call
            dev_in = {k: torch.empty_like(v) for k, v in t.items()}
            bi = sum(v.numel() * v.element_size() for v in host.values())
            e2e_path = "every input copied in whole, then the device call"

            def e2e_step():
                for k in host:
                    dev_in[k].copy_(host[k], non_blocking=True)
                call(dev_in)
                h_tok.copy_(out_tokens, non_blocking=True)
                h_num.copy_(out_num, non_blocking=True)
                h_alpha.copy_(out_alpha, non_blocking=True)
        else:
            # the host-buffer entry point: only the logit rows the rule reads are copied in
            dev_in = torch.empty(sv.spec_verify_staging_size(B, G, V, dcode), dtype=torch.uint8,
                                 device=dev)
            bi = sv.spec_verify_staged_h2d_bytes(host["draft_len"], host["temperature"], B, G, V,
                                                 dcode)
            e2e_path = "spec_verify_staged: host buffers, only the rows the rule reads copied in"

            def e2e_step():
                sv.spec_verify_staged(host["target_logits"], host["draft_logits"],
                                      host["draft_tokens"], host["draft_len"],
                                      host["temperature"], host["uniforms"], h_tok, h_num,
                                      h_alpha, dev_in, ws, stream)

        for _ in range(2):
            e2e_step()
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        n_e2e = max(1, min(args.steps, 5))
        e0.record(stream)
        for _ in range(n_e2e):
            e2e_step()
        e1.record(stream)
        barrier()
        ms_e2e, _ = job_totals(e0.elapsed_time(e1) / n_e2e, positions, dev)
        e2e = {"value": positions_all / (ms_e2e * 1e-3), "unit": UNIT,
               "h2d_bytes_per_step": int(bi), "d2h_bytes_per_step": int(bo),
               "ms_per_step": ms_e2e, "steps": n_e2e, "path": e2e_path}
        # The host link's own rate, a plain page-locked copy of 1 GiB (median of 3), and the floor it
        # sets for this step's host-to-device bytes.
        link_h = torch.empty(1 << 30, dtype=torch.uint8).pin_memory()
        link_d = torch.empty(1 << 30, dtype=torch.uint8, device=dev)
        link_ms = []
        for _ in range(4):
            a, b2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            link_d.copy_(link_h, non_blocking=True)
            b2.record(stream)
            torch.cuda.synchronize(dev)
            link_ms.append(a.elapsed_time(b2))
        link_gbs = (1 << 30) / (sorted(link_ms[1:])[1] * 1e-3) / 1e9
        e2e["host_link_gbs"] = link_gbs
        e2e["host_link_floor_ms"] = bi / (link_gbs * 1e9) * 1e3
        del host, dev_in, link_h, link_d

    cpu = parity = None
    if rank == 0 and world == 1 and not args.no_cpu:
        if args.onehot or args.filter:
            rate, rows, pos, secs = oracle_sample_rate(args.workload, args.cpu_seconds,
                                                       args.onehot, args.filter)
            cpu = {"value": rate, "unit": UNIT, "cores": 1, "kind": "oracle",
                   "sample": f"{rows} rows ({pos} positions) of the workload drawn on the host, "
                             f"{secs:.1f} s of single-thread fp64 oracle work"}
        else:
            step()                   # the timed batch's outputs, once more, for the comparison
            torch.cuda.synchronize(dev)
            gpu_out = (out_tokens.cpu().numpy(), out_num.cpu().numpy(), out_alpha.cpu().numpy())
            cpu, parity = cpu_leg(w, gpu_out, args.cpu_seconds)

    per_config = None
    if rank == 0 and world == 1 and not (args.onehot or args.filter or args.rows or args.no_per_config):
        del t
        torch.cuda.empty_cache()
        per_config = {}
        for key, flush in ((3, 256 << 20), (4, 0)):
            if key != args.workload:
                per_config[f"workload_{key}"] = time_workload(sv, key, args.steps, args.warmup, dev,
                                                              flush)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": cfg.dtype, "data": "synthetic",
            "config": {"workload": workload_name(cfg, args), "B": B,
                       "gamma_max": G, "V": V, "logits": cfg.dtype,
                       "greedy_rows": int((w.temperature == 0).sum()),
                       "positions_per_gpu": positions, "positions_all_gpus": int(positions_all),
                       "padded_positions_per_gpu": B * (G + 1),
                       "algorithmic_bytes_per_step": algo_bytes,
                       "l2": "inputs larger than L2 (no flush)", "parallelism": f"replicas x{world}"},
            # --filter: the threshold kernel, the list kernel, then the masked streaming kernel
            # (three launches a step; the step's time is the roofline's)
            "gpu_launches": args.steps * (3 if args.filter else 1),
            "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": peak, "unit": "GB/s",
                         "frac": achieved_gbs / peak, "peak_kind": peak_kind,
                         "frac_of_8tbs": achieved_gbs / NOMINAL_HBM_GBS, "traffic": traffic,
                         "kernel": ("sv_threshold_kernel + sv_listed_kernel + masked "
                                    if args.filter else "")
                         + "sv_stream_kernel" + ("<bf16>" if cfg.dtype == "bf16" else "<f32>")},
            "clocks": clock_info,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "parity": parity,
            "per_config": per_config,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


# ------------------------------------------------------------------------------------------------
# Tree verification (--tree)
# ------------------------------------------------------------------------------------------------

TREE_B, TREE_TOPK, TREE_HEADS, TREE_V = 256, 2, 4, 128256


def tree_parents():
    """The page's Medusa tree: the root, then the top-k candidates of each head under every node of
    the previous level (parents before children)."""
    import numpy as np
    parents, level = [-1], [0]
    for _ in range(TREE_HEADS):
        new = []
        for par in level:
            for _ in range(TREE_TOPK):
                new.append(len(parents))
                parents.append(par)
        level = new
    return np.array(parents, np.int32)


def tree_inputs(B, seed, backend):
    """Target logits at every node (N(0, 2.5^2) plus the Zipf bias of the V=128256 workload) and node
    tokens that equal the target's argmax at their parent with probability 0.7 (else uniform)."""
    import numpy as np
    par = tree_parents()
    N = len(par)
    if backend == "numpy":
        rng = np.random.default_rng(seed)
        bias = -1.1 * np.log1p(rng.permutation(TREE_V)).astype(np.float32)
        zt = (rng.standard_normal((B, N, TREE_V), dtype=np.float32) * 2.5 + bias)
        from workloads import bf16_round
        zt = bf16_round(zt)
        g = zt.argmax(-1)
        tok = np.where(rng.random((B, N)) < 0.7, g[:, np.maximum(par, 0)],
                       rng.integers(0, TREE_V, (B, N))).astype(np.int32)
        return zt, tok, np.tile(par, (B, 1))
    import torch
    gen = torch.Generator(device="cuda").manual_seed(seed)
    bias = -1.1 * torch.log1p(torch.randperm(TREE_V, device="cuda", generator=gen).float())
    zt = (torch.randn((B, N, TREE_V), device="cuda", generator=gen) * 2.5 + bias).to(torch.bfloat16)
    g = zt.float().argmax(-1)
    pidx = torch.from_numpy(np.maximum(par, 0)).cuda().long()
    rnd = torch.randint(0, TREE_V, (B, N), device="cuda", generator=gen)
    keep = torch.rand((B, N), device="cuda", generator=gen) < 0.7
    tok = torch.where(keep, g[:, pidx], rnd).to(torch.int32).contiguous()
    return zt, tok, torch.from_numpy(np.tile(par, (B, 1))).cuda()


def run_tree(args):
    import numpy as np
    import torch
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    import speculative_decoding_verification_55_gb300 as sv
    sv.build_library()
    B = min(args.rows, TREE_B) if args.rows else TREE_B
    zt, tok, par = tree_inputs(B, rank_seed(7, rank), "torch")
    N = zt.shape[1]
    stream = torch.cuda.current_stream(dev)
    ws = sv.workspace_for(B, N - 1, TREE_V, sv.SV_DTYPE_BF16, dev, stream)
    outs = [torch.empty((B, N), dtype=torch.int32, device=dev), torch.empty((B,), dtype=torch.int32, device=dev),
            torch.empty((B, N + 1), dtype=torch.int32, device=dev), torch.empty((B, N), dtype=torch.int32, device=dev)]

    def call(z, t, p):
        sv.spec_verify_tree_greedy(z, t, p, None, outs[0], outs[1], outs[2], outs[3], ws, stream)

    for _ in range(max(args.warmup, 3)):
        call(zt, tok, par)
    torch.cuda.synchronize(dev)

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        call(zt, tok, par)
    ev1.record(stream)
    barrier()
    clock_info = clocks.stop()
    nodes = B * N
    ms_step, nodes_all = job_totals(ev0.elapsed_time(ev1) / args.steps, nodes, dev)
    algo = B * N * TREE_V * 2 + B * N * 8 + B * (N + N + 1 + N + 1) * 4
    achieved = algo / (ms_step * 1e-3) / 1e9
    peak, peak_kind = measured_peaks()

    e2e = None
    if not args.no_e2e:
        host = [x.cpu().pin_memory() for x in (zt, tok, par)]
        dev_in = [torch.empty_like(x) for x in (zt, tok, par)]
        h_out = [torch.empty_like(o, device="cpu").pin_memory() for o in outs]
        bi = sum(x.numel() * x.element_size() for x in host)
        bo = sum(x.numel() * x.element_size() for x in h_out)

        def e2e_step():
            for d_, h_ in zip(dev_in, host):
                d_.copy_(h_, non_blocking=True)
            call(*dev_in)
            for h_, o_ in zip(h_out, outs):
                h_.copy_(o_, non_blocking=True)

        for _ in range(2):
            e2e_step()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n_e2e = max(1, min(args.steps, 5))
        e0.record(stream)
        for _ in range(n_e2e):
            e2e_step()
        e1.record(stream)
        barrier()
        ms_e2e, _ = job_totals(e0.elapsed_time(e1) / n_e2e, nodes, dev)
        e2e = {"value": nodes_all / (ms_e2e * 1e-3), "unit": UNIT, "h2d_bytes_per_step": int(bi),
               "d2h_bytes_per_step": int(bo), "ms_per_step": ms_e2e, "steps": n_e2e}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        from oracle.spec_verify_oracle import oracle_tree_greedy
        hz, ht, hp = tree_inputs(16, 99, "numpy")
        t0 = time.perf_counter()
        oracle_tree_greedy(hz, ht, hp)
        secs = time.perf_counter() - t0
        cpu = {"value": 16 * N / secs, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"16 trees of the workload drawn on the host, {secs:.1f} s of single-thread "
                         f"fp64 oracle work"}
    if rank == 0:
        line = {
            "metric": METRIC, "value": nodes_all / (ms_step * 1e-3), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": f"tree_greedy_b{B}_n{N}_v{TREE_V}_bf16", "B": B, "nodes": N,
                       "V": TREE_V, "tree": f"top {TREE_TOPK} of {TREE_HEADS} heads",
                       "positions_per_gpu": nodes, "algorithmic_bytes_per_step": algo,
                       "l2": "inputs larger than L2 (no flush)", "parallelism": f"replicas x{world}"},
            "gpu_launches": args.steps,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_kind": peak_kind,
                         "frac_of_8tbs": achieved / NOMINAL_HBM_GBS, "traffic": None,
                         "kernel": "sv_stream_kernel<bf16>"},
            "clocks": clock_info, "e2e": e2e, "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


# ------------------------------------------------------------------------------------------------
# KV-cache rollback (--rollback)
# ------------------------------------------------------------------------------------------------

RB_ENTRY = 80 * 2 * 8 * 128 * 2       # bytes of one token's cache entry: 80 layers of K and V
RB_L = 16                              # entries per row: the prefix (2..6) plus gamma + 1 (<= 9)


def rollback_inputs(seed):
    """Row lengths of the default workload (gamma_b 1..8), prefixes of 2..6 entries, accept counts
    drawn with alpha = 0.7 per position (k = first failure), 10% row errors."""
    import numpy as np
    from workloads import get_config
    from workloads.generate import _row_params
    cfg = get_config(DEFAULT_WORKLOAD)
    rng = np.random.default_rng(seed)
    g = np.asarray(_row_params(cfg, cfg.seed)[0])
    B = len(g)
    n = rng.integers(2, 7, B)
    k = np.minimum(rng.geometric(0.3, B) - 1, g)
    e = (k + 1).astype(np.int64)
    e[rng.random(B) < 0.1] = -1
    return n.astype(np.int32), g.astype(np.int32), e.astype(np.int32), (n + g).astype(np.int32)


def run_rollback(args):
    import numpy as np
    import torch
    from oracle.spec_verify_oracle import kv_rollback
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    import speculative_decoding_verification_55_gb300 as sv
    sv.build_library()
    n, g, e, d = rollback_inputs(5)
    B, G = len(n), int(g.max())
    ti = lambda a: torch.as_tensor(a, device=dev)
    n_t, g_t, e_t, d_t = ti(n), ti(g), ti(e), ti(d)
    tl = torch.empty(B, dtype=torch.int32, device=dev)
    dl = torch.empty(B, dtype=torch.int32, device=dev)
    cache = torch.ones((B, RB_L, RB_ENTRY), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        sv.spec_verify_kv_rollback(n_t, g_t, e_t, d_t, tl, dl, cache=cache, gamma_max=G, stream=stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    times = []
    clocks = ClockSampler(0)
    clocks.start()
    time.sleep(0.3)
    for _ in range(args.steps):
        flush.zero_()                  # the dropped entries are not in L2 when the step starts
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        step()
        b.record(stream)
        torch.cuda.synchronize(dev)
        times.append(a.elapsed_time(b))
    clock_info = clocks.stop()
    ms = float(np.median(times))
    _, _, dropped = kv_rollback(n, g, e, d, G)
    zero_bytes = sum(max(0, min(hi, RB_L) - max(lo, 0)) for lo, hi in dropped) * RB_ENTRY
    algo = zero_bytes + B * 6 * 4
    achieved = algo / (ms * 1e-3) / 1e9
    peak, peak_kind = measured_peaks()
    want_t, want_d, _ = kv_rollback(n, g, e, d, G)
    ok = np.array_equal(tl.cpu().numpy(), want_t) and np.array_equal(dl.cpu().numpy(), want_d)
    line = {
        "metric": "KV-cache rows rolled back per second and bytes zeroed (GB/s)", "value": B / (ms * 1e-3),
        "unit": "rows/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8",
        "data": "synthetic",
        "config": {"workload": f"kv_rollback_b{B}_entry{RB_ENTRY}", "B": B, "entries_per_row": RB_L,
                   "entry_bytes": RB_ENTRY, "bytes_zeroed_per_step": zero_bytes,
                   "algorithmic_bytes_per_step": algo, "l2": "256 MB written between steps",
                   "lengths_match_oracle": ok},
        "gpu_launches": args.steps,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "frac_of_8tbs": achieved / NOMINAL_HBM_GBS, "traffic": None,
                     "kernel": "sv_rollback_kernel"},
        "clocks": clock_info, "e2e": None, "cpu_baseline": None,
    }
    print(json.dumps(line), flush=True)
    return 0 if ok else 1


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    if args.tree:
        return run_tree(args)
    if args.rollback:
        return run_rollback(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
