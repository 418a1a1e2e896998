#!/usr/bin/env python3
"""Benchmark of the fused GRPO + IcePop token-level loss (forward + backward).

One step = one call of ``rl_loss_forward_backward`` over one batch of the
chosen workload (per-response prep, the fused row kernel, two fixed-order
reductions), inputs resident in HBM. Prints ONE JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--case C] [--impl ours|reference]

Multi-GPU runs are replicas: every rank processes its own batch, no
collective on the data path (``scaling: weak``); the timed region is bracketed
by a barrier + synchronize and the maximum over ranks is reported.
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
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "response tokens/s & HBM GB/s (% of peak), fused logprob+IcePop loss fwd+bwd"
SIDE_BYTES_PER_TOKEN = 22  # target 4, logp_old 4, logp_infer 4, mask 1, logp 4, entropy 4, flags 1


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--case", default="3", choices=["0", "1", "2", "3", "4", "gae", "topk"],
                    help="0-3: the fused loss over logits; 4: the fused projection + loss; gae: skip-observation "
                         "GAE; topk: deterministic top-k")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--e2e-chunks", type=int, default=16,
                    help="loss cases 0-3: N > 0 = the host-input call rl_loss_forward_backward_from_host with N "
                         "logits row blocks, each computed as soon as it lands (the e2e default, 16); 0 = copy "
                         "every input first, then the device call")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU time of the oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-also", action="store_true",
                    help="the default loss line leaves out its `also` object (short runs of the fused projection, "
                         "GAE and top-k)")
    ap.add_argument("--prompts", type=int, default=0,
                    help="use only the first P prompts' responses (small profiling runs); 0 = the whole case")
    ap.add_argument("--max-len", type=int, default=0, help="cap every response length (small profiling runs)")
    ap.add_argument("--vocab", type=int, default=0, help="case 4: vocabulary override (small profiling runs)")
    ap.add_argument("--rows", type=int, default=0, help="topk: query rows override (small profiling runs)")
    ap.add_argument("--graph", action="store_true",
                    help="loss cases 0-3: capture one step in a CUDA graph and time its replays (the per-kernel "
                         "profile is then not taken; the roofline uses the whole step)")
    return ap.parse_args()


def emit(line: dict, args) -> None:
    """Print the bench line, or hand it to the caller that runs this workload as a secondary one."""
    sink = getattr(args, "collect", None)
    if sink is not None:
        sink.append(line)
    else:
        print(json.dumps(line), flush=True)


def secondary_lines(args) -> dict:
    """Short runs of the other workloads on the hot path (the fused projection, GAE and top-k), for the
    `also` object of the default line: each one's time, rate, roofline fraction and clocks."""
    import copy
    import torch
    runs = {"case4_fused_projection": ("4", 3, 2), "gae": ("gae", 50, 3), "topk": ("topk", 20, 3)}
    also = {}
    for name, (case, steps, warmup) in runs.items():
        a = copy.copy(args)
        a.case, a.steps, a.warmup, a.e2e_steps, a.no_cpu_baseline, a.collect = case, steps, warmup, 1, True, []
        a.prompts = a.max_len = a.vocab = a.rows = 0
        {"4": main_projection, "gae": main_gae, "topk": main_topk}[case](a)
        torch.cuda.empty_cache()
        if not a.collect:
            continue
        ln = a.collect[0]
        keep = {k: ln[k] for k in ("metric", "value", "unit", "ms_per_step", "steps", "warmup", "roofline", "clocks",
                                   "step_tensor", "roofline_forward", "gpu_launches", "device_status") if k in ln}
        keep["workload"] = ln["config"]["workload"]
        also[name] = keep
    return also


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def measured_peaks(key: str = "hbm_gbs"):
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    fallback = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d[key]), "measured"
    except Exception:
        return fallback[key], "fallback"


# the source files each profiled kernel is compiled from
KERNEL_SOURCES = {
    "row_loss": ["row_loss.cu", "ptx.cuh", "common.cuh"],
    "proj_gemm": ["proj_gemm.cu", "proj.cuh", "ptx.cuh", "tmap.cuh", "common.cuh"],
    "proj_bwd": ["proj_gemm.cu", "proj.cuh", "ptx.cuh", "tmap.cuh", "common.cuh"],
    "gae": ["gae.cu", "scan_select.cuh", "ptx.cuh", "tmap.cuh", "common.cuh"],
    "topk": ["topk.cu", "scan_select.cuh", "ptx.cuh", "common.cuh"],
}


def kernel_traffic(kernel: str, case_id):
    """Per-launch DRAM bytes of ``kernel`` from the committed ncu summary, or
    None when that summary was taken on another version of the kernel source.
    ``case_id``: a loss case number, or the name of a profile's workload."""
    name = f"{kernel}_case{case_id}.md" if isinstance(case_id, int) else f"{kernel}_{case_id}.md"
    path = os.path.join(ROOT, "profiles", name)
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_bytes = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    m_hash = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    if not (m_bytes and m_hash) or m_hash.group(1) != kernel_source_hash(kernel):
        return None
    return float(m_bytes.group(1))


def kernel_source_hash(kernel: str) -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "rl_post_loss_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel]:
        h.update(open(os.path.join(csrc, name), "rb").read())
    return h.hexdigest()


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "note": "nvidia-smi unavailable"}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "note": "no samples"}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[3][k].lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "power_w_max": max(r[2] for r in rows), "samples": len(rows), "reasons": reasons}


def max_over_ranks(x: float) -> float:
    """The maximum of a per-rank value over the process group (identity without one)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(tokens_per_step: int, steps: int, world: int, ms: float) -> float:
    """Whole-job tokens/s of `world` replicas, each running `steps` steps of
    `tokens_per_step` tokens, timed by the slowest rank (`ms`)."""
    return world * steps * tokens_per_step / (ms / 1e3)


def algorithmic_bytes(batch) -> float:
    es = 2 if batch.dtype == "bf16" else 4
    return float(batch.num_tokens) * (2.0 * batch.vocab * es + SIDE_BYTES_PER_TOKEN)


def oracle_sample_rate(batch, seconds: float):
    """The fp64 oracle (as it stands) over a bounded sample of rows: forward +
    backward (dL/dlogits into a fresh fp64 buffer). Returns tokens/s, cores,
    sample description."""
    import numpy as np
    import torch
    import oracle
    p = oracle.LossParams(group_size=batch.group, eps_low=batch.eps_low, eps_high=batch.eps_high,
                          beta=batch.beta, adv_eps=batch.adv_eps, adv_mode=batch.adv_mode)
    odt = oracle.BF16 if batch.dtype == "bf16" else oracle.F32

    def logits_rows_np(b, ids):
        idx = torch.as_tensor(np.asarray(ids, np.int64), device=b.logits.device)
        lg = b.logits.index_select(0, idx)[:, :b.vocab].contiguous().cpu()
        return lg.view(torch.int16).numpy().view(np.uint16) if lg.dtype == torch.bfloat16 else lg.numpy()

    a = {k: getattr(batch, k).cpu().numpy() for k in
         ("targets", "logp_old", "logp_infer", "mask", "cu_seqlens", "rewards_or_adv")}
    n, adv, w = oracle.seq_prep(a["cu_seqlens"], a["mask"], a["rewards_or_adv"], p)
    T = batch.num_tokens
    probe = np.arange(min(T, 32))
    z = logits_rows_np(batch, probe)
    t0 = time.perf_counter()
    oracle.rows(probe, z, odt, batch.vocab, a["targets"], a["logp_old"], a["logp_infer"], a["mask"],
                a["cu_seqlens"], adv, w, p, want_dz=True)
    per_row = (time.perf_counter() - t0) / len(probe)
    # bounded by the time budget and by a 2 GB fp64 dL/dlogits buffer
    nrows = int(max(32, min(T, seconds / max(per_row, 1e-9), 2e9 / (8.0 * batch.vocab))))
    ids = np.linspace(0, T - 1, nrows).astype(np.int64)
    z = logits_rows_np(batch, ids)
    done, reps = 0, 0
    t0 = time.perf_counter()
    while True:  # repeat the sample until the time budget is spent
        oracle.seq_prep(a["cu_seqlens"], a["mask"], a["rewards_or_adv"], p)
        oracle.rows(ids, z, odt, batch.vocab, a["targets"], a["logp_old"], a["logp_infer"], a["mask"],
                    a["cu_seqlens"], adv, w, p, want_dz=True)
        done += nrows
        reps += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    cores = int(os.environ.get("OMP_NUM_THREADS", len(os.sched_getaffinity(0))))
    return done / dt, cores, (f"{nrows} of {T} rows (evenly spaced) x {reps}, V={batch.vocab}, "
                              f"fp64 fwd+bwd, {dt:.1f} s")


def run_reference(args):
    """The oracle on the host cores, on bounded samples of the same workload."""
    rank, world, local = dist_env()
    if rank != 0:
        return 0
    import torch
    from rl_post_loss_gb300 import synthetic
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    batch = make_case_batch(args.case, args.prompts, dev, max_len=args.max_len)
    per_step = max(2.0, 150.0 / max(1, args.steps + args.warmup))
    rates = []
    desc, cores = "", 0
    for k in range(args.warmup + args.steps):
        rate, cores, desc = oracle_sample_rate(batch, per_step)
        if k >= args.warmup:
            rates.append(rate)
    value = statistics.mean(rates)
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "impl": "reference", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * batch.num_tokens / value,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(batch, args.case),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


L2_BYTES = 129e6


def make_case_batch(case_id: int, prompts: int, device, seed: int = 0, max_len: int = 0):
    from rl_post_loss_gb300 import synthetic
    lengths = None
    if prompts or max_len:
        c = synthetic.CASES[case_id]
        base = 20261202 + case_id + 1000 * seed
        lengths = synthetic.make_lengths(c, base)
        if prompts:
            lengths = lengths[:prompts * c["group"]]
        if max_len:
            lengths = [min(n, max_len) for n in lengths]
    return synthetic.make_batch(case_id, device, seed=seed, lengths=lengths)


def workload_config(batch, case_id):
    from rl_post_loss_gb300 import synthetic
    c = synthetic.CASES[case_id]
    return {"workload": f"case {case_id}: {c['name']}", "tokens": batch.num_tokens, "responses": batch.num_seqs,
            "group": batch.group, "vocab": batch.vocab, "logits_dtype": batch.dtype,
            "mask1_tokens": int(batch.mask.sum().item()), "beta": batch.beta,
            "eps": [batch.eps_low, batch.eps_high], "adv_mode": batch.adv_mode,
            "parallelism": "replicas",
            "l2": ("no flush: each step streams the whole logits and dlogits arrays (%.2f GB), larger than "
                   "the 129 MB L2" % (algorithmic_bytes(batch) / 1e9)) if algorithmic_bytes(batch) > 2 * L2_BYTES
            else "L2 flushed between steps (256 MB memset inside the timed region)"}


def main():
    args = parse_args()
    if args.case == "gae":
        return main_gae(args)
    if args.case == "topk":
        return main_topk(args)
    args.case = int(args.case)
    if args.impl == "reference":
        return run_reference(args)
    if args.case == 4:
        return main_projection(args)
    import torch
    import torch.distributed as dist
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    from rl_post_loss_gb300 import build as nvbuild
    from rl_post_loss_gb300 import capi, synthetic
    if not os.path.exists(nvbuild.LIB_PATH):
        if rank == 0:
            nvbuild.build()
        else:
            for _ in range(600):
                if os.path.exists(nvbuild.LIB_PATH):
                    break
                time.sleep(1)
    capi.load()
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    batch = make_case_batch(args.case, args.prompts, "cuda", seed=rank, max_len=args.max_len)
    rl = capi.handle_for_batch(batch)
    flush = None
    if algorithmic_bytes(batch) <= 2 * L2_BYTES:
        flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    out = capi.alloc_outputs(batch)
    stream = torch.cuda.current_stream()

    for _ in range(args.warmup):
        capi.run_batch(rl, batch, out)
    torch.cuda.synchronize()
    bits = rl.device_status()

    graph = None
    if args.graph:
        # one step captured once (the warm-up above did the per-device setup); replays launch nothing from the host
        graph = torch.cuda.CUDAGraph()
        l0 = rl.launch_count()
        with torch.cuda.graph(graph):
            capi.run_batch(rl, batch, out)
        launches_per_step = rl.launch_count() - l0
        torch.cuda.synchronize()
    else:
        rl.profile_start(args.steps)
    launches0 = rl.launch_count()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        start.record(stream)
        for _ in range(args.steps):
            if flush is not None:
                flush.zero_()
            if graph is not None:
                graph.replay()
            else:
                capi.run_batch(rl, batch, out)
        stop.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
    ms = start.elapsed_time(stop)
    if graph is not None:
        launches = launches_per_step * args.steps
        prof = {}
    else:
        launches = rl.launch_count() - launches0
        prof = rl.profile_read()
    ms = max_over_ranks(ms)

    T = batch.num_tokens
    value = replica_throughput(T, args.steps, world, ms)
    if graph is not None:  # no per-kernel times: the whole step stands in for the row kernel
        row_avg_ms = ms / args.steps
    else:
        row_n, row_ms = prof["row_loss"]
        row_avg_ms = row_ms / max(1, row_n)
    bytes_per_launch = algorithmic_bytes(batch)
    peak, peak_kind = measured_peaks()
    achieved = bytes_per_launch / (row_avg_ms / 1e3) / 1e9
    traffic = kernel_traffic("row_loss", args.case)

    # end to end through the public API: pinned host inputs -> device, call, loss -> host. With
    # --e2e-chunks N > 0 (the default) the host-input entry point copies the logits in N row blocks
    # and computes each block as soon as it lands; with 0 every input is copied first and the device
    # call follows.
    dev_in = capi.batch_inputs(batch)
    host = {}
    for k, t in dev_in.items():
        host[k] = torch.empty_strided(t.shape, t.stride(), dtype=t.dtype, pin_memory=True)
        host[k].copy_(t)
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    loss_host = torch.empty(1, dtype=torch.float64).pin_memory()
    e_start, e_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # the host link as this run sees it: the same copies alone, as many times as the e2e steps
    # (one untimed first), just before them
    for k in range(args.e2e_steps + 1):
        if k == 1:
            torch.cuda.synchronize()
            e_start.record(stream)
        for name, t in host.items():
            dev_in[name].copy_(t, non_blocking=True)
    e_stop.record(stream)
    torch.cuda.synchronize()
    copy_ms = e_start.elapsed_time(e_stop) / args.e2e_steps
    for k in range(args.e2e_steps + 1):
        if k == 1:
            torch.cuda.synchronize()
            e_start.record(stream)
        if args.e2e_chunks > 0:
            capi.run_batch_from_host(rl, host, dev_in, out, num_chunks=args.e2e_chunks)
        else:
            for name, t in host.items():
                dev_in[name].copy_(t, non_blocking=True)
            capi.run_batch(rl, batch, out)
        loss_host.copy_(out["loss_f64"], non_blocking=True)
        stream.synchronize()
        _ = float(loss_host[0])
    e_stop.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e_start.elapsed_time(e_stop) / args.e2e_steps
    e2e_ms = max_over_ranks(e2e_ms)
    e2e_value = replica_throughput(T, 1, world, e2e_ms)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, cores, desc = oracle_sample_rate(batch, args.cpu_seconds)
        cpu = {"value": rate, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": desc}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
                "config": dict(workload_config(batch, args.case), **({"cuda_graph": True} if graph is not None else {})),
                "hbm_gbs": world * args.steps * bytes_per_launch / (ms / 1e3) / 1e9,
                "roofline": {"bound": "hbm", "kernel": "row_loss" if graph is None else "whole step (CUDA graph)",
                             "achieved": achieved, "peak": peak,
                             "peak_kind": f"{peak_kind} copy bandwidth", "unit": "GB/s", "frac": achieved / peak,
                             "traffic": traffic, "algorithmic_bytes_per_launch": bytes_per_launch,
                             "avg_launch_ms": row_avg_ms},
                "kernel_ms": {k: v[1] / max(1, v[0]) for k, v in prof.items()},
                "clocks": clocks.summary(),
                "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                        "d2h_bytes_per_step": 8, "ms_per_step": e2e_ms,
                        "h2d_gbs_in_step": h2d / (e2e_ms / 1e3) / 1e9,
                        "copy_alone_ms": copy_ms, "h2d_gbs_copy_alone": h2d / (copy_ms / 1e3) / 1e9,
                        "outputs": "the loss (8 B) comes back to the host; dlogits stays on the device for "
                                   "the caller's backward",
                        "call": ("rl_loss_forward_backward_from_host, %d logits blocks" % args.e2e_chunks
                                 if args.e2e_chunks > 0 else "copies, then rl_loss_forward_backward")},
                "gpu_launches": launches, "device_status": capi.status_bits_to_names(bits),
                "cpu_baseline": cpu}
    if world == 1 and not args.no_also and not args.graph and not (args.prompts or args.max_len or args.vocab):
        # the other workloads of the hot path, measured in the same run (after this workload's buffers go)
        del batch, out, host, dev_in, rl
        torch.cuda.empty_cache()
        line["also"] = secondary_lines(args)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def projection_sample_rate(pb, seconds: float):
    """The fp64 oracle of the fused path on a bounded sample of rows: the
    projection of each row (a float64 matmul), its loss terms, dL/dz and
    dL/dh. Returns tokens/s, cores, sample description."""
    import numpy as np
    import oracle
    b = pb.batch
    H = pb.hidden_dim
    p = oracle.LossParams(group_size=b.group, eps_low=b.eps_low, eps_high=b.eps_high, beta=b.beta,
                          adv_eps=b.adv_eps, adv_mode=b.adv_mode)
    a = {k: getattr(b, k).cpu().numpy() for k in
         ("targets", "logp_old", "logp_infer", "mask", "cu_seqlens", "rewards_or_adv")}
    bits = lambda t: t.contiguous().cpu().view(__import__("torch").int16).numpy().view(np.uint16)
    w64 = oracle.bf16_bits_to_f64(bits(pb.w[:, :H]))
    hb = bits(pb.hidden[:, :H])
    n, adv, w = oracle.seq_prep(a["cu_seqlens"], a["mask"], a["rewards_or_adv"], p)
    T = b.num_tokens
    done, reps, k = 0, 0, 16
    t0 = time.perf_counter()
    while True:
        ids = (np.arange(k) * 997 + reps * 131) % T
        oracle.projection_rows(ids, hb, None, a["targets"], a["logp_old"], a["logp_infer"], a["mask"],
                               a["cu_seqlens"], adv, w, p, want_dh=True, w64=w64)
        done += k
        reps += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    cores = int(os.environ.get("OMP_NUM_THREADS", len(os.sched_getaffinity(0))))
    return done / dt, cores, (f"{done} rows of {T} (16 per batch, spread), fp64 projection + loss + dL/dz + dL/dh "
                              f"per row (dL/dW excluded), {dt:.1f} s")


def main_projection(args):
    """Case 4: the fused sequence-chunked projection + loss, forward and backward."""
    import torch
    import torch.distributed as dist
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    from rl_post_loss_gb300 import build as nvbuild
    from rl_post_loss_gb300 import capi, synthetic
    if not os.path.exists(nvbuild.LIB_PATH):
        if rank == 0:
            nvbuild.build()
        else:
            for _ in range(600):
                if os.path.exists(nvbuild.LIB_PATH):
                    break
                time.sleep(1)
    capi.load()
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    over = {}
    if args.prompts:
        over["prompts"] = args.prompts
    if args.vocab:
        over["vocab"] = args.vocab
    pb = synthetic.make_projection_batch("cuda", seed=rank, **over)
    b = pb.batch
    rl = capi.projection_handle(pb)
    out = capi.alloc_projection_outputs(pb)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        capi.run_projection(rl, pb, out)
    torch.cuda.synchronize()
    bits = rl.device_status()
    rl.profile_start(args.steps)
    launches0 = rl.launch_count()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        start.record(stream)
        for _ in range(args.steps):
            capi.run_projection(rl, pb, out)
        stop.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
    ms = start.elapsed_time(stop)
    launches = rl.launch_count() - launches0
    prof = rl.profile_read()
    ms = max_over_ranks(ms)
    T, H, V = b.num_tokens, pb.hidden_dim, b.vocab
    value = replica_throughput(T, args.steps, world, ms)
    flops_alg = 6.0 * T * V * H  # projection, dL/dh and dL/dW GEMMs
    g_n, g_ms = prof["proj_gemm"]
    gemm_flops = 2.0 * T * V * H / max(1, g_n // args.steps)  # per launch (one chunk)
    peak, peak_kind = measured_peaks("bf16_tflops_sustained")
    achieved = gemm_flops / (g_ms / max(1, g_n) / 1e3) / 1e12
    b_n, b_ms = prof["proj_bwd"]
    bwd_flops = 4.0 * T * V * H / max(1, b_n // args.steps)  # dL/dh and dL/dW of one chunk per launch
    bwd_achieved = bwd_flops / (b_ms / max(1, b_n) / 1e3) / 1e12
    step_tflops = flops_alg / (ms / args.steps / 1e3) / 1e12

    host = {"hidden": pb.hidden.cpu().pin_memory(), "w": pb.w.cpu().pin_memory()}
    host.update({k: getattr(b, k).cpu().pin_memory() for k in
                 ("targets", "logp_old", "logp_infer", "mask", "cu_seqlens", "rewards_or_adv")})
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    loss_host = torch.empty(1, dtype=torch.float64).pin_memory()
    e_start, e_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for k in range(args.e2e_steps + 1):
        if k == 1:
            torch.cuda.synchronize()
            e_start.record(stream)
        pb.hidden.copy_(host["hidden"], non_blocking=True)
        pb.w.copy_(host["w"], non_blocking=True)
        for name in ("targets", "logp_old", "logp_infer", "mask", "cu_seqlens", "rewards_or_adv"):
            getattr(b, name).copy_(host[name], non_blocking=True)
        capi.run_projection(rl, pb, out)
        loss_host.copy_(out["loss_f64"], non_blocking=True)
        stream.synchronize()
        _ = float(loss_host[0])
    e_stop.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e_start.elapsed_time(e_stop) / args.e2e_steps
    e2e_ms = max_over_ranks(e2e_ms)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, cores, desc = projection_sample_rate(pb, args.cpu_seconds)
        cpu = {"value": rate, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": desc}
    if rank == 0:
        c = synthetic.PROJ_CASE
        line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": {"workload": f"case 4: {c['name']}", "tokens": T, "responses": b.num_seqs,
                           "group": b.group, "vocab": V, "hidden": H, "chunk_tokens": pb.chunk,
                           "mask1_tokens": int(b.mask.sum().item()), "parallelism": "replicas",
                           "l2": "no flush: each step streams W (1.9 GB) once per chunk and writes a 1.24-GB bf16 "
                                 "chunk twice per chunk, far larger than the 129 MB L2"},
                "roofline": {"bound": "tensor", "kernel": "proj_bwd", "achieved": bwd_achieved, "peak": peak,
                             "peak_kind": f"{peak_kind} sustained cuBLAS bf16 TFLOP/s", "unit": "TFLOP/s",
                             "frac": bwd_achieved / peak, "traffic": kernel_traffic("proj_bwd", 4),
                             "algorithmic_flops_per_launch": bwd_flops, "avg_launch_ms": b_ms / max(1, b_n)},
                "roofline_forward": {"bound": "tensor", "kernel": "proj_gemm", "achieved": achieved, "peak": peak,
                                     "unit": "TFLOP/s", "frac": achieved / peak,
                                     "traffic": kernel_traffic("proj_gemm", 4),
                                     "algorithmic_flops_per_launch": gemm_flops, "avg_launch_ms": g_ms / max(1, g_n)},
                "step_tensor": {"algorithmic_tflops": step_tflops, "frac": step_tflops / peak,
                                "executed_flops_per_step": flops_alg, "note": "6 N V H per step"},
                "kernel_ms": {k: v[1] / args.steps for k, v in prof.items() if v[0]},
                "clocks": clocks.summary(),
                "e2e": {"value": replica_throughput(T, 1, world, e2e_ms), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                        "d2h_bytes_per_step": 8, "ms_per_step": e2e_ms},
                "gpu_launches": launches, "device_status": capi.status_bits_to_names(bits), "cpu_baseline": cpu}
        emit(line, args)
    if world > 1:
        dist.destroy_process_group()
    return 0


def _device_setup():
    import torch
    import torch.distributed as dist
    rank, world, local = dist_env()
    if torch.cuda.is_available():
        torch.cuda.set_device(local)
    from rl_post_loss_gb300 import build as nvbuild
    if not os.path.exists(nvbuild.LIB_PATH):
        if rank == 0:
            nvbuild.build()
        else:
            for _ in range(600):
                if os.path.exists(nvbuild.LIB_PATH):
                    break
                time.sleep(1)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return rank, world, local


def _timed(fn, steps: int, warmup: int, local: int, flush=None):
    """Device time (ms) of `steps` calls of fn on the current stream, max over ranks."""
    import torch
    import torch.distributed as dist
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        if dist.is_initialized():
            dist.barrier()
        torch.cuda.synchronize()
        start.record(stream)
        for _ in range(steps):
            if flush is not None:
                flush.zero_()
            fn()
        stop.record(stream)
        torch.cuda.synchronize()
        if dist.is_initialized():
            dist.barrier()
    return max_over_ranks(start.elapsed_time(stop)), clocks.summary()


def main_gae(args):
    """Skip-observation GAE with the cross-trajectory discount over a CompactionRL-sized batch."""
    import numpy as np
    import torch
    if args.impl == "reference":
        from rl_post_loss_gb300 import synthetic
        rank, world, local = dist_env()
        if rank != 0:
            return 0
        gb = synthetic.make_gae_batch("cpu")
        per_step = max(2.0, 150.0 / max(1, args.steps + args.warmup))
        rates = []
        desc, cores = "", 1
        for i in range(args.warmup + args.steps):
            rate, cores, desc = _gae_oracle_rate(gb, per_step)
            if i >= args.warmup:
                rates.append(rate)
        config = {"workload": "gae: " + synthetic.GAE_CASE["name"], "tokens": gb.num_tokens,
                  "segments": int(gb.cu_seqlens.shape[0]) - 1, "gamma": gb.gamma, "lambda": gb.lam,
                  "parallelism": "replicas"}
        print(json.dumps(_reference_line(GAE_METRIC, "tokens/s", statistics.mean(rates), desc, cores, config, args,
                                         world, gb.num_tokens)), flush=True)
        return 0
    rank, world, local = _device_setup()
    from rl_post_loss_gb300 import capi, synthetic
    capi.load()
    gb = synthetic.make_gae_batch("cuda", seed=rank)
    T, S = gb.num_tokens, int(gb.cu_seqlens.shape[0]) - 1
    adv = torch.empty(T, dtype=torch.float32, device="cuda")
    run = lambda: capi.gae(gb.rewards, gb.values, gb.mask, gb.cu_seqlens, gb.gamma, gb.lam, True,
                           rollout_ids=gb.rollout_ids, advantages=adv)
    ms, clocks = _timed(run, args.steps, args.warmup, local)
    value = replica_throughput(T, args.steps, world, ms)
    bytes_per_token = 4 + 4 + 1 + 4  # rewards, values, mask in; advantages out
    peak, kind = measured_peaks()
    achieved = T * bytes_per_token / (ms / args.steps / 1e3) / 1e9
    # e2e: host inputs -> device, GAE, advantages -> host
    host = {k: getattr(gb, k).cpu().pin_memory() for k in ("rewards", "values", "mask", "cu_seqlens", "rollout_ids")}
    out_host = torch.empty(T, dtype=torch.float32).pin_memory()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for k in range(args.e2e_steps + 1):
        if k == 1:
            torch.cuda.synchronize()
            e0.record(stream)
        for name, t in host.items():
            getattr(gb, name).copy_(t, non_blocking=True)
        run()
        out_host.copy_(adv, non_blocking=True)
        stream.synchronize()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.e2e_steps)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, cores, desc = _gae_oracle_rate(gb, args.cpu_seconds)
        cpu = {"value": rate, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": desc}
    if rank == 0:
        line = {"metric": GAE_METRIC,
                "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f32", "data": "synthetic",
                "config": {"workload": "gae: " + synthetic.GAE_CASE["name"], "tokens": T, "segments": S,
                           "gamma": gb.gamma, "lambda": gb.lam, "parallelism": "replicas",
                           "l2": "no flush: each step reads %.0f MB and writes %.0f MB, more than the 129 MB L2"
                                 % (T * 9 / 1e6, T * 4 / 1e6)},
                "roofline": {"bound": "hbm", "kernel": "gae", "achieved": achieved, "peak": peak,
                             "peak_kind": f"{kind} copy bandwidth", "unit": "GB/s", "frac": achieved / peak,
                             "traffic": kernel_traffic("gae", "256x65536"), "algorithmic_bytes_per_launch": T * bytes_per_token,
                             "avg_launch_ms": ms / args.steps},
                "clocks": clocks,
                "e2e": {"value": replica_throughput(T, 1, world, e2e_ms), "unit": "tokens/s",
                        "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in host.values()),
                        "d2h_bytes_per_step": T * 4, "ms_per_step": e2e_ms},
                "gpu_launches": args.steps, "cpu_baseline": cpu}
        emit(line, args)
    return 0


def _gae_oracle_rate(gb, seconds: float):
    """The oracle's GAE (sequential fp64 recursion, one core) on the whole batch, repeated."""
    import oracle
    npb = {k: getattr(gb, k).cpu().numpy() for k in ("rewards", "values", "mask", "cu_seqlens", "rollout_ids")}
    done, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < seconds or done == 0:
        oracle.gae(npb["cu_seqlens"], npb["rewards"], npb["values"], npb["mask"], gb.gamma, gb.lam, True,
                   npb["rollout_ids"])
        done += gb.num_tokens
    dt = time.perf_counter() - t0
    return done / dt, 1, f"the whole batch x {done // gb.num_tokens}, fp64 sequential recursion, {dt:.1f} s"


def _topk_oracle_rate(b, seconds: float):
    """The oracle's top-k (a stable sort per row, one core) on evenly spaced rows, repeated."""
    import numpy as np
    from oracle import topk as otopk
    s = b.scores.cpu().numpy() if b.scores.device.type == "cpu" else None
    lengths = b.lengths.cpu().numpy()
    rows = np.linspace(0, b.rows - 1, 16).astype(int)
    host_rows = {int(q): (s[q] if s is not None else b.scores[q].cpu().numpy())[:int(lengths[q])] for q in rows}
    done, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < seconds or done == 0:
        for q in rows:
            otopk.topk_row(host_rows[int(q)], b.k)
            done += 1
    dt = time.perf_counter() - t0
    return done / dt, 1, f"{done} rows ({len(rows)} evenly spaced rows, repeated), stable sort per row, {dt:.1f} s"


def _reference_line(metric, unit, value, desc, cores, config, args, world, per_step_units):
    return {"metric": metric, "value": value, "unit": unit, "impl": "reference", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * per_step_units / value,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config,
            "cpu_baseline": {"value": value, "unit": unit, "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


TOPK_METRIC = "query rows/s, deterministic DSA-indexer top-k (k=2048)"
GAE_METRIC = "response tokens/s, skip-observation GAE with cross-trajectory discount"


def main_topk(args):
    """Deterministic top-k (k = 2048) over DSA indexer scores of a 202,752-token context."""
    import torch
    from rl_post_loss_gb300 import synthetic
    rank, world, local = dist_env() if args.impl == "reference" else _device_setup()
    if args.impl == "reference":
        if rank != 0:
            return 0
        b = synthetic.make_topk_batch("cuda" if torch.cuda.is_available() else "cpu")
        per_step = max(2.0, 150.0 / max(1, args.steps + args.warmup))
        rates = []
        desc, cores = "", 1
        for i in range(args.warmup + args.steps):
            rate, cores, desc = _topk_oracle_rate(b, per_step)
            if i >= args.warmup:
                rates.append(rate)
        print(json.dumps(_reference_line(TOPK_METRIC, "rows/s", statistics.mean(rates), desc, cores,
                                         _topk_config(b), args, world, b.rows)), flush=True)
        return 0
    from rl_post_loss_gb300 import capi
    capi.load()
    b = synthetic.make_topk_batch("cuda", seed=rank, **({"rows": args.rows} if args.rows else {}))
    out_idx = torch.empty((b.rows, b.k), dtype=torch.int32, device="cuda")
    out_val = torch.empty((b.rows, b.k), dtype=torch.float32, device="cuda")
    run = lambda: capi.topk(b.scores, b.k, lengths=b.lengths, out_idx=out_idx, out_val=out_val)
    ms, clocks = _timed(run, args.steps, args.warmup, local)
    value = replica_throughput(b.rows, args.steps, world, ms)
    n_sum = int(b.lengths.sum().item())
    bytes_per_launch = 4 * n_sum + 4 * b.rows + 8 * b.rows * b.k  # scores read, lengths, positions + scores written
    peak, kind = measured_peaks()
    achieved = bytes_per_launch / (ms / args.steps / 1e3) / 1e9
    # e2e: pinned host scores -> device, top-k, positions -> host
    host = b.scores.cpu().pin_memory()
    idx_host = torch.empty((b.rows, b.k), dtype=torch.int32).pin_memory()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i in range(args.e2e_steps + 1):
        if i == 1:
            torch.cuda.synchronize()
            e0.record(stream)
        b.scores.copy_(host, non_blocking=True)
        run()
        idx_host.copy_(out_idx, non_blocking=True)
        stream.synchronize()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.e2e_steps)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, cores, desc = _topk_oracle_rate(b, args.cpu_seconds)
        cpu = {"value": rate, "unit": "rows/s", "cores": cores, "kind": "oracle", "sample": desc}
    if rank == 0:
        line = {"metric": TOPK_METRIC, "value": value, "unit": "rows/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": _topk_config(b),
                "roofline": {"bound": "hbm", "kernel": "topk", "achieved": achieved, "peak": peak,
                             "peak_kind": f"{kind} copy bandwidth", "unit": "GB/s", "frac": achieved / peak,
                             "traffic": kernel_traffic("topk", "4096x202752"), "algorithmic_bytes_per_launch": bytes_per_launch,
                             "avg_launch_ms": ms / args.steps},
                "clocks": clocks,
                "e2e": {"value": replica_throughput(b.rows, 1, world, e2e_ms), "unit": "rows/s",
                        "h2d_bytes_per_step": host.numel() * 4, "d2h_bytes_per_step": b.rows * b.k * 4,
                        "ms_per_step": e2e_ms},
                "gpu_launches": args.steps, "cpu_baseline": cpu}
        emit(line, args)
    return 0


def _topk_config(b):
    from rl_post_loss_gb300 import synthetic
    return {"workload": "topk: " + synthetic.TOPK_CASE["name"], "rows": b.rows, "ld": b.ld, "k": b.k,
            "keys_per_launch": int(b.lengths.sum().item()), "order": "score desc, position asc",
            "parallelism": "replicas",
            "l2": "no flush: each step reads %.2f GB of scores, more than the 129 MB L2" % (
                4 * int(b.lengths.sum().item()) / 1e9)}


if __name__ == "__main__":
    sys.exit(main())
