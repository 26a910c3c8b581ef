#!/usr/bin/env python3
"""Benchmark of the token-sparse MLA forward (one JSON line on stdout).

Default workload: the bf16 decode batch -- 32 sequences x 16384 cached tokens
in a paged cache (block 64, random block table), one query token per sequence,
h = 8 heads, top-k = 2048 distinct valid slots per token.  A step is one
sparse_mla_fwd call over the whole batch.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

L2: each step uses the next of R independently drawn input sets (own cache,
indices and queries); R is chosen so that R x gathered bytes >= 2 x L2, so a
step never finds its rows in L2 from the previous steps.

--impl reference times the CPU oracle (fp64, OpenMP) on the host cores on the
same workload, a bounded number of tokens per step.
--workload dcp_merge times sparse_mla_merge instead: the combine of 4 split-list
partial results per row at the fp8 batch's shape (T = 32768, h = 8); --workload
v_up times sparse_mla_v_up (T = 32768, h = 8, v_head_dim 128); --workload topk times
sparse_mla_topk (the prefill chunk's 16384 causal rows over 32768 positions, k = 2048);
--workload masked_dense times the masked dense route (scatter of the lists into a bit mask,
then masked MHA) on a 4096-token GLM-5 prefill chunk that is the whole request.
Multi-GPU (torchrun): every rank runs its own replica of the workload (the
path shards by query token with no exchange), weak scaling.
"""

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time
from pathlib import Path

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

import torch  # noqa: E402

from workloads import (config_by_name, gathered_bytes, make_merge_parts, make_v_up_weights,  # noqa: E402
                       make_workload, pad_heads)

METRIC = "query-tokens/s and gathered-KV HBM GB/s (fraction of roofline) at topk=2048"
UNIT = "query-tokens/s"
L2_BYTES_DEFAULT = 129 * 1024 * 1024
CSRC = ROOT / "token_sparse_mla_gb300" / "csrc"


def kernel_source_hash() -> str:
    """Hash of every kernel source; an ncu traffic figure is used only for the same sources."""
    h = hashlib.sha256()
    for f in sorted(list(CSRC.glob("*.cuh")) + list(CSRC.glob("*.cu"))):
        h.update(f.name.encode())
        h.update(f.read_bytes())
    return h.hexdigest()[:16]


def kernel_name(h: int) -> str:
    """The kernel a launch with h heads runs (8/16: warp-MMA kernel; 32/64: tcgen05 kernel)."""
    return "sparse_mla_fwd_small_kernel" if h <= 16 else "sparse_mla_fwd_tc_kernel"


def flops_per_entry(h: int) -> int:
    """Dense work per valid list entry: h heads x (576 QK + 512 PV) multiply-adds."""
    return 2 * h * (576 + 512)


def measured_peaks() -> dict:
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def ncu_traffic(workload: str, h: int, pad: bool):
    """Per-launch DRAM bytes from the committed ncu summary, if it is for this kernel source."""
    p = ROOT / "profiles" / "ncu_traffic.json"
    if not p.exists():
        return None
    try:
        d = json.loads(p.read_text())
    except ValueError:
        return None
    if d.get("kernel_source_hash") != kernel_source_hash():
        return None
    key = f"{workload}/h{h}{'/pad64' if pad else ''}"
    e = d.get("entries", {}).get(key)
    return None if e is None else float(e["dram_bytes_per_launch"])


class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        self.t0 = time.time()

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self) -> dict:
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        dist.init_process_group(backend=backend)
        return dist.get_rank(), world, int(os.environ.get("LOCAL_RANK", "0"))
    return 0, 1, 0


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Max of a host float over all ranks (1 rank: itself)."""
    if world <= 1:
        return float(x)
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def oracle_rate(w, budget_s: float, max_tokens_per_call: int = 32):
    """Time the oracle on the host cores over tokens of workload w, for about budget_s seconds."""
    import oracle
    oracle.build()
    threads = oracle.max_threads()
    toks = list(range(min(w.T, max_tokens_per_call)))
    done, elapsed, calls = 0, 0.0, 0
    while elapsed < budget_s or calls == 0:
        t0 = time.perf_counter()
        oracle.sparse_mla_fwd(w.q, w.kv, w.indices, w.scale, kv_format=w.kv_format, tokens=toks)
        elapsed += time.perf_counter() - t0
        done += len(toks)
        calls += 1
    return done / elapsed, threads, done, elapsed


def run_reference(args, rank, world):
    if rank != 0:
        return
    name = args.workload
    w = make_workload(name, h=args.h)
    if args.pad:
        w.q = pad_heads(w.q, 64)
    import oracle
    oracle.build()
    threads = oracle.max_threads()
    # calibrate one token, then size each step so the whole run stays within ~2 minutes
    t0 = time.perf_counter()
    oracle.sparse_mla_fwd(w.q, w.kv, w.indices, w.scale, kv_format=w.kv_format, tokens=[0])
    t_tok = max(time.perf_counter() - t0, 1e-4)
    per_step = max(1, min(w.T, int(120.0 / (args.steps + args.warmup) / t_tok)))
    toks = [i % w.T for i in range(per_step)]
    for _ in range(args.warmup):
        oracle.sparse_mla_fwd(w.q, w.kv, w.indices, w.scale, kv_format=w.kv_format, tokens=toks[:1])
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.sparse_mla_fwd(w.q, w.kv, w.indices, w.scale, kv_format=w.kv_format, tokens=toks)
    el = time.perf_counter() - t0
    value = per_step * args.steps / el
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": workload_config(w, args, splits=None, rot=1),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"{per_step} query tokens of the workload per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(w, args, splits, rot, ctas=None):
    cfg = w.cfg
    launch = getattr(args, "launch", "eager")
    return {"workload": cfg.name, "T": w.T, "h": int(w.q.shape[1]), "h_real": w.h,
            "launch": "CUDA graph of consecutive steps" if launch == "graph" else "eager launches",
            "padded_to_64": bool(args.pad), "topk": w.topk, "kv_format": cfg.kv_format,
            "num_slots": w.num_slots, "block_size": 64, "splits": splits, "ctas": ctas,
            "l2": f"rotating {rot} independently drawn input sets (cache, indices, q); "
                  f"{rot} x gathered bytes >= 2 x L2"}


def gpu_busy_wait(stream, us: float = 200.0):
    """Keep the GPU busy for about `us` microseconds on `stream` (torch's spin kernel), so the
    launches queued behind it by the host start back to back when it ends: a timed window that
    opens right after it measures the device, not the host's launch latency."""
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(us * 2000))


def median_of_windows(replay, steps_per_replay: int, stream, n_windows: int = 10, min_window_ms: float = 1.0):
    """Median over n_windows CUDA-event windows of the time per step; each window replays
    enough graphs to last at least min_window_ms.  Returns (ms per step, replays per window)."""
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    gpu_busy_wait(stream)
    ev0.record(stream)
    with torch.cuda.stream(stream):
        replay()
    ev1.record(stream)
    ev1.synchronize()
    est = max(ev0.elapsed_time(ev1), 1e-3)
    k = max(1, math.ceil(min_window_ms / est))
    times = []
    for _ in range(n_windows):
        gpu_busy_wait(stream, min(2000.0, 200.0 + 20.0 * k))
        ev0.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(k):
                replay()
        ev1.record(stream)
        ev1.synchronize()
        times.append(ev0.elapsed_time(ev1))
    return statistics.median(times) / (k * steps_per_replay), k


def forward_graph(q, kv, idx, scale, out, lse, kv_format, stream, n_steps):
    """A CUDA graph of n_steps forward calls on the same buffers."""
    import token_sparse_mla_gb300 as smla
    with torch.cuda.stream(stream):
        for _ in range(3):
            smla.sparse_mla_fwd(q, kv, idx, scale, out=out, lse=lse, kv_format=kv_format, stream=stream)
    smla.sync_status(stream)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(n_steps):
            smla.sparse_mla_fwd(q, kv, idx, scale, out=out, lse=lse, kv_format=kv_format, stream=stream)
    return g


def roofline_fields(h: int, gbytes: float, row_bytes: int, ms: float, peaks: dict) -> dict:
    """Bound, achieved figure and fraction of one launch: 64 heads fill the MMA tile, so the
    tensor roofline bounds them; fewer heads are bound by the gathered HBM bytes."""
    gbps = gbytes / (ms * 1e-3) / 1e9
    if h >= 64:
        tfl = gbytes / row_bytes * flops_per_entry(h) / (ms * 1e-3) / 1e12
        return {"bound": "tensor", "achieved": tfl, "unit": "TFLOP/s", "peak": peaks["bf16_tflops_sustained"],
                "frac": tfl / peaks["bf16_tflops_sustained"], "gathered_gbps": gbps,
                "hbm_frac": gbps / peaks["hbm_gbs"]}
    return {"bound": "hbm", "achieved": gbps, "unit": "GB/s", "peak": peaks["hbm_gbs"],
            "frac": gbps / peaks["hbm_gbs"], "gathered_gbps": gbps}


def per_config_runs(args, dev, stream, peaks: dict, main_entry: dict) -> dict:
    """Every single-GPU configuration beside the headline one, timed in the same run as the
    median of >= 10 CUDA-event windows of >= 1 ms (graphs of consecutive steps): the head-count
    sweep native and padded to 64 heads, the prefill chunk, and the fp8 batch native and padded."""
    res = {"decode_bf16": main_entry}

    def run(key, name, q, kv, idx, scale, row_bytes, kv_format, h_real):
        T, H = int(q.shape[0]), int(q.shape[1])
        out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((T, H), dtype=torch.float32, device=dev)
        gb = gathered_bytes(idx, int(kv.shape[0]), row_bytes)
        qd, kvd, idd = q.to(dev), kv.to(dev), idx.to(dev)
        g1 = forward_graph(qd, kvd, idd, scale, out, lse, kv_format, stream, 1)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        with torch.cuda.stream(stream):
            g1.replay()
        ev1.record(stream)
        ev1.synchronize()
        n = max(1, min(32, math.ceil(1.0 / max(ev0.elapsed_time(ev1), 1e-3))))
        g = forward_graph(qd, kvd, idd, scale, out, lse, kv_format, stream, n) if n > 1 else g1
        ms, k = median_of_windows(g.replay, n, stream)
        import token_sparse_mla_gb300 as smla
        smla.sync_status(stream)
        e = {"workload": name, "T": T, "h": H, "h_real": h_real, "padded_to_64": H != h_real,
             "kv_format": kv_format, "ms": ms, "query_tokens_per_s": T / (ms * 1e-3),
             "windows": 10, "steps_per_window": k * n, "gathered_bytes": gb,
             "kernel": kernel_name(H), **roofline_fields(H, gb, row_bytes, ms, peaks),
             "traffic": ncu_traffic(name, H, H != h_real)}
        res[key] = e
        del qd, kvd, idd, out, lse, g, g1
        torch.cuda.synchronize(dev)

    sw = make_workload("sweep", h=64)
    for h in (8, 16, 32, 64):
        qh = sw.q[:, :h].contiguous()
        run(f"sweep_h{h}", "sweep", qh, sw.kv, sw.indices, sw.scale, 1152, "bf16", h)
        if h < 64:
            run(f"sweep_h{h}_pad64", "sweep", pad_heads(qh, 64), sw.kv, sw.indices, sw.scale, 1152, "bf16", h)
    del sw
    pf = make_workload("prefill")
    run("prefill", "prefill", pf.q, pf.kv, pf.indices, pf.scale, 1152, "bf16", 64)
    del pf
    f8 = make_workload("fp8_mixed")
    run("fp8_mixed", "fp8_mixed", f8.q, f8.kv, f8.indices, f8.scale, 656, "fp8", 8)
    run("fp8_mixed_pad64", "fp8_mixed", pad_heads(f8.q, 64), f8.kv, f8.indices, f8.scale, 656, "fp8", 8)
    del f8
    return res


def run_ours(args, rank, world, local_rank):
    import token_sparse_mla_gb300 as smla
    dev = torch.device(f"cuda:{local_rank}")
    torch.cuda.set_device(dev)
    name = args.workload
    cfg = config_by_name(name)
    base = make_workload(name, h=args.h, seed=cfg.seed + 7919 * rank)
    gb_step = gathered_bytes(base.indices, base.num_slots, cfg.row_bytes)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size or L2_BYTES_DEFAULT
    rot = args.rot or max(1, min(8, math.ceil(2 * l2 / max(gb_step, 1))))
    sets = [base] + [make_workload(name, h=args.h, seed=cfg.seed + 100 * i + 7919 * rank)
                     for i in range(1, rot)]
    if args.pad:
        for w in sets:
            w.q = pad_heads(w.q, 64)
    T, H, topk = sets[0].T, int(sets[0].q.shape[1]), sets[0].topk
    qs = [w.q.to(dev) for w in sets]
    kvs = [w.kv.to(dev) for w in sets]
    ids = [w.indices.to(dev) for w in sets]
    outs = [torch.empty((T, H, 512), dtype=torch.bfloat16, device=dev) for _ in sets]
    lses = [torch.empty((T, H), dtype=torch.float32, device=dev) for _ in sets]
    gbytes = [gathered_bytes(w.indices, w.num_slots, cfg.row_bytes) for w in sets]
    stream = torch.cuda.Stream(dev)  # a side stream: CUDA graphs cannot capture the default one
    info = smla.launch_info(T, H, topk, cfg.kv_format)

    def step(i):
        k = i % rot
        smla.sparse_mla_fwd(qs[k], kvs[k], ids[k], sets[k].scale, out=outs[k], lse=lses[k],
                            kv_format=cfg.kv_format, stream=stream)

    # CUDA graphs of consecutive steps (the launch path a serving loop uses): one of `glen`
    # steps replayed K // glen times, and one of the K % glen remaining steps
    graphs = []

    def capture(n_steps):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n_steps):
                step(i)
        return g

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i)
    smla.sync_status(stream)
    glen = rot * max(1, 32 // rot)
    if args.launch == "graph":
        graphs = [capture(glen), capture(args.steps % glen) if args.steps % glen else None]
        for _ in range(2):
            graphs[0].replay()
        torch.cuda.synchronize(dev)

    def timed_steps(k_steps):
        if args.launch == "graph":
            for _ in range(k_steps // glen):
                graphs[0].replay()
            if k_steps % glen:
                graphs[1].replay()
        else:
            for i in range(k_steps):
                step(i)
    clocks = ClockSampler(local_rank)
    clocks.start()
    # keep the GPU busy (0.3 s by default) before the timed region so the clock samples see load
    t_pre = time.time()
    i = 0
    while time.time() - t_pre < args.prerun:
        with torch.cuda.stream(stream):
            timed_steps(glen)
        i += 1
        if i % 8 == 0:
            torch.cuda.synchronize(dev)
    barrier()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    gpu_busy_wait(stream)  # the K steps below are queued while this runs
    ev0.record(stream)
    with torch.cuda.stream(stream):
        timed_steps(args.steps)
    ev1.record(stream)
    barrier()
    t_dev = ev0.elapsed_time(ev1) / 1e3
    clocks.stop()
    smla.sync_status(stream)
    t_dev = max_over_ranks(t_dev, world, dev)
    value = world * T * args.steps / t_dev
    per_launch = t_dev / args.steps
    avg_gb = sum(gbytes[i % rot] for i in range(args.steps)) / args.steps
    peaks = measured_peaks()
    achieved = avg_gb / per_launch / 1e9
    traffic = ncu_traffic(name, base.h, args.pad)

    # the same workload as the median of >= 10 windows of >= 1 ms each
    win = None
    if args.launch == "graph":
        ms_w, k_w = median_of_windows(graphs[0].replay, glen, stream)
        win = {"ms_per_step": ms_w, "query_tokens_per_s": T / (ms_w * 1e-3), "windows": 10,
               "steps_per_window": k_w * glen,
               **roofline_fields(H, avg_gb, cfg.row_bytes, ms_w, peaks)}

    # ---- end to end through the packed host-buffer entry point: one H2D copy of the step's
    # inputs, the kernel and one D2H copy of its outputs per step; steps alternate between two
    # streams with their own workspaces, so one step's copies overlap its neighbour's kernel
    e2e = None
    if not args.no_e2e:
        lay = smla.host_io_layout(T, H, topk)
        ins = []
        for w in sets:
            b = torch.empty(lay["in_bytes"], dtype=torch.uint8).pin_memory()
            qv, iv, _, _ = smla.host_io_views(b, torch.empty(lay["out_bytes"], dtype=torch.uint8), T, H, topk)
            qv.copy_(w.q)
            iv.copy_(w.indices)
            ins.append(b)
        ss = [stream, torch.cuda.Stream(dev)]
        obs = [torch.empty(lay["out_bytes"], dtype=torch.uint8).pin_memory() for _ in ss]
        wss = [torch.empty(smla.host_workspace_bytes(T, H, topk), dtype=torch.uint8, device=dev) for _ in ss]
        e2e_steps = max(1, min(args.steps, args.e2e_steps))

        def estep(i):
            j, k = i % 2, i % rot
            smla.sparse_mla_fwd_host_packed(ins[k], kvs[k], T, H, topk, sets[k].scale, obs[j], wss[j],
                                            kv_format=cfg.kv_format, stream=ss[j])
        for i in range(max(4, args.warmup // 10)):
            estep(i)
        barrier()
        e0, e1, eb = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
                      torch.cuda.Event())
        gpu_busy_wait(ss[0])
        e0.record(ss[0])
        ss[1].wait_event(e0)
        for i in range(e2e_steps):
            estep(i)
        eb.record(ss[1])
        ss[0].wait_event(eb)
        e1.record(ss[0])
        barrier()
        t_e2e = e0.elapsed_time(e1) / 1e3
        smla.sync_status(ss[0])
        smla.sync_status(ss[1])
        t_e2e = max_over_ranks(t_e2e, world, dev)
        e2e = {"value": world * T * e2e_steps / t_e2e, "unit": UNIT, "h2d_bytes_per_step": lay["in_bytes"],
               "d2h_bytes_per_step": lay["out_bytes"], "steps": e2e_steps,
               "path": "sparse_mla_fwd_host_packed (pinned host [q | indices] in, [out | lse] back, one "
                       "copy each way per step; two streams alternate; cache resident)"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, threads, ntok, el = oracle_rate(base, args.cpu_seconds)
        cpu = {"value": rate, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"{ntok} query tokens (the workload's first {min(base.T, 32)} tokens, "
                         f"repeated) in {el:.1f} s"}

    rf = roofline_fields(H, avg_gb, cfg.row_bytes, per_launch * 1e3, peaks)
    if H >= 64:
        # 64 heads fill the MMA tile: the tensor roofline bounds the kernel (the gathered
        # bytes are reported beside it)
        roof = {"bound": "tensor", "achieved": rf["achieved"], "peak": peaks["bf16_tflops_sustained"],
                "unit": "TFLOP/s", "frac": rf["frac"],
                "traffic": traffic, "peak_source": peaks["source"] + " (bf16 sustained)",
                "per_launch_algorithmic_flops": avg_gb / cfg.row_bytes * flops_per_entry(H),
                "hbm_frac": achieved / peaks["hbm_gbs"], "kernel": kernel_name(H)}
    else:
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                "peak_source": peaks["source"] + " (copy bandwidth)",
                "per_launch_algorithmic_bytes": avg_gb, "kernel": kernel_name(H)}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": per_launch * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(base, args, info["splits"], rot, info["ctas"]),
        "gathered_gbps": achieved,
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "clocks": clocks.summary(),
        "gpu_launches": info["launches"] * args.steps,
        "median_of_windows": win,
    }
    if (name == "decode_bf16" and not args.pad and args.h is None and not args.no_per_config
            and args.launch == "graph"):
        entry = dict(win or {})
        entry.update({"workload": name, "T": T, "h": H, "h_real": H, "kv_format": cfg.kv_format})
        pc = per_config_runs(args, dev, stream, peaks, entry)
        line["per_config"] = pc

        def ratio(nat, pad):
            if nat in pc and pad in pc:
                return pc[pad]["ms"] / pc[nat]["ms"]
            return None
        line["native_over_padded"] = {
            "meaning": "time per token of the padded-to-64 arm / time per token of the native arm "
                       "(> 1: the native path is faster)",
            "sweep_h8": ratio("sweep_h8", "sweep_h8_pad64"),
            "sweep_h16": ratio("sweep_h16", "sweep_h16_pad64"),
            "sweep_h32": ratio("sweep_h32", "sweep_h32_pad64"),
            "fp8_mixed_h8": ratio("fp8_mixed", "fp8_mixed_pad64")}
    if rank == 0:
        print(json.dumps(line), flush=True)


# ---- the DCP merge (combine of split-list partial results), on the fp8 batch's shape
MERGE_SHAPE = {"n_parts": 4, "T": 32768, "h": 8}


def merge_bytes(lse_parts: torch.Tensor) -> int:
    """Algorithmic bytes of one merge: every LSE and the O (bf16) of every non-empty part read
    (an empty part's O is never needed), O and LSE written."""
    n = lse_parts.shape[0]
    rows = lse_parts[0].numel()
    nonempty = int((lse_parts != float("-inf")).sum().item())
    return nonempty * 512 * 2 + n * rows * 4 + rows * (512 * 2 + 4)


def merge_config(args, nbytes: int) -> dict:
    return {"workload": "dcp_merge", **MERGE_SHAPE,
            "parts": "synthetic partials: O ~ bf16(N(0, 0.1)), LSE ~ N(6, 1); each part empty with "
                     "probability 0.05, and head 0 of every token empty in all parts",
            "launch": "CUDA graph of consecutive steps" if args.launch == "graph" else "eager launches",
            "l2": f"{nbytes / 1e9:.2f} GB read and written per step > 2 x L2"}


def run_merge(args, rank, world, local_rank):
    import token_sparse_mla_gb300 as smla
    dev = torch.device(f"cuda:{local_rank}")
    torch.cuda.set_device(dev)
    n, T, H = MERGE_SHAPE["n_parts"], MERGE_SHAPE["T"], MERGE_SHAPE["h"]
    o_h, l_h = make_merge_parts(n, T, H, seed=6000 + 7919 * rank)
    o_d, l_d = o_h.to(dev), l_h.to(dev)
    out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(dev)

    def step():
        smla.sparse_mla_merge(o_d, l_d, out=out, lse=lse, stream=stream)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    smla.sync_status(stream)
    glen = 16
    graph = None
    if args.launch == "graph":
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for _ in range(glen):
                step()
        graph.replay()
        torch.cuda.synchronize(dev)
    steps = max(glen, (args.steps // glen) * glen) if graph is not None else args.steps

    def timed():
        if graph is not None:
            for _ in range(steps // glen):
                graph.replay()
        else:
            for _ in range(steps):
                step()
    clocks = ClockSampler(local_rank)
    clocks.start()
    with torch.cuda.stream(stream):
        timed()
    torch.cuda.synchronize(dev)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    with torch.cuda.stream(stream):
        timed()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    clocks.stop()
    smla.sync_status(stream)
    t_dev = max_over_ranks(ev0.elapsed_time(ev1) / 1e3, world, dev)
    per_launch = t_dev / steps
    nbytes = merge_bytes(l_h)
    achieved = nbytes / per_launch / 1e9
    peaks = measured_peaks()
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        tok = 256
        t0 = time.perf_counter()
        k = 0
        while time.perf_counter() - t0 < args.cpu_seconds or k == 0:
            oracle.merge(o_h[:, :tok], l_h[:, :tok])
            k += 1
        el = time.perf_counter() - t0
        cpu = {"value": k * tok / el, "unit": UNIT, "cores": oracle.max_threads(), "kind": "oracle",
               "sample": f"the first {tok} query tokens' rows, merged {k} times in {el:.1f} s"}
    line = {
        "metric": METRIC, "value": world * T * steps / t_dev, "unit": UNIT, "n_gpus": world,
        "steps": steps, "warmup": args.warmup, "ms_per_step": per_launch * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": merge_config(args, nbytes), "merged_gbps": achieved,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": ncu_traffic("dcp_merge", H, False),
                     "peak_source": peaks["source"] + " (copy bandwidth)",
                     "per_launch_algorithmic_bytes": nbytes, "kernel": "sparse_mla_merge_kernel"},
        "cpu_baseline": cpu, "e2e": None, "clocks": clocks.summary(), "gpu_launches": steps,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_merge_reference(args, rank, world):
    if rank != 0:
        return
    import oracle
    oracle.build()
    n, T, H = MERGE_SHAPE["n_parts"], MERGE_SHAPE["T"], MERGE_SHAPE["h"]
    o_h, l_h = make_merge_parts(n, T, H, seed=6000)
    tok = 256
    for _ in range(args.warmup):
        oracle.merge(o_h[:, :8], l_h[:, :8])
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.merge(o_h[:, :tok], l_h[:, :tok])
    el = time.perf_counter() - t0
    value = tok * args.steps / el
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": merge_config(args, merge_bytes(l_h)),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.max_threads(), "kind": "oracle",
                         "sample": f"{tok} query tokens' rows per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# ---- the v_up projection of the attention output (DeepSeek-V3.2 geometry, 8 heads)
V_UP_SHAPE = {"T": 32768, "h": 8, "v": 128}


def v_up_inputs(seed: int):
    g = torch.Generator().manual_seed(seed)
    o = (torch.randn(V_UP_SHAPE["T"], V_UP_SHAPE["h"], 512, generator=g) * 0.1).to(torch.bfloat16)
    return o, make_v_up_weights(V_UP_SHAPE["h"], V_UP_SHAPE["v"], seed=seed)


def v_up_bytes() -> int:
    T, h, v = V_UP_SHAPE["T"], V_UP_SHAPE["h"], V_UP_SHAPE["v"]
    return (T * h * 512 + h * v * 512 + T * h * v) * 2


def v_up_config(args) -> dict:
    return {"workload": "v_up", **V_UP_SHAPE,
            "inputs": "O ~ bf16(N(0, 0.1)) [T, h, 512], W ~ bf16(N(0, 1) / sqrt(512)) [h, v, 512]",
            "launch": "CUDA graph of consecutive steps" if args.launch == "graph" else "eager launches",
            "l2": f"{v_up_bytes() / 1e6:.0f} MB read and written per step > 2 x L2"}


def run_v_up(args, rank, world, local_rank):
    import token_sparse_mla_gb300 as smla
    dev = torch.device(f"cuda:{local_rank}")
    torch.cuda.set_device(dev)
    T, H, V = V_UP_SHAPE["T"], V_UP_SHAPE["h"], V_UP_SHAPE["v"]
    o_h, w_h = v_up_inputs(7100 + 7919 * rank)
    o_d, w_d = o_h.to(dev), w_h.to(dev)
    y = torch.empty((T, H, V), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.Stream(dev)

    def step():
        smla.sparse_mla_v_up(o_d, w_d, out=y, stream=stream)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    smla.sync_status(stream)
    glen = 16
    graph = None
    if args.launch == "graph":
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for _ in range(glen):
                step()
        graph.replay()
        torch.cuda.synchronize(dev)
    steps = max(glen, (args.steps // glen) * glen) if graph is not None else args.steps

    def timed():
        if graph is not None:
            for _ in range(steps // glen):
                graph.replay()
        else:
            for _ in range(steps):
                step()
    clocks = ClockSampler(local_rank)
    clocks.start()
    with torch.cuda.stream(stream):
        timed()
    torch.cuda.synchronize(dev)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    with torch.cuda.stream(stream):
        timed()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    clocks.stop()
    smla.sync_status(stream)
    t_dev = max_over_ranks(ev0.elapsed_time(ev1) / 1e3, world, dev)
    per_launch = t_dev / steps
    nbytes = v_up_bytes()
    achieved = nbytes / per_launch / 1e9
    flops = 2.0 * T * H * 512 * V
    peaks = measured_peaks()
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        tok = 512
        t0 = time.perf_counter()
        k = 0
        while time.perf_counter() - t0 < args.cpu_seconds or k == 0:
            oracle.v_up(o_h[:tok], w_h)
            k += 1
        el = time.perf_counter() - t0
        cpu = {"value": k * tok / el, "unit": UNIT, "cores": oracle.max_threads(), "kind": "oracle",
               "sample": f"the first {tok} query tokens, projected {k} times in {el:.1f} s"}
    line = {
        "metric": METRIC, "value": world * T * steps / t_dev, "unit": UNIT, "n_gpus": world,
        "steps": steps, "warmup": args.warmup, "ms_per_step": per_launch * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": v_up_config(args), "tflops": flops / per_launch / 1e12,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": ncu_traffic("v_up", H, False),
                     "peak_source": peaks["source"] + " (copy bandwidth)",
                     "per_launch_algorithmic_bytes": nbytes,
                     "tensor_frac": flops / per_launch / 1e12 / peaks["bf16_tflops_sustained"],
                     "kernel": "sparse_mla_v_up_kernel"},
        "cpu_baseline": cpu, "e2e": None, "clocks": clocks.summary(), "gpu_launches": steps,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_v_up_reference(args, rank, world):
    if rank != 0:
        return
    import oracle
    oracle.build()
    o_h, w_h = v_up_inputs(7100)
    tok = 512
    for _ in range(args.warmup):
        oracle.v_up(o_h[:8], w_h)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.v_up(o_h[:tok], w_h)
    el = time.perf_counter() - t0
    value = tok * args.steps / el
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": v_up_config(args),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.max_threads(), "kind": "oracle",
                         "sample": f"{tok} query tokens per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# ---- top-k selection of the index lists (the prefill chunk's shape: causal rows)
TOPK_SHAPE = {"T": 16384, "S": 32768, "topk": 2048}


def topk_inputs(seed: int):
    T, S = TOPK_SHAPE["T"], TOPK_SHAPE["S"]
    g = torch.Generator().manual_seed(seed)
    scores = torch.randn(T, S, generator=g)
    lens = torch.arange(S - T + 1, S + 1, dtype=torch.int32)  # query positions S-T .. S-1
    table = torch.randperm(S // 64, generator=g).to(torch.int32)
    return scores, lens, table


def topk_bytes(lens) -> int:
    """Scores read once over each row's history, the lengths, the lists written."""
    T = lens.numel()
    return int(lens.sum().item()) * 4 + T * 4 + T * TOPK_SHAPE["topk"] * 4


def topk_config(args, nbytes: int) -> dict:
    return {"workload": "topk", **TOPK_SHAPE,
            "inputs": "scores ~ N(0, 1) fp32 [T, S], causal histories S - T + 1 .. S, a random block table",
            "launch": "CUDA graph of consecutive steps" if args.launch == "graph" else "eager launches",
            "l2": f"{nbytes / 1e9:.2f} GB read and written per step > 2 x L2"}


def run_topk(args, rank, world, local_rank):
    import token_sparse_mla_gb300 as smla
    dev = torch.device(f"cuda:{local_rank}")
    torch.cuda.set_device(dev)
    T, S, K = TOPK_SHAPE["T"], TOPK_SHAPE["S"], TOPK_SHAPE["topk"]
    s_h, l_h, t_h = topk_inputs(7200 + 7919 * rank)
    s_d, l_d, t_d = s_h.to(dev), l_h.to(dev), t_h.to(dev)
    out = torch.empty((T, K), dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(dev)

    def step():
        smla.sparse_mla_topk(s_d, l_d, K, block_table=t_d, out=out, stream=stream)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    smla.sync_status(stream)
    glen = 4
    graph = None
    if args.launch == "graph":
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for _ in range(glen):
                step()
        graph.replay()
        torch.cuda.synchronize(dev)
    steps = max(glen, (args.steps // glen) * glen) if graph is not None else args.steps

    def timed():
        if graph is not None:
            for _ in range(steps // glen):
                graph.replay()
        else:
            for _ in range(steps):
                step()
    clocks = ClockSampler(local_rank)
    clocks.start()
    with torch.cuda.stream(stream):
        timed()
    torch.cuda.synchronize(dev)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    with torch.cuda.stream(stream):
        timed()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    clocks.stop()
    smla.sync_status(stream)
    t_dev = max_over_ranks(ev0.elapsed_time(ev1) / 1e3, world, dev)
    per_launch = t_dev / steps
    nbytes = topk_bytes(l_h)
    achieved = nbytes / per_launch / 1e9
    peaks = measured_peaks()
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        rows = 64
        t0 = time.perf_counter()
        k = 0
        while time.perf_counter() - t0 < args.cpu_seconds or k == 0:
            oracle.topk(s_h[:rows], l_h[:rows], K, block_table=t_h)
            k += 1
        el = time.perf_counter() - t0
        cpu = {"value": k * rows / el, "unit": UNIT, "cores": oracle.max_threads(), "kind": "oracle",
               "sample": f"the first {rows} rows, selected {k} times in {el:.1f} s"}
    line = {
        "metric": METRIC, "value": world * T * steps / t_dev, "unit": UNIT, "n_gpus": world,
        "steps": steps, "warmup": args.warmup, "ms_per_step": per_launch * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": topk_config(args, nbytes),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": ncu_traffic("topk", 0, False),
                     "peak_source": peaks["source"] + " (copy bandwidth)",
                     "per_launch_algorithmic_bytes": nbytes, "kernel": "sparse_mla_topk_kernel"},
        "cpu_baseline": cpu, "e2e": None, "clocks": clocks.summary(), "gpu_launches": steps,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_topk_reference(args, rank, world):
    if rank != 0:
        return
    import oracle
    oracle.build()
    s_h, l_h, t_h = topk_inputs(7200)
    rows = 64
    for _ in range(args.warmup):
        oracle.topk(s_h[:2], l_h[:2], TOPK_SHAPE["topk"], block_table=t_h)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.topk(s_h[:rows], l_h[:rows], TOPK_SHAPE["topk"], block_table=t_h)
    el = time.perf_counter() - t0
    value = rows * args.steps / el
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": topk_config(args, topk_bytes(l_h)),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.max_threads(), "kind": "oracle",
                         "sample": f"{rows} rows per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# ---- the masked dense route: a GLM-5 prefill chunk that is the whole request
MASKED_SHAPE = {"T": 4096, "S": 4096, "h": 64, "dqk": 256, "dv": 256, "topk": 2048}


def masked_inputs(seed: int):
    from workloads import causal_position_lists, make_masked_dense_inputs
    m = MASKED_SHAPE
    q, k, v = make_masked_dense_inputs(m["T"], m["S"], m["h"], m["dqk"], m["dv"], seed=seed)
    lists = causal_position_lists(m["T"], m["S"], m["topk"], seed=seed + 1)
    return q, k, v, lists


def masked_tile_work(mask_words: torch.Tensor) -> dict:
    """Dense work of the route: per 128-query tile, the 64-key tiles any of its rows attends to,
    each a 128 x 64 block of QK^T and PV; beside it the masked-in (token, position) pairs."""
    m = MASKED_SHAPE
    T, W = mask_words.shape
    nz = (mask_words != 0)
    if W % 2:
        nz = torch.cat([nz, torch.zeros(T, 1, dtype=torch.bool)], dim=1)
    key_tiles = nz.view(T, -1, 2).any(dim=2)                      # [T, key tiles]
    nq = (T + 127) // 128
    pad = nq * 128 - T
    if pad:
        key_tiles = torch.cat([key_tiles, torch.zeros(pad, key_tiles.shape[1], dtype=torch.bool)])
    active = int(key_tiles.view(nq, 128, -1).any(dim=1).sum().item())
    import numpy as np
    pairs = int(np.unpackbits(np.ascontiguousarray(mask_words.numpy()).view(np.uint8)).sum())
    per_pair = 2 * m["h"] * (m["dqk"] + m["dv"])
    return {"active_tiles": active, "tile_flops": active * 128 * 64 * per_pair,
            "pairs": pairs, "pair_flops": pairs * per_pair}


def masked_config(args) -> dict:
    return {"workload": "masked_dense", **MASKED_SHAPE,
            "geometry": "GLM-5: 64 heads, q/k 192 nope + 64 rope, v 256",
            "inputs": "q, k, v ~ bf16(N(0, 1) * 0.5); lists = top-2048 of uniform keys over each causal history",
            "launch": "CUDA graph of consecutive steps" if args.launch == "graph" else "eager launches",
            "step": "sparse_mla_scatter_mask + sparse_mla_masked_mha"}


def run_masked(args, rank, world, local_rank):
    import numpy as np
    import token_sparse_mla_gb300 as smla
    dev = torch.device(f"cuda:{local_rank}")
    torch.cuda.set_device(dev)
    m = MASKED_SHAPE
    q_h, k_h, v_h, l_h = masked_inputs(9400 + 7919 * rank)
    q_d, k_d, v_d, l_d = q_h.to(dev), k_h.to(dev), v_h.to(dev), l_h.to(dev)
    W = (m["S"] + 31) // 32
    mask = torch.empty((m["T"], W), dtype=torch.int32, device=dev)
    out = torch.empty((m["T"], m["h"], m["dv"]), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((m["T"], m["h"]), dtype=torch.float32, device=dev)
    scale = m["dqk"] ** -0.5
    stream = torch.cuda.Stream(dev)

    def step():
        smla.sparse_mla_scatter_mask(l_d, m["S"], out=mask, stream=stream)
        smla.sparse_mla_masked_mha(q_d, k_d, v_d, mask, scale, out=out, lse=lse, stream=stream)

    def mha_only():
        smla.sparse_mla_masked_mha(q_d, k_d, v_d, mask, scale, out=out, lse=lse, stream=stream)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    smla.sync_status(stream)
    work = masked_tile_work(mask.cpu())
    glen = 4

    def graph_of(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(glen):
                fn()
        return g
    g_step, g_mha = graph_of(step), graph_of(mha_only)
    steps = max(glen, (args.steps // glen) * glen)
    clocks = ClockSampler(local_rank)
    clocks.start()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    gpu_busy_wait(stream)
    ev0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(steps // glen):
            g_step.replay()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    clocks.stop()
    t_dev = max_over_ranks(ev0.elapsed_time(ev1) / 1e3, world, dev)
    per_step = t_dev / steps
    ms_mha, _ = median_of_windows(g_mha.replay, glen, stream)
    smla.sync_status(stream)
    peaks = measured_peaks()
    tfl = work["tile_flops"] / (ms_mha * 1e-3) / 1e12
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        toks = [0, 1000, 2047, 3000, 4095]
        mk = oracle.scatter_mask(l_h[toks], m["S"])
        t0 = time.perf_counter()
        n = 0
        while time.perf_counter() - t0 < args.cpu_seconds or n == 0:
            oracle.masked_mha(q_h[toks], k_h, v_h, mk, scale)
            n += 1
        el = time.perf_counter() - t0
        cpu = {"value": n * len(toks) / el, "unit": UNIT, "cores": oracle.max_threads(), "kind": "oracle",
               "sample": f"{len(toks)} query tokens (all 64 heads) attended {n} times in {el:.1f} s"}
    line = {
        "metric": METRIC, "value": world * m["T"] * steps / t_dev, "unit": UNIT, "n_gpus": world,
        "steps": steps, "warmup": args.warmup, "ms_per_step": per_step * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": masked_config(args),
        "roofline": {"bound": "tensor", "achieved": tfl, "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s",
                     "frac": tfl / peaks["bf16_tflops_sustained"], "traffic": ncu_traffic("masked_dense", m["h"], False),
                     "peak_source": peaks["source"] + " (bf16 sustained)", "kernel": "sparse_mla_masked_mha_kernel",
                     "per_launch_algorithmic_flops": work["tile_flops"], "kernel_ms": ms_mha,
                     "flops_basis": "dense 128 x 64 tiles that hold a masked-in position",
                     "masked_in_pair_flops": work["pair_flops"], "active_tiles": work["active_tiles"]},
        "cpu_baseline": cpu, "e2e": None, "clocks": clocks.summary(), "gpu_launches": 2 * steps,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_masked_reference(args, rank, world):
    if rank != 0:
        return
    import oracle
    oracle.build()
    m = MASKED_SHAPE
    q_h, k_h, v_h, l_h = masked_inputs(9400)
    toks = [0, 2047, 4095]
    scale = m["dqk"] ** -0.5
    for _ in range(args.warmup):
        oracle.masked_mha(q_h[toks[:1]], k_h, v_h, oracle.scatter_mask(l_h[toks[:1]], m["S"]), scale)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.masked_mha(q_h[toks], k_h, v_h, oracle.scatter_mask(l_h[toks], m["S"]), scale)
    el = time.perf_counter() - t0
    value = len(toks) * args.steps / el
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": masked_config(args),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.max_threads(), "kind": "oracle",
                         "sample": f"{len(toks)} query tokens (all heads) per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="decode_bf16")
    ap.add_argument("--h", type=int, default=None, help="head count (sweep workload)")
    ap.add_argument("--pad", action="store_true", help="zero-pad the heads to 64")
    ap.add_argument("--rot", type=int, default=0, help="input sets to rotate (0 = auto)")
    ap.add_argument("--e2e-steps", type=int, default=2000)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the other configurations (timed beside the decode batch by default)")
    ap.add_argument("--launch", choices=["graph", "eager"], default="graph",
                    help="replay the timed steps from CUDA graphs, or launch each step eagerly")
    ap.add_argument("--prerun", type=float, default=0.3,
                    help="seconds of untimed steps before the timed region (clock samples)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local_rank = dist_setup(args)
    if args.workload == "masked_dense":
        (run_masked_reference(args, rank, world) if args.impl == "reference"
         else run_masked(args, rank, world, local_rank))
    elif args.workload == "topk":
        (run_topk_reference(args, rank, world) if args.impl == "reference"
         else run_topk(args, rank, world, local_rank))
    elif args.workload == "v_up":
        (run_v_up_reference(args, rank, world) if args.impl == "reference"
         else run_v_up(args, rank, world, local_rank))
    elif args.workload == "dcp_merge":
        (run_merge_reference(args, rank, world) if args.impl == "reference"
         else run_merge(args, rank, world, local_rank))
    elif args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
