"""Throughput benchmark of the batch-invariant selected-token logprob path.

One step = one pass of the whole hot path on one GPU:
  1. linear_logp forward on a GRPO group: 64 completions x 1024 tokens
     (T = 65536), H = 4096, V = 128256, bf16, seeded synthetic data; the
     forward keeps its per-tile softmax terms (bf16) for the backward
     (rk_linear_logp_fwd_saved: tile kernel + merge);
  2. linear_logp backward on the same rows, g ~ N(0, 1), from those terms
     (rk_linear_logp_bwd_saved: the terms become dZ in one HBM-bound pass,
     the target and p >= 1/64 columns get exact fp32 weights, dh GEMM);
  3. the logits path on T = 2048 rows of V = 32000 bf16 logits (rotated over 4
     buffers so that no call finds its input in L2).
The backward that recomputes z with a second GEMM instead (rk_linear_logp +
rk_linear_logp_bwd) is timed as its own row.
`value` = tokens (rows of the GRPO group, summed over ranks) per second of
device time, inputs resident in HBM.  h (512 MB) and W (1.05 GB) exceed the
126 MB L2, so nothing carries over between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
    python bench.py --case {fwd,bwd,dw,full,saved,full_saved,logits,logits_bwd,
                            qwen_padded,qwen_packed} [--shape T,H,V] [--reps R]

`--case` runs one operator a few times on a small workload (for profiler
captures; default T=2048, H=4096, V=32000: W and the logits exceed L2) and
prints its mean device time.  qwen_padded / qwen_packed run the Qwen-shaped
forward on sequences 0-7, right-padded to [8, 2048] or varlen-packed.

Under torchrun (N > 1) every rank runs its own group (weak scaling, no data
collective); the timed region is bracketed by barriers and the max over ranks
is reported.  `--impl reference` times the fp64 CPU oracle on a bounded sample
of the same workload instead (rank 0 only, one thread per host CPU).

The end-to-end figure (`e2e`) runs the same step from pinned host buffers:
every step's inputs are copied in and its dh / logp copied out, on their own
streams, against four device buffer sets.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "linear_logp tokens/s & % BF16 tensor peak, bitwise batch-invariant"
UNIT = "tokens/s"
GRPO = dict(n_seqs=64, seq_len=1024, H=4096, V=128256)
LOGITS = dict(T=2048, V=32000)
N_LOGITS_BUFFERS = 4
LOGITS_REPEATS = 7
WORKLOAD = ("grpo_fwd_bwd: linear_logp fwd+bwd T=65536 (64x1024) H=4096 V=128256 bf16, "
            "+ logits path T=2048 V=32000 bf16")

# ncu dram__bytes_read.sum + dram__bytes_write.sum of the two tile-kernel
# launches of one step (the forward that keeps its softmax terms, the dh GEMM)
# on this very workload (`ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,
# gpu__time_duration.sum --clock-control none -k regex:linear_logp_tiles -c 2
# python bench.py --steps 3 --warmup 3 --no-cpu-baseline --no-rows`, one pass per
# launch), recorded with the SHA-1 of the kernel source; reported only while the
# source still matches.
TRAFFIC_RECORD = {
    "source_sha1": "7c79002ffa7c04acf135db1752e30e4c74bf36ad",
    "bytes_per_step": 104289638400,
    "per_launch_gb": {"fwd_saved": 37.15, "dh": 67.14},
}

# Unique bytes a step has to move: forward h + W read, partials + target
# logits + the softmax terms (T*V bf16) written; stash -> dZ pass: the terms
# read and dZ written in place, partials read; dh GEMM: dZ + W read, dh
# written.
def algorithmic_bytes_per_step(T: int, H: int, V: int) -> int:
    nt = (V + 255) // 256
    h, w = T * H * 2, V * H * 2
    dz = T * V * 2
    part = T * nt * 8
    return (h + w + part + T * 4 + dz) + (2 * dz + part) + (dz + w + T * H * 4)


def kernel_source_sha1() -> str:
    p = os.path.join(ROOT, "invariant_rl_logprob_gb300", "csrc", "linear_logp_tc.cu")
    with open(p, "rb") as f:
        return hashlib.sha1(f.read()).hexdigest()


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# ---------------------------------------------------------------------------
# distributed plumbing (weak scaling, timing max over ranks)
# ---------------------------------------------------------------------------

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, world_size: int) -> float:
    if world_size == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world_size: int) -> None:
    if world_size > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="rk_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        rows = []
        if self.path and os.path.exists(self.path):
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) >= 9:
                        rows.append(parts)
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = max(float(r[2]) for r in rows if r[2].replace(".", "").isdigit())
        loaded = [s for s in sm if s > 0.5 * smax] or sm
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for i, n in enumerate(names):
                if r[5 + i].lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max((float(r[3]) for r in rows
                                    if r[3].replace(".", "").isdigit()), default=None)}


# ---------------------------------------------------------------------------
# workload
# ---------------------------------------------------------------------------

def make_inputs(rank: int):
    from invariant_rl_logprob_gb300 import synth
    seed_shift = 100 * rank
    c = synth.WORKLOADS["grpo"]
    lengths = [GRPO["seq_len"]] * GRPO["n_seqs"]
    pool = synth.make_pool(GRPO["H"], GRPO["V"], lengths, c["seed"] + seed_shift, with_grad=True)
    logits = []
    for i in range(N_LOGITS_BUFFERS):
        z, tg, _ = synth.logits_batch(seed=synth.WORKLOADS["logits"]["seed"] + seed_shift + 10 * i)
        logits.append((z, tg))
    return pool, logits


def oracle_threads() -> int:
    """Host cores the oracle runs on (threads over rows; its C calls release
    the GIL, and every row is computed independently)."""
    try:
        n = len(os.sched_getaffinity(0))  # the CPUs this process may run on
    except (AttributeError, OSError):
        n = os.cpu_count() or 1
    return max(1, n)


def cpu_oracle_sample(pool, logits, rows_per_thread: int) -> tuple[float, int, str]:
    """Time the fp64 oracle, unchanged, on the host cores: each of `threads`
    threads takes rows_per_thread GRPO rows (fwd + bwd) and as many
    logits-path rows; returns (tokens/s, threads, description)."""
    import concurrent.futures as cf

    import oracle
    from invariant_rl_logprob_gb300 import synth
    oracle.build()
    threads = oracle_threads()
    n_rows = rows_per_thread * threads
    hb = synth.bf16_bits(pool.h)
    Wb = synth.bf16_bits(pool.W)
    tg = pool.targets.numpy()
    g = pool.g.double().numpy()
    rows = synth.sample_rows(pool.h.shape[0], n_rows, seed=4)
    zb = synth.bf16_bits(logits[0][0])
    ztg = logits[0][1].numpy()
    zrows = synth.sample_rows(zb.shape[0], min(n_rows, zb.shape[0]), seed=1)

    def work(k):
        rr = rows[k::threads]
        oracle.linear_logp(hb, Wb, tg, rows=rr)
        oracle.linear_logp_bwd(hb, Wb, tg, g, rows=rr)
        oracle.logp_from_logits(zb, ztg, rows=zrows[k::threads])

    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(threads) as ex:
        list(ex.map(work, range(threads)))
    dt = time.perf_counter() - t0
    # one GRPO row of the step carries 2048/65536 of a logits-path row with it;
    # the logits rows are timed in full and charged to the same token count
    desc = (f"{n_rows} GRPO rows (fwd + bwd, H=4096, V=128256) + {len(zrows)} logits-path rows "
            f"(V=32000), fp64 oracle, {threads} threads (one per host core, rows split "
            f"between them), {dt:.1f} s")
    return n_rows / dt, threads, desc


def run_reference(args) -> None:
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    from invariant_rl_logprob_gb300 import synth
    c = synth.WORKLOADS["grpo"]
    # only W and a handful of rows are needed on the host
    lengths = [GRPO["seq_len"]] * GRPO["n_seqs"]
    pool = synth.make_pool(GRPO["H"], GRPO["V"], lengths, c["seed"], with_grad=True)
    z, ztg, _ = synth.logits_batch()
    logits = [(z, ztg)]
    rows_per_step = oracle_threads()   # one row per host core per step
    times = []
    for i in range(args.warmup + args.steps):
        v, cores, desc = cpu_oracle_sample(pool, logits, 1)
        if i >= args.warmup:
            times.append(rows_per_step / v)
    ms = 1000.0 * statistics.mean(times)
    value = rows_per_step / (ms / 1000.0)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample": f"{rows_per_step} GRPO row(s) fwd+bwd + "
                   f"{rows_per_step} logits-path row(s) per step"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def hold_stream(stream, ms: float = 5.0) -> None:
    """Keep `stream` busy for about `ms` so that the launches queued after it
    run back to back on the device, whatever the host's per-call overhead."""
    import torch
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(ms * 2.1e6))


def sm_clock_mhz(stream) -> float:
    """The SM clock right now, measured on the device: a spin of a known
    number of SM cycles (torch.cuda._sleep) timed with CUDA events."""
    import torch
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    cycles = 1_000_000
    with torch.cuda.stream(stream):
        a.record(stream)
        torch.cuda._sleep(cycles)
        b.record(stream)
    b.synchronize()
    return cycles / (a.elapsed_time(b) * 1e3)


def time_loop(fn, reps: int, stream) -> float:
    """Mean device ms per call of `fn` over `reps` back-to-back calls (after 3
    warm-up calls; the calls are queued behind a device-side wait so that
    host overhead cannot leave gaps between them)."""
    import torch
    for _ in range(3):
        fn(0)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    hold_stream(stream, 2.0 + 0.05 * reps)
    a.record(stream)
    for i in range(reps):
        fn(i)
    b.record(stream)
    b.synchronize()
    return a.elapsed_time(b) / reps


def measure_rows(rk, pool, zs, peaks, dev, stream) -> dict:
    """The widened rows, each in its own loop on the GRPO / logits inputs."""
    import torch
    T, H, V = pool.h.shape[0], pool.H, pool.V
    Tl, Vl = LOGITS["T"], LOGITS["V"]
    h, W, tg = pool.h.to(dev), pool.W.to(dev), pool.targets.to(dev)
    out = {}
    # dense path lm_head on a 8192-row slice of the group (bf16 logits 2.1 GB)
    Td = 8192
    logits = torch.empty((Td, V), dtype=torch.bfloat16, device=dev)
    wsl = torch.empty(rk.lm_head_workspace_size(), dtype=torch.uint8, device=dev)
    ms = time_loop(lambda i: rk.lm_head(h[:Td], W, out=logits, workspace=wsl, stream=stream), 5,
                   stream)
    tf = 2.0 * Td * H * V / (ms / 1e3) / 1e12
    out["lm_head"] = {"shape": [Td, H, V], "ms_per_call": ms, "bound": "tensor", "achieved": tf,
                      "unit": "TFLOP/s", "peak": peaks["bf16_tflops"],
                      "frac": tf / peaks["bf16_tflops"], "peak_source": "burst bf16"}
    # logits-path backward (read bf16 logits, write fp32 dlogits), rotated inputs
    g = torch.randn(Tl, device=dev)
    lses = [rk.logp_from_logits(z, t, stream=stream)[1] for z, t in zs]
    dl = torch.empty((Tl, Vl), dtype=torch.float32, device=dev)

    def lbwd(i):
        z, t = zs[i % len(zs)]
        rk.logp_from_logits_bwd(z, t, lses[i % len(zs)], g, out=dl, stream=stream)
    ms = time_loop(lbwd, 40, stream)
    nbytes = Tl * Vl * 2 + Tl * Vl * 4 + Tl * 16
    gbs = nbytes / (ms / 1e3) / 1e9
    out["logits_bwd"] = {"shape": [Tl, Vl], "ms_per_call": ms, "bound": "hbm", "achieved": gbs,
                         "unit": "GB/s", "peak": peaks["hbm_gbs"], "frac": gbs / peaks["hbm_gbs"],
                         "bytes_per_call": nbytes}
    # per-token GRPO loss on the group's rows
    lp = torch.randn(T, device=dev) - 3
    lpo = lp + 0.1 * torch.randn(T, device=dev)
    lpr = lp + 0.1 * torch.randn(T, device=dev)
    adv = torch.randn(T, device=dev)
    ms = time_loop(lambda i: rk.grpo_token_loss(lp, lpo, adv, tg, logp_ref=lpr, beta=0.04,
                                                stream=stream), 40, stream)
    nbytes = T * (4 * 4 + 8 + 4 * 4)
    gbs = nbytes / (ms / 1e3) / 1e9
    out["grpo_token_loss"] = {"T": T, "ms_per_call": ms, "bound": "hbm", "achieved": gbs,
                              "unit": "GB/s", "peak": peaks["hbm_gbs"],
                              "frac": gbs / peaks["hbm_gbs"], "bytes_per_call": nbytes,
                              "note": "2.6 MB per call: launch-latency bound"}
    out["decode_greedy_T64"] = measure_decode(rk, h[:64].clone(), W, dev)
    # fused greedy step on the whole group
    wsg = torch.empty(rk.linear_greedy_workspace_size(T, H, V), dtype=torch.uint8, device=dev)
    ms = time_loop(lambda i: rk.linear_greedy(h, W, workspace=wsg, stream=stream), 3, stream)
    tf = 2.0 * T * H * V / (ms / 1e3) / 1e12
    out["linear_greedy"] = {"shape": [T, H, V], "ms_per_call": ms, "bound": "tensor",
                            "achieved": tf, "unit": "TFLOP/s",
                            "peak": peaks["bf16_tflops_sustained"],
                            "frac": tf / peaks["bf16_tflops_sustained"]}
    del logits, dl, wsg
    # weight gradient on the whole group: dZ recomputed over the canonical
    # tokens + the dW GEMM (K = tokens), 4*T*H*V flop
    g = torch.randn(T, device=dev)
    _, lse = rk.linear_logp(h, W, tg, stream=stream)
    wsd = torch.empty(rk.linear_logp_dw_workspace_size(T, H, V), dtype=torch.uint8, device=dev)
    dW = torch.empty((V, H), dtype=torch.float32, device=dev)
    ms = time_loop(lambda i: rk.linear_logp_dw(h, W, tg, lse, g, dW=dW, workspace=wsd,
                                               stream=stream), 3, stream)
    tf = 4.0 * T * H * V / (ms / 1e3) / 1e12
    out["linear_logp_dw"] = {"shape": [T, H, V], "ms_per_call": ms, "bound": "tensor",
                             "achieved": tf, "unit": "TFLOP/s",
                             "peak": peaks["bf16_tflops_sustained"],
                             "frac": tf / peaks["bf16_tflops_sustained"],
                             "algorithmic": "4*T*H*V flop (dZ recompute + dZ^T h)"}
    # the same with Zipf(1.1)-distributed targets (seeded), as common tokens
    # repeat in real batches: long entry lists on a few vocabulary rows
    import numpy as np
    rng = np.random.default_rng(11)
    pz = np.arange(1, V + 1, dtype=np.float64) ** -1.1
    tz = torch.as_tensor(rng.choice(V, size=T, p=pz / pz.sum()), dtype=torch.int64).to(dev)
    _, lsez = rk.linear_logp(h, W, tz, stream=stream)
    ms = time_loop(lambda i: rk.linear_logp_dw(h, W, tz, lsez, g, dW=dW, workspace=wsd,
                                               stream=stream), 3, stream)
    tf = 4.0 * T * H * V / (ms / 1e3) / 1e12
    out["linear_logp_dw_zipf_targets"] = {
        "shape": [T, H, V], "ms_per_call": ms, "bound": "tensor", "achieved": tf,
        "unit": "TFLOP/s", "peak": peaks["bf16_tflops_sustained"],
        "frac": tf / peaks["bf16_tflops_sustained"],
        "top_target_count": int(torch.bincount(tz).max().item())}
    del tz, lsez
    # the whole backward (dh + dW) from one shared softmax pass, 6*T*H*V flop
    del wsd
    wsd = torch.empty(rk.linear_logp_bwd_full_workspace_size(T, H, V), dtype=torch.uint8,
                      device=dev)
    dh = torch.empty((T, H), dtype=torch.float32, device=dev)
    ms = time_loop(lambda i: rk.linear_logp_bwd_full(h, W, tg, lse, g, dh=dh, dW=dW, workspace=wsd,
                                                     stream=stream), 3, stream)
    tf = 6.0 * T * H * V / (ms / 1e3) / 1e12
    out["linear_logp_bwd_full"] = {"shape": [T, H, V], "ms_per_call": ms, "bound": "tensor",
                                   "achieved": tf, "unit": "TFLOP/s",
                                   "peak": peaks["bf16_tflops_sustained"],
                                   "frac": tf / peaks["bf16_tflops_sustained"],
                                   "algorithmic": "6*T*H*V flop (dZ + dh + dW GEMMs)"}
    # the same from the forward's saved terms (read only): dZ converted, not
    # recomputed; the forward that keeps them is timed with it: 6*T*H*V flop
    # of GEMMs in the recompute form against 4*T*H*V here (fwd, dh, dW)
    saved = torch.empty(rk.linear_logp_saved_size(T, H, V), dtype=torch.uint8, device=dev)

    def full_saved(i):
        rk.linear_logp_fwd_saved(h, W, tg, lse=lse, saved=saved, stream=stream)
        rk.linear_logp_bwd_full_saved(h, W, tg, lse, g, saved, dh=dh, dW=dW, workspace=wsd,
                                      stream=stream)
    ms = time_loop(full_saved, 3, stream)
    tf = 6.0 * T * H * V / (ms / 1e3) / 1e12
    out["linear_logp_fwd_bwd_full_saved"] = {
        "shape": [T, H, V], "ms_per_call": ms, "tokens_per_s": T / (ms / 1e3), "bound": "tensor",
        "achieved_equiv": tf, "unit": "TFLOP/s",
        "algorithmic": "forward + dh + dW: 6*T*H*V flop of GEMMs in the recompute form, 4*T*H*V "
                       "in this one (no dZ GEMM); achieved_equiv counts 6*T*H*V",
        "note": "compare with linear_logp_bwd_full (backward alone, recompute) + the forward"}
    del wsd, dW, dh, saved
    # the backward that recomputes z with a second GEMM (no saved terms):
    # forward + backward, 6*T*H*V flop
    wsf = torch.empty(rk.linear_logp_workspace_size(T, H, V), dtype=torch.uint8, device=dev)
    wsb = torch.empty(rk.linear_logp_bwd_workspace_size(T, H, V), dtype=torch.uint8, device=dev)
    lp = torch.empty(T, dtype=torch.float32, device=dev)
    ls = torch.empty(T, dtype=torch.float32, device=dev)
    dh = torch.empty((T, H), dtype=torch.float32, device=dev)
    g1 = torch.randn(T, device=dev)

    def recompute_step(i):
        rk.linear_logp(h, W, tg, out=lp, lse=ls, workspace=wsf, stream=stream)
        rk.linear_logp_bwd(h, W, tg, ls, g1, dh=dh, workspace=wsb, stream=stream)
    ms = time_loop(recompute_step, 3, stream)
    tf = 6.0 * T * H * V / (ms / 1e3) / 1e12
    out["linear_logp_fwd_bwd_recompute"] = {
        "shape": [T, H, V], "ms_per_call": ms, "tokens_per_s": T / (ms / 1e3), "bound": "tensor",
        "achieved": tf, "unit": "TFLOP/s", "peak": peaks["bf16_tflops_sustained"],
        "frac": tf / peaks["bf16_tflops_sustained"],
        "algorithmic": "6*T*H*V flop (fwd, z recompute, dZ.W)"}
    del wsf, wsb, dh
    out.update(measure_config_rows(rk, peaks, dev, stream))
    return out


def measure_decode(rk, h, W, dev) -> dict:
    """A greedy decode step (one new token for each of 64 sequences), as a
    serving loop runs it: each step synchronised.  The same call eager and
    captured once in a CUDA graph and replayed; both give the same bits."""
    import torch
    T, H, V = h.shape[0], h.shape[1], W.shape[0]
    cs = torch.cuda.Stream(dev)
    ws = torch.empty(rk.linear_greedy_workspace_size(T, H, V), dtype=torch.uint8, device=dev)
    cs.wait_stream(torch.cuda.current_stream(dev))

    def greedy():
        return rk.linear_greedy(h, W, workspace=ws, stream=cs)
    for _ in range(5):
        ref = greedy()
    cs.synchronize()
    n = 200
    t0 = time.perf_counter()
    for _ in range(n):
        greedy()
        cs.synchronize()
    eager_us = (time.perf_counter() - t0) / n * 1e6
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cs):
        cap = greedy()
    with torch.cuda.stream(cs):
        for _ in range(5):
            graph.replay()
    cs.synchronize()
    same = bool(torch.equal(cap[0], ref[0]) and torch.equal(cap[1].view(torch.int32),
                                                             ref[1].view(torch.int32)))
    t0 = time.perf_counter()
    with torch.cuda.stream(cs):
        for _ in range(n):
            graph.replay()
            cs.synchronize()
    graph_us = (time.perf_counter() - t0) / n * 1e6
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(cs):
        a.record(cs)
        for _ in range(n):
            graph.replay()
        b.record(cs)
    b.synchronize()
    dev_us = a.elapsed_time(b) / n * 1e3
    del graph
    return {"shape": [T, H, V], "eager_us_per_step": eager_us, "graph_us_per_step": graph_us,
            "device_us_per_step": dev_us, "graph_bits_equal_eager": same,
            "timing": "host wall clock per step, each step synchronised (eager: the Python "
                      "binding's call; graph: one replay); device: back-to-back replays, "
                      "CUDA events"}


def measure_config_rows(rk, peaks, dev, stream) -> dict:
    """linear_logp forward on the Llama- and Qwen-shaped workloads: tokens/s
    and the fraction of the burst bf16 rate (each a loop of a few calls), with
    the work counted on active tokens only (2*H*V flop per active token)."""
    import torch

    from invariant_rl_logprob_gb300 import synth
    out = {}

    def fwd_row(lay, W, n_calls):
        h, tg = lay.h.to(dev), lay.targets.to(dev)
        cu = lay.cu_seqlens.to(dev) if lay.cu_seqlens is not None else None
        T, H, V = h.shape[0], h.shape[1], W.shape[0]
        act = lay.targets >= 0
        if lay.cu_seqlens is not None:
            r = torch.arange(T)
            act &= (r >= int(lay.cu_seqlens[0])) & (r < int(lay.cu_seqlens[-1]))
        n_act = int(act.sum())
        ws = torch.empty(rk.linear_logp_workspace_size(T, H, V), dtype=torch.uint8, device=dev)
        logp = torch.empty(T, dtype=torch.float32, device=dev)
        lse = torch.empty(T, dtype=torch.float32, device=dev)
        ms = time_loop(lambda i: rk.linear_logp(h, W, tg, cu, out=logp, lse=lse, workspace=ws,
                                                stream=stream), n_calls, stream)
        tf = 2.0 * n_act * H * V / (ms / 1e3) / 1e12
        return {"rows": T, "active_tokens": n_act, "H": H, "V": V, "ms_per_call": ms,
                "active_tokens_per_s": n_act / (ms / 1e3), "bound": "tensor", "achieved": tf,
                "unit": "TFLOP/s", "peak": peaks["bf16_tflops"],
                "frac": tf / peaks["bf16_tflops"], "peak_source": "burst bf16",
                "algorithmic": "2*H*V flop per active token"}

    pool = synth.llama_pool()
    W = pool.W.to(dev)
    lay = synth.packed(pool, list(range(len(pool.lengths))))
    out["llama_fwd_varlen"] = fwd_row(lay, W, 10)
    out["llama_fwd_varlen"]["sequences"] = len(pool.lengths)
    del W, pool, lay
    pool = synth.qwen_pool()
    W = pool.W.to(dev)
    out["qwen_fwd_padded_b8"] = fwd_row(synth.padded(pool, list(range(8)), 2048), W, 10)
    out["qwen_fwd_packed_seqs0_7"] = fwd_row(synth.packed(pool, list(range(8))), W, 10)
    del W, pool
    torch.cuda.empty_cache()
    return out


def run_gpu(args) -> None:
    import torch

    import invariant_rl_logprob_gb300 as rk
    from invariant_rl_logprob_gb300 import build as rk_build

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)
    if rank == 0 or ws == 1:
        rk_build.build()
    barrier(ws)
    rk.load_library()
    peaks = load_peaks()

    pool, logits_host = make_inputs(rank)
    T, H, V = pool.h.shape[0], pool.H, pool.V
    Tl, Vl = LOGITS["T"], LOGITS["V"]
    stream = torch.cuda.current_stream(dev)

    h = pool.h.to(dev)
    W = pool.W.to(dev)
    tg = pool.targets.to(dev)
    g = pool.g.to(dev)
    zs = [(z.to(dev), t.to(dev)) for z, t in logits_host]
    logp = torch.empty(T, dtype=torch.float32, device=dev)
    lse = torch.empty(T, dtype=torch.float32, device=dev)
    dh = torch.empty((T, H), dtype=torch.float32, device=dev)
    zlogp = torch.empty(Tl, dtype=torch.float32, device=dev)
    zlse = torch.empty(Tl, dtype=torch.float32, device=dev)
    saved = torch.empty(rk.linear_logp_saved_size(T, H, V), dtype=torch.uint8, device=dev)
    ws_bwd = torch.empty(rk.linear_logp_bwd_saved_workspace_size(T, H, V), dtype=torch.uint8,
                         device=dev)
    # fwd: live row blocks, tile kernel, merge; bwd: stash -> dZ, exact
    # entries, entry sort, dh tile kernel, bad-target / skipped rows; logits: 1
    launches_per_step = 3 + 5 + 1

    def fwd(hh, tt, lp, ls):
        rk.linear_logp_fwd_saved(hh, W, tt, out=lp, lse=ls, saved=saved, stream=stream)

    def bwd(hh, tt, ls, gg, dd):
        rk.linear_logp_bwd_saved(hh, W, tt, ls, gg, saved, dh=dd, workspace=ws_bwd, stream=stream)

    def step(i):
        fwd(h, tg, logp, lse)
        bwd(h, tg, lse, g, dh)
        z, zt = zs[i % len(zs)]
        rk.logp_from_logits(z, zt, out=zlogp, lse=zlse, stream=stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    err = rk.get_device_error(stream)
    if err:
        raise RuntimeError(f"device error word {err:#x} during warm-up")

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    barrier(ws)
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index) as clk:
        t_wall = time.perf_counter()
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for i in range(args.steps):
            e = ev[i]
            e[0].record(stream)
            fwd(h, tg, logp, lse)
            e[1].record(stream)
            bwd(h, tg, lse, g, dh)
            e[2].record(stream)
            z, zt = zs[(args.warmup + i) % len(zs)]
            rk.logp_from_logits(z, zt, out=zlogp, lse=zlse, stream=stream)
            e[3].record(stream)
        end.record(stream)
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - t_wall
    barrier(ws)
    total_ms = start.elapsed_time(end)
    fwd_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / args.steps
    bwd_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / args.steps
    lg_ms = sum(e[2].elapsed_time(e[3]) for e in ev) / args.steps
    err = rk.get_device_error(stream)
    if err:
        raise RuntimeError(f"device error word {err:#x} in the timed region")

    # the logits path on its own: loops over the rotated buffers (each call's
    # input is absent from L2), repeated right after the step loop, while the
    # SM clock is still recovering from the power-capped GEMMs, and on; each
    # repeat carries the SM clock measured on the device around it
    lg_reps = 50
    lg_runs = []
    for r in range(LOGITS_REPEATS):
        f0 = sm_clock_mhz(stream)
        ls0 = torch.cuda.Event(enable_timing=True)
        ls1 = torch.cuda.Event(enable_timing=True)
        hold_stream(stream, 2.0)
        ls0.record(stream)
        for i in range(lg_reps):
            z, zt = zs[i % len(zs)]
            rk.logp_from_logits(z, zt, out=zlogp, lse=zlse, stream=stream)
        ls1.record(stream)
        f1 = sm_clock_mhz(stream)
        lg_runs.append({"us_per_call": ls0.elapsed_time(ls1) * 1000.0 / lg_reps,
                        "sm_mhz_before": round(f0), "sm_mhz_after": round(f1)})
    torch.cuda.synchronize(dev)
    lg_us = sorted(r["us_per_call"] for r in lg_runs)
    lg_loop_ms = statistics.median(lg_us) / 1000.0

    dh_order = rk.last_tile_order("dh")
    ms_step_local = total_ms / args.steps
    ms_step = max_over_ranks(ms_step_local, ws)
    value = ws * T / (ms_step / 1000.0)

    # ---- end to end: host buffers in, results out, through the public API ----
    # Every step copies its inputs from pinned host memory and its results
    # back.  Four device buffer sets: the inputs of step i+3 (host-to-device
    # stream) and the results of step i-1 (device-to-host stream) move while
    # step i computes, so each copy has three steps to finish.  Events around
    # every copy showed single copies slowed by the shared host from 6-9 ms to
    # 65-150 ms, once or twice a run; with two sets such a copy stalled the
    # loop by up to 42 ms.  (With one stream for both directions the loop
    # stalled for 12-24 ms every few steps.)
    pin = lambda t: t.pin_memory()
    h_h, W_h, tg_h, g_h = pin(pool.h), pin(pool.W), pin(pool.targets), pin(pool.g)
    z_h = [(pin(z), pin(t)) for z, t in logits_host]
    dh_h = torch.empty((T, H), dtype=torch.float32).pin_memory()
    logp_h = torch.empty(T, dtype=torch.float32).pin_memory()
    zlogp_h = torch.empty(Tl, dtype=torch.float32).pin_memory()
    h2d = (h_h.numel() * 2 + W_h.numel() * 2 + tg_h.numel() * 8 + g_h.numel() * 4
           + Tl * Vl * 2 + Tl * 8)
    d2h = dh_h.numel() * 4 + logp_h.numel() * 4 + zlogp_h.numel() * 4
    sets = [dict(h=h, W=W, tg=tg, g=g, z=zs[0][0], zt=zs[0][1], logp=logp, lse=lse, dh=dh,
                 zlogp=zlogp, zlse=zlse)]
    n_sets = 4
    for _ in range(n_sets - 1):
        sets.append(dict(h=torch.empty_like(h), W=torch.empty_like(W), tg=torch.empty_like(tg),
                         g=torch.empty_like(g), z=torch.empty_like(zs[0][0]),
                         zt=torch.empty_like(zs[0][1]), logp=torch.empty_like(logp),
                         lse=torch.empty_like(lse), dh=torch.empty_like(dh),
                         zlogp=torch.empty_like(zlogp), zlse=torch.empty_like(zlse)))
    in_stream = torch.cuda.Stream(dev)
    out_stream = torch.cuda.Stream(dev)

    def h2d_into(b, i):
        zh, zth = z_h[i % len(z_h)]
        b["h"].copy_(h_h, non_blocking=True)
        b["W"].copy_(W_h, non_blocking=True)
        b["tg"].copy_(tg_h, non_blocking=True)
        b["g"].copy_(g_h, non_blocking=True)
        b["z"].copy_(zh, non_blocking=True)
        b["zt"].copy_(zth, non_blocking=True)

    def compute(b):
        rk.linear_logp_fwd_saved(b["h"], b["W"], b["tg"], out=b["logp"], lse=b["lse"],
                                 saved=saved, stream=stream)
        rk.linear_logp_bwd_saved(b["h"], b["W"], b["tg"], b["lse"], b["g"], saved, dh=b["dh"],
                                 workspace=ws_bwd, stream=stream)
        rk.logp_from_logits(b["z"], b["zt"], out=b["zlogp"], lse=b["zlse"], stream=stream)

    def d2h_from(b):
        dh_h.copy_(b["dh"], non_blocking=True)
        logp_h.copy_(b["logp"], non_blocking=True)
        zlogp_h.copy_(b["zlogp"], non_blocking=True)

    def e2e_run(n_steps):
        in_ready = [torch.cuda.Event() for _ in range(n_sets)]
        done = [torch.cuda.Event() for _ in range(n_sets)]
        out_read = [torch.cuda.Event() for _ in range(n_sets)]
        with torch.cuda.stream(in_stream):
            for j in range(min(n_sets - 1, n_steps)):  # the first steps' inputs
                h2d_into(sets[j], j)
                in_ready[j].record(in_stream)
        for i in range(n_steps):
            b = sets[i % n_sets]
            stream.wait_event(in_ready[i % n_sets])
            if i >= n_sets:
                stream.wait_event(out_read[i % n_sets])    # step i-n_sets's results read out
            compute(b)
            done[i % n_sets].record(stream)
            k = i + n_sets - 1  # the step whose inputs go in now
            if k < n_steps:
                with torch.cuda.stream(in_stream):
                    if k >= n_sets:
                        in_stream.wait_event(done[k % n_sets])  # step k-n_sets done with the set
                    c0 = torch.cuda.Event(enable_timing=True)
                    c0.record(in_stream)
                    h2d_into(sets[k % n_sets], k)
                    c1 = torch.cuda.Event(enable_timing=True)
                    c1.record(in_stream)
                    copy_ev["h2d"].append((c0, c1))
                    in_ready[k % n_sets].record(in_stream)
            with torch.cuda.stream(out_stream):
                out_stream.wait_event(done[i % n_sets])
                c0 = torch.cuda.Event(enable_timing=True)
                c0.record(out_stream)
                d2h_from(b)
                c1 = torch.cuda.Event(enable_timing=True)
                c1.record(out_stream)
                copy_ev["d2h"].append((c0, c1))
                out_read[i % n_sets].record(out_stream)
        stream.wait_stream(in_stream)
        stream.wait_stream(out_stream)

    copy_ev = {"h2d": [], "d2h": []}  # per-copy events (the copies' own durations)
    e2e_run(2)
    torch.cuda.synchronize(dev)
    copy_ev = {"h2d": [], "d2h": []}
    barrier(ws)
    s2 = torch.cuda.Event(enable_timing=True)
    e2 = torch.cuda.Event(enable_timing=True)
    s2.record(stream)
    e2e_run(args.steps)
    e2.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(s2.elapsed_time(e2) / args.steps, ws)
    e2e_value = ws * T / (e2e_ms / 1000.0)
    copy_ms = {}
    for key, evs in copy_ev.items():
        d = sorted(a.elapsed_time(b) for a, b in evs)
        if d:
            copy_ms[key] = {"median": statistics.median(d), "max": d[-1], "n": len(d)}
    err = rk.get_device_error(stream)
    if err:
        raise RuntimeError(f"device error word {err:#x} in the end-to-end loop")

    if rank != 0:
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    flops_fwd = 2.0 * T * H * V   # z = h W^T with the fused softmax partials
    flops_bwd = 2.0 * T * H * V   # dh = dZ W (dZ from the saved terms, no z recompute)
    tc_tflops = (flops_fwd + flops_bwd) / ((fwd_ms + bwd_ms) / 1000.0) / 1e12
    peak_tc = peaks["bf16_tflops_sustained"]
    lg_bytes = Tl * Vl * 2 + Tl * 8 + 2 * Tl * 4
    lg_gbs = lg_bytes / (lg_loop_ms / 1000.0) / 1e9
    lg_gbs_step = lg_bytes / (lg_ms / 1000.0) / 1e9
    traffic = None
    if (TRAFFIC_RECORD["source_sha1"] == kernel_source_sha1()
            and (T, H, V) == (65536, 4096, 128256)):
        traffic = TRAFFIC_RECORD["bytes_per_step"]

    rows = None
    if not args.no_rows:
        rows = measure_rows(rk, pool, zs, peaks, dev, stream)

    cpu = None
    if not args.no_cpu_baseline:
        v, cores, desc = cpu_oracle_sample(pool, logits_host, args.cpu_rows)
        cpu = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc}

    clocks = clk.summary()
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "global_batch": ws * T, "seq_len": GRPO["seq_len"],
                   "H": H, "V": V, "parallelism": f"replicas x{ws}" if ws > 1 else "single",
                   "l2": "inputs larger than L2 (h 512 MB, W 1.05 GB); logits rotated over "
                         f"{N_LOGITS_BUFFERS} buffers of {Tl * Vl * 2 / 1e6:.0f} MB"},
        "roofline": {"bound": "tensor", "achieved": tc_tflops, "peak": peak_tc,
                     "unit": "TFLOP/s", "frac": tc_tflops / peak_tc, "traffic": traffic,
                     "kernel": "linear_logp_tiles (the forward launch and the dh GEMM launch, "
                               "each timed with the rest of its call: the backward call also "
                               "holds the HBM-bound pass that turns the saved terms into dZ)",
                     "algorithmic": "4*T*H*V flop per step (2 fwd + 2 dZ.W)",
                     "traffic_unit": "DRAM bytes per step (2 tile launches, ncu)",
                     "traffic_per_launch_gb": TRAFFIC_RECORD["per_launch_gb"] if traffic else None,
                     "algorithmic_bytes": algorithmic_bytes_per_step(T, H, V),
                     "peak_source": f"{peaks['source']} bf16_tflops_sustained"},
        "components_ms": {"linear_logp_fwd_saved": fwd_ms, "linear_logp_bwd_saved": bwd_ms,
                          "logits_path": lg_ms},
        "fwd_tflops": flops_fwd / (fwd_ms / 1000.0) / 1e12,
        "bwd_tflops": flops_bwd / (bwd_ms / 1000.0) / 1e12,
        "logits_path": {"bound": "hbm", "achieved": lg_gbs, "peak": peaks["hbm_gbs"],
                        "unit": "GB/s", "frac": lg_gbs / peaks["hbm_gbs"],
                        "bytes_per_call": lg_bytes, "us_per_call": lg_loop_ms * 1000.0,
                        "tokens_per_s": Tl / (lg_loop_ms / 1000.0),
                        "us_per_call_min_median_max": [lg_us[0], statistics.median(lg_us),
                                                       lg_us[-1]],
                        "repeats": lg_runs,
                        "timing": f"median of {LOGITS_REPEATS} loops of {lg_reps} back-to-back "
                                  f"calls over {N_LOGITS_BUFFERS} rotated buffers, the first "
                                  "right after the step loop (CUDA events on the launching "
                                  "stream; queued behind a device-side wait); SM clock measured "
                                  "on the device before and after each loop",
                        "in_step": {"us_per_call": lg_ms * 1000.0, "achieved": lg_gbs_step,
                                    "frac": lg_gbs_step / peaks["hbm_gbs"],
                                    "note": "one call between two events in each step, right "
                                            "after the backward call (at the clock the power-"
                                            "capped GEMMs leave, and with no neighbouring call "
                                            "to hide its launch)"}},
        "rows": rows,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "copy_ms": copy_ms,
                "how": "pinned host -> device copies of every step's inputs and device -> "
                       "host copies of its dh/logp, each direction on its own stream, "
                       "four buffer sets against the compute stream (each copy has three "
                       "steps to finish); timed from the first "
                       "copy to the last"},
        "dh_tile_order": {2: "rounds (cooperative launch)", 1: "tiles from a counter"}.get(
            dh_order, "none"),
        "gpu_launches": launches_per_step * args.steps,
        "gpu_launches_note": f"{launches_per_step} librk kernels per step x {args.steps} steps "
                             "in the timed region",
        "clocks": clocks,
        "wall_s_timed": wall,
        "device": torch.cuda.get_device_name(dev),
    }
    print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_case(args) -> None:
    """One operator, a few launches, on a small workload (profiling)."""
    import torch

    import invariant_rl_logprob_gb300 as rk
    from invariant_rl_logprob_gb300 import build as rk_build
    from invariant_rl_logprob_gb300 import synth
    rk_build.build()
    dev = torch.device("cuda", 0)
    T, H, V = (int(x) for x in args.shape.split(","))
    if args.case in ("qwen_padded", "qwen_packed"):
        # the Qwen-shaped forward on sequences 0-7: [8, 2048] right-padded
        # (256-row blocks of padding skipped) or varlen-packed
        pool = synth.qwen_pool()
        seqs = list(range(8))
        lay = (synth.padded(pool, seqs, 2048) if args.case == "qwen_padded"
               else synth.packed(pool, seqs))
        W = pool.W.to(dev)
        h, tg = lay.h.to(dev), lay.targets.to(dev)
        cu = lay.cu_seqlens.to(dev) if lay.cu_seqlens is not None else None
        T, H, V = h.shape[0], h.shape[1], W.shape[0]
        fn = lambda: rk.linear_logp(h, W, tg, cu)
        n_act = sum(len(lay.rows_of[i]) for i in seqs)
        work = f"{2.0 * n_act * H * V / 1e12:.3f} TFLOP on {n_act} active of {T} rows"
    elif args.case in ("logits", "logits_bwd"):
        z, tg, _ = synth.logits_batch(T=T, V=V)
        z, tg = z.to(dev), tg.to(dev)
        if args.case == "logits":
            fn = lambda: rk.logp_from_logits(z, tg)
            nbytes = T * V * 2 + T * 16
        else:
            _, lse = rk.logp_from_logits(z, tg)
            g = torch.randn(T, device=dev)
            dl = torch.empty((T, V), dtype=torch.float32, device=dev)
            fn = lambda: rk.logp_from_logits_bwd(z, tg, lse, g, out=dl)
            nbytes = T * V * 6 + T * 16
        work = f"{nbytes / 1e6:.1f} MB"
    else:
        pool = synth.make_pool(H, V, [T], seed=4, with_grad=True)
        h, W, tg, g = (pool.h.to(dev), pool.W.to(dev), pool.targets.to(dev), pool.g.to(dev))
        _, lse = rk.linear_logp(h, W, tg)
        if args.case == "fwd":
            fn = lambda: rk.linear_logp(h, W, tg)
            flops = 2.0 * T * H * V
        elif args.case == "dw":
            ws = torch.empty(rk.linear_logp_dw_workspace_size(T, H, V), dtype=torch.uint8,
                             device=dev)
            dW = torch.empty((V, H), dtype=torch.float32, device=dev)
            fn = lambda: rk.linear_logp_dw(h, W, tg, lse, g, dW=dW, workspace=ws)
            flops = 4.0 * T * H * V
        elif args.case == "saved":
            # forward that keeps its softmax terms + the backward from them
            saved = torch.empty(rk.linear_logp_saved_size(T, H, V), dtype=torch.uint8, device=dev)
            wsb = torch.empty(rk.linear_logp_bwd_saved_workspace_size(T, H, V), dtype=torch.uint8,
                              device=dev)
            dh = torch.empty((T, H), dtype=torch.float32, device=dev)

            def fn():
                _, lse_s, _ = rk.linear_logp_fwd_saved(h, W, tg, saved=saved)
                rk.linear_logp_bwd_saved(h, W, tg, lse_s, g, saved, dh=dh, workspace=wsb)
            flops = 4.0 * T * H * V
        elif args.case == "full_saved":
            # forward that keeps its softmax terms + dh and dW from them
            saved = torch.empty(rk.linear_logp_saved_size(T, H, V), dtype=torch.uint8, device=dev)
            ws = torch.empty(rk.linear_logp_bwd_full_workspace_size(T, H, V), dtype=torch.uint8,
                             device=dev)
            dW = torch.empty((V, H), dtype=torch.float32, device=dev)
            dh = torch.empty((T, H), dtype=torch.float32, device=dev)

            def fn():
                _, lse_s, _ = rk.linear_logp_fwd_saved(h, W, tg, saved=saved)
                rk.linear_logp_bwd_full_saved(h, W, tg, lse_s, g, saved, dh=dh, dW=dW, workspace=ws)
            flops = 6.0 * T * H * V
        elif args.case == "full":
            ws = torch.empty(rk.linear_logp_bwd_full_workspace_size(T, H, V), dtype=torch.uint8,
                             device=dev)
            dW = torch.empty((V, H), dtype=torch.float32, device=dev)
            dh = torch.empty((T, H), dtype=torch.float32, device=dev)
            fn = lambda: rk.linear_logp_bwd_full(h, W, tg, lse, g, dh=dh, dW=dW, workspace=ws)
            flops = 6.0 * T * H * V
        else:
            ws = torch.empty(rk.linear_logp_bwd_workspace_size(T, H, V), dtype=torch.uint8,
                             device=dev)
            fn = lambda: rk.linear_logp_bwd(h, W, tg, lse, g, workspace=ws)
            flops = 4.0 * T * H * V
        work = f"{flops / 1e12:.3f} TFLOP"
    for _ in range(2):
        fn()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(args.reps):
        fn()
    e.record()
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / args.reps
    if rk.get_device_error():
        raise RuntimeError("device error word set")
    print(json.dumps({"case": args.case, "shape": [T, H, V], "reps": args.reps,
                      "ms_per_call": ms, "work": work}))


def main() -> None:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-rows", type=int, default=2,
                    help="GRPO rows (and logits-path rows) per host core in the oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-rows", action="store_true",
                    help="skip the separate timing of the widened rows")
    ap.add_argument("--case", choices=["fwd", "bwd", "logits", "logits_bwd", "dw", "full", "saved",
                                       "qwen_padded", "qwen_packed",
                                       "full_saved"],
                    default=None)
    ap.add_argument("--shape", default="2048,4096,32000")
    ap.add_argument("--reps", type=int, default=3)
    args = ap.parse_args()
    if args.case:
        run_case(args)
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
