"""Benchmark of the REINFORCE Zero learner step (fused logprob + unclipped
token-level IS loss, forward and backward) on synthetic workloads shaped like
the pages' runs.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
                  [--impl ours|reference]

One step = group advantages + the learner step over one batch already
resident in HBM (H, W, tokens, the rollout's recorded log mu and log-sum-exp
of every row, cu_seqlens, rewards), through rz_loss_fwd_bwd_ref (the kept
softmax terms taken against the recorded log-sum-exp: no dz pass); the same
step through rz_loss_fwd_bwd is timed beside it (`plain_route`).  Inputs (H
alone is 3.3-5.7 GB) are far larger than L2, so no flush is needed between
steps.  Rank 0 prints one JSON line.  Under torchrun each rank runs its own
shard of the batch (rz_loss_fwd_bwd_shard) and the step includes the
fixed-order exchange of dW; the max time over ranks counts.
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM bytes (read + write) per launch of the roofline kernel of each bench
# workload, from an ncu capture of that kernel (the committed ncu summary
# gives the command).  A figure is reported only while the kernel's sources
# hash to the value recorded with it; otherwise the line carries null.
GEMM_SOURCES = ["rz_gemm.cuh", "rz_lmhead.cu", "rz_lse.cuh", "rz_ptx.cuh", "rz_math.cuh",
                "rz_internal.h"]
LOGITS_SOURCES = ["rz_logits.cu", "rz_ptx.cuh", "rz_math.cuh", "rz_internal.h"]
TRAFFIC_CAPTURES = {
    # learner keep GEMM taking the terms against the recorded log-sum-exp, one
    # 38,912-row chunk at the 4B shape: 2.321 GB read + 2.932 GB written at
    # 9,728 rows (one raster group of 76 m-blocks); a 38,912-row chunk is four
    # such groups (x4).  Its operand re-reads vary from capture to capture
    # (1.94-2.36 GB read at 9,728 rows on the same kernel code).
    "qwen4b_lag64": {"bytes": 4 * (2.320705536e9 + 2.931853824e9), "sources": GEMM_SOURCES,
                     "sources_sha256_16": "c6598b72eec7cb31"},
    # given-logits row kernel (768 threads, two rows per SM): 5.414 GB read
    # + 4.893 GB written at 16,384 rows, scaled to the workload's 262,144
    # rows (x16)
    "moe30b_logits": {"bytes": 16 * (5.414485504e9 + 4.892578816e9), "sources": LOGITS_SOURCES,
                      "sources_sha256_16": "47be4dfd2aa2d274"},
}


def sources_hash(files):
    """Hash of the kernel sources with comments and blank space removed, so a
    comment edit does not retire a capture of unchanged code."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "invariant_logprobs_gb300", "csrc", f)) as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def captured_traffic(workload):
    cap = TRAFFIC_CAPTURES.get(workload)
    if cap is None or cap["bytes"] is None:
        return None
    try:
        ok = sources_hash(cap["sources"]) == cap["sources_sha256_16"]
    except OSError:
        ok = False
    return cap["bytes"] if ok else None
METRIC = "action tokens/s, fused logprob+IS-loss fwd/bwd (1 GB300); % bf16 tensor roofline"


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed
    region (200 ms period)."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        loaded = [s for s in sm if mx and s > 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ----------------------------------------------------------------- distributed
def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def sum_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return int(t.item())


def gather_over_ranks(x, world):
    if world == 1:
        return [x]
    import torch.distributed as dist
    out = [None] * world
    dist.all_gather_object(out, x)
    return out


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------- CPU oracle leg
def oracle_sample(b, n_tokens):
    """A bounded sample of the workload for the CPU oracle: the first responses
    whose total length reaches n_tokens (whole responses, so the per-response
    means are the workload's own; the last one is cut short if needed).  Its
    recorded log mu and advantages are the oracle's own, from the batch's
    W_mu and rewards (computed here, outside the timed call)."""
    import numpy as np
    import torch
    import oracle
    cu = b["cu"].cpu().numpy()
    B = cu.shape[0] - 1
    k = 1
    while k < B and cu[k] < n_tokens:
        k += 1
    T = min(int(cu[k]), n_tokens)
    cu_s = np.minimum(cu[:k + 1], T)
    f = lambda t: t.to("cpu", torch.float64).numpy()
    H = f(b["H"][:T])
    tokens = b["tokens"][:T].cpu().numpy().astype(np.int64)
    logmu, _ = oracle.token_logprob(H, f(b["W_mu"]), tokens)
    adv = oracle.group_advantage(f(b["rewards"]), b["G"])[:k]
    return {"H": H, "W": f(b["W"]), "tokens": tokens, "logmu": logmu, "cu": cu_s, "adv": adv,
            "T": T}


def logits_oracle_sample(logits, tokens, logmu, cu, rewards, G, n_tokens):
    """The given-logits counterpart of oracle_sample: the first n_tokens rows
    (whole responses where they fit, the last one cut short), bf16 logits
    widened exactly to fp32 on the host; advantages are the oracle's own."""
    import numpy as np
    import torch
    import oracle
    adv = oracle.group_advantage(rewards.to("cpu", torch.float64).numpy(), G)
    cu = cu.cpu().numpy()
    B = cu.shape[0] - 1
    k = 1
    while k < B and cu[k] < n_tokens:
        k += 1
    T = min(int(cu[k]), n_tokens)
    return {"logits": logits[:T].to("cpu", torch.float32).numpy(),
            "tokens": tokens[:T].cpu().numpy(), "logmu": logmu[:T].cpu().double().numpy(),
            "cu": np.minimum(cu[:k + 1], T), "adv": adv[:k], "T": T}


def time_logits_oracle(sample, reps=1):
    import oracle
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.logits_loss_fwd_bwd(sample["logits"], sample["tokens"], sample["logmu"],
                                   sample["cu"], sample["adv"])
    dt = (time.perf_counter() - t0) / reps
    return sample["T"] / dt, dt


def time_oracle(sample, reps=1):
    import oracle
    import numpy as np
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.loss_fwd_bwd(sample["H"], sample["W"], sample["tokens"], sample["logmu"],
                            sample["cu"], sample["adv"])
    dt = (time.perf_counter() - t0) / reps
    return sample["T"] / dt, dt


def cpu_threads():
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(k):
            return int(os.environ[k])
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


# ----------------------------------------------------------------- workloads
def build_learner_batch(name, dev, rank):
    import torch
    import invariant_logprobs_gb300 as rz
    from invariant_logprobs_gb300 import synth
    wl = synth.WORKLOADS[name]
    b = synth.make_batch(wl, device=dev, seed=wl.seed + 7919 * rank)
    # the rollout records log mu and the row's log-sum-exp with its (lagged)
    # weights, in one pass: our own rollout path
    b["lse"] = torch.empty(b["T"], dtype=torch.float32, device=dev)
    b["logmu"], _ = rz.rz_token_logprob(b["H"], b["W_mu"], b["tokens"], lse_out=b["lse"])
    b["adv"] = rz.rz_group_advantage(b["rewards"], b["G"])
    torch.cuda.synchronize()
    return wl, b


def run_ours(args):
    import torch
    import invariant_logprobs_gb300 as rz

    world, rank, local = dist_setup(args)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    rz.load()
    peaks, peak_src = load_peaks()

    if args.config == "moe30b_logits":
        out = measure_logits(args, world, rank, dev, peaks, peak_src, args.steps, args.warmup)
    else:
        out = measure_learner(args, world, rank, local, dev, peaks, peak_src)
    if world == 1 and not args.no_other_workloads:
        torch.cuda.empty_cache()
        out["other_workloads"] = other_workloads(args, rank, dev, peaks, peak_src)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


def other_workloads(args, rank, dev, peaks, peak_src):
    """The other two bench workloads, shorter (3 warm-ups, up to 5 timed
    steps each), so that one default run records all three: the 1.5B-shaped
    learner step and the HBM-bound given-logits step."""
    import torch
    steps = max(2, min(args.steps, 5))
    res = {}
    # first: right after a sustained run of the HBM-bound given-logits step
    # the W-read-bound small batches took 0.255 instead of 0.146 ms for a
    # few seconds
    res["invariance_d2048_rollout"] = rollout_batch_sizes(dev, peaks)
    torch.cuda.empty_cache()
    for name in ("qwen4b_lag64", "qwen1p5b_lag2", "moe30b_logits"):
        if name == args.config:
            continue
        if name == "moe30b_logits":
            r = measure_logits(args, 1, rank, dev, peaks, peak_src, steps, 3, full=False)
            res[name] = {k: r[k] for k in ("value", "unit", "ms_per_step", "steps", "warmup",
                                           "roofline", "step_breakdown", "config")}
        else:
            r = measure_learner(args, 1, rank, dev.index, dev, peaks, peak_src, name=name,
                                steps=steps, warmup=3, full=False)
            res[name] = {k: r[k] for k in ("value", "unit", "ms_per_step", "steps", "warmup",
                                           "algorithmic_tflops",
                                           "algorithmic_frac_of_sustained_bf16", "roofline",
                                           "step_breakdown", "config")}
        torch.cuda.empty_cache()
    return res


def rollout_batch_sizes(dev, peaks, d=2048, V=151936, sizes=(1, 7, 64, 513, 4096), reps=15):
    """rz_token_logprob at the batch sizes of the invariance sweep (d = 2048,
    V = 151936; bitwise batch invariance is a test, this is its speed):
    median device time per call over `reps` calls, each after a 256 MB write
    that pushes W out of L2 (the write-back of the dirty lines it leaves
    behind falls inside the timed call), and the mean over 10 calls issued
    back to back (W, 622 MB, is larger than L2, so each call reads it from
    DRAM again; what one call leaves in L2 is the part of W the next call
    reads last).  Small batches are bound by reading W (V d 2 bytes), so the
    line gives that rate against the measured copy bandwidth; large ones by
    the tensor cores (2 d V flop per row)."""
    import torch
    import invariant_logprobs_gb300 as rz
    g = torch.Generator(device=dev).manual_seed(2004)
    W = (torch.randn(V, d, generator=g, device=dev) * 0.02).to(torch.bfloat16)
    Hb = torch.randn(max(sizes), d, generator=g, device=dev).to(torch.bfloat16)
    tok = torch.randint(0, V, (max(sizes),), generator=g, device=dev, dtype=torch.int32)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    out = {}
    for T in sizes:
        lp = torch.empty(T, device=dev)
        ws = rz.alloc_workspace(rz.RZ_OP_TOKEN_LOGPROB, T, d, V, 0, dev)
        for _ in range(3):
            rz.rz_token_logprob(Hb[:T], W, tok[:T], logprob_out=lp, ws=ws)
        ms = []
        for _ in range(reps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            rz.rz_token_logprob(Hb[:T], W, tok[:T], logprob_out=lp, ws=ws)
            e1.record(stream)
            torch.cuda.synchronize()
            ms.append(e0.elapsed_time(e1))
        m = statistics.median(ms)
        bb = []
        for _ in range(5):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(10):
                rz.rz_token_logprob(Hb[:T], W, tok[:T], logprob_out=lp, ws=ws)
            e1.record(stream)
            torch.cuda.synchronize()
            bb.append(e0.elapsed_time(e1) / 10)
        mb = statistics.median(bb)
        w_gbs = V * d * 2 / (m / 1e3) / 1e9
        wb_gbs = V * d * 2 / (mb / 1e3) / 1e9
        out["T=%d" % T] = {"ms": m, "W_read_GBs": w_gbs, "W_read_frac_of_hbm": w_gbs / peaks["hbm_gbs"],
                           "tflops": 2.0 * d * V * T / (m / 1e3) / 1e12,
                           "ms_back_to_back": mb,
                           "W_read_frac_of_hbm_back_to_back": wb_gbs / peaks["hbm_gbs"]}
    out["note"] = ("ms: median of %d calls after a 256 MB L2 flush each; ms_back_to_back: "
                   "median over 5 runs of the mean of 10 calls issued back to back (W is "
                   "larger than L2); d = %d, V = %d; W_read_* counts W once per call"
                   % (reps, d, V))
    return out


def measure_learner(args, world, rank, local, dev, peaks, peak_src, name=None, steps=None,
                    warmup=None, full=True):
    """The learner step on one workload: `steps` timed steps after `warmup`
    untimed ones, then the per-class breakdown of two more; with `full`, also
    clocks, the rollout entry points, the same-box cuBLAS comparison, the
    end-to-end run and the CPU baseline."""
    import torch
    import invariant_logprobs_gb300 as rz
    name = name or args.config
    steps = args.steps if steps is None else steps
    warmup = args.warmup if warmup is None else warmup
    stream = torch.cuda.current_stream()
    wl, b = build_learner_batch(name, dev, rank)
    T, d, V, B = b["T"], b["d"], b["V"], b["B"]
    ws = rz.alloc_workspace(rz.RZ_OP_LOSS_FWD_BWD_REF, T, d, V, B, dev)
    dH = torch.empty((T, d), dtype=torch.bfloat16, device=dev)
    dW = torch.empty((V, d), dtype=torch.float32, device=dev)
    lp = torch.empty(T, dtype=torch.float32, device=dev)
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    d3 = torch.empty(1, dtype=torch.float32, device=dev)
    adv = torch.empty(B, dtype=torch.float32, device=dev)
    err = rz.new_err_flag(dev)
    # data-parallel over responses: each rank holds B of the batch's
    # B * world responses, normalises by the batch's count and joins the one
    # exchange step (dW in rank order, the loss share and D3 per rank)
    B_total = B * world
    ex_ev = []
    gathered = torch.empty((world, 2), dtype=torch.float32, device=dev)
    dW_sum = {}  # the exchanged dW of the latest step (every rank holds all of it)

    def exchange():
        from invariant_logprobs_gb300 import shard
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        dW_sum["dW"], g = shard.dp_exchange(dW, loss, d3, rz.rz_sum_partials)
        gathered.copy_(g)
        e1.record(stream)
        ex_ev.append((e0, e1))

    def step():
        rz.rz_group_advantage(b["rewards"], b["G"], adv_out=adv)
        if world == 1:
            rz.rz_loss_fwd_bwd_ref(b["H"], b["W"], b["tokens"], b["logmu"], b["lse"], b["cu"],
                                   adv, logprob_out=lp, dH=dH, dW=dW, loss_out=loss,
                                   d3_out=d3, ws=ws, err_flag=err)
        else:
            rz.rz_loss_fwd_bwd_shard(b["H"], b["W"], b["tokens"], b["logmu"], b["cu"], adv,
                                     B_total, logprob_out=lp, dH=dH, dW=dW, loss_out=loss,
                                     d3_out=d3, ws=ws, err_flag=err, ref_lse=b["lse"])
            exchange()

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    clk = ClockSampler(local)
    if full:
        clk.start()
        time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    ev[0].record(stream)
    for k in range(steps):
        step()
        ev[k + 1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    per_step = [ev[k].elapsed_time(ev[k + 1]) for k in range(steps)]
    total_ms = ev[0].elapsed_time(ev[-1])
    exchange_ms = (statistics.mean(a.elapsed_time(z) for a, z in ex_ev[-steps:])
                   if world > 1 else None)

    # the step split by kernel class: two more (untimed) steps with the
    # library's launch-class timing on (CUDA events on the launching stream)
    breakdown = profile_steps(rz, step, stream, 2)
    ms = max_over_ranks(total_ms / steps, world)
    T_all = sum_over_ranks(T, world)
    value = T_all / (ms / 1e3)
    flop_alg = 6.0 * d * V * T
    keep_ms, keep_launches = breakdown["classes"]["keep_gemm"]["ms"], \
        breakdown["classes"]["keep_gemm"]["launches"]
    keep_tf = 2.0 * d * V * T / (keep_ms / 1e3) / 1e12
    for cname in ("keep_gemm", "dH_gemm", "dW_gemm"):
        c = breakdown["classes"][cname]
        c["tflops"] = 2.0 * d * V * T / (c["ms"] / 1e3) / 1e12
    # on this route the library's dz class is the H scaling (sigma_t h_t):
    # 4 bytes per element of H moved
    sc = breakdown["classes"].pop("dz")
    sc["gbs"] = T * d * 4.0 / (sc["ms"] / 1e3) / 1e9
    breakdown["classes"]["scale_rows"] = sc
    out = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": steps, "warmup": warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; shapes and distributions of the workload, random-init weights)",
        "config": {"workload": wl.name, "tokens_per_step": T_all, "responses": B_total,
                   "group": wl.group, "d": d, "V": V, "lag_steps": wl.drift_steps,
                   "l2": "inputs larger than L2 (H %.1f GB), no flush" % (T * d * 2 / 1e9),
                   "parallelism": ("dp%d over responses, dW exchanged in rank order every step"
                                   % world) if world > 1 else "dp1"},
        "step_ms_median": statistics.median(per_step),
        "algorithmic_tflops": flop_alg / (ms / 1e3) / 1e12,
        "algorithmic_frac_of_sustained_bf16": flop_alg / (ms / 1e3) / 1e12 /
        peaks["bf16_tflops_sustained"],
        # the dominant kernel of the timed step: the learner's logits +
        # log-sum-exp GEMM that keeps the softmax terms (2dV flop per token),
        # timed per launch by the launch-class events of the profiled steps
        "roofline": {
            "kernel": "gemm_kernel<EpiLseKeepT<true>> (learner logits+LSE GEMM keeping the "
                      "terms against the recorded log-sum-exp, one launch per 38,912-row chunk)",
            "bound": "tensor", "achieved": keep_tf,
            "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s",
            "frac": keep_tf / peaks["bf16_tflops_sustained"],
            "peak_source": "%s bf16_tflops_sustained (the kernel runs inside a %.1f s step under "
                           "the power cap)" % (peak_src, ms / 1e3),
            "frac_of_burst": keep_tf / peaks["bf16_tflops"],
            "ms_per_launch": keep_ms / keep_launches, "launches_per_step": keep_launches,
            "flop_per_launch": 2.0 * d * V * T / keep_launches,
            "traffic": captured_traffic(wl.name),
            "traffic_unit": "DRAM bytes per 38,912-row launch (ncu capture of a smaller chunk, "
                            "scaled by rows; see the committed ncu summary)",
            # H chunk + W + the chunk's references read; bf16 terms and split
            # states written
            "algorithmic_bytes_per_launch": 38912 * d * 2 + V * d * 2 + 38912 * 4 +
            38912 * 2 * ((V + 7) // 8 * 8) +
            rz.workspace_size(rz.RZ_OP_TOKEN_LOGPROB, 38912, d, V, 0)},
        "step_breakdown": breakdown,
        "gpu_launches": steps * (launches_per_step(T, V) + (1 if world > 1 else 0)),
        "device_err_flag": int(err.item()),
        "loss": float(loss.item()), "d3": float(d3.item()),
    }
    if world > 1:
        g = gathered.double().cpu()
        T_r = gather_over_ranks(T, world)
        out["exchange"] = {
            "ms_per_step": exchange_ms, "share_of_step": exchange_ms / ms,
            "what": "dW [V, d] fp32 added in rank order (NCCL all-to-all of 1/N slices, "
                    "rz_sum_partials, NCCL all-gather) + the loss shares and D3 of every rank",
            "bytes_per_rank": 2.0 * (world - 1) / world * V * d * 4}
        out["loss"] = float(g[:, 0].sum())
        out["d3"] = float(sum(g[r, 1] * T_r[r] for r in range(world)) / sum(T_r))
    if not full:
        return out

    # the same step through rz_loss_fwd_bwd (running maxima + the dz pass)
    pr = time_plain_route(rz, b, adv, lp, dH, dW, loss, d3, err, stream, dev,
                          max(2, min(steps, 5)))
    pr["algorithmic_frac_of_sustained_bf16"] = flop_alg / (pr["ms_per_step"] / 1e3) / 1e12 / \
        peaks["bf16_tflops_sustained"]
    out["plain_route"] = pr

    # the rollout's LM-head logprob GEMM (one tcgen05 GEMM launch per 38,912
    # rows + a tiny merge) over the same rows, with the lagged weights
    lp2 = torch.empty(T, dtype=torch.float32, device=dev)
    ws_r = rz.alloc_workspace(rz.RZ_OP_TOKEN_LOGPROB, T, d, V, 0, dev)
    rz.rz_token_logprob(b["H"], b["W_mu"], b["tokens"], logprob_out=lp2, ws=ws_r)
    torch.cuda.synchronize()
    kr = max(2, min(steps, 5))
    rev = [torch.cuda.Event(enable_timing=True) for _ in range(kr + 1)]
    rev[0].record(stream)
    for k in range(kr):
        rz.rz_token_logprob(b["H"], b["W_mu"], b["tokens"], logprob_out=lp2, ws=ws_r)
        rev[k + 1].record(stream)
    torch.cuda.synchronize()
    roll_ms = statistics.mean(rev[k].elapsed_time(rev[k + 1]) for k in range(kr))
    # rollout with the sampling fused into the same GEMM pass
    tok_s = torch.empty(T, dtype=torch.int32, device=dev)
    ws_s = rz.alloc_workspace(rz.RZ_OP_SAMPLE, T, d, V, 0, dev)
    rz.rz_sample_logprob(b["H"], b["W_mu"], 1234, tokens_out=tok_s, logprob_out=lp2, ws=ws_s)
    torch.cuda.synchronize()
    rev[0].record(stream)
    for k in range(kr):
        rz.rz_sample_logprob(b["H"], b["W_mu"], 1234 + k, tokens_out=tok_s, logprob_out=lp2,
                             ws=ws_s)
        rev[k + 1].record(stream)
    torch.cuda.synchronize()
    samp_ms = statistics.mean(rev[k].elapsed_time(rev[k + 1]) for k in range(kr))
    del ws_s, tok_s, ws_r, lp2
    # same-box reference: cuBLAS bf16 GEMM of one chunk's shape, interleaved
    ours_tf, cub_tf = gemm_vs_cublas(b["H"], b["W_mu"], b["tokens"], rz, dev, stream)
    out["clocks"] = clk.stop()

    # end to end through the public API from pinned host buffers
    out["e2e"] = run_e2e(args, b, rz, dev, stream, ws, dH, dW, lp, loss, d3, adv, err,
                         B_total if world > 1 else None, exchange)
    roll_tf = 2.0 * d * V * T / (roll_ms / 1e3) / 1e12
    out["rollout_gemm"] = {
        "kernel": "gemm_kernel<EpiLsePartial> (rollout logprob GEMM via rz_token_logprob)",
        "achieved_tflops": roll_tf,
        "frac_of_sustained": roll_tf / peaks["bf16_tflops_sustained"],
        "frac_of_burst": roll_tf / peaks["bf16_tflops"],
        "note": "timed back to back for about a second; the sustained peak is cuBLAS in a "
                "4 s loop and the burst peak its best single run, so a kernel between the "
                "two reads above 1.0 of sustained"}
    out["same_box_interleaved"] = {
        "logprob_gemm_tflops": ours_tf, "cublas_bf16_tflops": cub_tf, "ratio": ours_tf / cub_tf,
        "note": "alternating 1.5 s runs, 3 rounds, medians; cuBLAS [38912,d]x[d,V] bf16 with "
                "its output written"}
    out["rollout_tokens_per_s"] = T / (roll_ms / 1e3)
    out["rollout_sample_tokens_per_s"] = T / (samp_ms / 1e3)
    if rank == 0 and not args.no_cpu_baseline:
        s = oracle_sample(b, args.cpu_tokens)
        v, dt = time_oracle(s)
        out["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": cpu_threads(),
                               "kind": "oracle",
                               "sample": "%d tokens (first responses) of the same batch at full "
                                         "d=%d, V=%d; fp64 numpy, %.1f s" % (s["T"], d, V, dt)}
    return out


def gemm_vs_cublas(H, W, tokens, rz, dev, stream, rows=155648, seconds=1.5, rounds=3):
    """Same-box reference for the logprob GEMM: alternate ~1.5 s of our
    rz_token_logprob on `rows` rows with ~1.5 s of torch.matmul (cuBLAS) bf16
    on [38912, d] x [d, V] (its output is written, ours is not), three times,
    so both run under the same power and thermal state.  Returns median
    TFLOP/s of each."""
    import torch
    T = min(rows, H.shape[0])
    Hs, ts = H[:T], tokens[:T]
    d, V = H.shape[1], W.shape[0]
    ws = rz.alloc_workspace(rz.RZ_OP_TOKEN_LOGPROB, T, d, V, 0, dev)
    lp = torch.empty(T, dtype=torch.float32, device=dev)
    Hc = H[:38912]
    out = torch.empty((Hc.shape[0], V), dtype=torch.bfloat16, device=dev)

    def ours():
        rz.rz_token_logprob(Hs, W, ts, logprob_out=lp, ws=ws)
        return 2.0 * d * V * T

    def cub():
        torch.matmul(Hc, W.t(), out=out)
        return 2.0 * Hc.shape[0] * d * V

    res = {"ours": [], "cublas": []}
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    for _ in range(rounds):
        for name, f in (("ours", ours), ("cublas", cub)):
            f()
            torch.cuda.synchronize()
            fl, t = 0.0, 0.0
            e0.record(stream)
            while t < seconds * 1e3:
                for _ in range(4):
                    fl += f()
                e1.record(stream)
                e1.synchronize()
                t = e0.elapsed_time(e1)
            res[name].append(fl / (t / 1e3) / 1e12)
    del out, ws
    return statistics.median(res["ours"]), statistics.median(res["cublas"])


def time_plain_route(rz, b, adv, lp, dH, dW, loss, d3, err, stream, dev, steps):
    """The learner step through rz_loss_fwd_bwd on the same batch: 2 warm-ups,
    `steps` timed steps, and its launch-class breakdown."""
    import torch
    T, d, V, B = b["T"], b["d"], b["V"], b["B"]
    ws = rz.alloc_workspace(rz.RZ_OP_LOSS_FWD_BWD, T, d, V, B, dev)

    def step():
        rz.rz_group_advantage(b["rewards"], b["G"], adv_out=adv)
        rz.rz_loss_fwd_bwd(b["H"], b["W"], b["tokens"], b["logmu"], b["cu"], adv,
                           logprob_out=lp, dH=dH, dW=dW, loss_out=loss, d3_out=d3, ws=ws,
                           err_flag=err)
    for _ in range(2):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    br = profile_steps(rz, step, stream, 1)
    del ws
    return {"entry_point": "rz_loss_fwd_bwd", "value": T / (ms / 1e3), "unit": "tokens/s",
            "ms_per_step": ms, "steps": steps,
            "classes_ms": {k: v["ms"] for k, v in br["classes"].items()}}


def profile_steps(rz, step, stream, n):
    """Run n more learner steps with the library's launch-class timing on;
    returns per-step milliseconds and kernel launches of each class, their
    sum, and the steps' own CUDA-event time for comparison."""
    import torch
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    rz.rz_profile_begin()
    e0.record(stream)
    for _ in range(n):
        step()
    e1.record(stream)
    prof = rz.rz_profile_end()
    total = e0.elapsed_time(e1) / n
    classes = {k: {"ms": v[0] / n, "launches": v[1] // n} for k, v in prof.items() if v[1] > 0}
    summed = sum(c["ms"] for c in classes.values())
    for c in classes.values():
        c["share"] = c["ms"] / summed
    return {"classes": classes, "sum_ms": summed, "step_ms": total, "steps": n,
            "note": "one CUDA event pair per launch class on the launching stream, two untimed "
                    "steps after the timed region"}


def launches_per_step(T, V):
    chunk = 38912  # rows per backward chunk at V = 151936 (2.125 bytes per logit kept)
    n_chunks = (T + chunk - 1) // chunk
    # advantage; response factors; per chunk: logits+lse GEMM, merge+coef, the H
    # row scaling, dH, dW; loss (2)
    return 1 + 1 + 5 * n_chunks + 2


def run_e2e(args, b, rz, dev, stream, ws, dH, dW, lp, loss, d3, adv, err, B_total=None,
            exchange=None):
    """The learner step through the public API from pinned host buffers:
    every step copies its inputs (H, tokens, log mu, cu_seqlens, rewards)
    host -> device and reads its loss and D3 back.  Two device input slots
    and a copy stream let step k+1's upload overlap step k's compute, as a
    training loop would run it."""
    import torch
    host = {k: b[k].cpu().pin_memory() for k in ("H", "tokens", "logmu", "lse", "cu", "rewards")}
    slots = [{k: torch.empty_like(b[k]) for k in host} for _ in range(2)]
    res = torch.empty(2, dtype=torch.float32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = 8
    copy_stream = torch.cuda.Stream(device=dev)
    copied = [torch.cuda.Event() for _ in range(2)]
    consumed = [torch.cuda.Event() for _ in range(2)]

    def upload(i):
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(consumed[i])
            for k in host:
                slots[i][k].copy_(host[k], non_blocking=True)
            copied[i].record(copy_stream)

    def compute(i):
        stream.wait_event(copied[i])
        x = slots[i]
        rz.rz_group_advantage(x["rewards"], b["G"], adv_out=adv)
        if B_total is None:
            rz.rz_loss_fwd_bwd_ref(x["H"], b["W"], x["tokens"], x["logmu"], x["lse"], x["cu"],
                                   adv, logprob_out=lp, dH=dH, dW=dW, loss_out=loss,
                                   d3_out=d3, ws=ws, err_flag=err)
        else:  # one shard of the data-parallel step, then the exchange
            rz.rz_loss_fwd_bwd_shard(x["H"], b["W"], x["tokens"], x["logmu"], x["cu"], adv,
                                     B_total, logprob_out=lp, dH=dH, dW=dW, loss_out=loss,
                                     d3_out=d3, ws=ws, err_flag=err, ref_lse=x["lse"])
            exchange()
        consumed[i].record(stream)
        res[0:1].copy_(loss, non_blocking=True)
        res[1:2].copy_(d3, non_blocking=True)

    def run(K, e0=None, e1=None):
        if e0 is not None:
            e0.record(stream)
            copy_stream.wait_event(e0)
        upload(0)
        for k in range(K):
            if k + 1 < K:
                upload((k + 1) % 2)
            compute(k % 2)
        if e1 is not None:
            e1.record(stream)
        torch.cuda.synchronize()

    run(2)
    K = max(2, min(args.steps, 8))
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    run(K, e0, e1)
    ms = e0.elapsed_time(e1) / K
    return {"value": b["T"] / (ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms,
            "note": "inputs (H, tokens, log mu, the recorded log-sum-exp, cu_seqlens, rewards) "
                    "uploaded from pinned host memory every step, the upload of step k+1 "
                    "overlapping the compute of step k; loss and D3 read back.  W stays resident and dH, dW stay on the device "
                    "for an on-device optimiser, as in a training loop"}


def measure_logits(args, world, rank, dev, peaks, peak_src, steps, warmup, full=True):
    """The given-logits step (rz_logits_loss_fwd_bwd) on the MoE-shaped
    workload; with `full`, also clocks and the CPU baseline."""
    import torch
    import invariant_logprobs_gb300 as rz
    from invariant_logprobs_gb300 import synth
    wl = synth.WORKLOADS["moe30b_logits"]
    b = synth.make_logits_batch(wl, device=dev, seed=wl.seed + 7919 * rank)
    T, V, B = b["T"], b["V"], b["B"]
    logpi = torch.empty(T, dtype=torch.float32, device=dev)
    for s in range(0, T, 8192):
        e = min(T, s + 8192)
        z = torch.log_softmax(b["logits"][s:e].float(), dim=-1)
        logpi[s:e] = z.gather(1, b["tokens"][s:e].long()[:, None])[:, 0]
        del z
    logmu = synth.logmu_near(logpi, synth.LOGMU_NOISE_STD, b["gen"])
    adv = rz.rz_group_advantage(b["rewards"], b["G"])
    lp = torch.empty(T, dtype=torch.float32, device=dev)
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    d3 = torch.empty(1, dtype=torch.float32, device=dev)
    ws = rz.alloc_workspace(rz.RZ_OP_LOGITS_LOSS, T, 0, V, B, dev)
    err = rz.new_err_flag(dev)
    stream = torch.cuda.current_stream()

    def step():
        rz.rz_logits_loss_fwd_bwd(b["logits"], b["tokens"], logmu, b["cu"], adv,
                                  logprob_out=lp, loss_out=loss, d3_out=d3, ws=ws, err_flag=err)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    clk = ClockSampler(dev.index)
    if full:
        clk.start()
        time.sleep(0.3)
    barrier(world)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    ev[0].record(stream)
    for k in range(steps):
        step()
        ev[k + 1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = clk.stop() if full else None
    breakdown = profile_steps(rz, step, stream, 2)
    ms = max_over_ranks(ev[0].elapsed_time(ev[-1]) / steps, world)
    rows_ms = breakdown["classes"]["logits_rows"]["ms"]
    alg_bytes = T * (4.0 * V + 12.0)
    out = {
        "metric": METRIC, "value": T * world / (ms / 1e3), "unit": "tokens/s",
        "n_gpus": world, "steps": steps, "warmup": warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic bf16 logits ~N(0,3) (in place: later steps read the previous dz)",
        "config": {"workload": wl.name, "tokens_per_step": T, "responses": B, "V": V,
                   "l2": "inputs larger than L2 (%.0f GB), no flush" % (T * V * 2 / 1e9),
                   "parallelism": "dp%d replicas" % world},
        # one launch of the row kernel per step, timed by the launch-class
        # events of the profiled steps
        "roofline": {"kernel": "logits_row_kernel", "bound": "hbm",
                     "achieved": alg_bytes / (rows_ms / 1e3) / 1e9, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": alg_bytes / (rows_ms / 1e3) / 1e9 / peaks["hbm_gbs"],
                     "peak_source": "%s hbm_gbs" % peak_src,
                     "ms_per_launch": rows_ms,
                     "traffic": captured_traffic(wl.name),
                     "traffic_unit": "DRAM bytes per launch (ncu capture of 16,384 rows scaled "
                                     "to 262,144; see the committed ncu summary)",
                     "algorithmic_bytes_per_launch": alg_bytes},
        "step_breakdown": breakdown,
        "gpu_launches": 4 * steps,  # response factors, row kernel, loss (2)
        "device_err_flag": int(err.item()),
    }
    if clocks is not None:
        out["clocks"] = clocks
    if full and rank == 0 and not args.no_cpu_baseline:
        s = logits_oracle_sample(b["logits"], b["tokens"], logmu, b["cu"], b["rewards"], b["G"],
                                 args.cpu_tokens)
        v, dt = time_logits_oracle(s)
        out["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": cpu_threads(),
                               "kind": "oracle",
                               "sample": "first %d rows of the same logits at V=%d (log pi, "
                                         "loss, dz for every row); fp64 numpy, %.1f s"
                                         % (s["T"], V, dt)}
    return out


# ----------------------------------------------------------------- reference arm
def reference_tokens(args):
    """Tokens per reference-arm step: --cpu-tokens for up to 10 steps, fewer
    for longer runs, so that the whole run stays within a few minutes."""
    if args.steps <= 10:
        return args.cpu_tokens
    return max(64, args.cpu_tokens * 10 // args.steps)


def run_reference(args):
    """The CPU oracle as it stands, on the host cores, on a bounded sample of
    the same workload; rank 0 only."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from invariant_logprobs_gb300 import synth
    if args.config == "moe30b_logits":
        return run_reference_logits(args, world)
    wl = synth.WORKLOADS[args.config]
    # draw the same distributions on the host (no GPU needed): a small batch
    # of whole responses at full d and V
    import dataclasses
    n = reference_tokens(args)
    small = dataclasses.replace(wl, n_prompts=1, group=2, len_lo=n // 2, len_hi=n // 2)
    b = synth.make_batch(small, device="cpu")
    s = oracle_sample(b, n)
    for _ in range(max(0, min(args.warmup, 1))):
        time_oracle(s)
    times = []
    for _ in range(args.steps):
        _, dt = time_oracle(s)
        times.append(dt)
    ms = 1e3 * statistics.mean(times)
    v = s["T"] / (ms / 1e3)
    out = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s",
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic (seeded)",
           "config": {"workload": wl.name, "d": wl.d, "V": wl.V,
                      "tokens_per_step": s["T"], "parallelism": "cpu oracle, rank 0"},
           "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cpu_threads(),
                            "kind": "oracle",
                            "sample": "%d tokens at full d=%d, V=%d per step" % (
                                s["T"], wl.d, wl.V)},
           "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)
    return 0


def run_reference_logits(args, world):
    """Reference arm of the given-logits workload: the oracle on one group of
    responses drawn with the same distributions (N(0,3) logits at full V,
    uniform tokens, log mu = log pi + N(0,0.05)), --cpu-tokens rows in all."""
    import dataclasses
    import numpy as np
    import torch
    from invariant_logprobs_gb300 import synth
    import oracle
    wl = synth.WORKLOADS["moe30b_logits"]
    n = max(wl.group, reference_tokens(args))
    small = dataclasses.replace(wl, len_lo=n // wl.group, len_hi=n // wl.group)
    b = synth.make_logits_batch(small, device="cpu", T=n // wl.group * wl.group)
    T = b["T"]
    logits = b["logits"].to(torch.float32).numpy()
    tokens, cu = b["tokens"].numpy(), b["cu"].numpy()
    adv = oracle.group_advantage(b["rewards"].double().numpy(), b["G"])
    logpi = oracle.logits_loss_fwd_bwd(logits, tokens, np.zeros(T), cu, adv,
                                       rows=np.zeros(0, np.int64))["logpi"]
    logmu = synth.logmu_near(torch.tensor(logpi), synth.LOGMU_NOISE_STD, b["gen"])
    s = {"logits": logits, "tokens": tokens, "logmu": logmu.double().numpy(), "cu": cu,
         "adv": adv, "T": T}
    for _ in range(max(0, min(args.warmup, 1))):
        time_logits_oracle(s)
    times = [time_logits_oracle(s)[1] for _ in range(args.steps)]
    ms = 1e3 * statistics.mean(times)
    v = T / (ms / 1e3)
    out = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s",
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic (seeded)",
           "config": {"workload": wl.name, "V": wl.V, "tokens_per_step": T,
                      "responses": b["B"], "parallelism": "cpu oracle, rank 0"},
           "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cpu_threads(),
                            "kind": "oracle",
                            "sample": "%d rows of %d responses at V=%d per step" % (
                                T, b["B"], wl.V)},
           "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)
    return 0


def run_profile(args):
    """Small fixed cases for ncu captures (not a benchmark), on `--rows`
    tokens of the workload's d and V: one rollout logprob call then `--steps`
    learner steps (learner), `--steps` given-logits steps (logits), fused
    sampling calls (sample) or rollout logprob calls (rollout).  The learner
    steps go through rz_loss_fwd_bwd_ref (learner) or rz_loss_fwd_bwd
    (learner_plain)."""
    import dataclasses
    import torch
    import invariant_logprobs_gb300 as rz
    from invariant_logprobs_gb300 import synth
    rz.load()
    dev = torch.device("cuda", 0)
    if args.profile == "logits":
        wl = synth.WORKLOADS["moe30b_logits"]
        b = synth.make_logits_batch(wl, device=dev, T=args.rows)
        logmu = torch.full((b["T"],), -12.0, device=dev)
        adv = rz.rz_group_advantage(b["rewards"], b["G"])
        for _ in range(args.steps):
            rz.rz_logits_loss_fwd_bwd(b["logits"], b["tokens"], logmu, b["cu"], adv)
        torch.cuda.synchronize()
        print("profile logits rows=%d ok" % b["T"])
        return 0
    wl = synth.WORKLOADS[args.config]
    per = max(1, args.rows // wl.B)
    wl = dataclasses.replace(wl, len_lo=per, len_hi=per, tokens="uniform")
    b = synth.make_batch(wl, device=dev)
    if args.profile in ("sample", "rollout"):
        # fewer rows than the workload has responses: its first rows (a
        # decode-sized batch takes the logits through the workspace)
        n = min(args.rows, b["T"])
        H, tok = b["H"][:n].contiguous(), b["tokens"][:n].contiguous()
        for k in range(args.steps):
            if args.profile == "sample":
                rz.rz_sample_logprob(H, b["W_mu"], 77 + k)
            else:
                rz.rz_token_logprob(H, b["W_mu"], tok)
        torch.cuda.synchronize()
        print("profile %s rows=%d ok" % (args.profile, n))
        return 0
    lse = torch.empty(b["T"], dtype=torch.float32, device=dev)
    logmu, _ = rz.rz_token_logprob(b["H"], b["W_mu"], b["tokens"], lse_out=lse)
    adv = rz.rz_group_advantage(b["rewards"], b["G"])
    for _ in range(args.steps):
        if args.profile == "learner_plain":
            rz.rz_loss_fwd_bwd(b["H"], b["W"], b["tokens"], logmu, b["cu"], adv)
        else:
            rz.rz_loss_fwd_bwd_ref(b["H"], b["W"], b["tokens"], logmu, lse, b["cu"], adv)
    torch.cuda.synchronize()
    print("profile %s rows=%d ok" % (args.profile, b["T"]))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", default="qwen4b_lag64",
                    choices=["qwen4b_lag64", "qwen1p5b_lag2", "moe30b_logits", "tiny"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-tokens", type=int, default=1024,
                    help="tokens of the CPU oracle's timed sample (about 10 s at the 4B shape)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="time only --config (by default the other two bench workloads follow, "
                         "briefly, under other_workloads)")
    ap.add_argument("--profile", choices=["learner", "learner_plain", "logits", "sample", "rollout"], default=None,
                    help="small fixed case for ncu captures (no timing output)")
    ap.add_argument("--rows", type=int, default=16384)
    args = ap.parse_args()
    if args.profile:
        return run_profile(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
