#!/usr/bin/env python
"""Throughput of the nanochat-style pretraining step (forward + backward) on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload d20_bf16]
    python bench.py --impl reference ...     # the fp64 CPU oracle on host cores

One step = nc_step over one batch: embedding + norm, every block forward,
LM head + softcap + cross-entropy with its backward, every block backward,
embedding backward -- all weight gradients produced.  Inputs are synthetic
(Zipf(1.1) token ids, N(0, 1/fan_in) bf16 weights) and resident in HBM when
the timed region starts.  The working set (~40 GB at d20) is far larger than
the 126 MB L2, so no flush is needed between steps.

For N > 1 (one rank per GPU) every rank runs its own batch of the same
shape: the step shards by batch rows with no data-path collective, so
scaling is weak; the only collectives are the timing barrier and the max
over ranks.  `--gpus N` without a launcher starts the N ranks itself
(torch.distributed.run on 127.0.0.1); under a launcher WORLD_SIZE must equal
N.  Rank 0 prints one JSON line.

The headline is timed with nothing but the step on the stream.  A second,
separate pass of the same number of steps records CUDA events around every
named launch group; it gives the per-kernel attribution and the roofline of
the dominant kernel.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import nc_synth  # noqa: E402
from pretraining_step_pretrain_b300 import flops  # noqa: E402

METRIC = "train tokens/sec (fwd+bwd) at d20 shape, 1×B300; MFU vs bf16 tensor peak"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
NOMINAL_BF16_TFLOPS = 2250.0


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock / throttle samples every 200 ms while running."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-i", str(self.idx), "-lms", "200", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        power = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max(power) if power else None}


# ---------------------------------------------------------------- roofline
def algorithmic_cost(name, shape, B, T):
    """(kind, amount) per launch of a named launch group: FLOPs for tensor-core
    work, bytes for memory-bound work (minimum HBM traffic of the operation)."""
    d, H, h, f, V = shape.d_model, shape.n_head, shape.head_dim, shape.d_mlp, shape.vocab
    M, q = B * T, (H + 2) * h
    gemm = {"qkv": 2 * M * d * q, "out": 2 * M * H * h * d, "fc": 2 * M * d * f,
            "proj": 2 * M * f * d}
    causal_matmul = B * H * T * T * h          # one causal-half matmul (2 * T^2/2 * h)
    if name.startswith("fwd.") and name.endswith("_gemm"):
        return "tensor", gemm[name[4:-5]]
    if name.startswith("bwd.") and name.endswith("_gemm"):
        return "tensor", gemm[name[4:].split("_")[0]]
    if name in ("lm.logits_gemm", "lm.dw_gemm", "lm.dx_gemm"):
        return "tensor", 2 * M * d * V
    if name == "fwd.attention":
        return "tensor", 2 * causal_matmul
    if name == "bwd.attention":
        return "tensor", 5 * causal_matmul
    if name in ("fwd.norm1", "fwd.norm2", "lm.norm"):
        return "hbm", M * d * (4 + 2) + M * 4
    if name in ("bwd.norm1_bwd", "bwd.norm2_bwd", "lm.norm_bwd"):
        return "hbm", M * d * (2 + 2 + 4 + 4 + 2)
    if name == "fwd.qknorm_rope":
        return "hbm", M * q * 2 * 2
    if name == "bwd.qknorm_rope":
        return "hbm", M * (H + 1) * h * 2 * 3
    if name == "lm.dlogits":
        return "hbm", M * V * 2 * 2
    if name == "embed.norm":
        return "hbm", M * d * (2 + 4)
    if name == "embed_bwd":
        return "hbm", M * d * (4 + 2 + 4 + 4) + V * d * 4
    return None, 0


def aggregate_profile(recs):
    """[(launch group, ms)] -> rows sorted by total time, and the total."""
    agg = {}
    for name, ms in recs:
        a = agg.setdefault(name, [0.0, 0])
        a[0] += ms
        a[1] += 1
    total = sum(v[0] for v in agg.values())
    rows = sorted(agg.items(), key=lambda kv: -kv[1][0])
    return rows, total


TRAFFIC_FILE = os.path.join(ROOT, "profiles", "roofline_traffic.txt")


def measured_traffic(group):
    """DRAM bytes per launch of a launch group from an ncu capture listed in
    profiles/roofline_traffic.txt, or None when there is none or a listed
    kernel source changed since the capture (its sha256 prefix differs)."""
    import hashlib
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        for line in f:
            parts = line.split()
            if len(parts) < 4 or parts[0].startswith("#") or parts[0] != group:
                continue
            h = hashlib.sha256()
            for src in parts[3:]:
                path = os.path.join(ROOT, "pretraining_step_pretrain_b300", "csrc", src)
                if not os.path.exists(path):
                    return None
                with open(path, "rb") as g:
                    h.update(g.read())
            if h.hexdigest()[:16] != parts[2]:
                return None
            return float(parts[1])
    return None


# ---------------------------------------------------------------- CPU oracle
def blas_threads() -> int:
    """Threads the oracle's BLAS uses (threadpoolctl when present, else the
    OpenBLAS/OMP environment, else every host core)."""
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info()]
        if n and max(n) > 0:
            return max(n)
    except ImportError:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    return os.cpu_count() or 1


def host_cpu():
    """The host the oracle ran on: CPU model name (from /proc/cpuinfo) and the
    number of logical cores."""
    model = "unknown"
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    return {"model": model, "nproc": os.cpu_count() or 1}


def oracle_tokens_per_s(shape, B, T, min_seconds, max_steps, weights=None):
    """Time the fp64 oracle's full step on B rows of T tokens at `shape` on the
    host cores (as many BLAS threads as the environment gives it)."""
    import oracle
    if weights is None:
        weights = nc_synth.make_weights(shape, seed=1, bf16=True)
    P = {k: v.astype(np.float64) for k, v in weights.items()}
    ids, tg = nc_synth.make_tokens(shape.vocab, B, T, seed=0)
    oracle.step(shape, P, ids, tg)                       # first touch of every buffer
    times = []
    t_all = time.perf_counter()
    while len(times) < max_steps and (time.perf_counter() - t_all < min_seconds or not times):
        t0 = time.perf_counter()
        oracle.step(shape, P, ids, tg)
        times.append(time.perf_counter() - t0)
    return B * T * len(times) / sum(times), blas_threads(), len(times)


ONE_THREAD_ENV = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")


def oracle_one_thread(workload, tokens):
    """The same oracle timing in a child process whose BLAS runs one thread
    (the thread count is fixed when the BLAS library loads)."""
    env = dict(os.environ, **{k: "1" for k in ONE_THREAD_ENV})
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-sample", workload,
                        str(tokens)], env=env, capture_output=True, text=True, timeout=600)
    if r.returncode != 0:
        return {"error": r.stderr.strip().splitlines()[-1] if r.stderr.strip() else "failed"}
    return json.loads(r.stdout.strip().splitlines()[-1])


def cpu_baseline(w, weights, tokens, full_d20=False):
    """The fp64 oracle on the host cores: the bench workload's widths on one
    row of `tokens` tokens (all BLAS threads, then one thread), the tiny and
    small configurations' full steps, and optionally one whole 2048-token row
    at the depth-20 widths."""
    v, threads, n = oracle_tokens_per_s(w.shape, 1, tokens, 5.0, 2, weights)
    out = {"value": v, "unit": "tokens/s", "cores": threads, "host": host_cpu(),
           "kind": "oracle",
           "sample": f"{w.name} widths, 1 row x {tokens} tokens, {n} timed full oracle "
                     f"step(s) (forward + backward, fp64) after one untimed",
           "one_thread": oracle_one_thread(w.name, tokens),
           "full_steps": {}}
    for name in ("tiny_f32", "small_bf16"):
        o = nc_synth.WORKLOADS[name]
        tv, tt, tn = oracle_tokens_per_s(o.shape, o.batch, o.seq, 1.0, 5)
        out["full_steps"][name] = {"value": tv, "unit": "tokens/s", "cores": tt, "steps": tn,
                                   "batch": o.batch, "seq": o.seq}
    if full_d20:
        d20 = nc_synth.D20
        tv, tt, tn = oracle_tokens_per_s(d20.shape, 1, d20.seq, 0.0, 1)
        out["full_steps"]["d20_bf16_1x2048"] = {"value": tv, "unit": "tokens/s", "cores": tt,
                                                "steps": tn, "batch": 1, "seq": d20.seq}
    return out


# ---------------------------------------------------------------- arms
def run_reference(args, rank, world):
    if rank != 0:
        return
    w = nc_synth.WORKLOADS[args.workload]
    shape = w.shape
    T = args.ref_tokens
    weights = nc_synth.make_weights(shape, seed=1, bf16=True)
    import oracle
    P = {k: v.astype(np.float64) for k, v in weights.items()}
    ids, tg = nc_synth.make_tokens(shape.vocab, 1, T, seed=0)
    for _ in range(args.warmup):
        oracle.step(shape, P, ids, tg)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.step(shape, P, ids, tg)
    dt = time.perf_counter() - t0
    value = T * args.steps / dt
    threads = blas_threads()
    sample = f"{w.name} widths, 1 row x {T} tokens per step (fp64 numpy oracle)"
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
           "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": 1000 * dt / args.steps, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": config_dict(w, args.gpus),
           "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads,
                            "host": host_cpu(),
                            "kind": "oracle", "sample": sample},
           "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def config_dict(w, n):
    return {"workload": w.name, "depth": w.shape.depth, "d_model": w.shape.d_model,
            "n_head": w.shape.n_head, "head_dim": w.shape.head_dim, "n_kv_head": 1,
            "d_mlp": w.shape.d_mlp, "vocab": w.shape.vocab, "batch_per_gpu": w.batch,
            "global_batch": w.batch * n, "seq_len": w.seq,
            "parallelism": f"batch rows sharded over {n} GPU(s), no collective",
            "l2": "no flush: working set far larger than L2"}


# ---------------------------------------------------------------- multi-rank helpers
def rank_batch(w, rank):
    """This rank's shard of the job: its own B x T token rows (seed = rank);
    every rank holds the same weights."""
    return nc_synth.make_tokens(w.shape.vocab, w.batch, w.seq, seed=rank, dist=w.ids)


def max_over_ranks(x, world):
    """The slowest rank's value, returned on every rank (x when world == 1).
    The tensor lives where the process group's backend wants it: the GPU for
    NCCL, the host for gloo."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(B, T, world, steps, seconds):
    """Whole-job throughput: every rank's tokens over the slowest rank's time."""
    return B * T * world * steps / seconds


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    from pretraining_step_pretrain_b300 import nc
    torch.cuda.set_device(local_rank)
    w = nc_synth.WORKLOADS[args.workload]
    shape, B, T = w.shape, w.batch, w.seq
    weights = nc_synth.make_weights(shape, seed=1, bf16=(w.dtype == "bf16"))
    ids, tg = rank_batch(w, rank)
    st = nc.Step(shape, w.dtype, B, T, weights, device=f"cuda:{local_rank}")
    ids_d = torch.from_numpy(ids).cuda()
    tg_d = torch.from_numpy(tg).cuda()
    st.ids.copy_(ids_d)
    st.targets.copy_(tg_d)
    for _ in range(args.warmup):
        st.run()
    torch.cuda.synchronize()
    if st.status() != 0:
        raise RuntimeError("device error during warm-up")

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    stream = torch.cuda.current_stream()
    visible = [v.strip() for v in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if v]
    gpu_idx = local_rank
    if local_rank < len(visible) and visible[local_rank].isdigit():
        gpu_idx = int(visible[local_rank])
    clocks = ClockSampler(gpu_idx)
    # Headline: K steps with nothing else on the stream; one event after each
    # step (for the median), none inside it.
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    barrier()
    clocks.start()
    n0 = nc.launch_count()
    ev[0].record(stream)
    for i in range(args.steps):
        st.run()
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    launches = nc.launch_count() - n0
    clk = clocks.stop()
    barrier()
    step_ms = [ev[i].elapsed_time(ev[i + 1]) for i in range(args.steps)]
    ms = max_over_ranks(ev[0].elapsed_time(ev[-1]), world)
    if st.status() != 0:
        raise RuntimeError("device error during the timed steps")
    loss = float(st.loss.item())
    value = job_tokens_per_s(B, T, world, args.steps, ms / 1000.0)

    # Attribution: a separate pass of K steps with CUDA events recorded by the
    # library around every named launch group on the launching stream.
    nc.profile_start(60 * (shape.depth + 2) * args.steps)
    e0, e1 = ev[0], ev[-1]
    e0.record(stream)
    for _ in range(args.steps):
        st.run()
    e1.record(stream)
    torch.cuda.synchronize()
    recs = nc.profile_stop()
    prof_ms = e0.elapsed_time(e1)

    # end to end through the public call with host buffers
    ids_h = torch.from_numpy(ids).pin_memory()
    tg_h = torch.from_numpy(tg).pin_memory()
    st.run_host(ids_h, tg_h)
    barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        st.run_host(ids_h, tg_h)
    t_e2e = max_over_ranks(time.perf_counter() - t0, world)
    e2e = {"value": job_tokens_per_s(B, T, world, args.steps, t_e2e), "unit": "tokens/s",
           "h2d_bytes_per_step": 2 * B * T * 4, "d2h_bytes_per_step": 4}

    # per-launch-group attribution over the profiled steps
    rows, prof_total = aggregate_profile(recs)
    peaks, peak_src = load_peaks()
    top = None
    for name, (tot, cnt) in rows:
        kind, amount = algorithmic_cost(name, shape, B, T)
        if kind is not None:
            top = (name, tot, cnt, kind, amount)
            break
    roofline = None
    where = (f"CUDA events around each launch of the group on its stream, over {args.steps} "
             f"profiled steps run right after the headline steps")
    if top:
        name, tot, cnt, kind, amount = top
        per_launch_s = tot / cnt / 1000.0
        if kind == "tensor":
            achieved = amount / per_launch_s / 1e12
            peak = peaks["bf16_tflops_sustained"]
            roofline = {"kernel": name, "bound": "tensor", "achieved": achieved, "peak": peak,
                        "unit": "TFLOP/s", "frac": achieved / peak,
                        "traffic": measured_traffic(name),
                        "peak_source": f"{peak_src} bf16 sustained", "share": tot / prof_total,
                        "algorithmic_per_launch": amount, "timing": where}
        else:
            achieved = amount / per_launch_s / 1e9
            peak = peaks["hbm_gbs"]
            roofline = {"kernel": name, "bound": "hbm", "achieved": achieved, "peak": peak,
                        "unit": "GB/s", "frac": achieved / peak,
                        "traffic": measured_traffic(name),
                        "peak_source": f"{peak_src} copy bandwidth", "share": tot / prof_total,
                        "algorithmic_per_launch": amount, "timing": where}
    kernels = []
    for name, (tot, cnt) in rows[:16]:
        kind, amount = algorithmic_cost(name, shape, B, T)
        entry = {"name": name, "ms_per_step": tot / args.steps,
                 "share": tot / prof_total}
        if kind == "tensor":
            entry["tflops"] = amount * cnt / (tot / 1000.0) / 1e12
        elif kind == "hbm":
            entry["gbs"] = amount * cnt / (tot / 1000.0) / 1e9
        kernels.append(entry)

    # optimizer step (Muon + AdamW) on the step's gradients: time per step and
    # the Newton-Schulz GEMM rate; not part of the fwd+bwd metric above
    optim = None
    if not args.no_optimizer:
        o = nc.Optimizer(st)
        for t in range(1, 3):
            o.step(t, 1.0)
        torch.cuda.synchronize()
        n0 = nc.launch_count()
        e0.record(stream)
        for t in range(3, 3 + args.steps):
            o.step(t, 1.0)
        e1.record(stream)
        torch.cuda.synchronize()
        o_ms = e0.elapsed_time(e1) / args.steps
        ns_flops, adam_bytes = flops.optimizer_cost(shape)
        optim = {"ms_per_step": o_ms, "launches_per_step": (nc.launch_count() - n0) / args.steps,
                 "newton_schulz_flops": ns_flops, "adamw_bytes": adam_bytes,
                 "newton_schulz_tflops_if_all_time": ns_flops / (o_ms / 1000.0) / 1e12,
                 "note": "Muon for the block matrices (5 quintic Newton-Schulz steps, batched "
                         "tcgen05 GEMMs), AdamW for wte and w_lm; fp32 masters and state"}
        del o
        torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        del st
        torch.cuda.empty_cache()
        cpu = cpu_baseline(w, weights, args.cpu_tokens, full_d20=args.cpu_full_d20)

    f_tok = flops.flops_per_token(shape, T)
    f_tok_causal = flops.flops_per_token(shape, T, causal_actual=True)
    per_gpu = value / world
    out = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
           "ms_per_step_median": statistics.median(step_ms),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": w.dtype, "data": "synthetic: Zipf(1.1) token ids, N(0,1/fan_in) weights",
           "config": config_dict(w, world),
           "mfu": per_gpu * f_tok / (peaks["bf16_tflops"] * 1e12),
           "mfu_detail": {"flops_per_token_palm": f_tok, "flops_per_token_causal": f_tok_causal,
                          "vs_measured_burst": per_gpu * f_tok / (peaks["bf16_tflops"] * 1e12),
                          "vs_measured_sustained":
                              per_gpu * f_tok / (peaks["bf16_tflops_sustained"] * 1e12),
                          "vs_nominal_2250": per_gpu * f_tok / (NOMINAL_BF16_TFLOPS * 1e12),
                          "causal_actual_vs_measured_burst":
                              per_gpu * f_tok_causal / (peaks["bf16_tflops"] * 1e12),
                          "peak_source": peak_src},
           "loss": loss, "roofline": roofline, "kernels": kernels,
           "profiled_ms_per_step": prof_ms / args.steps, "cpu_baseline": cpu,
           "e2e": e2e, "gpu_launches": launches, "clocks": clk, "optimizer": optim}
    if rank == 0:
        print(json.dumps(out), flush=True)


def free_port() -> int:
    import socket
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def launch_ranks(n, argv):
    """Run this script as n ranks on this node (torch.distributed.run,
    rendezvous on 127.0.0.1); returns the launcher's exit code."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={n}", "--master-addr", "127.0.0.1",
           "--master-port", str(free_port()), os.path.abspath(__file__), *argv]
    return subprocess.call(cmd)


def launcher_check(rank, world):
    """Host-only check of the rank layout (no GPU work, no timing): every rank
    joins a gloo group and rank 0 prints the ranks it sees."""
    import torch
    import torch.distributed as dist
    dist.init_process_group("gloo")
    got = [None] * world
    dist.all_gather_object(got, {"rank": rank, "world": world,
                                 "local_rank": int(os.environ.get("LOCAL_RANK", 0))})
    if rank == 0:
        print(json.dumps({"launcher_check": True, "n_gpus": world, "ranks": got}), flush=True)
    dist.barrier()
    dist.destroy_process_group()
    del torch


def main(argv=None):
    argv = sys.argv[1:] if argv is None else argv
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="d20_bf16", choices=sorted(nc_synth.WORKLOADS))
    ap.add_argument("--cpu-tokens", type=int, default=256)
    ap.add_argument("--cpu-full-d20", action="store_true",
                    help="also time one whole 2048-token row of the oracle at the depth-20 widths")
    ap.add_argument("--ref-tokens", type=int, default=32)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-optimizer", action="store_true")
    ap.add_argument("--launcher-check", action="store_true",
                    help="start the ranks, report the rank layout, run nothing on a GPU")
    ap.add_argument("--oracle-sample", nargs=2, metavar=("WORKLOAD", "TOKENS"),
                    help="time the oracle alone on 1 row of TOKENS tokens and print it")
    args = ap.parse_args(argv)
    if args.oracle_sample:
        w = nc_synth.WORKLOADS[args.oracle_sample[0]]
        v, threads, n = oracle_tokens_per_s(w.shape, 1, int(args.oracle_sample[1]), 0.0, 1)
        print(json.dumps({"value": v, "unit": "tokens/s", "cores": threads, "steps": n}))
        return
    if args.gpus < 1:
        ap.error("--gpus must be >= 1")
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        sys.exit(launch_ranks(args.gpus, argv))
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local_rank = int(os.environ.get("LOCAL_RANK", 0))
    if world != args.gpus:
        print(f"bench.py: --gpus {args.gpus} but the launcher started {world} rank(s)",
              file=sys.stderr)
        sys.exit(2)
    if args.launcher_check:
        launcher_check(rank, world)
        return
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    run_ours(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
