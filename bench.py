"""Benchmark of the persistent GPT training step (162M GPT, seq 512, batch 8).

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config main]

Prints ONE JSON line (rank 0).  A step is one call of gpt_train_step: forward,
backward and AdamW of the whole model as one persistent kernel launch.  Inputs
are seeded synthetic Zipf(1.1) token batches (64 distinct batches, pre-uploaded),
standing in for the tokenized TinyStories stream of the pages; weights are the
seeded N(0, 0.02) initialisation.  The step's working set (fp32 master weights,
moments, gradients and activations: 6.5 GB for the 162M model) is far larger than
L2, so no L2 flush is inserted between steps.

Besides the device-timed steps (value) the line carries the same steps through
the host-buffer entry point (e2e) and as one multi-step call (multi_step_call).
--config selects another workload of inputs.CONFIGS (350m, 57m, ...).

Multi-GPU: the step does not shard here (no collective is in scope), so N > 1
runs N independent replicas, one per rank, and reports the aggregate tokens/s
over the max-over-ranks time ("scaling": "weak").

--impl reference times the CPU oracle (numpy, the machine's host cores) on a bounded
sample of the same workload; under torchrun only rank 0 runs it.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "train tokens/s & ms/step, 162M GPT seq512 b8 on 1 GB300; % bf16 tensor peak"
UNIT = "tokens/s"


def kernel_source_digest() -> str:
    """sha256 over the kernel's sources (csrc/ and the C header), to tell whether a
    stored ncu measurement still describes the kernel that runs."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "persistent_gpt_step_gb300", "csrc")
    files = sorted(os.path.join(csrc, f) for f in os.listdir(csrc)) + [os.path.join(ROOT, "include", "gpt.h")]
    for f in files:
        h.update(os.path.relpath(f, ROOT).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def measured_traffic(workload: str):
    """DRAM bytes (read + write) of one step launch from the committed ncu capture
    (profiles/step_kernel_main_traffic.json), or None when that capture was taken
    on another workload or on kernel sources that have changed since."""
    path = os.path.join(ROOT, "profiles", "step_kernel_main_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("workload") != workload or rec.get("kernel_source_sha256") != kernel_source_digest():
        return None
    return int(rec["dram_bytes_read"]) + int(rec["dram_bytes_write"])


def ptxas_report():
    """Registers, stack and spill bytes of each step-kernel instance, from the
    build's -Xptxas -v report (persistent_gpt_step_gb300/_build/ptxas.txt)."""
    import re
    path = os.path.join(ROOT, "persistent_gpt_step_gb300", "_build", "ptxas.txt")
    try:
        text = open(path).read()
    except OSError:
        return None
    out = {}
    names = {"I13__nv_bfloat16Lb1ELb0": "bf16", "I13__nv_bfloat16Lb1ELb1": "bf16_variant", "IfLb0ELb0": "fp32"}
    for key, label in names.items():
        m = re.search(r"Function properties for _ZN3pgs15gpt_step_kernel" + key + r"\S*\n\s*(\d+) bytes stack frame, "
                      r"(\d+) bytes spill stores, (\d+) bytes spill loads\n[^\n]*Used (\d+) registers", text)
        if m:
            out[label] = {"registers": int(m.group(4)), "stack_bytes": int(m.group(1)),
                          "spill_stores": int(m.group(2)), "spill_loads": int(m.group(3))}
    return out or None


def model_flops(cfg, n_params: int) -> float:
    """6 * params * tokens + causal attention (fwd + bwd = 3x fwd; fwd = 2 T^2 d per head)."""
    N = cfg.batch * cfg.seq_len
    attn = 6.0 * cfg.seq_len ** 2 * cfg.head_dim * cfg.batch * cfg.n_head * cfg.n_layer
    return 6.0 * n_params * N + attn


def matmul_flops(cfg) -> float:
    """Dense GEMM + attention FLOPs actually executed as products (no embedding gather)."""
    N, C, F, V, L = cfg.batch * cfg.seq_len, cfg.d_model, cfg.d_mlp, cfg.vocab, cfg.n_layer
    gemm = 3 * 2 * N * (L * (3 * C * C + C * C + 2 * C * F) + C * V)
    attn = 6.0 * cfg.seq_len ** 2 * cfg.head_dim * cfg.batch * cfg.n_head * cfg.n_layer
    return gemm + attn


def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d.get("bf16_tflops"), d.get("hbm_gbs"), "measured"
    return 1900.0, 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples during the timed region."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, interval_ms: int = 50):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", str(interval_ms)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[3:7]))
            except ValueError:
                continue
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v.lower() == "active"})
        max_mhz = max(r[1] for r in rows)
        loaded = [r[0] for r in rows if r[0] > 0.3 * max_mhz] or [r[0] for r in rows]
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max_mhz, "reasons": reasons,
                "samples": len(rows)}


def dist_setup(n_gpus: int):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = os.environ.get("BENCH_BACKEND", "nccl")
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def cpu_baseline(cfg, seed: int, budget_s: float = 15.0):
    """The oracle, as it stands, on the host cores: one-sequence steps of the
    workload's model until the time budget is spent (at least one)."""
    from oracle import gpt_oracle as O
    from persistent_gpt_step_gb300 import inputs as I
    sub = cfg.replace(batch=1)
    params = I.init_params(O.param_table(sub), seed)
    st = O.OracleState(sub, params, dtype=np.float64)
    t0 = time.perf_counter()
    steps = 0
    while True:
        tok, tgt = I.batch(sub, seed, steps)
        O.train_step(st, tok, tgt)
        steps += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    tokens = steps * sub.seq_len
    return {"value": tokens / dt, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{steps} oracle steps (fp64 numpy) of the same model on 1 x {sub.seq_len} tokens "
                      f"in {dt:.1f} s", "ms_per_step": 1000 * dt / steps}


def run_reference(args, cfg):
    rank, world, _ = int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), 0
    if rank != 0:
        return
    from oracle import gpt_oracle as O
    from persistent_gpt_step_gb300 import inputs as I
    # each timed step is a bounded sample: one sequence of the workload's model
    sub = cfg.replace(batch=1)
    params = I.init_params(O.param_table(sub), args.seed)
    st = O.OracleState(sub, params, dtype=np.float64)
    for s in range(args.warmup):
        O.train_step(st, *I.batch(sub, args.seed, s))
    t0 = time.perf_counter()
    for s in range(args.steps):
        O.train_step(st, *I.batch(sub, args.seed, args.warmup + s))
    dt = time.perf_counter() - t0
    value = args.steps * sub.seq_len / dt
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * dt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            # what this arm runs: the same model, one sequence of the workload's batch per step
            "config": {"workload": workload_name(sub), "global_batch": sub.batch, "seq_len": sub.seq_len,
                       "parallelism": "host cores", "params": O.num_params(cfg),
                       "sample_of": workload_name(cfg),
                       "tokens": "Zipf(1.1) synthetic" if cfg.tokens == "zipf" else "uniform synthetic"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                             "sample": f"{args.steps} oracle steps (fp64 numpy), each on 1 of the {cfg.batch} "
                                       f"sequences of a batch ({sub.seq_len} tokens)"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def workload_name(cfg) -> str:
    return (f"GPT {cfg.n_layer}L/{cfg.d_model}/{cfg.n_head}H F{cfg.d_mlp} V{cfg.vocab}, "
            f"seq {cfg.seq_len} x batch {cfg.batch}, AdamW fp32 master")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=4)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="main")
    ap.add_argument("--seed", type=int, default=1234)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    from persistent_gpt_step_gb300 import inputs as I
    cfg = I.CONFIGS[args.config]
    if args.impl == "reference":
        run_reference(args, cfg)
        return

    import torch
    from persistent_gpt_step_gb300 import binding as B
    rank, world, local = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    B.load()

    n_batches = 64
    host_batches = [I.batch(cfg, args.seed + 1000 * rank, s) for s in range(n_batches)]
    dev_batches = [(torch.from_numpy(t).to(dev), torch.from_numpy(g).to(dev)) for t, g in host_batches]
    stream = torch.cuda.current_stream(dev)
    model = B.GPT(cfg, seed=args.seed, stream=stream)
    arena_gb = model.arena_bytes / 1e9
    n_params = model.n_params
    N = cfg.batch * cfg.seq_len

    # ---- device-resident inputs -------------------------------------------------
    for s in range(args.warmup):
        model.train_step(*dev_batches[s % n_batches])
    torch.cuda.synchronize(dev)
    barrier(world)
    clocks = ClockSampler(local) if rank == 0 else None
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    kernel_ms = []
    losses = []
    ev0.record(stream)
    for s in range(args.steps):
        losses.append(model.train_step(*dev_batches[(args.warmup + s) % n_batches]))
        kernel_ms.append(model.last_kernel_ms())
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    t_dev = max_over_ranks(ev0.elapsed_time(ev1) / 1000.0, world, dev)

    # ---- end to end: host buffers through the C ABI (H2D/D2H inside) ----------
    pinned = [(torch.from_numpy(t).pin_memory(), torch.from_numpy(g).pin_memory()) for t, g in host_batches[:8]]
    model.train_step(*[x.numpy() for x in pinned[0]])
    torch.cuda.synchronize(dev)
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for s in range(args.steps):
        t, g = pinned[s % len(pinned)]
        model.train_step(t.numpy(), g.numpy())
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    t_e2e = max_over_ranks(e0.elapsed_time(e1) / 1000.0, world, dev)

    # ---- the same K steps as one multi-step call (no host sync between steps) ---
    ring = [dev_batches[(args.warmup + s) % n_batches] for s in range(args.steps)]
    ring_tok = torch.stack([t for t, _ in ring]).contiguous()
    ring_tgt = torch.stack([g for _, g in ring]).contiguous()
    torch.cuda.synchronize(dev)
    barrier(world)
    m0, m1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    m0.record(stream)
    model.train_steps(ring_tok, ring_tgt)
    m1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    # the sampler ran through the three timed regions (device, end-to-end, multi-step)
    clk = clocks.stop() if clocks else None
    t_multi = max_over_ranks(m0.elapsed_time(m1) / 1000.0, world, dev)
    model.close()

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    flops = model_flops(cfg, n_params)
    peak_tf, peak_hbm, peak_kind = read_peaks()
    kern_s = statistics.mean(kernel_ms) / 1000.0
    achieved = flops / kern_s / 1e12
    line = {
        "metric": METRIC,
        "value": world * args.steps * N / t_dev,
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": 1000.0 * t_dev / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": workload_name(cfg), "global_batch": cfg.batch * world, "seq_len": cfg.seq_len,
                   "parallelism": "replicas" if world > 1 else "single-gpu",
                   "params": n_params, "l2": f"working set ({arena_gb:.1f} GB arena) > L2; no flush",
                   "tokens": "Zipf(1.1) synthetic, 64 pre-uploaded batches"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak_tf, "unit": "TFLOP/s",
                     "frac": achieved / peak_tf if peak_tf else None,
                     "traffic": measured_traffic(workload_name(cfg)),
                     "peak_kind": f"{peak_kind} bf16 burst",
                     "flops_per_launch": flops, "matmul_flops_per_launch": matmul_flops(cfg),
                     "kernel": "pgs::gpt_step_kernel<bf16> (the whole step)",
                     "kernel_ms": 1000 * kern_s},
        "e2e": {"value": world * args.steps * N / t_e2e, "unit": UNIT,
                "h2d_bytes_per_step": 2 * N * 4, "d2h_bytes_per_step": 4 * 4 + 4},
        "multi_step_call": {"value": world * args.steps * N / t_multi, "unit": UNIT, "steps_per_call": args.steps,
                            "ms_per_step": 1000.0 * t_multi / args.steps},
        "gpu_launches": args.steps,
        "ptxas": ptxas_report(),
        "clocks": clk,
        "loss_first_last": [losses[0], losses[-1]],
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, args.seed)
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
