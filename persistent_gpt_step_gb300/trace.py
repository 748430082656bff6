"""Per-family time table of one training step from the in-kernel trace.

python -m persistent_gpt_step_gb300.trace [--config main] [--steps 3] [--save t.npz]
                                          [--windows 0,1.85,2.55,7.0,8.0]
python -m persistent_gpt_step_gb300.trace --load t.npz --windows ...   (no GPU needed)

The kernel stamps every task's claim, start (after its dependency waits) and
end (after its release) with %globaltimer.  Per operation family this prints
the summed busy time (sum of end - start over its tasks, divided by the number
of blocks: the family's share of the step if blocks never idled), the summed
dependency-wait time and the wall-clock span from its first start to its last
end — the shape of the per-family table on "Coppelius training on the RTX
3090" (section "Where a step's time goes"), measured inside one launch.
"""

from __future__ import annotations

import argparse
import json
import sys

import numpy as np

FAMILIES = ["embed", "layernorm-fwd", "gemm", "attention-fwd", "cross-entropy", "loss",
            "layernorm-bwd", "column-sum", "attention-bwd", "embedding-bwd-wte",
            "embedding-bwd-wpe", "adamw", "attention-bwd-pre", "attention-bwd-kv", "attention-bwd-q",
            "token-sort", "nop"]


def family_table(trace: np.ndarray, task_ops: np.ndarray, op_types, grid: int):
    """Rows (family, tasks, busy_ms_per_block, wait_ms_per_block, span_ms)."""
    claim = trace[:, 0].astype(np.int64)
    start = trace[:, 1].astype(np.int64)
    end = trace[:, 2].astype(np.int64)
    t0 = start.min()
    fam_of_task = np.asarray(op_types)[task_ops]
    rows = []
    for f in sorted(set(fam_of_task.tolist())):
        sel = fam_of_task == f
        busy = (end[sel] - start[sel]).sum() / 1e6 / grid
        wait = (start[sel] - claim[sel]).sum() / 1e6 / grid
        span = (end[sel].max() - start[sel].min()) / 1e6
        rows.append((FAMILIES[f], int(sel.sum()), busy, wait, span,
                     (start[sel].min() - t0) / 1e6, (end[sel].max() - t0) / 1e6))
    total = (end.max() - claim.min()) / 1e6
    return rows, total


def window_shares(trace: np.ndarray, task_ops: np.ndarray, op_types, grid: int, bounds_ms):
    """Per window [bounds_ms[i], bounds_ms[i+1]) of the launch (ms from its first
    claim) and per family: the share of the grid's time its tasks executed (start to
    end) and waited (claim to start) inside the window.  Tasks of one GEMM run
    overlap (tile i+1's mainloop runs under tile i's epilogue), so a window's GEMM
    share counts that overlap twice.  Returns [(lo, hi, {family: (exec, wait)})]."""
    claim = trace[:, 0].astype(np.int64)
    start = trace[:, 1].astype(np.int64)
    end = trace[:, 2].astype(np.int64)
    t0 = claim.min()
    c, s, e = (claim - t0) / 1e6, (start - t0) / 1e6, (end - t0) / 1e6
    fam = np.asarray(op_types)[task_ops]
    out = []
    for lo, hi in zip(bounds_ms[:-1], bounds_ms[1:]):
        cap = (hi - lo) * grid
        ex = np.clip(np.minimum(e, hi) - np.maximum(s, lo), 0, None)
        wt = np.clip(np.minimum(s, hi) - np.maximum(c, lo), 0, None)
        shares = {}
        for f in sorted(set(fam.tolist())):
            sel = fam == f
            x, w = ex[sel].sum() / cap, wt[sel].sum() / cap
            if x > 0 or w > 0:
                shares[FAMILIES[f]] = (float(x), float(w))
        out.append((lo, hi, shares))
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--config", default="main")
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--json", default=None)
    ap.add_argument("--ops", action="store_true", help="print every op's first start / last end")
    ap.add_argument("--save", default=None, help="write the raw trace and the task graph to this .npz")
    ap.add_argument("--load", default=None, help="analyse a trace saved with --save instead of running (no GPU)")
    ap.add_argument("--windows", default=None,
                    help="comma-separated window bounds in ms from the launch start: per-window family shares")
    args = ap.parse_args()
    if args.load:
        d = np.load(args.load)
        tr, task_ops, op_types, grid = d["trace"], d["task_ops"], list(d["op_types"]), int(d["grid"])
        rows, total = family_table(tr, task_ops, op_types, grid)
        print(f"saved trace: {len(tr)} tasks, grid {grid}, kernel {float(d['kernel_ms']):.3f} ms, "
              f"traced span {total:.3f} ms")
        for r in sorted(rows, key=lambda r: -r[2]):
            print(f"{r[0]:20s} {r[1]:7d} {r[2]:9.3f} {r[3]:9.3f} {r[4]:9.3f} {r[5]:8.3f} {r[6]:8.3f}")
        if args.windows:
            print_windows(window_shares(tr, task_ops, op_types, grid, [float(x) for x in args.windows.split(",")]))
        return 0
    import torch

    from . import binding as B
    from . import inputs as I
    cfg = I.CONFIGS[args.config]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    tasks, op_types, op_ntasks, op_dims = B.describe_graph(cfg, sms, dims=True)
    task_ops = np.array([t[0] for t in tasks])
    with B.GPT(cfg, seed=1234) as m:
        n, grid, _ = m.graph_info()
        assert n == len(tasks), (n, len(tasks))
        m.trace_enable(True)
        for s in range(args.steps):
            tok, tgt = I.batch(cfg, 1234, s)
            m.train_step(torch.from_numpy(tok).cuda(), torch.from_numpy(tgt).cuda())
        tr = m.trace()
        kms = m.last_kernel_ms()
    if args.save:
        waits = np.full((len(tasks), 3, 3), -1, dtype=np.int64)
        for i, t in enumerate(tasks):
            for w, (first, count, need) in enumerate(t[3]):
                waits[i, w] = (first, count, need)
        np.savez_compressed(args.save, trace=tr, task_ops=task_ops, task_idx=np.array([t[1] for t in tasks]),
                            task_sig=np.array([t[2] for t in tasks]), task_sig2=np.array([t[4] for t in tasks]),
                            task_waits=waits, op_types=np.asarray(op_types), op_dims=np.asarray(op_dims),
                            grid=grid, kernel_ms=kms)
    rows, total = family_table(tr, task_ops, op_types, grid)
    print(f"config {args.config}: {n} tasks, grid {grid}, kernel {kms:.3f} ms, traced span {total:.3f} ms")
    print(f"{'family':20s} {'tasks':>7s} {'busy ms':>9s} {'wait ms':>9s} {'span ms':>9s} {'first':>8s} {'last':>8s}")
    for r in sorted(rows, key=lambda r: -r[2]):
        print(f"{r[0]:20s} {r[1]:7d} {r[2]:9.3f} {r[3]:9.3f} {r[4]:9.3f} {r[5]:8.3f} {r[6]:8.3f}")
    # per-op spans of the GEMMs (first start to last end), with their achieved rate
    start = tr[:, 1].astype(np.int64)
    end = tr[:, 2].astype(np.int64)
    t0 = start.min()
    print(f"\n{'gemm op':>7s} {'M':>6s} {'N':>6s} {'K':>6s} {'BN':>4s} {'tiles':>6s} {'span us':>8s} {'TF/s':>7s} "
          f"{'begin':>8s}")
    for o, ty in enumerate(op_types):
        if ty != 2:
            continue
        sel = task_ops == o
        span = (end[sel].max() - start[sel].min()) / 1e3
        M, N, K, BN = op_dims[o][:4]
        print(f"{o:7d} {M:6d} {N:6d} {K:6d} {BN:4d} {op_ntasks[o]:6d} {span:8.1f} "
              f"{2.0 * M * N * K / span / 1e6:7.1f} {(start[sel].min() - t0) / 1e6:8.3f}")
    if args.ops:
        print(f"\n{'op':>5s} {'family':20s} {'tasks':>6s} {'start':>8s} {'end':>8s} {'busy/blk':>9s}")
        rows = []
        for o, ty in enumerate(op_types):
            sel = task_ops == o
            rows.append(((start[sel].min() - t0) / 1e6, o, ty, int(sel.sum()), (end[sel].max() - t0) / 1e6,
                         (end[sel] - start[sel]).sum() / 1e6 / grid))
        for st, o, ty, nt, en, busy in sorted(rows):
            print(f"{o:5d} {FAMILIES[ty]:20s} {nt:6d} {st:8.3f} {en:8.3f} {busy:9.4f}")
    if args.windows:
        print_windows(window_shares(tr, task_ops, op_types, grid, [float(x) for x in args.windows.split(",")]))
    if args.json:
        json.dump({"config": args.config, "kernel_ms": kms, "grid": grid, "rows": rows}, open(args.json, "w"))


def print_windows(wins):
    for lo, hi, shares in wins:
        print(f"\nwindow {lo:.2f}-{hi:.2f} ms")
        for f, (x, w) in sorted(shares.items(), key=lambda kv: -kv[1][0]):
            print(f"  {f:20s} exec {100 * x:5.1f} %  wait {100 * w:5.1f} %")


if __name__ == "__main__":
    sys.exit(main())
