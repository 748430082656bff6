"""Per-phase rates of the training step, one operation of every family at a time.

python -m persistent_gpt_step_gb300.phase_bench [--config main] [--reps 5] [--json out.json]
python -m persistent_gpt_step_gb300.phase_bench --config main_2l --once   (one launch per
    operation, for an ncu capture: the step is launch 1, the operations follow in the
    printed order)

After one full training step (so the arena holds real activations, logit
gradients and weight gradients), each selected operation of the step's graph
runs as its own launch of the same persistent kernel (gpt_run_ops), timed with
CUDA events on the handle's stream.  Per operation the table gives the device
time, the algorithmic work of one launch (FLOPs for GEMMs and attention, bytes for
the rest) and the achieved rate against the measured peak: the bf16 tensor peak
for contractions, the HBM copy bandwidth for the memory-bound families.  A
family whose working set stays in L2 (129 MB) can read above the HBM figure.

The families are those of the per-family table on "Coppelius training on the
RTX 3090" (section "Where a step's time goes"): GEMMs with their fused
epilogues, attention forward and its two backward families, LayerNorm forward
and backward, LayerNorm parameter column sums, cross-entropy, embedding and
embedding scatter, AdamW.
"""

from __future__ import annotations

import argparse
import json
import os

import torch

from . import binding as B
from . import inputs as I

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

OP_EMBED, OP_LN_FWD, OP_GEMM, OP_ATTN_FWD, OP_CE, OP_LOSS, OP_LN_BWD, OP_COLSUM = range(8)
OP_EMB_WTE, OP_EMB_WPE, OP_ADAMW, OP_ATT_PRE, OP_ATT_KV, OP_ATT_Q, OP_SORT = 9, 10, 11, 12, 13, 14, 15


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["bf16_tflops"]), float(d["hbm_gbs"]), "measured"
    return 1900.0, 6800.0, "fallback"


def label_ops(cfg, types, dims):
    """Name of every operation of the step graph (build order: forward, loss,
    backward layer by layer from the last, embeddings), with its layer."""
    N, C, F, V, L, T = cfg.batch * cfg.seq_len, cfg.d_model, cfg.d_mlp, cfg.vocab, cfg.n_layer, cfg.seq_len
    F2 = 2 * F if cfg.gated_mlp else F
    loss_op = types.index(OP_LOSS)
    names = []
    count = {}
    for i, (t, d) in enumerate(zip(types, dims)):
        bwd = i > loss_op
        M, Nn, K = d[0], d[1], d[2]
        if t == OP_GEMM:
            if not bwd:
                key = {(N, 3 * C, C): "gemm qkv (bf16 store + bias)", (N, C, C): "gemm attn-out (+ residual)",
                       (N, F2, C): "gemm mlp-up (+ GELU, GELU')", (N, C, F): "gemm mlp-down (+ residual)",
                       (N, V, C): "gemm lm-head (bf16 logits)"}.get((M, Nn, K), "gemm")
            elif (M, Nn) == (N, C) and K == V:
                key = "gemm lm-head dX (fp32, k-split)"
            elif (M, Nn, K) == (V, C, N):
                key = "gemm lm-head dW (fp32)"
            elif (M, Nn, K) == (N, F, C):
                key = "gemm mlp-down dX (x GELU')"
            elif (M, Nn, K) == (N, C, F2):
                key = "gemm mlp-up dX (fp32)"
            elif (M, Nn, K) == (N, C, C):
                key = "gemm attn-out dX (bf16)"
            elif (M, Nn, K) == (N, C, 3 * C):
                key = "gemm qkv dX (fp32)"
            elif M == C and K == N and Nn >= F:
                key = "gemm mlp-down dW|db (fp32)"
            elif M == F2 and K == N:
                key = "gemm mlp-up dW|db (fp32)"
            elif M == C and K == N:
                key = "gemm attn-out dW|db (fp32)"
            elif M == 3 * C and K == N:
                key = "gemm qkv dW|db (fp32)"
            else:
                key = "gemm"
        else:
            key = {OP_EMBED: "embedding", OP_LN_FWD: "layernorm fwd", OP_ATTN_FWD: "attention fwd",
                   OP_CE: "cross-entropy (+ grad)", OP_LOSS: "loss", OP_LN_BWD: "layernorm bwd",
                   OP_COLSUM: "layernorm gain/bias column sums", OP_EMB_WTE: "embedding bwd (token rows)",
                   OP_EMB_WPE: "embedding bwd (positions)", OP_ADAMW: "adamw", OP_ATT_PRE: "attention bwd D",
                   OP_ATT_KV: "attention bwd dK dV", OP_ATT_Q: "attention bwd dQ",
                   OP_SORT: "token sort"}.get(t, f"op{t}")
        names.append((key, count.get(key, 0)))
        count[key] = count.get(key, 0) + 1
    return names, count


def work(cfg, name, t, ntasks, d, n_params_of_op):
    """(amount, unit) of algorithmic work of one launch of the operation."""
    N, C, F, V, T, Bb, H = (cfg.batch * cfg.seq_len, cfg.d_model, cfg.d_mlp, cfg.vocab, cfg.seq_len, cfg.batch,
                            cfg.n_head)
    hd = C // H
    if t == OP_GEMM:
        return 2.0 * d[0] * d[1] * d[2], "flop"
    attn_fwd = 2.0 * T * T * hd * Bb * H  # causal: half of the 4 T^2 d of the dense products
    if t == OP_ATTN_FWD:
        return attn_fwd, "flop"
    if t == OP_ATT_KV:
        return attn_fwd * 4 / 2, "flop"   # S, dP, dV, dK recomputed / formed per key block
    if t == OP_ATT_Q:
        return attn_fwd * 3 / 2, "flop"   # S, dP, dQ per query block
    if t == OP_ATT_PRE:
        return 2.0 * N * C * 2 + 4.0 * Bb * H * T, "byte"
    if t == OP_EMBED:
        return 4.0 * N * C * 2 + 4.0 * T * C + 4.0 * N, "byte"
    if t == OP_LN_FWD:
        return 6.0 * N * C + 8.0 * N + 8.0 * C, "byte"
    if t == OP_LN_BWD:  # a layer's LN backward: dy, x, incoming residual gradient; out fp32 + bf16; partials
        return 4.0 * N * C * 3 + 6.0 * N * C + 8.0 * N + 8.0 * (N // 32) * C, "byte"
    if t == OP_CE:
        return 4.0 * N * V + 8.0 * N, "byte"
    if t == OP_ADAMW:
        return 30.0 * n_params_of_op, "byte"
    if t == OP_EMB_WTE:
        return 4.0 * N * C + 8.0 * N + 4.0 * V * C, "byte"
    if t == OP_EMB_WPE:
        return 4.0 * N * C + 4.0 * T * C, "byte"
    if t == OP_COLSUM:
        return 4.0 * (N // 32) * C + 4.0 * C, "byte"
    return 0.0, "byte"


def select(names, types, cfg):
    """Operation indices to measure: one of each family, at a middle layer."""
    L = cfg.n_layer
    want = {}
    for i, (key, k) in enumerate(names):
        if types[i] in (OP_LOSS,):
            continue
        per_layer = key.startswith("gemm") and "lm-head" not in key or key in (
            "attention fwd", "attention bwd D", "attention bwd dK dV", "attention bwd dQ")
        if key == "layernorm fwd":
            target = 2 * (L // 2)               # LN1 of the middle layer
        elif key == "layernorm bwd":
            target = 1                           # LN2 backward of the last layer (LN-final is 0)
        elif key == "adamw":
            continue
        elif per_layer:
            target = L // 2
        else:
            target = 0
        if k == target:
            want[key] = i
    return want


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--config", default="main")
    ap.add_argument("--reps", type=int, default=5)
    ap.add_argument("--once", action="store_true", help="one launch per operation, no warm-up (ncu captures)")
    ap.add_argument("--json", default=None)
    args = ap.parse_args()
    cfg = I.CONFIGS[args.config]
    torch.cuda.set_device(0)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    tasks, types, ntasks, dims = B.describe_graph(cfg, sms, dims=True)
    names, _ = label_ops(cfg, types, dims)
    tok, tgt = (torch.from_numpy(x).cuda() for x in I.batch(cfg, 1234, 0))
    peak_tf, peak_gbs, peak_kind = peaks()
    rows = []
    with B.GPT(cfg, seed=1234) as m:
        m.train_step(tok, tgt)
        table = m.tensor_table()
        want = select(names, types, cfg)
        # AdamW: the token embedding's update (the largest tensor)
        adam_ops = [i for i, t in enumerate(types) if t == OP_ADAMW]
        biggest = max(adam_ops, key=lambda i: ntasks[i])
        want["adamw (token embedding)"] = biggest
        wte_numel = [int(s[0]) * int(s[1]) for n, s, _ in table if n == "wte"][0]
        order = sorted(want.items(), key=lambda kv: kv[1])
        if args.once:
            for key, i in order:
                print(f"launch: op {i:4d} {key}", flush=True)
                m.run_ops(i, 1, tok, tgt, reps=1)
            return
        for key, i in order:
            m.run_ops(i, 1, tok, tgt, reps=1)  # warm-up (instruction cache, L2 state of this op)
            ms = m.run_ops(i, 1, tok, tgt, reps=args.reps)
            amount, unit = work(cfg, key, types[i], ntasks[i], dims[i],
                                wte_numel if types[i] == OP_ADAMW else 0)
            if unit == "flop":
                rate = amount / (ms * 1e-3) / 1e12
                frac = rate / peak_tf
                runit = "TFLOP/s"
            else:
                rate = amount / (ms * 1e-3) / 1e9
                frac = rate / peak_gbs
                runit = "GB/s"
            rows.append({"op": i, "family": key, "tasks": ntasks[i], "ms": ms, "work": amount, "work_unit": unit,
                         "rate": rate, "rate_unit": runit, "frac_of_peak": frac})
    print(f"| op | family | tasks | ms | algorithmic work | rate | of {peak_kind} peak |")
    print("|---|---|---|---|---|---|---|")
    for r in rows:
        w = f"{r['work'] / 1e9:.2f} GFLOP" if r["work_unit"] == "flop" else f"{r['work'] / 1e6:.1f} MB"
        print(f"| {r['op']} | {r['family']} | {r['tasks']} | {r['ms']:.4f} | {w} | {r['rate']:.0f} {r['rate_unit']} "
              f"| {r['frac_of_peak']:.3f} |")
    if args.json:
        with open(args.json, "w") as f:
            json.dump({"config": args.config, "peaks": {"bf16_tflops": peak_tf, "hbm_gbs": peak_gbs,
                                                       "kind": peak_kind}, "rows": rows}, f, indent=1)


if __name__ == "__main__":
    main()
