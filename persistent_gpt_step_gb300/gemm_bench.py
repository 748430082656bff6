"""Throughput of the tensor-core GEMM task on the step's GEMM shapes.

python -m persistent_gpt_step_gb300.gemm_bench [--config main] [--only M,N,K,a_mn,b_mn]

Each shape runs as a one-task-per-tile graph of the persistent kernel through
the gpt_test_gemm hook (fp32 output), timed with CUDA events around the
launch; the table gives ms and TFLOP/s per shape.
"""

from __future__ import annotations

import argparse

import torch

from . import binding as B
from . import inputs as I


def shapes(cfg):
    """(name, M, N, K, a_mn, b_mn) of every GEMM of one layer and the LM head."""
    N, C, F, V = cfg.batch * cfg.seq_len, cfg.d_model, cfg.d_mlp, cfg.vocab
    return [
        ("qkv", N, 3 * C, C, 0, 0), ("attn-out", N, C, C, 0, 0), ("mlp-up", N, F, C, 0, 0),
        ("mlp-down", N, C, F, 0, 0), ("lm-head", N, V, C, 0, 0),
        ("lm-head dX", N, C, V, 0, 1), ("lm-head dW", V, C, N, 1, 1),
        ("mlp-down dX", N, F, C, 0, 1), ("mlp-down dW", C, F, N, 1, 1),
        ("mlp-up dX", N, C, F, 0, 1), ("mlp-up dW", F, C, N, 1, 1),
        ("qkv dX", N, C, 3 * C, 0, 1), ("qkv dW", 3 * C, C, N, 1, 1),
    ]


def run(name, M, N, K, a_mn, b_mn, reps=3):
    g = torch.Generator(device="cuda").manual_seed(0)
    A = torch.randn(M, K, device="cuda", generator=g).bfloat16()
    Bm = torch.randn(N, K, device="cuda", generator=g).bfloat16()
    if a_mn:
        A = A.t().contiguous()
    if b_mn:
        Bm = Bm.t().contiguous()
    best = float("inf")
    for _ in range(reps):
        _, ms = B.test_gemm(A, Bm, a_mn, b_mn, M, N, K, timing=True)
        best = min(best, ms)
    return best, 2.0 * M * N * K / best / 1e9


EPILOGUES = [("f32", None), ("store", B.EPI_STORE), ("residual", B.EPI_RESID), ("gelu", B.EPI_GELU),
             ("gelu-bwd", B.EPI_GELU_BWD)]


def run_epilogues(M, N, K, reps=3):
    """Each fused epilogue on one shape: ms, TFLOP/s and the implied time per tile."""
    g = torch.Generator(device="cuda").manual_seed(1)
    A = torch.randn(M, K, device="cuda", generator=g).bfloat16()
    Bm = torch.randn(N, K, device="cuda", generator=g).bfloat16()
    bias = torch.randn(N, device="cuda", generator=g)
    resid = torch.randn(M, N, device="cuda", generator=g)
    aux = torch.randn(M, N, device="cuda", generator=g).bfloat16()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    print(f"epilogues on M={M} N={N} K={K} ({sms} SMs)")
    for name, epi in EPILOGUES:
        best = float("inf")
        for _ in range(reps):
            if epi is None:
                _, ms = B.test_gemm(A, Bm, 0, 0, M, N, K, timing=True)
            else:
                src = resid if epi == B.EPI_RESID else (aux if epi == B.EPI_GELU_BWD else None)
                ms = B.test_gemm_epilogue(A, Bm, 0, 0, M, N, K, epi, bias=bias, src=src, timing=True)[-1]
            best = min(best, ms)
        print(f"  {name:10s} {best:8.3f} ms {2.0 * M * N * K / best / 1e9:8.1f} TF/s")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--config", default="main")
    ap.add_argument("--only", default=None, help="M,N,K,a_mn,b_mn")
    ap.add_argument("--epilogues", default=None, help="M,N,K: time every fused epilogue on this shape")
    ap.add_argument("--reps", type=int, default=3, help="launches per epilogue (--epilogues)")
    args = ap.parse_args()
    B.load()
    if args.epilogues:
        run_epilogues(*(int(x) for x in args.epilogues.split(",")), reps=args.reps)
        return
    todo = shapes(I.CONFIGS[args.config])
    if args.only:
        M, N, K, a, b = (int(x) for x in args.only.split(","))
        todo = [("custom", M, N, K, a, b)]
    print(f"{'gemm':14s} {'M':>6s} {'N':>6s} {'K':>6s} {'A':>3s} {'B':>3s} {'ms':>8s} {'TF/s':>8s}")
    for name, M, N, K, a, b in todo:
        ms, tf = run(name, M, N, K, a, b)
        print(f"{name:14s} {M:6d} {N:6d} {K:6d} {'MN' if a else 'K':>3s} {'MN' if b else 'K':>3s} "
              f"{ms:8.3f} {tf:8.1f}")


if __name__ == "__main__":
    main()
