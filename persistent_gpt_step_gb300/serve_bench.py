"""Throughput of the serving partition on a workload's model (162M by default).

python -m persistent_gpt_step_gb300.serve_bench [--config main] [--blocks 24] [--tokens 256]
                                                [--per-step 8] [--steps 20]

1. Serving alone: one launch in which `blocks` blocks generate `tokens` tokens
   greedily (batch 1) after a 16-token prompt; tokens/s = generated tokens /
   the launch's device time.
2. Training with serving beside it: `steps` training steps (162M: 8 x 512
   tokens each) while `blocks` blocks run `per-step` decode steps per training
   step from the weights training updates; reports ms per training step and the
   serving tokens/s over the same device time, and the training step alone on
   all blocks for comparison.  ("Open Flapping Airplanes" record, section "What
   ran": training, serving and Doom share one kernel by SM role; "How one
   persistent kernel runs three jobs": the B200 run gives serving 24 SMs.)
"""

from __future__ import annotations

import argparse
import json

import torch

from . import binding as B
from . import inputs as I


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--config", default="main")
    ap.add_argument("--blocks", type=int, default=24)
    ap.add_argument("--tokens", type=int, default=256)
    ap.add_argument("--per-step", type=int, default=8)
    ap.add_argument("--steps", type=int, default=20)
    args = ap.parse_args()
    cfg = I.CONFIGS[args.config]
    torch.cuda.set_device(0)
    batches = [tuple(torch.from_numpy(x).cuda() for x in I.batch(cfg, 1234, s)) for s in range(args.steps + 3)]
    prompt = I.batch(cfg, 77, 0)[0][0, :16]
    out = {"config": args.config, "blocks": args.blocks}
    with B.GPT(cfg, seed=1234) as m:
        # 1. serving alone
        m.serve_begin(prompt, max_new=args.tokens, blocks=args.blocks)
        m.serve_run(15)  # the prompt's steps (and a warm launch)
        ms = m.serve_run(args.tokens)
        n = len(m.serve_tokens())
        out["serve_only"] = {"tokens": n, "ms": ms, "tokens_per_s": n / (ms * 1e-3)}
        m.serve_end()
        # 2. training alone, then training with serving beside it
        for t, g in batches[:3]:
            m.train_step(t, g)
        tok = torch.stack([t for t, _ in batches[3:]]).contiguous()
        tgt = torch.stack([g for _, g in batches[3:]]).contiguous()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        m.train_steps(tok, tgt)
        e1.record()
        torch.cuda.synchronize()
        alone = e0.elapsed_time(e1) / args.steps
        m.serve_begin(prompt, max_new=min(args.per_step * args.steps + 1, cfg.seq_len - 16), blocks=args.blocks,
                      tokens_per_step=args.per_step)
        torch.cuda.synchronize()
        e0.record()
        m.train_steps(tok, tgt)
        e1.record()
        torch.cuda.synchronize()
        both = e0.elapsed_time(e1)
        gen = len(m.serve_tokens())
        out["train_alone_ms_per_step"] = alone
        out["train_with_serving"] = {"ms_per_step": both / args.steps, "serving_tokens": gen,
                                     "serving_tokens_per_s": gen / (both * 1e-3),
                                     "train_tokens_per_s": args.steps * cfg.batch * cfg.seq_len / (both * 1e-3)}
    print(json.dumps(out))


if __name__ == "__main__":
    main()
