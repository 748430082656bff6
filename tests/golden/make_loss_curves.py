"""Writes the oracle's per-step loss curves that the bf16 GPU parity tests compare
against (tests/golden/<config>_loss_curve_<steps>.txt).

Only the CPU oracle and the seeded input generators run here: the weights come
from the initialisation specification, the token batches from the Zipf(s = 1.1)
streams, and every loss is the fp32 oracle's forward loss before its update
(the reference loss curve of a bf16 training run: "Open Flapping Airplanes"
experiment record, sections "What ran" and "Measured results", a loss record
per step of the 8 x 512-token AdamW step).

Usage (from the repository root; about 20-40 s per 162M step on 8 cores):
    python tests/golden/make_loss_curves.py main 50
    python tests/golden/make_loss_curves.py 57m 50
    python tests/golden/make_loss_curves.py 350m 10
"""

from __future__ import annotations

import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from oracle import gpt_oracle as O  # noqa: E402
from persistent_gpt_step_gb300 import inputs as I  # noqa: E402

SEED = 1234


def path_for(name: str, steps: int) -> str:
    return os.path.join(HERE, f"{name}_loss_curve_{steps}.txt")


def read_curve(name: str, steps: int) -> np.ndarray:
    """Losses of a committed curve file (one per step, in order)."""
    vals = []
    with open(path_for(name, steps)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                s, v = line.split()
                assert int(s) == len(vals), (s, len(vals))
                vals.append(float(v))
    assert len(vals) == steps, (len(vals), steps)
    return np.array(vals)


def main(name: str, steps: int) -> None:
    cfg = I.CONFIGS[name]
    params = I.init_params(O.param_table(cfg), SEED)
    st = O.OracleState(cfg, params, dtype=np.float32)
    out = path_for(name, steps)
    tmp = out + ".partial"
    t0 = time.time()
    with open(tmp, "w") as f:
        f.write(f"# fp32 CPU oracle loss per step, configuration '{name}' "
                f"({cfg.n_layer}L d{cfg.d_model} H{cfg.n_head} F{cfg.d_mlp} V{cfg.vocab} "
                f"T{cfg.seq_len} B{cfg.batch}), seed {SEED}, Zipf batches 0..{steps - 1}, "
                f"constant lr {cfg.lr}\n")
        f.write(f"# written by: python tests/golden/make_loss_curves.py {name} {steps}\n")
        f.write("# step  pre-update mean cross-entropy\n")
        for s in range(steps):
            tok, tgt = I.batch(cfg, SEED, s)
            loss = O.train_step(st, tok, tgt)
            f.write(f"{s} {loss:.9g}\n")
            f.flush()
            print(f"{name} step {s}: {loss:.6f} ({time.time() - t0:.0f} s)", flush=True)
    os.replace(tmp, out)


if __name__ == "__main__":
    main(sys.argv[1], int(sys.argv[2]))
