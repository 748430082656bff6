"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the CPU oracle.

This module holds workload definitions (shapes and hyper-parameters) and the
random-number streams that feed a training step: initial weights and token
batches.  It holds none of the model's arithmetic and imports nothing else from
this package, so the oracle and the CUDA path can both be fed from it without
sharing any of the method's code.

Workloads.  The 162M GPT (12 layers, width 768, 12 heads, 8 x 512 tokens a step,
AdamW) is the model of the A100 reproduction ("Open Flapping Airplanes" experiment
record, section "What ran"); the same 162.4M model and 4,096 tokens a step are
the training workload of "How one persistent kernel runs three jobs" (section
"Fewer launches do not guarantee fastest training").  The tiny, small and 350M
configurations are a debugging, a mid-size and a scale-up variant of the same
architecture.  The dataset of those pages (tokenized TinyStories) is not
available here; seeded Zipf(s=1.1) unigram streams stand in for it, with the
same shapes (B sequences of T tokens, targets = inputs shifted by one).

Random streams (a written specification, implemented independently in the C
library's host code and here):

* SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014): ``out(state, n) = mix(state + (n + 1) * GAMMA)``
  with GAMMA = 0x9E3779B97F4A7C15 and ``mix`` the published finaliser
  (xor-shift 30, x 0xBF58476D1CE4E5B9, xor-shift 27, x 0x94D049BB133111EB,
  xor-shift 31), all modulo 2**64.  ``out(state, n)`` is the n-th output of the
  generator seeded with ``state``, computed counter-style.
* Tensor t of the canonical parameter order has key ``k_t = out(seed, t)``.
  Element e draws ``u1 = (out(k_t, 2e) >> 11) * 2**-53`` and
  ``u2 = (out(k_t, 2e + 1) >> 11) * 2**-53``; Box-Muller in double precision,
  ``z = sqrt(-2 ln(1 - u1)) * cos(2 pi u2)``; the weight is ``fp32(0.02 * z)``
  (round to nearest even).  Bias tensors start at 0, LayerNorm gains at 1 and
  LayerNorm biases at 0.
* Token batch of step s has key ``k = out(seed, 2**40 + s)``; draw j (row-major
  over a [B, T + 1] block) is ``u_j = (out(k, j) >> 11) * 2**-53``.  Uniform:
  ``floor(u_j * V)``.  Zipf(s): P(id = r - 1) is proportional to r**-s for
  r = 1..V; the id is the smallest r - 1 with ``cdf[r] >= u_j``, where ``cdf`` is
  the running double-precision sum of r**-s divided by its total.  Inputs are
  columns 0..T-1 and targets columns 1..T of the block.
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np

GAMMA = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB
DATA_TAG = 1 << 40


@dataclasses.dataclass(frozen=True)
class GPTConfig:
    """Shapes and hyper-parameters of one GPT training workload."""

    name: str
    n_layer: int
    d_model: int
    n_head: int
    d_mlp: int
    vocab: int
    seq_len: int
    batch: int
    dtype: str = "bf16"          # "fp32": every tensor fp32; "bf16": bf16 compute, fp32 master
    linear_bias: bool = True
    ln_bias: bool = True
    gelu_tanh: bool = True
    rope: bool = False            # rotary position embedding on q, k (no learned position table)
    gated_mlp: bool = False       # gated-GELU MLP: GELU(x W_g^T) * (x W_u^T), then W_2
    tie_embeddings: bool = False  # the LM head is the token embedding
    lr: float = 6e-4
    beta1: float = 0.9
    beta2: float = 0.95
    eps: float = 1e-8
    weight_decay: float = 0.1
    ln_eps: float = 1e-5
    wd_on_1d: bool = False
    tokens: str = "zipf"         # "zipf" or "uniform"
    zipf_s: float = 1.1
    steps: int = 10

    @property
    def head_dim(self) -> int:
        return self.d_model // self.n_head

    @property
    def n_tokens(self) -> int:
        return self.batch * self.seq_len

    def replace(self, **kw) -> "GPTConfig":
        return dataclasses.replace(self, **kw)


CONFIGS = {
    "tiny": GPTConfig("tiny", 2, 64, 4, 256, 256, 64, 4, dtype="fp32", lr=1e-3,
                      tokens="uniform", steps=10),
    "small": GPTConfig("small", 4, 256, 4, 1024, 4096, 256, 8, lr=6e-4, steps=100),
    "main": GPTConfig("main", 12, 768, 12, 3072, 50304, 512, 8, lr=6e-4, steps=4000),
    "350m": GPTConfig("350m", 24, 1024, 16, 4096, 50304, 1024, 8, lr=6e-4, steps=500),
    # the RTX 3090 page's 57.7M model: RoPE, gated-GELU FFN 1408, tied embeddings,
    # no linear biases, one 1,024-token sequence per step
    "57m": GPTConfig("57m", 16, 512, 8, 1408, 12288, 1024, 1, lr=6e-4, steps=2000, linear_bias=False,
                     rope=True, gated_mlp=True, tie_embeddings=True),
    # the 162M model's shapes with two layers: profiling captures of one operation
    # at the step's own sizes with a few GB on the device
    "main_2l": GPTConfig("main_2l", 2, 768, 12, 3072, 50304, 512, 8, lr=6e-4, steps=10),
    # the same architecture at a size the parity tests run quickly
    "small_gated": GPTConfig("small_gated", 4, 256, 4, 704, 4096, 256, 4, lr=6e-4, steps=50, linear_bias=False,
                             rope=True, gated_mlp=True, tie_embeddings=True),
}


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * np.uint64(_M1)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(_M2)
    return z ^ (z >> np.uint64(31))


def splitmix64(state: int, n: np.ndarray) -> np.ndarray:
    """Outputs number ``n`` (uint64 array) of SplitMix64 seeded with ``state``."""
    with np.errstate(over="ignore"):
        n = np.asarray(n, dtype=np.uint64)
        z = np.uint64(state % (1 << 64)) + (n + np.uint64(1)) * np.uint64(GAMMA)
        return _mix(z)


def splitmix64_scalar(state: int, n: int) -> int:
    return int(splitmix64(state, np.array([n], dtype=np.uint64))[0])


def _unit(words: np.ndarray) -> np.ndarray:
    return (words >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal_fp32(seed: int, tensor_index: int, numel: int, std: float = 0.02,
                chunk: int = 1 << 24) -> np.ndarray:
    """fp32 N(0, std) weights of one tensor, per the Box-Muller spec above."""
    key = splitmix64_scalar(seed, tensor_index)
    out = np.empty(numel, dtype=np.float32)
    for lo in range(0, numel, chunk):
        hi = min(numel, lo + chunk)
        e = np.arange(lo, hi, dtype=np.uint64)
        u1 = _unit(splitmix64(key, e * np.uint64(2)))
        u2 = _unit(splitmix64(key, e * np.uint64(2) + np.uint64(1)))
        z = np.sqrt(-2.0 * np.log(1.0 - u1)) * np.cos(2.0 * math.pi * u2)
        out[lo:hi] = (std * z).astype(np.float32)
    return out


def init_params(table, seed: int) -> np.ndarray:
    """Flat fp32 parameter vector in canonical order.

    ``table`` is a sequence of ``(name, shape, kind)`` with kind one of
    ``"normal"``, ``"zeros"``, ``"ones"``; tensor index = position in the table.
    """
    parts = []
    for t, (_name, shape, kind) in enumerate(table):
        numel = int(np.prod(shape))
        if kind == "normal":
            parts.append(normal_fp32(seed, t, numel))
        elif kind == "zeros":
            parts.append(np.zeros(numel, dtype=np.float32))
        elif kind == "ones":
            parts.append(np.ones(numel, dtype=np.float32))
        else:
            raise ValueError(f"unknown init kind {kind!r}")
    return np.concatenate(parts) if parts else np.zeros(0, np.float32)


_ZIPF_CACHE: dict = {}


def zipf_cdf(vocab: int, s: float) -> np.ndarray:
    key = (vocab, s)
    if key not in _ZIPF_CACHE:
        w = np.arange(1, vocab + 1, dtype=np.float64) ** (-s)
        c = np.cumsum(w)
        _ZIPF_CACHE[key] = c / c[-1]
    return _ZIPF_CACHE[key]


def token_block(seed: int, step: int, batch: int, seq_len: int, vocab: int,
                dist: str = "zipf", s: float = 1.1) -> np.ndarray:
    """int32 [batch, seq_len + 1] token ids for one step."""
    key = splitmix64_scalar(seed, DATA_TAG + step)
    n = batch * (seq_len + 1)
    u = _unit(splitmix64(key, np.arange(n, dtype=np.uint64)))
    if dist == "uniform":
        ids = np.floor(u * vocab).astype(np.int64)
    elif dist == "zipf":
        ids = np.searchsorted(zipf_cdf(vocab, s), u, side="left")
    else:
        raise ValueError(f"unknown token distribution {dist!r}")
    ids = np.minimum(ids, vocab - 1)
    return ids.astype(np.int32).reshape(batch, seq_len + 1)


def batch(cfg: GPTConfig, seed: int, step: int):
    """(tokens, targets), each int32 [B, T], for step ``step`` of workload ``cfg``."""
    blk = token_block(seed, step, cfg.batch, cfg.seq_len, cfg.vocab, cfg.tokens, cfg.zipf_s)
    return np.ascontiguousarray(blk[:, :-1]), np.ascontiguousarray(blk[:, 1:])
