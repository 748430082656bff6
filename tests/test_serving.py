"""The serving partition: greedy generation from the live weights on reserved
blocks of the persistent kernel, next to (or instead of) the training step.

Greedy tokens are checked against the oracle's decode loop teacher-forced on
the GPU's own tokens: every generated token must be a maximum of the oracle's
next-token logits (within the fp32 rounding of the GPU's arithmetic), which is
what is unique about a greedy choice; the oracle uses the same bf16-rounded
weight matrices the serving path reads (fp32 embeddings, LayerNorm parameters
and biases)."""

import numpy as np
import pytest

from oracle import gpt_oracle as O
from persistent_gpt_step_gb300 import binding as B
from persistent_gpt_step_gb300 import inputs as I

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from persistent_gpt_step_gb300 import build
    build.build()
    B.load()
    yield


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _bf16_round(x):
    """Round-to-nearest-even fp32 -> bf16 -> fp32 (the weight copy the kernels read)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32)


def _served_weights(cfg, params):
    """Matrices as the serving GEMVs read them (bf16), everything else fp32."""
    out = np.array(params, dtype=np.float32)
    off = 0
    for name, shape, _ in O.param_table(cfg):
        n = int(np.prod(shape))
        if len(shape) == 2 and name not in ("wte", "wpe"):
            out[off:off + n] = _bf16_round(out[off:off + n])
        off += n
    return out


def _check_greedy(cfg, params, prompt, gen, tol=2e-3):
    w = _served_weights(cfg, params)
    seq = [int(t) for t in prompt]
    for i, g in enumerate(gen):
        z = O.next_token_logits(cfg, w, seq)
        assert 0 <= g < cfg.vocab
        assert z[g] >= z.max() - tol * (1.0 + abs(z.max())), (i, g, int(np.argmax(z)), z[g], z.max())
        seq.append(int(g))


def test_serving_greedy_tokens_match_the_oracle():
    cfg = I.CONFIGS["small"]
    prompt = I.batch(cfg, 3, 0)[0][0, :8]
    with B.GPT(cfg, seed=3) as m:
        p = m.params()
        m.serve_begin(prompt, max_new=24, blocks=16)
        ms = m.serve_run(7 + 24)
        gen = m.serve_tokens()
        m.serve_end()
    assert len(gen) == 24 and ms > 0
    _check_greedy(cfg, p, prompt, gen)


def test_serving_in_two_launches_equals_one():
    cfg = I.CONFIGS["small"]
    prompt = I.batch(cfg, 4, 0)[0][0, :5]
    with B.GPT(cfg, seed=4) as m:
        m.serve_begin(prompt, max_new=12, blocks=8)
        m.serve_run(100)
        one = m.serve_tokens()
        m.serve_begin(prompt, max_new=12, blocks=24)
        m.serve_run(6)
        assert len(m.serve_tokens()) == 2  # steps 0..5: four prompt steps, two generated tokens
        m.serve_run(100)
        two = m.serve_tokens()
    assert np.array_equal(one, two)


def test_serving_budget_crosses_32_bits():
    """The session starts as if so many decode steps had run that its 64-bit
    ticket (steps x tasks per step) passes 2^32 within the first steps — the
    record's serving budget of 4,194,304 iterations x 2,225 tasks per token
    wrapped at exactly that point with a 32-bit product.  The tokens equal those
    of a session that starts at zero."""
    cfg = I.CONFIGS["small"]
    prompt = I.batch(cfg, 6, 0)[0][0, :4]
    with B.GPT(cfg, seed=6) as m:
        m.serve_begin(prompt, max_new=10, blocks=16)
        m.serve_run(100)
        ref = m.serve_tokens()
        # tasks per step of this model: embed, 7 ops per layer, final LN, LM-head slices, argmax
        C, F, H, L, V = cfg.d_model, cfg.d_mlp, cfg.n_head, cfg.n_layer, cfg.vocab
        per_step = 1 + L * (1 + 3 * C // 64 + H + C // 64 + 1 + F // 64 + C // 64) + 1 + V // 64 + 1
        first = (1 << 32) // per_step - 2
        assert first * per_step < (1 << 32) < (first + 4) * per_step
        m.serve_begin(prompt, max_new=10, blocks=16, first_step=first)
        m.serve_run(100)
        got = m.serve_tokens()
        assert int(np.prod([4194304, 2225], dtype=np.int64)) % (1 << 32) == 742391808
    assert np.array_equal(ref, got)


def test_training_beside_serving_is_unchanged():
    """Training with 16 blocks serving next to it gives bitwise the losses and
    parameters of training alone (every reduction has a fixed order, whichever
    blocks run the tasks), and the serving blocks generate from the weights as
    training changes them."""
    cfg = I.CONFIGS["small"]
    batches = [I.batch(cfg, 9, s) for s in range(3)]
    prompt = batches[0][0][0, :6]
    with B.GPT(cfg, seed=9) as a, B.GPT(cfg, seed=9) as b:
        la = [a.train_step(_dev(t), _dev(g)) for t, g in batches]
        b.serve_begin(prompt, max_new=20, blocks=16, tokens_per_step=4)
        lb = [b.train_step(_dev(t), _dev(g)) for t, g in batches]
        assert la == lb
        assert np.array_equal(a.params(), b.params())
        gen = b.serve_tokens()
        assert len(gen) == 3 * 4 - 5  # 12 decode steps: five consume the rest of the prompt
        assert ((gen >= 0) & (gen < cfg.vocab)).all()
        # a multi-step call with serving beside it equals single steps too
        tok = _dev(np.stack([x[0] for x in batches]))
        tgt = _dev(np.stack([x[1] for x in batches]))
        la2 = a.train_steps(tok, tgt)
        lb2 = b.train_steps(tok, tgt)
        assert np.array_equal(la2, lb2)
        assert np.array_equal(a.params(), b.params())
