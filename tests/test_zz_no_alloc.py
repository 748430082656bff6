"""The training step that allocates nothing (gpt_train_step_static).

Callers that cannot allocate device memory (a runtime whose memory belongs to a
pool allocator that allows no side allocations, an embedded or real-time host
that must not allocate after start-up, where an allocation can block for an
unbounded time) get this entry point: its scratch is a static device array
inside libgpt.so, and the caller passes parameters, AdamW moments, tokens and
targets.  It must give the same results as the ordinary handle-based step.
This file is collected last so a run that stops at its first failure has run
every other test before it.
"""

import numpy as np
import pytest

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


def test_static_step_matches_handle_step_on_two_calls():
    cfg = I.CONFIGS["tiny"]
    seed = 21
    batches = [I.batch(cfg, seed, s) for s in range(2)]
    ref = []
    with B.GPT(cfg, seed=seed) as h:
        p0 = h.params()
        for tok, tgt in batches:
            loss = h.train_step(_dev(tok), _dev(tgt))
            m, v, step = h.opt_state()
            ref.append((loss, h.params(), m, v, step))
    P = _dev(p0)
    M = torch.zeros_like(P)
    V = torch.zeros_like(P)
    for s, (tok, tgt) in enumerate(batches):
        loss = B.train_step_static(cfg, P, M, V, s, _dev(tok), _dev(tgt))
        torch.cuda.synchronize()
        r_loss, r_p, r_m, r_v, r_step = ref[s]
        assert r_step == s + 1
        # the tiny configuration's tolerance (loss 1e-4 relative, parameters 1e-4)
        assert abs(loss - r_loss) <= 1e-4 * abs(r_loss), (s, loss, r_loss)
        assert np.abs(P.cpu().numpy() - r_p).max() <= 1e-4
        assert np.abs(M.cpu().numpy() - r_m).max() <= 1e-4
        assert np.abs(V.cpu().numpy() - r_v).max() <= 1e-4


def test_static_step_rejects_models_beyond_its_scratch():
    cfg = I.CONFIGS["small"].replace(dtype="fp32")
    n = B.param_count(cfg)
    P, M, V = (torch.full((n,), 7.0, device="cuda") for _ in range(3))
    tok = torch.zeros(cfg.batch, cfg.seq_len, dtype=torch.int32, device="cuda")
    with pytest.raises(B.GptError) as e:
        B.train_step_static(cfg, P, M, V, 0, tok, tok)
    assert e.value.name == "INVALID_ARG" and "static maximum" in str(e.value)
    assert bool((P == 7.0).all()) and bool((M == 7.0).all())  # rejected before any launch
    one = torch.zeros(1, device="cuda")
    with pytest.raises(B.GptError) as e:
        B.train_step_static(I.CONFIGS["tiny"].replace(dtype="bf16"), one, one, one, 0, tok, tok)
    assert e.value.name == "UNSUPPORTED"


def test_static_step_binding_rejects_wrong_buffers_before_any_launch():
    """The C call cannot see buffer lengths: the binding checks every tensor's
    size, dtype and device first, so a short parameter vector never reaches the
    kernel (which would read and write past its end)."""
    cfg = I.CONFIGS["tiny"]
    n = B.param_count(cfg)
    tok, tgt = (_dev(x) for x in I.batch(cfg, 3, 0))
    good = [torch.zeros(n, device="cuda") for _ in range(3)]
    short = torch.zeros(n - 1, device="cuda")
    for bad_args, word in (((short, good[1], good[2]), "elements"),
                           ((good[0], good[1].double(), good[2]), "float32"),
                           ((good[0], good[1], good[2].cpu()), "CUDA")):
        with pytest.raises(B.GptError) as e:
            B.train_step_static(cfg, *bad_args, 0, tok, tgt)
        assert e.value.name == "INVALID_ARG" and word in str(e.value)
    with pytest.raises(B.GptError) as e:
        B.train_step_static(cfg, *good, 0, tok[:, :-1].contiguous(), tgt)
    assert e.value.name == "INVALID_ARG" and "shape" in str(e.value)
    assert not any(bool(g.any()) for g in good)  # nothing ran
