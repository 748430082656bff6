"""Pins of the CPU oracle against things other than itself (no GPU)."""

import math
import os

import numpy as np
import pytest

from oracle import gpt_oracle as O
from persistent_gpt_step_gb300 import inputs as I

GOLD = os.path.join(os.path.dirname(__file__), "golden")

TINY = I.CONFIGS["tiny"]
# an even smaller model for the exhaustive checks
MICRO = TINY.replace(name="micro", n_layer=2, d_model=16, n_head=2, d_mlp=32, vocab=11,
                     seq_len=6, batch=2)


def _tiny_inputs(cfg, seed=7, step=0):
    params = I.init_params(O.param_table(cfg), seed).astype(np.float64)
    tok, tgt = I.batch(cfg, seed, step)
    return params, tok, tgt


def _read_kv(path):
    out = {}
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        k, v = line.split(None, 1)
        out[k] = v
    return out


# ----------------------------------------------------------------- page values

def test_param_counts_match_pages():
    for line in open(os.path.join(GOLD, "param_counts.txt")):
        if not line.strip() or line.startswith("#"):
            continue
        name, L, C, H, F, V, T, lb, nb, count = line.split()
        cfg = TINY.replace(n_layer=int(L), d_model=int(C), n_head=int(H), d_mlp=int(F),
                           vocab=int(V), seq_len=int(T), linear_bias=bool(int(lb)),
                           ln_bias=bool(int(nb)))
        assert O.num_params(cfg) == int(count), name


def test_param_count_closed_form():
    for cfg in I.CONFIGS.values():
        L, C, V, T, F = cfg.n_layer, cfg.d_model, cfg.vocab, cfg.seq_len, cfg.d_mlp
        lb, nb = int(cfg.linear_bias), int(cfg.ln_bias)
        fw = 2 * F if cfg.gated_mlp else F     # rows of the first MLP matrix
        per_layer = (2 + 2 * nb) * C + (3 * C * C + lb * 3 * C) + (C * C + lb * C) + (fw * C + lb * fw) \
            + (C * F + lb * C)
        emb = V * C + (0 if cfg.rope else T * C) + (0 if cfg.tie_embeddings else V * C)
        assert O.num_params(cfg) == L * per_layer + emb + (1 + nb) * C, cfg.name


def test_gated_rope_tied_model_is_the_pages_57_7m():
    """The RTX 3090 page's model: 57.7M parameters (its config list and summary)."""
    assert round(O.num_params(I.CONFIGS["57m"]) / 1e5) / 10 == 57.7


def test_rope_rotation_preserves_pairs_and_depends_on_offsets_only():
    """Rotary embedding: each (2i, 2i+1) pair keeps its length, rotating by -theta undoes
    it, and the score of a query at position m with a key at n depends only on m - n."""
    rng = np.random.default_rng(3)
    T, d = 40, 16
    th = O.rope_angles(T, d)
    q, k = rng.normal(size=(T, d)), rng.normal(size=(T, d))
    rq = O.rope_rotate(q, th)
    assert np.allclose(rq[:, 0::2] ** 2 + rq[:, 1::2] ** 2, q[:, 0::2] ** 2 + q[:, 1::2] ** 2, rtol=1e-12)
    assert np.allclose(O.rope_rotate(rq, th, -1.0), q, rtol=1e-12, atol=1e-14)
    qv, kv = rng.normal(size=d), rng.normal(size=d)
    Q, K = O.rope_rotate(np.tile(qv, (T, 1)), th), O.rope_rotate(np.tile(kv, (T, 1)), th)
    for m, n, shift in ((9, 3, 17), (20, 20, 11), (5, 1, 30)):
        assert Q[m] @ K[n] == pytest.approx(Q[m + shift] @ K[n + shift], rel=1e-10)
    assert np.allclose(th[0], 0.0) and th[1, 0] == 1.0 and th[3, 1] == pytest.approx(3 * 10000 ** (-2 / d))


def test_know_nothing_loss_is_ln_vocab():
    g = _read_kv(os.path.join(GOLD, "know_nothing_loss.txt"))
    V = int(g["vocab"])
    cfg = MICRO.replace(vocab=V, seq_len=8, batch=2)
    rng = np.random.default_rng(0)
    params = rng.normal(0, 0.02, O.num_params(cfg))
    O.param_views(cfg, params)["w_lm"][...] = 0.0       # every token equally likely
    tok = rng.integers(0, V, (2, 8))
    tgt = rng.integers(0, V, (2, 8))
    loss, _ = O.forward(cfg, params, tok, tgt)
    assert round(loss, int(g["decimals"])) == float(g["loss"])
    assert abs(loss - math.log(V)) < 1e-12


def test_initial_loss_near_ln_vocab_uniform_tokens():
    params, tok, tgt = _tiny_inputs(TINY)
    loss, _ = O.forward(TINY, params, tok, tgt)
    assert abs(loss - math.log(TINY.vocab)) < 0.05


# ----------------------------------------------------------------- invariants

def test_softmax_rows_sum_to_one_and_dz_rows_to_zero():
    rng = np.random.default_rng(1)
    z = rng.normal(0, 3, (64, 300))
    p = O.softmax_rows(z)
    assert np.abs(p.sum(1) - 1).max() < 1e-6
    t = rng.integers(0, 300, 64)
    loss, rows, dz = O.cross_entropy(z, t)
    assert np.abs(dz.sum(1)).max() < 1e-12
    # the row loss is -log p[target]
    assert np.allclose(rows, -np.log(p[np.arange(64), t]), rtol=1e-12)


def test_cross_entropy_matches_logsumexp_definition():
    rng = np.random.default_rng(2)
    z = rng.normal(0, 2, (5, 7))
    t = rng.integers(0, 7, 5)
    loss, rows, _ = O.cross_entropy(z, t)
    ref = [math.log(sum(math.exp(v) for v in z[i])) - z[i, t[i]] for i in range(5)]
    assert np.allclose(rows, ref, rtol=1e-13)
    assert abs(loss - sum(ref) / 5) < 1e-13


def test_causality():
    params, tok, tgt = _tiny_inputs(TINY)
    _, c0 = O.forward(TINY, params, tok, tgt)
    tok2 = tok.copy()
    t = 37
    tok2[:, t] = (tok2[:, t] + 101) % TINY.vocab
    _, c1 = O.forward(TINY, params, tok2, tgt)
    z0 = c0["z"].reshape(TINY.batch, TINY.seq_len, -1)
    z1 = c1["z"].reshape(TINY.batch, TINY.seq_len, -1)
    assert np.array_equal(z0[:, :t], z1[:, :t])
    assert not np.allclose(z0[:, t:], z1[:, t:])


def test_attention_single_position_returns_v():
    rng = np.random.default_rng(3)
    q, k, v = (rng.normal(size=(2, 3, 1, 8)) for _ in range(3))
    o, p = O.causal_attention(q, k, v)
    assert np.array_equal(p, np.ones_like(p))
    assert np.allclose(o, v, rtol=0, atol=0)


def test_attention_matches_per_row_loop():
    rng = np.random.default_rng(4)
    q, k, v = (rng.normal(size=(1, 1, 5, 4)) for _ in range(3))
    o, _ = O.causal_attention(q, k, v)
    for i in range(5):
        s = [float(q[0, 0, i] @ k[0, 0, j]) / 2.0 for j in range(i + 1)]
        w = np.exp(np.array(s) - max(s))
        w /= w.sum()
        assert np.allclose(o[0, 0, i], (w[:, None] * v[0, 0, :i + 1]).sum(0), rtol=1e-13)


def test_layernorm_moments():
    rng = np.random.default_rng(5)
    x = rng.normal(3, 7, (10, 64))
    y, xhat, _ = O.layernorm(x, np.ones(64), np.zeros(64), 1e-5)
    assert np.abs(xhat.mean(1)).max() < 1e-12
    assert np.abs(xhat.var(1) - 1).max() < 1e-5     # eps shifts the variance by ~eps/49
    assert np.array_equal(y, xhat)


def test_gelu_special_values():
    x = np.linspace(-6, 6, 2001)
    assert O.gelu(np.array([0.0]))[0] == 0.0
    assert abs(O.gelu_grad(np.array([0.0]))[0] - 0.5) < 1e-15
    # the tanh form approximates the erf form within 1e-3 everywhere
    assert np.abs(O.gelu(x, True) - O.gelu(x, False)).max() < 1e-3
    assert abs(O.gelu(np.array([30.0]))[0] - 30.0) < 1e-12
    # derivative against central differences
    h = 1e-6
    fd = (O.gelu(x + h) - O.gelu(x - h)) / (2 * h)
    assert np.abs(fd - O.gelu_grad(x)).max() < 1e-8
    fd = (O.gelu(x + h, False) - O.gelu(x - h, False)) / (2 * h)
    assert np.abs(fd - O.gelu_grad(x, False)).max() < 1e-8


# ----------------------------------------------------------------- gradients

def _loss(cfg, params, tok, tgt):
    return O.forward(cfg, params, tok, tgt, keep=False)[0]


def _one_blas_thread():
    try:
        from threadpoolctl import threadpool_limits
        return threadpool_limits(1)
    except ImportError:          # not installed everywhere; only slower without it
        import contextlib
        return contextlib.nullcontext()


GATED = TINY.replace(name="tiny_gated", rope=True, gated_mlp=True, tie_embeddings=True, d_mlp=96)


@pytest.mark.parametrize("variant", ["gpt2", "gated_rope_tied", "gated_rope_tied_bias"])
def test_finite_differences_tiny_fp64(variant):
    """Central differences on >=200 scalars per tensor (all of the small ones)."""
    cfg = {"gpt2": TINY, "gated_rope_tied": GATED.replace(linear_bias=False),
           "gated_rope_tied_bias": GATED}[variant]
    with _one_blas_thread():
        _finite_differences_tiny_fp64(cfg)


def _finite_differences_tiny_fp64(cfg):
    params, tok, tgt = _tiny_inputs(cfg, seed=11)
    # non-trivial LN/bias values so their gradients are exercised
    rng = np.random.default_rng(12)
    views = O.param_views(cfg, params)
    for name, arr in views.items():
        if name.endswith(("_b", "_g", "b_qkv", "b_o", "b_1", "b_2", "b_gu")):
            arr += rng.normal(0, 0.1, arr.shape)
    _, cache = O.forward(cfg, params, tok, tgt)
    grad = O.backward(cfg, params, cache)
    gv = O.param_views(cfg, grad)
    off = 0
    for name, shape, _ in O.param_table(cfg):
        n = int(np.prod(shape))
        idx = np.arange(n) if n <= 256 else rng.choice(n, 200, replace=False)
        if name == "wte":   # rows of tokens that occur (the others have zero gradient)
            rows = np.unique(tok)[:40]
            idx = np.unique(np.concatenate([idx, (rows[:, None] * shape[1] + np.arange(5)).ravel()]))
        fd = np.empty(len(idx))
        for j, e in enumerate(idx):
            p0 = params[off + e]
            h = 1e-6 * max(1.0, abs(p0))
            params[off + e] = p0 + h
            lp = _loss(cfg, params, tok, tgt)
            params[off + e] = p0 - h
            lm = _loss(cfg, params, tok, tgt)
            params[off + e] = p0
            fd[j] = (lp - lm) / (2 * h)
        an = gv[name].reshape(-1)[idx]
        scale = max(np.abs(an).max(), 1e-12)
        err = np.abs(fd - an).max() / scale
        assert err <= 1e-4, (name, err)
        off += n


def _torch_loss(cfg, params, tok, tgt):
    """Independent re-statement with PyTorch CPU library operators (float64)."""
    import torch
    import torch.nn.functional as F
    t = torch.tensor(params, dtype=torch.float64, requires_grad=True)
    B, T = tok.shape
    z = _torch_logits(cfg, t, tok)
    loss = F.cross_entropy(z.view(B * T, -1), torch.tensor(tgt, dtype=torch.long).view(-1))
    loss.backward()
    return float(loss), t.grad.numpy()


def _torch_logits(cfg, t, tok):
    """Logits [B, T, V] of the same re-statement; t: the float64 parameter tensor."""
    import torch
    import torch.nn.functional as F
    views, off = {}, 0
    for name, shape, _ in O.param_table(cfg):
        n = int(np.prod(shape))
        views[name] = t[off:off + n].view(*shape)
        off += n
    B, T = tok.shape
    C, H = cfg.d_model, cfg.n_head
    tk = torch.tensor(tok, dtype=torch.long)
    x = F.embedding(tk, views["wte"])
    if not cfg.rope:
        x = x + views["wpe"][:T][None]
    d = C // H
    # rotary embedding as a complex product: pair (2i, 2i+1) times exp(j t w_i)
    w = 1.0 / (10000.0 ** (torch.arange(0, d, 2, dtype=torch.float64) / d))
    rot = torch.polar(torch.ones(T, d // 2, dtype=torch.float64), torch.arange(T, dtype=torch.float64)[:, None] * w)

    def rope(u):  # [B, H, T, d]
        c = torch.view_as_complex(u.reshape(B, H, T, d // 2, 2).contiguous())
        return torch.view_as_real(c * rot).reshape(B, H, T, d)

    for l in range(cfg.n_layer):
        p = f"h{l}."
        a = F.layer_norm(x, (C,), views[p + "ln1_g"], views.get(p + "ln1_b"), cfg.ln_eps)
        qkv = F.linear(a, views[p + "w_qkv"], views.get(p + "b_qkv"))
        q, k, v = qkv.split(C, dim=-1)
        q, k, v = (u.view(B, T, H, C // H).transpose(1, 2) for u in (q, k, v))
        if cfg.rope:
            q, k = rope(q), rope(k)
        o = F.scaled_dot_product_attention(q, k, v, is_causal=True)
        o = o.transpose(1, 2).reshape(B, T, C)
        x = x + F.linear(o, views[p + "w_o"], views.get(p + "b_o"))
        a = F.layer_norm(x, (C,), views[p + "ln2_g"], views.get(p + "ln2_b"), cfg.ln_eps)
        approx = "tanh" if cfg.gelu_tanh else "none"
        if cfg.gated_mlp:
            gu = F.linear(a, views[p + "w_gu"], views.get(p + "b_gu"))
            h = F.gelu(gu[..., 0::2], approximate=approx) * gu[..., 1::2]
        else:
            h = F.gelu(F.linear(a, views[p + "w_1"], views.get(p + "b_1")), approximate=approx)
        x = x + F.linear(h, views[p + "w_2"], views.get(p + "b_2"))
    x = F.layer_norm(x, (C,), views["lnf_g"], views.get("lnf_b"), cfg.ln_eps)
    return F.linear(x, views["wte" if cfg.tie_embeddings else "w_lm"])


@pytest.mark.parametrize("variant", ["tiny", "gated_rope_tied"])
def test_greedy_decode_against_torch_restatement(variant):
    """Every token of the oracle's greedy generation is the argmax of the PyTorch
    re-statement's next-token logits over the same prefix, and the logits it was
    chosen from match that re-statement; generation stops at no fixed point (the
    oracle recomputes the whole prefix for every token)."""
    torch = pytest.importorskip("torch")
    cfg = TINY if variant == "tiny" else GATED.replace(linear_bias=False)
    params, tok, _ = _tiny_inputs(cfg, seed=12)
    rng = np.random.default_rng(13)
    params = params + rng.normal(0, 0.3, params.shape)   # a model with strong preferences: no near-ties
    prompt = tok[0, :5]
    gen, zs = O.greedy_decode(cfg, params, prompt, 12)
    seq = list(prompt)
    t = torch.tensor(params, dtype=torch.float64)
    for i, g in enumerate(gen):
        z = _torch_logits(cfg, t, np.array([seq]))[0, -1].numpy()
        assert int(np.argmax(z)) == int(g), i
        assert np.allclose(zs[i], z, rtol=1e-10, atol=1e-10)
        seq.append(int(g))
    assert len(gen) == 12 and len(set(gen.tolist())) > 1


@pytest.mark.parametrize("variant", ["tiny", "nobias_erf", "gated_rope_tied", "gated_rope_tied_erf_bias"])
def test_against_torch_autograd_fp64(variant):
    cfg = {"tiny": TINY, "nobias_erf": TINY.replace(linear_bias=False, ln_bias=False, gelu_tanh=False),
           "gated_rope_tied": GATED.replace(linear_bias=False),
           "gated_rope_tied_erf_bias": GATED.replace(gelu_tanh=False)}[variant]
    params, tok, tgt = _tiny_inputs(cfg, seed=5)
    rng = np.random.default_rng(6)
    params = params + rng.normal(0, 0.05, params.shape)   # move LN / biases off their init
    loss, cache = O.forward(cfg, params, tok, tgt)
    grad = O.backward(cfg, params, cache)
    tl, tg = _torch_loss(cfg, params, tok, tgt)
    assert abs(loss - tl) < 1e-12 * abs(tl)
    assert np.abs(grad - tg).max() < 1e-10 * np.abs(tg).max()


# ----------------------------------------------------------------- AdamW

def test_adamw_first_two_steps_closed_form():
    cfg = MICRO
    rng = np.random.default_rng(8)
    n = O.num_params(cfg)
    p0 = rng.normal(0, 1, n)
    g1, g2 = rng.normal(0, 1e-2, n), rng.normal(0, 1e-2, n)
    lr, wd, b1, b2, eps = cfg.lr, cfg.weight_decay, cfg.beta1, cfg.beta2, cfg.eps
    dec = O.decay_mask(cfg)
    p, m, v = p0.copy(), np.zeros(n), np.zeros(n)
    O.adamw(cfg, p, g1, m, v, 1)
    # bias correction cancels on the first step: update = g / (|g| + eps)
    p1 = p0 * (1 - lr * wd * dec) - lr * g1 / (np.abs(g1) + eps)
    assert np.allclose(p, p1, rtol=1e-14, atol=1e-16)
    O.adamw(cfg, p, g2, m, v, 2)
    m2 = b1 * (1 - b1) * g1 + (1 - b1) * g2
    v2 = b2 * (1 - b2) * g1 ** 2 + (1 - b2) * g2 ** 2
    p2 = p1 * (1 - lr * wd * dec) - lr * (m2 / (1 - b1 ** 2)) / (np.sqrt(v2 / (1 - b2 ** 2)) + eps)
    assert np.allclose(p, p2, rtol=1e-13, atol=1e-16)


def test_adamw_first_two_steps_closed_form_with_scheduled_rates():
    """The same closed form with a different rate on each step (the rate scales both
    the decoupled decay and the Adam step of that update only)."""
    cfg = MICRO
    rng = np.random.default_rng(9)
    n = O.num_params(cfg)
    p0 = rng.normal(0, 1, n)
    g1, g2 = rng.normal(0, 1e-2, n), rng.normal(0, 1e-2, n)
    wd, b1, b2, eps = cfg.weight_decay, cfg.beta1, cfg.beta2, cfg.eps
    lr1, lr2 = 2.5e-4, 7.5e-4
    dec = O.decay_mask(cfg)
    p, m, v = p0.copy(), np.zeros(n), np.zeros(n)
    O.adamw(cfg, p, g1, m, v, 1, lr=lr1)
    p1 = p0 * (1 - lr1 * wd * dec) - lr1 * g1 / (np.abs(g1) + eps)
    assert np.allclose(p, p1, rtol=1e-14, atol=1e-16)
    O.adamw(cfg, p, g2, m, v, 2, lr=lr2)
    m2 = b1 * (1 - b1) * g1 + (1 - b1) * g2
    v2 = b2 * (1 - b2) * g1 ** 2 + (1 - b2) * g2 ** 2
    p2 = p1 * (1 - lr2 * wd * dec) - lr2 * (m2 / (1 - b1 ** 2)) / (np.sqrt(v2 / (1 - b2 ** 2)) + eps)
    assert np.allclose(p, p2, rtol=1e-13, atol=1e-16)


def test_lr_schedule_closed_forms():
    """Warmup + cosine: linear ramp values, lr_max at the end of the warmup, the mean
    of lr_max and lr_min half-way through the decay, lr_min at and after the end,
    the half-period symmetry of the cosine about that midpoint, monotone decay."""
    hi, lo, w, tot = 6e-4, 6e-5, 100, 4000
    for t in (1, 37, 100):
        assert O.lr_at(t, hi, lo, w, tot) == pytest.approx(hi * t / w, rel=1e-15)
    assert O.lr_at(w, hi, lo, w, tot) == pytest.approx(hi, rel=1e-15)
    assert O.lr_at(w + (tot - w) // 2, hi, lo, w, tot) == pytest.approx((hi + lo) / 2, rel=1e-12)
    assert O.lr_at(tot, hi, lo, w, tot) == lo and O.lr_at(tot + 5, hi, lo, w, tot) == lo
    for x in (1, 250, 1234):
        a = O.lr_at(w + x, hi, lo, w, tot) - lo
        b = hi - O.lr_at(tot - x, hi, lo, w, tot)
        assert a == pytest.approx(b, rel=1e-9)
    seq = [O.lr_at(t, hi, lo, w, tot) for t in range(w, tot + 1)]
    assert all(x >= y for x, y in zip(seq, seq[1:]))
    # no warmup: the first update already follows the cosine, just below lr_max
    assert lo < O.lr_at(1, hi, lo, 0, tot) < hi


def _decays_by_name(name: str) -> bool:
    """GPT-2 convention written from parameter names alone: weight decay on the
    weight matrices and embeddings (w_*, wte, wpe, w_lm), none on biases or
    LayerNorm gains and biases."""
    leaf = name.split(".")[-1]
    return leaf in ("wte", "wpe", "w_lm") or leaf.startswith("w_")


@pytest.mark.parametrize("variant", ["tiny", "gated_rope_tied"])
def test_adamw_matches_torch_optim_adamw(variant):
    """Three AdamW updates of the oracle against torch.optim.AdamW (float64, CPU),
    with two parameter groups built from the parameter names (decay / no decay)
    and a different learning rate on each update: a decayed LayerNorm gain or
    bias, an undecayed matrix, a wrong bias correction or a wrong moment update
    each fails this."""
    torch = pytest.importorskip("torch")
    cfg = MICRO if variant == "tiny" else MICRO.replace(rope=True, gated_mlp=True, tie_embeddings=True,
                                                         linear_bias=False)
    table = O.param_table(cfg)
    rng = np.random.default_rng(31)
    n = O.num_params(cfg)
    p0 = rng.normal(0, 0.5, n)
    grads = [rng.normal(0, 1e-2, n) for _ in range(3)]
    rates = [3e-3, 1e-3, 2e-3]
    # torch: one tensor per parameter, grouped by name
    tensors, off = [], 0
    for name, shape, _ in table:
        k = int(np.prod(shape))
        tensors.append((name, off, k, torch.tensor(p0[off:off + k], dtype=torch.float64, requires_grad=True)))
        off += k
    decay = [t for name, _, _, t in tensors if _decays_by_name(name)]
    no_decay = [t for name, _, _, t in tensors if not _decays_by_name(name)]
    assert decay and no_decay
    opt = torch.optim.AdamW([{"params": decay, "weight_decay": cfg.weight_decay},
                             {"params": no_decay, "weight_decay": 0.0}],
                            lr=rates[0], betas=(cfg.beta1, cfg.beta2), eps=cfg.eps)
    p, m, v = p0.copy(), np.zeros(n), np.zeros(n)
    for step, (g, lr) in enumerate(zip(grads, rates), start=1):
        for grp in opt.param_groups:
            grp["lr"] = lr
        for _, o, k, t in tensors:
            t.grad = torch.tensor(g[o:o + k], dtype=torch.float64)
        opt.step()
        O.adamw(cfg, p, g, m, v, step, lr=lr)
        ref = np.concatenate([t.detach().numpy() for _, _, _, t in tensors])
        assert np.allclose(p, ref, rtol=1e-13, atol=1e-15), (step, np.abs(p - ref).max())
        ref_m = np.concatenate([opt.state[t]["exp_avg"].numpy() for _, _, _, t in tensors])
        ref_v = np.concatenate([opt.state[t]["exp_avg_sq"].numpy() for _, _, _, t in tensors])
        assert np.allclose(m, ref_m, rtol=1e-13, atol=1e-18)
        assert np.allclose(v, ref_v, rtol=1e-13, atol=1e-20)


@pytest.mark.parametrize("gated", [False, True])
def test_decay_mask_follows_parameter_names(gated):
    """The decay mask against the GPT-2 naming rule (matrices and embeddings
    decay; biases and LayerNorm parameters do not), not against tensor ranks."""
    cfg = MICRO.replace(rope=gated, gated_mlp=gated, tie_embeddings=gated, linear_bias=not gated)
    mask = O.decay_mask(cfg)
    off = 0
    for name, shape, _ in O.param_table(cfg):
        n = int(np.prod(shape))
        assert (mask[off:off + n] == (1.0 if _decays_by_name(name) else 0.0)).all(), name
        off += n
    assert off == mask.size
    assert (O.decay_mask(cfg.replace(wd_on_1d=True)) == 1).all()


def test_train_step_decreases_loss_on_repeated_batch():
    cfg = MICRO.replace(lr=1e-2)
    params, tok, tgt = _tiny_inputs(cfg, seed=9)
    st = O.OracleState(cfg, params)
    losses = [O.train_step(st, tok, tgt) for _ in range(20)]
    assert losses[-1] < losses[0] - 0.5


def test_fp32_oracle_tracks_fp64_within_tolerance_tiny():
    """The fp32 tolerance (loss 1e-4 relative, params 1e-4 max-abs over 10 steps) is
    reachable by a correct fp32 implementation: the fp32 oracle meets it."""
    cfg = TINY
    params = I.init_params(O.param_table(cfg), 1234)
    s64 = O.OracleState(cfg, params, dtype=np.float64)
    s32 = O.OracleState(cfg, params, dtype=np.float32)
    for step in range(cfg.steps):
        tok, tgt = I.batch(cfg, 1234, step)
        l64 = O.train_step(s64, tok, tgt)
        l32 = O.train_step(s32, tok, tgt)
        assert abs(l32 - l64) <= 1e-4 * abs(l64)
    assert np.abs(s32.params - s64.params).max() <= 1e-4
