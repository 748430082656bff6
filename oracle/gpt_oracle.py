"""CPU oracle of one GPT training step: forward, backward and AdamW.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or links
this module: only the tests, the package's smoke check and the benchmark's CPU
baseline leg use it.  It shares no code with the CUDA path.

What it computes is the plain definition of the step the pages describe: a GPT
language model (token and learned position embedding, pre-LN transformer
blocks with causal multi-head attention and a GELU MLP, a final LayerNorm, an
untied LM head, mean softmax cross-entropy), its reverse-mode gradient and one
decoupled-weight-decay Adam (AdamW) update of every parameter
("Open Flapping Airplanes" experiment record, section "What ran": 12 layers,
width 768, 12 heads, 8 x 512 tokens a step, AdamW from seeded weights; the
training role of the persistent kernel is "forward pass, backward pass, and
weight updates", same section, table of SM roles).  The loss is the mean
cross-entropy over every row of the step ("Coppelius training on the RTX 3090",
figure "Loss": "mean over the 1,024 rows of each step's context").

Everything is numpy in a caller-chosen float type (float64 by default); matrix
products are library matmuls.  Where the pages are silent the readings are:
tanh-approximate GELU, LayerNorm eps 1e-5 with biased variance, linear biases on
QKV / attention-out / MLP, none on the LM head, attention scale 1/sqrt(d) with
mask j <= i, no dropout, AdamW eps 1e-8 with bias correction, weight decay on
2-D tensors only, constant learning rate, no gradient clipping, and the returned
loss is the forward loss before the update.

Canonical parameter order (also the flat layout of every parameter-sized
vector): wte [V,C], wpe [T,C], then per layer ln1_g, ln1_b, w_qkv [3C,C],
b_qkv [3C], w_o [C,C], b_o [C], ln2_g, ln2_b, w_1 [F,C], b_1 [F], w_2 [C,F],
b_2 [C]; then lnf_g, lnf_b, w_lm [V,C].  Weight matrices are stored
[out_features, in_features]; a linear layer computes y = x W^T + b.

The RTX 3090 page's 57.7M model ("Coppelius training on the RTX 3090": RoPE on
q/k, gated-GELU FFN, tied embedding and LM head) is the same model with three
switches: ``rope`` rotates each head's dimension pairs (2i, 2i+1) of q and k by
t * 10000^(-2i/d) at position t and drops wpe; ``gated_mlp`` replaces w_1 / b_1
by w_gu [2F,C] / b_gu [2F] whose rows 2f and 2f+1 are the gate and up
projections of feature f, the MLP output being GELU(gate) * up; and
``tie_embeddings`` drops w_lm, the LM head using wte.

Pins (see tests/test_oracle.py): central finite differences in float64 on the
tiny model and its gated / RoPE / tied variant, an independent float64 autograd
re-derivation with PyTorch CPU operators (rotary embedding as a complex
product), the rotary embedding's norm and relative-position properties, the
know-nothing loss ln V printed on the Coppelius page, loss near ln V at
initialisation, softmax rows summing to one, the closed form of the first two
AdamW steps (also with per-step rates), the learning-rate schedule's closed
forms, causality, T = 1 attention, LayerNorm moments, and the parameter counts
printed on the pages.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "param_table", "num_params", "param_views", "decay_mask", "forward", "backward",
    "adamw", "train_step", "OracleState", "layernorm", "gelu", "gelu_grad",
    "causal_attention", "softmax_rows", "cross_entropy", "next_token_logits", "greedy_decode",
]


# --------------------------------------------------------------------------- #
# Parameter table
# --------------------------------------------------------------------------- #

def param_table(cfg):
    """[(name, shape, init_kind)] in canonical order.

    Matrices and embeddings start N(0, 0.02), biases 0, LayerNorm gains 1 and
    LayerNorm biases 0 (seeded weights made on the host: "Open Flapping
    Airplanes" record, "What ran" and "Reproduce the run").
    """
    C, F, V, T = cfg.d_model, cfg.d_mlp, cfg.vocab, cfg.seq_len
    rope = getattr(cfg, "rope", False)
    gated = getattr(cfg, "gated_mlp", False)
    tied = getattr(cfg, "tie_embeddings", False)
    tab = [("wte", (V, C), "normal")]
    if not rope:
        tab.append(("wpe", (T, C), "normal"))
    for l in range(cfg.n_layer):
        p = f"h{l}."
        tab.append((p + "ln1_g", (C,), "ones"))
        if cfg.ln_bias:
            tab.append((p + "ln1_b", (C,), "zeros"))
        tab.append((p + "w_qkv", (3 * C, C), "normal"))
        if cfg.linear_bias:
            tab.append((p + "b_qkv", (3 * C,), "zeros"))
        tab.append((p + "w_o", (C, C), "normal"))
        if cfg.linear_bias:
            tab.append((p + "b_o", (C,), "zeros"))
        tab.append((p + "ln2_g", (C,), "ones"))
        if cfg.ln_bias:
            tab.append((p + "ln2_b", (C,), "zeros"))
        if gated:  # rows 2f and 2f+1: gate and up projection of feature f
            tab.append((p + "w_gu", (2 * F, C), "normal"))
        else:
            tab.append((p + "w_1", (F, C), "normal"))
        if cfg.linear_bias:
            tab.append((p + ("b_gu" if gated else "b_1"), (2 * F if gated else F,), "zeros"))
        tab.append((p + "w_2", (C, F), "normal"))
        if cfg.linear_bias:
            tab.append((p + "b_2", (C,), "zeros"))
    tab.append(("lnf_g", (C,), "ones"))
    if cfg.ln_bias:
        tab.append(("lnf_b", (C,), "zeros"))
    if not tied:
        tab.append(("w_lm", (V, C), "normal"))
    return tab


def num_params(cfg) -> int:
    return sum(int(np.prod(s)) for _, s, _ in param_table(cfg))


def param_views(cfg, flat: np.ndarray) -> dict:
    """Name -> view into the flat vector (shares memory)."""
    out, off = {}, 0
    for name, shape, _ in param_table(cfg):
        n = int(np.prod(shape))
        out[name] = flat[off:off + n].reshape(shape)
        off += n
    assert off == flat.size, (off, flat.size)
    return out


def decay_mask(cfg) -> np.ndarray:
    """1.0 where AdamW applies weight decay: 2-D tensors (all, if wd_on_1d)."""
    parts = []
    for _, shape, _ in param_table(cfg):
        d = 1.0 if (len(shape) == 2 or cfg.wd_on_1d) else 0.0
        parts.append(np.full(int(np.prod(shape)), d))
    return np.concatenate(parts)


# --------------------------------------------------------------------------- #
# Building blocks (plain definitions)
# --------------------------------------------------------------------------- #

def layernorm(x, g, b, eps):
    """y = (x - mean) / sqrt(var + eps) * g + b over the last axis (biased var)."""
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    rstd = 1.0 / np.sqrt(var + eps)
    xhat = (x - mu) * rstd
    y = xhat * g
    if b is not None:
        y = y + b
    return y, xhat, rstd


def layernorm_backward(dy, xhat, rstd, g):
    """(dx, dg, db) of layernorm given the saved normalised input."""
    dxhat = dy * g
    C = xhat.shape[-1]
    dx = rstd * (dxhat - dxhat.sum(-1, keepdims=True) / C
                 - xhat * (dxhat * xhat).sum(-1, keepdims=True) / C)
    dg = (dy * xhat).reshape(-1, C).sum(0)
    db = dy.reshape(-1, C).sum(0)
    return dx, dg, db


_K0 = math.sqrt(2.0 / math.pi)


def gelu(x, tanh_form=True):
    """GELU; tanh form 0.5 x (1 + tanh(sqrt(2/pi)(x + 0.044715 x^3))) or exact erf form."""
    if tanh_form:
        return 0.5 * x * (1.0 + np.tanh(_K0 * (x + 0.044715 * (x * x * x))))
    from scipy.special import erf
    return 0.5 * x * (1.0 + erf(x / math.sqrt(2.0)))


def gelu_grad(x, tanh_form=True):
    """d GELU / dx."""
    if tanh_form:
        u = _K0 * (x + 0.044715 * (x * x * x))
        t = np.tanh(u)
        return 0.5 * (1.0 + t) + 0.5 * x * (1.0 - t * t) * _K0 * (1.0 + 3 * 0.044715 * x * x)
    from scipy.special import erf
    return 0.5 * (1.0 + erf(x / math.sqrt(2.0))) + x * np.exp(-0.5 * x * x) / math.sqrt(2 * math.pi)


def softmax_rows(s):
    """Row softmax with the row maximum subtracted first."""
    m = s.max(axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / e.sum(axis=-1, keepdims=True)


def causal_attention(q, k, v):
    """q, k, v [B, H, T, d] -> (o [B, H, T, d], P [B, H, T, T]).

    S = q k^T / sqrt(d); S[i, j] = -inf for j > i; P = softmax over j; o = P v.
    """
    d = q.shape[-1]
    T = q.shape[-2]
    s = (q @ np.swapaxes(k, -1, -2)) / math.sqrt(d)
    mask = np.triu(np.ones((T, T), dtype=bool), k=1)
    s = np.where(mask, -np.inf, s)
    p = softmax_rows(s)
    return p @ v, p


def causal_attention_backward(q, k, v, p, do):
    """(dq, dk, dv) of causal_attention given its probabilities P."""
    d = q.shape[-1]
    dv = np.swapaxes(p, -1, -2) @ do
    dp = do @ np.swapaxes(v, -1, -2)
    ds = p * (dp - (p * dp).sum(-1, keepdims=True))
    ds = ds / math.sqrt(d)
    dq = ds @ k
    dk = np.swapaxes(ds, -1, -2) @ q
    return dq, dk, dv


def cross_entropy(z, targets):
    """Mean over rows of logsumexp(z_n) - z_n[t_n]; returns (loss, per-row loss, dz).

    dz = (softmax(z) - onehot(t)) / N is the gradient of the mean loss.
    """
    N = z.shape[0]
    m = z.max(axis=1, keepdims=True)
    lse = (m + np.log(np.exp(z - m).sum(axis=1, keepdims=True)))[:, 0]
    rows = lse - z[np.arange(N), targets]
    p = np.exp(z - lse[:, None])
    p[np.arange(N), targets] -= 1.0
    return rows.mean(), rows, p / N


# --------------------------------------------------------------------------- #
# Forward / backward of the whole model
# --------------------------------------------------------------------------- #

def rope_angles(T, d, base=10000.0):
    """theta[t, i] = t * base^(-2i/d): the rotation angle of pair i at position t
    (rotary position embedding, pairs (2i, 2i+1) of each head's dimensions)."""
    i = np.arange(d // 2, dtype=np.float64)
    return np.arange(T, dtype=np.float64)[:, None] * base ** (-2.0 * i / d)[None, :]


def rope_rotate(x, theta, sign=1.0):
    """Rotates pairs (2i, 2i+1) of the last axis of x [..., T, d] by sign * theta[T, d/2]."""
    c, s = np.cos(theta), sign * np.sin(theta)
    x0, x1 = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = x0 * c - x1 * s
    out[..., 1::2] = x0 * s + x1 * c
    return out


def _split_heads(x, B, T, H):
    # [B*T, C] -> [B, H, T, d]
    d = x.shape[1] // H
    return x.reshape(B, T, H, d).transpose(0, 2, 1, 3)


def _merge_heads(x):
    B, H, T, d = x.shape
    return x.transpose(0, 2, 1, 3).reshape(B * T, H * d)


def forward(cfg, params: np.ndarray, tokens: np.ndarray, targets: np.ndarray,
            dtype=np.float64, keep=True):
    """Loss of the step and (if ``keep``) the activations backward needs.

    params: flat parameter vector (any float type; cast to ``dtype``);
    tokens, targets: int [B, T] with ids in [0, V).
    """
    B, T = tokens.shape
    assert T <= cfg.seq_len
    C, H = cfg.d_model, cfg.n_head
    P = param_views(cfg, np.asarray(params, dtype=dtype))
    rope = getattr(cfg, "rope", False)
    gated = getattr(cfg, "gated_mlp", False)
    tied = getattr(cfg, "tie_embeddings", False)
    tok = tokens.reshape(-1)
    pos = np.tile(np.arange(T), B)
    x = P["wte"][tok]
    if not rope:
        x = x + P["wpe"][pos]
    theta = rope_angles(T, C // H) if rope else None
    cache = {"x0": x, "tok": tok, "pos": pos, "B": B, "T": T, "layers": [], "theta": theta}
    for l in range(cfg.n_layer):
        p = f"h{l}."
        lc = {"x_in": x}
        a1, lc["xhat1"], lc["rstd1"] = layernorm(x, P[p + "ln1_g"], P.get(p + "ln1_b"), cfg.ln_eps)
        qkv = a1 @ P[p + "w_qkv"].T
        if cfg.linear_bias:
            qkv = qkv + P[p + "b_qkv"]
        q, k, v = (_split_heads(qkv[:, i * C:(i + 1) * C], B, T, H) for i in range(3))
        if rope:
            q, k = rope_rotate(q, theta), rope_rotate(k, theta)
        o, pr = causal_attention(q, k, v)
        o = _merge_heads(o)
        y = o @ P[p + "w_o"].T
        if cfg.linear_bias:
            y = y + P[p + "b_o"]
        x_mid = x + y
        a2, lc["xhat2"], lc["rstd2"] = layernorm(x_mid, P[p + "ln2_g"], P.get(p + "ln2_b"), cfg.ln_eps)
        if gated:
            hg = a2 @ P[p + "w_gu"].T
            if cfg.linear_bias:
                hg = hg + P[p + "b_gu"]
            h = hg               # [N, 2F]: gate (even columns) and up (odd columns)
            g = gelu(hg[:, 0::2], cfg.gelu_tanh) * hg[:, 1::2]
        else:
            h = a2 @ P[p + "w_1"].T
            if cfg.linear_bias:
                h = h + P[p + "b_1"]
            g = gelu(h, cfg.gelu_tanh)
        y2 = g @ P[p + "w_2"].T
        if cfg.linear_bias:
            y2 = y2 + P[p + "b_2"]
        x = x_mid + y2
        lc.update(a1=a1, q=q, k=k, v=v, p=pr, o=o, a2=a2, h=h, g=g)
        if keep:
            cache["layers"].append(lc)
    af, cache["xhatf"], cache["rstdf"] = layernorm(x, P["lnf_g"], P.get("lnf_b"), cfg.ln_eps)
    z = af @ P["wte" if tied else "w_lm"].T
    loss, rows, dz = cross_entropy(z, targets.reshape(-1))
    cache.update(af=af, z=z, rows=rows, dz=dz, x_final=x)
    return float(loss), (cache if keep else None)


def backward(cfg, params: np.ndarray, cache, dtype=np.float64) -> np.ndarray:
    """Flat gradient of the mean loss w.r.t. every parameter (canonical order)."""
    P = param_views(cfg, np.asarray(params, dtype=dtype))
    grad = np.zeros(num_params(cfg), dtype=dtype)
    G = param_views(cfg, grad)
    B, T, C, H = cache["B"], cache["T"], cfg.d_model, cfg.n_head
    rope = getattr(cfg, "rope", False)
    gated = getattr(cfg, "gated_mlp", False)
    tied = getattr(cfg, "tie_embeddings", False)
    dz = cache["dz"]
    lm = "wte" if tied else "w_lm"
    G[lm][...] += dz.T @ cache["af"]
    daf = dz @ P[lm]
    dx, dg, db = layernorm_backward(daf, cache["xhatf"], cache["rstdf"], P["lnf_g"])
    G["lnf_g"][...] = dg
    if cfg.ln_bias:
        G["lnf_b"][...] = db
    for l in reversed(range(cfg.n_layer)):
        p = f"h{l}."
        lc = cache["layers"][l]
        # MLP: x = x_mid + gelu(a2 W1^T + b1) W2^T + b2
        G[p + "w_2"][...] = dx.T @ lc["g"]
        if cfg.linear_bias:
            G[p + "b_2"][...] = dx.sum(0)
        dgl = dx @ P[p + "w_2"]
        if gated:  # g = GELU(gate) * up
            gate, up = lc["h"][:, 0::2], lc["h"][:, 1::2]
            dh = np.empty_like(lc["h"])
            dh[:, 0::2] = dgl * up * gelu_grad(gate, cfg.gelu_tanh)
            dh[:, 1::2] = dgl * gelu(gate, cfg.gelu_tanh)
            w1 = "w_gu"
        else:
            dh = dgl * gelu_grad(lc["h"], cfg.gelu_tanh)
            w1 = "w_1"
        G[p + w1][...] = dh.T @ lc["a2"]
        if cfg.linear_bias:
            G[p + ("b_gu" if gated else "b_1")][...] = dh.sum(0)
        da2 = dh @ P[p + w1]
        dxm, dg, db = layernorm_backward(da2, lc["xhat2"], lc["rstd2"], P[p + "ln2_g"])
        G[p + "ln2_g"][...] = dg
        if cfg.ln_bias:
            G[p + "ln2_b"][...] = db
        dx_mid = dx + dxm
        # attention: x_mid = x_in + attn(a1) W_o^T + b_o
        G[p + "w_o"][...] = dx_mid.T @ lc["o"]
        if cfg.linear_bias:
            G[p + "b_o"][...] = dx_mid.sum(0)
        do = _split_heads(dx_mid @ P[p + "w_o"], B, T, H)
        dq, dk, dv = causal_attention_backward(lc["q"], lc["k"], lc["v"], lc["p"], do)
        if rope:  # q, k were rotated by theta: their gradients rotate back by -theta
            dq, dk = rope_rotate(dq, cache["theta"], -1.0), rope_rotate(dk, cache["theta"], -1.0)
        dqkv = np.concatenate([_merge_heads(dq), _merge_heads(dk), _merge_heads(dv)], axis=1)
        G[p + "w_qkv"][...] = dqkv.T @ lc["a1"]
        if cfg.linear_bias:
            G[p + "b_qkv"][...] = dqkv.sum(0)
        da1 = dqkv @ P[p + "w_qkv"]
        dxi, dg, db = layernorm_backward(da1, lc["xhat1"], lc["rstd1"], P[p + "ln1_g"])
        G[p + "ln1_g"][...] = dg
        if cfg.ln_bias:
            G[p + "ln1_b"][...] = db
        dx = dx_mid + dxi
    # embeddings: x0 = wte[tok] + wpe[pos]
    np.add.at(G["wte"], cache["tok"], dx)
    if not rope:
        np.add.at(G["wpe"], cache["pos"], dx)
    return grad


# --------------------------------------------------------------------------- #
# AdamW
# --------------------------------------------------------------------------- #

def adamw(cfg, p, g, m, v, step, lr=None):
    """One AdamW update in place; ``step`` is the count after this update (>= 1).

    p <- p - lr*wd*p (decayed tensors); m <- b1 m + (1-b1) g; v <- b2 v + (1-b2) g^2;
    p <- p - lr * (m / (1 - b1^t)) / (sqrt(v / (1 - b2^t)) + eps).
    """
    lr = cfg.lr if lr is None else lr
    wd = cfg.weight_decay * decay_mask(cfg).astype(p.dtype)
    p *= (1.0 - lr * wd)
    m *= cfg.beta1
    m += (1.0 - cfg.beta1) * g
    v *= cfg.beta2
    v += (1.0 - cfg.beta2) * g * g
    mhat = m / (1.0 - cfg.beta1 ** step)
    vhat = v / (1.0 - cfg.beta2 ** step)
    p -= lr * mhat / (np.sqrt(vhat) + cfg.eps)


@dataclass
class OracleState:
    """Parameters and optimizer state of the oracle (all in one float type)."""

    cfg: object
    params: np.ndarray
    m: np.ndarray = None
    v: np.ndarray = None
    step: int = 0
    dtype: type = np.float64
    last_grad: np.ndarray = field(default=None, repr=False)

    def __post_init__(self):
        self.params = np.array(self.params, dtype=self.dtype)
        if self.m is None:
            self.m = np.zeros_like(self.params)
        if self.v is None:
            self.v = np.zeros_like(self.params)


def lr_at(step, lr_max, lr_min, warmup, total):
    """Learning rate of update number ``step`` (1-based) under a linear warmup then
    cosine decay.

    The record mentions a 4,000-step learning-rate schedule without giving its
    form ("Open Flapping Airplanes" record, section "Reproducibility needs inputs
    and an environment record"); the reading here is the common one: for
    step <= warmup the rate rises linearly, lr_max * step / warmup; from there
    to ``total`` it follows half a cosine period from lr_max down to lr_min,
    lr_min + (lr_max - lr_min) (1 + cos(pi (step - warmup) / (total - warmup))) / 2;
    after ``total`` it stays at lr_min.
    """
    if warmup > 0 and step <= warmup:
        return lr_max * step / warmup
    if step >= total:
        return lr_min
    frac = (step - warmup) / (total - warmup)
    return lr_min + 0.5 * (lr_max - lr_min) * (1.0 + math.cos(math.pi * frac))


def next_token_logits(cfg, params, seq, dtype=np.float64) -> np.ndarray:
    """Logits [V] of the token that follows the 1-D id sequence ``seq`` (its last
    position's row of the LM head output), from a full forward pass over ``seq``."""
    tok = np.asarray(seq, dtype=np.int64)[None, :]
    _, cache = forward(cfg, params, tok, np.zeros_like(tok), dtype=dtype)
    return cache["z"][-1]


def greedy_decode(cfg, params, prompt, n_new, dtype=np.float64):
    """Autoregressive greedy generation (serving: "autoregressive text generation
    from the changing model", "Open Flapping Airplanes" record, section "What
    ran", table of SM roles; one generated token releases the next, "How one
    persistent kernel runs three jobs").  Each new token is the argmax of the next
    token's logits (the smallest id among equal maxima) given everything so far,
    recomputed by a full forward pass over the sequence (no cache).  Returns the
    n_new generated ids and the logits each was chosen from ([n_new, V])."""
    seq = [int(t) for t in prompt]
    out, zs = [], []
    for _ in range(n_new):
        z = next_token_logits(cfg, params, seq, dtype=dtype)
        t = int(np.argmax(z))
        out.append(t)
        zs.append(z)
        seq.append(t)
    return np.array(out, dtype=np.int64), np.array(zs)


def train_step(state: OracleState, tokens, targets, lr=None) -> float:
    """Forward, backward and AdamW (at learning rate ``lr``, default the config's);
    returns the pre-update mean loss."""
    loss, cache = forward(state.cfg, state.params, tokens, targets, dtype=state.dtype)
    g = backward(state.cfg, state.params, cache, dtype=state.dtype)
    state.step += 1
    adamw(state.cfg, state.params, g, state.m, state.v, state.step, lr=lr)
    state.last_grad = g
    return loss
