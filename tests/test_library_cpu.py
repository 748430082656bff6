"""Host-side tests of libgpt.so and the input generators (no GPU needed)."""

import ctypes
import os
import random
import re
import threading
import time

import numpy as np
import pytest

from oracle import gpt_oracle as O
from persistent_gpt_step_gb300 import binding as B
from persistent_gpt_step_gb300 import build as build_mod
from persistent_gpt_step_gb300 import inputs as I

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gpt.h")
GOLD = os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return B.load()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(gpt_[a-z_0-9]+)\s*\(", text)
    return sorted(set(names))


def test_every_declared_function_is_exported(lib):
    names = _declared_functions()
    assert len(names) >= 20
    for n in names:
        assert hasattr(lib, n), n
    bound = {s[0] for s in B.SIGNATURES}
    assert set(names) == bound, set(names) ^ bound


def test_config_struct_matches_header(lib):
    text = open(HEADER).read()
    body = re.search(r"typedef struct gpt_config \{(.*?)\} gpt_config;", text, re.S).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    fields = []
    for decl in body.split(";"):
        decl = decl.strip()
        if not decl:
            continue
        typ, names = decl.split(None, 1)
        fields += [(typ, n.strip()) for n in names.split(",")]
    assert [n for _, n in fields] == [f[0] for f in B.gpt_config._fields_]
    assert ctypes.sizeof(B.gpt_config) == 4 * len(fields)


def test_default_config_is_main_workload(lib):
    c = B.gpt_config()
    lib.gpt_default_config(ctypes.byref(c))
    main = I.CONFIGS["main"]
    for f in ("n_layer", "d_model", "n_head", "d_mlp", "vocab", "seq_len", "batch"):
        assert getattr(c, f) == getattr(main, f)
    assert c.dtype == B.DTYPE_BF16 and c.tie_embeddings == 0 and c.gelu_tanh == 1
    assert abs(c.lr - 6e-4) < 1e-9 and abs(c.beta2 - 0.95) < 1e-7 and abs(c.weight_decay - 0.1) < 1e-7


def test_task_budget_overflow_golden(lib):
    g = {}
    for line in open(os.path.join(GOLD, "scheduler_overflow.txt")):
        if line.strip() and not line.startswith("#"):
            k, v = line.split()
            g[k] = int(v)
    prod = B.task_budget(g["iterations"], g["tasks_per_iteration"])
    assert prod == g["product"]
    # the page's 32-bit arithmetic, reproduced: this is the failure the 64-bit budget avoids
    assert prod % (1 << 32) == g["wrapped"]
    assert (prod % (1 << 32)) // g["tasks_per_iteration"] == g["tokens_before_stop"]
    assert B.task_budget(1 << 62, 4) == -1
    assert B.task_budget(-1, 3) == -1


def test_arena_bytes_and_invalid_configs(lib):
    for name in ("tiny", "small", "main"):
        c = B.make_config(I.CONFIGS[name])
        assert lib.gpt_arena_bytes(ctypes.byref(c)) > 0
    bad = B.make_config(I.CONFIGS["tiny"].replace(d_model=63))
    assert lib.gpt_arena_bytes(ctypes.byref(bad)) == 0
    bad = B.make_config(I.CONFIGS["small"].replace(seq_len=100))  # bf16: B*T % 128
    assert lib.gpt_arena_bytes(ctypes.byref(bad)) == 0


@pytest.mark.parametrize("name", ["tiny", "small", "main", "350m", "57m", "small_gated"])
def test_param_count_matches_oracle_table(lib, name):
    cfg = I.CONFIGS[name]
    assert B.param_count(cfg) == O.num_params(cfg)


def test_param_count_rejects_invalid_config(lib):
    with pytest.raises(B.GptError):
        B.param_count(I.CONFIGS["tiny"].replace(d_model=65))


def test_create_without_gpu_fails_cleanly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    c = B.make_config(I.CONFIGS["tiny"])
    h = ctypes.c_void_p()
    rc = lib.gpt_create(ctypes.byref(c), 1, None, None, 0, ctypes.byref(h))
    assert rc in (-2, -8)
    assert h.value is None
    assert lib.gpt_last_error(None)


@pytest.mark.parametrize("name", ["tiny", "small", "small_gated", "57m"])
def test_library_tensor_table_and_host_init_match_spec(lib, name):
    """The C++ implementation of the init spec equals the test-side one."""
    cfg = I.CONFIGS[name]
    n = O.num_params(cfg)
    got = B.init_params_host(cfg, 1234, n)
    ref = I.init_params(O.param_table(cfg), 1234)
    diff = got != ref
    # double-precision log/cos may differ in the last ulp between libm builds;
    # that moves an fp32 weight by one ulp at most, and almost never
    assert diff.sum() <= 2
    if diff.any():
        ulp = np.abs(got.view(np.int32)[diff].astype(np.int64) - ref.view(np.int32)[diff].astype(np.int64))
        assert ulp.max() <= 1


def test_library_lr_schedule_matches_oracle(lib):
    """The host-side schedule the multi-step call uses against the oracle's
    (independently written) warmup + cosine schedule, and invalid schedules."""
    from ctypes import byref
    from oracle import gpt_oracle as O
    hi, lo, w, tot = 6e-4, 6e-5, 100, 4000
    s = B.lr_schedule(w, tot, hi, lo)
    hi32, lo32 = float(np.float32(hi)), float(np.float32(lo))
    for t in list(range(1, 130)) + [1000, 2050, 3998, 3999, 4000, 4001, 10 ** 6]:
        want = O.lr_at(t, hi32, lo32, w, tot)
        assert lib.gpt_lr_at(byref(s), 1.0, t) == pytest.approx(want, rel=2e-7, abs=1e-12), t
    assert lib.gpt_lr_at(None, 2.5e-4, 7) == pytest.approx(2.5e-4, rel=1e-7)
    assert lib.gpt_lr_at(byref(B.gpt_lr_schedule(B.GPT_LR_CONSTANT, 0, 1, 0.0, 0.0)), 1e-3, 3) == \
        pytest.approx(1e-3, rel=1e-7)
    for bad in (B.gpt_lr_schedule(7, 0, 10, 1e-3, 0.0), B.gpt_lr_schedule(1, 10, 10, 1e-3, 0.0),
                B.gpt_lr_schedule(1, 1, 10, 1e-4, 1e-3), B.gpt_lr_schedule(1, -1, 10, 1e-3, 0.0)):
        assert lib.gpt_lr_at(byref(bad), 1e-3, 1) < 0
    assert lib.gpt_lr_at(byref(s), 1e-3, 0) < 0


def test_init_statistics():
    w = I.normal_fp32(42, 3, 200000)
    assert abs(w.mean()) < 0.02 * 0.02
    assert abs(w.std() - 0.02) < 0.02 * 0.01


def test_splitmix64_published_vector():
    lines = [l.strip() for l in open(os.path.join(GOLD, "splitmix64.txt"))
             if l.strip() and not l.startswith("#")]
    seed = int(lines[0].split()[1])
    want = [int(x, 16) for x in lines[1:]]
    got = [int(v) for v in I.splitmix64(seed, np.arange(len(want)))]
    assert got == want


def test_token_batches():
    cfg = I.CONFIGS["small"]
    tok, tgt = I.batch(cfg, 5, 3)
    assert tok.shape == (cfg.batch, cfg.seq_len) and tok.dtype == np.int32
    assert np.array_equal(tok[:, 1:], tgt[:, :-1])       # targets = inputs shifted by one
    assert tok.min() >= 0 and tok.max() < cfg.vocab
    t2, _ = I.batch(cfg, 5, 3)
    assert np.array_equal(tok, t2)
    t3, _ = I.batch(cfg, 5, 4)
    assert not np.array_equal(tok, t3)


def test_zipf_frequencies():
    V, s = 1000, 1.1
    blk = I.token_block(9, 0, 64, 4096, V, "zipf", s)
    counts = np.bincount(blk.ravel(), minlength=V)[:10].astype(float)
    w = np.arange(1, V + 1, dtype=float) ** -s
    pmf = w / w.sum()
    n = blk.size
    assert np.all(np.abs(counts - n * pmf[:10]) < 5 * np.sqrt(n * pmf[:10]))
    uni = I.token_block(9, 0, 64, 4096, V, "uniform")
    assert abs(np.bincount(uni.ravel(), minlength=V).std() / (uni.size / V) - 1 / np.sqrt(uni.size / V)) < 0.05


# ----------------------------------------------------------------- task graph

@pytest.mark.parametrize("name", ["tiny", "small", "main", "350m", "small_gated", "57m"])
def test_task_graph_is_topological(lib, name):
    """Every counter a task waits on is signalled only by earlier tickets, as
    many times as the wait needs (the no-deadlock condition of the ticket loop)."""
    from collections import Counter
    tasks, types, ntk, dims = B.describe_graph(I.CONFIGS[name], dims=True)
    sig_count = Counter(t[2] for t in tasks) + Counter(t[4] for t in tasks if t[4] >= 0)
    seen = Counter()
    for op, idx, sig, waits, sig2 in tasks:
        ctr0, nblk = dims[op][4], dims[op][5]
        assert ctr0 <= sig < ctr0 + nblk
        assert sig2 == (ctr0 + nblk - 1 if nblk > 1 else -1)
        for first, count, need in waits:
            for c in range(first, first + count):
                assert sig_count[c] == need
                assert seen[c] == sig_count[c]       # all signallers are earlier tickets
        seen[sig] += 1
        if sig2 >= 0:
            seen[sig2] += 1
    assert sorted(Counter(t[0] for t in tasks).items()) == list(enumerate(ntk))
    # every parameter tensor gets exactly one AdamW op
    assert sum(1 for t in types if t == 11) == len(O.param_table(I.CONFIGS[name]))


@pytest.mark.parametrize("name", ["small_gated", "57m"])
def test_variant_graph_structure(lib, name):
    """The rotary / gated / tied variant: no position-table gradient op, the gated MLP's
    GEMMs are 2F wide, and (tied embedding) the token-embedding gradient op waits for
    the LM head's weight-gradient GEMM, whose result it adds to."""
    cfg = I.CONFIGS[name]
    tasks, types, ntk, dims = B.describe_graph(cfg, dims=True)
    N, C, F, V = cfg.batch * cfg.seq_len, cfg.d_model, cfg.d_mlp, cfg.vocab
    assert 10 not in types                                   # no position-embedding backward
    gemm = [(o, d) for o, (t, d) in enumerate(zip(types, dims)) if t == 2]
    shapes = {(d[0], d[1], d[2]) for _, d in gemm}
    assert (N, 2 * F, C) in shapes                           # up projection, gate and up interleaved
    assert (2 * F, C, N) in shapes and (N, C, 2 * F) in shapes  # its weight and input gradients
    lm_dw = [o for o, d in gemm if (d[0], d[1], d[2]) == (V, C, N)]
    assert len(lm_dw) == 1
    ctr0, nctr = dims[lm_dw[0]][4], dims[lm_dw[0]][5]
    wte_op = types.index(9)
    waited = {c for (op, _, _, waits, _) in tasks if op == wte_op for (f, n, _) in waits for c in range(f, f + n)}
    assert waited & set(range(ctr0, ctr0 + nctr))


def test_row_blocks_make_the_forward_a_wavefront(lib):
    """On the bf16 path a QKV tile waits only for its own 128-row block of LN1."""
    tasks, types, ntk, dims = B.describe_graph(I.CONFIGS["main"], dims=True)
    gemm_row_ops = [o for o, t in enumerate(types) if t == 2 and dims[o][5] > 1]
    assert gemm_row_ops
    o = gemm_row_ops[0]
    waits = [w for (op, _, _, ws, _) in tasks if op == o for w in ws]
    assert all(count == 1 for _, count, _ in waits)


def _simulate(tasks, n_counters, n_blocks, skip=None, timeout=5.0, seed=0):
    """Blocks as threads running the ticket loop with random delays."""
    counters = [0] * n_counters
    ticket = [0]
    lock = threading.Lock()
    done = []
    failed = []
    rng = random.Random(seed)

    def block():
        while True:
            with lock:
                t = ticket[0]
                ticket[0] += 1
            if t >= len(tasks) or failed:
                return
            op, idx, sig, waits, sig2 = tasks[t]
            t0 = time.time()
            for first, count, need in waits:
                for c in range(first, first + count):
                    while counters[c] < need:
                        if time.time() - t0 > timeout:
                            failed.append(t)
                            return
                        time.sleep(0)
            if rng.random() < 0.01:
                time.sleep(0.001)
            with lock:
                done.append(t)
                if t != skip:
                    counters[sig] += 1
                    if sig2 >= 0:
                        counters[sig2] += 1

    th = [threading.Thread(target=block) for _ in range(n_blocks)]
    for x in th:
        x.start()
    for x in th:
        x.join()
    return counters, done, failed


def _n_counters(dims):
    return max(d[4] + d[5] for d in dims)


@pytest.mark.parametrize("name", ["tiny", "small"])
def test_scheduler_simulation_completes(lib, name):
    tasks, types, ntk, dims = B.describe_graph(I.CONFIGS[name], dims=True)
    counters, done, failed = _simulate(tasks, _n_counters(dims), 16)
    assert not failed
    assert sorted(done) == list(range(len(tasks)))
    from collections import Counter
    want = Counter(t[2] for t in tasks) + Counter(t[4] for t in tasks if t[4] >= 0)
    assert counters == [want[c] for c in range(_n_counters(dims))]


def test_scheduler_simulation_skipped_release_times_out(lib):
    tasks, types, ntk, dims = B.describe_graph(I.CONFIGS["tiny"], dims=True)
    counters, done, failed = _simulate(tasks, _n_counters(dims), 8, skip=0, timeout=0.5)
    assert failed


def test_trace_window_shares_synthetic():
    """The trace tool's window table on a hand-made trace: grid 2, one GEMM task
    (claim 0, start 1 ms, end 3 ms) and one AdamW task (claim 2, start 2.5, end 4)."""
    from persistent_gpt_step_gb300 import trace as T
    ms = 1_000_000
    tr = np.array([[0, 1 * ms, 3 * ms, 0], [2 * ms, int(2.5 * ms), 4 * ms, 1]], dtype=np.uint64)
    ops = np.array([0, 1])
    types = [2, 11]  # gemm, adamw
    w = T.window_shares(tr, ops, types, 2, [0.0, 2.0, 4.0])
    (lo0, hi0, s0), (lo1, hi1, s1) = w
    assert s0["gemm"] == pytest.approx((1.0 / 4.0, 1.0 / 4.0))   # exec 1-2, wait 0-1 of 2 x 2 ms
    assert "adamw" not in s0
    assert s1["gemm"] == pytest.approx((1.0 / 4.0, 0.0))
    assert s1["adamw"] == pytest.approx((1.5 / 4.0, 0.5 / 4.0))

