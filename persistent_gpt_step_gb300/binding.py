"""ctypes binding of libgpt.so: the gpt.h calls with the same names, argument
marshalling only.  Every step of the training path runs in the library's CUDA
kernel; there is no Python or CPU fallback — if the library is missing or
cannot be loaded this module raises.
"""

from __future__ import annotations

import ctypes
import os
from ctypes import (POINTER, byref, c_char_p, c_float, c_int, c_int32, c_int64, c_size_t,
                    c_uint32, c_uint64, c_void_p)

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libgpt.so")

GPT_OK = 0
ERRORS = {
    -1: "INVALID_ARG", -2: "CUDA", -3: "OOM", -4: "TIMEOUT", -5: "NONFINITE",
    -6: "BAD_TOKEN", -7: "POISONED", -8: "UNSUPPORTED",
}
DTYPE_FP32, DTYPE_BF16 = 0, 1


class GptError(RuntimeError):
    """A negative status of a gpt_* call; ``code`` is the GPT_ERR_* value."""

    def __init__(self, code: int, msg: str):
        super().__init__(f"GPT_ERR_{ERRORS.get(code, code)}: {msg}")
        self.code = code
        self.name = ERRORS.get(code, str(code))


class gpt_config(ctypes.Structure):
    _fields_ = [
        ("n_layer", c_int32), ("d_model", c_int32), ("n_head", c_int32), ("d_mlp", c_int32),
        ("vocab", c_int32), ("seq_len", c_int32), ("batch", c_int32),
        ("dtype", c_int32),
        ("linear_bias", c_int32), ("ln_bias", c_int32), ("tie_embeddings", c_int32),
        ("gelu_tanh", c_int32),
        ("lr", c_float), ("beta1", c_float), ("beta2", c_float), ("eps", c_float),
        ("weight_decay", c_float), ("ln_eps", c_float),
        ("wd_on_1d", c_int32), ("wait_timeout_ms", c_uint32), ("deterministic", c_int32),
        ("rope", c_int32), ("gated_mlp", c_int32),
    ]


class gpt_lr_schedule(ctypes.Structure):
    _fields_ = [("kind", c_int32), ("warmup_steps", c_int32), ("total_steps", c_int64),
                ("lr_max", c_float), ("lr_min", c_float)]


GPT_LR_CONSTANT, GPT_LR_WARMUP_COSINE = 0, 1


def lr_schedule(warmup_steps: int, total_steps: int, lr_max: float, lr_min: float) -> gpt_lr_schedule:
    """A linear-warmup + cosine-decay schedule for GPT.train_steps."""
    return gpt_lr_schedule(GPT_LR_WARMUP_COSINE, warmup_steps, total_steps, lr_max, lr_min)


class gpt_task_info(ctypes.Structure):
    _fields_ = [("op", c_int32), ("idx", c_int32), ("sig", c_int32), ("sig2", c_int32), ("nwait", c_int32),
                ("wait_first", c_int32 * 3), ("wait_count", c_int32 * 3), ("wait_need", c_int32 * 3)]


_lib = None

# (name, restype, argtypes) of every function gpt.h declares
SIGNATURES = [
    ("gpt_default_config", None, [POINTER(gpt_config)]),
    ("gpt_arena_bytes", c_size_t, [POINTER(gpt_config)]),
    ("gpt_param_count", c_size_t, [POINTER(gpt_config)]),
    ("gpt_create", c_int, [POINTER(gpt_config), c_uint64, c_void_p, c_void_p, c_size_t, POINTER(c_void_p)]),
    ("gpt_train_step", c_int, [c_void_p, c_void_p, c_void_p, POINTER(c_float)]),
    ("gpt_train_step_host", c_int, [c_void_p, c_void_p, c_void_p, POINTER(c_float)]),
    ("gpt_lr_at", c_float, [POINTER(gpt_lr_schedule), c_float, c_int64]),
    ("gpt_train_steps", c_int, [c_void_p, c_void_p, c_void_p, c_int32, POINTER(gpt_lr_schedule), c_void_p]),
    ("gpt_num_params", c_size_t, [c_void_p]),
    ("gpt_num_tensors", c_int, [c_void_p]),
    ("gpt_tensor_info", c_int, [c_void_p, c_int, POINTER(c_char_p), POINTER(c_int64), POINTER(c_size_t)]),
    ("gpt_get_params", c_int, [c_void_p, c_void_p, c_size_t]),
    ("gpt_set_params", c_int, [c_void_p, c_void_p, c_size_t]),
    ("gpt_get_grads", c_int, [c_void_p, c_void_p, c_size_t]),
    ("gpt_get_opt_state", c_int, [c_void_p, c_void_p, c_void_p, POINTER(c_int64)]),
    ("gpt_set_opt_state", c_int, [c_void_p, c_void_p, c_void_p, c_int64]),
    ("gpt_debug_skip_release", c_int, [c_void_p, c_int64]),
    ("gpt_reset", c_int, [c_void_p]),
    ("gpt_run_ops", c_int, [c_void_p, c_int32, c_int32, c_void_p, c_void_p, c_int32, POINTER(c_float)]),
    ("gpt_serve_begin", c_int, [c_void_p, c_void_p, c_int32, c_int32, c_int32, c_int32, c_int64]),
    ("gpt_serve_run", c_int, [c_void_p, c_int32, POINTER(c_float)]),
    ("gpt_serve_tokens", c_int, [c_void_p, c_void_p, c_int32, POINTER(c_int32)]),
    ("gpt_serve_end", c_int, [c_void_p]),
    ("gpt_graph_info", c_int, [c_void_p, POINTER(c_int64), POINTER(c_int32), POINTER(c_int32)]),
    ("gpt_trace_enable", c_int, [c_void_p, c_int32]),
    ("gpt_get_trace", c_int, [c_void_p, c_void_p, c_size_t]),
    ("gpt_last_kernel_ms", c_int, [c_void_p, POINTER(c_float)]),
    ("gpt_last_error", c_char_p, [c_void_p]),
    ("gpt_destroy", None, [c_void_p]),
    ("gpt_task_budget", c_int64, [c_int64, c_int64]),
    ("gpt_init_params_host", c_int, [POINTER(gpt_config), c_uint64, c_void_p, c_size_t]),
    ("gpt_graph_describe", c_int, [POINTER(gpt_config), c_int32, POINTER(c_int64), POINTER(c_int32),
                                   POINTER(gpt_task_info), c_int64, POINTER(c_int32), POINTER(c_int32),
                                   POINTER(c_int32), c_int32]),
    ("gpt_train_step_static", c_int, [POINTER(gpt_config), c_void_p, c_void_p, c_void_p, c_int64,
                                      c_void_p, c_void_p, POINTER(c_float), c_void_p]),
    ("gpt_test_attention", c_int, [c_int32, c_int32, c_int32, c_int32, c_int32, c_void_p, c_void_p,
                                   c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
    ("gpt_test_gemm", c_int, [c_int32, c_int32, c_int32, c_int32, c_void_p, c_int64, c_int32,
                              c_void_p, c_int64, c_int32, c_void_p, c_int64, c_int32, c_void_p,
                              POINTER(c_float)]),
    ("gpt_test_gemm_epilogue", c_int, [c_int32, c_int32, c_int32, c_void_p, c_int64, c_int32,
                                       c_void_p, c_int64, c_int32, c_int32, c_int32, c_void_p, c_int64,
                                       c_void_p, c_int64, c_void_p, c_void_p, c_int64, c_void_p,
                                       POINTER(c_float)]),
]


def load(path: str = LIB_PATH):
    """Loads libgpt.so (built in-tree by build.py); raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with "
                           "`python -m persistent_gpt_step_gb300.build` (no fallback exists)")
    lib = ctypes.CDLL(path)
    for name, res, args in SIGNATURES:
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def make_config(cfg, wait_timeout_ms: int = 2000) -> gpt_config:
    """gpt_config from a workload definition (inputs.GPTConfig or any object
    with the same attribute names)."""
    c = gpt_config()
    load().gpt_default_config(byref(c))
    for f in ("n_layer", "d_model", "n_head", "d_mlp", "vocab", "seq_len", "batch"):
        setattr(c, f, int(getattr(cfg, f)))
    c.dtype = DTYPE_FP32 if getattr(cfg, "dtype", "bf16") == "fp32" else DTYPE_BF16
    c.linear_bias = int(bool(getattr(cfg, "linear_bias", True)))
    c.ln_bias = int(bool(getattr(cfg, "ln_bias", True)))
    c.gelu_tanh = int(bool(getattr(cfg, "gelu_tanh", True)))
    c.tie_embeddings = int(bool(getattr(cfg, "tie_embeddings", False)))
    c.rope = int(bool(getattr(cfg, "rope", False)))
    c.gated_mlp = int(bool(getattr(cfg, "gated_mlp", False)))
    for f in ("lr", "beta1", "beta2", "eps", "weight_decay", "ln_eps"):
        if hasattr(cfg, f):
            setattr(c, f, float(getattr(cfg, f)))
    c.wd_on_1d = int(bool(getattr(cfg, "wd_on_1d", False)))
    c.wait_timeout_ms = int(wait_timeout_ms)
    return c


def _ptr(t) -> int:
    """Address of a torch tensor or numpy array."""
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


class GPT:
    """One handle of the library: a GPT model with its optimizer state on the GPU.

    ``cfg`` is a workload definition (see ``inputs.CONFIGS``).  The device arena
    is a torch allocation (PyTorch supplies device memory and the stream); every
    computation runs in the library's persistent kernel.
    """

    def __init__(self, cfg, seed: int = 1234, stream=None, wait_timeout_ms: int = 2000,
                 torch_arena: bool = True):
        import torch
        lib = load()
        self.cfg = cfg
        self._c = make_config(cfg, wait_timeout_ms)
        self._torch = torch
        self.stream = stream if stream is not None else torch.cuda.current_stream()
        nbytes = lib.gpt_arena_bytes(byref(self._c))
        if nbytes == 0:
            raise GptError(-1, "invalid or unsupported config")
        self.arena_bytes = int(nbytes)
        self._arena = torch.empty(nbytes, dtype=torch.uint8, device="cuda") if torch_arena else None
        h = c_void_p()
        rc = lib.gpt_create(byref(self._c), c_uint64(seed), c_void_p(self.stream.cuda_stream),
                            c_void_p(self._arena.data_ptr() if torch_arena else 0),
                            c_size_t(nbytes if torch_arena else 0), byref(h))
        if rc != GPT_OK:
            raise GptError(rc, lib.gpt_last_error(None).decode())
        self._h = h
        self._lib = lib
        self.n_params = int(lib.gpt_num_params(h))

    # -- helpers ------------------------------------------------------------
    def _check(self, rc):
        if rc != GPT_OK:
            raise GptError(rc, self._lib.gpt_last_error(self._h).decode())

    def close(self):
        if getattr(self, "_h", None):
            self._lib.gpt_destroy(self._h)
            self._h = None
            self._arena = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    # -- the step -------------------------------------------------------------
    def train_step(self, tokens, targets) -> float:
        """One training step; returns the pre-update mean loss.

        tokens, targets: int32 [batch, seq_len]; CUDA tensors are passed as
        device pointers, numpy arrays / CPU tensors go through the host entry
        point (copied to the device by the library on its stream).
        """
        loss = c_float()
        is_dev = hasattr(tokens, "is_cuda") and tokens.is_cuda
        if is_dev:
            assert tokens.dtype == self._torch.int32 and targets.dtype == self._torch.int32
            assert tokens.is_contiguous() and targets.is_contiguous()
            rc = self._lib.gpt_train_step(self._h, c_void_p(tokens.data_ptr()),
                                          c_void_p(targets.data_ptr()), byref(loss))
        else:
            tok = tokens.numpy() if hasattr(tokens, "numpy") else tokens
            tgt = targets.numpy() if hasattr(targets, "numpy") else targets
            tok = np.ascontiguousarray(tok, dtype=np.int32)
            tgt = np.ascontiguousarray(tgt, dtype=np.int32)
            rc = self._lib.gpt_train_step_host(self._h, c_void_p(tok.ctypes.data),
                                               c_void_p(tgt.ctypes.data), byref(loss))
        self._check(rc)
        return float(loss.value)

    def train_steps(self, tokens, targets, schedule: gpt_lr_schedule | None = None) -> np.ndarray:
        """k training steps in one call (no host synchronisation between them).

        tokens, targets: CUDA int32 tensors [k, batch, seq_len]; schedule: a
        gpt_lr_schedule (None: the config's constant rate).  Returns the k
        pre-update losses; raises GptError as train_step does (the error names
        the first failing step; the steps before it are applied)."""
        assert tokens.is_cuda and targets.is_cuda
        assert tokens.dtype == self._torch.int32 and targets.dtype == self._torch.int32
        assert tokens.is_contiguous() and targets.is_contiguous() and tokens.shape == targets.shape
        k = int(tokens.shape[0])
        out = np.zeros(k, np.float32)
        rc = self._lib.gpt_train_steps(self._h, c_void_p(tokens.data_ptr()), c_void_p(targets.data_ptr()), k,
                                       byref(schedule) if schedule is not None else None,
                                       c_void_p(out.ctypes.data))
        self.last_losses = out
        self._check(rc)
        return out

    # -- state ----------------------------------------------------------------
    def params(self) -> np.ndarray:
        out = np.empty(self.n_params, np.float32)
        self._check(self._lib.gpt_get_params(self._h, c_void_p(out.ctypes.data), self.n_params))
        return out

    def set_params(self, p: np.ndarray):
        p = np.ascontiguousarray(p, dtype=np.float32)
        assert p.size == self.n_params
        self._check(self._lib.gpt_set_params(self._h, c_void_p(p.ctypes.data), self.n_params))

    def grads(self) -> np.ndarray:
        out = np.empty(self.n_params, np.float32)
        self._check(self._lib.gpt_get_grads(self._h, c_void_p(out.ctypes.data), self.n_params))
        return out

    def opt_state(self):
        m = np.empty(self.n_params, np.float32)
        v = np.empty(self.n_params, np.float32)
        step = c_int64()
        self._check(self._lib.gpt_get_opt_state(self._h, c_void_p(m.ctypes.data),
                                                c_void_p(v.ctypes.data), byref(step)))
        return m, v, int(step.value)

    def set_opt_state(self, m, v, step: int):
        m = np.ascontiguousarray(m, dtype=np.float32)
        v = np.ascontiguousarray(v, dtype=np.float32)
        self._check(self._lib.gpt_set_opt_state(self._h, c_void_p(m.ctypes.data),
                                                c_void_p(v.ctypes.data), c_int64(step)))

    def tensor_table(self):
        """[(name, shape, offset)] in canonical order."""
        out = []
        name = c_char_p()
        shape = (c_int64 * 2)()
        off = c_size_t()
        for i in range(self._lib.gpt_num_tensors(self._h)):
            self._check(self._lib.gpt_tensor_info(self._h, i, byref(name), shape, byref(off)))
            shp = (int(shape[0]),) if int(shape[1]) == 1 and not self._is_matrix(name.value) \
                else (int(shape[0]), int(shape[1]))
            out.append((name.value.decode(), shp, int(off.value)))
        return out

    @staticmethod
    def _is_matrix(name: bytes) -> bool:
        n = name.decode()
        return n in ("wte", "wpe", "w_lm") or n.split(".")[-1].startswith("w_")

    def graph_info(self):
        n = c_int64()
        g = c_int32()
        b = c_int32()
        self._check(self._lib.gpt_graph_info(self._h, byref(n), byref(g), byref(b)))
        return int(n.value), int(g.value), int(b.value)

    def trace_enable(self, on: bool = True):
        self._check(self._lib.gpt_trace_enable(self._h, int(on)))

    def trace(self) -> np.ndarray:
        """uint64 [n_tasks, 4]: claim, start, end (ns), SM id of the last step."""
        n = self.graph_info()[0]
        out = np.empty((n, 4), np.uint64)
        self._check(self._lib.gpt_get_trace(self._h, c_void_p(out.ctypes.data), out.size))
        return out

    def role_states(self) -> np.ndarray:
        """uint64 [grid, 8]: the last wait each GEMM role entered in the last step."""
        n, grid, _ = self.graph_info()
        out = np.empty(4 * n + 8 * grid, np.uint64)
        self._check(self._lib.gpt_get_trace(self._h, c_void_p(out.ctypes.data), out.size))
        return out[4 * n:].reshape(grid, 8)

    def last_kernel_ms(self) -> float:
        ms = c_float()
        self._check(self._lib.gpt_last_kernel_ms(self._h, byref(ms)))
        return float(ms.value)

    def debug_skip_release(self, task_index: int):
        self._check(self._lib.gpt_debug_skip_release(self._h, c_int64(task_index)))

    def reset(self):
        self._check(self._lib.gpt_reset(self._h))

    # -- serving partition ----------------------------------------------------
    def serve_begin(self, prompt, max_new: int, blocks: int = 16, tokens_per_step: int = 0,
                    first_step: int = 0):
        """gpt_serve_begin: greedy generation from the live weights on `blocks`
        reserved blocks (prompt: host int ids)."""
        p = np.ascontiguousarray(prompt, dtype=np.int32)
        self._check(self._lib.gpt_serve_begin(self._h, c_void_p(p.ctypes.data), int(p.size), int(max_new),
                                              int(blocks), int(tokens_per_step), c_int64(first_step)))

    def serve_run(self, max_steps: int) -> float:
        """gpt_serve_run: a serving-only launch of up to max_steps decode steps;
        returns its device milliseconds."""
        ms = c_float()
        self._check(self._lib.gpt_serve_run(self._h, int(max_steps), byref(ms)))
        return float(ms.value)

    def serve_tokens(self) -> np.ndarray:
        """The tokens generated so far."""
        n = c_int32()
        self._check(self._lib.gpt_serve_tokens(self._h, None, 0, byref(n)))
        out = np.zeros(max(int(n.value), 1), np.int32)
        self._check(self._lib.gpt_serve_tokens(self._h, c_void_p(out.ctypes.data), out.size, byref(n)))
        return out[:int(n.value)]

    def serve_end(self):
        self._check(self._lib.gpt_serve_end(self._h))

    def run_ops(self, op_first: int, op_count: int, tokens, targets, reps: int = 1) -> float:
        """gpt_run_ops: operations [op_first, op_first + op_count) of the step graph
        as their own launch, ``reps`` times; returns the mean milliseconds per launch.
        tokens, targets: CUDA int32 tensors [batch, seq_len]."""
        assert tokens.is_cuda and targets.is_cuda
        assert tokens.dtype == self._torch.int32 and targets.dtype == self._torch.int32
        ms = c_float()
        self._check(self._lib.gpt_run_ops(self._h, op_first, op_count, c_void_p(tokens.data_ptr()),
                                          c_void_p(targets.data_ptr()), reps, byref(ms)))
        return float(ms.value)


def task_budget(iterations: int, tasks_per_iteration: int) -> int:
    return int(load().gpt_task_budget(c_int64(iterations), c_int64(tasks_per_iteration)))


def test_gemm(A, B, a_mn: bool, b_mn: bool, M: int, N: int, K: int, ksplit: int = 1, stream=None,
              timing: bool = False):
    """Runs gpt_test_gemm on torch CUDA tensors; returns C (fp32 [ksplit, M, N]),
    and with timing=True (C, kernel milliseconds)."""
    import torch
    lib = load()
    dtype = DTYPE_BF16 if A.dtype == torch.bfloat16 else DTYPE_FP32
    C = torch.full((ksplit, M, N), float("nan"), dtype=torch.float32, device=A.device)
    s = stream if stream is not None else torch.cuda.current_stream()
    ms = c_float()
    rc = lib.gpt_test_gemm(dtype, M, N, K, c_void_p(A.data_ptr()), A.stride(0), int(a_mn),
                           c_void_p(B.data_ptr()), B.stride(0), int(b_mn), c_void_p(C.data_ptr()), N,
                           ksplit, c_void_p(s.cuda_stream), byref(ms))
    if rc != GPT_OK:
        raise GptError(rc, lib.gpt_last_error(None).decode())
    return (C, float(ms.value)) if timing else C


EPI_STORE, EPI_RESID, EPI_GELU, EPI_GELU_BWD = 0, 1, 2, 4


def test_gemm_epilogue(A, B, a_mn: bool, b_mn: bool, M: int, N: int, K: int, epi: int, bias=None, src=None,
                       gelu_tanh: bool = True, stream=None, timing: bool = False):
    """Runs gpt_test_gemm_epilogue on bf16 torch CUDA tensors A, B.  Returns
    out (bf16, or fp32 for the residual epilogue; GELU' for the GELU
    epilogue), plus out2 (GELU) for the GELU epilogue, plus kernel
    milliseconds with timing=True."""
    import torch
    lib = load()
    dev = A.device
    out = torch.full((M, N), float("nan"), dtype=torch.float32 if epi == EPI_RESID else torch.bfloat16, device=dev)
    out2 = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=dev) if epi == EPI_GELU else None
    s = stream if stream is not None else torch.cuda.current_stream()
    ms = c_float()
    rc = lib.gpt_test_gemm_epilogue(M, N, K, c_void_p(A.data_ptr()), A.stride(0), int(a_mn),
                                    c_void_p(B.data_ptr()), B.stride(0), int(b_mn), epi, int(gelu_tanh),
                                    c_void_p(out.data_ptr()), N,
                                    c_void_p(out2.data_ptr() if out2 is not None else None), N,
                                    c_void_p(bias.data_ptr() if bias is not None else None),
                                    c_void_p(src.data_ptr() if src is not None else None),
                                    src.stride(0) if src is not None else 0, c_void_p(s.cuda_stream), byref(ms))
    if rc != GPT_OK:
        raise GptError(rc, lib.gpt_last_error(None).decode())
    res = (out, out2) if epi == EPI_GELU else (out,)
    return (*res, float(ms.value)) if timing else (res if len(res) > 1 else res[0])


def init_params_host(cfg, seed: int, n: int) -> np.ndarray:
    """The library's own (C++) seeded initial weights; no GPU needed."""
    lib = load()
    out = np.empty(n, np.float32)
    c = make_config(cfg)
    rc = lib.gpt_init_params_host(byref(c), c_uint64(seed), c_void_p(out.ctypes.data), n)
    if rc != GPT_OK:
        raise GptError(rc, lib.gpt_last_error(None).decode())
    return out


def describe_graph(cfg, num_sms: int = 152, dims: bool = False):
    """The step's task graph, built on the host.

    Returns (tasks, op_types, op_tasks[, op_dims]): tasks in ticket order as
    (op, idx, sig, [(first_counter, n_counters, need), ...], sig2); op_dims per op:
    (M, N, K, tile width) for GEMMs (zeros otherwise), first counter, counters."""
    lib = load()
    c = make_config(cfg)
    nt, no = c_int64(), c_int32()
    rc = lib.gpt_graph_describe(byref(c), num_sms, byref(nt), byref(no), None, 0, None, None, None, 0)
    if rc != GPT_OK:
        raise GptError(rc, lib.gpt_last_error(None).decode())
    tasks = (gpt_task_info * nt.value)()
    types = (c_int32 * no.value)()
    ntk = (c_int32 * no.value)()
    odims = (c_int32 * (6 * no.value))()
    rc = lib.gpt_graph_describe(byref(c), num_sms, byref(nt), byref(no), tasks, nt.value, types, ntk,
                                odims, no.value)
    if rc != GPT_OK:
        raise GptError(rc, lib.gpt_last_error(None).decode())
    out = [(t.op, t.idx, t.sig, [(t.wait_first[w], t.wait_count[w], t.wait_need[w]) for w in range(t.nwait)],
            t.sig2) for t in tasks]
    if dims:
        return out, list(types), list(ntk), [tuple(odims[6 * i:6 * i + 6]) for i in range(no.value)]
    return out, list(types), list(ntk)


def param_count(cfg) -> int:
    """Number of parameters of a model with this workload definition (host only)."""
    n = int(load().gpt_param_count(byref(make_config(cfg))))
    if n == 0:
        raise GptError(-1, "invalid config")
    return n


def _check_device_tensor(name, t, dtype, numel=None, shape=None):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise GptError(-1, f"{name} must be a CUDA tensor")
    if t.device.index != torch.cuda.current_device():
        raise GptError(-1, f"{name} is on cuda:{t.device.index}, not the current device")
    if t.dtype != dtype:
        raise GptError(-1, f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise GptError(-1, f"{name} must be contiguous")
    if numel is not None and t.numel() != numel:
        raise GptError(-1, f"{name} has {t.numel()} elements, the model needs {numel}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise GptError(-1, f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def train_step_static(cfg, params, m, v, step: int, tokens, targets, stream=None,
                      wait_timeout_ms: int = 2000) -> float:
    """gpt_train_step_static on CUDA tensors (fp32 params/m/v updated in place).

    The C call cannot check buffer lengths, so every tensor's device, dtype,
    contiguity and size is checked here before any launch; a mismatch raises
    GptError(INVALID_ARG).  Invalid configs and bf16 (which the call rejects by
    itself, before touching any buffer) reach the library unchanged."""
    import torch
    lib = load()
    c = make_config(cfg, wait_timeout_ms)
    n = int(lib.gpt_param_count(byref(c)))
    if n > 0 and c.dtype == DTYPE_FP32:
        for name, t in (("params", params), ("m", m), ("v", v)):
            _check_device_tensor(name, t, torch.float32, numel=n)
        for name, t in (("tokens", tokens), ("targets", targets)):
            _check_device_tensor(name, t, torch.int32, shape=(c.batch, c.seq_len))
    s = stream if stream is not None else torch.cuda.current_stream()
    loss = c_float()
    rc = lib.gpt_train_step_static(byref(c), c_void_p(params.data_ptr()), c_void_p(m.data_ptr()),
                                   c_void_p(v.data_ptr()), c_int64(step), c_void_p(tokens.data_ptr()),
                                   c_void_p(targets.data_ptr()), byref(loss), c_void_p(s.cuda_stream))
    if rc != GPT_OK:
        raise GptError(rc, lib.gpt_last_error(None).decode())
    return float(loss.value)


def test_attention(qkv, dout, B: int, T: int, H: int, d: int, stream=None):
    """Runs gpt_test_attention on CUDA tensors; returns (o, lse, dqkv)."""
    import torch
    lib = load()
    dtype = DTYPE_BF16 if qkv.dtype == torch.bfloat16 else DTYPE_FP32
    C = H * d
    o = torch.full((B * T, C), float("nan"), dtype=qkv.dtype, device=qkv.device)
    dqkv = torch.full((B * T, 3 * C), float("nan"), dtype=qkv.dtype, device=qkv.device)
    lse = torch.full((B, H, T), float("nan"), dtype=torch.float32, device=qkv.device)
    scratch = torch.empty(B * H * 2 * T * d, dtype=torch.float32, device=qkv.device)
    s = stream if stream is not None else torch.cuda.current_stream()
    rc = lib.gpt_test_attention(dtype, B, T, H, d, c_void_p(qkv.data_ptr()), c_void_p(o.data_ptr()),
                                c_void_p(lse.data_ptr()), c_void_p(dout.data_ptr()), c_void_p(dqkv.data_ptr()),
                                c_void_p(scratch.data_ptr()), c_void_p(s.cuda_stream))
    if rc != GPT_OK:
        raise GptError(rc, lib.gpt_last_error(None).decode())
    return o, lse, dqkv
