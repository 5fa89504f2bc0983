"""Python binding of libgpt2b300.so -- one GPT-2 training step on a B300.

Argument marshalling only: every step of the training path runs in the
library's CUDA kernels.  PyTorch supplies device memory (the arena) and the
CUDA stream.  The module-level functions carry the C ABI's names
(``gpt2_build``, ``gpt2_forward``, ``gpt2_zero_grad``, ``gpt2_backward``,
``gpt2_update`` ...); ``GPT2`` wraps a handle.

The calls follow the decomposition of llm.c's train_gpt2.c described on the
page «llm.c：Andrej Karpathy带你从零复现LLM», section
«核心代码解读：train_gpt2.c», items 2-3.  If the compiled library is missing,
every call raises: there is no fallback path.
"""
from __future__ import annotations

import ctypes as ct
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgpt2b300.so")

GPT2_OK = 0
GPT2_ERR_ARG = -1
GPT2_ERR_SHAPE = -2
GPT2_ERR_TOKEN_RANGE = -3
GPT2_ERR_STATE = -4
GPT2_ERR_ARENA = -5
GPT2_ERR_CUDA = -6
GPT2_ERR_DEVICE_TIMEOUT = -7
GPT2_WARN_NONFINITE = 1
GPT2_PREC_FP32 = 0
GPT2_PREC_BF16 = 1

# every symbol the header declares
EXPORTS = [
    "gpt2_arena_bytes", "gpt2_build", "gpt2_forward", "gpt2_forward_device", "gpt2_sample", "gpt2_sync",
    "gpt2_zero_grad",
    "gpt2_backward", "gpt2_update", "gpt2_train_step_device", "gpt2_free", "gpt2_num_parameters",
    "gpt2_get_params", "gpt2_set_params", "gpt2_get_grads", "gpt2_get_opt_state", "gpt2_set_opt_state",
    "gpt2_get_logits", "gpt2_last_launch_count", "gpt2_status_string", "gpt2_train_step", "gpt2_kernel_timer",
    "gpt2_kernel_timer_read", "gpt2op_matmul_workspace_bytes", "gpt2op_matmul_forward", "gpt2op_matmul_backward",
    "gpt2op_matmul_backward_noalloc", "gpt2op_attention_workspace_bytes", "gpt2op_attention_forward",
    "gpt2op_attention_backward_workspace_bytes", "gpt2op_attention_backward", "gpt2_set_wait_limit_ns",
    "gpt2_plan_bf16_matmul",
]


class gpt2_config(ct.Structure):
    _fields_ = [(n, ct.c_int) for n in ("max_seq_len", "vocab_size", "padded_vocab_size", "num_layers",
                                        "num_heads", "channels", "gemm_precision", "llama")]


class GPT2Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


_LIB = None


def lib() -> ct.CDLL:
    """Load libgpt2b300.so (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m gpt_train_step_02_b300.build`")
        L = ct.CDLL(LIB_PATH)
        P, I, F, LL, SZ = ct.c_void_p, ct.c_int, ct.c_float, ct.c_longlong, ct.c_size_t
        CFG = ct.POINTER(gpt2_config)
        sig = {
            "gpt2_arena_bytes": (SZ, [CFG, I, I]),
            "gpt2_build": (I, [ct.POINTER(P), CFG, ct.c_uint64, I, I, P, SZ, P]),
            "gpt2_forward": (I, [P, P, P, I, I, P]),
            "gpt2_forward_device": (I, [P, P, P, I, I]),
            "gpt2_sample": (I, [P, P, I, I, P]),
            "gpt2_sync": (I, [P, P]),
            "gpt2_zero_grad": (I, [P]),
            "gpt2_backward": (I, [P]),
            "gpt2_update": (I, [P, F, F, F, F, F, I]),
            "gpt2_train_step_device": (I, [P, P, P, I, I, F, F, F, F, F, I, I]),
            "gpt2_free": (I, [P]),
            "gpt2_num_parameters": (LL, [P]),
            "gpt2_get_params": (I, [P, P, LL]),
            "gpt2_set_params": (I, [P, P, LL]),
            "gpt2_get_grads": (I, [P, P, LL]),
            "gpt2_get_opt_state": (I, [P, P, P, LL]),
            "gpt2_set_opt_state": (I, [P, P, P, LL]),
            "gpt2_get_logits": (I, [P, P, LL]),
            "gpt2_last_launch_count": (LL, [P]),
            "gpt2_status_string": (ct.c_char_p, [I]),
            "gpt2_train_step": (I, [P, P, P, I, I, F, F, F, F, F, I, P]),
            "gpt2_kernel_timer": (I, [P, I]),
            "gpt2_set_wait_limit_ns": (I, [ct.c_ulonglong]),
            "gpt2_plan_bf16_matmul": (I, [I, I, I, I, I, I, P, P]),
            "gpt2op_matmul_workspace_bytes": (SZ, [I, I, I]),
            "gpt2op_matmul_forward": (I, [P, P, P, P, I, I, I, I, P, P]),
            "gpt2op_matmul_backward": (I, [P, P, P, P, P, P, I, I, I, I, P, P]),
            "gpt2op_matmul_backward_noalloc": (I, [P, P, P, P, P, P, I, I, I, I, P]),
            "gpt2op_attention_workspace_bytes": (SZ, [I, I, I]),
            "gpt2op_attention_forward": (I, [P, P, P, I, I, I, I, I, P, P]),
            "gpt2op_attention_backward_workspace_bytes": (SZ, [I, I, I, I]),
            "gpt2op_attention_backward": (I, [P, P, P, I, I, I, I, I, P, P]),
            "gpt2_kernel_timer_read": (I, [P, ct.POINTER(ct.c_double), ct.POINTER(LL), ct.POINTER(ct.c_double)]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = L
    return _LIB


def status_string(status: int) -> str:
    return lib().gpt2_status_string(int(status)).decode()


def _check(rc: int, where: str, allow=(GPT2_OK,)) -> int:
    if rc not in allow:
        raise GPT2Error(rc, where)
    return rc


def make_config(w) -> gpt2_config:
    """gpt2_config from any object with the GPT-2 shape fields."""
    prec = getattr(w, "gemm_precision", GPT2_PREC_FP32)
    return gpt2_config(w.max_seq_len, w.vocab_size, w.padded_vocab_size, w.num_layers, w.num_heads, w.channels,
                       prec, int(getattr(w, "llama", 0)))


def _hptr(a: np.ndarray) -> ct.c_void_p:
    return ct.c_void_p(a.ctypes.data)


# --- the C ABI under its own names ------------------------------------------
def gpt2_arena_bytes(cfg: gpt2_config, maxB: int, maxT: int) -> int:
    return int(lib().gpt2_arena_bytes(ct.byref(cfg), maxB, maxT))


def gpt2_build(cfg: gpt2_config, seed: int, maxB: int, maxT: int, arena_ptr: int | None, arena_bytes: int,
               stream_ptr: int | None) -> ct.c_void_p:
    h = ct.c_void_p()
    _check(lib().gpt2_build(ct.byref(h), ct.byref(cfg), seed, maxB, maxT, arena_ptr, arena_bytes, stream_ptr),
           "gpt2_build")
    return h


def gpt2_forward(h, inputs: np.ndarray, targets: np.ndarray | None, want_loss: bool = True):
    inputs = np.ascontiguousarray(inputs, dtype=np.int32)
    B, T = inputs.shape
    tp = None
    if targets is not None:
        targets = np.ascontiguousarray(targets, dtype=np.int32)
        assert targets.shape == inputs.shape
        tp = _hptr(targets)
    loss = ct.c_float(0.0)
    rc = lib().gpt2_forward(h, _hptr(inputs), tp, B, T, ct.byref(loss) if want_loss else None)
    _check(rc, "gpt2_forward", allow=(GPT2_OK, GPT2_WARN_NONFINITE))
    return float(loss.value) if want_loss else None


def gpt2_forward_device(h, d_inputs: int, d_targets: int | None, B: int, T: int) -> None:
    _check(lib().gpt2_forward_device(h, d_inputs, d_targets, B, T), "gpt2_forward_device")


def gpt2_sample(h, prompt: np.ndarray, n_total: int, coins: np.ndarray) -> np.ndarray:
    """Generate tokens n_prompt .. n_total-1 after the prompt; coins: one
    uniform draw in [0, 1) per generated token.  Returns all n_total ids."""
    prompt = np.ascontiguousarray(prompt, dtype=np.int32).ravel()
    coins = np.ascontiguousarray(coins, dtype=np.float32).ravel()
    n_prompt = prompt.size
    assert coins.size == n_total - n_prompt
    tokens = np.zeros(n_total, np.int32)
    tokens[:n_prompt] = prompt
    _check(lib().gpt2_sample(h, _hptr(tokens), n_prompt, n_total, _hptr(coins)), "gpt2_sample")
    return tokens


def gpt2_sync(h) -> float:
    loss = ct.c_float(0.0)
    _check(lib().gpt2_sync(h, ct.byref(loss)), "gpt2_sync", allow=(GPT2_OK, GPT2_WARN_NONFINITE))
    return float(loss.value)


def gpt2_zero_grad(h) -> None:
    _check(lib().gpt2_zero_grad(h), "gpt2_zero_grad")


def gpt2_backward(h) -> None:
    _check(lib().gpt2_backward(h), "gpt2_backward")


def gpt2_update(h, lr, beta1, beta2, eps, weight_decay, t) -> None:
    _check(lib().gpt2_update(h, lr, beta1, beta2, eps, weight_decay, int(t)), "gpt2_update")


def gpt2_train_step_device(h, d_inputs: int, d_targets: int, B: int, T: int, lr, beta1, beta2, eps, weight_decay,
                           t, use_graph: bool = True) -> None:
    _check(lib().gpt2_train_step_device(h, d_inputs, d_targets, B, T, lr, beta1, beta2, eps, weight_decay, int(t),
                                        int(use_graph)), "gpt2_train_step_device")


def gpt2_train_step(h, inputs: np.ndarray, targets: np.ndarray, lr, beta1, beta2, eps, weight_decay, t) -> float:
    """One step from host (ideally pinned) int32 token arrays; returns the loss."""
    B, T = inputs.shape
    loss = ct.c_float(0.0)
    _check(lib().gpt2_train_step(h, _hptr(inputs), _hptr(targets), B, T, lr, beta1, beta2, eps, weight_decay, int(t),
                                 ct.byref(loss)), "gpt2_train_step", allow=(GPT2_OK, GPT2_WARN_NONFINITE))
    return float(loss.value)


TIMER_KINDS = {"off": 0, "gemm": 1, "adamw": 2, "xent": 3, "attn_fwd": 4, "attn_bwd": 5, "layernorm": 6,
               "encoder": 7}


def gpt2_kernel_timer(h, kind: str) -> None:
    _check(lib().gpt2_kernel_timer(h, TIMER_KINDS[kind]), "gpt2_kernel_timer")


def gpt2_kernel_timer_read(h):
    ms, n, work = ct.c_double(0), ct.c_longlong(0), ct.c_double(0)
    _check(lib().gpt2_kernel_timer_read(h, ct.byref(ms), ct.byref(n), ct.byref(work)), "gpt2_kernel_timer_read")
    return float(ms.value), int(n.value), float(work.value)


def set_wait_limit_ns(ns: int) -> None:
    """Limit of the device-side pipeline waits (0 restores the 1 s default)."""
    _check(lib().gpt2_set_wait_limit_ns(int(ns)), "gpt2_set_wait_limit_ns")


def plan_bf16_matmul(M: int, N: int, K: int, no_split: bool = False, logits: bool = False,
                     num_sms: int = 148) -> tuple:
    """(tile width, K splits) the bf16 tensor-core matmul takes for an M x N x K
    product on num_sms SMs.  Host-side: no device is touched."""
    bn, sp = ct.c_int(0), ct.c_int(0)
    _check(lib().gpt2_plan_bf16_matmul(int(M), int(N), int(K), int(bool(no_split)), int(bool(logits)), int(num_sms),
                                       ct.byref(bn), ct.byref(sp)), "gpt2_plan_bf16_matmul")
    return int(bn.value), int(sp.value)


def gpt2_free(h) -> None:
    _check(lib().gpt2_free(h), "gpt2_free")


class GPT2:
    """A handle plus the torch-owned arena it lives in."""

    def __init__(self, w, seed: int = 1337, maxB: int | None = None, maxT: int | None = None,
                 arena: str = "torch", stream=None):
        import torch

        self.w = w
        self.cfg = make_config(w)
        self.maxB = maxB or w.B
        self.maxT = maxT or w.T
        self.arena_bytes = gpt2_arena_bytes(self.cfg, self.maxB, self.maxT)
        if self.arena_bytes == 0:
            raise GPT2Error(GPT2_ERR_ARG, "gpt2_arena_bytes")
        self._arena = None
        aptr = None
        if arena == "torch":
            self._arena = torch.empty(self.arena_bytes, dtype=torch.uint8, device="cuda")
            aptr = self._arena.data_ptr()
        # a dedicated stream: the legacy default stream cannot be graph-captured
        self.stream = stream if stream is not None else torch.cuda.Stream()
        self.h = gpt2_build(self.cfg, seed, self.maxB, self.maxT, aptr, self.arena_bytes, self.stream.cuda_stream)
        self.n = int(lib().gpt2_num_parameters(self.h))

    def close(self):
        if getattr(self, "h", None):
            gpt2_free(self.h)
            self.h = None
        self._arena = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # the five calls
    def forward(self, inputs, targets=None, want_loss=True):
        return gpt2_forward(self.h, inputs, targets, want_loss)

    def _order_after_torch(self):
        """Make the handle's stream wait for work torch queued on its current
        stream (e.g. the copy that produced a device token tensor)."""
        import torch

        cur = torch.cuda.current_stream()
        if cur.cuda_stream != self.stream.cuda_stream:
            self.stream.wait_stream(cur)

    def forward_device(self, d_inputs, d_targets=None):
        B, T = d_inputs.shape
        self._order_after_torch()
        gpt2_forward_device(self.h, d_inputs.data_ptr(), None if d_targets is None else d_targets.data_ptr(), B, T)

    def sample(self, prompt, n_total: int, coins) -> np.ndarray:
        """The pages' generation loop; see gpt2_sample."""
        return gpt2_sample(self.h, prompt, n_total, coins)

    def sync(self) -> float:
        return gpt2_sync(self.h)

    def zero_grad(self):
        gpt2_zero_grad(self.h)

    def backward(self):
        gpt2_backward(self.h)

    def update(self, lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0, t=1):
        gpt2_update(self.h, lr, beta1, beta2, eps, weight_decay, t)

    def step(self, inputs, targets, t, lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0) -> float:
        """forward (returns the loss) -> zero_grad -> backward -> update."""
        loss = self.forward(inputs, targets)
        self.zero_grad()
        self.backward()
        self.update(lr, beta1, beta2, eps, weight_decay, t)
        return loss

    def train_step(self, inputs, targets, t, lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0):
        return gpt2_train_step(self.h, inputs, targets, lr, beta1, beta2, eps, weight_decay, t)

    def train_step_device(self, d_inputs, d_targets, t, lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8,
                          weight_decay=0.0, use_graph=True):
        B, T = d_inputs.shape
        self._order_after_torch()
        gpt2_train_step_device(self.h, d_inputs.data_ptr(), d_targets.data_ptr(), B, T, lr, beta1, beta2, eps,
                               weight_decay, t, use_graph)

    # inspection
    def get_params(self) -> np.ndarray:
        out = np.empty(self.n, np.float32)
        _check(lib().gpt2_get_params(self.h, _hptr(out), self.n), "gpt2_get_params")
        return out

    def set_params(self, p: np.ndarray):
        p = np.ascontiguousarray(p, dtype=np.float32)
        assert p.size == self.n
        _check(lib().gpt2_set_params(self.h, _hptr(p), self.n), "gpt2_set_params")

    def get_grads(self) -> np.ndarray:
        out = np.empty(self.n, np.float32)
        _check(lib().gpt2_get_grads(self.h, _hptr(out), self.n), "gpt2_get_grads")
        return out

    def get_opt_state(self):
        m = np.empty(self.n, np.float32)
        v = np.empty(self.n, np.float32)
        _check(lib().gpt2_get_opt_state(self.h, _hptr(m), _hptr(v), self.n), "gpt2_get_opt_state")
        return m, v

    def set_opt_state(self, m: np.ndarray, v: np.ndarray):
        m = np.ascontiguousarray(m, dtype=np.float32)
        v = np.ascontiguousarray(v, dtype=np.float32)
        _check(lib().gpt2_set_opt_state(self.h, _hptr(m), _hptr(v), self.n), "gpt2_set_opt_state")

    def get_logits(self, B: int, T: int) -> np.ndarray:
        n = B * T * self.cfg.padded_vocab_size
        out = np.empty(n, np.float32)
        _check(lib().gpt2_get_logits(self.h, _hptr(out), n), "gpt2_get_logits")
        return out.reshape(B, T, self.cfg.padded_vocab_size)

    def last_launch_count(self) -> int:
        return int(lib().gpt2_last_launch_count(self.h))


# --- kernel-level entry points (torch CUDA tensors in, results in place) -------
def _dptr(t):
    """Device pointer of a contiguous fp32 CUDA tensor (None -> NULL)."""
    if t is None:
        return None
    import torch

    if t.dtype not in (torch.float32, torch.uint8) or not t.is_cuda or not t.is_contiguous():
        raise TypeError(f"expected a contiguous float32 CUDA tensor, got {t.dtype} on {t.device}")
    return t.data_ptr()


def matmul_forward(out, x, W, bias=None, precision=GPT2_PREC_FP32, stream=None):
    """out = x W^T (+ bias), on the library's tensor-core kernels."""
    import torch

    OC, IC = W.shape
    N = x.numel() // IC
    ws = torch.empty(lib().gpt2op_matmul_workspace_bytes(N, IC, OC), dtype=torch.uint8, device=x.device)
    s = stream or torch.cuda.current_stream()
    _check(lib().gpt2op_matmul_forward(_dptr(out), _dptr(x), _dptr(W), _dptr(bias), N, IC, OC, precision,
                                       _dptr(ws), s.cuda_stream), "gpt2op_matmul_forward")


def matmul_backward(dx, dW, dbias, dy, x, W, precision=GPT2_PREC_FP32, stream=None):
    """dx = dy W; dW += dy^T x; dbias += column sums of dy."""
    import torch

    OC, IC = W.shape
    N = x.numel() // IC
    ws = torch.empty(lib().gpt2op_matmul_workspace_bytes(N, IC, OC), dtype=torch.uint8, device=x.device)
    s = stream or torch.cuda.current_stream()
    _check(lib().gpt2op_matmul_backward(_dptr(dx), _dptr(dW), _dptr(dbias), _dptr(dy), _dptr(x), _dptr(W), N, IC,
                                        OC, precision, _dptr(ws), s.cuda_stream), "gpt2op_matmul_backward")


def attention_forward(y, lse, qkv, NH, precision=GPT2_PREC_FP32, stream=None):
    """Causal attention forward: y (B,T,C), lse (B,NH,T) from qkv (B,T,3C)."""
    import torch

    B, T, C3 = qkv.shape
    C = C3 // 3
    ws = torch.empty(lib().gpt2op_attention_workspace_bytes(B, T, C), dtype=torch.uint8, device=qkv.device)
    s = stream or torch.cuda.current_stream()
    _check(lib().gpt2op_attention_forward(_dptr(y), _dptr(lse), _dptr(qkv), B, T, C, NH, precision, _dptr(ws),
                                          s.cuda_stream), "gpt2op_attention_forward")


def attention_backward(dqkv, dy, qkv, NH, precision=GPT2_PREC_FP32, stream=None):
    """dqkv (B,T,3C) from the upstream gradient dy (B,T,C) of causal attention."""
    import torch

    B, T, C3 = qkv.shape
    C = C3 // 3
    ws = torch.empty(lib().gpt2op_attention_backward_workspace_bytes(B, T, C, NH), dtype=torch.uint8,
                     device=qkv.device)
    s = stream or torch.cuda.current_stream()
    _check(lib().gpt2op_attention_backward(_dptr(dqkv), _dptr(dy), _dptr(qkv), B, T, C, NH, precision, _dptr(ws),
                                           s.cuda_stream), "gpt2op_attention_backward")


def matmul_backward_noalloc(dx, dW, dbias, dy, x, W, precision=GPT2_PREC_FP32, stream=None):
    """matmul_backward for callers that cannot allocate device memory: the
    library takes its scratch from a fixed array of its own (8 MiB per GPU,
    held until exit) instead of a workspace.  Calls that overlap on one GPU
    race on that array.  Raises GPT2Error (GPT2_ERR_SHAPE) when
    ceil(N/64) * OC > 1,048,576 with a bias gradient."""
    import torch

    OC, IC = W.shape
    N = x.numel() // IC
    s = stream or torch.cuda.current_stream()
    _check(lib().gpt2op_matmul_backward_noalloc(_dptr(dx), _dptr(dW), _dptr(dbias), _dptr(dy), _dptr(x), _dptr(W),
                                                N, IC, OC, precision, s.cuda_stream),
           "gpt2op_matmul_backward_noalloc")
