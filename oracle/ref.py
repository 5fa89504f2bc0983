"""ctypes wrapper around the CPU oracle (``gpt2_ref.c``).

TEST INFRASTRUCTURE ONLY: imported by tests/, by ``__graft_entry__.smoke()``
and by bench.py's CPU-baseline leg.  The CUDA package never imports it.

``RefModel`` mirrors the five calls of llm.c's train_gpt2.c named on the page
«llm.c：Andrej Karpathy带你从零复现LLM», section «核心代码解读：train_gpt2.c»,
item 3 (build, forward, zero_grad, backward, update), with numpy views onto
the oracle's flat parameter, gradient, optimizer-state and activation
buffers.  ``ops(dtype)`` exposes the per-layer functions of item 1;
``sample_mult`` and ``generate`` follow item 5 (sampling generation).
"""
from __future__ import annotations

import ctypes as ct
import os

import numpy as np

from . import build as _build

PARAM_NAMES = [
    "wte", "wpe", "ln1w", "ln1b", "qkvw", "qkvb", "attprojw", "attprojb",
    "ln2w", "ln2b", "fcw", "fcb", "fcprojw", "fcprojb", "lnfw", "lnfb",
]
ACT_NAMES = [
    "encoded", "ln1", "ln1_mean", "ln1_rstd", "qkv", "atty", "preatt", "att", "attproj",
    "residual2", "ln2", "ln2_mean", "ln2_rstd", "fch", "fch_gelu", "fcproj", "residual3",
    "lnf", "lnf_mean", "lnf_rstd", "logits", "probs", "losses",
]


class RefConfig(ct.Structure):
    _fields_ = [(n, ct.c_int) for n in
                ("max_seq_len", "vocab_size", "padded_vocab_size", "num_layers", "num_heads", "channels", "llama")]


_LIBS: dict = {}


def _lib(dtype) -> ct.CDLL:
    key = "f32" if np.dtype(dtype) == np.float32 else "f64"
    if key not in _LIBS:
        paths = _build.build()
        lib = ct.CDLL(paths[key])
        P = ct.c_void_p
        I, LL, D = ct.c_int, ct.c_longlong, ct.c_double
        lib.ref_create.restype = P
        lib.ref_create.argtypes = [ct.POINTER(RefConfig), I, I]
        lib.ref_destroy.argtypes = [P]
        for n in ("ref_params", "ref_grads", "ref_m", "ref_v"):
            getattr(lib, n).restype = P
            getattr(lib, n).argtypes = [P]
        lib.ref_act.restype = P
        lib.ref_act.argtypes = [P, I]
        lib.ref_num_parameters.restype = LL
        lib.ref_num_parameters.argtypes = [ct.POINTER(RefConfig), I]
        lib.ref_num_activations.restype = LL
        lib.ref_num_activations.argtypes = [ct.POINTER(RefConfig), I, I, I]
        lib.ref_param_offset.restype = LL
        lib.ref_param_offset.argtypes = [ct.POINTER(RefConfig), I]
        lib.ref_forward.restype = D
        lib.ref_forward.argtypes = [P, P, P, I, I]
        lib.ref_zero_grad.argtypes = [P]
        lib.ref_backward.restype = I
        lib.ref_backward.argtypes = [P]
        lib.ref_update.argtypes = [P, D, D, D, D, D, I]
        _LIBS[key] = lib
    return _LIBS[key]


def make_config(max_seq_len, vocab_size, padded_vocab_size, num_layers, num_heads, channels,
                llama: int = 0) -> RefConfig:
    return RefConfig(max_seq_len, vocab_size, padded_vocab_size, num_layers, num_heads, channels, int(llama))


def config_from(w) -> RefConfig:
    """Build a RefConfig from any object with the GPT-2 shape fields (and an
    optional ``llama`` flag: RMSNorm, RoPE, no position table, no biases)."""
    return make_config(w.max_seq_len, w.vocab_size, w.padded_vocab_size, w.num_layers, w.num_heads, w.channels,
                       getattr(w, "llama", 0))


def num_parameters(cfg: RefConfig, padded: bool = True) -> int:
    return int(_lib(np.float32).ref_num_parameters(ct.byref(cfg), int(padded)))


def num_activations(cfg: RefConfig, B: int, T: int, padded: bool = True) -> int:
    return int(_lib(np.float32).ref_num_activations(ct.byref(cfg), B, T, int(padded)))


def param_offsets(cfg: RefConfig) -> dict:
    lib = _lib(np.float32)
    offs = [int(lib.ref_param_offset(ct.byref(cfg), i)) for i in range(17)]
    return {n: (offs[i], offs[i + 1] - offs[i]) for i, n in enumerate(PARAM_NAMES)}


def _ptr(a: np.ndarray) -> ct.c_void_p:
    return ct.c_void_p(a.ctypes.data)


class RefModel:
    """The oracle's GPT2 struct: flat params, grads, AdamW m and v, activations."""

    def __init__(self, cfg: RefConfig, maxB: int, maxT: int, dtype=np.float32):
        self.cfg = cfg
        self.dtype = np.dtype(dtype)
        self.lib = _lib(dtype)
        self.maxB, self.maxT = maxB, maxT
        self.h = self.lib.ref_create(ct.byref(cfg), maxB, maxT)
        if not self.h:
            raise MemoryError("oracle allocation failed")
        self.n = num_parameters(cfg, True)
        self.offsets = param_offsets(cfg)
        self.B = self.T = 0

    def close(self):
        if self.h:
            self.lib.ref_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _view(self, addr, n) -> np.ndarray:
        ctype = ct.c_float if self.dtype == np.float32 else ct.c_double
        return np.ctypeslib.as_array(ct.cast(addr, ct.POINTER(ctype)), shape=(n,))

    @property
    def params(self) -> np.ndarray:
        return self._view(self.lib.ref_params(self.h), self.n)

    @property
    def grads(self) -> np.ndarray:
        return self._view(self.lib.ref_grads(self.h), self.n)

    @property
    def m(self) -> np.ndarray:
        return self._view(self.lib.ref_m(self.h), self.n)

    @property
    def v(self) -> np.ndarray:
        return self._view(self.lib.ref_v(self.h), self.n)

    def tensor(self, flat: np.ndarray, name: str) -> np.ndarray:
        off, n = self.offsets[name]
        return flat[off: off + n]

    def act(self, name: str) -> np.ndarray:
        """Activation tensor ``name`` of the last forward (flat view)."""
        c = self.cfg
        B, T = self.B, self.T
        L, C, NH, Vp = c.num_layers, c.channels, c.num_heads, c.padded_vocab_size
        BT = B * T
        sizes = {
            "encoded": BT * C, "ln1": L * BT * C, "ln1_mean": L * BT, "ln1_rstd": L * BT,
            "qkv": L * BT * 3 * C, "atty": L * BT * C, "preatt": L * B * NH * T * T,
            "att": L * B * NH * T * T, "attproj": L * BT * C, "residual2": L * BT * C,
            "ln2": L * BT * C, "ln2_mean": L * BT, "ln2_rstd": L * BT, "fch": L * BT * 4 * C,
            "fch_gelu": L * BT * 4 * C, "fcproj": L * BT * C, "residual3": L * BT * C,
            "lnf": BT * C, "lnf_mean": BT, "lnf_rstd": BT, "logits": BT * Vp, "probs": BT * Vp,
            "losses": BT,
        }
        i = ACT_NAMES.index(name)
        return self._view(self.lib.ref_act(self.h, i), sizes[name])

    def set_params(self, p: np.ndarray):
        self.params[:] = np.asarray(p, dtype=self.dtype)

    def forward(self, inputs: np.ndarray, targets: np.ndarray | None) -> float:
        inputs = np.ascontiguousarray(inputs, dtype=np.int32)
        B, T = inputs.shape
        tp = None
        if targets is not None:
            targets = np.ascontiguousarray(targets, dtype=np.int32)
            tp = _ptr(targets)
        loss = self.lib.ref_forward(self.h, _ptr(inputs), tp, B, T)
        if loss in (-2.0, -3.0):
            raise ValueError("oracle rejected the batch (shape or token range)")
        self.B, self.T = B, T
        return float(loss)

    def zero_grad(self):
        self.lib.ref_zero_grad(self.h)

    def backward(self) -> int:
        return int(self.lib.ref_backward(self.h))

    def update(self, lr, beta1, beta2, eps, weight_decay, t):
        self.lib.ref_update(self.h, lr, beta1, beta2, eps, weight_decay, int(t))

    def step(self, inputs, targets, t, lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0) -> float:
        """forward -> zero_grad -> backward -> update, the order of the llm.c loop."""
        loss = self.forward(inputs, targets)
        self.zero_grad()
        rc = self.backward()
        if rc != 0:
            raise RuntimeError(f"oracle backward failed: {rc}")
        self.update(lr, beta1, beta2, eps, weight_decay, t)
        return loss


class Ops:
    """Per-layer functions of the oracle, taking and returning numpy arrays."""

    def __init__(self, dtype=np.float64):
        self.dtype = np.dtype(dtype)
        self.lib = _lib(dtype)

    def _a(self, x):
        return np.ascontiguousarray(x, dtype=self.dtype)

    def encoder_forward(self, ids, wte, wpe):
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        B, T = ids.shape
        C = wte.shape[1]
        wte, wpe = self._a(wte), self._a(wpe)
        out = np.zeros((B, T, C), self.dtype)
        self.lib.encoder_forward(_ptr(out), _ptr(ids), _ptr(wte), _ptr(wpe), B, T, C)
        return out

    def encoder_backward(self, dx, ids, Vrows, maxT):
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        B, T = ids.shape
        C = dx.shape[-1]
        dx = self._a(dx)
        dwte = np.zeros((Vrows, C), self.dtype)
        dwpe = np.zeros((maxT, C), self.dtype)
        self.lib.encoder_backward(_ptr(dwte), _ptr(dwpe), _ptr(dx), _ptr(ids), B, T, C)
        return dwte, dwpe

    def layernorm_forward(self, x, w, b):
        x, w, b = self._a(x), self._a(w), self._a(b)
        C = x.shape[-1]
        N = x.size // C
        y = np.zeros_like(x)
        mean = np.zeros(N, self.dtype)
        rstd = np.zeros(N, self.dtype)
        self.lib.layernorm_forward(_ptr(y), _ptr(mean), _ptr(rstd), _ptr(x), _ptr(w), _ptr(b), N, C)
        return y, mean, rstd

    def layernorm_backward(self, dy, x, w, mean, rstd):
        dy, x, w, mean, rstd = map(self._a, (dy, x, w, mean, rstd))
        C = x.shape[-1]
        N = x.size // C
        dx = np.zeros_like(x)
        dw = np.zeros(C, self.dtype)
        db = np.zeros(C, self.dtype)
        self.lib.layernorm_backward(_ptr(dx), _ptr(dw), _ptr(db), _ptr(dy), _ptr(x), _ptr(w),
                                    _ptr(mean), _ptr(rstd), N, C)
        return dx, dw, db

    def rmsnorm_forward(self, x, w):
        """y = x * rstd * w, rstd = 1/sqrt(mean(x^2) + 1e-5) per row."""
        x, w = self._a(x), self._a(w)
        C = x.shape[-1]
        N = x.size // C
        y = np.zeros_like(x)
        rstd = np.zeros(N, self.dtype)
        self.lib.rmsnorm_forward(_ptr(y), _ptr(rstd), _ptr(x), _ptr(w), N, C)
        return y, rstd

    def rmsnorm_backward(self, dy, x, w, rstd):
        dy, x, w, rstd = map(self._a, (dy, x, w, rstd))
        C = x.shape[-1]
        N = x.size // C
        dx = np.zeros_like(x)
        dw = np.zeros(C, self.dtype)
        self.lib.rmsnorm_backward(_ptr(dx), _ptr(dw), _ptr(dy), _ptr(x), _ptr(w), _ptr(rstd), N, C)
        return dx, dw

    def rope_apply(self, qkv, NH, inverse=False):
        """Rotary position embedding of the q and k blocks of qkv (B,T,3C) (a copy)."""
        qkv = self._a(qkv).copy()
        B, T, C3 = qkv.shape
        self.lib.rope_apply(_ptr(qkv), B, T, C3 // 3, NH, int(bool(inverse)))
        return qkv

    def matmul_forward(self, x, W, bias=None):
        x, W = self._a(x), self._a(W)
        OC, IC = W.shape
        N = x.size // IC
        out = np.zeros(x.shape[:-1] + (OC,), self.dtype)
        bp = None
        if bias is not None:
            bias = self._a(bias)
            bp = _ptr(bias)
        self.lib.matmul_forward(_ptr(out), _ptr(x), _ptr(W), bp, N, IC, OC)
        return out

    def matmul_backward(self, dy, x, W, with_bias=True):
        dy, x, W = self._a(dy), self._a(x), self._a(W)
        OC, IC = W.shape
        N = x.size // IC
        dx = np.zeros_like(x)
        dW = np.zeros_like(W)
        db = np.zeros(OC, self.dtype) if with_bias else None
        self.lib.matmul_backward(_ptr(dx), _ptr(dW), _ptr(db) if with_bias else None, _ptr(dy), _ptr(x),
                                 _ptr(W), N, IC, OC)
        return dx, dW, db

    def attention_forward(self, qkv, NH):
        qkv = self._a(qkv)
        B, T, C3 = qkv.shape
        C = C3 // 3
        out = np.zeros((B, T, C), self.dtype)
        preatt = np.zeros((B, NH, T, T), self.dtype)
        att = np.zeros((B, NH, T, T), self.dtype)
        self.lib.attention_forward(_ptr(out), _ptr(preatt), _ptr(att), _ptr(qkv), B, T, C, NH)
        return out, preatt, att

    def attention_backward(self, dout, qkv, att, NH):
        dout, qkv, att = self._a(dout), self._a(qkv), self._a(att)
        B, T, C3 = qkv.shape
        C = C3 // 3
        dqkv = np.zeros_like(qkv)
        self.lib.attention_backward(_ptr(dqkv), _ptr(dout), _ptr(qkv), _ptr(att), B, T, C, NH)
        return dqkv

    def gelu_forward(self, x):
        x = self._a(x)
        y = np.zeros_like(x)
        self.lib.gelu_forward(_ptr(y), _ptr(x), ct.c_longlong(x.size))
        return y

    def gelu_backward(self, x, dy):
        x, dy = self._a(x), self._a(dy)
        dx = np.zeros_like(x)
        self.lib.gelu_backward(_ptr(dx), _ptr(x), _ptr(dy), ct.c_longlong(x.size))
        return dx

    def residual_forward(self, a, b):
        a, b = self._a(a), self._a(b)
        out = np.zeros_like(a)
        self.lib.residual_forward(_ptr(out), _ptr(a), _ptr(b), ct.c_longlong(a.size))
        return out

    def residual_backward(self, dout):
        dout = self._a(dout)
        da = np.zeros_like(dout)
        db = np.zeros_like(dout)
        self.lib.residual_backward(_ptr(da), _ptr(db), _ptr(dout), ct.c_longlong(dout.size))
        return da, db

    def softmax_forward(self, logits, V):
        logits = self._a(logits)
        Vp = logits.shape[-1]
        N = logits.size // Vp
        probs = np.zeros_like(logits)
        self.lib.softmax_forward(_ptr(probs), _ptr(logits), N, V, Vp)
        return probs

    def crossentropy_forward(self, probs, targets):
        probs = self._a(probs)
        targets = np.ascontiguousarray(targets, dtype=np.int32).reshape(-1)
        Vp = probs.shape[-1]
        N = probs.size // Vp
        losses = np.zeros(N, self.dtype)
        self.lib.crossentropy_forward(_ptr(losses), _ptr(probs), _ptr(targets), N, Vp)
        return losses

    def crossentropy_softmax_backward(self, dlosses, probs, targets, V):
        probs = self._a(probs)
        dlosses = self._a(dlosses).reshape(-1)
        targets = np.ascontiguousarray(targets, dtype=np.int32).reshape(-1)
        Vp = probs.shape[-1]
        N = probs.size // Vp
        dlogits = np.zeros_like(probs)
        self.lib.crossentropy_softmax_backward(_ptr(dlogits), _ptr(dlosses), _ptr(probs), _ptr(targets), N, V, Vp)
        return dlogits

    def adamw_update(self, p, g, m, v, lr, b1, b2, eps, wd, t):
        p, g, m, v = (self._a(a).copy() for a in (p, g, m, v))
        self.lib.adamw_update(_ptr(p), _ptr(g), _ptr(m), _ptr(v), ct.c_longlong(p.size), ct.c_double(lr),
                              ct.c_double(b1), ct.c_double(b2), ct.c_double(eps), ct.c_double(wd), int(t))
        return p, m, v


def ops(dtype=np.float64) -> Ops:
    return Ops(dtype)


# ---------------------------------------------------------------------------
# Generation: the page «llm.c：Andrej Karpathy带你从零复现LLM», section
# «核心代码解读：train_gpt2.c», item 5 -- sample_mult draws an index from a
# probability distribution and the main loop generates a sequence with it.
# The pages do not print the function; the reading here is inverse-CDF
# sampling with the uniform draw passed in.
# ---------------------------------------------------------------------------
def softmax64(logits) -> np.ndarray:
    """softmax of a 1-D logits vector in float64 (max-subtracted)."""
    x = np.asarray(logits, dtype=np.float64).ravel()
    e = np.exp(x - x.max())
    return e / e.sum()


def sample_mult(probs, coin: float) -> int:
    """The first index whose cumulative probability exceeds coin (a uniform
    draw in [0, 1)); when rounding leaves coin at or above every prefix, the
    last index with a nonzero probability.  Prefix sums in float64, in index
    order."""
    p = np.asarray(probs, dtype=np.float64).ravel()
    cdf = np.cumsum(p)
    i = int(np.searchsorted(cdf, coin, side="right"))  # first i with cdf[i] > coin
    if i >= p.size:
        nz = np.nonzero(p > 0)[0]
        i = int(nz[-1]) if nz.size else p.size - 1
    return i


def sample_is_valid(probs, coin: float, index: int, tol: float) -> bool:
    """Whether index is the inverse-CDF draw for coin up to a tolerance tol on
    the cumulative probabilities: cdf[index-1] - tol <= coin < cdf[index] + tol
    and probs[index] > 0 (several indices qualify when coin lies within tol of
    a boundary)."""
    p = np.asarray(probs, dtype=np.float64).ravel()
    if not 0 <= index < p.size or p[index] <= 0:
        return False
    cdf = np.cumsum(p)
    lo = cdf[index - 1] if index > 0 else 0.0
    return lo - tol <= coin < cdf[index] + tol


def generate(model: RefModel, prompt, n_total: int, coins, vocab_size: int) -> np.ndarray:
    """The generation loop on the oracle: for t = len(prompt) .. n_total-1, a
    forward without targets over the n_total positions (positions not yet
    generated hold prompt[0]), then tokens[t] = sample_mult(softmax of logits
    row t-1 over the real vocabulary, coins[t - len(prompt)])."""
    prompt = np.asarray(prompt, dtype=np.int32).ravel()
    tokens = np.full(n_total, prompt[0], np.int32)
    tokens[:prompt.size] = prompt
    for t in range(prompt.size, n_total):
        model.forward(tokens[None, :], None)
        logits = model.act("logits").reshape(n_total, -1)[t - 1, :vocab_size]
        tokens[t] = sample_mult(softmax64(logits), float(coins[t - prompt.size]))
    return tokens
