"""Seeded synthetic inputs shared by the oracle tests, the GPU tests and bench.py.

This module holds no arithmetic of the training step itself.  It only draws
the numbers that both sides are fed: initial parameters and token batches.
It is deliberately independent of both the CUDA package and ``oracle/``;
each of those is handed the arrays produced here.

Generators (our own specification; the llm.c pages give no seeds):

* SplitMix64 (S. Vigna's published mixer).  Draw ``i`` of stream ``seed`` is
  ``mix(seed + (i + 1) * 0x9E3779B97F4A7C15)``, so every draw is addressable
  by its counter and a GPU kernel can reproduce any element independently.
* 53-bit uniforms ``(x >> 11) * 2**-53`` in [0, 1).
* Box-Muller normals: normal ``i`` uses the uniform pair ``(2j, 2j+1)`` with
  ``j = i // 2``; even ``i`` takes the cosine branch, odd ``i`` the sine one,
  ``r = sqrt(-2 ln(1 - u0))``.
* Zipf(s) token ids: rank ``k = 1..V`` has probability proportional to
  ``k**-s``; id ``k - 1``; sampled by inverse CDF on a float64 cumulative
  table (smallest k whose cumulative mass exceeds u).

Workloads follow the five GPT-2 shapes the build is measured on; the llm.c
pages' own console log (page «千行C代码训完GPT-2», section «快速入门») quotes
GPT-2 124M with max_seq_len 1024, vocab 50257, 12 layers, 12 heads and 768
channels.
"""
from __future__ import annotations

import math
import os
from dataclasses import dataclass

import numpy as np

GOLDEN_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

INIT_SEED = 1337
TOKEN_SEED = 42


@dataclass(frozen=True)
class Workload:
    """One GPT-2 shape plus the batch it is run with."""

    name: str
    num_layers: int
    channels: int
    num_heads: int
    vocab_size: int
    padded_vocab_size: int
    max_seq_len: int
    B: int
    T: int
    precision: str  # "fp32" or "bf16" (bf16 operands, fp32 accumulate / master)
    tokens: str  # "uniform" or "zipf"
    steps: int
    lr: float = 1e-4
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.0
    llama: int = 0  # 1: RMSNorm, RoPE, no position table, no biases

    @property
    def BT(self) -> int:
        return self.B * self.T

    @property
    def gemm_precision(self) -> int:
        return 0 if self.precision == "fp32" else 1


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_L2_C64", 2, 64, 4, 512, 512, 32, 2, 32, "fp32", "uniform", 10),
        Workload("gpt2_124m_B4_T64_fp32", 12, 768, 12, 50257, 50304, 1024, 4, 64, "fp32", "zipf", 10),
        Workload("gpt2_124m_B16_T1024_bf16", 12, 768, 12, 50257, 50304, 1024, 16, 1024, "bf16", "zipf", 20),
        Workload("gpt2_350m_B8_T1024_bf16", 24, 1024, 16, 50304, 50304, 1024, 8, 1024, "bf16", "zipf", 20),
        Workload("gpt2_774m_B4_T1024_bf16", 36, 1280, 20, 50304, 50304, 1024, 4, 1024, "bf16", "zipf", 20),
    ]
}


def splitmix64(seed: int, counters: np.ndarray) -> np.ndarray:
    """Draw ``counters[k]`` of the SplitMix64 stream seeded with ``seed``."""
    c = np.asarray(counters, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + (c + np.uint64(1)) * GOLDEN_GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def uniform53(seed: int, counters: np.ndarray) -> np.ndarray:
    """Uniform float64 in [0, 1) from the top 53 bits of each draw."""
    return (splitmix64(seed, counters) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def _normals_chunk(seed: int, start: int, n: int) -> np.ndarray:
    j0 = start >> 1
    j1 = (start + n + 1) >> 1
    pair = np.arange(j0, j1, dtype=np.uint64)
    u0 = uniform53(seed, pair * np.uint64(2))
    u1 = uniform53(seed, pair * np.uint64(2) + np.uint64(1))
    r = np.sqrt(-2.0 * np.log1p(-u0))
    ang = 2.0 * math.pi * u1
    both = np.empty(2 * (j1 - j0), dtype=np.float64)
    both[0::2] = r * np.cos(ang)
    both[1::2] = r * np.sin(ang)
    off = start - 2 * j0
    return both[off: off + n]


def normals(seed: int, start: int, n: int) -> np.ndarray:
    """Standard normals with counters ``start .. start+n-1`` (Box-Muller)."""
    if n <= 0:
        return np.zeros(0, dtype=np.float64)
    chunk = 1 << 21
    if n <= chunk:
        return _normals_chunk(seed, start, n)
    from concurrent.futures import ThreadPoolExecutor

    out = np.empty(n, dtype=np.float64)

    def work(s):
        m = min(chunk, n - s)
        out[s: s + m] = _normals_chunk(seed, start + s, m)

    with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
        list(ex.map(work, range(0, n, chunk)))
    return out


# ---------------------------------------------------------------------------
# parameter layout (flat, padded vocab) -- the order of the 16 tensors of the
# llm.c ParameterTensors struct (page «llm.c：Andrej Karpathy带你从零复现LLM»,
# section «核心代码解读：train_gpt2.c», item 2); orientation (out, in).
# ---------------------------------------------------------------------------
PARAM_NAMES = [
    "wte", "wpe", "ln1w", "ln1b", "qkvw", "qkvb", "attprojw", "attprojb",
    "ln2w", "ln2b", "fcw", "fcb", "fcprojw", "fcprojb", "lnfw", "lnfb",
]


def param_shapes(w: Workload, padded: bool = True) -> dict:
    L, C = w.num_layers, w.channels
    Vr = w.padded_vocab_size if padded else w.vocab_size
    shapes = {
        "wte": (Vr, C), "wpe": (w.max_seq_len, C),
        "ln1w": (L, C), "ln1b": (L, C),
        "qkvw": (L, 3 * C, C), "qkvb": (L, 3 * C),
        "attprojw": (L, C, C), "attprojb": (L, C),
        "ln2w": (L, C), "ln2b": (L, C),
        "fcw": (L, 4 * C, C), "fcb": (L, 4 * C),
        "fcprojw": (L, C, 4 * C), "fcprojb": (L, C),
        "lnfw": (C,), "lnfb": (C,),
    }
    if w.llama:  # the tensors keep their places with no elements
        for name in ("wpe", "ln1b", "qkvb", "attprojb", "ln2b", "fcb", "fcprojb", "lnfb"):
            shapes[name] = (0,)
    return shapes


def param_offsets(w: Workload) -> dict:
    off, out = 0, {}
    for name, shp in param_shapes(w).items():
        n = int(np.prod(shp))
        out[name] = (off, n)
        off += n
    return out


def num_params(w: Workload, padded: bool = True) -> int:
    return int(sum(int(np.prod(s)) for s in param_shapes(w, padded).values()))


_INIT_CACHE: dict = {}


def init_params(w: Workload, seed: int = INIT_SEED, wte_std: float = 0.02) -> np.ndarray:
    """Initial flat fp32 parameters (a fresh copy; draws are memoised).

    Matrices N(0, 0.02) (attention and MLP output projections additionally
    scaled by 1/sqrt(2L)); biases 0; layernorm gains 1 and shifts 0; padded
    wte rows [V, Vp) are 0.  Element ``i`` of the flat buffer uses normal
    counter ``i`` so any element can be regenerated on its own.
    """
    key = (w, seed, wte_std)
    if key in _INIT_CACHE:
        return _INIT_CACHE[key].copy()
    offs = param_offsets(w)
    n_total = num_params(w)
    out = np.zeros(n_total, dtype=np.float32)
    proj_std = 0.02 / math.sqrt(2.0 * w.num_layers)
    stds = {"wte": wte_std, "wpe": 0.02, "qkvw": 0.02, "attprojw": proj_std, "fcw": 0.02, "fcprojw": proj_std}
    chunk = 1 << 25
    for name, (off, n) in offs.items():
        if name in stds:
            nreal = n
            if name == "wte":
                nreal = w.vocab_size * w.channels
            for s in range(0, nreal, chunk):
                m = min(chunk, nreal - s)
                out[off + s: off + s + m] = stds[name] * normals(seed, off + s, m)
        elif name in ("ln1w", "ln2w", "lnfw"):
            out[off: off + n] = 1.0
    _INIT_CACHE.clear()
    _INIT_CACHE[key] = out
    return out.copy()


# ---------------------------------------------------------------------------
# token streams (the llm.c data files are raw int32 token ids; page
# «千行C代码训完GPT-2», section «快速入门»)
# ---------------------------------------------------------------------------
_ZIPF_CACHE: dict = {}


def zipf_cdf(V: int, s: float = 1.1) -> np.ndarray:
    key = (V, s)
    if key not in _ZIPF_CACHE:
        k = np.arange(1, V + 1, dtype=np.float64)
        p = k ** (-s)
        c = np.cumsum(p)
        _ZIPF_CACHE[key] = c / c[-1]
    return _ZIPF_CACHE[key]


def token_stream(w: Workload, start: int, n: int, seed: int = TOKEN_SEED) -> np.ndarray:
    """``n`` int32 token ids with counters ``start .. start+n-1``."""
    u = uniform53(seed, np.arange(start, start + n, dtype=np.uint64))
    if w.tokens == "uniform":
        ids = np.floor(u * w.vocab_size).astype(np.int64)
    else:
        ids = np.searchsorted(zipf_cdf(w.vocab_size), u, side="right")
    return np.minimum(ids, w.vocab_size - 1).astype(np.int32)


def batch(w: Workload, step: int = 0, seed: int = TOKEN_SEED, B: int | None = None, T: int | None = None):
    """(inputs, targets), each int32 (B, T): B*T+1 consecutive stream tokens,
    targets shifted by one (next-token prediction)."""
    B = w.B if B is None else B
    T = w.T if T is None else T
    n = B * T + 1
    x = token_stream(w, step * n, n, seed)
    return x[:-1].reshape(B, T).copy(), x[1:].reshape(B, T).copy()


def randn(seed: int, shape, scale: float = 1.0, dtype=np.float32) -> np.ndarray:
    """Seeded standard normals (counter-based, as above) of the given shape."""
    n = int(np.prod(shape))
    return (scale * normals(seed, 0, n)).astype(dtype).reshape(shape)
