"""Host-side checks of the C-ABI library (no GPU needed): it loads, exports
every symbol include/gpt2b300.h declares, rejects bad configs and shapes
before touching the device, and plans arenas of the expected size."""
import ctypes as ct
import os
import re

import pytest

import gpt_train_step_02_b300 as g
import synth
from gpt_train_step_02_b300 import build as gbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    gbuild.build()


def header_symbols():
    src = open(os.path.join(ROOT, "include", "gpt2b300.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gpt2(?:op)?_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    syms = header_symbols()
    assert len(syms) >= 19
    lib = ct.CDLL(g.LIB_PATH)
    for s in syms:
        assert hasattr(lib, s), s
    assert sorted(g.EXPORTS) == syms


def test_library_links_no_cuda_runtime_dynamically():
    # static cudart: the library loads on a machine without a GPU
    out = os.popen(f"ldd {g.LIB_PATH}").read()
    assert "libcudart" not in out


def test_status_strings():
    for code in (0, -1, -2, -3, -4, -5, -6, -7, 1):
        assert g.status_string(code) not in ("", "unknown status")
    assert g.status_string(12345) == "unknown status"


def test_arena_bytes_and_config_validation():
    for w in synth.WORKLOADS.values():
        n = g.gpt2_arena_bytes(g.make_config(w), w.B, w.T)
        np_ = synth.num_params(w)
        assert n > 4 * 4 * np_  # params, grads, m, v at least
        assert n % 256 == 0
    w = synth.WORKLOADS["tiny_L2_C64"]
    c = g.make_config(w)
    assert g.gpt2_arena_bytes(c, 0, 4) == 0
    assert g.gpt2_arena_bytes(c, 2, w.max_seq_len + 1) == 0
    bad = g.make_config(w)
    bad.num_heads = 5  # 64 % 5 != 0
    assert g.gpt2_arena_bytes(bad, 2, 8) == 0
    bad = g.make_config(w)
    bad.vocab_size = bad.padded_vocab_size + 1
    assert g.gpt2_arena_bytes(bad, 2, 8) == 0


def test_build_rejects_bad_arguments_without_touching_the_device():
    L = g.lib()
    h = ct.c_void_p()
    w = synth.WORKLOADS["tiny_L2_C64"]
    c = g.make_config(w)
    assert L.gpt2_build(None, ct.byref(c), 1, 2, 8, None, 0, None) == g.GPT2_ERR_ARG
    bad = g.make_config(w)
    bad.gemm_precision = 7
    assert L.gpt2_build(ct.byref(h), ct.byref(bad), 1, 2, 8, None, 0, None) == g.GPT2_ERR_ARG
    assert L.gpt2_build(ct.byref(h), ct.byref(c), 1, 2, w.max_seq_len + 1, None, 0, None) == g.GPT2_ERR_SHAPE
    # caller arena too small / misaligned
    assert L.gpt2_build(ct.byref(h), ct.byref(c), 1, 2, 8, ct.c_void_p(1 << 20), 16, None) == g.GPT2_ERR_ARENA
    n = g.gpt2_arena_bytes(c, 2, 8)
    assert L.gpt2_build(ct.byref(h), ct.byref(c), 1, 2, 8, ct.c_void_p((1 << 20) + 8), n, None) == g.GPT2_ERR_ARENA
    # NULL handle everywhere
    assert L.gpt2_forward(None, None, None, 1, 1, None) == g.GPT2_ERR_ARG
    assert L.gpt2_backward(None) == g.GPT2_ERR_ARG
    assert L.gpt2_zero_grad(None) == g.GPT2_ERR_ARG
    assert L.gpt2_update(None, 1e-4, 0.9, 0.999, 1e-8, 0.0, 1) == g.GPT2_ERR_ARG
    assert L.gpt2_free(None) == g.GPT2_ERR_ARG
    assert L.gpt2_num_parameters(None) == -1
