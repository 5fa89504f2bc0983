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


# The bf16 matmul planner (host logic, no device): the plans the design notes
# and the launch lists record for the GPT-2 product shapes on 148 SMs.
PLAN_CASES = [
    # (M, N, K): (tile width, K splits)
    ((4096, 1280, 1280), (192, 1)),    # 774M attention projection, B*T = 4096: 224 tiles, not 160 of 256
    ((4096, 1280, 5120), (192, 1)),    # 774M MLP output projection
    ((2304, 768, 16384), (192, 2)),    # 124M QKV weight gradient
    ((768, 768, 16384), (128, 4)),     # 124M attention-projection weight gradient
    ((3072, 768, 16384), (256, 2)),    # 124M MLP weight gradients
    ((768, 3072, 16384), (256, 2)),
    ((16384, 3072, 768), (256, 1)),    # 124M MLP input projection, forward
    ((16384, 768, 50304), (256, 1)),   # 124M LM-head input gradient
]


@pytest.mark.parametrize("mnk,plan", PLAN_CASES)
def test_bf16_matmul_plans_of_the_gpt2_products(mnk, plan):
    assert g.plan_bf16_matmul(*mnk) == plan


@pytest.mark.parametrize("mnk", [c[0] for c in PLAN_CASES] + [(256, 768, 768), (300, 96, 260), (128, 64, 64)])
def test_bf16_matmul_plan_invariants(mnk):
    M, N, K = mnk
    bn, s = g.plan_bf16_matmul(M, N, K)
    assert bn in (128, 192, 256) and s >= 1
    kt = -(-K // 64)
    if s > 1:
        # only grids below one wave are split, at least four K tiles a split,
        # the fp32 partials within the 8M-float workspace
        assert -(-M // 128) * -(-N // bn) < 148
        assert kt // s >= 4 or -(-kt // s) >= 4
        assert s * M * N <= 8 << 20
    # epilogues that take column sums are never split; the LM head's
    # row-statistics epilogue is never split and never 192 wide
    assert g.plan_bf16_matmul(M, N, K, no_split=True)[1] == 1
    bn_l, s_l = g.plan_bf16_matmul(M, N, K, logits=True)
    assert s_l == 1 and bn_l in (128, 256)


def test_bf16_matmul_plan_rejects_bad_arguments():
    for args in [(0, 768, 768), (256, 0, 768), (256, 768, -1)]:
        with pytest.raises(g.GPT2Error):
            g.plan_bf16_matmul(*args)
    with pytest.raises(g.GPT2Error):
        g.plan_bf16_matmul(256, 768, 768, num_sms=0)
