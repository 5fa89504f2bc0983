"""Per-layer parity of the causal attention forward against the oracle's
attention_forward (the page «llm.c：Andrej Karpathy带你从零复现LLM», section
«核心代码解读：train_gpt2.c», item 1), through the C ABI.

* fp32: the CUDA-core kernels, against the fp32 oracle, 1e-5 relative: the
  streaming ones, and for head size 64 with T <= 64 the one-CTA-per-head ones
  (register-tiled products, causal blocks skipped, one backward launch).
* bf16 with head size 64 and T % 128 == 0: the tensor-core kernel, against
  the oracle fed the same bf16-rounded qkv.  The kernel also rounds the
  softmax weights P to bf16 for the P V product (relative 2^-9 each) while
  the row sums take the fp32 weights, so y is a combination of the v rows
  with weights off by at most 2^-9 relative.  Tolerance: max |dy| <= 1e-2
  max |v|, |d lse| <= 1e-2.
* bf16 with another head size, or T <= 64: the CUDA-core kernels with
  rounded operands.
Inputs come from ``synth``; expected values from ``oracle/`` only."""
import numpy as np
import pytest

import synth
from oracle import ref

pytestmark = pytest.mark.gpu

OPS = ref.ops(np.float32)


def bf16(a):
    """Round to the nearest bf16 (ties to even), returned as float32."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def oracle_lse(preatt):
    """Row log-sum-exp of the scaled scores over the causal keys t2 <= t."""
    B, NH, T, _ = preatt.shape
    s = preatt.astype(np.float64)
    mask = np.tril(np.ones((T, T), bool))
    s = np.where(mask, s, -np.inf)
    mx = s.max(-1, keepdims=True)
    return (mx[..., 0] + np.log(np.exp(s - mx).sum(-1))).astype(np.float32)


def run_gpu(qkv, NH, precision):
    import torch
    import gpt_train_step_02_b300 as g

    B, T, C3 = qkv.shape
    C = C3 // 3
    y = torch.full((B, T, C), float("nan"), device="cuda")
    lse = torch.full((B, NH, T), float("nan"), device="cuda")
    g.attention_forward(y, lse, torch.tensor(qkv, device="cuda"), NH, precision=precision)
    return y.cpu().numpy(), lse.cpu().numpy()


# CUDA-core shapes: several 64-row chunks with a ragged tail (T = 200), head
# sizes 16, 64 and 128, a single position, a partial 8-row CTA (T = 13); the
# short-sequence kernels (head size 64, T <= 64) at the GPT-2 124M shape of
# the B=4, T=64 step, with ragged T (37, 61: partial 4-row blocks) and T = 1
FP32_SHAPES = [(2, 32, 64, 4), (1, 13, 64, 4), (2, 64, 768, 12), (1, 1, 64, 4), (1, 200, 128, 2), (1, 70, 256, 2),
               (4, 64, 768, 12), (2, 37, 128, 2), (3, 61, 192, 3), (1, 1, 128, 2)]


@pytest.mark.parametrize("B,T,C,NH", FP32_SHAPES)
def test_attention_forward_fp32(B, T, C, NH):
    import gpt_train_step_02_b300 as g

    qkv = synth.randn(301, (B, T, 3 * C))
    y, lse = run_gpu(qkv, NH, g.GPT2_PREC_FP32)
    ry, preatt, _ = OPS.attention_forward(qkv, NH)
    assert np.abs(y - ry).max() <= 1e-5 * max(np.abs(ry).max(), 1.0)
    assert np.abs(lse - oracle_lse(preatt)).max() <= 1e-4


# (16, 256, 768, 12) has 384 (query tile, head, batch) items: more than the
# persistent forward's 296 CTAs, so some CTAs run two items
@pytest.mark.parametrize("B,T,C,NH", [(2, 128, 128, 2), (1, 256, 64, 1), (2, 384, 128, 2), (1, 1024, 768, 12),
                                      (16, 256, 768, 12)])
def test_attention_forward_bf16_tensor_cores(B, T, C, NH):
    import gpt_train_step_02_b300 as g

    qkv = synth.randn(302, (B, T, 3 * C))
    y, lse = run_gpu(qkv, NH, g.GPT2_PREC_BF16)
    q = bf16(qkv)
    ry, preatt, _ = OPS.attention_forward(q, NH)
    vmax = np.abs(q[..., 2 * C:]).max()
    assert np.isfinite(y).all() and np.isfinite(lse).all()
    assert np.abs(y - ry).max() <= 1e-2 * vmax, np.abs(y - ry).max()
    assert np.abs(lse - oracle_lse(preatt)).max() <= 1e-2
    # the first query row attends to itself only: y = its own v exactly
    hs = C // NH
    np.testing.assert_allclose(y[:, 0, :], q[:, 0, 2 * C:], rtol=0, atol=0)
    del hs


def test_attention_forward_bf16_other_head_size():
    import gpt_train_step_02_b300 as g

    B, T, C, NH = 2, 32, 64, 4  # hs = 16: the CUDA-core kernel with bf16 operands
    qkv = synth.randn(303, (B, T, 3 * C))
    y, lse = run_gpu(qkv, NH, g.GPT2_PREC_BF16)
    ry, preatt, _ = OPS.attention_forward(bf16(qkv), NH)
    assert np.abs(y - ry).max() <= 1e-2 * np.abs(ry).max()
    assert np.abs(lse - oracle_lse(preatt)).max() <= 1e-3


@pytest.mark.parametrize("B,T,C,NH", [(2, 48, 128, 2), (1, 64, 768, 12)])
def test_attention_forward_bf16_short_sequences(B, T, C, NH):
    """Head size 64, T <= 64: the one-CTA-per-head kernel with operands and
    the P entering P V rounded to bf16, against the oracle fed the rounded qkv."""
    import gpt_train_step_02_b300 as g

    qkv = synth.randn(304, (B, T, 3 * C))
    y, lse = run_gpu(qkv, NH, g.GPT2_PREC_BF16)
    q = bf16(qkv)
    ry, preatt, _ = OPS.attention_forward(q, NH)
    assert np.abs(y - ry).max() <= 1e-2 * np.abs(ry).max()
    assert np.abs(lse - oracle_lse(preatt)).max() <= 1e-3
    np.testing.assert_allclose(y[:, 0, :], q[:, 0, 2 * C:], rtol=0, atol=0)


def run_gpu_backward(qkv, dy, NH, precision):
    import torch
    import gpt_train_step_02_b300 as g

    dqkv = torch.full(qkv.shape, float("nan"), device="cuda")
    g.attention_backward(dqkv, torch.tensor(dy, device="cuda"), torch.tensor(qkv, device="cuda"), NH,
                         precision=precision)
    return dqkv.cpu().numpy()


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return np.linalg.norm(a - b) / np.linalg.norm(b)


@pytest.mark.parametrize("B,T,C,NH", FP32_SHAPES)
def test_attention_backward_fp32(B, T, C, NH):
    import gpt_train_step_02_b300 as g

    qkv = synth.randn(311, (B, T, 3 * C))
    dy = synth.randn(312, (B, T, C))
    got = run_gpu_backward(qkv, dy, NH, g.GPT2_PREC_FP32)
    _, _, att = OPS.attention_forward(qkv, NH)
    ref_d = OPS.attention_backward(dy, qkv, att, NH)
    assert np.abs(got - ref_d).max() <= 1e-4 * np.abs(ref_d).max()


@pytest.mark.parametrize("B,T,C,NH", [(2, 128, 128, 2), (1, 384, 64, 1), (1, 1024, 768, 12), (16, 256, 768, 12)])
def test_attention_backward_bf16_tensor_cores(B, T, C, NH):
    """Tensor-core dK/dV and dQ kernels against the oracle fed the same
    bf16-rounded qkv and dy.  P and dS are rounded to bf16 for the products
    (relative 2^-9 each), so the bar is 1e-2 relative L2 per q, k, v block and
    3e-2 of the largest gradient entrywise."""
    import gpt_train_step_02_b300 as g

    qkv = synth.randn(313, (B, T, 3 * C))
    dy = synth.randn(314, (B, T, C))
    got = run_gpu_backward(qkv, dy, NH, g.GPT2_PREC_BF16)
    q, d = bf16(qkv), bf16(dy)
    _, _, att = OPS.attention_forward(q, NH)
    ref_d = OPS.attention_backward(d, q, att, NH)
    assert np.isfinite(got).all()
    for part in range(3):  # dq, dk, dv
        gp, rp = got[..., part * C:(part + 1) * C], ref_d[..., part * C:(part + 1) * C]
        assert rel_l2(gp, rp) <= 1e-2, (part, rel_l2(gp, rp))
        assert np.abs(gp - rp).max() <= 3e-2 * np.abs(rp).max(), part
    # the last key of each sequence is seen only by the last query
    last_k = ref_d[:, -1, C:2 * C]
    np.testing.assert_allclose(got[:, -1, C:2 * C], last_k, atol=3e-2 * np.abs(ref_d[..., C:2 * C]).max())


@pytest.mark.parametrize("B,T,C,NH", [(2, 48, 128, 2), (1, 64, 768, 12)])
def test_attention_backward_bf16_short_sequences(B, T, C, NH):
    """Head size 64, T <= 64 with bf16 operands: the one-launch backward with
    q, k, v, dy, P (for dV) and dS rounded to bf16, against the oracle fed the
    rounded qkv and dy; bars as for the tensor-core backward."""
    import gpt_train_step_02_b300 as g

    qkv = synth.randn(315, (B, T, 3 * C))
    dy = synth.randn(316, (B, T, C))
    got = run_gpu_backward(qkv, dy, NH, g.GPT2_PREC_BF16)
    q, d = bf16(qkv), bf16(dy)
    _, _, att = OPS.attention_forward(q, NH)
    ref_d = OPS.attention_backward(d, q, att, NH)
    assert np.isfinite(got).all()
    for part in range(3):
        gp, rp = got[..., part * C:(part + 1) * C], ref_d[..., part * C:(part + 1) * C]
        assert rel_l2(gp, rp) <= 1e-2, (part, rel_l2(gp, rp))
        assert np.abs(gp - rp).max() <= 3e-2 * np.abs(rp).max(), part
