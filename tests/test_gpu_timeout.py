"""The device-side timeout path, made to run without a fault or a hang.

Every tensor-core kernel bounds its pipeline waits (mbarrier phases of TMA
copies and MMAs): past the limit it records a timeout in the error word,
stops issuing work, lets the copies and MMAs it already issued land (those
drain waits keep the full 1 s), frees its tensor memory and returns, and
every CTA of a split-K cluster still reaches both cluster barriers.  The
tests lower the limit to 1 ns through ``gpt2_set_wait_limit_ns`` -- below
1 us every wait gives up at its first call -- and check that:

* the per-layer calls (a split-K 3xTF32 matmul, the fp32 tensor-core
  attention, the persistent bf16 tensor-core attention forward and
  backward) return GPT2_ERR_DEVICE_TIMEOUT;
* a model step reports GPT2_ERR_DEVICE_TIMEOUT at its synchronisation, the
  handle is poisoned (every later call returns the same status);
* with the default limit restored, the context is still usable: the same
  calls and a fresh handle match the oracle again.
Expected values come from ``oracle/`` only; inputs from ``synth``."""
import numpy as np
import pytest

import synth
from oracle import ref

pytestmark = pytest.mark.gpu

OPS = ref.ops(np.float32)


@pytest.fixture()
def short_waits():
    import gpt_train_step_02_b300 as g

    g.set_wait_limit_ns(1)
    try:
        yield g
    finally:
        g.set_wait_limit_ns(0)  # back to the 1 s default, whatever happened


def bf16(a):
    """Round to the nearest bf16 (ties to even), returned as float32."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return np.linalg.norm(a - b) / np.linalg.norm(b)


def rel_err(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return np.abs(a - b).max() / max(np.abs(b).max(), 1e-30)


def test_split_k_matmul_times_out_then_recovers(short_waits):
    import torch

    g = short_waits
    N, IC, OC = 256, 768, 768  # 12 output tiles, K split over clusters of 8 CTAs
    x = synth.randn(501, (N, IC))
    W = synth.randn(502, (OC, IC), 0.02)
    tx, tW = torch.tensor(x, device="cuda"), torch.tensor(W, device="cuda")
    out = torch.zeros((N, OC), device="cuda")
    with pytest.raises(g.GPT2Error) as e:
        g.matmul_forward(out, tx, tW, None)
    assert e.value.status == g.GPT2_ERR_DEVICE_TIMEOUT
    g.set_wait_limit_ns(0)
    g.matmul_forward(out, tx, tW, None)
    assert rel_err(out.cpu().numpy(), OPS.matmul_forward(x, W, None)) < 1e-5


def test_fp32_tensor_core_attention_times_out_then_recovers(short_waits):
    import torch

    g = short_waits
    B, T, C, NH = 2, 64, 128, 2  # head size 64, T <= 64: the 3xTF32 tcgen05 attention
    qkv = synth.randn(503, (B, T, 3 * C))
    y = torch.zeros((B, T, C), device="cuda")
    lse = torch.zeros((B, NH, T), device="cuda")
    tq = torch.tensor(qkv, device="cuda")
    with pytest.raises(g.GPT2Error) as e:
        g.attention_forward(y, lse, tq, NH)
    assert e.value.status == g.GPT2_ERR_DEVICE_TIMEOUT
    g.set_wait_limit_ns(0)
    g.attention_forward(y, lse, tq, NH)
    ry, _, _ = OPS.attention_forward(qkv, NH)
    assert np.abs(y.cpu().numpy() - ry).max() <= 1e-5 * max(np.abs(ry).max(), 1.0)


def test_bf16_tensor_core_attention_times_out_then_recovers(short_waits):
    """The persistent tensor-core attention kernels (bf16 operands, head size
    64, T % 128 == 0): the forward, the dK/dV and the dQ kernel all give up,
    each of their threads drains what it issued, and the same call then
    matches the oracle fed the bf16-rounded inputs (bars of the attention
    backward parity test: 1e-2 relative L2 per block, 3e-2 entrywise)."""
    import torch

    g = short_waits
    B, T, C, NH = 2, 256, 128, 2
    qkv = synth.randn(505, (B, T, 3 * C))
    dy = synth.randn(506, (B, T, C))
    tq, td = torch.tensor(qkv, device="cuda"), torch.tensor(dy, device="cuda")
    dqkv = torch.zeros_like(tq)
    with pytest.raises(g.GPT2Error) as e:
        g.attention_backward(dqkv, td, tq, NH, precision=g.GPT2_PREC_BF16)
    assert e.value.status == g.GPT2_ERR_DEVICE_TIMEOUT
    g.set_wait_limit_ns(0)
    g.attention_backward(dqkv, td, tq, NH, precision=g.GPT2_PREC_BF16)
    got = dqkv.cpu().numpy()
    q, d = bf16(qkv), bf16(dy)
    _, _, att = OPS.attention_forward(q, NH)
    ref_d = OPS.attention_backward(d, q, att, NH)
    for part in range(3):
        gp, rp = got[..., part * C:(part + 1) * C], ref_d[..., part * C:(part + 1) * C]
        assert rel_l2(gp, rp) <= 1e-2, (part, rel_l2(gp, rp))
        assert np.abs(gp - rp).max() <= 3e-2 * np.abs(rp).max(), part


def test_model_step_timeout_poisons_the_handle(short_waits):
    g = short_waits
    # GPT-2 124M's layer shapes at one layer: split-K products, the fp32
    # tensor-core attention (head size 64, T = 64)
    w = synth.Workload("timeout_L1_C768", 1, 768, 12, 512, 512, 64, 2, 64, "fp32", "uniform", 1)
    p0 = synth.init_params(w)
    inp, tgt = synth.batch(w)
    m = g.GPT2(w)
    m.set_params(p0)
    with pytest.raises(g.GPT2Error) as e:
        m.step(inp, tgt, 1)
    assert e.value.status == g.GPT2_ERR_DEVICE_TIMEOUT
    g.set_wait_limit_ns(0)
    # poisoned: every later call on this handle reports the same error
    for call in (lambda: m.forward(inp, tgt), m.zero_grad, m.backward, m.get_params):
        with pytest.raises(g.GPT2Error) as e:
            call()
        assert e.value.status == g.GPT2_ERR_DEVICE_TIMEOUT
    m.close()
    # a fresh handle on the same device works and matches the oracle
    m2 = g.GPT2(w)
    m2.set_params(p0)
    loss = m2.forward(inp, tgt)
    m2.close()
    o = ref.RefModel(ref.config_from(w), w.B, w.T, np.float32)
    o.set_params(p0)
    lo = o.forward(inp, tgt)
    o.close()
    assert abs(loss - lo) <= 1e-5 * abs(lo), (loss, lo)
