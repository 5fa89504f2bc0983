"""The device-side timeout path, made to run without a fault or a hang.

Every tensor-core kernel bounds its pipeline waits (mbarrier phases of TMA
copies and MMAs): past the limit it records a timeout in the error word,
stops issuing work, lets the copies and MMAs it already issued land (those
drain waits keep the full 1 s), frees its tensor memory and returns, and
every CTA of a split-K cluster still reaches both cluster barriers.  The
tests lower the limit to 1 ns through ``gpt2_set_wait_limit_ns`` -- below
1 us every wait gives up at its first call -- and check that:

* the per-layer calls (a split-K 3xTF32 matmul, the fp32 tensor-core
  attention) return GPT2_ERR_DEVICE_TIMEOUT;
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
