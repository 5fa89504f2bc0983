"""GPU parity of the Llama-style variant (config field ``llama``: RMSNorm in
place of layernorm, rotary position embedding of q and k, no position table,
no linear biases -- the architectures the page «千行C代码训完GPT-2» (新智元)
names as llm.c's next step) against the oracle's same variant, through the C
ABI.  Bars as for GPT-2: fp32 loss 1e-5 relative, logits 1e-4, each gradient
tensor 1e-3 relative L2, fixed-batch trajectory 1e-4 per step; bf16 operands
(tensor-core attention, rotary embedding applied to the bf16 copies too) loss
within 2e-2 and each gradient tensor within 3e-2 relative L2 (bf16 rounding,
u = 2^-9, through a few chained products gives about 1e-2).
Inputs come from ``synth``; expected values from ``oracle/`` only."""
import numpy as np
import pytest

import synth
from oracle import ref

pytestmark = pytest.mark.gpu

TINY_LL = synth.Workload("tiny_llama", 2, 64, 4, 512, 512, 32, 2, 32, "fp32", "uniform", 10, llama=1)
BF16_LL = synth.Workload("llama_bf16_hs64", 2, 128, 2, 512, 512, 256, 2, 256, "bf16", "uniform", 1, llama=1)


def gpu_model(w, **kw):
    import gpt_train_step_02_b300 as g

    return g.GPT2(w, **kw)


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    nb = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (nb if nb > 0 else 1.0)


def perturbed(w, seed=5):
    """Init plus seeded noise on the RMSNorm gains, so every gradient is generic."""
    p = synth.init_params(w)
    rng = np.random.default_rng(seed)
    for name, (o, n) in synth.param_offsets(w).items():
        if name in ("ln1w", "ln2w", "lnfw"):
            p[o:o + n] += (0.1 * rng.standard_normal(n)).astype(np.float32)
    return p


def check_grads(w, gg, go, tol):
    worst = {}
    for name, (o, n) in synth.param_offsets(w).items():
        if n == 0:
            continue
        e = rel_l2(gg[o:o + n], go[o:o + n])
        worst[name] = e
        assert e <= tol, (name, e)
    return worst


def test_llama_layout_and_init():
    w = TINY_LL
    m = gpu_model(w, seed=synth.INIT_SEED)
    assert m.get_params().size == synth.num_params(w) == ref.num_parameters(ref.config_from(w))
    pg = m.get_params()
    m.close()
    ps = synth.init_params(w)
    ulp = np.abs(pg.view(np.int32).astype(np.int64) - ps.view(np.int32).astype(np.int64))
    assert ulp.max() <= 1


@pytest.mark.parametrize("B,T", [(2, 32), (1, 7)])
def test_llama_tiny_forward_backward_parity(B, T):
    w = TINY_LL
    p0 = perturbed(w)
    inp, tgt = synth.batch(w, B=B, T=T)
    m = gpu_model(w, maxB=2, maxT=32)
    m.set_params(p0)
    o = ref.RefModel(ref.config_from(w), 2, 32, np.float32)
    o.set_params(p0)
    lg = m.forward(inp, tgt)
    lo = o.forward(inp, tgt)
    assert abs(lg - lo) <= 1e-5 * abs(lo), (lg, lo)
    np.testing.assert_allclose(m.get_logits(B, T), o.act("logits").reshape(B, T, -1), rtol=0, atol=1e-4)
    m.zero_grad()
    m.backward()
    o.zero_grad()
    o.backward()
    check_grads(w, m.get_grads(), o.grads, 1e-3)
    m.close()
    o.close()


def test_llama_tiny_trajectory():
    w = TINY_LL
    p0 = synth.init_params(w)
    inp, tgt = synth.batch(w)
    m = gpu_model(w)
    m.set_params(p0)
    o = ref.RefModel(ref.config_from(w), w.B, w.T, np.float32)
    o.set_params(p0)
    lg = [m.step(inp, tgt, t) for t in range(1, 11)]
    lo = [o.step(inp, tgt, t) for t in range(1, 11)]
    np.testing.assert_allclose(lg, lo, atol=1e-4, rtol=0)
    assert all(b < a for a, b in zip(lo, lo[1:]))
    m.close()
    o.close()


def test_llama_bf16_tensor_core_gradients():
    w = BF16_LL
    p0 = perturbed(w)
    inp, tgt = synth.batch(w)
    m = gpu_model(w)
    m.set_params(p0)
    o = ref.RefModel(ref.config_from(w), w.B, w.T, np.float32)
    o.set_params(p0)
    lg = m.forward(inp, tgt)
    lo = o.forward(inp, tgt)
    assert abs(lg - lo) <= 2e-2, (lg, lo)
    m.zero_grad()
    m.backward()
    o.zero_grad()
    o.backward()
    worst = check_grads(w, m.get_grads(), o.grads, 3e-2)
    assert max(worst.values()) > 0.0
    m.close()
    o.close()


def test_llama_generation_valid_under_the_oracle():
    w = TINY_LL
    p0 = synth.init_params(w)
    coins = np.random.default_rng(21).random(20).astype(np.float32) * np.float32(0.999)
    m = gpu_model(w, maxB=1, maxT=24)
    m.set_params(p0)
    toks = m.sample([7, 3, 9, 1], 24, coins)
    m.close()
    o = ref.RefModel(ref.config_from(w), 1, 24, np.float32)
    o.set_params(p0)
    for t in range(4, 24):
        o.forward(toks[None, :], None)
        probs = ref.softmax64(o.act("logits").reshape(24, -1)[t - 1, :w.vocab_size])
        assert ref.sample_is_valid(probs, float(coins[t - 4]), int(toks[t]), 1e-5), t
    o.close()
