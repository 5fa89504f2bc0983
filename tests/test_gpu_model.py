"""GPU parity of the whole training step against the CPU oracle, through the
C ABI.  Tolerances (fp32): loss 1e-5 relative, logits max-abs 1e-4, each of
the 16 gradient tensors relative L2 1e-3, fixed-batch AdamW trajectory within
1e-4 per step.  bf16 matmul operands: loss within 2e-2, trajectory within 2%.
Inputs come from ``synth`` only; expected values from ``oracle/`` only."""
import json
import math
import os

import numpy as np
import pytest

import synth
from oracle import ref

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
TINY = synth.WORKLOADS["tiny_L2_C64"]
G124 = synth.WORKLOADS["gpt2_124m_B4_T64_fp32"]


def gpu_model(w, **kw):
    import torch
    import gpt_train_step_02_b300 as g

    assert torch.cuda.is_available()
    return g.GPT2(w, **kw)


def oracle_model(w, params, B=None, T=None):
    m = ref.RefModel(ref.config_from(w), B or w.B, T or w.T, np.float32)
    m.set_params(params)
    return m


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    nb = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (nb if nb > 0 else 1.0)


def check_grads(w, gg, go, tol=1e-3):
    worst = {}
    for name, (o, n) in synth.param_offsets(w).items():
        e = rel_l2(gg[o:o + n], go[o:o + n])
        worst[name] = e
        assert e <= tol, (name, e)
    return worst


def perturbed(w, seed=5):
    """Init plus seeded noise on biases and layernorm terms (generic grads)."""
    p = synth.init_params(w)
    rng = np.random.default_rng(seed)
    for name, (o, n) in synth.param_offsets(w).items():
        if name in ("ln1w", "ln2w", "lnfw"):
            p[o:o + n] += (0.1 * rng.standard_normal(n)).astype(np.float32)
        elif name in ("ln1b", "ln2b", "lnfb", "qkvb", "attprojb", "fcb", "fcprojb"):
            p[o:o + n] = (0.02 * rng.standard_normal(n)).astype(np.float32)
    return p


# ---------------------------------------------------------------------------
def test_init_matches_input_generator():
    for w in (TINY, G124):
        m = gpu_model(w, seed=synth.INIT_SEED)
        pg = m.get_params()
        ps = synth.init_params(w)
        m.close()
        # both sides evaluate Box-Muller in float64 and round once to fp32
        ulp = np.abs(pg.view(np.int32).astype(np.int64) - ps.view(np.int32).astype(np.int64))
        assert ulp.max() <= 1, ulp.max()
        assert (ulp > 0).mean() < 1e-5


@pytest.mark.parametrize("B,T", [(2, 32), (1, 13), (2, 7), (1, 1)])
def test_tiny_forward_backward_parity(B, T):
    w = TINY
    p0 = perturbed(w)
    inp, tgt = synth.batch(w, B=B, T=T)
    m = gpu_model(w, maxB=2, maxT=32)
    m.set_params(p0)
    o = oracle_model(w, p0, 2, 32)
    lg = m.forward(inp, tgt)
    lo = o.forward(inp, tgt)
    assert abs(lg - lo) <= 1e-5 * abs(lo), (lg, lo)
    logits = m.get_logits(B, T)
    lo_logits = o.act("logits").reshape(B, T, -1)
    assert np.abs(logits - lo_logits).max() <= 1e-4
    m.zero_grad()
    m.backward()
    o.zero_grad()
    o.backward()
    check_grads(w, m.get_grads(), o.grads)
    m.close()
    o.close()


def test_tiny_trajectory_10_steps():
    w = TINY
    p0 = synth.init_params(w)
    inp, tgt = synth.batch(w)
    m = gpu_model(w)
    m.set_params(p0)
    o = oracle_model(w, p0)
    lg = [m.step(inp, tgt, t) for t in range(1, w.steps + 1)]
    lo = [o.step(inp, tgt, t) for t in range(1, w.steps + 1)]
    np.testing.assert_allclose(lg, lo, atol=1e-4, rtol=0)
    assert all(b < a for a, b in zip(lg, lg[1:]))
    gold = json.load(open(os.path.join(HERE, "golden", "oracle_traj_tiny_L2_C64.json")))["losses"]
    np.testing.assert_allclose(lg, gold, atol=1e-4, rtol=0)
    m.close()


def test_forward_without_targets_and_state_errors():
    import gpt_train_step_02_b300 as g

    w = TINY
    p0 = perturbed(w)
    inp, _ = synth.batch(w)
    m = gpu_model(w)
    m.set_params(p0)
    with pytest.raises(g.GPT2Error) as e:
        m.backward()  # nothing forwarded yet
    assert e.value.status == g.GPT2_ERR_STATE
    assert m.forward(inp, None) == -1.0
    o = oracle_model(w, p0)
    o.forward(inp, None)
    assert np.abs(m.get_logits(w.B, w.T) - o.act("logits").reshape(w.B, w.T, -1)).max() <= 1e-4
    with pytest.raises(g.GPT2Error) as e:
        m.backward()
    assert e.value.status == g.GPT2_ERR_STATE
    m.close()


def test_token_range_errors_host_and_device():
    import torch
    import gpt_train_step_02_b300 as g

    w = TINY
    m = gpu_model(w)
    inp, tgt = synth.batch(w)
    bad = inp.copy()
    bad[1, 3] = w.vocab_size
    with pytest.raises(g.GPT2Error) as e:
        m.forward(bad, tgt)
    assert e.value.status == g.GPT2_ERR_TOKEN_RANGE
    badt = tgt.copy()
    badt[0, 0] = -1
    with pytest.raises(g.GPT2Error) as e:
        m.forward(inp, badt)
    assert e.value.status == g.GPT2_ERR_TOKEN_RANGE
    # device path: detected on the device, reported at the next sync
    m.forward_device(torch.tensor(bad, device="cuda"), torch.tensor(tgt, device="cuda"))
    with pytest.raises(g.GPT2Error) as e:
        m.sync()
    assert e.value.status == g.GPT2_ERR_TOKEN_RANGE
    # the handle stays usable
    l1 = m.forward(inp, tgt)
    m.forward_device(torch.tensor(inp, device="cuda"), torch.tensor(tgt, device="cuda"))
    assert m.sync() == l1
    # shape errors
    with pytest.raises(g.GPT2Error) as e:
        m.forward(np.zeros((3, 4), np.int32), None)
    assert e.value.status == g.GPT2_ERR_SHAPE
    m.close()


def test_backward_accumulates_and_runs_are_bitwise_deterministic():
    w = TINY
    p0 = perturbed(w)
    inp, tgt = synth.batch(w)
    grads = []
    for _ in range(2):
        m = gpu_model(w)
        m.set_params(p0)
        m.forward(inp, tgt)
        m.zero_grad()
        m.backward()
        g1 = m.get_grads()
        m.backward()
        g2 = m.get_grads()
        m.close()
        grads.append((g1, g2))
    assert np.array_equal(grads[0][0], grads[1][0])
    assert np.array_equal(grads[0][1], grads[1][1])
    g1, g2 = grads[0]
    for name, (o, n) in synth.param_offsets(w).items():
        if name == "wte":
            np.testing.assert_allclose(g2[o:o + n], 2 * g1[o:o + n], rtol=1e-5, atol=1e-9)
        else:
            assert np.array_equal(g2[o:o + n], 2 * g1[o:o + n]), name


def test_device_step_matches_host_calls():
    import torch

    w = TINY
    p0 = synth.init_params(w)
    inp, tgt = synth.batch(w)
    a = gpu_model(w)
    b = gpu_model(w)
    a.set_params(p0)
    b.set_params(p0)
    di, dt = torch.tensor(inp, device="cuda"), torch.tensor(tgt, device="cuda")
    for t in range(1, 4):
        la = a.step(inp, tgt, t)
        b.train_step_device(di, dt, t)
        lb = b.sync()
        assert la == lb
    assert np.array_equal(a.get_params(), b.get_params())
    ma, va = a.get_opt_state()
    mb, vb = b.get_opt_state()
    assert np.array_equal(ma, mb) and np.array_equal(va, vb)
    a.close()
    b.close()


def test_fused_step_gradients_equal_zero_grad_then_backward():
    """The fused step stores each gradient once instead of clearing the
    buffer and accumulating: its gradients must equal zero_grad + backward
    exactly, also when a shorter sequence follows a longer one (the wpe rows
    past T are cleared, not left from the previous step)."""
    import torch

    w = TINY
    p0 = perturbed(w)
    a = gpu_model(w)
    b = gpu_model(w)
    a.set_params(p0)
    b.set_params(p0)
    for t, (B, T) in enumerate([(2, 32), (2, 16), (1, 7)], start=1):
        inp, tgt = synth.batch(w, B=B, T=T)
        la = a.step(inp, tgt, t)
        b.train_step_device(torch.tensor(inp, device="cuda"), torch.tensor(tgt, device="cuda"), t)
        lb = b.sync()
        assert la == lb, (t, la, lb)
        assert np.array_equal(a.get_grads(), b.get_grads()), t
        assert np.array_equal(a.get_params(), b.get_params()), t
    a.close()
    b.close()


def test_checkpoint_resume_is_bitwise():
    w = TINY
    p0 = synth.init_params(w)
    inp, tgt = synth.batch(w)
    a = gpu_model(w)
    a.set_params(p0)
    for t in range(1, 11):
        a.step(inp, tgt, t)
    b = gpu_model(w)
    b.set_params(p0)
    for t in range(1, 6):
        b.step(inp, tgt, t)
    p5 = b.get_params()
    m5, v5 = b.get_opt_state()
    b.close()
    c = gpu_model(w, seed=999)
    c.set_params(p5)
    c.set_opt_state(m5, v5)
    for t in range(6, 11):
        c.step(inp, tgt, t)
    assert np.array_equal(a.get_params(), c.get_params())
    a.close()
    c.close()


def test_bf16_operands_tiny():
    w = synth.Workload("tiny_bf16", 2, 64, 4, 512, 512, 32, 2, 32, "bf16", "uniform", 10)
    p0 = synth.init_params(w)
    inp, tgt = synth.batch(w)
    m = gpu_model(w)
    m.set_params(p0)
    o = oracle_model(w, p0)
    lg = [m.step(inp, tgt, t) for t in range(1, 11)]
    lo = [o.step(inp, tgt, t) for t in range(1, 11)]
    assert abs(lg[0] - lo[0]) <= 2e-2
    np.testing.assert_allclose(lg, lo, rtol=0.02)
    m.close()


def test_bf16_tensor_core_attention_small():
    """bf16 workload whose attention takes the tensor-core kernels (head
    size 64, T a multiple of 128): the 10-step fixed-batch trajectory stays
    within 2% per step of the fp32 oracle, as the bf16 bar requires."""
    w = synth.Workload("small_bf16_hs64", 2, 128, 2, 512, 512, 256, 2, 256, "bf16", "uniform", 10)
    p0 = synth.init_params(w)
    inp, tgt = synth.batch(w)
    m = gpu_model(w)
    m.set_params(p0)
    o = oracle_model(w, p0)
    lg = [m.step(inp, tgt, t) for t in range(1, 11)]
    lo = [o.step(inp, tgt, t) for t in range(1, 11)]
    assert abs(lg[0] - lo[0]) <= 2e-2
    np.testing.assert_allclose(lg, lo, rtol=0.02)
    assert all(b < a for a, b in zip(lg, lg[1:]))
    m.close()


def test_bf16_tensor_core_gradients():
    """Every parameter gradient of one bf16 step on a workload that takes the
    tensor-core attention (head size 64, T % 128 == 0), whose MLP input and
    QKV bias gradients come from column sums taken in the matmul and
    attention epilogues, against the fp32 oracle.  bf16 operand rounding
    (u = 2^-9) through a few chained products gives about 1e-2 relative L2
    per tensor; the bar is 3e-2."""
    w = synth.Workload("grad_bf16_hs64", 2, 128, 2, 512, 512, 256, 2, 256, "bf16", "uniform", 1)
    p0 = perturbed(w)
    inp, tgt = synth.batch(w)
    m = gpu_model(w)
    m.set_params(p0)
    o = oracle_model(w, p0)
    lg = m.forward(inp, tgt)
    lo = o.forward(inp, tgt)
    assert abs(lg - lo) <= 2e-2, (lg, lo)
    m.zero_grad()
    m.backward()
    o.zero_grad()
    o.backward()
    worst = check_grads(w, m.get_grads(), o.grads, tol=3e-2)
    assert max(worst.values()) > 0.0  # bf16 rounding is visible, so the bf16 path really ran
    m.close()
    o.close()


@pytest.mark.parametrize("tokens", ["uniform", "zipf"])
def test_embedding_backward_beyond_the_single_cta_sort(tokens):
    """B*T = 20480 tokens, more than the single-CTA bitonic sort holds: the
    embedding backward sorts positions with the two-pass radix sort.  Loss and
    every gradient tensor against the oracle (fp32 bars), and two backward
    passes bitwise equal (the sort's ranks and the per-id sums have a fixed
    order).  With Zipf(1.1) ids, id 0 takes about a fifth of the positions."""
    w = synth.Workload(f"tiny_B640_{tokens}", 2, 64, 4, 512, 512, 32, 640, 32, "fp32", tokens, 1)
    p0 = perturbed(w)
    inp, tgt = synth.batch(w)
    m = gpu_model(w)
    m.set_params(p0)
    lg = m.forward(inp, tgt)
    m.zero_grad()
    m.backward()
    g1 = m.get_grads()
    m.zero_grad()
    m.backward()
    g2 = m.get_grads()
    m.close()
    assert np.array_equal(g1, g2)
    o = oracle_model(w, p0)
    lo = o.forward(inp, tgt)
    o.zero_grad()
    o.backward()
    go = o.grads.copy()
    o.close()
    assert abs(lg - lo) <= 1e-5 * abs(lo), (lg, lo)
    check_grads(w, g1, go)


def bf16_round(a):
    """Round to the nearest bf16 (ties to even), returned as float32."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


@pytest.mark.parametrize("V,Vp,T,tokens", [(500, 512, 64, "uniform"), (50257, 50304, 128, "zipf")])
def test_bf16_logits_row_statistics_and_loss(V, Vp, T, tokens):
    """bf16 forward with targets: the LM-head matmul stores the logits in bf16
    and the rows' softmax statistics and the targets' logits in fp32; the
    cross-entropy merges the statistics.  The stored logits must be exactly
    the bf16 rounding of the same matmul's fp32 logits (a forward without
    targets), and the loss must equal the softmax cross-entropy of those fp32
    logits over the V real columns, evaluated here in float64 (the
    statistics are exact up to fp32 rounding).  The two vocabularies take
    128- and 256-column tiles (64- and 128-column statistic blocks), with
    padded columns in the last tile."""
    w = synth.Workload(f"xent_bf16_V{V}", 1, 64, 4, V, Vp, T, 2, T, "bf16", tokens, 1)
    p0 = perturbed(w)
    inp, tgt = synth.batch(w)
    m = gpu_model(w)
    m.set_params(p0)
    assert m.forward(inp, None) == -1.0
    l32 = m.get_logits(w.B, w.T).astype(np.float32)
    loss = m.forward(inp, tgt)
    l16 = m.get_logits(w.B, w.T)
    m.close()
    assert np.array_equal(l16, bf16_round(l32))
    x = l32.reshape(-1, Vp)[:, :V].astype(np.float64)
    mx = x.max(axis=1, keepdims=True)
    lse = mx[:, 0] + np.log(np.exp(x - mx).sum(axis=1))
    ref_loss = float(np.mean(lse - x[np.arange(x.shape[0]), tgt.reshape(-1)]))
    assert abs(loss - ref_loss) <= 2e-6 * abs(ref_loss), (loss, ref_loss)


# ---------------------------------------------------------------------------
# GPT-2 124M, fp32, B=4, T=64 (the workload of the pages' console log)
# ---------------------------------------------------------------------------
@pytest.fixture(scope="module")
def g124_step():
    w = G124
    p0 = synth.init_params(w)
    inp, tgt = synth.batch(w)
    o = oracle_model(w, p0)
    lo = o.forward(inp, tgt)
    logits_o = o.act("logits").reshape(w.B, w.T, -1).copy()
    o.zero_grad()
    o.backward()
    go = o.grads.copy()
    o.close()
    return p0, inp, tgt, lo, logits_o, go


def test_124m_forward_backward_parity(g124_step):
    w = G124
    p0, inp, tgt, lo, logits_o, go = g124_step
    m = gpu_model(w)
    m.set_params(p0)
    lg = m.forward(inp, tgt)
    assert abs(lg - lo) <= 1e-5 * abs(lo), (lg, lo)
    assert abs(lo - math.log(50257)) < 0.5
    logits = m.get_logits(w.B, w.T)
    assert np.abs(logits - logits_o).max() <= 1e-4
    assert np.all(logits[..., w.vocab_size:] == 0.0)  # padded wte rows are zero
    m.zero_grad()
    m.backward()
    worst = check_grads(w, m.get_grads(), go)
    print("124M grad rel-L2:", {k: f"{v:.2e}" for k, v in worst.items()})
    m.close()


def test_124m_trajectory_10_steps():
    w = G124
    gold = json.load(open(os.path.join(HERE, "golden", f"oracle_traj_{w.name}.json")))["losses"]
    p0 = synth.init_params(w)
    inp, tgt = synth.batch(w)
    m = gpu_model(w)
    m.set_params(p0)
    lg = [m.step(inp, tgt, t) for t in range(1, w.steps + 1)]
    print("124M trajectory gpu:", lg)
    np.testing.assert_allclose(lg, gold, atol=1e-4, rtol=0)
    m.close()
