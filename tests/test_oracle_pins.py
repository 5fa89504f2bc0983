"""Pins of the CPU oracle against what the llm.c pages and the mathematics fix.

Each test names the fact it pins (P1..P12).  The oracle is never compared
with itself here: the expected values are printed numbers from the pages
(tests/golden/pages_console_log.json), closed forms, invariants, brute force
or finite differences.
"""
import json
import math
import os
import subprocess
import sys

import numpy as np
import pytest

import synth
from oracle import ref

HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = json.load(open(os.path.join(HERE, "golden", "pages_console_log.json")))

TINY = synth.WORKLOADS["tiny_L2_C64"]
G124 = synth.WORKLOADS["gpt2_124m_B4_T64_fp32"]


def cfg_124m_from_log():
    g = GOLDEN
    return ref.make_config(g["max_seq_len"], g["vocab_size"], 50304, g["num_layers"], g["num_heads"], g["channels"])


# --------------------------------------------------------------------------
# P1-P3: the counts printed in the console log
# --------------------------------------------------------------------------
def test_P1_parameter_count_matches_console_log():
    cfg = cfg_124m_from_log()
    assert ref.num_parameters(cfg, padded=False) == GOLDEN["num_parameters"] == 124439808
    # padded layout: 47 extra zero rows of wte
    assert ref.num_parameters(cfg, padded=True) == 124439808 + (50304 - 50257) * 768
    assert ref.num_parameters(ref.config_from(TINY)) == 134912


def test_P1_layout_agrees_with_input_generator():
    for w in (TINY, G124):
        offs = ref.param_offsets(ref.config_from(w))
        assert offs == synth.param_offsets(w)
        assert ref.num_parameters(ref.config_from(w)) == synth.num_params(w)


def test_P2_activation_count_matches_console_log():
    cfg = cfg_124m_from_log()
    # B*T = 256 (P3) with T = 64; unpadded vocab as printed
    assert ref.num_activations(cfg, 4, 64, padded=False) == GOLDEN["num_activations"] == 73323776


def test_P3_batch_counts_fix_BT_256():
    g = GOLDEN
    cands = [bt for bt in range(1, 4097) if g["train_tokens"] // bt == g["train_num_batches"]
             and g["val_tokens"] // bt == g["val_num_batches"]]
    assert cands == [256]
    assert G124.B * G124.T == 256


# --------------------------------------------------------------------------
# helpers
# --------------------------------------------------------------------------
def perturbed_params(w, seed=7, scale=1.0):
    """Initial params plus seeded noise on biases and layernorm affine terms,
    so that every gradient is generic (not structurally zero)."""
    p = synth.init_params(w).astype(np.float64)
    rng = np.random.default_rng(seed)
    offs = synth.param_offsets(w)
    for name in ("ln1w", "ln2w", "lnfw"):
        o, n = offs[name]
        p[o:o + n] += scale * 0.1 * rng.standard_normal(n)
    for name in ("ln1b", "ln2b", "lnfb", "qkvb", "attprojb", "fcb", "fcprojb"):
        o, n = offs[name]
        p[o:o + n] = scale * 0.02 * rng.standard_normal(n)
    # padded wte rows stay zero
    o, _ = offs["wte"]
    p[o + w.vocab_size * w.channels: o + w.padded_vocab_size * w.channels] = 0.0
    return p


def tiny_model(dtype=np.float64, params=None, maxB=None, maxT=None, w=TINY):
    m = ref.RefModel(ref.config_from(w), maxB or w.B, maxT or w.T, dtype)
    m.set_params(perturbed_params(w) if params is None else params)
    return m


# --------------------------------------------------------------------------
# P4: layernorm moments
# --------------------------------------------------------------------------
def test_P4_layernorm_output_moments():
    ops = ref.ops(np.float64)
    rng = np.random.default_rng(0)
    for sigma in (0.03, 1.0, 10.0):
        x = 0.5 + sigma * rng.standard_normal((37, 96))
        y, mean, rstd = ops.layernorm_forward(x, np.ones(96), np.zeros(96))
        var_in = x.var(axis=1)
        assert np.all(np.abs(y.mean(axis=1)) < 1e-6)
        np.testing.assert_allclose(y.var(axis=1), var_in / (var_in + 1e-5), rtol=1e-10)
        np.testing.assert_allclose(mean, x.mean(axis=1), rtol=1e-12)
        np.testing.assert_allclose(rstd, 1.0 / np.sqrt(var_in + 1e-5), rtol=1e-12)
    # affine: gamma scales, beta shifts
    x = rng.standard_normal((5, 32))
    g, b = rng.standard_normal(32), rng.standard_normal(32)
    y0, _, _ = ops.layernorm_forward(x, np.ones(32), np.zeros(32))
    y1, _, _ = ops.layernorm_forward(x, g, b)
    np.testing.assert_allclose(y1, y0 * g + b, rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------
# P5: attention rows and vocab rows are probability distributions
# --------------------------------------------------------------------------
def test_P5_attention_and_probs_rows_sum_to_one():
    m = tiny_model(np.float64)
    inp, tgt = synth.batch(TINY)
    m.forward(inp, tgt)
    B, T, NH, L = TINY.B, TINY.T, TINY.num_heads, TINY.num_layers
    att = m.act("att").reshape(L, B, NH, T, T)
    rows = att.sum(axis=-1)
    np.testing.assert_allclose(rows, 1.0, atol=1e-12)
    mask = np.triu(np.ones((T, T), bool), k=1)
    assert np.all(att[..., mask] == 0.0)
    assert np.all(att[..., ~mask] > 0.0)
    probs = m.act("probs").reshape(B * T, -1)
    np.testing.assert_allclose(probs.sum(axis=1), 1.0, atol=1e-12)


def test_P5_padded_vocab_columns_have_zero_probability():
    w = synth.Workload("pad", 1, 32, 2, 100, 128, 16, 2, 8, "fp32", "uniform", 3)
    m = ref.RefModel(ref.config_from(w), 2, 8, np.float32)
    m.set_params(perturbed_params(w))
    inp, tgt = synth.batch(w)
    m.forward(inp, tgt)
    probs = m.act("probs").reshape(16, 128)
    assert np.all(probs[:, 100:] == 0.0)
    np.testing.assert_allclose(probs.sum(axis=1, dtype=np.float64), 1.0, atol=1e-6)


# --------------------------------------------------------------------------
# P6: initial loss near ln V
# --------------------------------------------------------------------------
def test_P6_initial_loss_tiny():
    inp, tgt = synth.batch(TINY)
    m = ref.RefModel(ref.config_from(TINY), TINY.B, TINY.T, np.float64)
    m.set_params(synth.init_params(TINY, wte_std=1e-4))
    assert abs(m.forward(inp, tgt) - math.log(512)) < 1e-3
    m.set_params(synth.init_params(TINY))
    assert abs(m.forward(inp, tgt) - math.log(512)) < 0.05 * math.log(512)


@pytest.mark.slow
def test_P6_initial_loss_124m():
    w = G124
    m = ref.RefModel(ref.config_from(w), w.B, w.T, np.float32)
    m.set_params(synth.init_params(w))
    inp, tgt = synth.batch(w)
    loss = m.forward(inp, tgt)
    # logits std ~ 0.02*sqrt(C) gives E[loss] ~ ln V + (0.02^2 C)/2 ~ 10.98
    assert abs(loss - math.log(50257)) < 0.05 * math.log(50257)
    assert 10.8 < loss < 11.2
    m.close()


# --------------------------------------------------------------------------
# P7: gradients against central finite differences (double build)
# --------------------------------------------------------------------------
def test_P7_finite_difference_gradients():
    w = synth.Workload("fd", 2, 32, 4, 64, 64, 16, 2, 12, "fp32", "uniform", 1)
    p0 = perturbed_params(w, seed=11)
    inp, tgt = synth.batch(w)
    m = ref.RefModel(ref.config_from(w), w.B, w.T, np.float64)
    m.set_params(p0)
    m.forward(inp, tgt)
    m.zero_grad()
    assert m.backward() == 0
    g = m.grads.copy()

    def loss_at(p):
        m.set_params(p)
        return m.forward(inp, tgt)

    h = 1e-5
    rng = np.random.default_rng(3)
    offs = synth.param_offsets(w)
    worst = 0.0
    for name, (o, n) in offs.items():
        idx = o + rng.choice(n, size=min(n, 12), replace=False)
        if name == "wpe":  # only rows < T receive gradient; also test those
            idx = o + rng.choice(w.T * w.channels, size=12, replace=False)
        for i in idx:
            pp = p0.copy(); pp[i] += h
            pm = p0.copy(); pm[i] -= h
            fd = (loss_at(pp) - loss_at(pm)) / (2 * h)
            err = abs(fd - g[i])
            assert err <= 1e-6 * abs(g[i]) + 2e-9, (name, i, fd, g[i])
            worst = max(worst, err)
        # directional derivative along a random direction inside the tensor
        d = np.zeros_like(p0)
        d[o:o + n] = rng.standard_normal(n)
        fd = (loss_at(p0 + h * d) - loss_at(p0 - h * d)) / (2 * h)
        gd = float(g[o:o + n] @ d[o:o + n])
        assert abs(fd - gd) <= 1e-6 * abs(gd) + 1e-8, (name, fd, gd)
    m.close()


# --------------------------------------------------------------------------
# P8: brute-force causality
# --------------------------------------------------------------------------
def test_P8_causality_changing_token_t_leaves_earlier_logits_bit_identical():
    m = tiny_model(np.float32)
    inp, tgt = synth.batch(TINY)
    m.forward(inp, tgt)
    l0 = m.act("logits").reshape(TINY.B, TINY.T, -1).copy()
    t = 17
    inp2 = inp.copy()
    inp2[:, t] = (inp2[:, t] + 123) % TINY.vocab_size
    m.forward(inp2, tgt)
    l1 = m.act("logits").reshape(TINY.B, TINY.T, -1)
    assert np.array_equal(l0[:, :t], l1[:, :t])
    assert not np.array_equal(l0[:, t], l1[:, t])


def test_P8_zero_queries_give_uniform_causal_average():
    ops = ref.ops(np.float64)
    rng = np.random.default_rng(5)
    B, T, C, NH = 2, 9, 24, 3
    qkv = rng.standard_normal((B, T, 3 * C))
    qkv[:, :, :C] = 0.0  # q = 0 -> all scores 0
    out, _, att = ops.attention_forward(qkv, NH)
    for t in range(T):
        np.testing.assert_allclose(att[:, :, t, :t + 1], 1.0 / (t + 1), rtol=1e-14)
        v = qkv[:, :t + 1, 2 * C:]
        np.testing.assert_allclose(out[:, t], v.mean(axis=1), rtol=1e-12, atol=1e-14)


def test_P8_single_position_attention_returns_v():
    ops = ref.ops(np.float64)
    rng = np.random.default_rng(6)
    qkv = rng.standard_normal((3, 1, 3 * 40))
    out, _, att = ops.attention_forward(qkv, 5)
    np.testing.assert_array_equal(out[:, 0], qkv[:, 0, 80:])
    assert np.all(att == 1.0)


# --------------------------------------------------------------------------
# P10: AdamW first step closed form
# --------------------------------------------------------------------------
def test_P10_adamw_first_step_closed_form():
    ops = ref.ops(np.float64)
    rng = np.random.default_rng(8)
    n = 4096
    p = rng.standard_normal(n)
    g = rng.standard_normal(n) * np.exp(rng.uniform(-12, 2, n))
    lr, eps = 1e-4, 1e-8
    p1, m1, v1 = ops.adamw_update(p, g, np.zeros(n), np.zeros(n), lr, 0.9, 0.999, eps, 0.0, 1)
    np.testing.assert_allclose(p1, p - lr * g / (np.abs(g) + eps), rtol=1e-13, atol=1e-19)
    big = np.abs(g) > 1e-3
    np.testing.assert_allclose(p1[big] - p[big], -lr * np.sign(g[big]), rtol=1e-4)
    np.testing.assert_allclose(m1, 0.1 * g, rtol=1e-12)
    np.testing.assert_allclose(v1, 0.001 * g * g, rtol=1e-12)
    # decoupled weight decay: a zero gradient leaves only the decay term
    p2, _, _ = ops.adamw_update(p, np.zeros(n), np.zeros(n), np.zeros(n), lr, 0.9, 0.999, eps, 0.1, 1)
    np.testing.assert_allclose(p2, p * (1 - lr * 0.1), rtol=1e-14)


# --------------------------------------------------------------------------
# P11: invariants
# --------------------------------------------------------------------------
def test_P11_backward_accumulates():
    m = tiny_model(np.float32)
    inp, tgt = synth.batch(TINY)
    m.forward(inp, tgt)
    m.zero_grad()
    assert m.backward() == 0
    g1 = m.grads.copy()
    assert m.backward() == 0
    g2 = m.grads.copy()
    offs = synth.param_offsets(TINY)
    for name, (o, n) in offs.items():
        if name == "wte":  # two contributions per backward (LM head + embedding): rounding differs
            np.testing.assert_allclose(g2[o:o + n], 2 * g1[o:o + n], rtol=1e-5, atol=1e-9)
        else:
            assert np.array_equal(g2[o:o + n], 2 * g1[o:o + n]), name
    m.zero_grad()
    assert np.all(m.grads == 0)


def test_P11_backward_needs_forward_with_targets():
    m = tiny_model(np.float32)
    inp, _ = synth.batch(TINY)
    assert m.backward() == -4
    assert m.forward(inp, None) == -1.0
    assert m.backward() == -4


def test_P11_fixed_batch_loss_strictly_decreases_and_pad_rows_stay_zero():
    w = synth.Workload("pad", 2, 32, 2, 100, 128, 16, 2, 16, "fp32", "uniform", 10)
    m = ref.RefModel(ref.config_from(w), w.B, w.T, np.float32)
    m.set_params(synth.init_params(w))
    inp, tgt = synth.batch(w)
    losses = [m.step(inp, tgt, t, lr=1e-3) for t in range(1, 11)]
    assert all(b < a for a, b in zip(losses, losses[1:])), losses
    o, _ = synth.param_offsets(w)["wte"]
    pad = slice(o + 100 * 32, o + 128 * 32)
    assert np.all(m.params[pad] == 0.0) and np.all(m.grads[pad] == 0.0)


def test_P11_tiny_config_ten_steps_lr_1e4_decreases():
    m = ref.RefModel(ref.config_from(TINY), TINY.B, TINY.T, np.float32)
    m.set_params(synth.init_params(TINY))
    inp, tgt = synth.batch(TINY)
    losses = [m.step(inp, tgt, t) for t in range(1, 11)]
    assert all(b < a for a, b in zip(losses, losses[1:])), losses


def test_P11_zipf_unigram_entropy_floor():
    p = np.diff(np.concatenate([[0.0], synth.zipf_cdf(50257)]))
    H = float(-(p * np.log(p)).sum())
    assert abs(H - 6.4647) < 5e-4
    assert abs(p[0] - 0.139) < 1e-3


# --------------------------------------------------------------------------
# P12: determinism across thread counts
# --------------------------------------------------------------------------
_DET_SCRIPT = r"""
import sys, hashlib, numpy as np
sys.path.insert(0, %r)
import synth
from oracle import ref
w = synth.Workload("det", 2, 48, 4, 200, 256, 24, 3, 24, "fp32", "uniform", 2)
m = ref.RefModel(ref.config_from(w), w.B, w.T, np.float32)
m.set_params(synth.init_params(w))
inp, tgt = synth.batch(w)
for t in (1, 2):
    m.step(inp, tgt, t)
m.forward(inp, tgt); m.zero_grad(); m.backward()
h = hashlib.sha256(m.params.tobytes() + m.grads.tobytes() + m.act("logits").tobytes()).hexdigest()
print(h)
"""


def test_P12_oracle_bit_identical_across_thread_counts():
    root = os.path.dirname(HERE)
    outs = []
    for nt in ("1", "3", "8"):
        env = dict(os.environ, OMP_NUM_THREADS=nt)
        r = subprocess.run([sys.executable, "-c", _DET_SCRIPT % root], env=env, capture_output=True, text=True,
                           check=True)
        outs.append(r.stdout.strip())
    assert outs[0] == outs[1] == outs[2]


# ---------------------------------------------------------------------------
# Sampling (the page's item 5, sample_mult): inverse-CDF draws with the
# uniform coin passed in.  Pins: the definition at exact binary boundaries,
# zero-probability entries, the rounding tail, and the closed-form counts of
# stratified coins.
# ---------------------------------------------------------------------------
def test_sample_mult_boundaries():
    p = [0.125, 0.25, 0.625]  # cumulative 0.125, 0.375, 1.0, exact in binary
    cases = [(0.0, 0), (0.124, 0), (0.125, 1), (0.374, 1), (0.375, 2), (0.999, 2)]
    for coin, want in cases:
        assert ref.sample_mult(p, coin) == want, (coin, want)


def test_sample_mult_skips_zero_probabilities():
    p = [0.0, 0.5, 0.0, 0.5, 0.0]
    draws = {ref.sample_mult(p, c) for c in np.linspace(0.0, 0.999, 101)}
    assert draws == {1, 3}
    assert ref.sample_mult(p, 0.0) == 1


def test_sample_mult_rounding_tail_takes_last_nonzero():
    # probabilities summing below the coin (as rounding can leave them)
    assert ref.sample_mult([0.25, 0.25, 0.0], 0.75) == 1


def test_sample_mult_stratified_counts():
    p = [0.2, 0.5, 0.3]
    n = 1000
    counts = np.bincount([ref.sample_mult(p, (i + 0.5) / n) for i in range(n)], minlength=3)
    assert counts.tolist() == [200, 500, 300]


def test_softmax64_closed_form():
    np.testing.assert_allclose(ref.softmax64([0.0, np.log(3.0)]), [0.25, 0.75], rtol=1e-15)


def test_sample_is_valid():
    p = [0.125, 0.25, 0.625]
    assert ref.sample_is_valid(p, 0.2, 1, 0.0)
    assert not ref.sample_is_valid(p, 0.2, 2, 0.0)
    assert ref.sample_is_valid(p, 0.3749999, 2, 1e-6)  # within tol of the 0.375 boundary


# ---------------------------------------------------------------------------
# Llama-style variant ([LL]: RMSNorm in place of layernorm, RoPE on q and k,
# no position table, no biases).  Pins: closed forms, the invariances that
# define the two layers (scale invariance; rotation, identity at t = 0 and
# dependence of q.k on the position difference only), the transpose used by
# the backward, the parameter count, and whole-model finite differences.
# ---------------------------------------------------------------------------
LL_OPS = ref.ops(np.float64)


def test_LL_rmsnorm_closed_form_and_scale_invariance():
    x = np.array([[3.0, 4.0], [-1.0, 2.0]])
    w = np.array([2.0, 0.5])
    y, rstd = LL_OPS.rmsnorm_forward(x, w)
    np.testing.assert_allclose(y[0], [6.0 / np.sqrt(12.5 + 1e-5), 2.0 / np.sqrt(12.5 + 1e-5)], rtol=1e-14)
    np.testing.assert_allclose(rstd, 1.0 / np.sqrt((x * x).mean(1) + 1e-5), rtol=1e-14)
    xr = np.random.default_rng(0).standard_normal((4, 32))
    y1, _ = LL_OPS.rmsnorm_forward(xr, np.ones(32))
    y5, _ = LL_OPS.rmsnorm_forward(5.0 * xr, np.ones(32))
    np.testing.assert_allclose(y5, y1, rtol=1e-5)  # eps 1e-5 is the only scale-dependent term
    np.testing.assert_allclose(np.sqrt((y1 * y1).mean(1)), 1.0, rtol=1e-4)


def test_LL_rmsnorm_backward_finite_differences():
    rng = np.random.default_rng(1)
    x, w, dy = rng.standard_normal((3, 8)), rng.standard_normal(8), rng.standard_normal((3, 8))
    _, rstd = LL_OPS.rmsnorm_forward(x, w)
    dx, dw = LL_OPS.rmsnorm_backward(dy, x, w, rstd)
    h = 1e-6
    f = lambda xx, ww: float((LL_OPS.rmsnorm_forward(xx, ww)[0] * dy).sum())
    for i in range(3):
        for j in range(8):
            xp, xm = x.copy(), x.copy()
            xp[i, j] += h
            xm[i, j] -= h
            assert abs((f(xp, w) - f(xm, w)) / (2 * h) - dx[i, j]) <= 1e-7 * (1 + abs(dx[i, j]))
    for j in range(8):
        wp, wm = w.copy(), w.copy()
        wp[j] += h
        wm[j] -= h
        assert abs((f(x, wp) - f(x, wm)) / (2 * h) - dw[j]) <= 1e-7 * (1 + abs(dw[j]))


def test_LL_rope_closed_form_identity_and_v_untouched():
    # one head of size 2: the single pair turns by t radians (frequency 10000^0)
    qkv = np.zeros((1, 3, 6))
    qkv[0, :, 0] = 1.0  # q = (1, 0) at every position
    qkv[0, :, 4] = 7.0  # v
    r = LL_OPS.rope_apply(qkv, 1)
    for t in range(3):
        np.testing.assert_allclose(r[0, t, 0:2], [np.cos(t), np.sin(t)], rtol=0, atol=1e-15)
    np.testing.assert_array_equal(r[0, :, 4:6], qkv[0, :, 4:6])
    x = np.random.default_rng(2).standard_normal((2, 1, 3 * 16))  # position 0 only
    np.testing.assert_array_equal(LL_OPS.rope_apply(x, 2), x)


def test_LL_rope_scores_depend_on_position_difference_only():
    rng = np.random.default_rng(3)
    C, NH, T = 16, 2, 9
    hs = C // NH
    q, k = rng.standard_normal(hs), rng.standard_normal(hs)

    def score(tq, tk):
        x = np.zeros((1, T, 3 * C))
        x[0, tq, 0:hs] = q  # head 0 query at position tq
        x[0, tk, C:C + hs] = k  # head 0 key at position tk
        r = LL_OPS.rope_apply(x, NH)
        return float(r[0, tq, 0:hs] @ r[0, tk, C:C + hs])

    for tq, tk, d in [(2, 0, 5), (4, 4, 3), (0, 3, 2), (6, 1, 2)]:
        assert abs(score(tq, tk) - score(tq + d, tk + d)) <= 1e-12 * (1 + abs(score(tq, tk)))
    assert abs(score(2, 0) - score(3, 0)) > 1e-6  # and it does depend on the difference


def test_LL_rope_inverse_is_the_transpose():
    rng = np.random.default_rng(4)
    x, y = rng.standard_normal((2, 7, 3 * 24)), rng.standard_normal((2, 7, 3 * 24))
    rx = LL_OPS.rope_apply(x, 3)
    np.testing.assert_allclose(LL_OPS.rope_apply(rx, 3, inverse=True), x, atol=1e-14)
    lhs = float((rx * y).sum())
    rhs = float((x * LL_OPS.rope_apply(y, 3, inverse=True)).sum())
    assert abs(lhs - rhs) <= 1e-12 * abs(lhs)


LLAMA_FD = synth.Workload("llama_fd", 2, 32, 4, 64, 64, 16, 2, 12, "fp32", "uniform", 1, llama=1)


def test_LL_parameter_count():
    w = LLAMA_FD
    L, C, Vp = w.num_layers, w.channels, w.padded_vocab_size
    want = Vp * C + L * (C + 3 * C * C + C * C + C + 4 * C * C + 4 * C * C) + C
    assert ref.num_parameters(ref.config_from(w)) == want == synth.num_params(w)
    offs = ref.param_offsets(ref.config_from(w))
    assert offs == synth.param_offsets(w)


def test_LL_finite_difference_gradients():
    w = LLAMA_FD
    p0 = perturbed_params(w, seed=17)
    inp, tgt = synth.batch(w)
    m = ref.RefModel(ref.config_from(w), w.B, w.T, np.float64)
    m.set_params(p0)
    m.forward(inp, tgt)
    m.zero_grad()
    assert m.backward() == 0
    g = m.grads.copy()

    def loss_at(p):
        m.set_params(p)
        return m.forward(inp, tgt)

    h = 1e-5
    rng = np.random.default_rng(5)
    for name, (o, n) in synth.param_offsets(w).items():
        if n == 0:
            continue
        for i in o + rng.choice(n, size=min(n, 10), replace=False):
            pp = p0.copy(); pp[i] += h
            pm = p0.copy(); pm[i] -= h
            fd = (loss_at(pp) - loss_at(pm)) / (2 * h)
            assert abs(fd - g[i]) <= 1e-6 * abs(g[i]) + 2e-9, (name, i, fd, g[i])
        d = np.zeros_like(p0)
        d[o:o + n] = rng.standard_normal(n)
        fd = (loss_at(p0 + h * d) - loss_at(p0 - h * d)) / (2 * h)
        gd = float(g[o:o + n] @ d[o:o + n])
        assert abs(fd - gd) <= 1e-6 * abs(gd) + 1e-8, (name, fd, gd)
    m.close()
