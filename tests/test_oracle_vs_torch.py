"""P9: every oracle operation against PyTorch CPU float64 library routines.

The llm.c pages check the C code against PyTorch (page «千行C代码训完GPT-2»,
section «测试»: logits and loss of one forward, then ten Adam steps).  Here
each layer of the double build is checked against torch's own routine for the
same definition (F.layer_norm, F.linear, F.scaled_dot_product_attention,
F.gelu(approximate="tanh"), F.cross_entropy, torch.optim.AdamW), forward and
backward through autograd, and the whole tiny model once end to end.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import synth
from oracle import ref

OPS = ref.ops(np.float64)
RTOL = 1e-10


def close(a, b, rtol=RTOL):
    a = np.asarray(a, dtype=np.float64)
    b = b.detach().numpy() if isinstance(b, torch.Tensor) else np.asarray(b, dtype=np.float64)
    scale = max(np.abs(b).max(), 1e-300)
    err = np.abs(a - b).max() / scale
    assert err < rtol, err


def leaf(x):
    return torch.tensor(np.asarray(x, dtype=np.float64), dtype=torch.float64, requires_grad=True)


def test_encoder_vs_embedding():
    rng = np.random.default_rng(0)
    V, maxT, C, B, T = 50, 16, 24, 3, 11
    ids = rng.integers(0, V, (B, T)).astype(np.int32)
    ids[0, :4] = 7  # repeated ids exercise the scatter-add
    wte, wpe = rng.standard_normal((V, C)), rng.standard_normal((maxT, C))
    dx = rng.standard_normal((B, T, C))
    out = OPS.encoder_forward(ids, wte, wpe)
    twte, twpe = leaf(wte), leaf(wpe)
    tout = F.embedding(torch.tensor(ids, dtype=torch.long), twte) + twpe[:T]
    close(out, tout)
    tout.backward(torch.tensor(dx))
    dwte, dwpe = OPS.encoder_backward(dx, ids, V, maxT)
    close(dwte, twte.grad)
    close(dwpe, twpe.grad)


def test_layernorm_vs_torch():
    rng = np.random.default_rng(1)
    x = 0.3 + 2.0 * rng.standard_normal((4, 7, 48))
    w, b = rng.standard_normal(48), rng.standard_normal(48)
    dy = rng.standard_normal(x.shape)
    y, mean, rstd = OPS.layernorm_forward(x, w, b)
    tx, tw, tb = leaf(x), leaf(w), leaf(b)
    ty = F.layer_norm(tx, (48,), tw, tb, eps=1e-5)
    close(y, ty)
    ty.backward(torch.tensor(dy))
    dx, dw, db = OPS.layernorm_backward(dy, x, w, mean, rstd)
    close(dx, tx.grad)
    close(dw, tw.grad)
    close(db, tb.grad)


@pytest.mark.parametrize("with_bias", [True, False])
def test_matmul_vs_linear(with_bias):
    rng = np.random.default_rng(2)
    x = rng.standard_normal((3, 5, 40))
    W = rng.standard_normal((56, 40))
    b = rng.standard_normal(56) if with_bias else None
    dy = rng.standard_normal((3, 5, 56))
    out = OPS.matmul_forward(x, W, b)
    tx, tW = leaf(x), leaf(W)
    tb = leaf(b) if with_bias else None
    tout = F.linear(tx, tW, tb)
    close(out, tout)
    tout.backward(torch.tensor(dy))
    dx, dW, db = OPS.matmul_backward(dy, x, W, with_bias)
    close(dx, tx.grad)
    close(dW, tW.grad)
    if with_bias:
        close(db, tb.grad)


@pytest.mark.parametrize("T", [1, 5, 33])
def test_attention_vs_sdpa(T):
    rng = np.random.default_rng(3 + T)
    B, NH, hs = 2, 3, 8
    C = NH * hs
    qkv = rng.standard_normal((B, T, 3 * C))
    dout = rng.standard_normal((B, T, C))
    out, preatt, att = OPS.attention_forward(qkv, NH)
    tqkv = leaf(qkv)
    q, k, v = tqkv.split(C, dim=-1)
    sh = lambda z: z.view(B, T, NH, hs).transpose(1, 2)
    ty = F.scaled_dot_product_attention(sh(q), sh(k), sh(v), is_causal=True)
    ty = ty.transpose(1, 2).reshape(B, T, C)
    close(out, ty)
    # the stored attention matrix is the causal softmax of the scores
    s = (sh(q) @ sh(k).transpose(-1, -2)) / np.sqrt(hs)
    s = s.masked_fill(torch.triu(torch.ones(T, T, dtype=torch.bool), 1), float("-inf"))
    close(att, torch.softmax(s, -1))
    ty.backward(torch.tensor(dout))
    dqkv = OPS.attention_backward(dout, qkv, att, NH)
    close(dqkv, tqkv.grad)


def test_gelu_vs_torch_tanh():
    rng = np.random.default_rng(4)
    x = 3.0 * rng.standard_normal(1000)
    dy = rng.standard_normal(1000)
    tx = leaf(x)
    ty = F.gelu(tx, approximate="tanh")
    close(OPS.gelu_forward(x), ty)
    ty.backward(torch.tensor(dy))
    close(OPS.gelu_backward(x, dy), tx.grad)


def test_residual():
    rng = np.random.default_rng(5)
    a, b, d = rng.standard_normal((3, 100))
    close(OPS.residual_forward(a, b), torch.tensor(a + b))
    da, db = OPS.residual_backward(d)
    close(da, torch.tensor(d))
    close(db, torch.tensor(d))


@pytest.mark.parametrize("V,Vp", [(37, 37), (37, 48)])
def test_softmax_crossentropy_vs_torch(V, Vp):
    rng = np.random.default_rng(6)
    N = 13
    logits = 4.0 * rng.standard_normal((N, Vp))
    targets = rng.integers(0, V, N).astype(np.int32)
    probs = OPS.softmax_forward(logits, V)
    tl = leaf(logits)
    close(probs[:, :V], torch.softmax(tl[:, :V], -1))
    assert np.all(probs[:, V:] == 0)
    losses = OPS.crossentropy_forward(probs, targets)
    tloss = F.cross_entropy(tl[:, :V], torch.tensor(targets, dtype=torch.long), reduction="none")
    close(losses, tloss)
    tloss.mean().backward()
    dlogits = OPS.crossentropy_softmax_backward(np.full(N, 1.0 / N), probs, targets, V)
    close(dlogits, tl.grad)


@pytest.mark.parametrize("wd", [0.0, 0.1])
def test_adamw_vs_torch_optim(wd):
    rng = np.random.default_rng(7)
    n = 500
    p0 = rng.standard_normal(n)
    tp = torch.nn.Parameter(torch.tensor(p0))
    opt = torch.optim.AdamW([tp], lr=1e-3, betas=(0.9, 0.999), eps=1e-8, weight_decay=wd)
    p, m, v = p0.copy(), np.zeros(n), np.zeros(n)
    for t in range(1, 11):
        g = rng.standard_normal(n) * (0.1 * t)
        tp.grad = torch.tensor(g)
        opt.step()
        p, m, v = OPS.adamw_update(p, g, m, v, 1e-3, 0.9, 0.999, 1e-8, wd, t)
        close(p, tp.detach(), rtol=1e-12)
        st = opt.state[tp]
        close(m, st["exp_avg"], rtol=1e-12)
        close(v, st["exp_avg_sq"], rtol=1e-12)


# --------------------------------------------------------------------------
# whole model, tiny config, end to end through autograd
# --------------------------------------------------------------------------
def torch_gpt2_loss(flat, w, inputs, targets):
    """GPT-2 written with torch library ops (layer_norm, linear, SDPA, gelu,
    cross_entropy); weights are views into the flat tensor."""
    C, L, NH, V, Vp = w.channels, w.num_layers, w.num_heads, w.vocab_size, w.padded_vocab_size
    B, T = inputs.shape
    hs = C // NH
    shapes = synth.param_shapes(w)
    P, off = {}, 0
    for name in synth.PARAM_NAMES:
        n = int(np.prod(shapes[name]))
        P[name] = flat[off: off + n].view(shapes[name])
        off += n
    ids = torch.tensor(inputs, dtype=torch.long)
    x = F.embedding(ids, P["wte"]) + P["wpe"][:T]
    for l in range(L):
        h = F.layer_norm(x, (C,), P["ln1w"][l], P["ln1b"][l], eps=1e-5)
        q, k, v = F.linear(h, P["qkvw"][l], P["qkvb"][l]).split(C, dim=-1)
        sh = lambda z: z.view(B, T, NH, hs).transpose(1, 2)
        y = F.scaled_dot_product_attention(sh(q), sh(k), sh(v), is_causal=True).transpose(1, 2).reshape(B, T, C)
        x = x + F.linear(y, P["attprojw"][l], P["attprojb"][l])
        h = F.layer_norm(x, (C,), P["ln2w"][l], P["ln2b"][l], eps=1e-5)
        h = F.gelu(F.linear(h, P["fcw"][l], P["fcb"][l]), approximate="tanh")
        x = x + F.linear(h, P["fcprojw"][l], P["fcprojb"][l])
    x = F.layer_norm(x, (C,), P["lnfw"], P["lnfb"], eps=1e-5)
    logits = x @ P["wte"].T
    loss = F.cross_entropy(logits[..., :V].reshape(-1, V), torch.tensor(targets, dtype=torch.long).reshape(-1))
    return loss, logits


@pytest.mark.parametrize("V,Vp", [(512, 512), (500, 512)])
def test_whole_tiny_model_vs_autograd(V, Vp):
    w = synth.Workload("t", 2, 64, 4, V, Vp, 32, 2, 32, "fp32", "uniform", 1)
    rng = np.random.default_rng(9)
    p = synth.init_params(w).astype(np.float64)
    offs = synth.param_offsets(w)
    for name in ("ln1b", "ln2b", "lnfb", "qkvb", "attprojb", "fcb", "fcprojb"):
        o, n = offs[name]
        p[o:o + n] = 0.02 * rng.standard_normal(n)
    inp, tgt = synth.batch(w)
    m = ref.RefModel(ref.config_from(w), w.B, w.T, np.float64)
    m.set_params(p)
    loss = m.forward(inp, tgt)
    m.zero_grad()
    m.backward()
    tp = leaf(p)
    tloss, tlogits = torch_gpt2_loss(tp, w, inp, tgt)
    assert abs(loss - tloss.item()) < 1e-12 * abs(loss)
    close(m.act("logits"), tlogits.reshape(-1))
    tloss.backward()
    g = m.grads
    for name, (o, n) in offs.items():
        close(g[o:o + n], tp.grad[o:o + n], rtol=1e-9)
    m.close()
