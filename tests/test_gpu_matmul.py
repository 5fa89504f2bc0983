"""Per-layer parity of the tensor-core matmul (tcgen05, 3xTF32) against the
oracle's matmul_forward / matmul_backward (the page «llm.c：Andrej Karpathy
带你从零复现LLM», section «核心代码解读：train_gpt2.c», item 1).  Shapes cover
ragged M, N and K (partial 128x128 tiles and partial 32-wide K tiles),
split-K (small N with long K), products with more tiles than SMs (the
persistent kernel, one CTA per SM walking the tiles) and both operand
layouts of each product."""
import numpy as np
import pytest

import synth
from oracle import ref

pytestmark = pytest.mark.gpu

OPS = ref.ops(np.float32)

SHAPES = [  # (N rows, IC, OC)
    (64, 64, 192),      # tiny config QKV
    (13, 68, 100),      # ragged everything
    (1, 64, 64),        # one row
    (300, 96, 260),     # M spans 3 tiles with a tail
    (256, 768, 2304),   # 124M QKV at B*T=256: split-K
    (256, 3072, 768),   # 124M MLP output projection: split-K over 3072
    (256, 768, 50304),  # LM head (tied wte), 393 column tiles: forward and weight gradient persistent
    (1000, 200, 2500),  # forward with 160 tiles (> 148 SMs, persistent), ragged M, N and K
    (300, 1100, 2100),  # weight gradient with 153 tiles (persistent, both operands MN-major), ragged K = 300
    (256, 1024, 3072),  # 350M QKV (K = 1024)
    (256, 4096, 1024),  # 350M MLP output projection (K = 4096)
    (256, 1280, 3840),  # 774M QKV (K = 1280)
    (256, 5120, 1280),  # 774M MLP output projection (K = 5120)
]


def tol(K):
    """3xTF32 products are ~2^-20 relative; the tensor core's fp32
    accumulation adds an error that grows with the summed length K."""
    return 1e-5 if K <= 4096 else 1e-4


def rel_err(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return np.abs(a - b).max() / max(np.abs(b).max(), 1e-30)


@pytest.mark.parametrize("N,IC,OC", SHAPES)
def test_matmul_forward_backward_fp32(N, IC, OC):
    import torch
    import gpt_train_step_02_b300 as g

    x = synth.randn(101, (N, IC))
    W = synth.randn(102, (OC, IC), 0.02)
    b = synth.randn(103, (OC,), 0.1)
    dy = synth.randn(104, (N, OC))
    dW0 = synth.randn(105, (OC, IC), 0.01)
    db0 = synth.randn(106, (OC,), 0.01)

    tx, tW, tb, tdy = (torch.tensor(a, device="cuda") for a in (x, W, b, dy))
    out = torch.empty((N, OC), dtype=torch.float32, device="cuda")
    g.matmul_forward(out, tx, tW, tb)
    ref_out = OPS.matmul_forward(x, W, b)
    assert rel_err(out.cpu().numpy(), ref_out) < tol(IC)

    out0 = torch.empty((N, OC), dtype=torch.float32, device="cuda")
    g.matmul_forward(out0, tx, tW, None)
    assert rel_err(out0.cpu().numpy(), OPS.matmul_forward(x, W, None)) < tol(IC)

    dx = torch.empty((N, IC), dtype=torch.float32, device="cuda")
    tdW = torch.tensor(dW0, device="cuda")
    tdb = torch.tensor(db0, device="cuda")
    g.matmul_backward(dx, tdW, tdb, tdy, tx, tW)
    rdx, rdW, rdb = OPS.matmul_backward(dy, x, W, True)
    assert rel_err(dx.cpu().numpy(), rdx) < tol(OC)
    assert rel_err(tdW.cpu().numpy() - dW0, rdW) < tol(N)
    assert rel_err(tdb.cpu().numpy() - db0, rdb) < 1e-5


def bf16(a):
    """Round to the nearest bf16 (ties to even), returned as float32."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


SHAPES_BF16 = [  # (N rows, IC, OC); IC and OC multiples of 8 (16-byte bf16 rows)
    (64, 64, 192),      # tiny config QKV: one 128-wide column tile
    (13, 72, 104),      # ragged everything, N <= 128 (128-wide tiles)
    (300, 96, 264),     # M spans 3 tiles with a tail; 256-wide column tiles with a tail
    (256, 768, 2304),   # 124M QKV at B*T=256
    (256, 3072, 768),   # MLP output projection: K split for the weight gradient
    (1024, 768, 768),   # attention projection at B*T=1024: K-split weight gradient
    (256, 768, 50304),  # LM head (tied wte), 197 column tiles
    (2048, 1024, 3072),  # 350M QKV at B*T = 2048 (K = 1024)
    (1024, 4096, 1024),  # 350M MLP output projection (K = 4096)
    (1024, 1280, 3840),  # 774M QKV (K = 1280)
    (1024, 5120, 1280),  # 774M MLP output projection (K = 5120)
    # 774M at B*T = 4096: 192-wide column tiles (the forward's K-major and the
    # input gradient's MN-major B), 192-wide tiles split in two for the
    # attention projection's weight gradient
    (4096, 1280, 1280),
    (4096, 5120, 1280),
]


@pytest.mark.parametrize("N,IC,OC", SHAPES_BF16)
def test_matmul_bf16_forward_backward(N, IC, OC):
    """bf16 tensor-core products against the oracle fed the same bf16-rounded
    operands (the products are exact in fp32; only the fp32 accumulation
    order differs)."""
    import torch
    import gpt_train_step_02_b300 as g

    x = synth.randn(111, (N, IC))
    W = synth.randn(112, (OC, IC), 0.02)
    b = synth.randn(113, (OC,), 0.1)
    dy = synth.randn(114, (N, OC))
    dW0 = synth.randn(115, (OC, IC), 0.01)
    db0 = synth.randn(116, (OC,), 0.01)
    tx, tW, tb, tdy = (torch.tensor(a, device="cuda") for a in (x, W, b, dy))
    P = g.GPT2_PREC_BF16

    out = torch.empty((N, OC), dtype=torch.float32, device="cuda")
    g.matmul_forward(out, tx, tW, tb, precision=P)
    ref_out = OPS.matmul_forward(bf16(x), bf16(W), b)
    assert rel_err(out.cpu().numpy(), ref_out) < tol(IC)
    if IC >= 64:  # really bf16: the unrounded product differs
        assert rel_err(out.cpu().numpy() - b, OPS.matmul_forward(x, W, None)) > 1e-4

    dx = torch.empty((N, IC), dtype=torch.float32, device="cuda")
    tdW = torch.tensor(dW0, device="cuda")
    tdb = torch.tensor(db0, device="cuda")
    g.matmul_backward(dx, tdW, tdb, tdy, tx, tW, precision=P)
    rdx, rdW, _ = OPS.matmul_backward(bf16(dy), bf16(x), bf16(W), False)
    _, _, rdb = OPS.matmul_backward(dy, x, W, True)  # the bias gradient sums the fp32 dy
    assert rel_err(dx.cpu().numpy(), rdx) < tol(OC)
    assert rel_err(tdW.cpu().numpy() - dW0, rdW) < tol(N)
    assert rel_err(tdb.cpu().numpy() - db0, rdb) < 1e-5


def test_matmul_bf16_rejects_rows_that_are_not_16_bytes():
    import torch
    import gpt_train_step_02_b300 as g

    N, IC, OC = 16, 68, 64  # IC % 8 != 0: a bf16 row of 136 bytes
    x = torch.zeros((N, IC), device="cuda")
    W = torch.zeros((OC, IC), device="cuda")
    out = torch.zeros((N, OC), device="cuda")
    with pytest.raises(g.GPT2Error) as e:
        g.matmul_forward(out, x, W, None, precision=g.GPT2_PREC_BF16)
    assert e.value.status == g.GPT2_ERR_SHAPE
