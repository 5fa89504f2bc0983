"""The matmul backward for callers that cannot allocate device memory.

Some callers have no way to hand the library a workspace. One example is a
plugin whose host application's allocator already owns all of the device's
memory. Another is a loop that must not call cudaMalloc, because cudaMalloc
can synchronise the device. For these callers,
``gpt2op_matmul_backward_noalloc`` takes its scratch from a fixed array in
the library's own device memory.

These tests check, through the C ABI, that the variant gives the same dx,
dW and dbias as ``gpt2op_matmul_backward`` with a caller workspace. The check
runs on two calls in a row, so the second call runs on the scratch the first
one left behind. They also check that a shape whose bias partials exceed the
fixed array is rejected before any device work.

The file is collected last, so a run that stops at its first failure has
already run every other test.
"""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

SHAPES = [  # (N rows, IC, OC)
    (256, 768, 768),    # split-K products and a bias gradient
    (300, 96, 260),     # ragged tiles
    (256, 3072, 768),   # long K for the input gradient
]


def rel_err(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return np.abs(a - b).max() / max(np.abs(b).max(), 1e-30)


def tol(K):
    """The tolerance of the fp32 matmul parity tests: 3xTF32 products are
    about 2^-20 relative; the fp32 accumulation error grows with K."""
    return 1e-5 if K <= 4096 else 1e-4


@pytest.mark.parametrize("N,IC,OC", SHAPES)
def test_noalloc_backward_matches_workspace_backward_on_two_calls(N, IC, OC):
    import torch

    import gpt_train_step_02_b300 as g

    dev = torch.device("cuda", 0)
    x = torch.from_numpy(synth.randn(201, (N, IC))).to(dev)
    W = torch.from_numpy(synth.randn(202, (OC, IC), 0.02)).to(dev)
    dy = torch.from_numpy(synth.randn(203, (N, OC))).to(dev)
    dW0 = torch.from_numpy(synth.randn(204, (OC, IC), 0.01)).to(dev)
    db0 = torch.from_numpy(synth.randn(205, (OC,), 0.01)).to(dev)

    dx_ref = torch.empty(N, IC, device=dev)
    dW_ref, db_ref = dW0.clone(), db0.clone()
    g.matmul_backward(dx_ref, dW_ref, db_ref, dy, x, W)
    ref = [t.cpu().numpy() for t in (dx_ref, dW_ref, db_ref)]

    for call in range(2):
        dx = torch.full((N, IC), float("nan"), device=dev)
        dW, db = dW0.clone(), db0.clone()
        g.matmul_backward_noalloc(dx, dW, db, dy, x, W)
        got = [t.cpu().numpy() for t in (dx, dW, db)]
        assert np.isfinite(got[0]).all(), call
        assert rel_err(got[0], ref[0]) <= tol(OC), (call, "dx", rel_err(got[0], ref[0]))
        assert rel_err(got[1] - dW0.cpu().numpy(), ref[1] - dW0.cpu().numpy()) <= tol(N), (call, "dW")
        assert rel_err(got[2] - db0.cpu().numpy(), ref[2] - db0.cpu().numpy()) <= tol(N), (call, "db")


def test_noalloc_backward_rejects_shapes_beyond_its_scratch():
    import torch

    import gpt_train_step_02_b300 as g

    # ceil(N/64) * OC = 1025 * 1024 > 1,048,576 partials; the buffers are
    # allocated at full size all the same, so nothing could be out of bounds
    N, IC, OC = 64 * 1025, 4, 1024
    dev = torch.device("cuda", 0)
    x = torch.zeros(N, IC, device=dev)
    W = torch.zeros(OC, IC, device=dev)
    dy = torch.zeros(N, OC, device=dev)
    dx = torch.zeros(N, IC, device=dev)
    dW = torch.zeros(OC, IC, device=dev)
    db = torch.zeros(OC, device=dev)
    with pytest.raises(g.GPT2Error) as e:
        g.matmul_backward_noalloc(dx, dW, db, dy, x, W)
    assert e.value.status == g.GPT2_ERR_SHAPE
