"""The matmul backward for callers that cannot allocate device memory.

Some callers have no way to hand the library a workspace. One example is a
plugin whose host application's allocator already owns all of the device's
memory. Another is a loop that must not call cudaMalloc, because cudaMalloc
can synchronise the device. For these callers,
``gpt2op_matmul_backward_noalloc`` takes its scratch from a fixed array in
the library's own device memory.

These tests check, through the C ABI, that the variant gives bitwise the
same dx, dW and dbias as ``gpt2op_matmul_backward`` with a caller workspace
(the same deterministic kernels run on the same inputs), and that both agree
with the oracle's matmul_backward within the fp32 matmul tolerance.  The check
runs on two calls in a row, so the second call runs on the scratch the first
one left behind; one case makes the second call smaller than the first, so
column-sum partials left over from the larger shape would show.  They also
check that a shape whose bias partials exceed the fixed array is rejected
before any device work.

The file is collected last, so a run that stops at its first failure has
already run every other test.
"""
import numpy as np
import pytest

import synth
from oracle import ref

pytestmark = pytest.mark.gpu

OPS = ref.ops(np.float32)

SHAPES = [  # (N rows, IC, OC) of the first call, N of the second call
    (256, 768, 768, 256),    # split-K products and a bias gradient
    (300, 96, 260, 300),     # ragged tiles
    (256, 3072, 768, 256),   # long K for the input gradient
    (700, 96, 260, 130),     # second call smaller: stale partials of the first would show
]


def rel_err(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return np.abs(a - b).max() / max(np.abs(b).max(), 1e-30)


def tol(K):
    """The tolerance of the fp32 matmul parity tests: 3xTF32 products are
    about 2^-20 relative; the fp32 accumulation error grows with K."""
    return 1e-5 if K <= 4096 else 1e-4


def case(N, IC, OC, seed):
    return (synth.randn(seed, (N, IC)), synth.randn(seed + 1, (OC, IC), 0.02), synth.randn(seed + 2, (N, OC)),
            synth.randn(seed + 3, (OC, IC), 0.01), synth.randn(seed + 4, (OC,), 0.01))


@pytest.mark.parametrize("N,IC,OC,N2", SHAPES)
def test_noalloc_backward_matches_workspace_backward_on_two_calls(N, IC, OC, N2):
    import torch

    import gpt_train_step_02_b300 as g

    dev = torch.device("cuda", 0)
    for call, (n, seed) in enumerate([(N, 201), (N2, 301)]):
        x, W, dy, dW0, db0 = case(n, IC, OC, seed)
        tx, tW, tdy = (torch.from_numpy(a).to(dev) for a in (x, W, dy))

        dx_ws = torch.empty(n, IC, device=dev)
        dW_ws, db_ws = torch.from_numpy(dW0).to(dev), torch.from_numpy(db0).to(dev)
        g.matmul_backward(dx_ws, dW_ws, db_ws, tdy, tx, tW)
        ws = [t.cpu().numpy() for t in (dx_ws, dW_ws, db_ws)]

        dx = torch.full((n, IC), float("nan"), device=dev)
        dW, db = torch.from_numpy(dW0).to(dev), torch.from_numpy(db0).to(dev)
        g.matmul_backward_noalloc(dx, dW, db, tdy, tx, tW)
        got = [t.cpu().numpy() for t in (dx, dW, db)]

        for name, a, b in zip(("dx", "dW", "db"), got, ws):
            assert np.array_equal(a, b), (call, name, rel_err(a, b))
        rdx, rdW, rdb = OPS.matmul_backward(dy, x, W, True)
        assert rel_err(got[0], rdx) <= tol(OC), (call, "dx", rel_err(got[0], rdx))
        assert rel_err(got[1] - dW0, rdW) <= tol(n), (call, "dW", rel_err(got[1] - dW0, rdW))
        assert rel_err(got[2] - db0, rdb) <= 1e-5, (call, "db", rel_err(got[2] - db0, rdb))


def test_noalloc_backward_rejects_shapes_beyond_its_scratch():
    import torch

    import gpt_train_step_02_b300 as g

    # ceil(N/64) * OC = 1025 * 2048 > 2,097,152 partials; the buffers are
    # allocated at full size all the same, so nothing could be out of bounds
    N, IC, OC = 64 * 1025, 4, 2048
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
