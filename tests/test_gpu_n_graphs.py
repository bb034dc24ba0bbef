"""GPU: the entry points inside CUDA graphs.  Every call is asynchronous on
the caller's stream and launches only stream-ordered work (kernels, and one
memset for the split tail's counters), so a captured sequence replays the
same work: the replayed results equal eager calls bit for bit.  The first
call on a device (one-time kernel attributes and cluster occupancy) is made
before the capture."""
import numpy as np
import pytest

import mixed_precision_matmul_gb300 as mpg
import synthetic

pytestmark = pytest.mark.gpu


def _capture(fn):
    import torch
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        out = fn()
    return g, out


@pytest.mark.parametrize("mode,dt,opts", [
    ("bf16", "bf16", {}),                                   # one-CTA tiles
    ("bf16", "bf16", {"cta_pair": 1, "tail_split": 1}),     # CTA pairs, split tail (memset + kernel)
    ("split3", "f32", {"prepass": 1}),                      # conversion pass, then the product
    ("tf32", "f32", {"splitk": 3}),                         # split-K partials and their reduction
])
def test_product_replays_like_eager_calls(mode, dt, opts):
    import torch
    mpg.build()
    m, n, k = 520, 300, 1000
    a = synthetic.normal((m, k), 181)
    b = synthetic.normal((k, n), 182)
    c0 = synthetic.normal((m, n), 183)
    td = {"bf16": torch.bfloat16, "f32": torch.float32}[dt]
    A = torch.from_numpy(a).cuda().to(td)
    B = torch.from_numpy(b).cuda().to(td)
    o = mpg.options(**opts)
    C_eager = torch.from_numpy(c0).cuda()
    mpg.gemm(A, B, C_eager, alpha=1.25, beta=0.5, mode=mode, opts=o)
    torch.cuda.synchronize()
    C_graph = torch.from_numpy(c0).cuda()
    g, _ = _capture(lambda: mpg.gemm(A, B, C_graph, alpha=1.25, beta=0.5, mode=mode, opts=o))
    for _ in range(3):                       # C = 1.25 AB + 0.5 C, applied again at each replay
        C_graph.copy_(torch.from_numpy(c0).cuda())
        g.replay()
        torch.cuda.synchronize()
        assert mpg.device_status() == mpg.OK
        assert np.array_equal(C_graph.cpu().numpy().view(np.uint32), C_eager.cpu().numpy().view(np.uint32))


def test_fused_attention_replays_like_eager_calls():
    import torch
    mpg.build()
    q = synthetic.normal((300, 128), 191)
    kk = synthetic.normal((2000, 128), 192).astype(np.float16)
    vv = synthetic.normal((2000, 128), 193).astype(np.float16)
    Q, K, V = (torch.from_numpy(x).cuda() for x in (q, kk, vv))
    O_eager = mpg.attention(Q, K, V, scale=0.1)
    torch.cuda.synchronize()
    O_graph = torch.zeros_like(O_eager)
    g, _ = _capture(lambda: mpg.attention(Q, K, V, O=O_graph, scale=0.1))
    g.replay()
    torch.cuda.synchronize()
    assert mpg.device_status() == mpg.OK
    assert np.array_equal(O_graph.cpu().numpy().view(np.uint32), O_eager.cpu().numpy().view(np.uint32))
