"""Products captured in a CUDA graph and replayed: split-K launches take their epoch from
device memory, so a replay (whose kernel parameters are frozen at capture) never accepts
the flags of the previous replay. Checked bit for bit with integer inputs that change
between replays, for the CTA-pair kernel and the exact-fp32 chunked kernel."""
import pytest
import torch

import workloads as W
from gpu_util import to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import dense_tiled_gemm_05_gb300 as g
    return g


@pytest.mark.parametrize("dtype,precision", [("bf16", "default"), ("f32", "exact")])
def test_split_k_graph_replays(g, dtype, precision):
    M, N, K = 1030, 530, 1200
    h = g.Gemm(0)
    h.set_option("stream_k", 2)
    p = W.integer_problem(M, N, K, dtype, seed=11, precision=precision)
    a, b = to_device(p.A), to_device(p.B)
    c = torch.empty((M, N), device="cuda")
    assert h.plan(a, b, out_dtype="f32", precision=precision)["split_tiles"] > 0
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for _ in range(2):  # workspaces sized, code loaded
            h.matmul(a, b, out=c, precision=precision)
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        h.matmul(a, b, out=c, precision=precision)
    for seed in (21, 22, 23, 24):
        q = W.integer_problem(M, N, K, dtype, seed=seed, precision=precision)
        a.copy_(q.A.cuda())
        b.copy_(q.B.cuda())
        graph.replay()
        torch.cuda.synchronize()
        assert h.status() == 0
        assert torch.equal(c.cpu().to(torch.int64), q.A.to(torch.int64) @ q.B.to(torch.int64))
    h.close()
