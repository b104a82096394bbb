"""gemm_set_kernel_events: caller-owned CUDA events recorded around the main GEMM kernel of
a product (after its staging copies), which the benchmark uses to time that kernel alone."""
import ctypes

import pytest
import torch

import workloads as W
from gpu_util import oracle_rows, rel_err, tolerance

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import dense_tiled_gemm_05_gb300 as g
    from dense_tiled_gemm_05_gb300 import build as gbuild
    gbuild.build()
    return g


def test_kernel_events_bracket_the_main_kernel(g):
    # Exact fp32 splits both operands before its kernel runs: the events' interval lies
    # inside the whole call's and is shorter. A half-given pair is refused and leaves the
    # hook as it was; turning the hook off stops the recording.
    h = g.Gemm(0)
    p = W.fp32_square(2048, "exact", seed=31)
    a, b = p.A.cuda(), p.B.cuda()
    s0, s1, k0, k1 = (torch.cuda.Event(enable_timing=True) for _ in range(4))
    for ev in (k0, k1):
        ev.record()  # creates the CUDA events
    torch.cuda.synchronize()
    h.set_kernel_events(k0, k1)
    assert g.lib().gemm_set_kernel_events(h.handle, ctypes.c_void_p(k0.cuda_event), None) == 1
    assert h.plan(a, b, precision="exact")["path"] == "tcgen05_3xtf32"
    s0.record()
    c = h.matmul(a, b, precision="exact")
    s1.record()
    torch.cuda.synchronize()
    assert h.status() == 0
    whole, kernel = s0.elapsed_time(s1), k0.elapsed_time(k1)
    assert 0 < kernel < whole
    h.set_kernel_events()
    before = k1.elapsed_time(s1)
    h.matmul(a, b, precision="exact")
    torch.cuda.synchronize()
    assert k1.elapsed_time(s1) == before  # not recorded again
    rows = list(range(0, 2048, 67))
    C64, D = oracle_rows(p, rows)
    assert rel_err(c[rows], C64, D) <= tolerance(p)
    h.close()
