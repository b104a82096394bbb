"""gemm_tune: the measured choice of tile shape, split-K, stage width and raster group for
one problem signature, kept on the handle and used by later calls with that signature."""
import pytest
import torch

import workloads as W
from gpu_util import run_gpu, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture()
def h():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import dense_tiled_gemm_05_gb300 as g
    hh = g.Gemm(0)
    yield hh
    hh.close()


def test_tune_keeps_the_fastest_and_applies_it(h):
    p = W.integer_problem(2048, 2048, 1024, "bf16", seed=61, b_layout="col")
    a, b = to_device(p.A), to_device(p.B)
    before = h.plan(a, b, out_dtype="f32")
    r = h.tune(a, b, out_dtype="f32", iters=3)
    assert r["candidates"] >= 8
    assert 0 < r["best_us"] <= r["default_us"]
    after = h.plan(a, b, out_dtype="f32")
    assert after["tile_n"] == r["block_n"] and after["cta_pair"] == (r["cta_pair"] == 2)
    assert after["tile_k"] == 64 * r["stage_k"]
    # the tuned configuration computes the same exact integer product
    c = run_gpu(h, p)
    assert torch.equal(c.cpu().to(torch.int64), p.A.to(torch.int64) @ p.B.to(torch.int64))
    # another signature keeps the planner's own choice; clearing restores the default
    q = W.integer_problem(2048, 2048, 1088, "bf16", seed=62, b_layout="col")
    qa, qb = to_device(q.A), to_device(q.B)
    import dense_tiled_gemm_05_gb300 as g
    assert h.plan(qa, qb, out_dtype="f32") == g.Gemm(0).plan(qa, qb, out_dtype="f32")
    h.tune_clear()
    assert h.plan(a, b, out_dtype="f32") == before


def test_tune_single_candidate_paths(h):
    p = W.fp32_square(512, "exact")
    r = h.tune(to_device(p.A), to_device(p.B), out_dtype="f32", precision="exact", iters=1)
    assert r["candidates"] == 1 and r["best_us"] == r["default_us"]
