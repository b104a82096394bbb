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
    assert after["tile_m"] == (2 * r["tile_rows"] if r["cta_pair"] == 2 else 128)
    assert r["tile_rows"] == 128  # compute-bound: no shorter tiles tried
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


def test_tune_tries_shorter_pair_tiles(h):
    # bandwidth-bound (bf16 6000 x 128 x 4096): 96-row CTAs are among the candidates
    p = W.integer_problem(6000, 128, 4096, "bf16", seed=63, b_layout="col")
    a, b = to_device(p.A), to_device(p.B)
    r = h.tune(a, b, out_dtype="f32", iters=3)
    assert r["tile_rows"] in (96, 128)
    assert 0 < r["best_us"] <= r["default_us"]
    after = h.plan(a, b, out_dtype="f32")
    assert after["tile_m"] == (2 * r["tile_rows"] if r["cta_pair"] == 2 else 128)
    c = run_gpu(h, p)
    assert torch.equal(c.cpu().to(torch.int64), p.A.to(torch.int64) @ p.B.to(torch.int64))
    # forcing 96 rows as the tuner would: the same exact product
    h.tune_clear()
    h.set_option("tile_rows", 96)
    assert h.plan(a, b, out_dtype="f32")["tile_m"] == 192
    c = run_gpu(h, p)
    assert torch.equal(c.cpu().to(torch.int64), p.A.to(torch.int64) @ p.B.to(torch.int64))


def test_tune_single_candidate_paths(h):
    p = W.fp32_square(512, "exact")
    r = h.tune(to_device(p.A), to_device(p.B), out_dtype="f32", precision="exact", iters=1)
    assert r["candidates"] == 1 and r["best_us"] == r["default_us"]
