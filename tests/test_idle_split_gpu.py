"""Few tiles, long K: each tile's K-loop shared out over otherwise idle CTA pairs.

"Chapter 13: The Blocked Matmul Kernel" section 13.1 sums a tile's K-blocks into one fp32
accumulator. When a product has so few output tiles that most SMs would idle, the planner
cuts every tile's K-loop into a few pieces (about sqrt(K-blocks / 4) of them) on as many
CTA pairs; the pieces' fp32 sums are added by the tile's owner in a fixed order. The set
of products summed is unchanged, so integer-valued inputs stay exact; real inputs are
checked against the fp64 oracle with the section's tolerance, and two runs must agree bit
for bit (the order of the partial sums is fixed).
"""
import pytest
import torch

import workloads as W
from gpu_util import oracle_rows, rel_err, run_gpu, sample_rows, to_device, tolerance

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def h():
    import dense_tiled_gemm_05_gb300 as g
    from dense_tiled_gemm_05_gb300 import build as gbuild
    gbuild.build()
    hh = g.Gemm(0)
    yield hh
    hh.close()


def int_exact(c, p):
    return torch.equal(c.cpu().to(torch.int64), p.A.to(torch.int64) @ p.B.to(torch.int64))


@pytest.mark.parametrize("M,N,K,dtype,b_layout", [
    (256, 256, 8192, "bf16", "col"),     # one tile, six pieces
    (128, 128, 32768, "bf16", "col"),    # one tile, eleven pieces
    (1024, 128, 8192, "bf16", "col"),    # four tiles
    (1000, 300, 9000, "f16", "col"),     # ragged in M, N and K
    (100, 200, 20000, "bf16", "row"),    # shorter than one CTA's rows; N-major B
    (640, 136, 12345, "f16", "row"),     # ragged, staged operands
])
def test_idle_split_integer_exact(h, M, N, K, dtype, b_layout):
    p = W.integer_problem(M, N, K, dtype, seed=M + N + K, b_layout=b_layout)
    plan = h.plan(to_device(p.A), to_device(p.B), out_dtype="f32")
    assert plan["cta_pair"] == 1 and plan["split_tiles"] == plan["grid_m"] * plan["grid_n"], plan
    assert plan["ctas"] <= torch.cuda.get_device_properties(0).multi_processor_count
    c = run_gpu(h, p)
    assert int_exact(c, p)


@pytest.mark.parametrize("M,N,K,out_dtype", [(256, 256, 8192, "bf16"), (1000, 300, 9000, "f32"),
                                             (3000, 128, 8192, "bf16")])
def test_idle_split_real_vs_oracle(h, M, N, K, out_dtype):
    p = W.bf16_skinny(M=M, N=N, K=K, seed=K + 3)
    p = W.Problem(p.name, p.A, p.B, out_dtype, p.precision)
    plan = h.plan(to_device(p.A), to_device(p.B), out_dtype=out_dtype)
    assert plan["split_tiles"] > 0, plan
    c1 = run_gpu(h, p)
    c2 = run_gpu(h, p)
    assert torch.equal(c1, c2)
    rows = sample_rows(p.M, n_random=24)
    C64, D = oracle_rows(p, rows)
    assert rel_err(c1[rows], C64, D) <= tolerance(p)


def test_idle_split_tf32(h):
    A = W.make_operand(300, 8192, "f32", "row", 71)
    B = W.make_operand(8192, 200, "f32", "col", 72)
    p = W.Problem("tf32_idle_split", A, B, "f32", "tf32")
    plan = h.plan(to_device(p.A), to_device(p.B), out_dtype="f32", precision="tf32")
    assert plan["cta_pair"] == 1 and plan["split_tiles"] > 0, plan
    c = run_gpu(h, p)
    rows = sample_rows(p.M, n_random=24)
    C64, D = oracle_rows(p, rows)
    assert rel_err(c[rows], C64, D) <= tolerance(p)


def test_short_k_keeps_whole_tiles(h):
    # 64 K-blocks: no split; one 128-row tile of M keeps single-CTA tiles
    p = W.integer_problem(128, 4096, 4096, "bf16", seed=9, b_layout="col")
    plan = h.plan(to_device(p.A), to_device(p.B), out_dtype="f32")
    assert plan["cta_pair"] == 0 and plan["split_tiles"] == 0
    assert int_exact(run_gpu(h, p), p)
