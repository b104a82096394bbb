"""Shorter tiles of the CTA-pair kernel, and the once-read operand schedule.

Two schedule choices of the tensor-core kernels that leave each output element's sum, the
K-loop of "Chapter 13: The Blocked Matmul Kernel" section 13.1, the same set of products:

* rows per CTA (GEMM_OPT_TILE_ROWS): each CTA of a pair loads r <= 128 rows of A into the
  128-row MMA, and only those r accumulator lanes are stored; section 13.2's masks at the
  tile's edges then fall inside a warp (the epilogue stores the valid lanes only);
* an operand that one tile row or column reads alone is loaded as first-to-evict from L2 and
  whole tiles begin their K-loops at staggered K-blocks (the order of the K-blocks in the
  fp32 sum changes, not the set).

Integer-valued inputs make every order of the sum exact, so those cases are compared bit
for bit with the exact integer product; real-valued ones against the fp64 oracle within the
section's tolerance.
"""
import pytest
import torch

import workloads as W
from gpu_util import check_sums, oracle_rows, rel_err, run_gpu, sample_rows, to_device, tolerance

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    import dense_tiled_gemm_05_gb300 as g
    from dense_tiled_gemm_05_gb300 import build as gbuild
    gbuild.build()
    return g


def int_exact(c, p):
    return torch.equal(c.cpu().to(torch.int64), p.A.to(torch.int64) @ p.B.to(torch.int64))


def tile_edge_rows(M, r, n_random=24, seed=0):
    """Every CTA's first and last row for tiles of r rows per CTA, plus random rows."""
    rows = sample_rows(M, tile=r, n_random=n_random, seed=seed)
    rows += [min(t0 + r - 1, M - 1) for t0 in range(r, M, 2 * r)]
    rows += [t0 for t0 in range(r, M, 2 * r)]
    return sorted(set(rows))


@pytest.mark.parametrize("r", [64, 72, 104, 112, 120])
@pytest.mark.parametrize("b_layout", ["col", "row"])
def test_forced_rows_integer_exact(g, r, b_layout):
    h = g.Gemm(0)
    h.set_option("cta_pair", 2)  # rows per CTA are a property of the pair kernel
    h.set_option("tile_rows", r)
    # ragged M (tails inside a warp and inside a CTA), ragged N and K; K of 64 is one block
    for n, (M, N, K) in enumerate([(1000, 300, 1025), (2 * r * 3 + 17, 257, 64),
                                   (4099, 130, 2048), (r, 256, 200)]):
        p = W.integer_problem(M, N, K, "bf16", seed=300 + 7 * r + n, b_layout=b_layout)
        plan = h.plan(to_device(p.A), to_device(p.B), out_dtype="f32")
        assert plan["cta_pair"] == 1 and plan["tile_m"] == 2 * r, plan
        c = run_gpu(h, p)
        assert int_exact(c, p), (M, N, K)
    h.close()


@pytest.mark.parametrize("out_dtype", ["bf16", "f16", "f32"])
def test_forced_rows_real_vs_oracle(g, out_dtype):
    # TMA-store epilogue for the full warps, plain stores for the warp the tile ends in
    h = g.Gemm(0)
    h.set_option("cta_pair", 2)
    h.set_option("tile_rows", 104)
    p = W.bf16_skinny(M=3000, N=256, K=1500, seed=21)
    p = W.Problem(p.name, p.A, p.B, out_dtype, p.precision)
    plan = h.plan(to_device(p.A), to_device(p.B), out_dtype=out_dtype)
    assert plan["tile_m"] == 208 and plan["tma_store"] == 1
    c = run_gpu(h, p)
    rows = tile_edge_rows(p.M, 104)
    C64, D = oracle_rows(p, rows)
    assert rel_err(c[rows], C64, D) <= tolerance(p)
    s_err, tol = check_sums(p, c)
    assert s_err <= tol, s_err
    h.close()


def test_forced_rows_direct_epilogue(g):
    # A C row that does not end on 16 bytes (N = 301 fp32): every warp stores with plain
    # stores, the warp the tile ends in only its valid lanes.
    h = g.Gemm(0)
    h.set_option("cta_pair", 2)
    h.set_option("tile_rows", 88)
    p = W.integer_problem(1234, 301, 777, "f16", seed=77, b_layout="col")
    plan = h.plan(to_device(p.A), to_device(p.B), out_dtype="f32")
    assert plan["tma_store"] == 0 and plan["tile_m"] == 176
    c = run_gpu(h, p)
    assert int_exact(c, p)
    h.close()


def test_forced_rows_tf32(g):
    h = g.Gemm(0)
    h.set_option("cta_pair", 2)
    h.set_option("tile_rows", 96)
    A = W.make_operand(1111, 700, "f32", "row", 91)
    B = W.make_operand(700, 333, "f32", "col", 92)
    p = W.Problem("tf32_rows96", A, B, "f32", "tf32")
    plan = h.plan(to_device(p.A), to_device(p.B), out_dtype="f32", precision="tf32")
    assert plan["cta_pair"] == 1 and plan["tile_m"] == 192
    c = run_gpu(h, p)
    rows = tile_edge_rows(p.M, 96)
    C64, D = oracle_rows(p, rows)
    assert rel_err(c[rows], C64, D) <= tolerance(p)
    h.close()


@pytest.mark.parametrize("r", [80, 112])
def test_forced_rows_with_split_k(g, r):
    # Several rounds whose last ones are split along K: partial pieces store all 128
    # accumulator lanes to the workspace, owners add them, and only the tile's rows are
    # stored. Integer inputs stay exact; two runs agree bit for bit.
    h = g.Gemm(0)
    h.set_option("cta_pair", 2)  # rows per CTA are a property of the pair kernel
    h.set_option("tile_rows", r)
    h.set_option("stream_k", 2)
    h.set_option("max_ctas", 16)
    p = W.integer_problem(2000, 700, 3000, "bf16", seed=500 + r, b_layout="col")
    plan = h.plan(to_device(p.A), to_device(p.B), out_dtype="f32")
    assert plan["tile_m"] == 2 * r and plan["split_tiles"] > 0, plan
    c = run_gpu(h, p)
    assert int_exact(c, p)
    q = W.ragged(2000, 700, 3000, seed=r, dtype="bf16")
    c1, c2 = run_gpu(h, q), run_gpu(h, q)
    assert torch.equal(c1, c2)
    rows = tile_edge_rows(q.M, r)
    C64, D = oracle_rows(q, rows)
    assert rel_err(c1[rows], C64, D) <= tolerance(q)
    h.close()


def test_tile_rows_option_checks(g):
    h = g.Gemm(0)
    a = torch.empty(16384, 8192, dtype=torch.bfloat16, device="cuda")
    b = torch.empty(128, 8192, dtype=torch.bfloat16, device="cuda").t()
    for bad in (-8, 8, 56, 100, 129, 136, 256):
        with pytest.raises(g.GemmError) as e:
            h.set_option("tile_rows", bad)
        assert e.value.status == "GEMM_ERR_INVALID_ARG"
    # forced rows are taken as given, even on a product that fills every cluster
    h.set_option("tile_rows", 96)
    p = h.plan(torch.empty(8192, 8192, dtype=torch.bfloat16, device="cuda"),
               torch.empty(8192, 8192, dtype=torch.bfloat16, device="cuda").t(), sm_count=148)
    assert p["tile_m"] == 192 and p["grid_m"] == 43
    # refused where the kernel cannot take fewer rows: single-CTA tiles, an M-major A,
    # the chunked kernels
    h.set_option("cta_pair", 1)
    with pytest.raises(g.GemmError):
        h.plan(a, b)
    h.set_option("cta_pair", 0)
    a_col = torch.empty(8192, 1024, dtype=torch.bfloat16, device="cuda").t()  # 1024 x 8192
    with pytest.raises(g.GemmError) as e:
        h.plan(a_col, b)
    assert e.value.status == "GEMM_ERR_UNSUPPORTED"
    f = torch.empty(1024, 1024, device="cuda")
    with pytest.raises(g.GemmError):
        h.plan(f, f, precision="exact")
    with pytest.raises(g.GemmError):
        h.plan(f.half(), f.half(), out_dtype="f16", precision="f16acc")
    # forced split-K with default rows keeps 128 rows
    h.set_option("tile_rows", 0)
    h.set_option("stream_k", 2)
    p = h.plan(a, b, sm_count=148)
    assert p["tile_m"] == 256 and p["split_tiles"] > 0
    h.close()


@pytest.mark.parametrize("M,N,K,b_layout,once", [
    (5000, 100, 3000, "col", True),   # one tile column: A read once (pairs)
    (3000, 120, 2500, "row", True),   # one tile column, N-major B
    (200, 3000, 3000, "col", True),   # one tile row of pairs: B read once
    (100, 5000, 2000, "col", True),   # single-CTA tiles, one tile row: B read once
    (128, 128, 4096, "row", True),    # one tile in all: both read once
    (1000, 1000, 1000, "col", False),  # neither
])
def test_once_read_operands_integer_exact(g, M, N, K, b_layout, once):
    h = g.Gemm(0)
    p = W.integer_problem(M, N, K, "bf16", seed=M + N + K, b_layout=b_layout)
    plan = h.plan(to_device(p.A), to_device(p.B), out_dtype="f32")
    assert (plan["grid_m"] == 1 or plan["grid_n"] == 1) == once, plan
    c = run_gpu(h, p)
    assert int_exact(c, p)
    # real-valued, bf16 out, against the oracle
    q = W.bf16_skinny(M=M, N=N, K=K, seed=M + 1, b_layout=b_layout)
    c = run_gpu(h, q)
    rows = tile_edge_rows(q.M, plan["tile_m"] // (2 if plan["cta_pair"] else 1), seed=M)
    C64, D = oracle_rows(q, rows)
    assert rel_err(c[rows], C64, D) <= tolerance(q)
    h.close()


def test_skinny_rows_full_size(g):
    # bf16 16384 x 128 x 8192, the bench's skinny shape, on 112-row CTAs (74 tiles)
    h = g.Gemm(0)
    h.set_option("tile_rows", 112)
    p = W.bf16_skinny()
    plan = h.plan(to_device(p.A), to_device(p.B), out_dtype="bf16")
    assert plan["tile_m"] == 224 and plan["grid_m"] == 74
    c = run_gpu(h, p)
    r = plan["tile_m"] // 2
    rows = tile_edge_rows(p.M, r, n_random=16)
    C64, D = oracle_rows(p, rows)
    assert rel_err(c[rows], C64, D) <= tolerance(p)
    s_err, tol = check_sums(p, c)
    assert s_err <= tol, s_err
    h.close()
