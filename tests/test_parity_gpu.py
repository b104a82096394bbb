"""GPU parity: the library (through its C ABI) against the CPU oracle, element by
element on the seeded workloads, on every kernel path, layout and dtype, plus the
edge cases of the method (ragged M/N/K, K == 0, empty outputs, padded and
misaligned operands, untouched bytes outside C, determinism)."""
import itertools

import numpy as np
import pytest
import torch

import workloads as W
from gpu_util import (check_full, check_sampled, check_sums, oracle_rows, rel_err, run_gpu,
                      sample_rows, to_device, tolerance)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def h():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import dense_tiled_gemm_05_gb300 as g
    from dense_tiled_gemm_05_gb300 import build as gbuild
    gbuild.build()
    return g.Gemm(0)


def full_check(h, p, **kw):
    c = run_gpu(h, p, **kw)
    C64, D = oracle_rows(p)
    err = rel_err(c, C64, D)
    assert err <= tolerance(p), "%s: rel err %.3g > %.3g" % (p.name, err, tolerance(p))
    return c, err


# ------------------------------------------------------------ the pages' cases

@pytest.mark.parametrize("dtype,precision", [("f32", "exact"), ("f16", "default"),
                                             ("bf16", "default"), ("f32", "tf32")])
def test_two_by_two(h, dtype, precision):
    p = W.two_by_two(dtype)
    p.precision = precision
    p.out_dtype = "f32"
    c = run_gpu(h, p)
    assert c.cpu().tolist() == [[19.0, 22.0], [43.0, 50.0]]


def test_small_exact_8x8x8_on_4x4x4_tiles(h):
    p = W.small_exact()
    plan = h.plan(to_device(p.A), to_device(p.B), out_dtype="f32", precision="exact")
    assert (plan["tile_m"], plan["grid_m"], plan["grid_n"], plan["k_iters"]) == (4, 2, 2, 2)
    full_check(h, p)


@pytest.mark.parametrize("M,K,N", [(8, 8, 8), (5, 7, 6)])
@pytest.mark.parametrize("dtype,precision", [("f32", "exact"), ("f32", "tf32"),
                                             ("f16", "default")])
def test_arange_examples(h, M, K, N, dtype, precision):
    p = W.arange_tenths(M, K, N, dtype)
    p.precision, p.out_dtype = precision, "f32"
    full_check(h, p)


@pytest.mark.parametrize("dtype,precision", [("f32", "exact"), ("f32", "tf32"),
                                             ("f16", "default"), ("bf16", "default")])
def test_sentinel_k_mask(h, dtype, precision):
    # Operands sliced from parents whose k >= 5 columns/rows hold 999: the library must
    # read none of them (the missing-K-mask failure would add ~2,994,003 everywhere).
    p = W.sentinel_padded(dtype=dtype)
    p.precision, p.out_dtype = precision, "f32"
    c, _ = full_check(h, p)
    assert float(c.abs().max()) < 20.0


# ----------------------------------------------------------------- ragged sweep

def test_ragged_sweep_all_216(h):
    worst, failures = 0.0, []
    for (M, N, K) in W.ragged_combos():
        p = W.ragged(M, N, K)
        c = run_gpu(h, p)
        C64, D = oracle_rows(p)
        err = rel_err(c, C64, D)
        worst = max(worst, err)
        if err > tolerance(p):
            failures.append(((M, N, K), err))
    assert not failures, failures[:10]
    assert worst < 1e-2


def test_ragged_sweep_fp32_exact_all_216(h):
    # fp32 inputs in exact mode: the accuracy gate for running exact fp32 on the tensor
    # cores as three tf32 products (max |err| / sum |a b| <= 1e-6 on every combination).
    worst, failures = 0.0, []
    for (M, N, K) in W.ragged_combos():
        p = W.ragged(M, N, K, dtype="f32")
        c = run_gpu(h, p)
        C64, D = oracle_rows(p)
        err = rel_err(c, C64, D)
        worst = max(worst, err)
        if err > tolerance(p):
            failures.append(((M, N, K), err))
    assert not failures, failures[:10]
    print("worst exact-mode relative error over the sweep: %.3g" % worst)


@pytest.mark.parametrize("M,N,K", [(1025, 17, 1023), (127, 1000, 1025), (17, 1023, 1000),
                                   (1, 1025, 127)])
def test_ragged_guard_bands(h, M, N, K):
    # A and B live in padded parents whose tails hold 999; C lives in a NaN-filled parent
    # with a wider row pitch. The result must equal the zero-tailed run bit for bit and
    # every byte of C's parent outside [0, M) x [0, N) must keep its NaN pattern.
    seed = 7 * M + N + K
    results = []
    for tail in (0.0, 999.0):
        A = W.make_operand(M, K, "f16", "row", seed, ld_pad=13)
        B = W.make_operand(K, N, "f16", "row", seed + 1, ld_pad=9)
        A.as_strided((M, 13), (A.stride(0), 1), A.storage_offset() + K).fill_(tail)
        B.as_strided((K, 9), (B.stride(0), 1), B.storage_offset() + N).fill_(tail)
        # C at an odd offset and pitch (plain-store epilogue), then at a 16-byte aligned
        # offset and pitch (TMA-store epilogue, clipped by the tensor map).
        for col0, pitch in ((2, N + 5), (4, (N + 8 + 3) // 4 * 4)):
            parent = torch.full((M + 2, pitch), float("nan"), dtype=torch.float32, device="cuda")
            out = parent[1:M + 1, col0:col0 + N]
            c = run_gpu(h, W.Problem("guard", A, B, "f32"), out=out)
            mask = torch.ones_like(parent, dtype=torch.bool)
            mask[1:M + 1, col0:col0 + N] = False
            bad = (mask & ~torch.isnan(parent)).nonzero()
            assert bad.numel() == 0, "C pitch %d offset %d: guard cells written, e.g. %s" % (
                pitch, col0, bad[:6].tolist())
            results.append(c.cpu())
        if tail == 999.0:
            C64, D = oracle_rows(W.Problem("guard", A, B, "f32"))
            assert rel_err(c, C64, D) <= 1e-2
    assert all(torch.equal(results[0], r) for r in results[1:])


# --------------------------------------------------- integer exactness (P7)

INT_SHAPES = [(1, 1, 1), (128, 256, 64), (129, 257, 65), (300, 520, 1025), (777, 33, 200),
              (64, 600, 8), (1000, 1000, 17)]


@pytest.fixture(scope="module", params=[(1, 256), (1, 128), (2, 256), (2, 128)],
                ids=["cta128x256", "cta128x128", "pair256x256", "pair256x128"])
def h_tiles(request, h):
    """A handle forced to one tile kind: single-CTA (128 rows) or CTA-pair (256 rows),
    128 or 256 columns wide."""
    import dense_tiled_gemm_05_gb300 as g
    hh = g.Gemm(0)
    hh.set_option("cta_pair", request.param[0])
    hh.set_option("block_n", request.param[1])
    yield hh
    hh.close()


@pytest.mark.parametrize("dtype,precision", [("bf16", "default"), ("f16", "default"),
                                             ("f32", "tf32"), ("f32", "exact")])
@pytest.mark.parametrize("a_layout,b_layout", list(itertools.product(["row", "col"], repeat=2)))
def test_integer_inputs_bit_exact(h_tiles, dtype, precision, a_layout, b_layout):
    for n, (M, N, K) in enumerate(INT_SHAPES):
        p = W.integer_problem(M, N, K, dtype, seed=100 + n, a_layout=a_layout,
                              b_layout=b_layout, precision=precision, ld_pad=n % 3)
        c = run_gpu(h_tiles, p)
        ref = p.A.to(torch.int64) @ p.B.to(torch.int64)
        assert torch.equal(c.cpu().to(torch.int64), ref), (M, N, K)
        assert torch.equal(c.cpu(), ref.to(torch.float32))


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_fma_kernel_integer_exact(h, dtype):
    import dense_tiled_gemm_05_gb300 as g
    h2 = g.Gemm(0)
    h2.set_option("force_path", 2)
    for n, (M, N, K) in enumerate([(1, 1, 1), (129, 257, 65), (300, 200, 1025), (8, 8, 8)]):
        for al, bl in itertools.product(["row", "col"], repeat=2):
            p = W.integer_problem(M, N, K, dtype, seed=300 + n, a_layout=al, b_layout=bl)
            assert h2.plan(to_device(p.A), to_device(p.B), out_dtype="f32",
                           precision=p.precision)["path"] == "fma"
            c = run_gpu(h2, p)
            assert torch.equal(c.cpu().to(torch.int64), p.A.to(torch.int64) @ p.B.to(torch.int64))
    h2.close()


@pytest.mark.parametrize("out_dtype", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("in_dtype", ["f16", "bf16"])
def test_output_dtypes_round_once(h, in_dtype, out_dtype):
    # Integer inputs keep the fp32 accumulator exact; the only rounding is the final one,
    # round-to-nearest-even into the output type.
    p = W.integer_problem(300, 260, 1000, in_dtype, seed=5, out_dtype=out_dtype)
    c = run_gpu(h, p)
    exact = (p.A.to(torch.int64) @ p.B.to(torch.int64)).to(torch.float64)
    expect = exact.to(torch.float32).to(W.TORCH_DTYPES[out_dtype])
    assert c.dtype == W.TORCH_DTYPES[out_dtype]
    assert torch.equal(c.cpu(), expect)


def test_accumulation_precision_example(h):
    # fp16 in, fp32 accumulate, fp16 out (the chapter's 4 x 1024 x 4 comparison): one
    # rounding at the store, so the result is the fp16 rounding of the fp32 sum.
    import oracle
    p = W.accumulation_13_3_1()
    c = run_gpu(h, p).double().cpu().numpy()
    C64, _ = oracle_rows(p)
    r16 = oracle.round_to(C64, "f16")
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(C64), 2.0 ** -14))) - 10)
    assert np.all(np.abs(c - r16) <= ulp)  # at most one fp16 step from the exact rounding
    assert np.max(np.abs(c - C64)) <= 9.737179152580211e-05 + ulp.max()


# --------------------------------------------------------- degenerate shapes

def test_k_zero_writes_zeros_and_empty_is_noop(h):
    a = torch.empty(37, 0, dtype=torch.bfloat16, device="cuda")
    b = torch.empty(0, 45, dtype=torch.bfloat16, device="cuda")
    out = torch.full((37, 45), float("nan"), dtype=torch.float32, device="cuda")
    h.matmul(a, b, out=out)
    assert h.status() == 0
    assert torch.equal(out, torch.zeros_like(out)) and not torch.signbit(out).any()
    out2 = torch.full((0, 45), 1.0, device="cuda")
    h.matmul(torch.empty(0, 8, dtype=torch.float16, device="cuda"),
             torch.empty(8, 45, dtype=torch.float16, device="cuda"), out=out2)
    assert h.status() == 0


def test_misaligned_operands_are_staged(h):
    # Operands starting 2 bytes past an aligned address: TMA cannot read them in place.
    M, N, K = 200, 300, 260
    for n, (al, bl) in enumerate(itertools.product(["row", "col"], repeat=2)):
        p = W.integer_problem(M, N, K, "bf16", seed=40 + n, a_layout=al, b_layout=bl)
        a = to_device(p.A)
        b = to_device(p.B)
        abuf = torch.empty(a.numel() + 8, dtype=a.dtype, device="cuda")
        bbuf = torch.empty(b.numel() + 8, dtype=b.dtype, device="cuda")
        a2 = torch.as_strided(abuf, a.shape, a.stride(), 1)
        b2 = torch.as_strided(bbuf, b.shape, b.stride(), 1)
        a2.copy_(a)
        b2.copy_(b)
        plan = h.plan(a2, b2, out_dtype="f32")
        assert plan["stage_a"] == 1 and plan["stage_b"] == 1
        c = h.matmul(a2, b2, out_dtype="f32")
        assert h.status() == 0
        ref = p.A.to(torch.int64) @ p.B.to(torch.int64)
        assert torch.equal(c.cpu().to(torch.int64), ref)


# ------------------------------------------------- schedule and determinism

def test_schedule_options_do_not_change_bits(h):
    # With whole tiles only, every output tile is the same K-loop whatever the raster order,
    # grid size or staging: the bits cannot depend on the schedule. (Split-K changes the
    # fp32 summation order of the split tiles; it is covered by its own tests.)
    import dense_tiled_gemm_05_gb300 as g
    p = W.bf16_square(1024)
    a, b = to_device(p.A), to_device(p.B)
    h0 = g.Gemm(0)
    h0.set_option("stream_k", 1)
    base = h0.matmul(a, b)
    assert h0.status() == 0
    h0.close()
    for opts in ({"max_ctas": 3}, {"group_m": 1}, {"group_m": 5, "max_ctas": 17},
                 {"force_staging": 1}):
        h2 = g.Gemm(0)
        h2.set_option("stream_k", 1)
        for k, v in opts.items():
            h2.set_option(k, v)
        c = h2.matmul(a, b)
        assert h2.status() == 0
        assert torch.equal(c, base), opts
        h2.close()
    C64, D = oracle_rows(p)
    assert rel_err(base, C64, D) <= 1e-2


@pytest.mark.parametrize("cta_pair,max_ctas", [(1, 7), (2, 6)])
def test_mid_size_full_compare_many_tiles_per_cta(h, cta_pair, max_ctas):
    import dense_tiled_gemm_05_gb300 as g
    h2 = g.Gemm(0)
    h2.set_option("cta_pair", cta_pair)
    h2.set_option("max_ctas", max_ctas)  # many tiles per CTA: both TMEM buffers, many phases
    for p in (W.integer_problem(2048, 1100, 1000, "bf16", seed=9, b_layout="col"),
              W.integer_problem(1500, 1024, 700, "f32", seed=10, precision="tf32")):
        c = run_gpu(h2, p)
        ref = p.A.to(torch.int64) @ p.B.to(torch.int64)
        assert torch.equal(c.cpu().to(torch.int64), ref)
    h2.close()


@pytest.mark.parametrize("M,N,K,max_ctas", [(2048, 2048, 2048, 0), (1500, 1300, 700, 10),
                                            (600, 600, 1000, 16), (256, 256, 8192, 0),
                                            (1030, 530, 1200, 8)])
def test_split_k_integer_exact(h, M, N, K, max_ctas):
    # Shapes whose last round of tiles is split along K: pieces of tiles are summed by
    # their owners from fp32 partials in a fixed order. Integer inputs keep every partial
    # exact, so the result must match the int64 product bit for bit. (256 x 256 x 8192 is
    # a single tile shared by every cluster: one owner adds dozens of partials.)
    import dense_tiled_gemm_05_gb300 as g
    h2 = g.Gemm(0)
    h2.set_option("cta_pair", 2)
    h2.set_option("block_n", 256)
    h2.set_option("stream_k", 2)  # split whenever the schedule allows, even for small shapes
    if max_ctas:
        h2.set_option("max_ctas", max_ctas)
    p = W.integer_problem(M, N, K, "bf16", seed=M + K, b_layout="col")
    plan = h2.plan(to_device(p.A), to_device(p.B), out_dtype="f32")
    assert plan["split_tiles"] > 0, plan
    for _ in range(2):  # twice: the second launch reuses the workspace with a new epoch
        c = run_gpu(h2, p)
        assert torch.equal(c.cpu().to(torch.int64), p.A.to(torch.int64) @ p.B.to(torch.int64))
    h2.close()


def test_split_k_matches_whole_tiles_and_is_deterministic(h):
    import dense_tiled_gemm_05_gb300 as g
    p = W.bf16_square(4096)
    a, b = to_device(p.A), to_device(p.B)
    assert h.plan(a, b)["split_tiles"] > 0
    c1 = h.matmul(a, b)
    c2 = h.matmul(a, b)
    assert h.status() == 0
    assert torch.equal(c1, c2)  # fixed reduction order: bitwise repeatable
    whole = g.Gemm(0)
    whole.set_option("stream_k", 1)
    assert whole.plan(a, b)["split_tiles"] == 0
    c3 = whole.matmul(a, b)
    assert whole.status() == 0
    whole.close()
    rows = list(range(0, 4096, 97))
    C64, D = oracle_rows(p, rows)
    assert rel_err(c1[rows], C64, D) <= 1e-2 and rel_err(c3[rows], C64, D) <= 1e-2
    # the two schedules only differ in fp32 summation order before the bf16 rounding
    assert float((c1.float() - c3.float()).abs().max()) <= 2 * 2.0 ** -8 * float(c3.float().abs().max())


def test_deterministic(h):
    p = W.bf16_square(2048)
    a, b = to_device(p.A), to_device(p.B)
    c1 = h.matmul(a, b)
    c2 = h.matmul(a, b)
    assert h.status() == 0
    assert torch.equal(c1, c2)


# ------------------------------------------------------- full-size configs
#
# Every element of every full-size product is compared with the oracle's fp64 product
# (the whole 8192^3 takes about 15 s on the host's cores), plus every row and column sum.

_ORACLE = {}


def oracle_full(p):
    """The oracle's full (C, D) for a workload; fp32 inputs shared by both precision modes
    are computed once."""
    key = (p.name.replace("_tf32", "").replace("_exact", ""), p.M, p.N, p.K)
    if key not in _ORACLE:
        _ORACLE.clear()  # one full-size result held at a time (8192^2 fp64 is 1 GB)
        _ORACLE[key] = oracle_rows(p)
    return _ORACLE[key]


def full_size_check(p, c):
    err = check_full(p, c, oracle_full(p))
    assert err <= tolerance(p), "%s: rel err %.3g > %.3g" % (p.name, err, tolerance(p))
    s_err, tol = check_sums(p, c)
    assert s_err <= tol, s_err
    return err


def test_bf16_4096_col_major_b(h):
    p = W.bf16_square(4096)
    full_size_check(p, run_gpu(h, p))


@pytest.mark.parametrize("precision,force_path", [("tf32", 0), ("exact", 0), ("exact", 2)],
                         ids=["tf32", "exact_3xtf32", "exact_fma"])
def test_fp32_4096_modes(h, precision, force_path):
    import dense_tiled_gemm_05_gb300 as g
    p = W.fp32_square(4096, precision)
    h2 = g.Gemm(0)
    h2.set_option("force_path", force_path)
    c = run_gpu(h2, p)
    h2.close()
    full_size_check(p, c)


@pytest.mark.parametrize("a_layout,b_layout", [("row", "row"), ("col", "col"), ("col", "row")])
def test_tf32_mn_major_in_place_and_transposed(h, a_layout, b_layout):
    # An MN-major fp32 operand in tf32 mode is read in place by the tensor cores (128-byte
    # swizzle with 32-byte atoms); GEMM_OPT_TF32_TRANSPOSE = 1 copies it K-major first.
    # Both are compared with the oracle on a ragged problem of several tiles, and with the
    # exact integer product.
    import dense_tiled_gemm_05_gb300 as g
    A = W.make_operand(1500, 1000, "f32", a_layout, 61)
    B = W.make_operand(1000, 1300, "f32", b_layout, 62)
    p = W.Problem("tf32_%s_%s" % (a_layout, b_layout), A, B, "f32", "tf32")
    q = W.integer_problem(700, 900, 1000, "f32", seed=63, a_layout=a_layout, b_layout=b_layout,
                          precision="tf32")
    C64, D = oracle_rows(p)
    outs = []
    for transpose in (0, 1):
        h2 = g.Gemm(0)
        h2.set_option("tf32_transpose", transpose)
        plan = h2.plan(to_device(p.A), to_device(p.B), out_dtype="f32", precision="tf32")
        assert plan["a_mn_major"] == (a_layout == "col" and not transpose)
        assert plan["b_mn_major"] == (b_layout == "row" and not transpose)
        assert plan["stage_b"] == (b_layout == "row" and transpose == 1)
        c = run_gpu(h2, p)
        assert rel_err(c, C64, D) <= tolerance(p)
        outs.append(c)
        ci = run_gpu(h2, q)
        assert torch.equal(ci.cpu().to(torch.int64), q.A.to(torch.int64) @ q.B.to(torch.int64))
        h2.close()
    scale = torch.from_numpy(D).to(outs[0].device).clamp_min(1e-30)
    assert float(((outs[0].double() - outs[1].double()).abs() / scale).max()) <= 2 * tolerance(p)


def test_bf16_8192(h):
    p = W.bf16_square(8192, seed=5)
    c = run_gpu(h, p)
    full_size_check(p, c)
    # the tile-boundary rows (0, 127, 128, 255 mod 256) once more through the row sampler
    assert check_sampled(p, c) <= tolerance(p)


def test_bf16_skinny(h):
    p = W.bf16_skinny()
    full_size_check(p, run_gpu(h, p))


@pytest.mark.parametrize("block_n", [128, 256])
@pytest.mark.parametrize("stream_k", [1, 2])
def test_wide_stages_integer_exact(block_n, stream_k):
    # Two 128-byte K-blocks per pipeline stage: K = 64 (the second block entirely past K,
    # read as zeros), ragged K, and K long enough for split-K pieces of 128-wide K-blocks.
    import dense_tiled_gemm_05_gb300 as g
    h2 = g.Gemm(0)
    h2.set_option("stage_k", 2)
    h2.set_option("block_n", block_n)
    h2.set_option("stream_k", stream_k)
    for n, (M, N, K) in enumerate([(300, 257, 64), (513, 300, 1025), (1030, 530, 1200),
                                   (256, 256, 8192)]):
        p = W.integer_problem(M, N, K, "bf16", seed=40 + n, b_layout="col")
        plan = h2.plan(to_device(p.A), to_device(p.B), out_dtype="f32")
        assert plan["tile_k"] == 128 and plan["stages"] == (3 if block_n == 256 else 4)
        c = run_gpu(h2, p)
        assert torch.equal(c.cpu().to(torch.int64), p.A.to(torch.int64) @ p.B.to(torch.int64))
    # operands the wide stages do not take are refused, not silently narrowed
    p = W.integer_problem(300, 200, 64, "bf16", seed=49)  # row-major B: MN-major
    with pytest.raises(g.GemmError):
        run_gpu(h2, p)
    h2.close()


@pytest.mark.parametrize("M,N,K,max_ctas", [(1030, 530, 1200, 0), (600, 600, 1000, 16),
                                            (256, 256, 4096, 0), (1500, 1300, 700, 10)])
def test_exact_split_k(M, N, K, max_ctas):
    # Exact fp32 with the last rounds split along K: partial pieces store their fp32
    # register sums, owners add them in worker order. Integer inputs must stay bit exact;
    # real inputs within the exact-mode bound; two runs bitwise equal.
    import dense_tiled_gemm_05_gb300 as g
    h2 = g.Gemm(0)
    h2.set_option("stream_k", 2)
    if max_ctas:
        h2.set_option("max_ctas", max_ctas)
    p = W.integer_problem(M, N, K, "f32", seed=M + 3 * K)
    plan = h2.plan(to_device(p.A), to_device(p.B), out_dtype="f32", precision="exact")
    assert plan["path"] == "tcgen05_3xtf32" and plan["split_tiles"] > 0, plan
    c = run_gpu(h2, p)
    assert torch.equal(c.cpu().to(torch.int64), p.A.to(torch.int64) @ p.B.to(torch.int64))
    q = W.ragged(M, N, K, seed=K, dtype="f32")
    c1 = run_gpu(h2, q)
    c2 = run_gpu(h2, q)
    assert torch.equal(c1, c2)
    rows = sample_rows(q.M, n_random=16)
    C64, D = oracle_rows(q, rows)
    assert rel_err(c1[rows], C64, D) <= tolerance(q)
    h2.close()


def test_north_star_signature_gemm_run(h):
    # gemm_run: the plain C signature (row-major A and B, legacy default stream), called
    # through ctypes with raw device pointers, on the pages' 2 x 2 check, a ragged fp16
    # problem and an fp32 exact one.
    import ctypes
    import dense_tiled_gemm_05_gb300 as g
    L = g.lib()
    for p in (W.two_by_two("f32"), W.ragged(1000, 17, 1025, seed=5), W.small_exact()):
        a, b = to_device(p.A.contiguous()), to_device(p.B.contiguous())
        c = torch.full((p.M, p.N + 3), float("nan"), device="cuda")
        code = L.gemm_run(h.handle, p.M, p.N, p.K, ctypes.c_void_p(a.data_ptr()), p.K,
                          ctypes.c_void_p(b.data_ptr()), p.N, ctypes.c_void_p(c.data_ptr()),
                          p.N + 3, g._dtype_code(a.dtype), g._dtype_code("f32"),
                          g.PREC[p.precision])
        assert code == 0
        torch.cuda.synchronize()
        assert h.status() == 0
        C64, D = oracle_rows(p)
        assert rel_err(c[:, :p.N], C64, D) <= tolerance(p)
        assert torch.isnan(c[:, p.N:]).all()
        if p.M == 2:  # the pages' printed single-tile result, bit for bit
            assert torch.equal(c[:, :2].cpu(), torch.tensor([[19.0, 22.0], [43.0, 50.0]]))


@pytest.mark.parametrize("dtype,precision", [("bf16", "default"), ("f16", "default"),
                                             ("f32", "tf32")])
@pytest.mark.parametrize("a_layout,b_layout", [("col", "row"), ("row", "row"), ("col", "col")])
@pytest.mark.parametrize("block_n,stream_k", [(256, 1), (256, 2), (128, 0)])
def test_mn_major_panel_loads_integer_exact(h, dtype, precision, a_layout, b_layout, block_n,
                                            stream_k):
    # CTA pairs load an MN-major operand whose M or N is a whole number of 128-byte panels
    # with one 3D copy a stage (all of a CTA's panels at once); other extents keep one 2D
    # copy a panel. Both must give the exact integer product: extents that are and are not
    # whole panels (32 tf32 or 64 16-bit elements), ragged K, split-K pieces.
    import dense_tiled_gemm_05_gb300 as g
    h2 = g.Gemm(0)
    h2.set_option("cta_pair", 2)
    h2.set_option("block_n", block_n)
    h2.set_option("stream_k", stream_k)
    shapes = [(512, 512, 1000), (384, 320, 129), (256, 96, 64), (1024, 2048, 777),
              (640, 192, 1025), (300, 130, 200)]
    for n, (M, N, K) in enumerate(shapes):
        p = W.integer_problem(M, N, K, dtype, seed=900 + n, a_layout=a_layout,
                              b_layout=b_layout, precision=precision)
        plan = h2.plan(to_device(p.A), to_device(p.B), out_dtype="f32", precision=precision)
        assert plan["cta_pair"] == 1 and plan["tile_n"] == block_n, plan
        c = run_gpu(h2, p)
        assert torch.equal(c.cpu().to(torch.int64), p.A.to(torch.int64) @ p.B.to(torch.int64)), (
            M, N, K)
    h2.close()
