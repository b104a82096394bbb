"""Pins for the CPU oracle: each test ties it to something other than itself.

The values come from the pages (golden files under tests/golden, each with its
citation), from closed forms, from exact integer arithmetic, from IEEE format
definitions, and from invariants of the product (identity, zero, transposition,
tile-order independence). A plausible slip anywhere in the oracle -- a dropped
term, a wrong sign, a swapped index, a transposed operand, a bad decoder or an
off-by-one in the K range -- fails at least one of them.
"""
import itertools

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from workloads import storage_numpy


def run_oracle(p, rows=None, threads=0):
    a, al, lda = storage_numpy(p.A)
    b, bl, ldb = storage_numpy(p.B)
    return oracle.gemm_f64(a, b, p.M, p.N, p.K, lda=lda, ldb=ldb, a_dtype=p.in_dtype,
                           b_dtype=W.dtype_name(p.B.dtype), a_layout=al, b_layout=bl, rows=rows,
                           threads=threads)


def as_layout(x, layout):
    """Same logical values, stored row- or column-major."""
    return x.contiguous() if layout == "row" else x.t().contiguous().t()


# --------------------------------------------------------------- page values

@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16", "f64"])
@pytest.mark.parametrize("a_layout,b_layout", list(itertools.product(["row", "col"], repeat=2)))
def test_two_by_two(golden, dtype, a_layout, b_layout):
    g = golden("two_by_two.txt")
    p = W.two_by_two(dtype)
    assert p.A.double().flatten().tolist() == g["A"][0]
    assert p.B.double().flatten().tolist() == g["B"][0]
    p.A, p.B = as_layout(p.A, a_layout), as_layout(p.B, b_layout)
    C, D = run_oracle(p)
    assert C.flatten().tolist() == g["C"][0]
    assert D.flatten().tolist() == g["C"][0]  # all products positive


def closed_form(M, K, N):
    """C for A[i,k] = 0.1(K i + k), B[k,j] = 0.1(N k + j), summed symbolically over k."""
    S1 = K * (K - 1) / 2
    S2 = (K - 1) * K * (2 * K - 1) / 6
    i = np.arange(M)[:, None].astype(np.float64)
    j = np.arange(N)[None, :].astype(np.float64)
    return 0.01 * (K * N * S1 * i + K * K * i * j + N * S2 + S1 * j)


@pytest.mark.parametrize("M,K,N", [(8, 8, 8), (5, 7, 6), (4, 5, 4), (3, 1, 9)])
def test_arange_closed_form(M, K, N):
    # Chapter 13, Worked Examples 13.1.1 and 13.2.1 use these operands.
    exact = closed_form(M, K, N)
    C, D = run_oracle(W.arange_tenths(M, K, N, "f64"))
    assert np.all(np.abs(C - exact) <= 1e-13 * np.maximum(D, 1.0))
    C32, D32 = run_oracle(W.arange_tenths(M, K, N, "f32"))
    assert np.all(np.abs(C32 - exact) <= 3e-7 * np.maximum(D32, 1e-30))
    if (M, K, N) == (8, 8, 8):
        assert abs(C[0, 0] - 11.2) < 1e-12 and abs(C[7, 7] - 169.96) < 1e-11


def test_printed_reference_matrix(golden):
    # Section 13.2, Worked Example 13.2.2's printed ground truth (4 decimals).
    ref = np.array(golden("sentinel_4x5x4.txt")["reference"])
    C, _ = run_oracle(W.arange_tenths(4, 5, 4, "f32"))
    assert np.max(np.abs(C - ref)) < 5e-5


def test_sentinel_missing_k_mask(golden):
    g = golden("sentinel_4x5x4.txt")
    p = W.sentinel_padded()
    Ap, Bp = p.meta["A_parent"], p.meta["B_parent"]
    a = Ap.numpy().reshape(-1)
    b = Bp.numpy().reshape(-1)
    kw = dict(lda=8, ldb=4, a_dtype="f32", b_dtype="f32", BM=4, BN=4, BK=4)
    plain, _ = run_oracle(p)
    masked = oracle.gemm_blocked(a, b, 4, 4, 5, **kw)
    assert np.max(np.abs(masked - plain)) < 1e-12
    assert np.max(np.abs(masked - np.array(g["reference"]))) < 5e-5
    # Without the K mask the second K-chunk reads k = 5, 6, 7 from the sentinel region.
    buggy = oracle.gemm_blocked(a, b, 4, 4, 5, mask_k=False, a_k_alloc=8, b_k_alloc=8, **kw)
    assert np.max(np.abs(buggy - (plain + 3 * 999.0 * 999.0))) < 1e-6
    # The page's numbers come from fp32 arithmetic: within a couple of fp32 ulps (0.25 here).
    assert np.max(np.abs(buggy - np.array(g["buggy"]))) <= 0.5
    # An unmasked read past what the caller says it allocated is refused, not performed.
    with pytest.raises(ValueError):
        oracle.gemm_blocked(a, b, 4, 4, 5, mask_k=False, a_k_alloc=5, b_k_alloc=5, **kw)


def test_accumulation_precision_pins(golden):
    g = golden("accumulation_4x1024x4.txt")
    p = W.accumulation_13_3_1()
    C, _ = run_oracle(p)
    a, _, _ = storage_numpy(p.A)
    b, _, _ = storage_numpy(p.B)
    # fp32 accumulator, one rounding to fp16 at the store.
    out32 = oracle.round_to(C, "f16")
    assert np.max(np.abs(out32 - C)) == g["fp32acc_max_abs_diff"][0][0]
    # fp16 accumulator, rounded after every K-chunk of 8.
    out16 = oracle.gemm_f16acc(a, b, 4, 4, 1024, lda=1024, ldb=4, a_dtype="f16", b_dtype="f16",
                               BK=8)
    assert np.max(np.abs(out16 - C)) == g["fp16acc_max_abs_diff"][0][0]


# ------------------------------------------------------- special structure

def test_identity_and_zero():
    A = W.make_operand(5, 7, "f32", "row", 11)
    I = torch.eye(7, dtype=torch.float32)
    C, D = run_oracle(W.Problem("id", A, I, "f32"))
    assert np.array_equal(C, A.double().numpy())
    assert np.array_equal(D, A.double().abs().numpy())
    Z = torch.zeros(7, 3, dtype=torch.float32)
    C, D = run_oracle(W.Problem("zero", A, Z, "f32"))
    assert np.all(C == 0) and not np.any(np.signbit(C)) and np.all(D == 0)
    # K == 0: the empty sum is +0.
    E = torch.zeros(4, 0, dtype=torch.float32)
    C, D = run_oracle(W.Problem("k0", E, torch.zeros(0, 6), "f32"))
    assert C.shape == (4, 6) and np.all(C == 0) and not np.any(np.signbit(C))


def _int64_product(p):
    A = p.A.to(torch.int64).numpy()
    B = p.B.to(torch.int64).numpy()
    return A @ B, np.abs(A) @ np.abs(B)


def test_integer_brute_force_tiny():
    dtypes = ["f32", "f16", "bf16"]
    layouts = list(itertools.product(["row", "col"], repeat=2))
    n = 0
    for M, N, K in itertools.product(range(1, 10), repeat=3):
        al, bl = layouts[n % 4]
        p = W.integer_problem(M, N, K, dtypes[n % 3], seed=n, a_layout=al, b_layout=bl,
                              ld_pad=n % 3)
        C, D = run_oracle(p)
        ref, mag = _int64_product(p)
        assert np.array_equal(C, ref.astype(np.float64)), (M, N, K)
        assert np.array_equal(D, mag.astype(np.float64)), (M, N, K)
        n += 1


@pytest.mark.parametrize("M,N,K", [(1025, 17, 1023), (127, 1000, 1), (1, 1, 1025),
                                   (17, 1025, 127), (1000, 127, 1025)])
def test_integer_brute_force_ragged_sizes(M, N, K):
    p = W.integer_problem(M, N, K, "f16", seed=M + N + K)
    C, _ = run_oracle(p)
    ref, _ = _int64_product(p)
    assert np.array_equal(C, ref.astype(np.float64))


def test_transpose_identity():
    # (A B)^T = B^T A^T: the same products, so the fp64 results agree bit for bit.
    A = W.make_operand(23, 31, "f32", "row", 5)
    B = W.make_operand(31, 17, "f32", "row", 6)
    C, D = run_oracle(W.Problem("ab", A, B, "f32"))
    Ct, Dt = run_oracle(W.Problem("btat", B.t(), A.t(), "f32"))  # column-major views
    assert np.array_equal(Ct, C.T) and np.array_equal(Dt, D.T)


def test_tile_order_independence():
    rng = np.random.default_rng(7)
    for (M, N, K), (BM, BN, BK) in [((13, 11, 29), (4, 4, 4)), ((13, 11, 29), (5, 3, 7)),
                                    ((8, 8, 8), (4, 4, 4)), ((17, 9, 40), (16, 16, 8))]:
        tiles = -(-M // BM) * -(-N // BN)
        kb = -(-K // BK)
        for dtype, kind in [("f32", "int"), ("f16", "int"), ("f32", "uniform")]:
            A = W.make_operand(M, K, dtype, "row", 1, kind)
            B = W.make_operand(K, N, dtype, "row", 2, kind)
            p = W.Problem("t", A, B, "f32")
            plain, D = run_oracle(p)
            a, _, lda = storage_numpy(A)
            b, _, ldb = storage_numpy(B)
            for _ in range(3):
                blk = oracle.gemm_blocked(a, b, M, N, K, lda=lda, ldb=ldb, a_dtype=dtype,
                                          b_dtype=dtype, BM=BM, BN=BN, BK=BK,
                                          tile_order=rng.permutation(tiles),
                                          kblock_order=rng.permutation(kb))
                if kind == "int":
                    assert np.array_equal(blk, plain)
                else:
                    assert np.all(np.abs(blk - plain) <= 1e-14 * D)


def test_row_subset_matches_full():
    p = W.ragged(127, 17, 1000)
    C, D = run_oracle(p)
    rows = [126, 0, 64, 63, 5]
    Cs, Ds = run_oracle(p, rows=rows, threads=3)
    assert np.array_equal(Cs, C[rows]) and np.array_equal(Ds, D[rows])


def test_magnitude_sum():
    A = W.make_operand(9, 33, "f32", "row", 3, lo=0.0, hi=1.0)
    B = W.make_operand(33, 12, "f32", "col", 4, lo=0.0, hi=1.0)
    C, D = run_oracle(W.Problem("nonneg", A, B, "f32"))
    assert np.array_equal(C, D)
    p = W.ragged(17, 127, 1023)
    C, D = run_oracle(p)
    assert np.all(D >= np.abs(C))


def test_f64_agrees_with_blas():
    A = W.make_operand(64, 300, "f64", "row", 8)
    B = W.make_operand(300, 48, "f64", "col", 9)
    C, D = run_oracle(W.Problem("f64", A, B, "f64"))
    assert np.all(np.abs(C - A.numpy() @ B.numpy()) <= 1e-13 * D)


# ------------------------------------------------------------ format pins

def test_decode_f16_exhaustive():
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.decode("f16", int(x)) for x in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_decode_bf16_exhaustive():
    bits = np.arange(65536, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    got = np.array([oracle.decode("bf16", int(x)) for x in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # Spot values from the format definitions.
    assert oracle.decode("f16", 0x3C00) == 1.0 and oracle.decode("f16", 0x0001) == 2.0 ** -24
    assert oracle.decode("f16", 0x7BFF) == 65504.0 and oracle.decode("bf16", 0x3F80) == 1.0


def test_round_to_nearest_even():
    rng = np.random.default_rng(3)
    x = np.concatenate([
        rng.standard_normal(20000) * 10.0 ** rng.integers(-9, 6, 20000),
        [1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11, 65504.0, 65519.99, 65520.0, 2.0 ** -25,
         3 * 2.0 ** -26, 2.0 ** -24 * 1.5, -0.0, 0.0, 1e-30, -7e5]])
    with np.errstate(over="ignore"):
        ref16 = x.astype(np.float16).astype(np.float64)
    assert np.array_equal(oracle.round_to(x, "f16"), ref16)
    assert np.array_equal(oracle.round_to(x, "f32"), x.astype(np.float32).astype(np.float64))
    x32 = x.astype(np.float32).astype(np.float64)  # exact fp32 values: single rounding to bf16
    ref_bf = torch.from_numpy(x32.astype(np.float32)).to(torch.bfloat16).double().numpy()
    assert np.array_equal(oracle.round_to(x32, "bf16"), ref_bf)
    # Ties go to the even neighbour.
    assert oracle.round_to([1 + 2.0 ** -11], "f16")[0] == 1.0
    assert oracle.round_to([1 + 3 * 2.0 ** -11], "f16")[0] == 1 + 2.0 ** -9


def test_rejects_bad_arguments():
    a = np.zeros(12, np.float32)
    with pytest.raises(ValueError):  # lda below the row length
        oracle.gemm_f64(a, a, 3, 4, 4, lda=3, ldb=4, a_dtype="f32", b_dtype="f32")
    with pytest.raises(ValueError):  # storage too small for the stated shape
        oracle.gemm_f64(a, a, 4, 4, 4, lda=4, ldb=4, a_dtype="f32", b_dtype="f32")
    with pytest.raises(ValueError):  # row index out of range
        oracle.gemm_f64(a, a, 3, 3, 4, lda=4, ldb=3, a_dtype="f32", b_dtype="f32", rows=[3])
    with pytest.raises(TypeError):  # storage dtype mismatch
        oracle.gemm_f64(a, a, 3, 3, 4, lda=4, ldb=3, a_dtype="f16", b_dtype="f32")
