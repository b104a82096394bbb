"""Pins of the row-softmax oracle ("Triton from zero, Lesson 4: Block Pointers", homework 4:
per row, y = exp(x - max) / sum(exp(x - max)), with the tile's masked columns at -inf) to
values fixed by the mathematics, not by the oracle itself: closed forms, invariances, the
special values the -inf padding produces, and an independent library routine."""
import math

import numpy as np
import pytest

import oracle

scipy_special = pytest.importorskip("scipy.special")


def sm(x, dtype="f64", ldx=None):
    x = np.asarray(x)
    M, N = x.shape
    return oracle.softmax_rows(x, M, N, ldx=ldx or N, x_dtype=dtype)


def test_logs_of_integers():
    y = sm(np.array([[0.0, math.log(2), math.log(3)]]))
    np.testing.assert_allclose(y[0], [1 / 6, 2 / 6, 3 / 6], rtol=1e-15, atol=0)


def test_constant_rows_are_uniform():
    for n in (1, 2, 7, 1000):
        y = sm(np.full((3, n), 5.25))
        np.testing.assert_allclose(y, np.full((3, n), 1.0 / n), rtol=1e-14, atol=0)


def test_two_values_are_the_logistic_function():
    for a, b in [(0.0, 0.0), (1.0, -2.0), (-30.0, 40.0), (700.0, 699.0), (-1e-3, 2e-3)]:
        y = sm(np.array([[a, b]]))
        p = 1.0 / (1.0 + math.exp(b - a))
        assert abs(y[0, 0] - p) <= 1e-15 * max(p, 1e-300) + 1e-300
        assert abs(y[0, 1] - (1.0 - p)) <= 1e-15


def test_rows_of_a_geometric_series():
    # X[i, j] = i * j: y[i, j] = r^j / sum_k r^k with r = e^i (closed form of the series),
    # so each row is different and a row/column mix-up or a wrong row stride shows.
    M, N = 5, 9
    X = np.fromfunction(lambda i, j: i * j, (M, N), dtype=np.float64)
    y = sm(X)
    for i in range(M):
        if i == 0:
            ref = np.full(N, 1.0 / N)
        else:
            r = math.exp(-i)  # relative to the row's maximum at j = N - 1
            total = (1.0 - r ** N) / (1.0 - r)
            ref = np.array([r ** (N - 1 - j) / total for j in range(N)])
        np.testing.assert_allclose(y[i], ref, rtol=1e-13, atol=0)


def test_shift_invariance_without_overflow():
    rng = np.random.default_rng(1)
    X = rng.normal(size=(4, 33))
    y0 = sm(X)
    for c in (1000.0, -1000.0, 1e5):
        np.testing.assert_allclose(sm(X + c), y0, rtol=1e-10, atol=1e-15)
    assert np.all(np.isfinite(sm(X * 800.0)))  # max subtraction keeps exp in range


def test_minus_infinity_is_the_padding_value():
    inf = math.inf
    y = sm(np.array([[1.0, -inf, 2.0, -inf], [-inf, 3.0, -inf, -inf]]))
    assert y[0, 1] == 0.0 and y[0, 3] == 0.0
    np.testing.assert_allclose(y[0, [0, 2]], [1 / (1 + math.e), math.e / (1 + math.e)],
                               rtol=1e-15)
    assert y[1, 1] == 1.0 and np.all(y[1, [0, 2, 3]] == 0.0)
    # -inf padding changes nothing: the padded row equals the unpadded one
    x = np.array([[0.5, -1.5, 2.25]])
    padded = np.concatenate([x, np.full((1, 5), -inf)], axis=1)
    np.testing.assert_array_equal(sm(padded)[:, :3], sm(x))


def test_special_values_give_nan():
    inf, nan = math.inf, math.nan
    y = sm(np.array([[-inf, -inf], [1.0, nan], [inf, 1.0]]))
    assert np.all(np.isnan(y))


def test_matches_an_independent_routine_and_sums_to_one():
    rng = np.random.default_rng(2)
    X = rng.normal(scale=4.0, size=(16, 257))
    y = sm(X)
    np.testing.assert_allclose(y, scipy_special.softmax(X, axis=1), rtol=1e-13, atol=1e-300)
    np.testing.assert_allclose(y.sum(axis=1), 1.0, rtol=1e-14)
    # order preserving within a row
    for i in range(4):
        order = np.argsort(X[i])
        assert np.all(np.diff(y[i][order]) >= 0)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_stored_formats_and_leading_dimension(dtype):
    import torch
    rng = np.random.default_rng(3)
    vals = rng.normal(size=(6, 40)).astype(np.float32)
    t = torch.from_numpy(vals).to({"f32": torch.float32, "f16": torch.float16,
                                   "bf16": torch.bfloat16}[dtype])
    exact = t.double().numpy()[:, :31]
    # storage with a row pitch of 40 and NaN beyond column 31: only 31 columns count
    t[:, 31:] = float("nan")
    raw = t.view(torch.int16).numpy().view(np.uint16) if dtype != "f32" else t.numpy()
    y = oracle.softmax_rows(raw.reshape(-1), 6, 31, ldx=40, x_dtype=dtype)
    np.testing.assert_allclose(y, scipy_special.softmax(exact, axis=1), rtol=1e-13)
