"""Python access to the CPU oracle for the blocked matrix multiply.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only importers. It never imports the GPU
package, and the GPU package never imports it.

Operands are passed as raw storage in numpy arrays:

* ``f32`` -> ``np.float32``; ``f64`` -> ``np.float64``;
* ``f16`` and ``bf16`` -> ``np.uint16`` holding the bit patterns.

A logical ``rows x cols`` operand with layout ``"row"`` has element (r, c) at
flat index ``r * ld + c``; with layout ``"col"`` at ``c * ld + r``. For A the
logical shape is M x K, for B it is K x N ("Chapter 13: The Blocked Matmul
Kernel", section 13.1: C[M,N] = A[M,K] @ B[K,N]).
"""
import ctypes
import os

import numpy as np

from . import build as _build

DTYPES = {"f32": 0, "f16": 1, "bf16": 2, "f64": 3}
LAYOUTS = {"row": 0, "col": 1}
_STORAGE = {"f32": np.float32, "f16": np.uint16, "bf16": np.uint16, "f64": np.float64}
_ERRORS = {-1: "invalid argument", -2: "unmasked read outside the buffer", -3: "out of memory"}

_lib = None


def lib():
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        i64, i32, vp, dp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p
        L.oracle_gemm_f64.argtypes = [i64, i64, i64, vp, i64, i32, i32, vp, i64, i32, i32,
                                      vp, i64, dp, dp, i32]
        L.oracle_gemm_f64.restype = i32
        L.oracle_gemm_blocked.argtypes = [i64, i64, i64, vp, i64, i32, i32, i64,
                                          vp, i64, i32, i32, i64, i64, i64, i64, i32,
                                          vp, vp, dp, i64]
        L.oracle_gemm_blocked.restype = i32
        L.oracle_gemm_f16acc.argtypes = [i64, i64, i64, vp, i64, i32, i32, vp, i64, i32, i32,
                                         i64, dp, i64]
        L.oracle_gemm_f16acc.restype = i32
        L.oracle_softmax_rows.argtypes = [i64, i64, vp, i64, i32, dp, i64]
        L.oracle_softmax_rows.restype = i32
        L.oracle_round.argtypes = [dp, i64, i32]
        L.oracle_round.restype = i32
        L.oracle_decode.argtypes = [i32, ctypes.c_uint64]
        L.oracle_decode.restype = ctypes.c_double
        L.oracle_num_threads.argtypes = []
        L.oracle_num_threads.restype = i32
        _lib = L
    return _lib


def _check(rc):
    if rc != 0:
        raise ValueError("oracle: " + _ERRORS.get(rc, "error %d" % rc))


def _operand(x, dtype, layout, rows, cols, ld):
    """Validate storage size so the C code never reads outside ``x``."""
    if dtype not in DTYPES or layout not in LAYOUTS:
        raise ValueError("unknown dtype/layout %r/%r" % (dtype, layout))
    x = np.ascontiguousarray(x).reshape(-1)
    if x.dtype != _STORAGE[dtype]:
        raise TypeError("%s storage must be %s, got %s" % (dtype, _STORAGE[dtype], x.dtype))
    outer, inner = (rows, cols) if layout == "row" else (cols, rows)
    need = 0 if rows == 0 or cols == 0 else (outer - 1) * ld + inner
    if x.size < need:
        raise ValueError("operand storage holds %d elements, needs %d" % (x.size, need))
    return x


def num_threads() -> int:
    return lib().oracle_num_threads()


def gemm_f64(a, b, M, N, K, *, lda, ldb, a_dtype, b_dtype, a_layout="row", b_layout="row",
             rows=None, threads=0):
    """Return ``(C, D)`` in fp64 for the selected rows (all rows by default).

    ``C[r, j] = sum_k A[rows[r], k] * B[k, j]`` and ``D[r, j] = sum_k |A B|``.
    """
    a = _operand(a, a_dtype, a_layout, M, K, lda)
    b = _operand(b, b_dtype, b_layout, K, N, ldb)
    if rows is None:
        rows_arr, n_rows = None, M
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1)
        n_rows = rows_arr.size
    C = np.zeros((n_rows, N), dtype=np.float64)
    D = np.zeros((n_rows, N), dtype=np.float64)
    rc = lib().oracle_gemm_f64(M, N, K, a.ctypes.data, lda, DTYPES[a_dtype], LAYOUTS[a_layout],
                               b.ctypes.data, ldb, DTYPES[b_dtype], LAYOUTS[b_layout],
                               None if rows_arr is None else rows_arr.ctypes.data, n_rows,
                               C.ctypes.data, D.ctypes.data, threads)
    _check(rc)
    return C, D


def gemm_blocked(a, b, M, N, K, *, lda, ldb, a_dtype, b_dtype, BM, BN, BK, a_layout="row",
                 b_layout="row", mask_k=True, a_k_alloc=None, b_k_alloc=None,
                 tile_order=None, kblock_order=None):
    """The pages' tiled algorithm (tile grid, K-loop, masks) in fp64; returns C[M, N].

    With ``mask_k=False`` the K mask is omitted; ``a_k_alloc``/``b_k_alloc`` then
    state how many k positions the buffers really hold.
    """
    a_k_alloc = K if a_k_alloc is None else a_k_alloc
    b_k_alloc = K if b_k_alloc is None else b_k_alloc
    a = _operand(a, a_dtype, a_layout, M, max(K, a_k_alloc), lda)
    b = _operand(b, b_dtype, b_layout, max(K, b_k_alloc), N, ldb)
    C = np.zeros((M, N), dtype=np.float64)
    to = None if tile_order is None else np.ascontiguousarray(tile_order, dtype=np.int64)
    ko = None if kblock_order is None else np.ascontiguousarray(kblock_order, dtype=np.int64)
    tiles = -(-M // BM) * -(-N // BN)
    if to is not None and to.size != tiles:
        raise ValueError("tile_order must have %d entries" % tiles)
    if ko is not None and ko.size != -(-K // BK):
        raise ValueError("kblock_order must have %d entries" % -(-K // BK))
    rc = lib().oracle_gemm_blocked(M, N, K, a.ctypes.data, lda, DTYPES[a_dtype], LAYOUTS[a_layout],
                                   a_k_alloc, b.ctypes.data, ldb, DTYPES[b_dtype],
                                   LAYOUTS[b_layout], b_k_alloc, BM, BN, BK, int(bool(mask_k)),
                                   None if to is None else to.ctypes.data,
                                   None if ko is None else ko.ctypes.data,
                                   C.ctypes.data, max(N, 1))
    _check(rc)
    return C


def gemm_f16acc(a, b, M, N, K, *, lda, ldb, a_dtype, b_dtype, BK, a_layout="row",
                b_layout="row"):
    """fp16-accumulator product (each K-chunk rounded to fp16); returns fp16 values as fp64."""
    a = _operand(a, a_dtype, a_layout, M, K, lda)
    b = _operand(b, b_dtype, b_layout, K, N, ldb)
    C = np.zeros((M, N), dtype=np.float64)
    rc = lib().oracle_gemm_f16acc(M, N, K, a.ctypes.data, lda, DTYPES[a_dtype], LAYOUTS[a_layout],
                                  b.ctypes.data, ldb, DTYPES[b_dtype], LAYOUTS[b_layout], BK,
                                  C.ctypes.data, max(N, 1))
    _check(rc)
    return C


def softmax_rows(x, M, N, *, ldx, x_dtype):
    """Row softmax of the M x N row-major matrix in ``x`` (raw storage, leading dimension
    ``ldx``), in fp64: y = exp(x - max) / sum(exp(x - max)) per row."""
    x = np.ascontiguousarray(x, dtype=_STORAGE[x_dtype]).reshape(-1)
    if M > 0 and N > 0 and x.size < (M - 1) * ldx + N:
        raise ValueError("x is smaller than its logical extent")
    Y = np.zeros((M, N), dtype=np.float64)
    _check(lib().oracle_softmax_rows(M, N, x.ctypes.data, ldx, DTYPES[x_dtype], Y.ctypes.data,
                                     max(N, 1)))
    return Y


def round_to(x, dtype):
    """Round fp64 values to the nearest ``dtype`` value (ties to even); returns a new array."""
    y = np.array(x, dtype=np.float64, copy=True, order="C")
    _check(lib().oracle_round(y.ctypes.data, y.size, DTYPES[dtype]))
    return y


def decode(dtype, bits):
    """Decode one stored bit pattern of ``dtype`` into a Python float."""
    return lib().oracle_decode(DTYPES[dtype], int(bits))
