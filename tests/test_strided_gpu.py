"""gemm_run_strided: C = A @ B for arbitrary 2-D views (the six strides of "Chapter 13: The
Blocked Matmul Kernel", section 13.4). Row- and column-major views run in place; sliced,
strided and broadcast views are gathered; a column-major C is produced as C^T = B^T A^T; a
strided C goes through a temporary and must leave the elements between its own untouched."""
import itertools

import numpy as np
import pytest
import torch

import workloads as W
from gpu_util import oracle_rows, rel_err, tolerance

pytestmark = pytest.mark.gpu

TORCH = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}


@pytest.fixture(scope="module")
def h():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import dense_tiled_gemm_05_gb300 as g
    hh = g.Gemm(0)
    yield hh
    hh.close()


def ints(shape, dtype, seed):
    gen = torch.Generator().manual_seed(seed)
    return torch.randint(-4, 5, shape, generator=gen).to(TORCH[dtype]).cuda()


def view(kind, rows, cols, dtype, seed):
    """A rows x cols view of a larger integer-valued base tensor, of the given kind."""
    if kind == "row":
        return ints((rows, cols), dtype, seed)
    if kind == "col":
        return ints((cols, rows), dtype, seed).t()
    if kind == "inner2":                       # strides (2 * cols, 2)
        return ints((rows, 2 * cols), dtype, seed)[:, ::2]
    if kind == "odd":                          # strides (6 * cols, 3)
        return ints((2 * rows, 3 * cols), dtype, seed)[::2, ::3]
    if kind == "col_wide":                     # strides (1, 3 * rows)
        return ints((3 * cols, rows), dtype, seed)[::3].t()
    if kind == "bcast":                        # one row repeated: strides (0, 1)
        return ints((1, cols), dtype, seed).expand(rows, cols)
    raise ValueError(kind)


KINDS = ["row", "col", "inner2", "odd", "col_wide", "bcast"]


def exact(a, b):
    return (a.cpu().to(torch.int64) @ b.cpu().to(torch.int64)).to(torch.float64)


@pytest.mark.parametrize("dtype,precision", [("bf16", "default"), ("f32", "exact")])
@pytest.mark.parametrize("a_kind,b_kind", list(itertools.product(KINDS, KINDS)))
def test_strided_operands_bit_exact(h, dtype, precision, a_kind, b_kind):
    M, N, K = 300, 257, 96
    a = view(a_kind, M, K, dtype, 1)
    b = view(b_kind, K, N, dtype, 2)
    c = h.matmul(a, b, out_dtype="f32", precision=precision)
    torch.cuda.synchronize()
    assert h.status() == 0
    assert torch.equal(c.cpu().double(), exact(a, b))


@pytest.mark.parametrize("c_kind", ["col", "inner2", "odd"])
@pytest.mark.parametrize("a_kind,b_kind", [("row", "row"), ("col", "inner2"), ("odd", "col")])
def test_strided_outputs_bit_exact(h, c_kind, a_kind, b_kind):
    M, N, K = 130, 70, 1025
    a = view(a_kind, M, K, "bf16", 3)
    b = view(b_kind, K, N, "bf16", 4)
    if c_kind == "col":
        base = torch.full((N, M), float("nan"), device="cuda")
        c = base.t()
    elif c_kind == "inner2":
        base = torch.full((M, 2 * N), float("nan"), device="cuda")
        c = base[:, ::2]
    else:
        base = torch.full((2 * M, 3 * N), float("nan"), device="cuda")
        c = base[::2, ::3]
    h.matmul(a, b, out=c)
    torch.cuda.synchronize()
    assert h.status() == 0
    assert torch.equal(c.cpu().double(), exact(a, b))
    # every element of the base that is not an element of C is untouched
    mask = torch.ones_like(base, dtype=torch.bool)
    if c_kind == "col":
        mask[:] = False
    elif c_kind == "inner2":
        mask[:, ::2] = False
    else:
        mask[::2, ::3] = False
    assert torch.isnan(base[mask]).all()


@pytest.mark.parametrize("dtype", ["f16", "f32"])
def test_strided_random_vs_oracle(h, dtype):
    """Real-valued operands through gathers, compared with the oracle on contiguous copies."""
    M, N, K = 257, 300, 1000
    gen = torch.Generator().manual_seed(11)
    a_base = (torch.rand(M, 2 * K, generator=gen) * 2 - 1).to(TORCH[dtype])
    b_base = (torch.rand(3 * N, K, generator=gen) * 2 - 1).to(TORCH[dtype])
    a_cpu, b_cpu = a_base[:, ::2], b_base[::3].t()
    a, b = a_base.cuda()[:, ::2], b_base.cuda()[::3].t()
    prec = "exact" if dtype == "f32" else "default"
    c = h.matmul(a, b, out_dtype="f32", precision=prec)
    torch.cuda.synchronize()
    assert h.status() == 0
    p = W.Problem("strided", a_cpu.contiguous(), b_cpu.contiguous(), "f32", prec)
    C64, D = oracle_rows(p)
    assert rel_err(c, C64, D) <= tolerance(p)


def test_strided_degenerate(h):
    a = view("inner2", 5, 0, "bf16", 5)
    b = view("row", 0, 7, "bf16", 6)
    base = torch.full((5, 14), float("nan"), device="cuda")
    h.matmul(a, b, out=base[:, ::2])
    torch.cuda.synchronize()
    assert torch.equal(base[:, ::2].cpu(), torch.zeros(5, 7))
    assert torch.isnan(base[:, 1::2]).all()
    # one row, one column, single element
    for M, N, K in [(1, 9, 33), (9, 1, 33), (1, 1, 1)]:
        a = view("odd", M, K, "bf16", 7)
        b = view("inner2", K, N, "bf16", 8)
        c = h.matmul(a, b, out_dtype="f32")
        torch.cuda.synchronize()
        assert torch.equal(c.cpu().double(), exact(a, b))
