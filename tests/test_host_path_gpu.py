"""gemm_run_host: the product of operands held in host memory, with the copies to and
from the device pipelined against the product inside the library (row panels of A and
column panels of B in, blocks of C out, on the handle's own streams). Compared with the exact product (integer inputs) and with
the oracle, for single- and multi-panel shapes, both operand layouts, pinned and pageable
buffers, K = 0, and back-to-back calls that reuse the handle's device copies."""
import itertools

import numpy as np
import pytest
import torch

import workloads as W
from gpu_util import oracle_rows, rel_err, sample_rows, tolerance

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def h():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import dense_tiled_gemm_05_gb300 as g
    hh = g.Gemm(0)
    yield hh
    hh.close()


def to_host(x, pinned=True):
    """A host copy of a logical view's storage span (pinned or pageable), same view."""
    layout, ld = W.layout_of(x)
    r, c = x.shape
    outer, inner = (r, c) if layout == "row" else (c, r)
    n = (outer - 1) * ld + inner if r and c else 0
    if n == 0:
        return torch.empty(x.shape, dtype=x.dtype, pin_memory=pinned)
    flat = torch.empty((n,), dtype=x.dtype, pin_memory=pinned)
    flat.copy_(torch.as_strided(x, (n,), (1,), x.storage_offset()))
    return torch.as_strided(flat, x.shape, x.stride(), 0)


def run_host(h, p, pinned=True, out=None):
    a, b = to_host(p.A, pinned), to_host(p.B, pinned)
    c = h.matmul_host(a, b, out=out, out_dtype=p.out_dtype, precision=p.precision)
    torch.cuda.synchronize()
    assert h.status() == 0
    return c


# (M, N, K): one panel each; several row panels of A with a ragged tail; an output row of
# 1001 fp32 values (not a multiple of 16 bytes, so the device copy is padded); several
# panels of both operands
HOST_SHAPES = [(1, 1, 1), (300, 257, 65), (4500, 130, 96), (8200, 72, 40), (2049, 1001, 33),
               (1500, 3000, 24)]


@pytest.mark.parametrize("dtype,precision", [("bf16", "default"), ("f32", "exact")])
@pytest.mark.parametrize("a_layout,b_layout", list(itertools.product(["row", "col"], repeat=2)))
def test_host_path_integer_bit_exact(h, dtype, precision, a_layout, b_layout):
    for n, (M, N, K) in enumerate(HOST_SHAPES):
        p = W.integer_problem(M, N, K, dtype, seed=500 + n, a_layout=a_layout,
                              b_layout=b_layout, precision=precision, ld_pad=n % 3)
        c = run_host(h, p)
        assert not c.is_cuda
        ref = p.A.to(torch.int64) @ p.B.to(torch.int64)
        assert torch.equal(c.to(torch.int64), ref), (M, N, K)


@pytest.mark.parametrize("panel", [256, 1024, 1 << 20])
def test_host_path_panel_widths(panel):
    """Explicit panel widths: many 256-wide panels (more than the 32-panel cap, which
    widens them), the default-sized ones, and one panel per operand."""
    import dense_tiled_gemm_05_gb300 as g
    hh = g.Gemm(0)
    hh.set_option("host_panel", panel)
    for n, (M, N, K) in enumerate([(4500, 1300, 96), (257, 64, 64), (9000, 700, 48),
                                   (300, 9001, 40)]):
        p = W.integer_problem(M, N, K, "bf16", seed=700 + n, b_layout="col")
        c = run_host(hh, p)
        assert torch.equal(c.to(torch.int64), p.A.to(torch.int64) @ p.B.to(torch.int64))
    with pytest.raises(g.GemmError):
        hh.set_option("host_panel", 100)
    hh.close()


def test_host_path_random_vs_oracle(h):
    p = W.ragged(4608, 768, 1000, seed=77, dtype="bf16")
    c = run_host(h, p)
    rows = sample_rows(p.M, tile=256)
    C64, D = oracle_rows(p, rows)
    assert rel_err(c[rows], C64, D) <= tolerance(p)


def test_host_path_pageable(h):
    p = W.ragged(2500, 300, 200, seed=78, dtype="f16")
    c = run_host(h, p, pinned=False)
    C64, D = oracle_rows(p)
    assert rel_err(c, C64, D) <= tolerance(p)


def test_host_path_k_zero(h):
    a = torch.empty((5, 0), dtype=torch.bfloat16, pin_memory=True)
    b = torch.empty((0, 7), dtype=torch.bfloat16, pin_memory=True)
    out = torch.full((5, 7), float("nan"), dtype=torch.float32, pin_memory=True)
    h.matmul_host(a, b, out=out)
    torch.cuda.synchronize()
    assert h.status() == 0
    assert torch.equal(out, torch.zeros(5, 7))


def test_host_path_back_to_back(h):
    """Two calls enqueued without a synchronisation in between reuse the handle's device
    copies of A, B and C; the second must not overwrite them while the first still reads
    them, and both results must be complete after one synchronisation."""
    p1 = W.integer_problem(4200, 96, 160, "bf16", seed=601)
    p2 = W.integer_problem(4200, 96, 160, "bf16", seed=602)
    a1, b1, a2, b2 = to_host(p1.A), to_host(p1.B), to_host(p2.A), to_host(p2.B)
    c1 = h.matmul_host(a1, b1, out_dtype="f32")
    c2 = h.matmul_host(a2, b2, out_dtype="f32")
    torch.cuda.synchronize()
    assert h.status() == 0
    assert torch.equal(c1.to(torch.int64), p1.A.to(torch.int64) @ p1.B.to(torch.int64))
    assert torch.equal(c2.to(torch.int64), p2.A.to(torch.int64) @ p2.B.to(torch.int64))


def test_host_path_after_device_work_on_stream(h):
    """The copies start only after work enqueued earlier on the caller's stream: the host
    output buffer is filled by a device-to-host copy first, then overwritten by the product."""
    p = W.integer_problem(700, 64, 48, "bf16", seed=603)
    a, b = to_host(p.A), to_host(p.B)
    out = torch.empty((700, 64), dtype=torch.float32, pin_memory=True)
    junk = torch.full((700, 64), 12345.0, device="cuda")
    torch.cuda._sleep(1_000_000)  # keep the stream busy so that ordering matters
    out.copy_(junk, non_blocking=True)
    h.matmul_host(a, b, out=out)
    torch.cuda.synchronize()
    assert h.status() == 0
    assert torch.equal(out.to(torch.int64), p.A.to(torch.int64) @ p.B.to(torch.int64))
    np.testing.assert_array_equal(out.numpy(), (p.A.double() @ p.B.double()).numpy())
