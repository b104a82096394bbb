"""gemm_run_noalloc, the entry point for callers that may not allocate device memory when
they need a product (a plugin inside a runtime that owns every device allocation, a
deployment that reserves all memory up front, a callback that must not synchronise the
device the way cudaMalloc can). It stages operands in a fixed device array compiled into
the library instead of a workspace grown with cudaMalloc.

Called here through the C ABI and compared with gemm_run_ex (the handle path) on
problems whose operands must be staged, so the fixed array is really used, on calls in
a row that overwrite each other's staged copies."""
import ctypes

import pytest
import torch

import workloads as W
from gpu_util import oracle_rows, rel_err, to_device, tolerance

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import dense_tiled_gemm_05_gb300 as g
    from dense_tiled_gemm_05_gb300 import build as gbuild
    gbuild.build()
    return g


def noalloc(g, a, b, out, precision, status=None):
    al, lda = g.operand_layout(a)
    bl, ldb = g.operand_layout(b)
    M, K = a.shape
    N = b.shape[1]
    stream = torch.cuda.current_stream().cuda_stream
    return g.lib().gemm_run_noalloc(
        M, N, K, ctypes.c_void_p(a.data_ptr()), lda, ctypes.c_void_p(b.data_ptr()), ldb,
        ctypes.c_void_p(out.data_ptr()), max(out.stride(0), N, 1), g._dtype_code(a.dtype),
        g._dtype_code(out.dtype), g.PREC[precision], al, bl,
        None if status is None else ctypes.c_void_p(status.data_ptr()), ctypes.c_void_p(stream))


def test_noalloc_matches_run_ex_on_calls_in_a_row(g):
    h = g.Gemm(0)
    # The allocation-free path computes whole tiles only (no split-K workspace); compare
    # with the handle path on the same schedule so the bits must agree.
    h.set_option("stream_k", 1)
    # All need scratch: fp16 rows of 1025 elements and fp32 rows of 1001 are not 16-byte
    # multiples (staged copies), and exact fp32 splits both operands into tf32 hi and lo
    # parts. The tf32 problem runs twice: once with the array's own status word, once with
    # the caller's, so a timeout on that kernel would be seen.
    tf32 = W.Problem("tf32_1000x1000x1001", W.make_operand(1000, 1001, "f32", "row", 42),
                     W.make_operand(1001, 1000, "f32", "row", 43), "f32", "tf32")
    problems = [(W.ragged(1023, 1000, 1025), True), (tf32, False), (tf32, True),
                (W.ragged(1000, 700, 1025, seed=22, dtype="f32"), True),
                (W.ragged(1023, 1000, 1025), True)]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for p, own_status in problems:
        a, b = to_device(p.A), to_device(p.B)
        plan = h.plan(a, b, out_dtype=p.out_dtype, precision=p.precision)
        assert plan["stage_a"] or plan["stage_b"]
        assert plan["workspace_bytes"] <= (32 << 20) - 256  # fits the fixed array
        if p.precision == "exact":
            assert plan["path"] == "tcgen05_3xtf32", plan  # split operands in the array
        ref = h.matmul(a, b, out_dtype=p.out_dtype, precision=p.precision)  # gemm_run_ex
        assert h.status() == 0
        out = torch.full_like(ref, float("nan"))
        rc = noalloc(g, a, b, out, p.precision, status=status if own_status else None)
        assert rc == 0, g.STATUS.get(rc, rc)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        C64, D = oracle_rows(p)
        assert rel_err(out, C64, D) <= tolerance(p)
        scale = torch.from_numpy(D).to(out.device).clamp_min(1e-30)
        assert float(((out.double() - ref.double()).abs() / scale).max()) <= tolerance(p)
        assert torch.equal(out, ref)  # same kernels and staging: the same bits
    h.close()


def test_noalloc_rejects_staging_beyond_its_array(g):
    # A 4096 x 4097 fp32 B (rows of 16388 bytes, not a 16-byte multiple) needs a 64 MiB
    # staged copy, more than the 32 MiB array: refused before anything is launched, C
    # untouched.
    a = torch.zeros(64, 4096, dtype=torch.float32, device="cuda")
    b = torch.zeros(4096, 4097, dtype=torch.float32, device="cuda")[:, :4096]
    out = torch.full((64, 4096), 7.0, dtype=torch.float32, device="cuda")
    rc = noalloc(g, a, b, out, "tf32")
    assert rc == 2  # GEMM_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())


def test_noalloc_rejects_exact_split_beyond_its_array(g):
    # Exact fp32 2048^3 splits both operands into hi and lo parts: 8 * 4096 * 2048 bytes =
    # 64 MiB, more than the array holds. Refused (no silent fall-back to a slower kernel),
    # C untouched; the same problem through the handle path is correct.
    p = W.ragged(2048, 2048, 2048, seed=23, dtype="f32")
    a, b = to_device(p.A), to_device(p.B)
    out = torch.full((2048, 2048), 7.0, dtype=torch.float32, device="cuda")
    rc = noalloc(g, a, b, out, "exact")
    assert rc == 2  # GEMM_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())
    h = g.Gemm(0)
    c = h.matmul(a, b, precision="exact")
    assert h.status() == 0
    h.close()
    rows = list(range(0, 2048, 61)) + [2047]
    C64, D = oracle_rows(p, rows)
    assert rel_err(c[rows], C64, D) <= tolerance(p)
