"""The driver's entry points, on the host: smoke()'s products build, plan to the paths their
comments name, and the oracle computes them (smoke() itself needs the GPU)."""
import os
import sys

import dense_tiled_gemm_05_gb300 as g
import oracle
import workloads as W

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import __graft_entry__ as entry  # noqa: E402


def test_smoke_cases_plan_and_have_oracle_results():
    paths = []
    for p, tol in entry.smoke_cases():
        assert 0 < tol <= 1e-2
        plan = g.plan(p.A, p.B, out_dtype=p.out_dtype, precision=p.precision, sm_count=152)
        paths.append(plan["path"])
        a, al, lda = W.storage_numpy(p.A)
        b, bl, ldb = W.storage_numpy(p.B)
        C64, D = oracle.gemm_f64(a, b, p.M, p.N, p.K, lda=lda, ldb=ldb, a_dtype=p.in_dtype,
                                 b_dtype=W.dtype_name(p.B.dtype), a_layout=al, b_layout=bl)
        assert C64.shape == (p.M, p.N) and (D >= 0).all()
    assert paths == ["tcgen05", "tcgen05", "tcgen05", "fma", "fma"], paths
