"""Host-only decisions of the six-stride interface (gemm_plan_strided): which views are read
or written in place, which are gathered, and which arguments are refused. The pages' host
wrapper passes both strides of A, B and C ("Chapter 13: The Blocked Matmul Kernel", section
13.4); "Triton from zero, Lesson 4", homework 2, reads B^T as a (K, N) view with strides
(1, K)."""
import ctypes

import pytest
import torch

g = pytest.importorskip("dense_tiled_gemm_05_gb300")


@pytest.fixture(scope="module", autouse=True)
def built():
    from dense_tiled_gemm_05_gb300 import build as gbuild
    gbuild.build()


def f16(*shape):
    return torch.empty(*shape, dtype=torch.float16)


def test_row_and_column_major_views_in_place():
    a, b = f16(512, 256), f16(256, 384)
    p, s = g.plan_strided(a, b, out_dtype="f32")
    assert s == {"a_gathered": 0, "b_gathered": 0, "c_mode": 0, "buffer_bytes": 0}
    assert p["path"] == "tcgen05" and p["b_mn_major"] == 1
    # B^T viewed as (K, N) with strides (1, K): K-major, read in place
    bt = f16(384, 256).t()
    p, s = g.plan_strided(a, bt, out_dtype="f32")
    assert s["b_gathered"] == 0 and p["b_mn_major"] == 0
    # row slices with a leading stride wider than the row are still in place
    wide = f16(512, 300)[:, :256]
    assert g.plan_strided(wide, b, out_dtype="f32")[1]["a_gathered"] == 0


def test_general_views_are_gathered():
    a = f16(512, 512)[:, ::2]             # inner stride 2
    b = f16(256, 768)[:, ::2]
    p, s = g.plan_strided(a, b, out_dtype="f32")
    assert s["a_gathered"] == 1 and s["b_gathered"] == 1 and s["c_mode"] == 0
    # gathered A row-major with 16-byte lines; gathered B column-major (K-major for the MMA)
    assert p["a_mn_major"] == 0 and p["b_mn_major"] == 0 and p["stage_a"] == 0
    assert s["buffer_bytes"] >= 512 * 256 * 2 + 384 * 256 * 2
    # a broadcast row (stride 0) is gathered too
    bc = f16(1, 256).expand(512, 256)
    assert g.plan_strided(bc, f16(256, 64), out_dtype="f32")[1]["a_gathered"] == 1


def test_c_layouts():
    a, b = f16(300, 200), f16(200, 100)
    # column-major C: computed as C^T = B^T A^T into the same storage
    c = torch.empty(100, 300, dtype=torch.float32).t()
    p, s = g.plan_strided(a, b, out=c)
    assert s["c_mode"] == 1 and s["a_gathered"] == 0 and s["b_gathered"] == 0
    # the transposed problem has 100 rows: one single-CTA tile row (300 rows would take
    # CTA pairs)
    assert p["grid_m"] == 1 and p["cta_pair"] == 0
    # C with stride 2 along N: through a row-major temporary
    c2 = torch.empty(300, 200, dtype=torch.float32)[:, ::2]
    p, s = g.plan_strided(a, b, out=c2)
    assert s["c_mode"] == 2 and s["buffer_bytes"] >= 300 * 100 * 4
    # a single row of C with a non-unit stride is a column-major 1 x N matrix
    c3 = torch.empty(1, 400, dtype=torch.float32)[:, ::2]
    assert g.plan_strided(f16(1, 200), b, out=c3)[1]["c_mode"] == 1


def code(M, N, K, A, sa, B, sb, C, sc, in_dt=1, out_dt=0, prec=0):
    info, sinfo = g.PlanInfo(), g.StridedInfo()
    return g.lib().gemm_plan_strided(None, M, N, K, A, sa[0], sa[1], B, sb[0], sb[1], C, sc[0],
                                     sc[1], in_dt, out_dt, prec, 148, ctypes.byref(info),
                                     ctypes.byref(sinfo))


def test_refusals():
    A, B, C = 1 << 20, 1 << 24, 1 << 28
    assert code(16, 16, 16, A, (16, 1), B, (16, 1), C, (16, 1)) == 0
    assert code(16, 16, 16, A, (-16, 1), B, (16, 1), C, (16, 1)) == 1   # negative stride
    assert code(16, 16, 16, A, (16, 1), B, (16, 1), C, (8, 1)) == 1     # C rows overlap
    assert code(16, 16, 16, A, (16, 1), B, (16, 1), C, (1, 1)) == 1     # C elements alias
    assert code(16, 16, 16, A, (16, 1), B, (16, 1), C, (0, 1)) == 1     # C broadcast
    assert code(16, 16, 16, A, (16, 1), B, (16, 1), A + 32, (16, 1)) == 1  # C overlaps A
    assert code(16, 16, 16, A, (0, 0), B, (16, 1), C, (16, 1)) == 0     # A broadcast: fine
    assert code(16, 16, 16, A, (16, 1), B, (16, 1), None, (16, 1)) == 1
    assert code(16, 16, 16, None, (16, 1), B, (16, 1), C, (16, 1)) == 1
    assert code(16, 16, 0, None, (0, 0), None, (0, 0), C, (16, 1)) == 0  # K == 0: zeros
    assert code(0, 16, 16, None, (0, 0), None, (0, 0), None, (0, 0)) == 0  # empty
    assert code(16, 16, 16, A, (16, 1), B, (16, 1), C, (16, 1), in_dt=2, prec=1) == 2
    assert g.lib().gemm_run_strided(None, 4, 4, 4, A, 4, 1, B, 4, 1, C, 4, 1, 1, 0, 0,
                                    None) == 1
