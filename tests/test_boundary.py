"""Host-side tests of the C-ABI library: it loads without a GPU, exports every symbol
include/gemm.h declares, rejects bad arguments before launching anything, and plans
each workload the way the design says. Nothing here calls a GPU kernel."""
import ctypes
import os
import re

import pytest
import torch

import dense_tiled_gemm_05_gb300 as g
from dense_tiled_gemm_05_gb300 import build as gbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    gbuild.build()
    return g.lib()


def header_symbols():
    text = open(os.path.join(ROOT, "include", "gemm.h")).read()
    return sorted(set(re.findall(r"GEMM_API\s+[\w\s\*]+?\b(gemm_\w+)\s*\(", text)))


def test_exports_every_declared_symbol(L):
    declared = header_symbols()
    assert set(declared) == set(g.EXPORTS), declared
    for name in declared:
        assert hasattr(L, name), name
    # Nothing but the declared API is exported (hidden visibility for internals).
    out = os.popen("nm -D --defined-only %s" % g.LIB_PATH).read()
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert {s for s in exported if s.startswith("gemm_")} == set(declared)


def test_version_and_strerror(L):
    assert re.match(r"^\d+\.\d+\.\d+$", g.version())
    for code in range(8):
        assert L.gemm_strerror(code)
    assert L.gemm_strerror(99) == b"unknown status"


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU error path")
def test_create_without_gpu_reports_device_error(L):
    h = ctypes.c_void_p()
    assert L.gemm_create(ctypes.byref(h), 0) == 7  # GEMM_ERR_DEVICE
    assert h.value is None
    assert L.gemm_create(None, 0) == 1


def test_null_handle_is_rejected(L):
    assert L.gemm_run(None, 4, 4, 4, None, 4, None, 4, None, 4, 0, 0, 0) == 1
    assert L.gemm_get_status(None, None) == 1
    assert L.gemm_run_host(None, 4, 4, 4, None, 4, None, 4, None, 4, 0, 0, 0, 0, 0, None) == 1
    assert L.gemm_tune(None, 4, 4, 4, None, 4, None, 4, None, 4, 0, 0, 0, 0, 0, None, 1,
                       None) == 1
    assert L.gemm_tune_clear(None) == 1
    assert L.gemm_set_kernel_events(None, None, None) == 1
    assert L.gemm_set_option(None, 0, 1) == 1
    L.gemm_destroy(None)  # no-op


def t(shape, dtype, layout="row"):
    x = torch.zeros(shape[::-1] if layout == "col" else shape, dtype=dtype)
    return x.t() if layout == "col" else x


def test_plan_small_exact_uses_pages_tiles():
    # The pages' 8x8x8 example: 4x4x4 tiles, grid (2, 2), two K-iterations per tile.
    p = g.plan(t((8, 8), torch.float32), t((8, 8), torch.float32), precision="exact")
    assert p["path"] == "fma"
    assert (p["tile_m"], p["tile_n"], p["tile_k"]) == (4, 4, 4)
    assert (p["grid_m"], p["grid_n"], p["k_iters"]) == (2, 2, 2)
    assert g.plan(t((8, 8), torch.float32), t((8, 8), torch.float32))["path"] == "fma"


def test_plan_bf16_square_is_tcgen05_k_major():
    p = g.plan(t((4096, 4096), torch.bfloat16), t((4096, 4096), torch.bfloat16, "col"),
               sm_count=148)
    assert p["path"] == "tcgen05" and p["cta_pair"] == 1
    assert (p["tile_m"], p["tile_n"], p["tile_k"]) == (256, 256, 64)
    assert (p["grid_m"], p["grid_n"], p["k_iters"]) == (16, 16, 64)
    assert p["a_mn_major"] == 0 and p["b_mn_major"] == 0
    assert p["stage_a"] == 0 and p["stage_b"] == 0 and p["tma_store"] == 1
    assert p["ctas"] == 148 and p["workspace_bytes"] == 0 and p["stages"] == 6
    assert p["split_tiles"] == 108  # last rounds split along K (3.46 rounds of tiles)
    p = g.plan(t((8192, 8192), torch.bfloat16), t((8192, 8192), torch.bfloat16, "col"),
               sm_count=148)
    assert (p["tile_m"], p["tile_n"], p["grid_m"], p["grid_n"]) == (256, 256, 32, 32)
    assert (p["tile_k"], p["stages"]) == (64, 6)  # compute-bound: one K-block per stage
    p = g.plan(t((16384, 8192), torch.bfloat16), t((8192, 128), torch.bfloat16, "col"),
               sm_count=148)
    assert (p["tile_m"], p["tile_n"], p["grid_m"], p["grid_n"]) == (256, 128, 64, 1)
    assert p["ctas"] == 128 and p["split_tiles"] == 0
    # bandwidth-bound (125 flops per byte): two 128-byte K-blocks per stage, half the stages
    assert (p["tile_k"], p["k_iters"], p["stages"]) == (128, 64, 4)
    # A compute-bound problem whose single-CTA tiles all fit one round keeps single CTAs.
    p = g.plan(t((2048, 2048), torch.bfloat16), t((2048, 2048), torch.bfloat16, "col"),
               sm_count=148)
    assert p["cta_pair"] == 0 and (p["tile_m"], p["tile_n"], p["ctas"]) == (128, 256, 128)
    # One 128-row tile of M with a short K: single-CTA tiles.
    p = g.plan(t((128, 2048), torch.bfloat16), t((2048, 4096), torch.bfloat16, "col"),
               sm_count=148)
    # Fewer tiles than SMs: 32 tiles of 128 x 128 finish sooner than 16 of 128 x 256.
    assert p["cta_pair"] == 0 and (p["tile_m"], p["tile_n"], p["grid_m"]) == (128, 128, 1)
    assert p["ctas"] == 32
    # The same with K = 8192 (128 K-blocks): so few tiles leave most SMs idle, so CTA pairs
    # split each of the 16 tiles' K-loops over the idle clusters (six pieces a tile at
    # most; 74 clusters here)
    p = g.plan(t((128, 8192), torch.bfloat16), t((8192, 4096), torch.bfloat16, "col"),
               sm_count=148)
    assert p["cta_pair"] == 1 and (p["grid_m"], p["grid_n"]) == (1, 16)
    assert p["split_tiles"] == 16 and p["ctas"] == 148 and p["tile_k"] == 64
    # one tile: six pieces on six clusters for 128 K-blocks, sixteen for 1024
    p = g.plan(t((256, 8192), torch.bfloat16), t((8192, 256), torch.bfloat16, "col"),
               sm_count=148)
    assert p["cta_pair"] == 1 and p["split_tiles"] == 1 and p["ctas"] == 12
    p = g.plan(t((128, 65536), torch.bfloat16), t((65536, 128), torch.bfloat16, "col"),
               sm_count=148)
    assert p["cta_pair"] == 1 and p["split_tiles"] == 1 and p["ctas"] == 32


def test_plan_row_major_b_is_mn_major():
    p = g.plan(t((256, 512), torch.float16), t((512, 300), torch.float16))
    assert p["path"] == "tcgen05" and p["b_mn_major"] == 1 and p["a_mn_major"] == 0
    p = g.plan(t((256, 512), torch.float16, "col"), t((512, 304), torch.float16))
    assert p["a_mn_major"] == 1 and p["stage_a"] == 0


def test_plan_ragged_stages_misaligned_operands():
    # fp16 with K = 1025: a row is 2050 bytes, not a multiple of 16 -> staged copy.
    a, b = t((1023, 1025), torch.float16), t((1025, 17), torch.float16)
    p = g.plan(a, b, out_dtype="f32")
    assert p["stage_a"] == 1 and p["stage_b"] == 1 and p["tma_store"] == 0
    assert p["workspace_bytes"] >= 1023 * 1032 * 2 + 1025 * 24 * 2
    # K = 1000 (2000-byte rows) is TMA-legal in place; N = 1000 fp32 C rows are 4000 bytes.
    p = g.plan(t((17, 1000), torch.float16), t((1000, 1000), torch.float16), out_dtype="f32")
    assert p["stage_a"] == 0 and p["stage_b"] == 0 and p["tma_store"] == 1
    # A row of C that does not end on a 16-byte boundary is written with plain stores.
    p = g.plan(t((64, 64), torch.float16), t((64, 17), torch.float16), out_dtype="f32",
               ldc=28)
    assert p["tma_store"] == 0
    # A misaligned base pointer is staged, not rejected.
    a = t((64, 64), torch.float16)
    p = g.plan(a, t((64, 64), torch.float16), a_ptr=a.data_ptr() + 2)
    assert p["stage_a"] == 1


def test_plan_fp32_modes():
    a, b = t((4096, 4096), torch.float32), t((4096, 4096), torch.float32)
    p = g.plan(a, b, precision="tf32")
    assert p["path"] == "tcgen05" and p["tile_k"] == 32 and p["k_iters"] == 128
    # The tensor cores read a row-major (MN-major) tf32 B in place, in the 128-byte swizzle
    # with 32-byte atoms; a row-major A is K-major and read in place too.
    assert p["stage_a"] == 0 and p["stage_b"] == 0 and p["b_mn_major"] == 1
    assert p["workspace_bytes"] == 0
    p = g.plan(t((100, 60), torch.float32, "col"), t((60, 50), torch.float32, "col"),
               precision="tf32")
    assert p["stage_a"] == 0 and p["a_mn_major"] == 1 and p["stage_b"] == 0
    # GEMM_OPT_TF32_TRANSPOSE = 1: MN-major tf32 operands are copied K-major first
    h = g.Gemm.__new__(g.Gemm)
    hh = ctypes.c_void_p()
    if g.lib().gemm_create(ctypes.byref(hh), 0) == 0:  # only with a GPU; else plan by options
        h._h = hh
        h.set_option("tf32_transpose", 1)
        p = g.plan(a, b, precision="tf32", handle=h)
        assert p["stage_b"] == 1 and p["b_mn_major"] == 0
        assert p["workspace_bytes"] == 4096 * 4096 * 4
        h.close()
    for prec in ("exact", "default"):
        # Exact fp32: both operands split into tf32 [hi | lo] parts (2K columns each), read
        # as three K-long products.
        p = g.plan(a, b, precision=prec)
        assert p["path"] == "tcgen05_3xtf32" and p["tile_k"] == 32 and p["k_iters"] == 384
        assert p["stage_a"] == 1 and p["stage_b"] == 1
        assert p["a_mn_major"] == 0 and p["b_mn_major"] == 0
        assert p["workspace_bytes"] == 2 * 4096 * 2 * 4096 * 4
    # a ragged K pads each part to whole 32-long K-blocks: K = 1000 -> 1024 per part
    p = g.plan(t((300, 1000), torch.float32), t((1000, 200), torch.float32), precision="exact")
    assert p["path"] == "tcgen05_3xtf32" and p["k_iters"] == 3 * 32
    assert p["workspace_bytes"] == (300 + 200) * 2048 * 4
    # K = 1100 -> 1120 per part
    p = g.plan(t((300, 1100), torch.float32), t((1100, 200), torch.float32), precision="exact")
    assert p["workspace_bytes"] == 300 * 2240 * 4 + (256 - 300 * 2240 * 4 % 256) % 256 + 200 * 2240 * 4
    p = g.plan(t((16, 16), torch.float32), t((16, 16), torch.float32))
    assert p["path"] == "fma" and (p["tile_m"], p["tile_n"], p["tile_k"]) == (4, 4, 4)


def test_plan_fp16_accumulator():
    # Section 13.3's fp16 accumulator: chunks of one 16-long MMA on the tensor cores (CTA
    # pairs, 256 x 256 tiles); a row-major B is transposed into K-major form, since the
    # chunked kernel reads K-major operands only.
    a, b = t((4096, 1024), torch.float16), t((1024, 4096), torch.float16)
    p = g.plan(a, b, precision="f16acc", sm_count=148)
    assert p["path"] == "tcgen05_f16acc" and p["cta_pair"] == 1
    assert (p["tile_m"], p["tile_n"], p["tile_k"], p["k_iters"]) == (256, 256, 64, 16)
    assert p["stage_a"] == 0 and p["stage_b"] == 1 and p["b_mn_major"] == 0
    assert p["split_tiles"] == 0
    p = g.plan(a, t((4096, 1024), torch.float16).t(), precision="f16acc")
    assert p["stage_b"] == 0
    # the pages' 4 x 1024 @ 1024 x 4 example is tiny but keeps the tensor-core kernel
    p = g.plan(t((4, 1024), torch.float16), t((1024, 4), torch.float16), precision="f16acc")
    assert p["path"] == "tcgen05_f16acc"


def test_plan_degenerate_shapes():
    assert g.plan(t((0, 5), torch.float16), t((5, 7), torch.float16))["path"] == "none"
    assert g.plan(t((5, 3), torch.float16), t((3, 0), torch.float16))["path"] == "none"
    assert g.plan(t((5, 0), torch.float16), t((0, 7), torch.float16))["path"] == "zero_fill"


def plan_code(L, M, N, K, A, lda, B, ldb, C, ldc, in_dt=1, out_dt=0, prec=0, al=0, bl=0):
    info = g.PlanInfo()
    return L.gemm_plan(None, M, N, K, A, lda, B, ldb, C, ldc, in_dt, out_dt, prec, al, bl, 148,
                       ctypes.byref(info))


def test_plan_rejects_bad_arguments(L):
    A, B, C = 1 << 20, 1 << 24, 1 << 28
    assert plan_code(L, 16, 16, 16, A, 16, B, 16, C, 16) == 0
    assert plan_code(L, -1, 16, 16, A, 16, B, 16, C, 16) == 1        # negative size
    assert plan_code(L, 16, 16, 16, A, 15, B, 16, C, 16) == 1        # lda < K
    assert plan_code(L, 16, 16, 16, A, 16, B, 15, C, 16) == 1        # ldb < N
    assert plan_code(L, 16, 16, 16, A, 16, B, 16, C, 15) == 1        # ldc < N
    assert plan_code(L, 16, 16, 16, A, 8, B, 16, C, 16, al=1) == 1   # col-major A: lda < M
    assert plan_code(L, 16, 16, 16, None, 16, B, 16, C, 16) == 1     # null A
    assert plan_code(L, 16, 16, 16, A, 16, B, 16, None, 16) == 1     # null C
    assert plan_code(L, 16, 16, 16, A, 16, B, 16, C, 16, in_dt=7) == 1
    assert plan_code(L, 16, 16, 16, A, 16, B, 16, C, 16, al=3) == 1
    assert plan_code(L, 16, 16, 16, A, 16, B, 16, C, 16, prec=1) == 2  # tf32 with fp16 in
    assert plan_code(L, 16, 16, 16, A, 16, B, 16, C, 16, prec=3) == 0  # fp16 acc, fp16 in
    assert plan_code(L, 16, 16, 16, A, 16, B, 16, C, 16, prec=3, in_dt=2) == 2  # bf16 in
    assert plan_code(L, 16, 16, 16, A, 16, B, 16, C, 16, prec=3, in_dt=0) == 2  # fp32 in
    assert plan_code(L, 16, 16, 16, A, 16, B, 16, C, 16, prec=4) == 1  # unknown mode
    assert plan_code(L, 16, 16, 16, A + 1, 16, B, 16, C, 16) == 3      # odd fp16 address
    assert plan_code(L, 16, 16, 16, A, 16, B, 16, C + 2, 16) == 3      # fp32 C at 2 bytes
    assert plan_code(L, 16, 16, 16, A, 16, B, 16, A + 64, 16) == 1     # C overlaps A
    assert plan_code(L, 16, 16, 16, A, 16, B, 16, B - 16, 16) == 1     # C overlaps B
    assert plan_code(L, 0, 16, 16, None, 16, None, 16, None, 16) == 0  # empty: nothing needed
    assert plan_code(L, 16, 16, 0, None, 16, None, 16, C, 16) == 0     # K == 0: only C needed


def test_sources_share_nothing_with_the_oracle():
    csrc = os.path.join(ROOT, "dense_tiled_gemm_05_gb300")
    for dirpath, _, files in os.walk(csrc):
        for f in files:
            if f.endswith((".cu", ".cuh", ".h", ".py", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in text.lower(), f
    for f in os.listdir(os.path.join(ROOT, "oracle")):
        if f.endswith((".c", ".py")):
            text = open(os.path.join(ROOT, "oracle", f)).read()
            assert "dense_tiled_gemm_05_gb300" not in text and "gemm.h" not in text, f




def test_plan_tile_rows_default():
    """Rows per CTA of the pair kernel's tiles stay 128 unless the option asks otherwise
    (GEMM_OPT_TILE_ROWS; its checks need a handle and run with the GPU tests)."""
    for M, N, K in [(16384, 128, 8192), (24576, 128, 8192), (4096, 128, 8192), (5000, 100, 3000)]:
        p = g.plan(t((M, K), torch.bfloat16), t((K, N), torch.bfloat16, "col"), sm_count=148)
        assert p["cta_pair"] == 1 and p["tile_m"] == 256, (M, N, K)


def test_plan_split_k_rule():
    """Split-K shares out the last whole round plus the partial one when that is at most
    1.6 rounds' worth of tiles (and K has >= 64 K-blocks); few-tile long-K products split
    over idle clusters; compute-bound products take CTA pairs from 64 K-blocks on."""
    def plan(M, N, K, sms):
        return g.plan(t((M, K), torch.bfloat16), t((K, N), torch.bfloat16, "col"), sm_count=sms)
    # 100 tiles on 76 clusters: 1.32 rounds shared
    assert plan(2560, 2560, 8192, 152)["split_tiles"] == 100
    # 144 tiles: 1.89 rounds, kept whole
    assert plan(3072, 3072, 4096, 152)["split_tiles"] == 0
    # 8192^3: 1024 tiles; on 76 clusters the last 112 tiles (1.47 rounds) are shared, on 74
    # the last 136 (1.84) are not
    assert plan(8192, 8192, 8192, 152)["split_tiles"] == 112
    assert plan(8192, 8192, 8192, 148)["split_tiles"] == 0
    # short K (32 K-blocks): never
    assert plan(8192, 8192, 2048, 152)["split_tiles"] == 0
    # fewer tiles than clusters but more than half: whole tiles
    p = plan(2048, 2048, 8192, 152)
    assert p["cta_pair"] == 1 and p["split_tiles"] == 0 and p["ctas"] == 128
    # compute-bound, all single-CTA tiles in one round: single CTAs for 32 K-blocks, pairs
    # from 64 on
    assert plan(2048, 2048, 2048, 152)["cta_pair"] == 0
    assert plan(2048, 2048, 4096, 152)["cta_pair"] == 1
    # 2560^2: 256-wide tiles (128-wide ones cost 0.8 of a 256-wide one's time, too much
    # for the rounds they save)
    assert plan(2560, 2560, 8192, 152)["tile_n"] == 256


def test_plan_short_k_takes_the_fma_kernel():
    """A short K with a moderate output runs on the FMA kernel (one launch that reads any
    alignment); a longer K, a large output, or a tensor-core tile asked for keeps the
    tensor cores."""
    f16 = torch.float16
    assert g.plan(t((1000, 17), f16), t((17, 1000), f16), out_dtype="f32")["path"] == "fma"
    assert g.plan(t((1025, 1), f16), t((1, 1025), f16), out_dtype="f32")["path"] == "fma"
    assert g.plan(t((2048, 24), f16), t((24, 2048), f16), out_dtype="f32")["path"] == "fma"
    assert g.plan(t((1000, 127), f16), t((127, 1000), f16), out_dtype="f32")["path"] == "tcgen05"
    assert g.plan(t((1000, 25), f16), t((25, 1000), f16), out_dtype="f32")["path"] == "tcgen05"
    assert g.plan(t((8192, 16), f16), t((16, 8192), f16), out_dtype="f32")["path"] == "tcgen05"


def test_plan_fma_tile_kinds():
    """The FMA kernel's K-chunk: 4 for the pages' 4 x 4 x 4 tiles, 8 under the fp16
    accumulator (whose chunks are multiples of 8, e.g. the pages' BLOCK_K = 8), 16 for the
    other 128 x 128 tiles."""
    f16, f32 = torch.float16, torch.float32
    p = g.plan(t((1000, 17), f16), t((17, 1000), f16), out_dtype="f32")
    assert p["path"] == "fma" and (p["tile_m"], p["tile_n"], p["tile_k"]) == (128, 128, 16)
    assert p["k_iters"] == 2
    p = g.plan(t((16, 16), f32), t((16, 16), f32), precision="exact")
    assert p["path"] == "fma" and (p["tile_m"], p["tile_n"], p["tile_k"]) == (4, 4, 4)
    # a short K under the fp16 accumulator: the FMA kernel with 8-long chunks
    p = g.plan(t((64, 16), f16), t((16, 64), f16), out_dtype="f16", precision="f16acc")
    assert p["path"] == "fma" and (p["tile_k"], p["k_iters"]) == (8, 2)
    p = g.plan(t((64, 64), f16), t((64, 64), f16), out_dtype="f16", precision="f16acc")
    assert p["path"] == "tcgen05_f16acc"
    p = g.plan(t((8, 40), f16), t((40, 8), f16), out_dtype="f16", precision="f16acc")
    assert p["path"] == "tcgen05_f16acc"  # K = 40 is past the short-K limit
