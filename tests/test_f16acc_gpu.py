"""The fp16-accumulator mode (GEMM_PREC_F16_ACC): "Chapter 13: The Blocked Matmul Kernel",
section 13.3, Worked Example 13.3.1. The running total is an fp16 value; after every K-chunk
the chunk's dot product is rounded to fp16 and added to it with an fp16 add. Compared with
the oracle's definition of the same arithmetic (oracle.gemm_f16acc, pinned to the pages'
printed 0.001974425897060428): bitwise on integer inputs, where every chunk dot is exact in
fp32 so both sides take the same roundings, and within a few fp16 ulps on real inputs, where
a chunk dot summed in a different order may round to the neighbouring fp16 value."""
import itertools

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_util import oracle_rows, to_device

pytestmark = pytest.mark.gpu

F16ACC_MAX_ABS_DIFF = 0.001974425897060428  # Worked Example 13.3.1, BLOCK_K = 8


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import dense_tiled_gemm_05_gb300 as g
    return g


def handle(g, chunk, force_path=0):
    h = g.Gemm(0)
    h.set_option("acc_chunk", chunk)
    h.set_option("force_path", force_path)
    return h


def run(h, p, out_dtype=None):
    c = h.matmul(to_device(p.A), to_device(p.B), out_dtype=out_dtype or p.out_dtype,
                 precision="f16acc")
    torch.cuda.synchronize()
    assert h.status() == 0
    return c.cpu().double().numpy()


def oracle_f16acc(p, chunk):
    a, al, lda = W.storage_numpy(p.A)
    b, bl, ldb = W.storage_numpy(p.B)
    return oracle.gemm_f16acc(a, b, p.M, p.N, p.K, lda=lda, ldb=ldb, a_dtype="f16",
                              b_dtype="f16", BK=chunk, a_layout=al, b_layout=bl)


def f16_ulp(x):
    """Spacing of fp16 values at |x| (subnormal spacing below the normal range)."""
    ax = np.maximum(np.abs(x), 2.0 ** -14)
    return 2.0 ** (np.floor(np.log2(ax)) - 10)


# (M, N, K): the pages' 4 x 4 x 1024; ragged, several tiles, a ragged last chunk; a long K
# whose integer totals pass 2048, where fp16 itself starts rounding them
INT_SHAPES = [(4, 4, 1024), (300, 257, 1025), (129, 640, 4100)]


@pytest.mark.parametrize("chunk,force_path", [(8, 0), (16, 0), (48, 0), (256, 0), (16, 2)])
@pytest.mark.parametrize("a_layout,b_layout", list(itertools.product(["row", "col"], repeat=2)))
def test_f16acc_integer_bit_exact(g, chunk, force_path, a_layout, b_layout):
    h = handle(g, chunk, force_path)
    for n, (M, N, K) in enumerate(INT_SHAPES):
        p = W.integer_problem(M, N, K, "f16", seed=800 + n, a_layout=a_layout,
                              b_layout=b_layout, out_dtype="f16", precision="f16acc",
                              ld_pad=n % 3)
        ref = oracle_f16acc(p, chunk)
        c = run(h, p)
        assert np.array_equal(c, ref), (M, N, K, chunk, int(np.sum(c != ref)))
        if n == 1:  # the fp16 total widened exactly to fp32, and rounded to bf16
            assert np.array_equal(run(h, p, "f32"), ref)
            assert np.array_equal(run(h, p, "bf16"), oracle.round_to(ref, "bf16"))
    h.close()


@pytest.mark.parametrize("chunk", [8, 16])
def test_f16acc_pages_example(g, chunk):
    """Worked Example 13.3.1: fp16 4 x 1024 @ 1024 x 4 from seed 0; the fp16 accumulator
    drifts about twenty times further from the fp64 product than the fp32 one."""
    p = W.accumulation_13_3_1()
    C64, _ = oracle_rows(p)
    h = handle(g, chunk)
    c16 = run(h, p, "f16")
    ref = oracle_f16acc(p, chunk)
    assert np.all(np.abs(c16 - ref) <= f16_ulp(ref)), np.max(np.abs(c16 - ref))
    err16 = float(np.max(np.abs(c16 - C64)))
    c32 = h.matmul(to_device(p.A), to_device(p.B), out_dtype="f16").cpu().double().numpy()
    err32 = float(np.max(np.abs(c32 - C64)))
    assert err16 > 5 * err32
    if chunk == 8:  # the pages' BLOCK_K: their printed deviation, to within an fp16 ulp
        assert abs(err16 - F16ACC_MAX_ABS_DIFF) <= 2.0 ** -10
    h.close()


def running_total_bound(p, chunk, block=64):
    """max over chunks t of |sum of the first t chunk dots|, per element, in fp64: the
    largest magnitude the running total passes through, which sets the fp16 spacing at
    which a rounding decided differently on the two sides can shift the result."""
    M, N, K = p.M, p.N, p.K
    C = -(-K // chunk)
    A = np.zeros((M, C * chunk))
    A[:, :K] = p.A.double().numpy()
    Bt = np.zeros((N, C * chunk))
    Bt[:, :K] = p.B.double().numpy().T
    A3 = A.reshape(M, C, chunk)
    S = np.empty((M, N))
    for j0 in range(0, N, block):
        P = np.einsum("mck,nck->mnc", A3, Bt[j0:j0 + block].reshape(-1, C, chunk))
        S[:, j0:j0 + block] = np.max(np.abs(np.cumsum(P, axis=2)), axis=2)
    return S


@pytest.mark.parametrize("chunk", [16, 64])
@pytest.mark.parametrize("M,N,K", [(1000, 1023, 1025), (256, 512, 4096)])
def test_f16acc_random_within_ulps(g, chunk, M, N, K):
    """Real-valued inputs: a chunk dot summed in another order than the oracle's can round
    to the neighbouring fp16 value, and the running total then differs by about one fp16
    spacing at the magnitude it had; such events are rare, so nearly every element is
    bitwise equal and the rest are within a few spacings of the largest running total."""
    p = W.ragged(M, N, K, seed=900 + K, dtype="f16")
    h = handle(g, chunk)
    c = run(h, p, "f16")
    ref = oracle_f16acc(p, chunk)
    diff = np.abs(c - ref)
    bound = 4 * f16_ulp(running_total_bound(p, chunk))
    assert np.all(diff <= bound), float(np.max(diff / bound))
    assert np.mean(diff == 0) >= 0.99, float(np.mean(diff == 0))
    h.close()


def test_f16acc_guard_band_and_k_zero(g):
    h = handle(g, 16)
    p = W.integer_problem(300, 70, 200, "f16", seed=950, precision="f16acc", out_dtype="f16")
    big = torch.full((300, 80), float("nan"), dtype=torch.float16, device="cuda")
    out = big[:, :70]
    h.matmul(to_device(p.A), to_device(p.B), out=out, precision="f16acc")
    torch.cuda.synchronize()
    assert h.status() == 0
    assert np.array_equal(out.cpu().double().numpy(), oracle_f16acc(p, 16))
    assert torch.isnan(big[:, 70:]).all()
    a = torch.empty((5, 0), dtype=torch.float16, device="cuda")
    b = torch.empty((0, 7), dtype=torch.float16, device="cuda")
    z = h.matmul(a, b, precision="f16acc")
    torch.cuda.synchronize()
    assert torch.equal(z.cpu(), torch.zeros(5, 7, dtype=torch.float16))
    h.close()


def test_f16acc_rejections(g):
    h = g.Gemm(0)
    with pytest.raises(g.GemmError):
        h.set_option("acc_chunk", 12)
    bf = torch.ones((4, 4), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(g.GemmError):
        h.matmul(bf, bf, precision="f16acc")
    h.set_option("acc_chunk", 8)
    h.set_option("force_path", 1)  # tensor cores cannot round every 8 K
    f = torch.ones((4, 4), dtype=torch.float16, device="cuda")
    with pytest.raises(g.GemmError):
        h.matmul(f, f, precision="f16acc")
    h.close()


def test_f16acc_bench_size_sampled(g):
    """The measured fp16-accumulator workload (fp16 4096^3, N(0,1) * 0.1, chunk 16) in the
    bench's launch configuration: sampled rows against the oracle's definition."""
    p = W.f16acc_square(4096)
    h = g.Gemm(0)
    c = h.matmul(to_device(p.A), to_device(p.B), out_dtype="f16", precision="f16acc")
    torch.cuda.synchronize()
    assert h.status() == 0
    rows = [0, 255, 256, 2047, 4095, 1234]
    sub = W.Problem("rows", p.A[rows], p.B, "f16", "f16acc")
    ref = oracle_f16acc(sub, 16)
    got = c[rows].cpu().double().numpy()
    diff = np.abs(got - ref)
    bound = 4 * f16_ulp(running_total_bound(sub, 16))
    assert np.all(diff <= bound)
    assert np.mean(diff == 0) >= 0.99
    h.close()
