"""Row softmax on the GPU ("Triton from zero, Lesson 4: Block Pointers", homework 4) against
the fp64 oracle: every row length class of the kernels (one warp, one CTA with 1..32 values
per thread, the two-pass kernel for longer rows), ragged lengths, all dtype pairs, padded
leading dimensions with poisoned padding, in place, and the special values the formula
turns into 0 or NaN."""
import itertools
import math

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

TORCH = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
# relative bound (fp32 arithmetic, then the output rounding) and absolute floor (underflow)
TOL = {"f32": (1e-5, 1e-37), "f16": (2.0 ** -10, 2.0 ** -24), "bf16": (2.0 ** -7, 1e-37)}


@pytest.fixture(scope="module")
def h():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import dense_tiled_gemm_05_gb300 as g
    hh = g.Gemm(0)
    yield hh
    hh.close()


def raw(t):
    t = t.contiguous()
    if t.dtype in (torch.float16, torch.bfloat16):
        return t.view(torch.int16).numpy().view(np.uint16).reshape(-1)
    return t.numpy().reshape(-1)


def reference(x_store, M, N, ldx, dtype):
    return oracle.softmax_rows(raw(x_store), M, N, ldx=ldx, x_dtype=dtype)


def check(y, ref, out_dtype):
    rtol, atol = TOL[out_dtype]
    y = y.double().cpu().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(y), nan)
    err = np.abs(y[~nan] - ref[~nan])
    assert np.all(err <= rtol * ref[~nan] + atol), float(np.max(err - rtol * ref[~nan]))


def make(M, N, dtype, seed, ld_pad=0, scale=3.0):
    gen = torch.Generator().manual_seed(seed)
    store = (torch.randn(M, N + ld_pad, generator=gen) * scale).to(TORCH[dtype])
    if ld_pad:
        store[:, N:] = float("nan")  # poisoned padding: never read
    return store


SHAPES = [(1, 1), (3, 7), (5, 31), (4, 32), (4, 33), (64, 127), (17, 1000), (8, 1023),
          (8, 1025), (16, 4096), (4, 8192), (2, 32768), (2, 32772), (2, 100003)]


@pytest.mark.parametrize("M,N", SHAPES)
def test_softmax_f32_lengths(h, M, N):
    store = make(M, N, "f32", seed=N)
    y = h.softmax_rows(store.cuda())
    torch.cuda.synchronize()
    check(y, reference(store, M, N, N, "f32"), "f32")


@pytest.mark.parametrize("din,dout", list(itertools.product(["f32", "f16", "bf16"], repeat=2)))
@pytest.mark.parametrize("M,N,pad", [(33, 300, 0), (9, 4100, 3), (3, 40000, 8)])
def test_softmax_dtypes_and_padding(h, din, dout, M, N, pad):
    store = make(M, N, din, seed=7 * N + pad, ld_pad=pad)
    x = store.cuda()[:, :N]
    out_store = torch.full((M, N + 5), float("nan"), dtype=TORCH[dout], device="cuda")
    y = out_store[:, :N]
    h.softmax_rows(x, out=y)
    torch.cuda.synchronize()
    check(y, reference(store, M, N, N + pad, din), dout)
    assert torch.isnan(out_store[:, N:].float()).all()  # tails of Y untouched


def test_softmax_in_place_and_unaligned_rows(h):
    store = make(40, 1001, "f32", seed=3)
    ref = reference(store, 40, 1001, 1001, "f32")  # ld 1001: rows not 16-byte aligned
    x = store.cuda()
    h.softmax_rows(x, out=x)
    torch.cuda.synchronize()
    check(x, ref, "f32")


@pytest.mark.parametrize("N", [6, 5000, 50000])
def test_softmax_special_values(h, N):
    inf, nan = math.inf, math.nan
    rows = np.random.default_rng(N).normal(size=(6, N)).astype(np.float32)
    rows[0, :] = -inf
    rows[0, N // 2] = 1.5           # one finite value: 1 there, exactly 0 elsewhere
    rows[1, :] = -inf               # all -inf: NaN
    rows[2, N // 3] = nan           # NaN: NaN row
    rows[3, N - 1] = inf            # +inf: NaN row
    rows[4, :] *= 1000.0            # large magnitudes: no overflow
    rows[5, ::2] = -inf             # half the row masked
    store = torch.from_numpy(rows)
    y = h.softmax_rows(store.cuda())
    torch.cuda.synchronize()
    ref = reference(store, 6, N, N, "f32")
    check(y, ref, "f32")
    yc = y.cpu()
    assert yc[0, N // 2] == 1.0 and (yc[0, :N // 2] == 0).all()
    assert torch.isnan(yc[1:4]).all()
    assert (yc[5, ::2] == 0).all()


def test_softmax_rejects_overlap(h):
    import dense_tiled_gemm_05_gb300 as g
    x = torch.randn(8, 64, device="cuda")
    with pytest.raises(g.GemmError):
        h.softmax_rows(x[:, :32], out=x[:, 16:48])


def test_softmax_bench_size_sampled(h):
    """The measured workload, 16384 x 8192 fp32 (N(0,1) * 3 entries, the bench's seed), in the
    launch configuration the bench times: sampled rows against the oracle, and every row's
    sum equal to 1 within fp32 rounding."""
    import bench
    x = bench.softmax_input(16384, 8192)
    y = h.softmax_rows(x.cuda())
    torch.cuda.synchronize()
    rows = sorted(set([0, 1, 8191, 16383] + list(np.random.default_rng(5).integers(0, 16384, 60))))
    ref = oracle.softmax_rows(x[rows].numpy().reshape(-1), len(rows), 8192, ldx=8192,
                              x_dtype="f32")
    check(y[rows], ref, "f32")
    sums = y.double().sum(dim=1).cpu()
    assert torch.all((sums - 1.0).abs() < 1e-4)
