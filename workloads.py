"""Seeded synthetic inputs for the blocked GEMM workloads.

This module only draws random numbers (torch's CPU generator, so every host
produces the same bits) and casts them to the storage dtype with torch's
round-to-nearest-even cast. It holds none of the product's arithmetic; the
tests, the benchmark and the smoke check hand the same tensors to the GPU
library and to the CPU oracle.

A :class:`Problem` carries the two operands as *logical* torch views
(``A`` is M x K, ``B`` is K x N) whose strides encode the storage layout:

* row-major operand: stride ``(ld, 1)``;
* column-major operand: stride ``(1, ld)`` (storage is the transpose).

Workloads (value distributions, sizes and layouts):

* ``small_exact``: fp32 8x8x8, uniform[-1, 1], seed 0 -- plus the fixed 2x2 check;
* ``ragged``: fp16 in, fp32 out, M, N, K each in {1, 17, 127, 1000, 1023, 1025},
  uniform[-1, 1], row-major, tight leading dimensions, seed 1000 + combo index;
* ``bf16_square(n)``: bf16, A row-major, B column-major, N(0, 1)/sqrt(K), bf16 out;
* ``fp32_square(n)``: fp32 row-major, uniform[-1, 1], fp32 out (tf32 or exact mode);
* ``bf16_skinny``: bf16 M=16384, N=128, K=8192, N(0, 1)/sqrt(K), bf16 out.
"""
from dataclasses import dataclass, field
import itertools

import numpy as np
import torch

TORCH_DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16,
                "f64": torch.float64}
RAGGED_SIZES = (1, 17, 127, 1000, 1023, 1025)


@dataclass
class Problem:
    name: str
    A: torch.Tensor  # logical M x K view
    B: torch.Tensor  # logical K x N view
    out_dtype: str
    precision: str = "default"  # "default" | "tf32" | "exact"
    meta: dict = field(default_factory=dict)

    @property
    def M(self):
        return self.A.shape[0]

    @property
    def K(self):
        return self.A.shape[1]

    @property
    def N(self):
        return self.B.shape[1]

    @property
    def in_dtype(self):
        return dtype_name(self.A.dtype)


def dtype_name(t):
    for k, v in TORCH_DTYPES.items():
        if v == t:
            return k
    raise TypeError("unsupported dtype %s" % t)


def layout_of(x):
    """("row", ld) or ("col", ld) for a 2-D logical view."""
    r, c = x.shape
    s0, s1 = x.stride()
    if s1 == 1 and (s0 >= max(c, 1) or r <= 1):
        return "row", max(s0, c, 1)
    if s0 == 1 and (s1 >= max(r, 1) or c <= 1):
        return "col", max(s1, r, 1)
    raise ValueError("operand is neither row- nor column-major: shape %s stride %s"
                     % (tuple(x.shape), x.stride()))


def storage_numpy(x):
    """The raw storage behind a logical view as a flat numpy array plus (layout, ld).

    f16/bf16 come back as uint16 bit patterns. The flat array starts at the
    view's first element, so (layout, ld) index it directly.
    """
    layout, ld = layout_of(x)
    r, c = x.shape
    outer, inner = (r, c) if layout == "row" else (c, r)
    n = 0 if r == 0 or c == 0 else (outer - 1) * ld + inner
    flat = torch.as_strided(x, (n,), (1,), x.storage_offset()) if n else x.new_empty(0)
    flat = flat.contiguous()
    if x.dtype in (torch.float16, torch.bfloat16):
        arr = flat.view(torch.int16).numpy().view(np.uint16)
    else:
        arr = flat.numpy()
    return arr, layout, ld


def _gen(seed):
    return torch.Generator().manual_seed(int(seed))


def uniform(shape, dtype, seed, lo=-1.0, hi=1.0):
    g = _gen(seed)
    x = torch.rand(shape, generator=g, dtype=torch.float32) * (hi - lo) + lo
    return x.to(TORCH_DTYPES[dtype])


def normal_scaled(shape, dtype, seed, scale):
    g = _gen(seed)
    x = torch.randn(shape, generator=g, dtype=torch.float32) * scale
    return x.to(TORCH_DTYPES[dtype])


def integers(shape, dtype, seed, lo=-4, hi=4):
    """Integer values in [lo, hi]; exact in every supported input format."""
    g = _gen(seed)
    x = torch.randint(lo, hi + 1, shape, generator=g, dtype=torch.int32)
    return x.to(TORCH_DTYPES[dtype])


def make_operand(rows, cols, dtype, layout, seed, kind="uniform", ld_pad=0, **kw):
    """A logical rows x cols operand in the given layout, leading dim padded by ld_pad."""
    if layout == "row":
        store_shape = (rows, cols + ld_pad)
    else:
        store_shape = (cols, rows + ld_pad)
    if kind == "uniform":
        s = uniform(store_shape, dtype, seed, kw.get("lo", -1.0), kw.get("hi", 1.0))
    elif kind == "normal":
        s = normal_scaled(store_shape, dtype, seed, kw["scale"])
    elif kind == "int":
        s = integers(store_shape, dtype, seed, kw.get("lo", -4), kw.get("hi", 4))
    else:
        raise ValueError(kind)
    if layout == "row":
        return s[:, :cols]
    return s[:, :rows].t()


# ------------------------------------------------------------------ workloads

def two_by_two(dtype="f32"):
    """[[1,2],[3,4]] @ [[5,6],[7,8]]; its product is [[19,22],[43,50]]."""
    t = TORCH_DTYPES[dtype]
    A = torch.tensor([[1.0, 2.0], [3.0, 4.0]]).to(t)
    B = torch.tensor([[5.0, 6.0], [7.0, 8.0]]).to(t)
    out = "f32" if dtype in ("f16", "bf16") else dtype
    return Problem("two_by_two_%s" % dtype, A, B, out, "exact" if dtype == "f32" else "default")


def small_exact(seed=0):
    """fp32 8x8 @ 8x8, uniform[-1, 1], row-major, exact-fp32 mode."""
    A = make_operand(8, 8, "f32", "row", seed * 2 + 0)
    B = make_operand(8, 8, "f32", "row", seed * 2 + 1)
    return Problem("small_exact_8x8x8", A, B, "f32", "exact", {"tiles": (4, 4, 4)})


def ragged_combos():
    return list(itertools.product(RAGGED_SIZES, RAGGED_SIZES, RAGGED_SIZES))


def ragged(M, N, K, seed=None, dtype="f16"):
    """A[M,K] @ B[K,N] (fp16 by default), uniform[-1, 1], row-major with tight leading dims,
    fp32 out; fp32 inputs run in exact mode."""
    if seed is None:
        seed = 1000 + ragged_combos().index((M, N, K))
    A = make_operand(M, K, dtype, "row", 2 * seed)
    B = make_operand(K, N, dtype, "row", 2 * seed + 1)
    prec = "exact" if dtype == "f32" else "default"
    return Problem("ragged_%s_%dx%dx%d" % (dtype, M, N, K), A, B, "f32", prec)


def bf16_square(n, seed=2, b_layout="col"):
    """bf16 n^3: A row-major, B column-major, N(0,1)/sqrt(K), bf16 out."""
    s = 1.0 / np.sqrt(n)
    A = make_operand(n, n, "bf16", "row", 2 * seed, "normal", scale=s)
    B = make_operand(n, n, "bf16", b_layout, 2 * seed + 1, "normal", scale=s)
    return Problem("bf16_%d^3" % n, A, B, "bf16", "default")


def f16acc_square(n, seed=6):
    """fp16 n^3 in the fp16-accumulator mode: A row-major, B column-major, entries
    N(0,1) * 0.1 (the scale of the 13.3.1 example), fp16 out."""
    A = make_operand(n, n, "f16", "row", 2 * seed, "normal", scale=0.1)
    B = make_operand(n, n, "f16", "col", 2 * seed + 1, "normal", scale=0.1)
    return Problem("f16acc_%d^3" % n, A, B, "f16", "f16acc")


def fp32_square(n, precision, seed=3):
    """fp32 n^3 row-major, uniform[-1, 1], fp32 out, tf32 or exact mode."""
    A = make_operand(n, n, "f32", "row", 2 * seed)
    B = make_operand(n, n, "f32", "row", 2 * seed + 1)
    return Problem("fp32_%d^3_%s" % (n, precision), A, B, "f32", precision)


def bf16_skinny(M=16384, N=128, K=8192, seed=4, b_layout="col"):
    """bf16 M x N x K skinny (memory-bound), N(0,1)/sqrt(K), bf16 out."""
    s = 1.0 / np.sqrt(K)
    A = make_operand(M, K, "bf16", "row", 2 * seed, "normal", scale=s)
    B = make_operand(K, N, "bf16", b_layout, 2 * seed + 1, "normal", scale=s)
    return Problem("bf16_skinny_%dx%dx%d" % (M, N, K), A, B, "bf16", "default")


def integer_problem(M, N, K, dtype, seed, a_layout="row", b_layout="row", out_dtype="f32",
                    precision="default", ld_pad=0):
    """Integer-valued inputs in [-4, 4]: every partial sum is an exact fp32 integer for K <= 1025."""
    A = make_operand(M, K, dtype, a_layout, 2 * seed, "int", ld_pad=ld_pad)
    B = make_operand(K, N, dtype, b_layout, 2 * seed + 1, "int", ld_pad=ld_pad)
    if dtype == "f32" and precision == "default":
        precision = "exact"
    return Problem("int_%s_%dx%dx%d" % (dtype, M, N, K), A, B, out_dtype, precision)


def arange_tenths(M, K, N, dtype="f32"):
    """The pages' deterministic operands: A[i,k] = 0.1*(K*i + k), B[k,j] = 0.1*(N*k + j)."""
    t = TORCH_DTYPES[dtype]
    A = (torch.arange(M * K, dtype=torch.float64).reshape(M, K) * 0.1).to(t)
    B = (torch.arange(K * N, dtype=torch.float64).reshape(K, N) * 0.1).to(t)
    return Problem("arange_%dx%dx%d" % (M, K, N), A, B, dtype)


def sentinel_padded(M=4, K_real=5, N=4, K_pad=8, sentinel=999.0, dtype="f32"):
    """Operands sliced out of sentinel-filled parents (row tails past K hold the sentinel)."""
    t = TORCH_DTYPES[dtype]
    Ap = torch.full((M, K_pad), sentinel, dtype=torch.float64)
    Ap[:, :K_real] = torch.arange(M * K_real, dtype=torch.float64).reshape(M, K_real) * 0.1
    Bp = torch.full((K_pad, N), sentinel, dtype=torch.float64)
    Bp[:K_real, :] = torch.arange(K_real * N, dtype=torch.float64).reshape(K_real, N) * 0.1
    Ap, Bp = Ap.to(t), Bp.to(t)
    return Problem("sentinel_%dx%dx%d" % (M, K_real, N), Ap[:, :K_real], Bp[:K_real, :], dtype,
                   "exact" if dtype == "f32" else "default",
                   {"A_parent": Ap, "B_parent": Bp, "K_pad": K_pad})


def accumulation_13_3_1():
    """fp16 4x1024 @ 1024x4 from torch.manual_seed(0), randn*0.1 (A drawn first, then B)."""
    g = _gen(0)  # same stream as torch.manual_seed(0) on the default CPU generator
    A = (torch.randn(4, 1024, generator=g) * 0.1).to(torch.float16)
    B = (torch.randn(1024, 4, generator=g) * 0.1).to(torch.float16)
    return Problem("accumulation_4x1024x4", A, B, "f16")
