"""Helpers for the GPU parity tests: move seeded operands to the device with their
layout intact, run the library through its C ABI, and score the result against the
CPU oracle with the relative metric max |C_gpu - C| / sum_k |a_ik b_kj|."""
import numpy as np
import torch

import oracle
import workloads as W

# Relative-error bounds per input dtype / precision mode (max |err| / D).
TOL = {("f32", "exact"): 1e-6, ("f32", "default"): 1e-6, ("f32", "tf32"): 2e-3,
       ("f16", "default"): 1e-2, ("bf16", "default"): 1e-2}


def tolerance(p):
    return TOL[(p.in_dtype, p.precision)]


def to_device(x, device="cuda"):
    """Copy a logical view's storage span to the device and rebuild the same view."""
    layout, ld = W.layout_of(x)
    r, c = x.shape
    outer, inner = (r, c) if layout == "row" else (c, r)
    n = (outer - 1) * ld + inner if r and c else 0
    if n == 0:
        return torch.empty(x.shape, dtype=x.dtype, device=device)
    flat = torch.as_strided(x, (n,), (1,), x.storage_offset()).contiguous().to(device)
    return torch.as_strided(flat, x.shape, x.stride(), 0)


def run_gpu(h, p, out=None, stream=None):
    """Run the problem on the GPU through the library; returns C (device) after checking
    that the device status word is clean."""
    a, b = to_device(p.A), to_device(p.B)
    c = h.matmul(a, b, out=out, out_dtype=p.out_dtype, precision=p.precision, stream=stream)
    torch.cuda.synchronize()
    status = h.status()
    assert status == 0, "device status %d" % status
    return c


def oracle_rows(p, rows=None):
    a, al, lda = W.storage_numpy(p.A)
    b, bl, ldb = W.storage_numpy(p.B)
    return oracle.gemm_f64(a, b, p.M, p.N, p.K, lda=lda, ldb=ldb, a_dtype=p.in_dtype,
                           b_dtype=W.dtype_name(p.B.dtype), a_layout=al, b_layout=bl, rows=rows)


def rel_err(c_gpu, C64, D):
    """max |c - C64| / D over elements with D > 0; elements with D == 0 must be exactly 0."""
    c = c_gpu.double().cpu().numpy() if torch.is_tensor(c_gpu) else np.asarray(c_gpu)
    assert np.all(np.isfinite(c)), "non-finite output"
    zero = D == 0
    assert np.all(c[zero] == 0), "non-zero output where no product contributes"
    if not np.any(~zero):
        return 0.0
    return float(np.max(np.abs(c[~zero] - C64[~zero]) / D[~zero]))


def sample_rows(M, tile=256, n_random=256, seed=0):
    """Rows i = 0, 127, 128 and 255 mod 256 of every 256-row tile-row (the first and last
    rows of both CTAs of a pair tile, and of every 128-row single-CTA tile), the last row,
    plus n_random random rows."""
    rows = set()
    for t0 in range(0, M, tile):
        for r in (0, tile // 2 - 1, tile // 2, tile - 1):
            if t0 + r < M:
                rows.add(t0 + r)
    rows.add(M - 1)
    rng = np.random.default_rng(seed)
    rows.update(rng.integers(0, M, n_random).tolist())
    return sorted(rows)


def check_sampled(p, c_gpu, rows=None):
    rows = sample_rows(p.M) if rows is None else rows
    C64, D = oracle_rows(p, rows)
    return rel_err(c_gpu[rows], C64, D)


def check_full(p, c_gpu, oracle_result=None):
    """Every element of C against the oracle's full product (computed here unless given)."""
    C64, D = oracle_rows(p) if oracle_result is None else oracle_result
    return rel_err(c_gpu, C64, D)


def check_sums(p, c_gpu):
    """Row and column sums of the whole output against the oracle, for every row/column.

    sum_j C[i,j] = sum_k A[i,k] (sum_j B[k,j]) and sum_i C[i,j] = sum_k (sum_i A[i,k]) B[k,j],
    each bounded by the same relative metric with the summed magnitudes."""
    a, al, lda = W.storage_numpy(p.A)
    b, bl, ldb = W.storage_numpy(p.B)
    adt, bdt = p.in_dtype, W.dtype_name(p.B.dtype)
    M, N, K = p.M, p.N, p.K
    c = c_gpu.double().cpu().numpy()
    tol = tolerance(p)
    # rows: s = B 1 and u = |B| 1 (as K x 1), then t = A s, w = |A| u
    ones_n = np.ones(N, np.float64)
    # (B's own storage read as a K x N left operand, same layout and leading dimension)
    s, u = oracle.gemm_f64(b, ones_n, K, 1, N, lda=ldb, ldb=1, a_dtype=bdt, b_dtype="f64",
                           a_layout=bl)
    t, _ = oracle.gemm_f64(a, s.reshape(-1), M, 1, K, lda=lda, ldb=1, a_dtype=adt, b_dtype="f64",
                           a_layout=al)
    _, w = oracle.gemm_f64(a, u.reshape(-1), M, 1, K, lda=lda, ldb=1, a_dtype=adt, b_dtype="f64",
                           a_layout=al)
    row_err = np.max(np.abs(c.sum(axis=1) - t[:, 0]) / np.maximum(w[:, 0], 1e-300))
    # columns: q = 1^T A (as 1 x K), then r = q B, with magnitudes
    ones_m = np.ones(M, np.float64)
    q, qa = oracle.gemm_f64(ones_m, a, 1, K, M, lda=M, ldb=lda, a_dtype="f64", b_dtype=adt,
                            b_layout=al)
    r, _ = oracle.gemm_f64(q.reshape(-1), b, 1, N, K, lda=K, ldb=ldb, a_dtype="f64", b_dtype=bdt,
                           b_layout=bl)
    _, colmag = oracle.gemm_f64(qa.reshape(-1), b, 1, N, K, lda=K, ldb=ldb, a_dtype="f64",
                                b_dtype=bdt, b_layout=bl)
    col_err = np.max(np.abs(c.sum(axis=0) - r[0]) / np.maximum(colmag[0], 1e-300))
    return max(row_err, col_err), tol
