"""Failure detection on the GPU without a GPU fault: the tensor-core kernel's loader
is told to issue nothing, or to stop after some stage fills with copies still in flight,
so the MMA and epilogue roles' bounded mbarrier waits expire after a short limit; the
kernel records GEMM_ERR_TIMEOUT in the handle's status word, lets every copy it issued
land, releases its TMEM and returns. The same context then runs a normal GEMM correctly."""
import pytest
import torch

import workloads as W
from gpu_util import oracle_rows, rel_err, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import dense_tiled_gemm_05_gb300 as g
    from dense_tiled_gemm_05_gb300 import build as gbuild
    gbuild.build()
    return g


@pytest.mark.parametrize("cta_pair", [1, 2])
def test_bounded_wait_expires_and_context_stays_usable(g, cta_pair):
    p = W.bf16_square(512)
    a, b = to_device(p.A), to_device(p.B)
    h = g.Gemm(0)
    h.set_option("cta_pair", cta_pair)
    h.set_option("wait_timeout_us", 20000)  # 20 ms
    h.set_option("fault_stall_producer", 1)
    h.matmul(a, b)  # launches; the failure is found on the device
    assert h.status() == 6  # GEMM_ERR_TIMEOUT
    assert h.status() == 0  # reading the status clears it
    h.set_option("fault_stall_producer", 0)
    c = h.matmul(a, b)
    assert h.status() == 0
    C64, D = oracle_rows(p)
    assert rel_err(c, C64, D) <= 1e-2
    h.close()


def test_timeout_then_other_handles_unaffected(g):
    p = W.integer_problem(300, 400, 500, "f16", seed=3)
    a, b = to_device(p.A), to_device(p.B)
    bad, good = g.Gemm(0), g.Gemm(0)
    bad.set_option("wait_timeout_us", 10000)
    bad.set_option("fault_stall_producer", 1)
    bad.matmul(a, b, out_dtype="f32")
    c = good.matmul(a, b, out_dtype="f32")
    assert bad.status() == 6
    assert good.status() == 0
    assert torch.equal(c.cpu().to(torch.int64), p.A.to(torch.int64) @ p.B.to(torch.int64))
    bad.close()
    good.close()


def test_workspace_allocation_failure_is_reported(g, monkeypatch):
    # Host-side fault injection: the staging workspace cannot be allocated.
    monkeypatch.setenv("GEMM_FAULT_INJECT", "alloc")
    p = W.ragged(127, 17, 1025)  # misaligned rows: needs the staging workspace
    a, b = to_device(p.A), to_device(p.B)
    h = g.Gemm(0)
    with pytest.raises(g.GemmError) as e:
        h.matmul(a, b, out_dtype="f32")
    assert e.value.code == 4  # GEMM_ERR_NO_MEMORY
    monkeypatch.delenv("GEMM_FAULT_INJECT")
    c = h.matmul(a, b, out_dtype="f32")
    assert h.status() == 0
    C64, D = oracle_rows(p)
    assert rel_err(c, C64, D) <= 1e-2
    h.close()


def test_split_k_after_a_timeout(g):
    # A split-K launch that gives up on its waits leaves flags behind; the epoch protocol
    # must keep the next launches from mistaking them for this launch's partials.
    p = W.integer_problem(1030, 530, 1200, "bf16", seed=7, b_layout="col")
    a, b = to_device(p.A), to_device(p.B)
    ref = p.A.to(torch.int64) @ p.B.to(torch.int64)
    h = g.Gemm(0)
    h.set_option("stream_k", 2)
    assert h.plan(a, b, out_dtype="f32")["split_tiles"] > 0
    c = h.matmul(a, b, out_dtype="f32")
    assert h.status() == 0 and torch.equal(c.cpu().to(torch.int64), ref)
    h.set_option("wait_timeout_us", 20000)
    h.set_option("fault_stall_producer", 1)
    h.matmul(a, b, out_dtype="f32")
    assert h.status() == 6
    h.set_option("fault_stall_producer", 0)
    for _ in range(3):
        c = h.matmul(a, b, out_dtype="f32")
        assert h.status() == 0
        assert torch.equal(c.cpu().to(torch.int64), ref)
    h.close()


@pytest.mark.parametrize("kind,who", [("pair", 0), ("pair", 1), ("single", 0), ("exact", 0),
                                      ("exact", 1), ("pair_split", 0), ("pair_split", 1)])
def test_loader_stops_with_copies_in_flight(g, kind, who):
    # The loader of one CTA (rank `who` of a pair) stops after 20 stage fills, so the other
    # CTA's loader keeps issuing until the ring is full and the MMA issuer's bounded wait
    # expires with copies of both CTAs still in flight. Before either CTA of a pair leaves,
    # the leader accounts for every outstanding fill (the bytes that never come, or the
    # missing arrival) and waits for the copies that were issued. Nothing faults or hangs:
    # the kernel reports GEMM_ERR_TIMEOUT and the same context then computes correctly.
    dtype = "f32" if kind == "exact" else "bf16"
    # (every cluster of the split product still takes more than 20 K-blocks)
    M, N, K = {"exact": (700, 600, 1500), "pair_split": (4096, 2048, 4096)}.get(kind, (1100, 900, 4096))
    p = W.integer_problem(M, N, K, dtype, seed=61 + who, b_layout="col")
    a, b = to_device(p.A), to_device(p.B)
    ref = p.A.to(torch.int64) @ p.B.to(torch.int64)
    h = g.Gemm(0)
    h.set_option("cta_pair", 1 if kind == "single" else 2)
    if kind == "pair_split":
        h.set_option("stream_k", 2)
        assert h.plan(a, b, out_dtype="f32")["split_tiles"] > 0
    plan = h.plan(a, b, out_dtype="f32", precision=p.precision)
    assert plan["k_iters"] > 20 and plan["cta_pair"] == (0 if kind == "single" else 1)
    h.set_option("wait_timeout_us", 20000)
    h.set_option("fault_stall_producer", 2 * 20 + who)
    for _ in range(2):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        h.matmul(a, b, out_dtype="f32", precision=p.precision)
        e1.record()
        assert h.status() == 6  # GEMM_ERR_TIMEOUT
        # One 20 ms limit expires; the teardown's waits for the copies in flight end at once
        # (each would take another 20 ms if the outstanding fills were miscounted).
        assert e0.elapsed_time(e1) < 80.0, e0.elapsed_time(e1)
    h.set_option("fault_stall_producer", 0)
    for _ in range(2):
        c = h.matmul(a, b, out_dtype="f32", precision=p.precision)
        assert h.status() == 0
        assert torch.equal(c.cpu().to(torch.int64), ref)
    h.close()
