"""GPU parity of the stream-K schedule (the *_ws calls) against the fp64 oracle.

Stream-K splits the K loop of some tiles across CTAs and adds fp32 partials through a
workspace, so the summation order differs from the plain call while the acceptance rule
is the same; integer-valued problems stay bit-exact.
"""
import numpy as np
import pytest
import torch

from layout_algebra_gb300 import binding as G
from layout_algebra_gb300 import workloads as W
from tests.test_gemm_gpu import DEV, check, sample_entries

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def workspace():
    return G.make_workspace(DEV)


@pytest.fixture(params=[1, 2, 4, 5, 6, 7], ids=["single", "pair", "narrow", "pair224", "pair512", "pair448"])
def variant(request):
    G.set_kernel_variant(request.param)
    yield request.param
    G.set_kernel_variant(0)


@pytest.fixture(params=[0, 2], ids=["auto", "forced"])
def schedule(request):
    G.set_schedule(request.param)
    yield request.param
    G.set_schedule(0)


def run_ws(p, data, ws, D=None):
    A, B = data["A"].to(DEV), data["B"].to(DEV)
    C = data["C"].to(DEV) if data["C"] is not None else None
    out = G.gemm(A, B, p.M, p.N, p.K, lda=data["lda"], ldb=data["ldb"], majorA=p.majorA,
                 majorB=p.majorB, alpha=p.alpha, beta=p.beta, C=C, D=D, workspace=ws)
    st, detail = G.last_device_status()
    assert st == 0, "device status %d detail %#x" % (st, detail)
    return out


@pytest.mark.parametrize("shape", [(256, 512, 4096), (300, 520, 1000), (128, 256, 2048), (4096, 16, 4096),
                                   (1000, 1000, 777), (64, 64, 64)])
def test_split_tiles_match_oracle(variant, schedule, workspace, shape):
    """Few tiles and forced splitting: many CTAs add partials into one tile."""
    M, N, K = shape
    ld = -(-K // 8) * 8
    p = W.Problem("sk", M, N, K, "bf16", has_c=True, alpha=1.25, beta=0.5, dist="normal",
                  c_dist="normal", seed=M + N + K, lda=ld, ldb=ld)
    data = W.make(p)
    check(p, data, run_ws(p, data, workspace))


@pytest.mark.parametrize("majors", [("K", "K"), ("MN", "MN"), ("MN", "K"), ("K", "MN")])
def test_integer_split_is_exact(variant, workspace, majors):
    G.set_schedule(2)
    try:
        M, N, K = 384, 768, 2048
        p = W.Problem("ski", M, N, K, "f16", majorA=majors[0], majorB=majors[1], has_c=True,
                      alpha=1.0, beta=1.0, dist="int2", c_dist="int2", seed=7)
        data = W.make(p)
        check(p, data, run_ws(p, data, workspace), exact=True)
    finally:
        G.set_schedule(0)


def test_workspace_reuse_across_calls(workspace):
    """Back-to-back calls on one workspace (each launch tags its hand-offs anew)."""
    G.set_schedule(2)
    try:
        p = W.Problem("reuse", 512, 1024, 3000, "f16", dist="int2", seed=9, lda=3000, ldb=3000)
        data = W.make(p)
        outs = [run_ws(p, data, workspace) for _ in range(3)]
        q = W.Problem("reuse2", 256, 256, 512, "f16", dist="int2", seed=10)
        dq = W.make(q)
        check(q, dq, run_ws(q, dq, workspace), exact=True)
        outs.append(run_ws(p, data, workspace))
        for o in outs:
            check(p, data, o, exact=True)
    finally:
        G.set_schedule(0)


@pytest.mark.parametrize("name", ["gemm4096_f16", "gemm5000x3000x4104_ragged_f16",
                                  "gemm16384x1024x4096_mnmajor_f16"])
def test_workloads_with_workspace(workspace, name):
    p = W.WORKLOADS[name]
    data = W.make(p)
    D = run_ws(p, data, workspace)
    rows, cols = sample_entries(p.M, p.N, seed=p.seed + 100)
    check(p, data, D, rows, cols)


def test_workspace_errors(workspace):
    A = torch.zeros(64 * 64, dtype=torch.float16, device=DEV)
    s = torch.cuda.current_stream().cuda_stream
    lib = G.lib()
    nbytes = workspace.numel()
    base = workspace.data_ptr()
    # misaligned workspace
    assert lib.gb_gemm_f16_ws(64, 64, 64, 1.0, A.data_ptr(), 64, 0, A.data_ptr(), 64, 0, 0.0,
                              None, A.data_ptr(), base + 16, nbytes - 16, s) == 2
    # too small
    assert lib.gb_gemm_f16_ws(64, 64, 64, 1.0, A.data_ptr(), 64, 0, A.data_ptr(), 64, 0, 0.0,
                              None, A.data_ptr(), base, 1024, s) == 1
    # missing
    assert lib.gb_gemm_f16_ws(64, 64, 64, 1.0, A.data_ptr(), 64, 0, A.data_ptr(), 64, 0, 0.0,
                              None, A.data_ptr(), None, nbytes, s) == 1


def test_split_timeout_path_reports_and_recovers(workspace):
    """A k-block that is never copied makes the waits run out; the status is reported."""
    G.set_schedule(2)
    G.set_wait_timeout_ns(50_000_000)
    G.debug_skip_k_block(1)
    try:
        p = W.Problem("skto", 256, 512, 16384, "f16", dist="int2", seed=11)
        data = W.make(p)
        A, B = data["A"].to(DEV), data["B"].to(DEV)
        G.gemm(A, B, p.M, p.N, p.K, lda=data["lda"], ldb=data["ldb"], workspace=workspace)
        st, detail = G.last_device_status()
    finally:
        G.debug_skip_k_block(-1)
        G.set_wait_timeout_ns(0)
    assert st == 5 and (detail & 0xff) in (1, 2, 4, 7)
    try:
        check(p, data, run_ws(p, data, workspace), exact=True)
    finally:
        G.set_schedule(0)


def test_stream_k_graph_replay(workspace):
    """A captured stream-K GEMM replays correctly: owners clear the partial-ready flags they
    consumed, so a replay (same launch number) waits for fresh partials."""
    G.set_schedule(2)
    try:
        p = W.Problem("skg", 512, 768, 4096, "f16", dist="int2", seed=12)
        data = W.make(p)
        A, B = data["A"].to(DEV), data["B"].to(DEV)
        D = torch.empty(p.M * p.N, dtype=torch.float16, device=DEV)

        def call():
            G.gemm(A, B, p.M, p.N, p.K, lda=data["lda"], ldb=data["ldb"], D=D, workspace=workspace)

        call()                                   # first use: attributes, occupancy, plan
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            call()
        gen = torch.Generator().manual_seed(13)
        for trial in range(4):
            a = torch.randint(-2, 3, (p.M, p.K), generator=gen).to(torch.float16)
            A.copy_(a.reshape(-1).to(DEV))
            graph.replay()
            torch.cuda.synchronize()
            assert G.last_device_status() == (0, 0)
            q = dict(data, A=a.reshape(-1))
            check(p, q, D.cpu(), exact=True)
    finally:
        G.set_schedule(0)
