"""GPU parity: the sm_103a GEMM through its C ABI against the fp64 oracle.

Acceptance: |D - ref| <= 2^-9 (|alpha| sum|ab| + |beta c|) + one output ulp, and bit
equality on integer-valued problems.  Every full-size workload is compared on every
output (the 8192^3 one in a test marked slow), and also on sampled outputs
(tile-boundary rows and columns plus seeded random entries); smaller problems that still
span several tiles with ragged tails are compared element by element.
"""
import numpy as np
import pytest
import torch

from layout_algebra_gb300 import binding as G
from layout_algebra_gb300 import layout as L
from layout_algebra_gb300 import workloads as W
from oracle import gemm_ref as O

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


@pytest.fixture(params=[1, 2, 4, 5, 6, 7], ids=["single", "pair", "narrow", "pair224", "pair512", "pair448"])
def variant(request):
    """Run a test with the single-CTA kernel and with the CTA-pair kernel."""
    G.set_kernel_variant(request.param)
    yield request.param
    G.set_kernel_variant(0)


def code(p):
    return O.dtype_code(p.dtype)


def run(p, data, D=None, stream=None):
    A = data["A"].to(DEV)
    B = data["B"].to(DEV)
    C = data["C"].to(DEV) if data["C"] is not None else None
    out = G.gemm(A, B, p.M, p.N, p.K, lda=data["lda"], ldb=data["ldb"], majorA=p.majorA,
                 majorB=p.majorB, alpha=p.alpha, beta=p.beta, C=C, D=D, stream=stream)
    st, detail = G.last_device_status(stream)
    assert st == 0, "device status %d detail %#x" % (st, detail)
    return out


def oracle(p, data, rows=None, cols=None):
    C = W.bits(data["C"]) if data["C"] is not None else None
    return O.gemm(p.M, p.N, p.K, p.alpha, W.bits(data["A"]), data["lda"],
                  0 if p.majorA == "K" else 1, W.bits(data["B"]), data["ldb"],
                  0 if p.majorB == "K" else 1, p.beta, C, p.N, code(p), rows, cols)


def check(p, data, D, rows=None, cols=None, exact=False):
    dh = O.decode(code(p), W.bits(D.cpu()))
    ref, sab = oracle(p, data, rows, cols)
    if rows is None:
        d = dh[: p.M * p.N].reshape(p.M, p.N)
        c = (O.decode(code(p), W.bits(data["C"])).reshape(p.M, p.N)
             if data["C"] is not None else None)
    else:
        d = dh[rows * p.N + cols]
        c = (O.decode(code(p), W.bits(data["C"]))[rows * p.N + cols]
             if data["C"] is not None else None)
    if exact:
        want = O.decode(code(p), O.round_to(code(p), ref))
        bad = np.argwhere(d != want)
        assert bad.size == 0, "first mismatch at %s: %r vs %r" % (
            bad[0], d[tuple(bad[0])], want[tuple(bad[0])])
        return 0.0
    bound = O.bound(code(p), p.alpha, p.beta, ref, sab, c)
    ratio = np.abs(d - ref) / bound
    worst = float(np.max(ratio)) if ratio.size else 0.0
    assert np.all(np.isfinite(d)), "non-finite output"
    assert worst <= 1.0, "worst element at %.3f of the error budget" % worst
    return worst


def sample_entries(M, N, seed, n_random=20000):
    rng = np.random.default_rng(seed)
    rows, cols = [], []
    for r in sorted({0, 127, 128, M // 2, M - 129 if M > 129 else 0, M - 1}):
        rows.append(np.full(N, r))
        cols.append(np.arange(N))
    for c in sorted({0, 255, 256, N // 2, N - 257 if N > 257 else 0, N - 1}):
        rows.append(np.arange(M))
        cols.append(np.full(M, c))
    rows.append(rng.integers(0, M, n_random))
    cols.append(rng.integers(0, N, n_random))
    return np.concatenate(rows).astype(np.int64), np.concatenate(cols).astype(np.int64)


# --------------------------------------------------------------------------- workloads


def test_integer_workload_bit_exact():
    p = W.WORKLOADS["gemm256_int_f16"]
    data = W.make(p)
    D = run(p, data)
    check(p, data, D, exact=True)


@pytest.mark.parametrize("name", [n for n in W.WORKLOAD_ORDER if n != "gemm256_int_f16"])
def test_full_size_workload_sampled(name):
    p = W.WORKLOADS[name]
    data = W.make(p)
    D = run(p, data)
    rows, cols = sample_entries(p.M, p.N, seed=p.seed)
    worst = check(p, data, D, rows, cols)
    print("%s: worst sampled element at %.3f of budget" % (name, worst))


def test_ragged_workload_full_compare():
    """The ragged-tail workload compared on every output (not only samples)."""
    p = W.WORKLOADS["gemm5000x3000x4104_ragged_f16"]
    data = W.make(p)
    D = run(p, data)
    check(p, data, D)


def full_compare(name):
    """Every output of a named workload against the oracle.  The oracle gets the same
    logical A and B stored K-major (the generator draws the logical matrices before it lays
    them out, so only the storage differs): its k loop then reads both operands
    contiguously, which keeps a full pass of these sizes to tens of seconds on the host."""
    p = W.WORKLOADS[name]
    data = W.make(p)
    D = run(p, data)
    pk = p.with_(majorA="K", majorB="K", lda=None, ldb=None)
    data_k = data if pk == p else W.make(pk)
    worst = check(pk, data_k, D)
    print("%s: worst element at %.3f of budget over all %d outputs" % (name, worst, p.M * p.N))


def test_full_compare_4096():
    full_compare("gemm4096_f16")


def test_full_compare_mnmajor():
    """16384 x 1024 x 4096 with M-major A and N-major B: every output."""
    full_compare("gemm16384x1024x4096_mnmajor_f16")


@pytest.mark.slow
def test_full_compare_8192_bf16_c():
    """8192^3 bf16 with C, every one of its 67M outputs (about 1.1e12 fp64 multiply-adds on
    the host: minutes)."""
    full_compare("gemm8192_bf16_c")


# --------------------------------------------------------------------------- shapes and majors


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("majors", [("K", "K"), ("MN", "MN"), ("K", "MN"), ("MN", "K")])
def test_multi_tile_ragged_all_majors(variant, dtype, majors):
    M, N, K = 300, 520, 200        # 3 x 3 tiles, tails of 44 rows / 8 columns, 4 k-blocks
    lda = K if majors[0] == "K" else 304
    p = W.Problem("mt", M, N, K, dtype, majorA=majors[0], majorB=majors[1], has_c=True,
                  alpha=1.25, beta=0.5, dist="normal", c_dist="normal", seed=31, lda=lda)
    data = W.make(p)
    check(p, data, run(p, data))


@pytest.mark.parametrize("var", [6, 7], ids=["pair512", "pair448"])
@pytest.mark.parametrize("has_c", [True, False], ids=["C", "noC"])
@pytest.mark.parametrize("majors", [("K", "K"), ("MN", "MN")])
def test_wide_forms_several_tiles_per_pair(var, has_c, majors):
    # 20 x 4 = 80 tiles on 76 pairs: four pairs run a second tile, whose copies reuse the
    # ring stages that the first tile's epilogue borrowed as staging; ragged last row and
    # column of tiles (36 rows, 40 columns short), 5 k-blocks
    tile_n = 512 if var == 6 else 448
    M, N, K = 20 * 256 - 36, 4 * tile_n - 40, 320
    lda = K if majors[0] == "K" else M + 4
    ldb = K if majors[1] == "K" else N
    p = W.Problem("wide", M, N, K, "bf16", majorA=majors[0], majorB=majors[1], has_c=has_c,
                  alpha=1.25, beta=0.5 if has_c else 0.0, dist="normal", c_dist="normal",
                  seed=91 + var, lda=lda, ldb=ldb)
    data = W.make(p)
    G.set_kernel_variant(var)
    try:
        D = run(p, data)
    finally:
        G.set_kernel_variant(0)
    check(p, data, D)


@pytest.mark.parametrize("majors", [("K", "K"), ("MN", "MN"), ("MN", "K"), ("K", "MN")])
def test_integer_ragged_exact(variant, majors):
    M, N, K = 129, 77, 40
    lda = K if majors[0] == "K" else 136
    ldb = K if majors[1] == "K" else 80
    p = W.Problem("int", M, N, K, "f16", majorA=majors[0], majorB=majors[1], has_c=True,
                  alpha=1.0, beta=1.0, dist="int2", c_dist="int2", seed=41, lda=lda, ldb=ldb)
    data = W.make(p)
    check(p, data, run(p, data), exact=True)


@pytest.mark.parametrize("shape", [(1, 8, 8), (1, 1, 1), (7, 3, 5), (128, 256, 64),
                                   (129, 257, 65), (256, 512, 1000), (8, 2000, 16)])
def test_small_and_boundary_shapes(variant, shape):
    M, N, K = shape
    lda = -(-K // 8) * 8
    ldb = -(-K // 8) * 8
    p = W.Problem("s", M, N, K, "f16", has_c=True, alpha=0.75, beta=-1.0, dist="uniform",
                  c_dist="uniform", seed=M * 7 + N * 3 + K, lda=lda, ldb=ldb)
    data = W.make(p)
    check(p, data, run(p, data))


def test_long_k():
    p = W.Problem("longk", 256, 256, 16384, "bf16", dist="uniform", seed=51)
    data = W.make(p)
    check(p, data, run(p, data))


def test_output_past_2_31_elements():
    """D of 2^31 elements (4 GiB): element offsets past the int32 range in the epilogue and a
    tile grid of 8192 x 4 tiles; sampled outputs (first, middle and last rows, random
    entries) against the oracle."""
    M, N, K = 1 << 21, 1024, 64
    p = W.Problem("big", M, N, K, "f16", dist="uniform", seed=61)
    data = W.make(p)
    D = torch.empty(M * N, dtype=torch.float16, device=DEV)
    G.gemm(data["A"].to(DEV), data["B"].to(DEV), M, N, K, lda=K, ldb=K, D=D)
    st, detail = G.last_device_status()
    assert st == 0, "device status %d detail %#x" % (st, detail)
    rng = np.random.default_rng(7)
    rows = np.concatenate([np.repeat([0, M // 2, M - 256, M - 1], N), rng.integers(0, M, 20000)])
    cols = np.concatenate([np.tile(np.arange(N), 4), rng.integers(0, N, 20000)])
    idx = torch.from_numpy(rows * N + cols).to(DEV)
    d = O.decode(O.F16, W.bits(D[idx].cpu()))
    ref, sab = O.gemm(M, N, K, 1.0, W.bits(data["A"]), K, 0, W.bits(data["B"]), K, 0, 0.0, None, N, O.F16,
                      rows, cols)
    bound = O.bound(O.F16, 1.0, 0.0, ref, sab, None)
    assert np.all(np.abs(d - ref) <= bound)
    del D
    torch.cuda.empty_cache()


def test_k_zero_gives_beta_c(variant):
    p = W.Problem("k0", 200, 264, 0, "f16", has_c=True, alpha=2.0, beta=0.5,
                  c_dist="uniform", seed=61)
    data = W.make(p)
    C = data["C"].to(DEV)
    D = G.gemm(torch.empty(8, dtype=torch.float16, device=DEV),
               torch.empty(8, dtype=torch.float16, device=DEV), p.M, p.N, 0, lda=8, ldb=8,
               alpha=p.alpha, beta=p.beta, C=C)
    assert G.last_device_status()[0] == 0
    check(p, data, D, exact=True)          # 0.5 * c is exact


def test_alpha_zero_and_beta_zero(variant):
    p = W.Problem("a0", 130, 260, 70, "bf16", has_c=True, alpha=0.0, beta=1.5,
                  dist="normal", c_dist="normal", seed=62, lda=72, ldb=72)
    data = W.make(p)
    check(p, data, run(p, data))
    q = W.Problem("b0", 130, 260, 72, "bf16", has_c=False, alpha=1.0, beta=0.0,
                  dist="normal", seed=63)
    dq = W.make(q)
    check(q, dq, run(q, dq))


def test_empty_problem_writes_nothing():
    D = torch.full((64,), 7.0, dtype=torch.float16, device=DEV)
    A = torch.zeros(64, dtype=torch.float16, device=DEV)
    for M, N in ((0, 8), (8, 0)):
        st = G.raw_call(torch.float16, M, N, 8, 1.0, A.data_ptr(), 8, 0, A.data_ptr(), 8, 0,
                        0.0, None, D.data_ptr(), torch.cuda.current_stream().cuda_stream)
        assert st == 0
    torch.cuda.synchronize()
    assert torch.all(D == 7.0)


def test_canary_outside_d_untouched(variant):
    p = W.Problem("can", 200, 300, 64, "f16", dist="uniform", seed=64)
    data = W.make(p)
    D = torch.full((p.M * p.N + 4096,), -3.0, dtype=torch.float16, device=DEV)
    run(p, data, D=D)
    assert torch.all(D[p.M * p.N:] == -3.0)
    check(p, data, D[: p.M * p.N])


def test_non_default_stream_and_repeat():
    p = W.Problem("st", 512, 768, 512, "bf16", has_c=True, alpha=1.0, beta=1.0,
                  dist="normal", seed=65)
    data = W.make(p)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        D1 = run(p, data, stream=s)
        D2 = run(p, data, stream=s)
    s.synchronize()
    assert torch.equal(D1, D2)             # same inputs, same kernel: same bits
    check(p, data, D1)


def test_host_buffers_end_to_end():
    p = W.Problem("e2e", 384, 512, 256, "f16", has_c=True, alpha=0.5, beta=2.0,
                  dist="uniform", seed=66)
    data = W.make(p)
    D = G.gemm(data["A"].pin_memory(), data["B"].pin_memory(), p.M, p.N, p.K,
               lda=data["lda"], ldb=data["ldb"], alpha=p.alpha, beta=p.beta,
               C=data["C"].pin_memory())
    torch.cuda.synchronize()
    assert not D.is_cuda
    check(p, data, D)


@pytest.mark.parametrize("dtype,M,majorA,pinned", [("bf16", 4096, "K", True), ("f16", 5000, "K", True),
                                                  ("f16", 2304, "MN", True), ("bf16", 4352, "MN", False),
                                                  ("f16", 3000, "K", False)])
def test_host_buffers_row_blocks_match_device_call(dtype, M, majorA, pinned):
    """Host operands through gb_gemm_*_host (A, C up and D down in row blocks overlapped with
    the GEMM, inside the library); pinned and pageable buffers, both majors of A.  The result
    equals one device call over all rows, bit for bit."""
    N, K = 520, 200
    lda = K if majorA == "K" else M + 8
    p = W.Problem("e2eb", M, N, K, dtype, majorA=majorA, has_c=True, alpha=1.25, beta=0.5,
                  dist="normal", c_dist="normal", seed=M + 3, lda=lda)
    data = W.make(p)
    assert len(G.row_blocks(M)) == min(8, M // 1024)
    host = (lambda t: t.pin_memory()) if pinned else (lambda t: t.clone())
    D_h = torch.full((M * N,), float("nan"), dtype=W.torch_dtype(dtype))
    if pinned:
        D_h = D_h.pin_memory()
    Dh = G.gemm(host(data["A"]), host(data["B"]), M, N, K, lda=lda, ldb=data["ldb"], majorA=majorA,
                alpha=p.alpha, beta=p.beta, C=host(data["C"]), D=D_h)
    torch.cuda.synchronize()
    Dd = run(p, data)
    assert Dh is D_h and not Dh.is_cuda
    assert torch.equal(Dh.view(torch.int16), Dd.cpu().view(torch.int16))
    check(p, data, Dh, *sample_entries(M, N, seed=5, n_random=4000))


def test_host_call_ordering_on_two_streams():
    """Host-operand calls share the library's staging buffer: calls issued back to back on
    two streams, each with its own operands, still each get their own result."""
    outs = []
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    probs = [W.Problem("hs%d" % i, 2048 + 256 * i, 264, 136, "f16", has_c=True, alpha=1.0, beta=1.0,
                       dist="int2", c_dist="int2", seed=90 + i) for i in range(4)]
    datas = [W.make(p) for p in probs]
    for i, (p, d) in enumerate(zip(probs, datas)):
        outs.append(G.gemm(d["A"].pin_memory(), d["B"].pin_memory(), p.M, p.N, p.K, lda=d["lda"],
                           ldb=d["ldb"], alpha=p.alpha, beta=p.beta, C=d["C"].pin_memory(),
                           stream=streams[i % 2]))
    torch.cuda.synchronize()
    for p, d, D in zip(probs, datas, outs):
        check(p, d, D, exact=True)


def test_host_entry_rejects_device_pointers():
    p = W.Problem("hd", 64, 64, 64, "f16", dist="int2", seed=3)
    data = W.make(p)
    A, B = data["A"].to(DEV), data["B"].to(DEV)
    D = torch.empty(64 * 64, dtype=torch.float16)
    st = G.lib().gb_gemm_f16_host(64, 64, 64, 1.0, A.data_ptr(), 64, 0, B.data_ptr(), 64, 0, 0.0,
                                  None, D.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 1


def test_device_misalignment_rejected():
    buf = torch.zeros(4096, dtype=torch.float16, device=DEV)
    s = torch.cuda.current_stream().cuda_stream
    st = G.raw_call(torch.float16, 64, 64, 64, 1.0, buf.data_ptr() + 2, 64, 0, buf.data_ptr(),
                    64, 0, 0.0, None, buf.data_ptr(), s)
    assert st == 2


# --------------------------------------------------------------------------- failure path


def test_wait_timeout_is_reported_and_context_survives(variant):
    p = W.Problem("to", 256, 256, 512, "f16", dist="int2", seed=71)
    data = W.make(p)
    G.set_wait_timeout_ns(50_000_000)
    G.debug_skip_k_block(3)        # the copy stage never issues k-block 3: its wait runs out
    try:
        A, B = data["A"].to(DEV), data["B"].to(DEV)
        G.gemm(A, B, p.M, p.N, p.K, lda=data["lda"], ldb=data["ldb"])
        st, detail = G.last_device_status()
    finally:
        G.debug_skip_k_block(-1)
        G.set_wait_timeout_ns(0)
    assert st == 5
    # the first wait to run out: the MMA on the missing k-block (2), the epilogue behind it
    # (4), a copy stage waiting for a slot (1) or for the last releases before exit (6)
    assert detail & 0xff in (1, 2, 4, 6)
    assert G.last_device_status() == (0, 0)   # record cleared
    check(p, data, run(p, data), exact=True)  # the context still works


# --------------------------------------------------------------------------- device-side maps


@pytest.mark.parametrize("var", [1, 2, 4, 5, 6, 7])
@pytest.mark.parametrize("M,N,tile", [(5000, 3000, (19, 11)), (5000, 3000, (0, 0)),
                                      (256, 128, (0, 0)), (8192, 8192, (17, 30))])
def test_epilogue_map_matches_host_layout(var, M, N, tile):
    """The device evaluation of the C/D tile map equals the host layout library's."""
    G.set_kernel_variant(var)
    try:
        plan = G.plan("f16", M, N, 64, 64, "K", 64, "K")
    finally:
        G.set_kernel_variant(0)
    tm, tn = int(plan["tile_m"]), int(plan["tile_n"])
    # the last tile along a mode when the index is beyond this variant's grid
    tile = (min(tile[0], (M + tm - 1) // tm - 1), min(tile[1], (N + tn - 1) // tn - 1))
    out = torch.empty(tm * tn, dtype=torch.int64, device=DEV)
    st = __import__("layout_algebra_gb300._native", fromlist=["lib"]).lib().gb_debug_epilogue_map(
        var, M, N, tile[0], tile[1], out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 0
    got = out.cpu().numpy().reshape(tm, tn)
    origin, tl = L.local_tile("(%d,%d):(%d,1)" % (M, N, N), "(%d,%d)" % (tm, tn), list(tile))
    rr, cc = np.meshgrid(np.arange(tm), np.arange(tn), indexing="ij")
    idx = (rr + tm * cc).ravel()                     # colexicographic index of (r, c)
    want = (origin + L.evaluate(tl, idx)).reshape(tm, tn)
    inside = ((tile[0] * tm + rr) < M) & ((tile[1] * tn + cc) < N)
    want = np.where(inside, want, -1)
    assert np.array_equal(got, want)
    assert np.array_equal(got[inside], ((tile[0] * tm + rr) * N + tile[1] * tn + cc)[inside])


def _swizzle_offset(row, byte_in_row):
    """128-byte swizzle: the 16-byte chunk index is XORed with the row index mod 8."""
    chunk = (byte_in_row // 16) ^ (row % 8)
    return row * 128 + chunk * 16 + byte_in_row % 16


@pytest.mark.parametrize("which,major,tile,kb", [(0, "K", 1, 2), (0, "MN", 1, 1), (1, "K", 0, 3),
                                                 (1, "MN", 1, 0), (0, "K", 2, 3)])
def test_stage_bytes_match_swizzle_model(which, major, tile, kb):
    M, N, K = 300, 520, 200
    lda = K if (which == 1 or major == "K") else 304
    ldb = K if (which == 0 or major == "K") else N
    majorA = major if which == 0 else "K"
    majorB = major if which == 1 else "K"
    p = W.Problem("tma", M, N, K, "f16", majorA=majorA, majorB=majorB, dist="normal", seed=81,
                  lda=lda, ldb=ldb)
    data = W.make(p, logical=True)
    A, B = data["A"].to(DEV), data["B"].to(DEV)
    nbytes = 128 * 64 * 2 if which == 0 else 256 * 64 * 2
    out = torch.zeros(nbytes // 2, dtype=torch.int16, device=DEV)
    lib = __import__("layout_algebra_gb300._native", fromlist=["lib"]).lib()
    st = lib.gb_debug_stage_bytes(0, which, M, N, K, A.data_ptr(), lda, G.major_code(majorA),
                                  B.data_ptr(), ldb, G.major_code(majorB), tile, kb,
                                  out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 0
    assert G.last_device_status()[0] == 0
    got = out.cpu().numpy().view(np.uint16)
    # logical operand as (rows, K): A is M x K; B^T is N x K
    mat = W.bits(data["a"]).reshape(M, K) if which == 0 else W.bits(data["b"].t().contiguous()).reshape(N, K)
    rows_total = M if which == 0 else N
    rows_tile = 128 if which == 0 else 256
    want = np.zeros(nbytes // 2, dtype=np.uint16)
    for r in range(rows_tile):
        for k in range(64):
            gr, gk = tile * rows_tile + r, kb * 64 + k
            v = mat[gr, gk] if (gr < rows_total and gk < K) else 0
            if major == "K":
                off = _swizzle_offset(r, 2 * k)
            else:
                box, inner = divmod(r, 64)
                off = box * 8192 + _swizzle_offset(k, 2 * inner)
            want[off // 2] = v
    assert np.array_equal(got, want)
