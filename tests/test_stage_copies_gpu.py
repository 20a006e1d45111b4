"""GPU parity of the stage-deep copies of the CTA-pair kernel.

When K is a multiple of the k-block, the pair kernel copies both k-blocks of a stage with
one tensor copy per operand: a K-major operand with a three-dimensional copy (k-block elements, rows,
k-blocks), an MN-major one (rows a multiple of 64) with one four-dimensional copy; a last
stage holding a single k-block still receives a whole box, its second k-block zero-filled
past K.  These cases pin that path against the fp64 oracle: odd and even k-block counts,
padded leading dimensions, mixed majors, rows that do and do not allow the MN-major stage
copy, 16-bit and FP8 inputs.
"""
import numpy as np
import pytest
import torch

from layout_algebra_gb300 import binding as G
from layout_algebra_gb300 import workloads as W
from oracle import gemm_ref as O

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


@pytest.fixture(params=[2, 5, 6, 7], ids=["pair", "pair224", "pair512", "pair448"])
def pair(request):
    G.set_kernel_variant(request.param)
    yield
    G.set_kernel_variant(0)


def run16(p, data):
    C = data["C"].to(DEV) if data["C"] is not None else None
    D = G.gemm(data["A"].to(DEV), data["B"].to(DEV), p.M, p.N, p.K, lda=data["lda"],
               ldb=data["ldb"], majorA=p.majorA, majorB=p.majorB, alpha=p.alpha, beta=p.beta, C=C)
    st, detail = G.last_device_status()
    assert st == 0, "device status %d detail %#x" % (st, detail)
    return D


def ref16(p, data):
    C = W.bits(data["C"]) if data["C"] is not None else None
    return O.gemm(p.M, p.N, p.K, p.alpha, W.bits(data["A"]), data["lda"],
                  0 if p.majorA == "K" else 1, W.bits(data["B"]), data["ldb"],
                  0 if p.majorB == "K" else 1, p.beta, C, p.N, O.dtype_code(p.dtype))


# K multiples of the k-block (64) with even and odd k-block counts, and K tails (100, 200,
# 1000: the stage reaching past K / 64 whole k-blocks goes through the two-dimensional maps)
@pytest.mark.parametrize("K", [64, 100, 192, 200, 320, 1000, 1024])
@pytest.mark.parametrize("majors", [("K", "K"), ("K", "MN"), ("MN", "K"), ("MN", "MN")])
@pytest.mark.parametrize("MN", [(300, 520), (320, 576)], ids=["rows_ragged", "rows_x64"])
def test_integer_exact_k_blocks(pair, K, majors, MN):
    # (300, 520): MN-major operands fall back to per-k-block copies (rows not a multiple of
    # 64); (320, 576): they take the four-dimensional stage copies, with whole 64-row chunks
    # past M and N zero-filled in the last tiles
    M, N = MN
    # leading dimensions: multiples of 8 elements, padded past K / M
    lda = -(-K // 8) * 8 + 16 if majors[0] == "K" else -(-M // 8) * 8 + 8
    ldb = -(-K // 8) * 8 + 8 if majors[1] == "K" else N
    p = W.Problem("sd", M, N, K, "f16", majorA=majors[0], majorB=majors[1], has_c=True,
                  alpha=1.0, beta=1.0, dist="int2", c_dist="int2", seed=K + 7, lda=lda, ldb=ldb)
    data = W.make(p)
    d = O.decode(O.F16, W.bits(run16(p, data).cpu())).reshape(M, N)
    ref, _ = ref16(p, data)
    want = O.decode(O.F16, O.round_to(O.F16, ref)).reshape(M, N)
    bad = np.argwhere(d != want)
    assert bad.size == 0, "first mismatch at %s" % (bad[0],)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_random_odd_k_blocks_default_variant(dtype):
    p = W.Problem("sdr", 512, 768, 448, dtype, has_c=True, alpha=1.25, beta=0.5, dist="normal",
                  c_dist="normal", seed=97)
    data = W.make(p)
    d = O.decode(O.dtype_code(dtype), W.bits(run16(p, data).cpu())).reshape(p.M, p.N)
    ref, sab = ref16(p, data)
    c = O.decode(O.dtype_code(dtype), W.bits(data["C"])).reshape(p.M, p.N)
    bound = O.bound(O.dtype_code(dtype), p.alpha, p.beta, ref, sab, c)
    assert np.all(np.abs(d - ref) <= bound)


@pytest.mark.parametrize("K", [128, 200, 384, 640, 1000])
def test_fp8_integer_exact_k_blocks(pair, K):
    ld = -(-K // 16) * 16   # FP8 rows: multiples of 16 bytes
    p = W.Problem("sd8", 320, 272, K, "f16", dist="int2", seed=K, a_fmt="e4m3", b_fmt="e5m2", lda=ld, ldb=ld)
    data = W.make(p)
    D = G.gemm_fp8(data["A"].to(DEV), data["B"].to(DEV), p.M, p.N, p.K, lda=data["lda"],
                   ldb=data["ldb"], a_format=p.a_fmt, b_format=p.b_fmt, out_dtype=torch.float16)
    st, detail = G.last_device_status()
    assert st == 0, "device status %d detail %#x" % (st, detail)
    ref, _ = O.gemm(p.M, p.N, p.K, 1.0, W.bits(data["A"]), data["lda"], O.K_MAJOR,
                    W.bits(data["B"]), data["ldb"], O.K_MAJOR, 0.0, None, p.N, O.F16,
                    a_dtype=O.dtype_code(p.a_fmt), b_dtype=O.dtype_code(p.b_fmt))
    d = O.decode(O.F16, W.bits(D.cpu())).reshape(p.M, p.N)
    want = O.decode(O.F16, O.round_to(O.F16, ref)).reshape(p.M, p.N)
    assert np.array_equal(d, want)
