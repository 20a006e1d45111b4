"""GPU parity of the FP8-input GEMM (gb_gemm_fp8) against the fp64 oracle.

FP8 operands (E4M3 / E5M2, K-major) with 16-bit C and D.  Every product of two FP8 values
is exact in fp32, so the error sources are the fp32 accumulation order and the final
rounding, as for 16-bit inputs: the same bound |d - r| <= 2^-9 (|alpha| S + |beta c|) +
one output ulp applies, and integer-valued problems must match exactly.
"""
import numpy as np
import pytest
import torch

from layout_algebra_gb300 import binding as G
from layout_algebra_gb300 import workloads as W
from oracle import gemm_ref as O

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
FP8 = {"e4m3": (O.E4M3, 448.0), "e5m2": (O.E5M2, 57344.0)}


@pytest.fixture(params=[1, 2, 4, 5, 6, 7], ids=["single", "pair", "narrow", "pair224", "pair512", "pair448"])
def variant(request):
    G.set_kernel_variant(request.param)
    yield request.param
    G.set_kernel_variant(0)


def run(p, data, workspace=None, **kw):
    A, B = data["A"].to(DEV), data["B"].to(DEV)
    C = data["C"].to(DEV) if data["C"] is not None else None
    D = G.gemm_fp8(A, B, p.M, p.N, p.K, lda=data["lda"], ldb=data["ldb"], a_format=p.a_fmt,
                   b_format=p.b_fmt, out_dtype=W.torch_dtype(p.dtype), alpha=p.alpha,
                   beta=p.beta, C=C, workspace=workspace, **kw)
    st, detail = G.last_device_status()
    assert st == 0, "device status %d detail %#x" % (st, detail)
    return D


def reference(p, data, rows=None, cols=None):
    code = O.dtype_code(p.dtype)
    C = W.bits(data["C"]) if data["C"] is not None else None
    return O.gemm(p.M, p.N, p.K, p.alpha, W.bits(data["A"]), data["lda"], O.K_MAJOR,
                  W.bits(data["B"]), data["ldb"], O.K_MAJOR, p.beta, C, p.N, code,
                  rows=rows, cols=cols, a_dtype=O.dtype_code(p.a_fmt),
                  b_dtype=O.dtype_code(p.b_fmt))


def check(p, data, D, rows=None, cols=None):
    code = O.dtype_code(p.dtype)
    ref, sab = reference(p, data, rows, cols)
    d = O.decode(code, W.bits(D.cpu()))
    c = None
    if data["C"] is not None:
        c = O.decode(code, W.bits(data["C"]))
    if rows is None:
        d = d.reshape(p.M, p.N)
        c = None if c is None else c.reshape(p.M, p.N)
    else:
        d = d.reshape(p.M, p.N)[rows, cols]
        c = None if c is None else c.reshape(p.M, p.N)[rows, cols]
    err = np.abs(d - ref)
    bnd = O.bound(code, p.alpha, p.beta, ref, sab, c)
    assert np.all(np.isfinite(d))
    assert np.all(err <= bnd), "worst %.3g of bound" % float(np.max(err / bnd))


@pytest.mark.parametrize("fa,fb", [("e4m3", "e4m3"), ("e5m2", "e5m2"), ("e4m3", "e5m2"),
                                   ("e5m2", "e4m3")])
def test_integer_exact(variant, fa, fb):
    # |sum| <= 4 K = 1024: exact in fp16
    p = W.Problem("i8", 320, 272, 256, "f16", dist="int2", seed=101, a_fmt=fa, b_fmt=fb)
    data = W.make(p)
    D = run(p, data)
    ref, _ = reference(p, data)
    d = O.decode(O.F16, W.bits(D.cpu())).reshape(p.M, p.N)
    assert np.array_equal(d, ref)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("fa,fb", [("e4m3", "e4m3"), ("e4m3", "e5m2"), ("e5m2", "e4m3")])
def test_random_ragged(variant, dtype, fa, fb):
    # M, N off the tile grid; K = 200 is one 128-wide k-block and a 72-wide zero-filled tail
    p = W.Problem("r8", 300, 520, 200, dtype, has_c=True, alpha=0.75, beta=0.5,
                  dist="normal", c_dist="normal", seed=102, a_fmt=fa, b_fmt=fb, lda=208,
                  ldb=224)
    data = W.make(p)
    check(p, data, run(p, data))


@pytest.mark.parametrize("K", [1, 16, 100, 128, 129, 1000])
def test_k_edges(variant, K):
    ld = ((K + 15) // 16) * 16
    p = W.Problem("k8", 257, 264, K, "bf16", dist="uniform", seed=103, a_fmt="e4m3",
                  b_fmt="e4m3", lda=ld, ldb=ld)
    data = W.make(p)
    check(p, data, run(p, data))


def test_k_zero_is_beta_c():
    p = W.Problem("k0", 130, 136, 0, "bf16", has_c=True, alpha=2.0, beta=-1.5, seed=104,
                  a_fmt="e4m3", b_fmt="e4m3", lda=16, ldb=16)
    data = W.make(p)
    check(p, data, run(p, data))


def test_scales_folded_into_alpha():
    # dequantised operands sA*A and sB*B: the caller passes alpha*sA*sB
    sA, sB = 0.03125, 3.0
    p = W.Problem("s8", 256, 512, 384, "bf16", has_c=True, alpha=1.5 * sA * sB, beta=1.0,
                  dist="normal", sigma=20.0, c_dist="normal", seed=105, a_fmt="e4m3",
                  b_fmt="e5m2")
    data = W.make(p)
    check(p, data, run(p, data))


def test_stream_k_fp8():
    ws = G.make_workspace(DEV)
    G.set_schedule(2)
    try:
        p = W.Problem("sk8", 512, 768, 4096, "bf16", has_c=True, alpha=0.5, beta=1.0,
                      dist="normal", c_dist="normal", seed=106, a_fmt="e4m3", b_fmt="e4m3")
        data = W.make(p)
        check(p, data, run(p, data, workspace=ws))
    finally:
        G.set_schedule(0)


def test_fp8_in_fp8_out_fused(variant):
    p = W.Problem("ff8", 384, 1040, 512, "bf16", has_c=True, alpha=0.25, beta=0.25,
                  dist="normal", c_dist="normal", seed=107, a_fmt="e4m3", b_fmt="e4m3")
    data = W.make(p)
    g = torch.Generator().manual_seed(8)
    bias = torch.randn(p.N, generator=g).to(torch.bfloat16)
    amax = torch.zeros(1, dtype=torch.float32, device=DEV)
    D = run(p, data, bias=bias.to(DEV), activation="gelu", amax=amax, out_format="e4m3",
            out_scale=8.0)
    ref, sab = reference(p, data)
    c = O.decode(O.BF16, W.bits(data["C"])).reshape(p.M, p.N)
    v = O.fused(ref, O.decode(O.BF16, W.bits(bias))[None, :], "gelu")
    err = O.LIPSCHITZ["gelu"] * 2.0 ** -9 * (abs(p.alpha) * sab + np.abs(p.beta * c))
    d = O.decode(O.E4M3, W.bits(D.cpu())).reshape(p.M, p.N)
    target = np.clip(v * 8.0, -448.0, 448.0)
    assert np.all(np.abs(d - target) <= err * 8.0 + O.ulp_fp8(O.E4M3, target))
    assert abs(float(amax.item()) - np.max(np.abs(v))) <= np.max(err) + 1e-6 * np.max(np.abs(v))


def test_full_size_sampled():
    # the throughput problem at its full size, in the launch configuration the bench times
    p = W.FP8_WORKLOADS["gemm8192_e4m3_bf16_c"]
    data = W.make(p)
    D = run(p, data)
    rng = np.random.default_rng(109)
    rows = np.concatenate([rng.integers(0, p.M, 1500), [0, p.M - 1, 255, 256]])
    cols = np.concatenate([rng.integers(0, p.N, 1500), [p.N - 1, 0, 256, 255]])
    check(p, data, D, rows, cols)


def test_argument_errors():
    A = torch.zeros(64 * 64, dtype=torch.uint8, device=DEV)
    with pytest.raises(G.GemmError) as e:      # lda not a multiple of 16 bytes
        G.gemm_fp8(A, A, 64, 64, 40, lda=40, ldb=48, a_format="e4m3", b_format="e4m3")
    assert e.value.status == 2
    for fa, fb, od in ((2, 0, 0), (0, -1, 0), (0, 0, 5)):
        st = G.lib().gb_gemm_fp8(fa, fb, od, 64, 64, 64, 1.0, A.data_ptr(), 64, A.data_ptr(), 64,
                                 0.0, None, A.data_ptr(), None, None, 0,
                                 torch.cuda.current_stream().cuda_stream)
        assert st == 1


def test_host_operands_row_blocks():
    """FP8 host operands through the row-block staging path equal one device call."""
    p = W.Problem("h8", 2304, 272, 256, "bf16", has_c=True, alpha=0.75, beta=0.5, dist="uniform",
                  c_dist="normal", seed=211, a_fmt="e4m3", b_fmt="e4m3")
    data = W.make(p)
    Dh = G.gemm_fp8(data["A"].pin_memory(), data["B"].pin_memory(), p.M, p.N, p.K,
                    lda=data["lda"], ldb=data["ldb"], a_format=p.a_fmt, b_format=p.b_fmt,
                    out_dtype=torch.bfloat16, alpha=p.alpha, beta=p.beta, C=data["C"].pin_memory())
    torch.cuda.synchronize()
    Dd = run(p, data)
    assert not Dh.is_cuda
    assert torch.equal(Dh.view(torch.int16), Dd.cpu().view(torch.int16))


def test_host_operands_fused_bias_amax_fp8_out():
    """gb_gemm_fp8_host with a host bias, a host amax and an E4M3 output, in two row blocks:
    the same bytes and amax as the device call."""
    p = W.Problem("h8f", 2304, 272, 256, "bf16", has_c=True, alpha=0.5, beta=0.25, dist="normal",
                  c_dist="normal", seed=212, a_fmt="e4m3", b_fmt="e4m3")
    data = W.make(p)
    g = torch.Generator().manual_seed(9)
    bias = torch.randn(p.N, generator=g).to(torch.bfloat16)
    kw = dict(lda=data["lda"], ldb=data["ldb"], a_format=p.a_fmt, b_format=p.b_fmt,
              out_dtype=torch.bfloat16, alpha=p.alpha, beta=p.beta, activation="gelu",
              out_format="e4m3", out_scale=4.0)
    amax_h = torch.full((1,), 0.5, dtype=torch.float32).pin_memory()
    Dh = G.gemm_fp8(data["A"].pin_memory(), data["B"].pin_memory(), p.M, p.N, p.K,
                    C=data["C"].pin_memory(), bias=bias.pin_memory(), amax=amax_h, **kw)
    torch.cuda.synchronize()
    amax_d = torch.full((1,), 0.5, dtype=torch.float32, device=DEV)
    Dd = G.gemm_fp8(data["A"].to(DEV), data["B"].to(DEV), p.M, p.N, p.K, C=data["C"].to(DEV),
                    bias=bias.to(DEV), amax=amax_d, **kw)
    torch.cuda.synchronize()
    assert not Dh.is_cuda and Dh.dtype == torch.float8_e4m3fn
    assert torch.equal(Dh.view(torch.uint8), Dd.cpu().view(torch.uint8))
    assert float(amax_h.item()) == float(amax_d.item()) and float(amax_h.item()) > 0.5
