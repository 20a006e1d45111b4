"""GPU parity of the fused epilogue (gb_gemm_ex): bias, ReLU/GELU, amax, FP8 outputs.

Reference: the fp64 GEMM, then the column's bias and the activation in fp64.  Bound: the
GEMM bound scaled by the activation's Lipschitz constant, plus one output ulp (FP8 outputs
are compared after scaling and clamping the reference to the format's range).
"""
import math

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


def make_bias(p, dist="normal", seed=0):
    g = torch.Generator().manual_seed(seed)
    if dist == "int2":
        b = torch.randint(-2, 3, (p.N,), generator=g).float()
    else:
        b = torch.randn(p.N, generator=g)
    return b.to(W.torch_dtype(p.dtype))


def run_fused(p, data, bias, **kw):
    A, B = data["A"].to(DEV), data["B"].to(DEV)
    C = data["C"].to(DEV) if data["C"] is not None else None
    amax = torch.zeros(1, dtype=torch.float32, device=DEV)
    D = G.gemm_fused(A, B, p.M, p.N, p.K, lda=data["lda"], ldb=data["ldb"], majorA=p.majorA,
                     majorB=p.majorB, alpha=p.alpha, beta=p.beta, C=C,
                     bias=None if bias is None else bias.to(DEV), amax=amax, **kw)
    st, detail = G.last_device_status()
    assert st == 0, "device status %d detail %#x" % (st, detail)
    return D, float(amax.item())


def reference(p, data, bias, act):
    code = O.dtype_code(p.dtype)
    C = W.bits(data["C"]) if data["C"] is not None else None
    ref, sab = O.gemm(p.M, p.N, p.K, p.alpha, W.bits(data["A"]), data["lda"],
                      0 if p.majorA == "K" else 1, W.bits(data["B"]), data["ldb"],
                      0 if p.majorB == "K" else 1, p.beta, C, p.N, code)
    b = None if bias is None else O.decode(code, W.bits(bias))[None, :]
    v = O.fused(ref, b, act)
    c = O.decode(code, C).reshape(p.M, p.N) if C is not None else 0.0
    err = O.LIPSCHITZ[act] * math.ldexp(1.0, -9) * (abs(p.alpha) * sab + np.abs(p.beta * c))
    return v, err


def check_16(p, D, v, err):
    code = O.dtype_code(p.dtype)
    d = O.decode(code, W.bits(D.cpu())).reshape(p.M, p.N)
    assert np.all(np.abs(d - v) <= err + O.ulp_out(code, v))


def check_fp8(p, D, v, err, fmt, scale):
    code, maxfin = FP8[fmt]
    d = O.decode(code, D.cpu().view(torch.uint8).numpy().astype(np.uint16)).reshape(p.M, p.N)
    target = np.clip(v * scale, -maxfin, maxfin)
    assert np.all(np.isfinite(d))
    assert np.all(np.abs(d - target) <= err * scale + O.ulp_fp8(code, target))


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("act", ["gelu", "relu", "none"])
def test_bias_activation_16bit(variant, dtype, act):
    p = W.Problem("fe", 300, 520, 200, dtype, has_c=True, alpha=1.25, beta=0.5, dist="normal",
                  c_dist="normal", seed=91)
    data = W.make(p)
    bias = make_bias(p, seed=1)
    D, amax = run_fused(p, data, bias, activation=act)
    v, err = reference(p, data, bias, act)
    check_16(p, D, v, err)
    assert abs(amax - np.max(np.abs(v))) <= np.max(err) + 1e-6 * np.max(np.abs(v))


def test_relu_integer_exact(variant):
    p = W.Problem("fi", 257, 136, 64, "f16", has_c=True, alpha=1.0, beta=1.0, dist="int2",
                  c_dist="int2", seed=92)
    data = W.make(p)
    bias = make_bias(p, "int2", seed=2)
    D, amax = run_fused(p, data, bias, activation="relu")
    v, _ = reference(p, data, bias, "relu")
    d = O.decode(O.F16, W.bits(D.cpu())).reshape(p.M, p.N)
    assert np.array_equal(d, v)
    assert amax == np.max(np.abs(v))


@pytest.mark.parametrize("fmt,scale", [("e4m3", 16.0), ("e5m2", 256.0), ("e4m3", 1000.0)])
@pytest.mark.parametrize("N", [1040, 1000])        # 16-byte FP8 stores / byte stores
def test_fp8_outputs(variant, fmt, scale, N):
    p = W.Problem("f8", 520, N, 256, "bf16", has_c=True, alpha=1.0, beta=0.25, dist="uniform",
                  c_dist="normal", seed=93)
    data = W.make(p)
    bias = make_bias(p, seed=3)
    D, amax = run_fused(p, data, bias, activation="gelu", out_format=fmt, out_scale=scale)
    v, err = reference(p, data, bias, "gelu")
    check_fp8(p, D, v, err, fmt, scale)
    assert abs(amax - np.max(np.abs(v))) <= np.max(err) + 1e-6 * np.max(np.abs(v))


def test_fp8_integer_exact(variant):
    # |v| <= 2*4 + 2 = 10: every value is an integer E4M3 represents exactly
    p = W.Problem("f8i", 384, 512, 2, "f16", dist="int2", seed=94, lda=8, ldb=8)
    data = W.make(p)
    bias = make_bias(p, "int2", seed=4)
    D, _ = run_fused(p, data, bias, activation="relu", out_format="e4m3", out_scale=1.0)
    v, _ = reference(p, data, bias, "relu")
    d = O.decode(O.E4M3, D.cpu().view(torch.uint8).numpy().astype(np.uint16)).reshape(p.M, p.N)
    assert np.array_equal(d, v)


def test_fused_with_stream_k():
    ws = G.make_workspace(DEV)
    G.set_schedule(2)
    try:
        p = W.Problem("fsk", 512, 768, 2048, "bf16", has_c=True, alpha=0.5, beta=1.0,
                      dist="normal", c_dist="normal", seed=95)
        data = W.make(p)
        bias = make_bias(p, seed=5)
        D, amax = run_fused(p, data, bias, activation="gelu", workspace=ws)
        v, err = reference(p, data, bias, "gelu")
        check_16(p, D, v, err)
        assert abs(amax - np.max(np.abs(v))) <= np.max(err) + 1e-6 * np.max(np.abs(v))
    finally:
        G.set_schedule(0)


def test_fused_argument_errors():
    A = torch.zeros(64 * 64, dtype=torch.float16, device=DEV)
    for kw in (dict(activation="none", out_format="e4m3", out_scale=0.0),
               dict(activation="none", out_format="e5m2", out_scale=float("inf"))):
        with pytest.raises(G.GemmError) as e:
            G.gemm_fused(A, A, 64, 64, 64, lda=64, ldb=64, **kw)
        assert e.value.status == 1
    from layout_algebra_gb300._native import Epilogue
    import ctypes
    bad = Epilogue(None, 7, None, 0, 1.0)
    st = G.lib().gb_gemm_ex(0, 64, 64, 64, 1.0, A.data_ptr(), 64, 0, A.data_ptr(), 64, 0, 0.0,
                            None, A.data_ptr(), ctypes.byref(bad), None, 0,
                            torch.cuda.current_stream().cuda_stream)
    assert st == 1
