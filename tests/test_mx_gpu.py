"""GPU parity of the block-scaled FP8 GEMM (gb_gemm_mxfp8) against the fp64 oracle.

Scales are E8M0 powers of two, one per 32 K elements of each row of A and column of B; the
GPU takes them packed by gb_mx_pack_scales, the oracle takes the plain row-major codes.
Scaled FP8 products are still exact in fp32, so the 16-bit acceptance bound applies to the
scaled products, and integer-valued problems must match exactly.
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
ATOM = "((32,4),4):((16,4),1)"    # (row in 128, scale in k-block) -> byte of a 512-byte atom


@pytest.fixture(params=[1, 2, 4, 5, 6, 7], ids=["single", "pair", "narrow_falls_back", "pair224_falls_back", "pair512_falls_back", "pair448_falls_back"])
def variant(request):
    G.set_kernel_variant(request.param)
    yield request.param
    G.set_kernel_variant(0)


def run(p, data, workspace=None, **kw):
    A, B = data["A"].to(DEV), data["B"].to(DEV)
    C = data["C"].to(DEV) if data["C"] is not None else None
    sfa = G.mx_pack_scales(0, p.M, p.K, data["SFA"].to(DEV), data["ld_sf"])
    sfb = G.mx_pack_scales(1, p.N, p.K, data["SFB"].to(DEV), data["ld_sf"])
    D = G.gemm_mxfp8(A, B, p.M, p.N, p.K, lda=data["lda"], ldb=data["ldb"], sfa=sfa, sfb=sfb,
                     a_format=p.a_fmt, b_format=p.b_fmt, out_dtype=W.torch_dtype(p.dtype),
                     alpha=p.alpha, beta=p.beta, C=C, workspace=workspace, **kw)
    st, detail = G.last_device_status()
    assert st == 0, "device status %d detail %#x" % (st, detail)
    return D


def reference(p, data, rows=None, cols=None):
    code = O.dtype_code(p.dtype)
    C = W.bits(data["C"]) if data["C"] is not None else None
    return O.gemm_mx(p.M, p.N, p.K, p.alpha, W.bits(data["A"]), data["lda"], O.dtype_code(p.a_fmt),
                     data["SFA"].numpy(), data["ld_sf"], W.bits(data["B"]), data["ldb"],
                     O.dtype_code(p.b_fmt), data["SFB"].numpy(), data["ld_sf"], p.beta, C, p.N, code,
                     rows=rows, cols=cols)


def check(p, data, D, rows=None, cols=None):
    code = O.dtype_code(p.dtype)
    ref, sab = reference(p, data, rows, cols)
    d = O.decode(code, W.bits(D.cpu())).reshape(p.M, p.N)
    c = O.decode(code, W.bits(data["C"])).reshape(p.M, p.N) if data["C"] is not None else None
    if rows is not None:
        d = d[rows, cols]
        c = None if c is None else c[rows, cols]
    err = np.abs(d - ref)
    bnd = O.bound(code, p.alpha, p.beta, ref, sab, c)
    assert np.all(np.isfinite(d))
    assert np.all(err <= bnd), "worst %.3g of bound" % float(np.max(err / bnd))


def mx_problem(name, M, N, K, dtype="bf16", **kw):
    kw.setdefault("a_fmt", "e4m3")
    kw.setdefault("b_fmt", "e4m3")
    kw.setdefault("scale_codes", (122, 132))
    return W.Problem(name, M, N, K, dtype, **kw)


# --------------------------------------------------------------------------- packing


@pytest.mark.parametrize("operand,rows,K", [(0, 300, 200), (1, 300, 200), (0, 128, 128),
                                            (1, 449, 1000), (0, 5, 33)])
def test_pack_layout(operand, rows, K):
    nsf = -(-K // 32)
    ld = nsf + 3
    g = torch.Generator().manual_seed(rows * 7 + K)
    src = torch.randint(0, 255, (rows, ld), generator=g).to(torch.uint8)
    got = G.mx_pack_scales(operand, rows, K, src.reshape(-1).to(DEV), ld).cpu().numpy()
    kbs = -(-K // 128)
    blk_rows, atom_bytes = (128, 512) if operand == 0 else (224, 1024)
    assert got.size == -(-rows // blk_rows) * kbs * atom_bytes
    want = np.full(got.size, 127, np.uint8)
    r, s = np.meshgrid(np.arange(rows), np.arange(nsf), indexing="ij")
    kb, kk = s // 4, s % 4
    if operand == 0:
        blk, rr = r // 128, r % 128
        off = (blk * kbs + kb) * 512 + L.evaluate(ATOM, (rr + 128 * kk).ravel()).reshape(rr.shape)
    else:
        blk, rn = r // 224, r % 224
        grp, i = rn // 32, rn % 32
        rr = 32 * (grp % 4) + i
        off = ((blk * kbs + kb) * 1024 + (grp // 4) * 512
               + L.evaluate(ATOM, (rr + 128 * kk).ravel()).reshape(rr.shape))
    want[off.ravel()] = src[:, :nsf].numpy().ravel()
    assert np.array_equal(got, want)


# --------------------------------------------------------------------------- GEMM parity


@pytest.mark.parametrize("fa,fb", [("e4m3", "e4m3"), ("e5m2", "e4m3"), ("e4m3", "e5m2")])
def test_integer_exact(variant, fa, fb):
    # int2 values times scales 1 or 2: |sum| <= 16 K = 2048, exact in fp16
    p = mx_problem("mi", 320, 480, 128, "f16", dist="int2", seed=201, a_fmt=fa, b_fmt=fb,
                   scale_codes=(127, 128))
    data = W.make(p)
    D = run(p, data)
    ref, _ = reference(p, data)
    d = O.decode(O.F16, W.bits(D.cpu())).reshape(p.M, p.N)
    assert np.array_equal(d, ref)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_random_ragged(variant, dtype):
    # M, N off the tile grid; K = 200: one k-block of 128 and a 72-wide tail whose last scale
    # block holds 8 elements
    p = mx_problem("mr", 300, 520, 200, dtype, has_c=True, alpha=0.75, beta=0.5, dist="normal",
                   c_dist="normal", seed=202, a_fmt="e4m3", b_fmt="e5m2", lda=208, ldb=224)
    data = W.make(p)
    check(p, data, run(p, data))


@pytest.mark.parametrize("K", [1, 32, 33, 128, 129, 1000])
def test_k_edges(variant, K):
    ld = ((K + 15) // 16) * 16
    p = mx_problem("mk", 257, 232, K, dist="uniform", seed=203, lda=ld, ldb=ld,
                   scale_codes=(110, 140))
    data = W.make(p)
    check(p, data, run(p, data))


def test_wide_scale_range():
    # scales 2^-20 .. 2^20 across blocks: the block structure, not the value range, decides
    p = mx_problem("mw", 256, 448, 512, has_c=True, alpha=1.0, beta=1.0, dist="normal",
                   c_dist="normal", seed=204, scale_codes=(107, 147))
    data = W.make(p)
    check(p, data, run(p, data))


def test_stream_k_mx():
    ws = G.make_workspace(DEV)
    G.set_schedule(2)
    try:
        p = mx_problem("msk", 512, 672, 4096, has_c=True, alpha=0.5, beta=1.0, dist="normal",
                       c_dist="normal", seed=205)
        data = W.make(p)
        check(p, data, run(p, data, workspace=ws))
    finally:
        G.set_schedule(0)


def test_fused_fp8_out(variant):
    p = mx_problem("mf", 384, 1040, 512, has_c=True, alpha=0.25, beta=0.25, dist="normal",
                   c_dist="normal", seed=206)
    data = W.make(p)
    bias = torch.randn(p.N, generator=torch.Generator().manual_seed(9)).to(torch.bfloat16)
    amax = torch.zeros(1, dtype=torch.float32, device=DEV)
    D = run(p, data, bias=bias.to(DEV), activation="gelu", amax=amax, out_format="e4m3",
            out_scale=4.0)
    ref, sab = reference(p, data)
    c = O.decode(O.BF16, W.bits(data["C"])).reshape(p.M, p.N)
    v = O.fused(ref, O.decode(O.BF16, W.bits(bias))[None, :], "gelu")
    err = O.LIPSCHITZ["gelu"] * 2.0 ** -9 * (abs(p.alpha) * sab + np.abs(p.beta * c))
    d = O.decode(O.E4M3, W.bits(D.cpu())).reshape(p.M, p.N)
    target = np.clip(v * 4.0, -448.0, 448.0)
    assert np.all(np.abs(d - target) <= err * 4.0 + O.ulp_fp8(O.E4M3, target))
    assert abs(float(amax.item()) - np.max(np.abs(v))) <= np.max(err) + 1e-6 * np.max(np.abs(v))


def test_full_size_sampled():
    # the throughput problem at its full size, in the launch configuration the bench times
    p = W.FP8_WORKLOADS["gemm8192_mxfp8_bf16_c"]
    data = W.make(p)
    D = run(p, data)
    rng = np.random.default_rng(207)
    rows = np.concatenate([rng.integers(0, p.M, 1500), [0, p.M - 1, 255, 256, 4095]])
    cols = np.concatenate([rng.integers(0, p.N, 1500), [p.N - 1, 0, 223, 224, 8191]])
    check(p, data, D, rows, cols)


def test_argument_errors():
    A = torch.zeros(256 * 256, dtype=torch.uint8, device=DEV)
    h = torch.cuda.current_stream().cuda_stream
    lib = G.lib()
    # missing scales with K > 0
    assert lib.gb_gemm_mxfp8(0, 0, 1, 256, 256, 128, 1.0, A.data_ptr(), 128, None, A.data_ptr(), 128,
                             A.data_ptr(), 0.0, None, A.data_ptr(), None, None, 0, h) == 1
    # misaligned scales
    assert lib.gb_gemm_mxfp8(0, 0, 1, 256, 256, 128, 1.0, A.data_ptr(), 128, A.data_ptr() + 8,
                             A.data_ptr(), 128, A.data_ptr(), 0.0, None, A.data_ptr(), None, None, 0,
                             h) == 2
    # pack: short pitch, bad operand
    assert lib.gb_mx_pack_scales(0, 10, 128, A.data_ptr(), 3, A.data_ptr(), h) == 1
    assert lib.gb_mx_pack_scales(2, 10, 128, A.data_ptr(), 4, A.data_ptr(), h) == 1
