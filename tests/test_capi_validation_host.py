"""Argument checks of every GEMM entry point of the C ABI, on the host (no GPU needed).

Each call below breaks exactly one documented rule and must return its status before any
device is touched (the library checks arguments first), so the pointers are placeholders
that are never dereferenced.  No call here has valid arguments: on a machine with a GPU a
valid call would launch.
"""
import ctypes

import pytest
import torch

from layout_algebra_gb300 import _native

# Host-only checks: on a machine with a GPU they add nothing (the GPU tests cover the same
# statuses with real buffers), and a case that slipped through validation would launch.
pytestmark = pytest.mark.skipif(torch.cuda.is_available(), reason="host-only argument checks")

OK, INVALID, MISALIGNED = 0, 1, 2
P = 1 << 20            # a 256-byte-aligned placeholder address
E4M3, E5M2 = 0, 1      # gb_fp8_format
F16, BF16 = 0, 1


def epi(bias=None, act=0, amax=None, out=0, scale=1.0):
    return _native.Epilogue(bias, act, amax, out, scale)


def gemm_ex(e, M=64, N=64, K=64, ws=None):
    return _native.lib().gb_gemm_ex(F16, M, N, K, 1.0, P, K, 0, P, K, 0, 0.0, None, P,
                                    ctypes.byref(e), ws, 0 if ws is None else 1 << 30, None)


@pytest.mark.parametrize("e,status", [
    (epi(act=3), INVALID),                         # unknown activation
    (epi(act=-1), INVALID),
    (epi(out=3), INVALID),                         # unknown output format
    (epi(out=1, scale=0.0), INVALID),              # FP8 output needs a positive finite scale
    (epi(out=2, scale=float("inf")), INVALID),
    (epi(amax=P + 2), MISALIGNED),                 # amax is a float
    (epi(bias=P + 1), MISALIGNED),                 # bias holds 16-bit values
])
def test_fused_epilogue_arguments(e, status):
    assert gemm_ex(e) == status


def test_workspace_alignment():
    lib = _native.lib()
    # 16-byte aligned but not 256-byte aligned
    assert lib.gb_gemm_f16_ws(64, 64, 64, 1.0, P, 64, 0, P, 64, 0, 0.0, None, P, P + 16, 1 << 30,
                              None) == MISALIGNED
    assert gemm_ex(epi(act=1), ws=P + 128) == MISALIGNED


@pytest.mark.parametrize("args,status", [
    ((5, E4M3, BF16, 64, 64, 64, 64, 64), INVALID),     # unknown A format
    ((E4M3, 2, BF16, 64, 64, 64, 64, 64), INVALID),     # unknown B format
    ((E4M3, E5M2, 7, 64, 64, 64, 64, 64), INVALID),     # output must be fp16 or bf16
    ((E4M3, E4M3, F16, -1, 64, 64, 64, 64), INVALID),   # negative size
    ((E4M3, E4M3, F16, 64, 64, 40, 24, 48), INVALID),   # lda < K
    ((E4M3, E4M3, F16, 64, 64, 24, 24, 48), MISALIGNED),  # 24-byte rows of A
    ((E5M2, E4M3, BF16, 64, 64, 32, 32, 40), MISALIGNED),  # 40-byte rows of B
])
def test_fp8_arguments(args, status):
    a, b, out, M, N, K, lda, ldb = args
    assert _native.lib().gb_gemm_fp8(a, b, out, M, N, K, 1.0, P, lda, P, ldb, 0.0, None, P, None,
                                     None, 0, None) == status


def test_fp8_pointer_alignment():
    lib = _native.lib()
    assert lib.gb_gemm_fp8(E4M3, E4M3, BF16, 64, 64, 64, 1.0, P + 8, 64, P, 64, 0.0, None, P, None,
                           None, 0, None) == MISALIGNED
    assert lib.gb_gemm_fp8(E4M3, E4M3, BF16, 64, 64, 64, 1.0, P, 64, P, 64, 0.5, None, P, None,
                           None, 0, None) == INVALID          # beta != 0 needs C


@pytest.mark.parametrize("sfa,sfb,status", [
    (None, P, INVALID),            # block-scaled inputs need both scale arrays
    (P, None, INVALID),
    (P + 8, P, MISALIGNED),        # packed scales are copied by tensor copies
    (P, P + 4, MISALIGNED),
])
def test_block_scaled_scale_arguments(sfa, sfb, status):
    assert _native.lib().gb_gemm_mxfp8(E4M3, E4M3, BF16, 256, 256, 256, 1.0, P, 256, sfa, P, 256, sfb,
                                       0.0, None, P, None, None, 0, None) == status


def test_block_scaled_formats():
    assert _native.lib().gb_gemm_mxfp8(E4M3, 3, BF16, 256, 256, 256, 1.0, P, 256, P, P, 256, P,
                                       0.0, None, P, None, None, 0, None) == INVALID


def test_scale_factor_sizes():
    """Packed scale bytes: A in 512-byte atoms per (128 rows, 128-element k-block), B in two
    atoms per (224 columns, k-block)."""
    lib = _native.lib()
    n = ctypes.c_size_t()
    assert lib.gb_mx_scales_bytes(0, 300, 1000, ctypes.byref(n)) == OK and n.value == 3 * 8 * 512
    assert lib.gb_mx_scales_bytes(1, 300, 100, ctypes.byref(n)) == OK and n.value == 2 * 1 * 1024
    assert lib.gb_mx_scales_bytes(1, 224, 128, ctypes.byref(n)) == OK and n.value == 1024
    assert lib.gb_mx_scales_bytes(0, 0, 128, ctypes.byref(n)) == OK and n.value == 0
    assert lib.gb_mx_scales_bytes(2, 8, 8, ctypes.byref(n)) == INVALID
    assert lib.gb_mx_scales_bytes(0, -1, 8, ctypes.byref(n)) == INVALID
    assert lib.gb_mx_scales_bytes(0, 8, 8, None) == INVALID
    # packing: nothing to do for no rows; a source row shorter than K/32 scales is refused
    assert lib.gb_mx_pack_scales(0, 0, 128, P, 4, P, None) == OK
    assert lib.gb_mx_pack_scales(0, 128, 128, P, 3, P, None) == INVALID
    assert lib.gb_mx_pack_scales(1, 128, 128, None, 4, P, None) == INVALID


def test_schedule_and_dtype_arguments():
    lib = _native.lib()
    for bad in (-1, 3):
        assert lib.gb_set_schedule(bad) == INVALID
    assert lib.gb_gemm_ex(5, 64, 64, 64, 1.0, P, 64, 0, P, 64, 0, 0.0, None, P, None, None, 0,
                          None) == INVALID
    assert lib.gb_gemm_noalloc(5, 64, 64, 64, 1.0, P, 64, 0, P, 64, 0, 0.0, None, P, None) == INVALID


@pytest.mark.parametrize("fn", ["gb_gemm_f16_host", "gb_gemm_bf16_host"])
@pytest.mark.parametrize("args,status", [
    ((-1, 64, 64, 1.0, P, 64, 0, P, 64, 0, 0.0, None, P), INVALID),     # negative M
    ((64, 64, 64, 1.0, P, 32, 0, P, 64, 0, 0.0, None, P), INVALID),     # lda < K
    ((64, 64, 64, 1.0, P, 68, 0, P, 64, 0, 0.0, None, P), MISALIGNED),  # lda*2 not a multiple of 16
    ((64, 64, 64, 1.0, P, 64, 0, P, 64, 2, 0.0, None, P), INVALID),     # bad major
    ((64, 64, 64, 1.0, P, 64, 0, P, 64, 0, 1.0, None, P), INVALID),     # beta != 0 without C
    ((64, 64, 64, 1.0, P, 64, 0, P, 64, 0, 0.0, None, None), INVALID),  # no D
    ((64, 64, 64, 1.0, None, 64, 0, P, 64, 0, 0.0, None, P), INVALID),  # no A with K > 0
    ((0, 64, 64, 1.0, None, 0, 0, None, 0, 0, 0.0, None, None), OK),    # empty: nothing to do
])
def test_host_entry_arguments(fn, args, status):
    """The host-operand entry points check their arguments before any copy."""
    assert getattr(_native.lib(), fn)(*args, None) == status


def test_fp8_host_entry_arguments():
    lib = _native.lib()
    f = lib.gb_gemm_fp8_host
    assert f(E4M3, 7, BF16, 64, 64, 64, 1.0, P, 64, P, 64, 0.0, None, P, None, None) == INVALID
    assert f(E4M3, E4M3, 9, 64, 64, 64, 1.0, P, 64, P, 64, 0.0, None, P, None, None) == INVALID
    assert f(E4M3, E4M3, BF16, 64, 64, 64, 1.0, P, 72, P, 64, 0.0, None, P, None, None) == MISALIGNED
    assert f(E4M3, E5M2, F16, 64, 64, 64, 1.0, P, 64, P, 64, 0.0, None, P,
             ctypes.byref(epi(out=5)), None) == INVALID


def test_host_row_block_arguments():
    lib = _native.lib()
    bounds = (ctypes.c_int64 * 9)()
    n = ctypes.c_int()
    assert lib.gb_gemm_host_row_blocks(-1, bounds, ctypes.byref(n)) == INVALID
    assert lib.gb_gemm_host_row_blocks(10, None, ctypes.byref(n)) == INVALID
    assert lib.gb_gemm_host_row_blocks(10, bounds, ctypes.byref(n)) == OK and n.value == 1
