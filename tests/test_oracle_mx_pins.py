"""Pins for the oracle's block-scaled (MX) FP8 GEMM: scales of 2^(e-127) shared by 32 K elements."""
import math

import numpy as np
import pytest
import torch

from oracle import gemm_ref as O


def _fp8_codes(rng, n, code):
    c = rng.integers(0, 256, n).astype(np.uint16)
    bad = ((c & 0x7F) == 0x7F) if code == O.E4M3 else ((c & 0x7C) == 0x7C)
    c[bad] &= 0x83
    return c


def _torch_decode(code, c):
    tdt = torch.float8_e4m3fn if code == O.E4M3 else torch.float8_e5m2
    return torch.from_numpy(c.astype(np.uint8)).view(tdt).double().numpy()


@pytest.mark.parametrize("K", [32, 70, 129])
def test_mx_against_library_matmul(K):
    # torch's FP8 decode, numpy's ldexp for the block scales and a float64 matmul: none of
    # the oracle's code.  Scale pitches wider than ceil(K/32) catch a pitch mix-up; distinct
    # formats and scales for A and B catch a swapped operand.
    rng = np.random.default_rng(K)
    M, N = 7, 9
    kb = -(-K // 32)
    lda, ldb, ldsa, ldsb = K + 3, K + 5, kb + 2, kb + 1
    A = _fp8_codes(rng, M * lda, O.E4M3)
    B = _fp8_codes(rng, N * ldb, O.E5M2)
    SFA = rng.integers(120, 135, M * ldsa).astype(np.uint8)
    SFB = rng.integers(118, 131, N * ldsb).astype(np.uint8)
    C = O.round_to(O.BF16, rng.standard_normal(M * N))
    a = _torch_decode(O.E4M3, A).reshape(M, lda)[:, :K]
    b = _torch_decode(O.E5M2, B).reshape(N, ldb)[:, :K]
    ea = SFA.reshape(M, ldsa)[:, :kb].astype(np.int64) - 127
    eb = SFB.reshape(N, ldsb)[:, :kb].astype(np.int64) - 127
    a = np.ldexp(a, np.repeat(ea, 32, axis=1)[:, :K])
    b = np.ldexp(b, np.repeat(eb, 32, axis=1)[:, :K])
    want = 1.5 * (a @ b.T) - 0.25 * O.decode(O.BF16, C).reshape(M, N)
    ref, sab = O.gemm_mx(M, N, K, 1.5, A, lda, O.E4M3, SFA, ldsa, B, ldb, O.E5M2, SFB, ldsb,
                         -0.25, C, N, O.BF16)
    assert np.allclose(ref, want, rtol=0, atol=1e-12 * (np.max(sab) + 1.0))
    assert np.allclose(sab, np.abs(a) @ np.abs(b).T, rtol=1e-13)


def test_mx_unit_scales_reduce_to_plain_fp8():
    rng = np.random.default_rng(3)
    M, N, K = 5, 6, 96
    A = _fp8_codes(rng, M * K, O.E4M3)
    B = _fp8_codes(rng, N * K, O.E4M3)
    ones_a = np.full(M * 3, 127, np.uint8)
    ones_b = np.full(N * 3, 127, np.uint8)
    ref, _ = O.gemm_mx(M, N, K, 1.0, A, K, O.E4M3, ones_a, 3, B, K, O.E4M3, ones_b, 3, 0.0, None,
                       N, O.F16)
    plain, _ = O.gemm(M, N, K, 1.0, A, K, O.K_MAJOR, B, K, O.K_MAJOR, 0.0, None, N, O.F16,
                      a_dtype=O.E4M3, b_dtype=O.E4M3)
    assert np.array_equal(ref, plain)


def test_e8m0_values():
    one = O.round_to(O.E4M3, [1.0])          # 1.0 in E4M3
    for e, want in [(0, 2.0 ** -127), (127, 1.0), (130, 8.0), (254, 2.0 ** 127)]:
        ref, _ = O.gemm_mx(1, 1, 1, 1.0, one, 1, O.E4M3, np.array([e], np.uint8), 1, one, 1,
                           O.E4M3, np.array([127], np.uint8), 1, 0.0, None, 1, O.F16)
        assert ref[0, 0] == want
    ref, _ = O.gemm_mx(1, 1, 1, 1.0, one, 1, O.E4M3, np.array([255], np.uint8), 1, one, 1,
                       O.E4M3, np.array([127], np.uint8), 1, 0.0, None, 1, O.F16)
    assert math.isnan(ref[0, 0])


def test_mx_block_boundary_exact():
    # A = B = 1 everywhere; A's second block (k = 32..63) scaled by 2^3, B's third by 2^-2:
    # each output is 32 * (1 + 8 + 0.25) exactly
    M, N, K = 2, 3, 96
    one = O.round_to(O.E4M3, [1.0])[0]
    A = np.full(M * K, one, np.uint16)
    B = np.full(N * K, one, np.uint16)
    SFA = np.tile(np.array([127, 130, 127], np.uint8), M)
    SFB = np.tile(np.array([127, 127, 125], np.uint8), N)
    ref, _ = O.gemm_mx(M, N, K, 1.0, A, K, O.E4M3, SFA, 3, B, K, O.E4M3, SFB, 3, 0.0, None, N, O.F16)
    assert np.all(ref == 32 * (1 + 8 + 0.25))
