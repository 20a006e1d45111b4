"""Pins for the oracle's FP8 codecs, GELU and the fused-epilogue bound constants."""
import math

import numpy as np
import pytest
import torch

from oracle import gemm_ref as O


@pytest.mark.parametrize("code,tdt", [(O.E4M3, torch.float8_e4m3fn), (O.E5M2, torch.float8_e5m2)])
def test_fp8_decode_exhaustive(code, tdt):
    b = np.arange(256, dtype=np.uint16)
    got = O.decode(code, b)
    want = torch.from_numpy(b.astype(np.uint8)).view(tdt).double().numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


@pytest.mark.parametrize("code,maxfin,maxcode", [(O.E4M3, 448.0, 0x7E), (O.E5M2, 57344.0, 0x7B)])
def test_fp8_round_nearest_even_saturating(code, maxfin, maxcode):
    rng = np.random.default_rng(int(maxfin))
    x = np.ldexp(rng.random(20000) + 0.5, rng.integers(-20, 17, 20000))
    x *= np.where(rng.random(20000) < 0.5, -1.0, 1.0)
    got = O.round_to(code, x)
    val = O.decode(code, got)
    inside = np.abs(x) <= maxfin
    # saturation: beyond the largest finite value the result is that value
    assert np.all(np.abs(val[~inside]) == maxfin)
    assert np.all(np.sign(val[~inside]) == np.sign(x[~inside]))
    # inside: no neighbouring finite code is nearer
    for delta in (-1, 1):
        nb = got.astype(np.int64) + delta
        ok = inside & ((nb & 0x7F) <= maxcode) & ((nb & 0x7F) >= 0)
        nv = O.decode(code, nb[ok].astype(np.uint16))
        assert np.all(np.abs(x[ok] - val[ok]) <= np.abs(x[ok] - nv))
    # hand-placed ties go to the even code
    one = 0x38 if code == O.E4M3 else 0x3C
    step = 0.125 if code == O.E4M3 else 0.25
    assert O.round_to(code, [1 + step / 2])[0] == one            # between 1 (even) and 1+step
    assert O.round_to(code, [1 + 1.5 * step])[0] == one + 2      # between 1+step and 1+2step (even)
    assert O.round_to(code, [maxfin * 4])[0] == maxcode
    assert O.round_to(code, [-maxfin * 4])[0] == 0x80 | maxcode


def test_gelu_pins():
    # GELU(v) = v * Phi(v): textbook normal-CDF values
    assert math.isclose(float(O.gelu([1.0])[0]), 0.8413447460685429, rel_tol=1e-14)
    assert math.isclose(float(O.gelu([2.0])[0]), 2 * 0.9772498680518208, rel_tol=1e-14)
    assert O.gelu([0.0])[0] == 0.0
    v = np.linspace(-6, 6, 1001)
    assert np.allclose(O.gelu(v) - O.gelu(-v), v, atol=1e-14)   # erf is odd
    assert np.all(np.abs(O.gelu([-40.0, 40.0]) - np.array([0.0, 40.0])) < 1e-12)


def test_lipschitz_constants_bound_the_activations():
    v = np.linspace(-10, 10, 200001)
    for act in ("relu", "gelu"):
        y = O.fused(v, activation=act)
        slope = np.max(np.abs(np.diff(y) / np.diff(v)))
        assert slope <= O.LIPSCHITZ[act]


def test_fused_bias_then_activation():
    ref = np.array([[-1.0, 0.5], [2.0, -3.0]])
    bias = np.array([1.5, -1.0])
    assert np.array_equal(O.fused(ref, bias, "relu"), np.array([[0.5, 0.0], [3.5, 0.0]]))
    assert np.array_equal(O.fused(ref, bias, "none"), ref + bias)


def _fp8_codes(rng, n, code):
    """Random finite FP8 codes (NaN codes excluded; E5M2 infinities excluded)."""
    c = rng.integers(0, 256, n).astype(np.uint16)
    if code == O.E4M3:
        bad = (c & 0x7F) == 0x7F
    else:
        bad = (c & 0x7C) == 0x7C
    c[bad] &= 0x83          # a small finite value of the same sign instead
    return c


def _torch_decode(code, c):
    tdt = torch.float8_e4m3fn if code == O.E4M3 else torch.float8_e5m2
    return torch.from_numpy(c.astype(np.uint8)).view(tdt).double().numpy()


@pytest.mark.parametrize("fa,fb", [(O.E4M3, O.E5M2), (O.E5M2, O.E4M3), (O.E4M3, O.E4M3)])
def test_typed_gemm_against_library_matmul(fa, fb):
    # Decoding by torch's own FP8 types and a float64 matmul (a library routine) is
    # independent of the oracle's decoders and loop; a swapped A/B format fails it.
    rng = np.random.default_rng(7 + fa + 2 * fb)
    M, N, K = 9, 11, 37
    A = _fp8_codes(rng, M * K, fa)          # K-major: A[i*K + k]
    B = _fp8_codes(rng, N * K, fb)          # K-major: B[j*K + k]
    C = O.round_to(O.BF16, rng.standard_normal(M * N))
    a = _torch_decode(fa, A).reshape(M, K)
    b = _torch_decode(fb, B).reshape(N, K).T
    want = 0.75 * (a @ b) + 0.5 * O.decode(O.BF16, C).reshape(M, N)
    ref, sab = O.gemm(M, N, K, 0.75, A, K, O.K_MAJOR, B, K, O.K_MAJOR, 0.5, C, N, O.BF16,
                      a_dtype=fa, b_dtype=fb)
    assert np.allclose(ref, want, rtol=0, atol=1e-12 * (np.max(sab) + 1.0))
    assert np.allclose(sab, np.abs(a) @ np.abs(b), rtol=1e-13)
    if fa != fb:
        swapped, _ = O.gemm(M, N, K, 0.75, A, K, O.K_MAJOR, B, K, O.K_MAJOR, 0.5, C, N, O.BF16,
                            a_dtype=fb, b_dtype=fa)
        assert not np.allclose(swapped, want)


def test_typed_gemm_integer_exact():
    # integers -2..2 are exact in both FP8 formats: the result is an integer matmul
    rng = np.random.default_rng(11)
    M, N, K = 6, 5, 40
    ai = rng.integers(-2, 3, (M, K))
    bi = rng.integers(-2, 3, (K, N))
    A = O.round_to(O.E4M3, ai.astype(np.float64).ravel())
    B = O.round_to(O.E5M2, bi.T.astype(np.float64).ravel())
    ref, _ = O.gemm(M, N, K, 1.0, A, K, O.K_MAJOR, B, K, O.K_MAJOR, 0.0, None, N, O.F16,
                    a_dtype=O.E4M3, b_dtype=O.E5M2)
    assert np.array_equal(ref, (ai @ bi).astype(np.float64))


@pytest.mark.parametrize("code,tdt,maxcode", [(O.E4M3, torch.float8_e4m3fn, 0x7E),
                                               (O.E5M2, torch.float8_e5m2, 0x7B)])
def test_ulp_fp8_is_the_gap_to_the_next_code(code, tdt, maxcode):
    """ulp_fp8 (part of the FP8-output acceptance bound) equals, at every finite non-negative
    value of the format, the distance to the next larger finite value, read off torch's own
    float8 decoding (independent of the oracle's decoder)."""
    b = np.arange(maxcode + 1, dtype=np.uint8)     # 0 .. the largest finite code
    vals = torch.from_numpy(b).view(tdt).double().numpy()
    gaps = vals[1:] - vals[:-1]
    assert np.array_equal(O.ulp_fp8(code, vals[:-1]), gaps)
    # the sign does not matter
    assert np.array_equal(O.ulp_fp8(code, -vals[:-1]), gaps)


@pytest.mark.parametrize("code,points", [
    # OCP E4M3: 3 fraction bits, smallest normal exponent -6, largest finite 448 = 1.75 * 2^8
    (O.E4M3, [(0.0, 2.0 ** -9), (1.0, 2.0 ** -3), (448.0, 2.0 ** 5), (2.0 ** -6, 2.0 ** -9),
              (2.0 ** -7, 2.0 ** -9), (3.0, 2.0 ** -2)]),
    # OCP E5M2: 2 fraction bits, smallest normal exponent -14, largest finite 57344 = 1.75 * 2^15
    (O.E5M2, [(0.0, 2.0 ** -16), (1.0, 2.0 ** -2), (57344.0, 2.0 ** 13), (2.0 ** -14, 2.0 ** -16),
              (2.0 ** -15, 2.0 ** -16), (3.0, 2.0 ** -1)]),
])
def test_ulp_fp8_values_fixed_by_the_formats(code, points):
    """Spacings the two OCP FP8 formats fix by their field widths."""
    r = np.array([x for x, _ in points])
    want = np.array([u for _, u in points])
    assert np.array_equal(O.ulp_fp8(code, r), want)
