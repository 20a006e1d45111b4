"""Pins for the GEMM oracle: it is checked against things other than itself.

  * exhaustive decode of both 16-bit formats against library conversions;
  * round-to-nearest-even against numpy (binary16) and against a brute-force nearest
    search (bfloat16), plus hand-placed ties;
  * integer workloads against exact int64 products;
  * closed forms: identity, all-ones A (column sums), all-ones B (row sums);
  * exact rational brute force (fractions) on tiny shapes;
  * numpy's float64 matmul within the fp64 summation bound;
  * a planted transposition that the closed forms must catch.
"""
import math
import random
from fractions import Fraction

import numpy as np
import pytest
import torch

from layout_algebra_gb300 import workloads as W
from oracle import gemm_ref as O

U53 = math.ldexp(1.0, -53)


def _logical_bits(t):
    return W.bits(t)


def _run(p, data, rows=None, cols=None):
    code = O.dtype_code(p.dtype)
    C = W.bits(data["C"]) if data["C"] is not None else None
    return O.gemm(p.M, p.N, p.K, p.alpha, W.bits(data["A"]), data["lda"],
                  0 if p.majorA == "K" else 1, W.bits(data["B"]), data["ldb"],
                  0 if p.majorB == "K" else 1, p.beta, C, p.N, code, rows, cols)


# ----------------------------------------------------------------------------- formats


def test_decode_f16_exhaustive():
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = O.decode(O.F16, allbits)
    want = allbits.view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def test_decode_bf16_exhaustive():
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    want = torch.from_numpy(allbits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    got = O.decode(O.BF16, allbits)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def _random_doubles(n, seed):
    rng = np.random.default_rng(seed)
    mags = np.ldexp(rng.random(n) + 0.5, rng.integers(-140, 130, n))
    signs = np.where(rng.random(n) < 0.5, -1.0, 1.0)
    return mags * signs


def test_round_f16_matches_numpy_and_ties():
    x = _random_doubles(200000, 1)
    x = x[np.abs(x) < 1e6]
    # values sitting exactly half-way between neighbouring binary16 numbers
    lo = np.arange(0, 0x7bff, 7, dtype=np.uint16)
    a = lo.view(np.float16).astype(np.float64)
    b = (lo + 1).view(np.float16).astype(np.float64)
    mids = (a + b) / 2
    x = np.concatenate([x, mids, -mids, [65504.0, 65519.0, 65520.0, 70000.0, 0.0, -0.0]])
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    got = O.round_to(O.F16, x)
    assert np.array_equal(got, want)
    # hand-placed ties: 1 + 2^-11 sits between 1 (even) and 1 + 2^-10 (odd)
    assert O.round_to(O.F16, [1 + 2.0**-11])[0] == 0x3C00
    assert O.round_to(O.F16, [1 + 3 * 2.0**-11])[0] == 0x3C02
    assert O.round_to(O.F16, [2.0**-25])[0] == 0x0000      # half the smallest subnormal
    assert O.round_to(O.F16, [3 * 2.0**-25])[0] == 0x0002


def test_round_bf16_is_nearest_even():
    x = _random_doubles(50000, 2)
    got = O.round_to(O.BF16, x)
    val = O.decode(O.BF16, got)
    finite = np.isfinite(val)
    # neighbours one code below and above in magnitude (same sign)
    for delta in (-1, 1):
        nb = (got.astype(np.int64) + delta)
        ok = (nb & 0x7fff) < 0x7f80
        nb = nb[ok & finite].astype(np.uint16)
        xv = x[ok & finite]
        nv = O.decode(O.BF16, nb)
        rv = val[ok & finite]
        assert np.all(np.abs(xv - rv) <= np.abs(xv - nv))
    # ties go to the even code
    for base in (0x3F80, 0x4049, 0x0001, 0x7F00):
        a = O.decode(O.BF16, np.array([base], np.uint16))[0]
        b = O.decode(O.BF16, np.array([base + 1], np.uint16))[0]
        r = O.round_to(O.BF16, [(a + b) / 2])[0]
        assert r == (base if base % 2 == 0 else base + 1)
    big = math.ldexp(255.0, 120)
    assert O.round_to(O.BF16, [big])[0] == 0x7F7F
    assert O.round_to(O.BF16, [big + math.ldexp(1.0, 119)])[0] == 0x7F80   # the tie overflows


def test_ulp_out_values():
    assert O.ulp_out(O.F16, 1.0) == 2.0**-10
    assert O.ulp_out(O.F16, 1.5) == 2.0**-10
    assert O.ulp_out(O.F16, 2.0) == 2.0**-9
    assert O.ulp_out(O.F16, 0.0) == 2.0**-24
    assert O.ulp_out(O.F16, 1e-7) == 2.0**-24
    assert O.ulp_out(O.BF16, 1.0) == 2.0**-7
    assert O.ulp_out(O.BF16, -300.0) == 2.0**1
    assert O.ulp_out(O.BF16, 0.0) == 2.0**-133


# ----------------------------------------------------------------------------- GEMM


def test_integer_workload_is_exact():
    p = W.WORKLOADS["gemm256_int_f16"]
    data = W.make(p, logical=True)
    ref, _ = _run(p, data)
    a = data["a"].to(torch.int64).numpy()
    b = data["b"].to(torch.int64).numpy()
    exact = a @ b
    assert np.array_equal(ref, exact.astype(np.float64))
    # the fp16 outputs are exact too: |sum| <= 256*4 < 2^11
    back = O.decode(O.F16, O.round_to(O.F16, ref))
    assert np.array_equal(back, ref)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("majors", [("K", "K"), ("MN", "MN"), ("K", "MN"), ("MN", "K")])
def test_identity_closed_form(dtype, majors):
    M = K = 48
    N = 40
    p = W.Problem("id", M, N, K, dtype, majorA=majors[0], majorB=majors[1], has_c=True,
                  alpha=0.75, beta=-1.5, dist="uniform", seed=11)
    data = W.make(p, logical=True)
    eye = torch.eye(M, dtype=W.torch_dtype(dtype))
    lda, _ = W.leading_dims(p)
    data["A"] = W.store_a(eye, p.majorA, lda)
    ref, _ = _run(p, data)
    b = data["b"].double().numpy()
    c = data["c"].double().numpy()
    want = 0.75 * b + (-1.5) * c      # each entry is one product plus one term: exact in fp64
    assert np.array_equal(ref, want)


@pytest.mark.parametrize("which", ["A", "B"])
def test_all_ones_closed_forms(which):
    M, N, K = 33, 29, 300
    p = W.Problem("ones", M, N, K, "f16", dist="uniform", seed=12)
    data = W.make(p, logical=True)
    lda, ldb = W.leading_dims(p)
    if which == "A":
        data["A"] = W.store_a(torch.ones(M, K, dtype=torch.float16), "K", lda)
        col = data["b"].double().numpy()
        want = np.array([[math.fsum(col[:, j]) for j in range(N)]] * M)       # column sums
        mag = np.array([[math.fsum(np.abs(col[:, j])) for j in range(N)]] * M)
    else:
        data["B"] = W.store_b(torch.ones(K, N, dtype=torch.float16), "K", ldb)
        row = data["a"].double().numpy()
        want = np.array([[math.fsum(row[i, :])] * N for i in range(M)])      # row sums
        mag = np.array([[math.fsum(np.abs(row[i, :]))] * N for i in range(M)])
    ref, sab = _run(p, data)
    assert np.all(np.abs(ref - want) <= K * U53 * mag)
    assert np.allclose(sab, mag, rtol=1e-12, atol=0)


def test_planted_transpose_is_caught():
    """Reading B with the wrong major must break the column-sum closed form."""
    M, N, K = 16, 24, 24
    p = W.Problem("plant", M, N, K, "f16", dist="uniform", seed=13)
    data = W.make(p, logical=True)
    lda, ldb = W.leading_dims(p)
    data["A"] = W.store_a(torch.ones(M, K, dtype=torch.float16), "K", lda)
    col = data["b"].double().numpy()
    want = np.array([[math.fsum(col[:, j]) for j in range(N)]] * M)
    # planted mistake: tell the oracle that B is N-major while it is stored K-major
    ref, _ = O.gemm(M, N, K, 1.0, W.bits(data["A"]), lda, 0, W.bits(data["B"]), ldb, 1,
                    0.0, None, N, O.F16)
    assert not np.allclose(ref, want)


@pytest.mark.parametrize("seed", range(12))
def test_bruteforce_fractions_tiny(seed):
    rnd = random.Random(seed)
    M, N, K = rnd.randint(1, 6), rnd.randint(1, 6), rnd.randint(1, 8)
    dtype = "f16" if seed % 2 == 0 else "bf16"
    majors = [("K", "K"), ("MN", "MN"), ("K", "MN"), ("MN", "K")][seed % 4]
    alpha = rnd.choice([1.0, -0.5, 1.25, 3.0])
    beta = rnd.choice([0.0, 0.5, -2.0])
    p = W.Problem("tiny", M, N, K, dtype, majorA=majors[0], majorB=majors[1],
                  has_c=beta != 0.0, alpha=alpha, beta=beta, dist="normal", seed=100 + seed)
    data = W.make(p, logical=True)
    ref, sab = _run(p, data)
    a = data["a"].double().numpy()
    b = data["b"].double().numpy()
    c = data["c"].double().numpy() if data["c"] is not None else None
    for i in range(M):
        for j in range(N):
            s = sum(Fraction(a[i, k]) * Fraction(b[k, j]) for k in range(K))
            exact = Fraction(alpha) * s
            if beta != 0:
                exact += Fraction(beta) * Fraction(c[i, j])
            mag = sum(abs(Fraction(a[i, k]) * Fraction(b[k, j])) for k in range(K))
            tol = abs(alpha) * K * U53 * float(mag) + 4 * U53 * abs(float(exact)) + 1e-300
            assert abs(Fraction(ref[i, j]) - exact) <= Fraction(tol)
            assert math.isclose(sab[i, j], float(mag), rel_tol=1e-12, abs_tol=0)


@pytest.mark.parametrize("majors", [("K", "K"), ("MN", "MN"), ("K", "MN"), ("MN", "K")])
def test_numpy_crosscheck_and_majors(majors):
    M, N, K = 37, 53, 91
    base = W.Problem("x", M, N, K, "bf16", has_c=True, alpha=1.25, beta=0.5,
                     dist="normal", seed=21)
    p = base.with_(majorA=majors[0], majorB=majors[1])
    data = W.make(p, logical=True)
    ref, sab = _run(p, data)
    a = data["a"].double().numpy()
    b = data["b"].double().numpy()
    c = data["c"].double().numpy()
    want = 1.25 * (a @ b) + 0.5 * c
    assert np.all(np.abs(ref - want) <= 2 * K * U53 * (1.25 * sab + np.abs(0.5 * c)) + 1e-300)
    # every major stores the same logical matrices: identical results, bit for bit
    ref_kk, _ = _run(base, W.make(base))
    assert np.array_equal(ref, ref_kk)


def test_padded_leading_dims_and_entries():
    p = W.Problem("pad", 20, 24, 40, "f16", majorA="MN", majorB="K", lda=32, ldb=48,
                  has_c=True, alpha=2.0, beta=1.0, dist="uniform", seed=5)
    data = W.make(p)
    full, fsab = _run(p, data)
    q = p.with_(lda=None, ldb=None)
    packed, _ = _run(q, W.make(q))
    assert np.array_equal(full, packed)
    rows = np.array([0, 19, 7, 3], np.int64)
    cols = np.array([0, 23, 11, 5], np.int64)
    part, psab = _run(p, data, rows, cols)
    assert np.array_equal(part, full[rows, cols])
    assert np.array_equal(psab, fsab[rows, cols])


def test_beta_zero_reads_no_c():
    p = W.Problem("nc", 8, 8, 8, "f16", dist="int2", seed=3)
    data = W.make(p, logical=True)
    ref, _ = _run(p, data)
    assert np.array_equal(ref, (data["a"].double() @ data["b"].double()).numpy())
    with pytest.raises(ValueError):
        O.gemm(8, 8, 8, 1.0, W.bits(data["A"]), 8, 0, W.bits(data["B"]), 8, 0, 1.0, None, 8,
               O.F16)


def test_k_zero_is_beta_c():
    p = W.Problem("k0", 5, 7, 0, "f16", has_c=True, alpha=3.0, beta=0.5, dist="uniform",
                  c_dist="uniform", seed=9)
    data = W.make(p, logical=True)
    ref, sab = _run(p, data)
    assert np.array_equal(ref, 0.5 * data["c"].double().numpy())
    assert np.all(sab == 0)


def test_bound_formula():
    ref = np.array([1.0, 0.0, -3.0])
    s = np.array([10.0, 0.0, 4.0])
    c = np.array([2.0, 1.0, 0.0])
    b = O.bound(O.F16, 1.25, 0.5, ref, s, c)
    want = [2.0**-9 * (12.5 + 1.0) + 2.0**-10, 2.0**-9 * 0.5 + 2.0**-24,
            2.0**-9 * 5.0 + 2.0**-9]
    assert np.allclose(b, want, rtol=0, atol=0)
