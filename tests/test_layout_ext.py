"""Layout-library extensions: logical_product, the swizzle functor, the print CLI."""
import os
import random
import subprocess
import sys

import pytest

from layout_algebra_gb300 import layout as L
from oracle import layout_ref as R

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rand_layout(rnd, modes):
    shape = [rnd.choice([1, 2, 3, 4]) for _ in range(modes)]
    stride = [rnd.choice([1, 2, 3, 4, 6, 8]) for _ in range(modes)]
    if modes == 1:
        return "%d:%d" % (shape[0], stride[0])
    return "(%s):(%s)" % (",".join(map(str, shape)), ",".join(map(str, stride)))


def test_product_examples():
    # a 2x2 tile repeated 3 times: copies start at 0, 4, 8
    assert L.logical_product("(2,2):(1,2)", "3:1") == "((2,2),3):((1,2),4)"
    # a 4-element run laid out by a 2x3 row-major pattern of copies
    assert L.logical_product("4:1", "(2,3):(3,1)") == "(4,(2,3)):(1,(12,4))"


def test_product_is_the_mirror_of_divide():
    """Dividing the product of a tile by the tile gives back the tile and the pattern."""
    prod = L.logical_product("(2,2):(1,2)", "3:1")
    assert L.coalesce(prod) == "12:1"
    assert L.logical_divide("12:1", "4:1") == "(4,3):(1,4)"


def test_random_products_by_definition():
    rnd = random.Random(5)
    checked = 0
    for _ in range(1500):
        a = _rand_layout(rnd, rnd.randint(1, 2))
        b = _rand_layout(rnd, rnd.randint(1, 2))
        pa, pb = R.parse(a), R.parse(b)
        try:
            want = R.product_table(pa, pb)
        except ValueError:
            continue
        try:
            got = L.logical_product(a, b)
        except L.LayoutError:
            continue
        n = L.size(got)
        assert n == R.size(pa[0]) * R.size(pb[0])
        assert list(L.evaluate(got, list(range(n)))) == want, (a, b, got)
        checked += 1
    assert checked > 200


def _tma_swizzle_model(row, byte_in_row):
    """The 128-byte swizzle the GPU stage-bytes test checks against real copies."""
    return row * 128 + (((byte_in_row // 16) ^ (row % 8)) * 16) + byte_in_row % 16


def test_swizzle_matches_the_copy_engine_model():
    offs = [r * 128 + b for r in range(64) for b in range(128)]
    got = L.swizzle(3, 4, 3, offs)
    want = [_tma_swizzle_model(r, b) for r in range(64) for b in range(128)]
    assert list(got) == want


def test_swizzle_properties():
    x = list(range(4096))
    y = L.swizzle(3, 4, 3, x)
    assert sorted(y) == x                       # a permutation of each 1 KiB atom
    assert list(L.swizzle(3, 4, 3, y)) == x     # an involution
    assert list(L.swizzle(0, 4, 3, x)) == x     # no bits: identity
    assert all(a // 1024 == b // 1024 for a, b in zip(x, y))
    with pytest.raises(L.LayoutError):
        L.swizzle(4, 4, 3, [0])                 # bits above shift are not a swizzle


def test_print_layout_cli():
    r = subprocess.run([sys.executable, "-m", "layout_algebra_gb300.print_layout", "(2,3):(3,1)"],
                       capture_output=True, text=True, cwd=ROOT, timeout=120)
    assert r.returncode == 0, r.stderr
    rows = [line for line in r.stdout.splitlines() if "|" in line]
    assert [[int(v) for v in line.split("|")[1:-1]] for line in rows] == [[0, 1, 2], [3, 4, 5]]


# ------------------------------------------------------------------ local_tile with a projection
# "Layouts as Algebra", "The kernel, in three lines": one block tiler (BM, BN, BK) serves A, B
# and C, each keeping the modes it has; A keeps (BM, BK) and every k-tile, giving the
# (BLK_M, BLK_K, k) shape of the sgemm example.

@pytest.mark.parametrize("M,N,K,BM,BN,BK,m,n", [(512, 384, 256, 128, 64, 32, 2, 3),
                                                 (256, 256, 128, 128, 128, 64, 1, 0)])
def test_projected_tiles_of_a_gemm(M, N, K, BM, BN, BK, m, n):
    tiler = "(%d,%d,%d)" % (BM, BN, BK)
    # A (M,K) row-major, step (1, X, 1), all k-tiles kept
    oa, la = L.local_tile_proj("(%d,%d):(%d,1)" % (M, K, K), tiler, [m, n, None], [1, 0, 1])
    assert R.parse(la)[0] == (BM, BK, K // BK)
    for i in range(0, BM, 7):
        for k in range(0, BK, 5):
            for kt in range(K // BK):
                assert oa + R.evaluate_coord(R.parse(la), [i, k, kt]) == (m * BM + i) * K + kt * BK + k
    # B (N,K) K-major, step (X, 1, 1)
    ob, lb = L.local_tile_proj("(%d,%d):(%d,1)" % (N, K, K), tiler, [m, n, None], [0, 1, 1])
    assert R.parse(lb)[0] == (BN, BK, K // BK)
    for j in range(0, BN, 3):
        for kt in range(K // BK):
            assert ob + R.evaluate_coord(R.parse(lb), [j, 1, kt]) == (n * BN + j) * K + kt * BK + 1
    # C (M,N) row-major, step (1, 1, X): one tile, no trailing mode
    oc, lc = L.local_tile_proj("(%d,%d):(%d,1)" % (M, N, N), tiler, [m, n, None], [1, 1, 0])
    assert R.parse(lc)[0] == (BM, BN)
    for i in range(0, BM, 11):
        for j in range(0, BN, 13):
            assert oc + R.evaluate_coord(R.parse(lc), [i, j]) == (m * BM + i) * N + n * BN + j


def test_projection_matches_plain_local_tile():
    # with every mode kept and every coordinate fixed it is local_tile itself
    for coord in ([0, 0], [3, 1], [1, 2]):
        o1, l1 = L.local_tile("(64,48):(1,64)", "(16,16)", coord)
        o2, l2 = L.local_tile_proj("(64,48):(1,64)", "(16,16)", coord, [1, 1])
        assert (o1, R.table(R.parse(l1))) == (o2, R.table(R.parse(l2)))


def test_projection_errors():
    with pytest.raises(L.LayoutError):    # keeps three modes of a rank-2 layout
        L.local_tile_proj("(64,48):(48,1)", "(16,16,8)", [0, 0, 0], [1, 1, 1])
    with pytest.raises(L.LayoutError):    # coordinate beyond the grid
        L.local_tile_proj("(64,48):(48,1)", "(16,16,8)", [4, 0, None], [1, 0, 1])
