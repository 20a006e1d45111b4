"""Host layout library (C ABI) against the pages' worked examples and the definitional oracle."""
import json
import os
import random

import pytest

from layout_algebra_gb300 import layout as L
from oracle import layout_ref as R

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "layout_pages.json")))


def same_function(a_text, b_text):
    a, b = R.parse(a_text), R.parse(b_text)
    return R.size(a[0]) == R.size(b[0]) and R.table(a) == R.table(b)


@pytest.mark.parametrize("case", GOLDEN["eval_points"], ids=lambda c: c["id"])
def test_eval_points(case):
    if "coord" in case:
        assert L.evaluate_coord(case["layout"], case["coord"]) == case["offset"]
    for coord, off in case.get("points", []):
        assert L.evaluate_coord(case["layout"], coord) == off
    for x, off in case.get("flat", []):
        assert L.evaluate(case["layout"], x) == off
    if "size" in case:
        assert L.size(case["layout"]) == case["size"]
        assert L.cosize(case["layout"]) == case["cosize"]


@pytest.mark.parametrize("case", GOLDEN["tables"], ids=lambda c: c["id"])
def test_tables(case):
    n = L.size(case["layout"])
    assert list(L.evaluate(case["layout"], list(range(n)))) == case["values"]


@pytest.mark.parametrize("case", GOLDEN["coalesce"], ids=lambda c: c["in"])
def test_coalesce(case):
    out = L.coalesce(case["in"])
    assert out == case["out"]
    assert same_function(out, case["in"])


def test_composition_page_example():
    (c,) = GOLDEN["composition"]
    out = L.composition(c["a"], c["b"])
    assert out == c["out"]
    a, b = R.parse(c["a"]), R.parse(c["b"])
    assert R.table(R.parse(out)) == R.compose_table(a, b)


@pytest.mark.parametrize("case", GOLDEN["complement"], ids=lambda c: c["out"])
def test_complement(case):
    out = L.complement(case["b"], case["m"])
    assert out == case["out"]
    assert R.table(R.parse(out)) == R.complement_by_search(R.parse(case["b"]), case["m"])


@pytest.mark.parametrize("case", GOLDEN["logical_divide"], ids=lambda c: c["a"] + "/" + c["tiler"])
def test_logical_divide(case):
    assert L.logical_divide(case["a"], case["tiler"]) == case["out"]


@pytest.mark.parametrize("case", GOLDEN["zipped_divide"], ids=lambda c: c["a"] + "/" + c["tiler"])
def test_zipped_divide(case):
    assert L.zipped_divide(case["a"], case["tiler"]) == case["out"]


def test_two_sided_gate_32768():
    """Every element of (256,128):(128,1) through zipped_divide vs the hand-written address."""
    z = L.zipped_divide("(256,128):(128,1)", "(16,16)")
    n = 0
    for r in range(256):
        for c in range(128):
            got = L.evaluate_coord(z, [r % 16, c % 16, r // 16, c // 16])
            assert got == (r // 16 * 16 + r % 16) * 128 + (c // 16 * 16 + c % 16)
            n += 1
    assert n == 32768


def test_divide_identity_256():
    """Mode 0 at tile (0,0) and at tile (9,5) is the 16x16 sub-block of the matrix."""
    mA = "(256,128):(128,1)"
    for tile in ([0, 0], [9, 5]):
        origin, t = L.local_tile(mA, "(16,16)", tile)
        assert t == "(16,16):(128,1)"
        for i in range(16):
            for j in range(16):
                r, c = tile[0] * 16 + i, tile[1] * 16 + j
                assert origin + L.evaluate_coord(t, [i, j]) == L.evaluate_coord(mA, [r, c])


def test_tiled_panel_discrepancy():
    t = GOLDEN["tiled_panel"]
    assert L.coalesce(t["labelled"]) == "16:1"
    assert same_function(t["labelled"], t["labelled_equals"].replace("(4,4):(1,4)", "16:1"))
    grid_text = L.print_layout(t["printed_square_layout"])
    rows = [line for line in grid_text.splitlines() if "|" in line]
    parsed = [[int(x) for x in line.split("|")[1:-1]] for line in rows]
    assert parsed == t["printed_square"]


@pytest.mark.parametrize("case", GOLDEN["sizes"], ids=lambda c: c["layout"])
def test_sizes(case):
    assert L.size(case["layout"]) == case["size"]
    assert L.cosize(case["layout"]) == case["cosize"]


def test_local_tile_sgemm_shapes():
    # gA (BLK_M, BLK_K, k): (M,K):(K,1) tiled by (128,32) keeps 128x32 tiles with K/32 of them
    M, K = 512, 256
    z = L.zipped_divide("(%d,%d):(%d,1)" % (M, K, K), "(128,32)")
    assert z == "((128,32),(4,8)):((%d,1),(%d,32))" % (K, 128 * K)
    origin, t = L.local_tile("(%d,%d):(%d,1)" % (M, K, K), "(128,32)", [2, 3])
    assert t == "(128,32):(%d,1)" % K and origin == 2 * 128 * K + 3 * 32


def test_local_partition_thread_layouts():
    for thr in ("(8,4):(1,8)", "(8,4):(4,1)"):
        seen = set()
        for tid in range(32):
            origin, rest = L.local_partition("(16,16):(16,1)", thr, tid)
            n = L.size(rest)
            offs = [origin + int(v) for v in L.evaluate(rest, list(range(n)))]
            assert len(offs) == 8
            seen.update(offs)
        assert seen == set(range(256))     # the 32 threads cover the tile exactly once


def test_errors():
    with pytest.raises(L.LayoutError):
        L.composition("(6,2):(8,2)", "5:4")       # stride 4 does not divide 6
    with pytest.raises(L.LayoutError):
        L.complement("(2,2):(1,1)", 8)            # overlapping modes
    with pytest.raises(L.LayoutError):
        L.size("(2,3):(1)")                       # incongruent
    with pytest.raises(L.LayoutError):
        L.evaluate("4:1", 4)                      # out of range


def _random_layout(rnd, max_modes=3):
    n = rnd.randint(1, max_modes)
    shape = [rnd.choice([1, 2, 3, 4, 6, 8]) for _ in range(n)]
    stride = [rnd.choice([0, 1, 2, 3, 4, 8, 12, 16]) for _ in range(n)]
    if n == 1:
        return "%d:%d" % (shape[0], stride[0])
    return "(%s):(%s)" % (",".join(map(str, shape)), ",".join(map(str, stride)))


def test_random_coalesce_preserves_function():
    rnd = random.Random(1)
    for _ in range(400):
        a = _random_layout(rnd, 4)
        assert same_function(L.coalesce(a), a) or L.size(a) == 1


def test_random_composition_by_definition():
    """Wherever the library returns A o B, it equals A(B(x)) point by point."""
    rnd = random.Random(2)
    checked = 0
    for _ in range(3000):
        a = _random_layout(rnd, 3)
        b = _random_layout(rnd, 2)
        pa, pb = R.parse(a), R.parse(b)
        if max(R.table(pb)) >= R.size(pa[0]):
            continue
        try:
            r = L.composition(a, b)
        except L.LayoutError:
            continue
        assert L.size(r) == L.size(b)
        assert R.table(R.parse(r)) == R.compose_table(pa, pb), (a, b, r)
        checked += 1
    assert checked > 300


def test_random_complement_by_search():
    rnd = random.Random(3)
    checked = 0
    for _ in range(1500):
        b = _random_layout(rnd, 2)
        pb = R.parse(b)
        if len(set(R.table(pb))) != R.size(pb[0]):
            continue
        m = rnd.choice([8, 16, 24, 48, 64])
        starts = R.complement_by_search(pb, m)
        try:
            c = L.complement(b, m)
        except L.LayoutError:
            assert starts is None or R.size(pb[0]) == 1
            continue
        if starts is None:
            continue
        assert R.table(R.parse(c)) == starts, (b, m, c)
        checked += 1
    assert checked > 100


def test_random_logical_divide_by_definition():
    rnd = random.Random(4)
    for _ in range(200):
        n = rnd.choice([8, 12, 16, 24, 32, 10, 20])
        d = rnd.choice([1, 2, 3])
        t = rnd.choice([2, 4])
        a = "%d:%d" % (n, d)
        out = L.logical_divide(a, "%d:1" % t)
        want = R.divide_table(R.parse(a), R.parse("%d:1" % t))
        lay = R.parse(out)
        for x, v in want.items():
            assert R.evaluate(lay, x) == v
