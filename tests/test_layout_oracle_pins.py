"""Pins for the definitional layout oracle against values the pages print."""
import json
import os

import pytest

from oracle import layout_ref as R

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "layout_pages.json")))


@pytest.mark.parametrize("case", GOLDEN["eval_points"], ids=lambda c: c["id"])
def test_eval_points(case):
    lay = R.parse(case["layout"])
    if "coord" in case:
        assert R.evaluate_coord(lay, case["coord"]) == case["offset"]
    for coord, off in case.get("points", []):
        assert R.evaluate_coord(lay, coord) == off
    for x, off in case.get("flat", []):
        assert R.evaluate(lay, x) == off
    if "size" in case:
        assert R.size(lay[0]) == case["size"]
        assert R.cosize(lay) == case["cosize"]


@pytest.mark.parametrize("case", GOLDEN["tables"], ids=lambda c: c["id"])
def test_tables(case):
    assert R.table(R.parse(case["layout"])) == case["values"]


@pytest.mark.parametrize("case", GOLDEN["unravel"], ids=lambda c: str(c["index"]))
def test_unravel(case):
    assert R.unravel(tuple(case["shape"]), case["index"]) == case["coord"]


def test_composition_by_definition():
    (c,) = GOLDEN["composition"]
    a, b, r = R.parse(c["a"]), R.parse(c["b"]), R.parse(c["out"])
    by_def = R.compose_table(a, b)
    assert by_def == [0, 24, 2, 26, 8, 32, 10, 34, 16, 40, 18, 42]
    assert R.table(r) == by_def


@pytest.mark.parametrize("case", GOLDEN["complement"], ids=lambda c: c["out"])
def test_complement_by_search(case):
    starts = R.complement_by_search(R.parse(case["b"]), case["m"])
    assert starts == R.table(R.parse(case["out"]))


def test_complement_search_strided():
    # 4:2 touches even offsets; copies start at 0, 1 then 8, 9: (2,2):(1,8)
    assert R.complement_by_search(R.parse("4:2"), 16) == [0, 1, 8, 9]


@pytest.mark.parametrize("case", GOLDEN["zipped_divide"], ids=lambda c: c["a"])
def test_divide_gate_two_sided(case):
    """The pages' two-sided gate: the divided layout versus the hand-written tile address."""
    a = R.parse(case["a"])
    z = R.parse(case["out"])
    tile_shape = R.mode(z, 0)[0]
    grid_shape = R.mode(z, 1)[0]
    (tr, tc), (gr, gc) = tile_shape, grid_shape
    rows, cols = a[0]
    for r in range(rows):
        for c in range(cols):
            coord = [r % tr, c % tc, r // tr, c // tc]
            assert R.evaluate_coord(z, coord) == R.evaluate_coord(a, [r, c])


def test_day16_index_gate():
    """(256,128):(128,1) zipped by 16x16 against the page's day16Index expression."""
    z = R.parse("((16,16),(16,8)):((128,1),(2048,16))")
    kK, kTile = 128, 16
    n = 0
    for tile_row in range(16):
        for tile_col in range(8):
            for rit in range(16):
                for cit in range(16):
                    row = tile_row * kTile + rit
                    col = tile_col * kTile + cit
                    assert R.evaluate_coord(z, [rit, cit, tile_row, tile_col]) == row * kK + col
                    n += 1
    assert n == 32768
    # element (37, 44): tile (2, 2), in-tile (5, 12) -> 4780
    assert R.evaluate_coord(z, [5, 12, 2, 2]) == 4780


def test_tiled_panel_discrepancy():
    t = GOLDEN["tiled_panel"]
    lab = R.parse(t["labelled"])
    assert R.table(lab) == list(range(16))
    assert R.coalesced_equal(lab, R.parse("16:1"))
    # as a 2-D layout with modes ((2,2),(2,2)) it equals column-major (4,4):(1,4)
    assert R.grid(lab) == R.grid(R.parse(t["labelled_equals"]))
    assert R.grid(R.parse(t["printed_square_layout"])) == t["printed_square"]


@pytest.mark.parametrize("case", GOLDEN["sizes"], ids=lambda c: c["layout"])
def test_sizes(case):
    lay = R.parse(case["layout"])
    assert R.size(lay[0]) == case["size"]
    assert R.cosize(lay) == case["cosize"]


@pytest.mark.parametrize("case", GOLDEN["tv_layouts"], ids=lambda c: c["layout"])
def test_tv_layouts(case):
    lay = R.parse(case["layout"])
    t = case["thread"]
    assert [R.evaluate_coord(lay, [t, v]) for v in range(4)] == case["values"]
    assert [R.evaluate_coord(lay, [th, 0]) for th in range(8)] == case["step0"]


def test_logical_divide_by_definition():
    d = R.divide_table(R.parse("8:1"), R.parse("4:1"))
    assert [d[x] for x in range(8)] == R.table(R.parse("(4,2):(1,4)"))


def test_ragged_divide_drops_off_edge():
    d = R.divide_table(R.parse("10:1"), R.parse("4:1"))
    assert sorted(d) == list(range(10))     # 3 tiles of 4, the last two entries off the edge


def test_product_table_pins():
    # a compact tile repeated by a contiguous pattern fills 0..n-1 in order
    assert R.product_table(R.parse("4:1"), R.parse("3:1")) == list(range(12))
    assert R.product_table(R.parse("(2,2):(1,2)"), R.parse("3:1")) == list(range(12))
    # worked by hand: 2:2 touches {0,2}; its copies start at 0 and 1 -> 0,2,1,3
    assert R.product_table(R.parse("2:2"), R.parse("2:1")) == [0, 2, 1, 3]
    # a strided pattern of copies: copy j of 2:1 sits at 2*B(j), B = 2:2 -> 0,1,4,5
    assert R.product_table(R.parse("2:1"), R.parse("2:2")) == [0, 1, 4, 5]
