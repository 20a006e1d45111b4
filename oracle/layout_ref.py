"""Definitional shape:stride layout semantics (TEST INFRASTRUCTURE ONLY).

Each function restates a definition from the pages in the most literal form available:
a layout is evaluated point by point, composition is function composition point by
point, and the complement is found by search.  Nothing here is fast or clever; the
product's host layout library (C++) computes the same objects symbolically and is
checked against these tables.

Definitions followed:
  * A layout is a pair Shape:Stride mapping a coordinate to sum(coord_i * stride_i).
    "Day 84: CUTLASS and CuTe layouts", section "A layout is a shape and a stride";
    "3.5 CUTLASS II", section 3.5.3.
  * A flat index is unravelled against the shape first mode fastest (colexicographic).
    "Layouts as Algebra", section "The formula gets a name"; "3.5 CUTLASS II", 3.5.4.
  * Shapes and strides are congruent trees.  "Layouts as Algebra", "A shape is a tree".
  * size = number of coordinates; cosize = largest offset + 1.  "3.5 CUTLASS II", 3.5.5.
  * (A o B)(x) = A(B(x)).  "Layouts as Algebra", "Composition, worked by hand".
  * logical_divide(A, B) = A o (B, B*), B* the complement of B: the layout of everything
    B misses.  "Layouts as Algebra", "Divide is tiling"; "Day 84", "A layout is a shape
    and a stride".
"""
import re

# --------------------------------------------------------------------------- parsing


def _parse_tuple(s, i):
    """Parse an integer or a parenthesised tuple starting at s[i]; return (value, next)."""
    if s[i] == "(":
        items = []
        i += 1
        while True:
            v, i = _parse_tuple(s, i)
            items.append(v)
            if s[i] == ",":
                i += 1
                continue
            if s[i] == ")":
                return tuple(items), i + 1
            raise ValueError("bad tuple near %r" % s[i:])
    m = re.match(r"-?\d+", s[i:])
    if not m:
        raise ValueError("expected integer near %r" % s[i:])
    return int(m.group(0)), i + len(m.group(0))


def parse(text):
    """'((2,2),3):((24,2),8)' -> (shape_tree, stride_tree)."""
    s = text.replace(" ", "").replace("_", "")
    shape, i = _parse_tuple(s, 0)
    if s[i] != ":":
        raise ValueError("missing ':' in %r" % text)
    stride, j = _parse_tuple(s, i + 1)
    if j != len(s):
        raise ValueError("trailing text in %r" % text)
    if not congruent(shape, stride):
        raise ValueError("shape and stride are not congruent in %r" % text)
    return shape, stride


def congruent(a, b):
    if isinstance(a, tuple) != isinstance(b, tuple):
        return False
    if isinstance(a, tuple):
        return len(a) == len(b) and all(congruent(x, y) for x, y in zip(a, b))
    return True


def flatten(t):
    if not isinstance(t, tuple):
        return (t,)
    out = ()
    for x in t:
        out += flatten(x)
    return out


def size(shape):
    n = 1
    for s in flatten(shape):
        n *= s
    return n


# --------------------------------------------------------------------------- evaluation


def unravel(shape, x):
    """Flat index -> flat natural coordinate, first mode fastest."""
    coord = []
    for s in flatten(shape):
        coord.append(x % s)
        x //= s
    return coord


def evaluate(layout, x):
    """Offset of flat index x (0 <= x < size)."""
    shape, stride = layout
    if not 0 <= x < size(shape):
        raise IndexError(x)
    return sum(c * d for c, d in zip(unravel(shape, x), flatten(stride)))


def evaluate_coord(layout, coord):
    """Offset of a natural coordinate given as a flat sequence of per-leaf indices."""
    shape, stride = layout
    fs, fd = flatten(shape), flatten(stride)
    if len(coord) != len(fs) or any(not 0 <= c < s for c, s in zip(coord, fs)):
        raise IndexError(coord)
    return sum(c * d for c, d in zip(coord, fd))


def table(layout):
    return [evaluate(layout, x) for x in range(size(layout[0]))]


def cosize(layout):
    return max(table(layout)) + 1


def mode(layout, i):
    """The i-th top-level mode as a layout of its own."""
    shape, stride = layout
    if not isinstance(shape, tuple):
        if i != 0:
            raise IndexError(i)
        return layout
    return shape[i], stride[i]


# --------------------------------------------------------------------------- algebra by definition


def compose_table(a, b):
    """[A(B(x)) for x in domain(B)]: composition read as function composition."""
    return [evaluate(a, evaluate(b, x)) for x in range(size(b[0]))]


def complement_by_search(b, m):
    """Offsets at which translated copies of B's image tile a prefix [0, N), N >= m.

    Definition restated: the complement lists, in increasing order, where the copies of
    "everything B touches" must start so that together with B they cover every offset of
    a contiguous prefix [0, N) exactly once, with N at least the target m.  Found
    greedily: the next start is always the smallest offset not yet covered; the search
    stops at the first point where the target is reached and the covered set has no
    holes.  Returns the list of starts, or None when B's image cannot be tiled this way
    (then no complement exists).
    """
    image = table(b)
    if len(set(image)) != len(image):
        return None
    span = max(image) + 1
    covered = set()
    starts = []
    nxt = 0
    while nxt < m or len(covered) != max(covered) + 1:
        for v in image:
            if nxt + v in covered:
                return None
        for v in image:
            covered.add(nxt + v)
        starts.append(nxt)
        nxt = 0
        while nxt in covered:
            nxt += 1
        if nxt > (m + span) * (span + 1):
            return None
    return starts


def concat_eval(layouts, x):
    """Evaluate the tuple layout (L0, L1, ...) at flat index x (first mode fastest)."""
    total = 0
    for lay in layouts:
        n = size(lay[0])
        total += evaluate(lay, x % n)
        x //= n
    return total


def divide_table(a, b, m=None):
    """Point-by-point table of logical_divide(A, B) = A o (B, B*), in-domain entries only.

    Returns a dict {flat index of (B, B*) : A((B, B*)(x))} for every x whose image lies
    inside A's domain (entries that fall off a ragged edge are left out: those are the
    ones a kernel must predicate away).
    """
    n = size(a[0]) if m is None else m
    starts = complement_by_search(b, n)
    if starts is None:
        raise ValueError("complement does not exist")
    sb = size(b[0])
    out = {}
    for t, st in enumerate(starts):
        for x in range(sb):
            pos = st + evaluate(b, x)
            if pos < size(a[0]):
                out[x + sb * t] = evaluate(a, pos)
    return out


def coalesced_equal(a, b):
    """True when two layouts are the same function on the same domain."""
    return size(a[0]) == size(b[0]) and table(a) == table(b)


def grid(layout):
    """2-D offset grid of a rank-2 layout: rows index mode 0, columns index mode 1."""
    r = mode(layout, 0)
    c = mode(layout, 1)
    rows = []
    for i in range(size(r[0])):
        rows.append([evaluate(r, i) + evaluate(c, j) for j in range(size(c[0]))])
    return rows


def product_table(a, b):
    """logical_product(A, B) point by point: copy j of A starts where the complement of A
    (the offsets its translated copies occupy) puts B(j).  Index i + size(A) * j."""
    sa = size(a[0])
    starts = complement_by_search(a, sa * cosize(b))
    if starts is None:
        raise ValueError("complement does not exist")
    return [evaluate(a, i) + starts[evaluate(b, j)] for j in range(size(b[0])) for i in range(sa)]
