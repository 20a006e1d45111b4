"""Python face of the host layout library (text in the pages' Shape:Stride notation).

Every function marshals strings and integers to the C ABI in include/layout_algebra.h
and returns its result; the algebra itself runs in the native library.
"""
import ctypes

import numpy as np

from ._native import lib

_CAP = 1 << 16


class LayoutError(ValueError):
    def __init__(self, code, what):
        self.code = code
        super().__init__("%s: %s" % (what, lib().la_error_string(code).decode()))


def _b(s):
    return s.encode() if isinstance(s, str) else s


def _text(fn, *args, cap=_CAP):
    buf = ctypes.create_string_buffer(cap)
    rc = fn(*args, buf, cap)
    if rc != 0:
        raise LayoutError(rc, fn.__name__)
    return buf.value.decode()


def size(layout):
    out = ctypes.c_int64()
    rc = lib().la_size(_b(layout), ctypes.byref(out))
    if rc:
        raise LayoutError(rc, "la_size")
    return out.value


def cosize(layout):
    out = ctypes.c_int64()
    rc = lib().la_cosize(_b(layout), ctypes.byref(out))
    if rc:
        raise LayoutError(rc, "la_cosize")
    return out.value


def evaluate(layout, idx):
    """Offsets of flat (colexicographic) indices; idx is an int or a sequence."""
    scalar = np.isscalar(idx)
    a = np.ascontiguousarray(np.atleast_1d(np.asarray(idx, dtype=np.int64)))
    out = np.empty_like(a)
    rc = lib().la_eval(_b(layout), a.ctypes.data, a.size, out.ctypes.data)
    if rc:
        raise LayoutError(rc, "la_eval")
    return int(out[0]) if scalar else out


def evaluate_coord(layout, coord):
    c = np.ascontiguousarray(np.asarray(coord, dtype=np.int64))
    out = ctypes.c_int64()
    rc = lib().la_eval_coord(_b(layout), c.ctypes.data, c.size, ctypes.byref(out))
    if rc:
        raise LayoutError(rc, "la_eval_coord")
    return out.value


def coalesce(layout):
    return _text(lib().la_coalesce, _b(layout))


def composition(a, b):
    return _text(lib().la_composition, _b(a), _b(b))


def complement(layout, cotarget):
    return _text(lib().la_complement, _b(layout), int(cotarget))


def logical_divide(layout, tiler):
    return _text(lib().la_logical_divide, _b(layout), _b(tiler))


def zipped_divide(layout, tiler):
    return _text(lib().la_zipped_divide, _b(layout), _b(tiler))


def local_tile(layout, tiler, grid_coord):
    g = np.ascontiguousarray(np.asarray(grid_coord, dtype=np.int64))
    origin = ctypes.c_int64()
    s = _text(lib().la_local_tile, _b(layout), _b(tiler), g.ctypes.data, g.size,
              ctypes.byref(origin))
    return origin.value, s


def local_tile_proj(layout, tiler, grid_coord, step):
    """local_tile with a projection step: grid_coord entries of None keep that grid mode
    (every tile along it) as a trailing mode; step entries of 0 (or None) drop a tiler mode.
    Returns (origin, layout)."""
    n = len(step)
    g = np.ascontiguousarray([-1 if c is None else int(c) for c in grid_coord], dtype=np.int64)
    st = np.ascontiguousarray([0 if x in (None, 0) else 1 for x in step], dtype=np.int32)
    if g.size != n:
        raise ValueError("grid_coord and step must have the same length")
    origin = ctypes.c_int64()
    s = _text(lib().la_local_tile_proj, _b(layout), _b(tiler), g.ctypes.data, st.ctypes.data, n,
              ctypes.byref(origin))
    return origin.value, s


def local_partition(layout, thr, tid):
    origin = ctypes.c_int64()
    s = _text(lib().la_local_partition, _b(layout), _b(thr), int(tid), ctypes.byref(origin))
    return origin.value, s


def print_layout(layout):
    return _text(lib().la_print_layout, _b(layout))


def logical_product(a, b):
    return _text(lib().la_logical_product, _b(a), _b(b))


def swizzle(bits, base, shift, offsets):
    """Sw<bits,base,shift> applied to an int or a sequence of offsets."""
    scalar = np.isscalar(offsets)
    x = np.ascontiguousarray(np.atleast_1d(np.asarray(offsets, dtype=np.int64)))
    out = np.empty_like(x)
    rc = lib().la_swizzle(int(bits), int(base), int(shift), x.ctypes.data, x.size, out.ctypes.data)
    if rc:
        raise LayoutError(rc, "la_swizzle")
    return int(out[0]) if scalar else out

