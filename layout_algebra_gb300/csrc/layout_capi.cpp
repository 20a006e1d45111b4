// C ABI over the host layout library: text in, text out, status codes (layout_algebra.h).
#include <cstring>
#include <string>

#include "../../include/layout_algebra.h"
#include "layout.hpp"

namespace {

int put(const std::string& s, char* out, size_t cap) {
  if (!out || cap == 0) return LA_ERR_ARG;
  if (s.size() + 1 > cap) {
    out[0] = '\0';
    return LA_ERR_BUFFER;
  }
  std::memcpy(out, s.c_str(), s.size() + 1);
  return LA_OK;
}

template <class F>
int guarded(F&& f) {
  try {
    return f();
  } catch (const la::Error& e) {
    return static_cast<int>(e.code);
  } catch (const std::bad_alloc&) {
    return LA_ERR_RANGE;
  } catch (...) {
    return LA_ERR_ARG;
  }
}

}  // namespace

extern "C" {

const char* la_error_string(int code) {
  switch (code) {
    case LA_OK: return "ok";
    case LA_ERR_PARSE: return "parse error";
    case LA_ERR_INCONGRUENT: return "shape and stride are not congruent";
    case LA_ERR_NOT_COMPOSABLE: return "composition is not defined for these layouts";
    case LA_ERR_NO_COMPLEMENT: return "no complement exists";
    case LA_ERR_RANGE: return "out of range";
    case LA_ERR_BUFFER: return "output buffer too small";
    case LA_ERR_ARG: return "invalid argument";
    default: return "unknown error";
  }
}

int la_size(const char* layout, int64_t* size) {
  if (!layout || !size) return LA_ERR_ARG;
  return guarded([&] {
    *size = la::size(la::parse_layout(layout));
    return LA_OK;
  });
}

int la_cosize(const char* layout, int64_t* cosize) {
  if (!layout || !cosize) return LA_ERR_ARG;
  return guarded([&] {
    *cosize = la::cosize(la::parse_layout(layout));
    return LA_OK;
  });
}

int la_eval(const char* layout, const int64_t* idx, int64_t n, int64_t* offsets) {
  if (!layout || n < 0 || (n > 0 && (!idx || !offsets))) return LA_ERR_ARG;
  return guarded([&] {
    la::Layout l = la::parse_layout(layout);
    for (int64_t i = 0; i < n; ++i) offsets[i] = la::eval(l, idx[i]);
    return LA_OK;
  });
}

int la_eval_coord(const char* layout, const int64_t* coord, int ncoord, int64_t* offset) {
  if (!layout || !offset || ncoord < 0 || (ncoord > 0 && !coord)) return LA_ERR_ARG;
  return guarded([&] {
    std::vector<int64_t> c(coord, coord + ncoord);
    *offset = la::eval_coord(la::parse_layout(layout), c);
    return LA_OK;
  });
}

int la_coalesce(const char* layout, char* out, size_t cap) {
  if (!layout) return LA_ERR_ARG;
  return guarded([&] { return put(la::to_string(la::coalesce(la::parse_layout(layout))), out, cap); });
}

int la_composition(const char* a, const char* b, char* out, size_t cap) {
  if (!a || !b) return LA_ERR_ARG;
  return guarded([&] {
    return put(la::to_string(la::composition(la::parse_layout(a), la::parse_layout(b))), out, cap);
  });
}

int la_complement(const char* layout, int64_t cotarget, char* out, size_t cap) {
  if (!layout) return LA_ERR_ARG;
  return guarded([&] {
    return put(la::to_string(la::complement(la::parse_layout(layout), cotarget)), out, cap);
  });
}

int la_logical_divide(const char* layout, const char* tiler, char* out, size_t cap) {
  if (!layout || !tiler) return LA_ERR_ARG;
  return guarded([&] {
    return put(la::to_string(la::logical_divide(la::parse_layout(layout), la::parse_tiler(tiler))),
               out, cap);
  });
}

int la_zipped_divide(const char* layout, const char* tiler, char* out, size_t cap) {
  if (!layout || !tiler) return LA_ERR_ARG;
  return guarded([&] {
    return put(la::to_string(la::zipped_divide(la::parse_layout(layout), la::parse_tiler(tiler))),
               out, cap);
  });
}

int la_local_tile(const char* layout, const char* tiler, const int64_t* grid, int ngrid,
                  int64_t* origin, char* out, size_t cap) {
  if (!layout || !tiler || !origin || ngrid < 0 || (ngrid > 0 && !grid)) return LA_ERR_ARG;
  return guarded([&] {
    std::vector<int64_t> g(grid, grid + ngrid);
    la::Layout t = la::local_tile(la::parse_layout(layout), la::parse_tiler(tiler), g, origin);
    return put(la::to_string(t), out, cap);
  });
}

int la_local_tile_proj(const char* layout, const char* tiler, const int64_t* grid, const int* step, int n,
                       int64_t* origin, char* out, size_t cap) {
  if (!layout || !tiler || !origin || n <= 0 || !grid || !step) return LA_ERR_ARG;
  return guarded([&] {
    std::vector<int64_t> g(grid, grid + n);
    std::vector<int> st(step, step + n);
    la::Layout t = la::local_tile_proj(la::parse_layout(layout), la::parse_tiler(tiler), g, st, origin);
    return put(la::to_string(t), out, cap);
  });
}

int la_local_partition(const char* layout, const char* thr, int64_t tid, int64_t* origin,
                       char* out, size_t cap) {
  if (!layout || !thr || !origin) return LA_ERR_ARG;
  return guarded([&] {
    la::Layout r = la::local_partition(la::parse_layout(layout), la::parse_layout(thr), tid, origin);
    return put(la::to_string(r), out, cap);
  });
}

int la_logical_product(const char* a, const char* b, char* out, size_t cap) {
  if (!a || !b) return LA_ERR_ARG;
  return guarded([&] {
    return put(la::to_string(la::logical_product(la::parse_layout(a), la::parse_layout(b))), out, cap);
  });
}

int la_swizzle(int bits, int base, int shift, const int64_t* in, int64_t n, int64_t* out) {
  if (n < 0 || (n > 0 && (!in || !out))) return LA_ERR_ARG;
  return guarded([&] {
    for (int64_t i = 0; i < n; ++i) out[i] = la::swizzle(bits, base, shift, in[i]);
    return LA_OK;
  });
}

int la_print_layout(const char* layout, char* out, size_t cap) {
  if (!layout) return LA_ERR_ARG;
  return guarded([&] { return put(la::print_layout(la::parse_layout(layout)), out, cap); });
}

}  // extern "C"
