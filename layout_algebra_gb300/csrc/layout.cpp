// Host-side shape:stride layout algebra (see layout.hpp for the definitions followed).
#include "layout.hpp"

#include <algorithm>
#include <cctype>
#include <limits>
#include <sstream>

namespace la {

namespace {

constexpr int64_t kUnbounded = std::numeric_limits<int64_t>::max();

using Mode = std::pair<int64_t, int64_t>;   // (extent, stride)

void flatten_into(const IntTuple& t, std::vector<int64_t>& out) {
  if (t.leaf) {
    out.push_back(t.value);
    return;
  }
  for (const auto& k : t.kids) flatten_into(k, out);
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

int64_t checked_mul(int64_t a, int64_t b) {
  int64_t r;
  if (__builtin_mul_overflow(a, b, &r)) throw Error(LA_ERR_RANGE, "integer overflow");
  return r;
}

// A flat list of modes as a layout: a leaf when there is exactly one mode, a tuple
// otherwise (an empty list is the size-1 layout 1:0).
Layout from_modes(const std::vector<Mode>& m) {
  if (m.empty()) return leaf_layout(1, 0);
  if (m.size() == 1) return leaf_layout(m[0].first, m[0].second);
  std::vector<Layout> ls;
  for (const auto& x : m) ls.push_back(leaf_layout(x.first, x.second));
  return tuple_layout(ls);
}

// A o (s:d), A given as coalesced flat modes.
//  Step 1 divides the stride d out of A's modes: a mode wholly covered by d is skipped,
//  a mode that d divides keeps every d-th element.  Step 2 keeps the first s elements
//  of what is left.  A's last mode is read as unbounded, so the walk may run past
//  size(A) (that is what a ragged tile grid needs).
//  `maxdig[j]` receives the largest coordinate the walk reaches in A's mode j (all but
//  the last mode), which the caller uses to check that B's modes do not interfere.
std::vector<Mode> compose_leaf(const std::vector<Mode>& a, int64_t s, int64_t d,
                               std::vector<int64_t>* maxdig) {
  if (maxdig) maxdig->assign(a.empty() ? 0 : a.size() - 1, 0);
  if (s == 1) return {};
  if (d == 0) return {{s, 0}};
  struct Part {
    int64_t extent, stride;
    size_t mode;
    int64_t step;   // distance in mode `mode`'s coordinate between consecutive elements
  };
  std::vector<Part> divided;
  int64_t rest = d;
  for (size_t i = 0; i < a.size(); ++i) {
    int64_t si = a[i].first, di = a[i].second;
    if (i + 1 == a.size()) {
      divided.push_back({kUnbounded, checked_mul(di, rest), i, rest});
      break;
    }
    if (rest == 1) {
      divided.push_back({si, di, i, 1});
    } else if (rest % si == 0) {
      rest /= si;
    } else if (si % rest == 0) {
      divided.push_back({si / rest, checked_mul(di, rest), i, rest});
      rest = 1;
    } else {
      throw Error(LA_ERR_NOT_COMPOSABLE, "stride divisibility condition fails");
    }
  }
  std::vector<Mode> out;
  int64_t rem = s;
  for (const auto& m : divided) {
    if (rem == 1) break;
    int64_t take;
    if (m.extent == kUnbounded) {
      take = rem;
    } else if (m.extent == 1) {
      continue;
    } else if (rem <= m.extent) {
      take = rem;
    } else {
      if (rem % m.extent != 0) throw Error(LA_ERR_NOT_COMPOSABLE, "shape divisibility condition fails");
      take = m.extent;
    }
    out.push_back({take, m.stride});
    if (maxdig && m.mode < maxdig->size()) (*maxdig)[m.mode] = m.step * (take - 1);
    rem /= take;
  }
  return out;
}

// Composition keeps B's nesting: every leaf s:d of B becomes A o (s:d).  The pieces add
// up to A(B(x)) only if no combination of B's coordinates makes A's coordinates carry
// from one mode into the next; the per-mode maxima are summed here and checked.
Layout compose_tree(const std::vector<Mode>& a, const IntTuple& bs, const IntTuple& bd,
                    std::vector<int64_t>& used) {
  if (bs.leaf) {
    std::vector<int64_t> mx;
    Layout r = from_modes(compose_leaf(a, bs.value, bd.value, &mx));
    for (size_t j = 0; j < mx.size(); ++j) {
      used[j] += mx[j];
      if (used[j] >= a[j].first)
        throw Error(LA_ERR_NOT_COMPOSABLE, "modes of B interfere inside A");
    }
    return r;
  }
  std::vector<Layout> parts;
  for (size_t i = 0; i < bs.kids.size(); ++i) parts.push_back(compose_tree(a, bs.kids[i], bd.kids[i], used));
  return tuple_layout(parts);
}

// ------------------------------------------------------------------------ parsing
struct Parser {
  std::string s;
  size_t i = 0;
  explicit Parser(const std::string& text) {
    for (char c : text)
      if (!std::isspace(static_cast<unsigned char>(c)) && c != '_') s.push_back(c);
  }
  bool done() const { return i >= s.size(); }
  char peek() const { return done() ? '\0' : s[i]; }
  void expect(char c) {
    if (peek() != c) throw Error(LA_ERR_PARSE, std::string("expected '") + c + "' in " + s);
    ++i;
  }
  IntTuple tuple() {
    if (peek() == '(') {
      ++i;
      std::vector<IntTuple> kids;
      for (;;) {
        kids.push_back(tuple());
        if (peek() == ',') {
          ++i;
          continue;
        }
        expect(')');
        break;
      }
      return IntTuple::Tup(std::move(kids));
    }
    size_t j = i;
    if (peek() == '-') ++i;
    while (!done() && std::isdigit(static_cast<unsigned char>(s[i]))) ++i;
    if (j == i || (s[j] == '-' && i == j + 1)) throw Error(LA_ERR_PARSE, "expected integer in " + s);
    try {
      return IntTuple::Int(std::stoll(s.substr(j, i - j)));
    } catch (const std::out_of_range&) {
      throw Error(LA_ERR_RANGE, "integer out of range in " + s);
    }
  }
  Layout layout() {
    Layout l;
    l.shape = tuple();
    expect(':');
    l.stride = tuple();
    if (!congruent(l.shape, l.stride)) throw Error(LA_ERR_INCONGRUENT, "shape and stride differ in " + s);
    for (int64_t e : flatten(l.shape))
      if (e <= 0) throw Error(LA_ERR_ARG, "extents must be positive in " + s);
    return l;
  }
};

// Split "a,b,c" at top-level commas.
std::vector<std::string> split_top(const std::string& s) {
  std::vector<std::string> out;
  int depth = 0;
  std::string cur;
  for (char c : s) {
    if (c == '(') ++depth;
    if (c == ')') --depth;
    if (c == ',' && depth == 0) {
      out.push_back(cur);
      cur.clear();
    } else {
      cur.push_back(c);
    }
  }
  out.push_back(cur);
  return out;
}

}  // namespace

// ------------------------------------------------------------------------ IntTuple
IntTuple IntTuple::Int(int64_t v) {
  IntTuple t;
  t.leaf = true;
  t.value = v;
  return t;
}

IntTuple IntTuple::Tup(std::vector<IntTuple> k) {
  IntTuple t;
  t.leaf = false;
  t.kids = std::move(k);
  return t;
}

const IntTuple& IntTuple::mode(int i) const {
  if (leaf) {
    if (i != 0) throw Error(LA_ERR_RANGE, "mode index out of range");
    return *this;
  }
  if (i < 0 || i >= static_cast<int>(kids.size())) throw Error(LA_ERR_RANGE, "mode index out of range");
  return kids[i];
}

Layout Layout::mode(int i) const { return Layout{shape.mode(i), stride.mode(i)}; }

// ------------------------------------------------------------------------ construction
Layout make_layout(const std::vector<int64_t>& shape, const std::vector<int64_t>& stride) {
  if (shape.size() != stride.size() || shape.empty()) throw Error(LA_ERR_INCONGRUENT, "make_layout");
  if (shape.size() == 1) return leaf_layout(shape[0], stride[0]);
  std::vector<Layout> m;
  for (size_t i = 0; i < shape.size(); ++i) m.push_back(leaf_layout(shape[i], stride[i]));
  return tuple_layout(m);
}

Layout leaf_layout(int64_t s, int64_t d) {
  if (s <= 0) throw Error(LA_ERR_ARG, "extents must be positive");
  return Layout{IntTuple::Int(s), IntTuple::Int(d)};
}

Layout tuple_layout(const std::vector<Layout>& modes) {
  std::vector<IntTuple> s, d;
  for (const auto& m : modes) {
    s.push_back(m.shape);
    d.push_back(m.stride);
  }
  return Layout{IntTuple::Tup(std::move(s)), IntTuple::Tup(std::move(d))};
}

Tiler tiler_of(const std::vector<int64_t>& tile_extents) {
  Tiler t;
  for (int64_t e : tile_extents) t.modes.push_back(leaf_layout(e, 1));
  return t;
}

// ------------------------------------------------------------------------ queries
bool congruent(const IntTuple& a, const IntTuple& b) {
  if (a.leaf != b.leaf) return false;
  if (a.leaf) return true;
  if (a.kids.size() != b.kids.size()) return false;
  for (size_t i = 0; i < a.kids.size(); ++i)
    if (!congruent(a.kids[i], b.kids[i])) return false;
  return true;
}

std::vector<int64_t> flatten(const IntTuple& t) {
  std::vector<int64_t> out;
  flatten_into(t, out);
  return out;
}

int64_t size(const IntTuple& shape) {
  int64_t n = 1;
  for (int64_t s : flatten(shape)) n = checked_mul(n, s);
  return n;
}

int64_t size(const Layout& l) { return size(l.shape); }

std::vector<int64_t> unravel(const IntTuple& shape, int64_t idx) {
  std::vector<int64_t> c;
  for (int64_t s : flatten(shape)) {
    c.push_back(idx % s);
    idx /= s;
  }
  return c;
}

int64_t eval_coord(const Layout& l, const std::vector<int64_t>& coord) {
  auto s = flatten(l.shape);
  auto d = flatten(l.stride);
  if (coord.size() != s.size()) throw Error(LA_ERR_ARG, "coordinate rank mismatch");
  int64_t off = 0;
  for (size_t i = 0; i < s.size(); ++i) {
    if (coord[i] < 0 || coord[i] >= s[i]) throw Error(LA_ERR_RANGE, "coordinate out of range");
    off += coord[i] * d[i];
  }
  return off;
}

int64_t eval(const Layout& l, int64_t idx) {
  if (idx < 0 || idx >= size(l)) throw Error(LA_ERR_RANGE, "index out of range");
  return eval_coord(l, unravel(l.shape, idx));
}

int64_t cosize(const Layout& l) {
  // largest offset + 1: each mode contributes its extreme coordinate independently
  auto s = flatten(l.shape);
  auto d = flatten(l.stride);
  int64_t hi = 0;
  for (size_t i = 0; i < s.size(); ++i)
    if (d[i] > 0) hi += (s[i] - 1) * d[i];
  return hi + 1;
}

std::vector<Mode> flat_modes(const Layout& l) {
  auto s = flatten(l.shape);
  auto d = flatten(l.stride);
  std::vector<Mode> m;
  for (size_t i = 0; i < s.size(); ++i) m.push_back({s[i], d[i]});
  return m;
}

// ------------------------------------------------------------------------ algebra
Layout coalesce(const Layout& l) {
  std::vector<Mode> out;
  for (const auto& m : flat_modes(l)) {
    if (m.first == 1) continue;
    if (!out.empty() && m.second == out.back().first * out.back().second) {
      out.back().first *= m.first;
      continue;
    }
    out.push_back(m);
  }
  if (out.empty()) return leaf_layout(1, 0);
  return from_modes(out);
}

Layout composition(const Layout& a, const Layout& b) {
  auto flat_a = flat_modes(coalesce(a));
  std::vector<int64_t> used(flat_a.empty() ? 0 : flat_a.size() - 1, 0);
  return compose_tree(flat_a, b.shape, b.stride, used);
}

Layout complement(const Layout& b, int64_t cotarget) {
  if (cotarget <= 0) throw Error(LA_ERR_ARG, "complement target must be positive");
  std::vector<Mode> m;
  for (const auto& x : flat_modes(b)) {
    if (x.first == 1 || x.second == 0) continue;
    if (x.second < 0) throw Error(LA_ERR_NO_COMPLEMENT, "negative stride");
    m.push_back(x);
  }
  std::sort(m.begin(), m.end(), [](const Mode& p, const Mode& q) {
    return p.second < q.second || (p.second == q.second && p.first < q.first);
  });
  std::vector<Mode> out;
  int64_t cur = 1;
  for (const auto& x : m) {
    if (x.second % cur != 0) throw Error(LA_ERR_NO_COMPLEMENT, "modes overlap or interleave");
    out.push_back({x.second / cur, cur});
    cur = checked_mul(x.first, x.second);
  }
  out.push_back({ceil_div(cotarget, cur), cur});
  Layout raw = from_modes(out);
  return coalesce(raw);
}

Layout logical_divide(const Layout& a, const Tiler& t) {
  if (t.whole) {
    Layout c = complement(t.layout, size(a));
    return composition(a, tuple_layout({t.layout, c}));
  }
  if (static_cast<int>(t.modes.size()) > a.rank()) throw Error(LA_ERR_ARG, "tiler has more modes than the layout");
  if (a.shape.leaf) {
    Tiler w;
    w.whole = true;
    w.layout = t.modes[0];
    return logical_divide(a, w);
  }
  std::vector<Layout> parts;
  for (int i = 0; i < a.rank(); ++i) {
    if (i < static_cast<int>(t.modes.size())) {
      Tiler w;
      w.whole = true;
      w.layout = t.modes[i];
      parts.push_back(logical_divide(a.mode(i), w));
    } else {
      parts.push_back(a.mode(i));
    }
  }
  return tuple_layout(parts);
}

Layout zipped_divide(const Layout& a, const Tiler& t) {
  Layout d = logical_divide(a, t);
  if (t.whole || a.shape.leaf) return d;
  std::vector<Layout> tiles, rest;
  for (int i = 0; i < d.rank(); ++i) {
    if (i < static_cast<int>(t.modes.size())) {
      Layout mi = d.mode(i);
      tiles.push_back(mi.mode(0));
      rest.push_back(mi.mode(1));
    } else {
      rest.push_back(d.mode(i));
    }
  }
  Layout tile = tiles.size() == 1 ? tiles[0] : tuple_layout(tiles);
  Layout grid = rest.size() == 1 ? rest[0] : tuple_layout(rest);
  return tuple_layout({tile, grid});
}

Layout logical_product(const Layout& a, const Layout& b) {
  const int64_t target = checked_mul(size(a), cosize(b));
  Layout c = complement(a, target);
  return tuple_layout({a, composition(c, b)});
}

int64_t swizzle(int bits, int base, int shift, int64_t x) {
  if (bits < 0 || base < 0 || shift < bits || bits + base + shift > 62)
    throw Error(LA_ERR_ARG, "swizzle needs 0 <= bits <= shift and bits + base + shift <= 62");
  const int64_t mask = ((int64_t(1) << bits) - 1) << base;
  return x ^ ((x >> shift) & mask);
}

Layout local_tile(const Layout& a, const Tiler& t, const std::vector<int64_t>& grid_coord,
                  int64_t* origin) {
  Layout z = zipped_divide(a, t);
  Layout grid = z.mode(1);
  if (origin) *origin = eval_coord(grid, grid_coord);
  return z.mode(0);
}

Layout local_tile_proj(const Layout& a, const Tiler& t, const std::vector<int64_t>& grid_coord,
                       const std::vector<int>& step, int64_t* origin) {
  if (t.whole) throw Error(LA_ERR_ARG, "a projected tiler names one tile per mode");
  const size_t n = t.modes.size();
  if (step.size() != n || grid_coord.size() != n) throw Error(LA_ERR_ARG, "tiler, coordinate and step ranks differ");
  Tiler kept;
  std::vector<int64_t> coord;
  for (size_t i = 0; i < n; ++i)
    if (step[i] != 0) {
      kept.modes.push_back(t.modes[i]);
      coord.push_back(grid_coord[i]);
    }
  if (static_cast<int>(kept.modes.size()) != a.rank())
    throw Error(LA_ERR_ARG, "the projection keeps a different number of modes than the layout has");
  Layout z = zipped_divide(a, kept);
  Layout tile = z.mode(0), grid = z.mode(1);
  if (grid.rank() != a.rank()) throw Error(LA_ERR_ARG, "grid rank");
  int64_t off = 0;
  std::vector<Layout> out;
  for (int i = 0; i < tile.rank(); ++i) out.push_back(tile.mode(i));
  for (int i = 0; i < grid.rank(); ++i) {
    Layout g = grid.mode(i);
    if (coord[i] < 0) {
      out.push_back(g);
    } else {
      if (coord[i] >= size(g)) throw Error(LA_ERR_RANGE, "grid coordinate out of range");
      off += eval(g, coord[i]);
    }
  }
  if (origin) *origin = off;
  return tuple_layout(out);
}

Layout local_partition(const Layout& a, const Layout& thr, int64_t tid, int64_t* origin) {
  // the thread's coordinate inside thr: the x with thr(x) == tid, unravelled
  int64_t n = size(thr);
  int64_t found = -1;
  for (int64_t x = 0; x < n; ++x)
    if (eval(thr, x) == tid) {
      found = x;
      break;
    }
  if (found < 0) throw Error(LA_ERR_RANGE, "thread index not in the thread layout's image");
  auto coord = unravel(thr.shape, found);
  // tile a by thr's shape, mode by mode, and index the tile mode with the coordinate
  auto ext = flatten(thr.shape);
  if (static_cast<int>(ext.size()) > a.rank()) throw Error(LA_ERR_ARG, "thread layout rank exceeds the tile's");
  Layout z = zipped_divide(a, tiler_of(ext));
  if (origin) *origin = eval_coord(z.mode(0), coord);
  return z.mode(1);
}

// ------------------------------------------------------------------------ text
std::string to_string(const IntTuple& t) {
  if (t.leaf) return std::to_string(t.value);
  std::string s = "(";
  for (size_t i = 0; i < t.kids.size(); ++i) {
    if (i) s += ",";
    s += to_string(t.kids[i]);
  }
  return s + ")";
}

std::string to_string(const Layout& l) { return to_string(l.shape) + ":" + to_string(l.stride); }

Layout parse_layout(const std::string& text) {
  Parser p(text);
  Layout l = p.layout();
  if (!p.done()) throw Error(LA_ERR_PARSE, "trailing text in " + p.s);
  return l;
}

Tiler parse_tiler(const std::string& text) {
  Parser p(text);
  const std::string& s = p.s;
  Tiler t;
  if (!s.empty() && s.front() == '<') {
    if (s.back() != '>') throw Error(LA_ERR_PARSE, "unterminated tiler " + s);
    for (const auto& part : split_top(s.substr(1, s.size() - 2))) {
      if (part.find(':') != std::string::npos) {
        t.modes.push_back(parse_layout(part));
      } else {
        Parser q(part);
        IntTuple v = q.tuple();
        if (!v.leaf || !q.done()) throw Error(LA_ERR_PARSE, "bad tile extent " + part);
        t.modes.push_back(leaf_layout(v.value, 1));
      }
    }
    return t;
  }
  if (s.find(':') != std::string::npos) {
    t.whole = true;
    t.layout = parse_layout(s);
    return t;
  }
  // a bare shape: one contiguous tile per mode
  Parser q(s);
  IntTuple v = q.tuple();
  if (!q.done()) throw Error(LA_ERR_PARSE, "trailing text in tiler " + s);
  if (v.leaf) {
    t.modes.push_back(leaf_layout(v.value, 1));
    return t;
  }
  for (const auto& k : v.kids) {
    if (!k.leaf) throw Error(LA_ERR_PARSE, "nested tile extents need the <...> form");
    t.modes.push_back(leaf_layout(k.value, 1));
  }
  return t;
}

std::string print_layout(const Layout& l) {
  if (l.rank() != 2) throw Error(LA_ERR_ARG, "print_layout needs a rank-2 layout");
  Layout r = l.mode(0), c = l.mode(1);
  int64_t nr = size(r), nc = size(c);
  if (nr * nc > (1 << 16)) throw Error(LA_ERR_RANGE, "layout too large to print");
  std::ostringstream os;
  os << to_string(l) << "\n";
  os << "     ";
  for (int64_t j = 0; j < nc; ++j) os << " " << std::string(j < 10 ? 4 : (j < 100 ? 3 : 2), ' ') << j;
  os << "\n";
  std::string sep = "     +";
  for (int64_t j = 0; j < nc; ++j) sep += "-----+";
  os << sep << "\n";
  for (int64_t i = 0; i < nr; ++i) {
    std::string idx = std::to_string(i);
    os << std::string(idx.size() < 4 ? 4 - idx.size() : 0, ' ') << idx << " |";
    for (int64_t j = 0; j < nc; ++j) {
      std::string v = std::to_string(eval(r, i) + eval(c, j));
      os << std::string(v.size() < 5 ? 5 - v.size() : 0, ' ') << v << "|";
    }
    os << "\n" << sep << "\n";
  }
  return os.str();
}

}  // namespace la
