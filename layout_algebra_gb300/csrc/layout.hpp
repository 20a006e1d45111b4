// Host-side shape:stride layout algebra.
//
// A layout is a pair of congruent integer trees, Shape:Stride, and is the function
//   coordinate -> sum_i coord_i * stride_i
// ("Day 84: CUTLASS and CuTe layouts", section "A layout is a shape and a stride";
//  "3.5 CUTLASS II", section 3.5.3).  A flat index is unravelled against the shape
// first mode fastest (colexicographic; "Layouts as Algebra", "The formula gets a name").
//
// Operations implemented here, each from the definition on the pages:
//   coalesce       merge s0:d0, s1:(s0*d0) into (s0*s1):d0, drop extent-1 modes
//                  ("Layouts as Algebra", "A shape is a tree"; "3.5 CUTLASS II" 3.5.6)
//   composition    (A o B)(x) = A(B(x)), distributed over B's modes
//                  ("Layouts as Algebra", "Composition, worked by hand")
//   complement     the layout of everything B misses, up to a target size
//                  ("Layouts as Algebra", "Divide is tiling")
//   logical_divide A o (B, B*): mode 0 inside the tile, mode 1 picks the tile
//   zipped_divide  logical_divide with the tile modes gathered first, the grid second
//                  ("Day 84", "A layout is a shape and a stride")
//   local_tile / local_partition  slice the grid mode / the tile mode
//                  ("Layouts as Algebra", "The kernel, in three lines")
//
// This library runs on the host only.  Errors are reported by throwing la::Error.
#pragma once

#include <cstdint>
#include <stdexcept>
#include <string>
#include <utility>
#include <vector>

namespace la {

enum Status : int {
  LA_OK = 0,
  LA_ERR_PARSE = 1,
  LA_ERR_INCONGRUENT = 2,
  LA_ERR_NOT_COMPOSABLE = 3,
  LA_ERR_NO_COMPLEMENT = 4,
  LA_ERR_RANGE = 5,
  LA_ERR_BUFFER = 6,
  LA_ERR_ARG = 7,
};

struct Error : std::runtime_error {
  Status code;
  Error(Status c, const std::string& what) : std::runtime_error(what), code(c) {}
};

// An integer tree: either a leaf holding `value`, or a tuple of children.
struct IntTuple {
  bool leaf = true;
  int64_t value = 0;
  std::vector<IntTuple> kids;

  static IntTuple Int(int64_t v);
  static IntTuple Tup(std::vector<IntTuple> k);
  int rank() const { return leaf ? 1 : static_cast<int>(kids.size()); }
  const IntTuple& mode(int i) const;
};

struct Layout {
  IntTuple shape;
  IntTuple stride;
  int rank() const { return shape.rank(); }
  Layout mode(int i) const;
};

// A tiler is either one layout applied to the whole (1-D) layout, or one tile layout per
// leading mode (an integer t means t:1).
struct Tiler {
  bool whole = false;
  Layout layout;                 // when whole
  std::vector<Layout> modes;     // otherwise
};

// ---------------------------------------------------------------- construction
Layout make_layout(const std::vector<int64_t>& shape, const std::vector<int64_t>& stride);
Layout leaf_layout(int64_t s, int64_t d);
Layout tuple_layout(const std::vector<Layout>& modes);   // (L0, L1, ...) as modes
Tiler tiler_of(const std::vector<int64_t>& tile_extents);

// ---------------------------------------------------------------- queries
bool congruent(const IntTuple& a, const IntTuple& b);
std::vector<int64_t> flatten(const IntTuple& t);
int64_t size(const IntTuple& shape);
int64_t size(const Layout& l);
int64_t cosize(const Layout& l);
std::vector<int64_t> unravel(const IntTuple& shape, int64_t idx);
int64_t eval(const Layout& l, int64_t idx);
int64_t eval_coord(const Layout& l, const std::vector<int64_t>& flat_coord);
std::vector<std::pair<int64_t, int64_t>> flat_modes(const Layout& l);

// ---------------------------------------------------------------- algebra
Layout coalesce(const Layout& l);
Layout composition(const Layout& a, const Layout& b);
Layout complement(const Layout& b, int64_t cotarget);
Layout logical_divide(const Layout& a, const Tiler& t);
Layout zipped_divide(const Layout& a, const Tiler& t);
// logical_product(A, B) = (A, A* o B), A* = complement(A, size(A) * cosize(B)): copies of A
// laid out by the pattern B ("Layouts as Algebra", "Divide is tiling": the mirror of divide).
Layout logical_product(const Layout& a, const Layout& b);
// Swizzle functor Sw<B,M,S>: x -> x ^ ((x >> S) & (((1 << B) - 1) << M)), i.e. the B bits
// above bit M+S are folded into the B bits above bit M.  The 128-byte shared-memory
// swizzle of the tensor copies, in byte offsets, is Sw<3,4,3>.
int64_t swizzle(int bits, int base, int shift, int64_t x);
// local_tile: the tile of zipped_divide(a, t) at grid coordinate `grid_coord`
// (one index per grid leaf).  Returns the tile layout and its origin offset.
Layout local_tile(const Layout& a, const Tiler& t, const std::vector<int64_t>& grid_coord,
                  int64_t* origin);
// local_tile with a projection: the tiler and coordinate name more modes than `a` has (the
// (BM, BN, BK) tiler of a GEMM, say) and step[i] != 0 keeps mode i of them for `a` (CuTe's
// Step<_1, X, _1> for A).  A coordinate of -1 keeps that grid mode whole, as a trailing mode
// of the result over its tiles.  Returns (tile modes..., kept grid modes...) and the
// offset of the fixed coordinates.
Layout local_tile_proj(const Layout& a, const Tiler& t, const std::vector<int64_t>& grid_coord,
                       const std::vector<int>& step, int64_t* origin);
// local_partition: thread `tid` of thread layout `thr` takes, from every thr-shaped
// block of `a`, the element at its own coordinate.  Returns the rest layout and the
// offset of the thread's first element.
Layout local_partition(const Layout& a, const Layout& thr, int64_t tid, int64_t* origin);

// ---------------------------------------------------------------- text
std::string to_string(const IntTuple& t);
std::string to_string(const Layout& l);
Layout parse_layout(const std::string& text);
Tiler parse_tiler(const std::string& text);
std::string print_layout(const Layout& l);   // rank-2 grid, rows = mode 0

}  // namespace la
