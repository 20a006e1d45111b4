/*
 * layout_algebra.h — C ABI of the host shape:stride layout library.
 *
 * Layouts cross this boundary as text in the pages' own notation, Shape:Stride with
 * nested parentheses, e.g. "((2,2),3):((24,2),8)" or "8:1" (a '_' prefix marking a
 * static integer is accepted and ignored).  A tiler is one of:
 *   "4:1"            one layout that divides the whole (1-D) layout,
 *   "(16,16)"        one contiguous tile per leading mode (t means t:1),
 *   "<4:1,(2,2):(1,4)>"  one tile layout per leading mode.
 *
 * All functions run on the host, allocate nothing the caller must free, are
 * thread-safe, and return 0 (LA_OK) or a positive error code (la_error_string names
 * it).  Output text goes to a caller-owned buffer `out` of `cap` bytes; when it does not
 * fit, LA_ERR_BUFFER is returned and `out` holds an empty string.
 *
 * Definitions (page — section):
 *   evaluation      "Day 84: CUTLASS and CuTe layouts" — "A layout is a shape and a
 *                   stride"; flat indices unravel first mode fastest: "Layouts as
 *                   Algebra" — "The formula gets a name".
 *   size, cosize    "3.5 CUTLASS II — CuTe layouts and tensors", 3.5.5.
 *   coalesce        "Layouts as Algebra" — "A shape is a tree".
 *   composition     "Layouts as Algebra" — "Composition, worked by hand".
 *   complement,     "Layouts as Algebra" — "Divide is tiling";
 *   logical_divide  "3.5 CUTLASS II", 3.5.6.
 *   zipped_divide   "Day 84" — "A layout is a shape and a stride".
 *   local_tile,     "Layouts as Algebra" — "The kernel, in three lines";
 *   local_partition "3.5 CUTLASS II", 3.5.6–3.5.7.
 *   thread layouts  "Layouts as Algebra" — "The threads are a layout too".
 */
#ifndef LAYOUT_ALGEBRA_H
#define LAYOUT_ALGEBRA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  LA_OK = 0,
  LA_ERR_PARSE = 1,          /* text is not Shape:Stride, or a tiler form above */
  LA_ERR_INCONGRUENT = 2,    /* shape and stride trees differ */
  LA_ERR_NOT_COMPOSABLE = 3, /* divisibility conditions of composition fail */
  LA_ERR_NO_COMPLEMENT = 4,  /* the layout's modes overlap: no complement exists */
  LA_ERR_RANGE = 5,          /* index/coordinate out of range, or integer overflow */
  LA_ERR_BUFFER = 6,         /* output buffer too small */
  LA_ERR_ARG = 7             /* NULL pointer, non-positive extent, bad rank */
};

const char* la_error_string(int code);

/* size (number of coordinates) and cosize (largest offset + 1). */
int la_size(const char* layout, int64_t* size);
int la_cosize(const char* layout, int64_t* cosize);

/* offsets[i] = layout(idx[i]) for n flat (colexicographic) indices. */
int la_eval(const char* layout, const int64_t* idx, int64_t n, int64_t* offsets);

/* offset of one natural coordinate given leaf by leaf (ncoord = number of leaves). */
int la_eval_coord(const char* layout, const int64_t* coord, int ncoord, int64_t* offset);

/* Algebra: results written as Shape:Stride text. */
int la_coalesce(const char* layout, char* out, size_t cap);
int la_composition(const char* a, const char* b, char* out, size_t cap);
int la_complement(const char* layout, int64_t cotarget, char* out, size_t cap);
int la_logical_divide(const char* layout, const char* tiler, char* out, size_t cap);
int la_zipped_divide(const char* layout, const char* tiler, char* out, size_t cap);

/* The tile of zipped_divide(layout, tiler) at grid coordinate `grid` (ngrid leaves):
   tile layout in `out`, offset of its first element in *origin. */
int la_local_tile(const char* layout, const char* tiler, const int64_t* grid, int ngrid,
                  int64_t* origin, char* out, size_t cap);

/* local_tile with a projection ("Layouts as Algebra" — "The kernel, in three lines": the
   block tiler (BM, BN, BK) is applied to A, B and C with a step that keeps the modes each
   one has).  tiler names n tile modes; step[i] != 0 keeps mode i (the kept modes must number
   the layout's rank); grid[i] is the tile coordinate along mode i, or -1 to keep that grid
   mode whole as a trailing mode of the result.  Writes the layout (tile modes, then the kept
   grid modes) to out and the offset of the fixed coordinates to *origin.  LA_ERR_ARG for a
   rank mismatch, LA_ERR_RANGE for a coordinate off the grid. */
int la_local_tile_proj(const char* layout, const char* tiler, const int64_t* grid, const int* step, int n,
                       int64_t* origin, char* out, size_t cap);

/* Thread `tid` of thread layout `thr`: its elements of `layout` (the rest layout in
   `out`) and the offset of its first element in *origin. */
int la_local_partition(const char* layout, const char* thr, int64_t tid, int64_t* origin,
                       char* out, size_t cap);

/* logical_product(A, B) = (A, complement(A, size(A)*cosize(B)) o B): copies of A laid out
   by the pattern B ("Layouts as Algebra" — "Divide is tiling", the mirror of divide). */
int la_logical_product(const char* a, const char* b, char* out, size_t cap);

/* Swizzle functor Sw<bits,base,shift> applied to n offsets:
   out[i] = x ^ ((x >> shift) & (((1 << bits) - 1) << base)), x = in[i].  Needs
   0 <= bits <= shift and bits + base + shift <= 62.  The tensor copies' 128-byte
   shared-memory swizzle is Sw<3,4,3> on byte offsets. */
int la_swizzle(int bits, int base, int shift, const int64_t* in, int64_t n, int64_t* out);

/* Offset grid of a rank-2 layout (rows = mode 0, columns = mode 1) as text. */
int la_print_layout(const char* layout, char* out, size_t cap);

#ifdef __cplusplus
}
#endif

#endif /* LAYOUT_ALGEBRA_H */
