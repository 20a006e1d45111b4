// Persistent tiled GEMM for sm_103a:  D = alpha * A * B + beta * C — host side and C ABI.
//
// What the pages define ("CUTLASS, in depth" — "The problem CUTLASS solves", "Kernel
// schedules", "Epilogue fusion"; "Layouts as Algebra" — "The kernel, in three lines"):
// a CTA owns a BM x BN output tile, walks K in BK steps and stages the A and B slices in
// shared memory; a producer fills a ring of stages and signals barriers, the consumer
// multiplies and releases them; after the last K step the epilogue applies alpha and
// beta and stores D.  Persistent CTAs loop over tiles in a grouped raster order.
//
// How it maps onto sm_103a (device code in gemm_kernel.cuh):
//   warp 0, one lane   tensor copies (TMA) of A/B into a ring of 128-byte-swizzled shared
//                      memory stages (a CTA pair: 3 stages of two k-blocks, one copy per
//                      operand per stage), counted on mbarriers;
//   warp 1, one lane   tcgen05.mma (fp32 accumulate) into one of two Tensor Memory
//                      accumulators; tcgen05.commit frees a stage when its MMAs retire and
//                      hands a finished accumulator to the epilogue; warp 1 also owns TMEM;
//   warps 2-5          epilogue: tcgen05.ld of their 32-lane quarter, alpha*acc + beta*C in
//                      fp32 (and the fused nodes), rounded to fp16/bf16 and written through
//                      shared-memory staging tiles by tensor copies clipped at M and N (C read
//                      the same way), or with per-thread 16-byte stores (FP8 outputs, N % 8
//                      != 0).  The second accumulator lets the epilogue of tile i overlap the
//                      main loop of tile i+1.
// This file: the layout-algebra planning of a call (tile grids, copy geometry, the C/D offset
// map: zipped_divide((M,N):(N,1), (BM,BN)) and the divides of A and B, see layout.cpp), tensor
// map encoding, the variant and schedule choice, the plan cache, and the C ABI.
//
// Every wait is bounded: past the limit the waiting thread records a code in the device
// status word, raises an abort flag in shared memory, and all roles leave their loops; the
// copy stage waits for its own copies in flight, the MMA stage for its own MMAs, and TMEM is
// always released before the CTA exits.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/gb300_gemm.h"
#include "layout.hpp"
#include "gemm_kernel.cuh"

namespace gb {

// The device status word: the first bounded wait that gave up records `site | cta << 8`;
// kernels receive its address in Params (they are compiled in other translation units).
__device__ uint32_t g_status;

// ------------------------------------------------------------------ scale-factor packing
// Block-scaled FP8 reads its E8M0 scales in 512-byte atoms, each holding 4 k-slices of 32
// elements (one k-block of 128) for 128 rows: scale (row 32 j + i, slice kk) at byte
// 16 i + 4 j + kk, the layout ((32,4),4):((16,4),1) from (row, slice) to bytes.  A packs one
// atom per (128 rows, k-block), atom (rb, kb) at (rb * KB + kb) * 512; B packs two atoms per
// (224 columns, k-block) at (nb * KB + kb) * 1024, its 32-column groups g = 0..6 in atom
// g / 4, group slot g % 4 (slot 3 of the second atom is padding).  Padding holds 127 (1.0).
__global__ void mx_pack_kernel(int operand, int64_t rows, int64_t K, const uint8_t* src, int64_t ld,
                               uint8_t* dst, int64_t total) {
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= total) return;
  const int64_t kbs = (K + 127) / 128, nsf = (K + 31) / 32;
  const int64_t atom_bytes = operand == 0 ? 512 : 1024;
  const int64_t blk = idx / atom_bytes, w = idx % atom_bytes;
  const int64_t rb = blk / kbs, kb = blk % kbs;
  const int64_t w2 = w % 512;
  const int64_t i = w2 / 16, slot = (w2 / 4) % 4, kk = w2 % 4;
  int64_t r;
  bool valid;
  if (operand == 0) {
    r = rb * 128 + 32 * slot + i;
    valid = true;
  } else {
    const int64_t g = (w / 512) * 4 + slot;
    r = rb * kMxTileN + 32 * g + i;
    valid = g < kMxTileN / 32;
  }
  const int64_t sfi = kb * 4 + kk;
  dst[idx] = (valid && r < rows && sfi < nsf) ? src[r * ld + sfi] : static_cast<uint8_t>(127);
}

// ------------------------------------------------------------------ test kernels
__global__ void epilogue_map_kernel(const Params p, int32_t tile_m, int32_t tile_n, int32_t mt, int32_t nt,
                                    int64_t* out) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= tile_m * tile_n) return;
  const int r = idx / tile_n, c = idx % tile_n;
  const int64_t row = static_cast<int64_t>(mt) * tile_m + r;
  const int64_t col = static_cast<int64_t>(nt) * tile_n + c;
  out[idx] = (row < p.M && col < p.N) ? d_offset(p, mt, nt, r, c) : -1;
}

// One CTA of 32 threads: copy one stage of A (which == 0) or B (which == 1) of the single
// variant exactly as its producer does, then dump the raw shared-memory bytes.
__global__ void __launch_bounds__(32, 1)
    stage_bytes_kernel(const __grid_constant__ CUtensorMap tm, const Params p, int which,
                       int32_t tile, int32_t kb, uint4* out) {
  using C = Cfg<false>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_1024(smem_raw);
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + C::kStageBytes);
  const int rows = which == 0 ? kRowsA : C::kRowsB;
  const int bytes = rows * kBK * 2;
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&ctl->full[0]), 1);
    ctl->abort = 0;
    ctl->status = p.status;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t full = smem_addr(&ctl->full[0]);
    mbar_arrive_expect_tx(full, bytes);
    issue_operand<false>(which == 0 ? p.majorA : p.majorB, &tm, smem_addr(smem), full, tile * rows,
                         rows, kb, p.bk_elems);
    wait_drain(full, 0u, p.timeout_ns, p.status);
  }
  __syncthreads();
  const uint4* src = reinterpret_cast<const uint4*>(smem);
  for (int i = threadIdx.x; i < bytes / 16; i += 32) out[i] = src[i];
}

}  // namespace gb

// ====================================================================== host side
namespace {

using gb::Params;

std::mutex g_mu;
uint64_t g_timeout_ns = gb::kDefaultTimeoutNs;
int64_t g_skip_kb = -1;
int g_force_variant = 0;   // 0: choose by shape; 1: single CTA; 2: CTA pair; 4: single CTA with
                           // narrow tiles; 5: CTA pair with 224-column tiles; 6: CTA pair with
                           // 512-column tiles (3 is not a variant)
int g_force_schedule = 0;  // 0: stream-K when a workspace is given, the tiles are fewer than the
                           // CTAs and every CTA gets two stage-blocks; 1: data-parallel only;
                           // 2: stream-K whenever possible

constexpr int kVariantSingle = 1;
constexpr int kVariantPair = 2;
constexpr int kVariantNarrow = 4;   // single CTA, 128 x 64 tiles (few output columns)
constexpr int kVariantPair224 = 5;  // CTA pair, 256 x 224 tiles (K-major B, 16-bit or FP8 inputs)
constexpr int kVariantPair512 = 6;  // CTA pair, 256 x 512 tiles (16-bit or FP8 inputs)
constexpr int kVariantPair448 = 7;  // CTA pair, 256 x 448 tiles (K-major B, 16-bit or FP8 inputs)

bool is_pair(int variant) {
  return variant == kVariantPair || variant == kVariantPair224 || variant == kVariantPair512 ||
         variant == kVariantPair448;
}

using gb::DeviceState;
using gb::Maps;
using gb::prepare_single;
using gb::launch_single;
using gb::prepare_pair;
using gb::launch_pair;

// Per-device launcher state; every write to it (probing, function attributes, cluster
// counts, the stream-K launch counter) happens with g_dev_mu held.
std::mutex g_dev_mu;
DeviceState g_dev[128];

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Copy geometry of one operand, read off its layout: the stride-1 mode is the copy's
// inner dimension; the other mode's stride is the row pitch.  `tile_rows` is the tile
// extent along the operand's rows (for the grid), `cta_rows` the rows one CTA stages.
struct OperandPlan {
  int64_t dim[2], row_bytes, box[2], boxes;
  int64_t grid_rows, k_blocks;
};

// Input element type: 16-bit (fp16/bf16) or 8-bit (E4M3/E5M2).  A 128-byte swizzle row holds
// 128 / bytes elements, which sets the K extent of a k-block.
struct InType {
  int a_fmt, b_fmt;   // instruction-descriptor formats: 0 fp16 / E4M3, 1 bf16 / E5M2
  bool f8;
  int bytes;          // 2 or 1
  bool mx = false;    // block-scaled FP8 (E8M0 scales per 32 K elements)
  int bk() const { return 128 / bytes; }
  int kind() const { return mx ? gb::kInMx : (f8 ? gb::kIn8 : gb::kIn16); }
};

InType in16(int dtype) { return InType{dtype == GB_BF16, dtype == GB_BF16, false, 2, false}; }

// Tile width and the B rows one copy stages per CTA, per variant and input kind.
int64_t tile_n_of(int variant, const InType& in) {
  if (variant == kVariantNarrow) return gb::kNarrowTileN;
  if (in.mx || variant == kVariantPair224) return gb::kMxTileN;
  if (variant == kVariantPair512) return gb::Cfg<true, gb::kIn16, gb::kShapeW512>::kTileN;
  if (variant == kVariantPair448) return gb::Cfg<true, gb::kIn16, gb::kShapeW448>::kTileN;
  return is_pair(variant) ? gb::Cfg<true>::kTileN : gb::Cfg<false>::kTileN;
}
int64_t mma_n_of(int variant, const InType& in) {
  if (variant == kVariantNarrow) return gb::kNarrowTileN;
  if (in.mx || variant == kVariantPair224) return gb::kMxTileN;
  if (variant == kVariantPair512) return gb::Cfg<true, gb::kIn16, gb::kShapeW512>::kMmaN;
  if (variant == kVariantPair448) return gb::Cfg<true, gb::kIn16, gb::kShapeW448>::kMmaN;
  return is_pair(variant) ? gb::Cfg<true>::kMmaN : gb::Cfg<false>::kMmaN;
}

gb_status plan_operand(int64_t rows, int64_t K, int64_t ld, int major, int64_t tile_rows,
                       int64_t cta_rows, OperandPlan* o, const InType& in) {
  if (in.f8 && major != GB_K_MAJOR) return GB_ERR_INVALID_ARG;   // 8-bit operands: K-major only
  la::Layout m = major == GB_K_MAJOR ? la::make_layout({rows, K}, {ld, 1}) : la::make_layout({rows, K}, {1, ld});
  la::Layout z = la::zipped_divide(m, la::tiler_of({tile_rows, in.bk()}));
  auto grid = la::flatten(z.mode(1).shape);   // (row tiles, k-blocks)
  o->grid_rows = grid[0];
  o->k_blocks = grid[1];
  auto modes = la::flat_modes(m);
  const int64_t s_rows = modes[0].second, s_k = modes[1].second;
  if (s_k == 1 && major == GB_K_MAJOR) {
    o->dim[0] = K;
    o->dim[1] = rows;
    o->row_bytes = s_rows * in.bytes;
    o->box[0] = in.bk();
    o->box[1] = cta_rows;
    o->boxes = 1;
  } else if (s_rows == 1) {
    o->dim[0] = rows;
    o->dim[1] = K;
    o->row_bytes = s_k * in.bytes;
    o->box[0] = gb::kSwz;
    o->box[1] = gb::kBK;
    o->boxes = cta_rows / gb::kSwz;
  } else {
    return GB_ERR_INVALID_ARG;
  }
  return GB_OK;
}

gb_status validate_sizes(int64_t M, int64_t N, int64_t K, int64_t lda, int majorA, int64_t ldb,
                         int majorB, int bytes = 2) {
  if (M < 0 || N < 0 || K < 0) return GB_ERR_INVALID_ARG;
  if (majorA != GB_K_MAJOR && majorA != GB_MN_MAJOR) return GB_ERR_INVALID_ARG;
  if (majorB != GB_K_MAJOR && majorB != GB_MN_MAJOR) return GB_ERR_INVALID_ARG;
  const int64_t lim = (int64_t(1) << 31) - 1;
  if (M > lim || N > lim || K > lim) return GB_ERR_INVALID_ARG;
  if (K > 0 && M > 0 && N > 0) {
    if (lda < (majorA == GB_K_MAJOR ? K : M)) return GB_ERR_INVALID_ARG;
    if (ldb < (majorB == GB_K_MAJOR ? K : N)) return GB_ERR_INVALID_ARG;
    if ((lda * bytes) % 16 != 0 || (ldb * bytes) % 16 != 0) return GB_ERR_MISALIGNED;
    if (lda * bytes >= (int64_t(1) << 40) || ldb * bytes >= (int64_t(1) << 40)) return GB_ERR_INVALID_ARG;
  }
  return GB_OK;
}

uint32_t make_idesc(const InType& in, int majorA, int majorB, int tile_m, int mma_n) {
  uint32_t d = 0;
  if (in.mx)
    d |= 1u << 23;                                     // scale factors: E8M0 (bits 4-5, 29-30: ids)
  else
    d |= 1u << 4;                                      // accumulator format: fp32
  d |= static_cast<uint32_t>(in.a_fmt) << 7;           // A format: 0 fp16/E4M3, 1 bf16/E5M2
  d |= static_cast<uint32_t>(in.b_fmt) << 10;          // B format
  d |= static_cast<uint32_t>(majorA) << 15;            // A: 0 K-major, 1 MN-major
  d |= static_cast<uint32_t>(majorB) << 16;            // B: 0 K-major, 1 MN-major
  d |= static_cast<uint32_t>(mma_n >> 3) << 17;        // N / 8
  d |= static_cast<uint32_t>(tile_m >> 4) << 24;       // M / 16 (256 for a CTA pair)
  return d;
}

// Kernel for a problem: a forced variant, else the form that keeps the most SMs busy while
// one wave of tiles covers the output ("CUTLASS, in depth" — "Worked example: tile choice and
// wave quantisation": a grid smaller than the GPU leaves SMs idle):
//   narrow 128 x 64 tiles when the output has at most 64 columns, or when its 128 x 64 tiles
//     fit in one wave (at most one per SM): small problems, whose time is the fixed cost of a
//     tile (set-up, the first copies' latency, the epilogue), run them on more SMs at once;
//   the single CTA (128 x 256) when the output has at most 128 rows, or when its 128 x 256
//     tiles fit in one wave;
//   otherwise the CTA pair, 256 x 224, 256 x 256 or 256 x 512 by the wave cost
//     (choose_pair_width).
// Measured from a CUDA graph on one GB300 (default before -> after): 256^3 9.1 -> 5.5 us,
// 512^3 10.3 -> 7.0, 1024^3 12.4 -> 10.0, 128 x 2048 x 1024 12.8 -> 9.4, 2048 x 2048 x 512
// 12.2 -> 11.2.  Block-scaled inputs have no narrow form and take the pair or the single CTA.
// Tile width of a CTA pair ("CUTLASS, in depth", "Worked example: tile choice and wave
// quantisation"): a persistent grid of G pairs runs ceil(tiles / G) waves of tiles, and a tile
// costs its k-blocks times the time of one k-block of that width, plus, for the 512-column tile
// whose accumulator fills TMEM, the epilogue it cannot overlap.  The per-k-block times are the
// measured ones of the three forms on a GB300 (16-bit inputs, data in L2-friendly order): 224
// columns 0.324 us, 256 columns 0.339 us, 512 columns 0.645 us, and about 1 us of exposed
// epilogue per 512-column tile.  The copy side bounds the narrower forms (a CTA copies 30 or 32
// KiB per k-block for 128 x 224 or 128 x 256 outputs, 48 KiB for 128 x 512), which is why the
// wide tile costs less per column.  For 4096^3 on 76 pairs: 4 waves of 224 (83 us) against 2 of
// 512 (85 us); for 8192^3: 7 waves of 512 (585 us) against 14 of 256 (608 us).  A K-major
// operand whose rows do not start on 128-byte lines (a leading dimension that is not a multiple
// of 128 bytes: every 128-byte copy row then spans two lines) makes the copies slower, the more
// so the more bytes a tile copies per flop: measured on 5000 x 3000 x 4104, 1.33 times the
// per-k-block time for 224 columns and 1.29 for 512.
int choose_pair_width(int64_t M, int64_t N, int64_t K, int pairs, bool allow224, bool allow512,
                      bool split_rows) {
  if (pairs <= 0) return kVariantPair;
  const int64_t m_tiles = (M + 255) / 256;
  const double k_blocks = static_cast<double>((K + gb::kBK - 1) / gb::kBK);
  const double narrow_factor = split_rows ? 1.33 : 1.0, wide_factor = split_rows ? 1.29 : 1.0;
  auto cost = [&](int64_t w, double per_kblock, double epi) {
    const int64_t waves = (m_tiles * ((N + w - 1) / w) + pairs - 1) / pairs;
    return static_cast<double>(waves) * (k_blocks * per_kblock + epi);
  };
  int v = kVariantPair;
  double best = cost(256, 0.339 * narrow_factor, 0.0);
  const double c224 = cost(gb::kMxTileN, 0.324 * narrow_factor, 0.0);
  if (allow224 && c224 < best) {
    v = kVariantPair224;
    best = c224;
  }
  const double c512 = cost(gb::kWideTileN, 0.645 * wide_factor, 1.0);
  if (allow512 && c512 < best) {
    v = kVariantPair512;
    best = c512;
  }
  // 2 x 224 columns: the 512-column tile's costs scaled by 7/8 (K-major B, like 224)
  if (allow512 && allow224 && cost(gb::kWide448TileN, 0.645 * 0.875 * wide_factor, 0.875) < best)
    v = kVariantPair448;
  return v;
}

int choose_variant(int64_t M, int64_t N, int64_t K, const InType& in, int majorA, int64_t lda, int majorB,
                   int64_t ldb, int sms, bool heavy_epilogue = false) {
  int forced;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    forced = g_force_variant;
  }
  const int64_t m128 = (M + gb::Cfg<false>::kTileM - 1) / gb::Cfg<false>::kTileM;
  const int64_t narrow_tiles = m128 * ((N + gb::kNarrowTileN - 1) / gb::kNarrowTileN);
  const int64_t single_tiles = m128 * ((N + gb::Cfg<false>::kTileN - 1) / gb::Cfg<false>::kTileN);
  int v;
  if (forced != 0)
    v = forced;
  else if (N <= gb::kNarrowTileN || narrow_tiles <= sms)
    v = kVariantNarrow;
  else if (M <= gb::Cfg<false>::kTileM || single_tiles <= sms)
    v = kVariantSingle;
  else
    // FP8 k-blocks run at twice the 16-bit MMA rate, so the 512-column tile's exposed epilogue
    // weighs twice as much against its main loop: measured slower for FP8 (8192^3 E4M3: 424 us
    // against 380 with 256 columns), so FP8 takes it only when forced.  A fused epilogue (bias,
    // activation, amax or an FP8 output) does more work per element, which nothing overlaps on
    // the wide tiles: measured on 8192^3 bf16 with C, bias and GELU 747 us with 512 columns
    // against 664 with 256, bias and ReLU 685 against 640, so these keep two accumulators
    v = choose_pair_width(M, N, K, sms / 2, !in.mx && majorB == GB_K_MAJOR,
                          !in.mx && !in.f8 && !heavy_epilogue,
                          (majorA == GB_K_MAJOR && (lda * in.bytes) % 128 != 0) ||
                              (majorB == GB_K_MAJOR && (ldb * in.bytes) % 128 != 0));
  if (in.mx && v == kVariantNarrow) v = M > gb::Cfg<false>::kTileM ? kVariantPair : kVariantSingle;
  if (in.mx && (v == kVariantPair512 || v == kVariantPair448)) v = kVariantPair;
  if (v == kVariantPair448 && majorB != GB_K_MAJOR) v = kVariantPair512;
  // 224-column tiles stage 112 B rows per CTA: K-major B only (an MN-major box is 64 wide)
  if (v == kVariantPair224 && (in.mx || majorB != GB_K_MAJOR)) v = kVariantPair;
  return v;
}

gb_status make_plan(int dtype, int variant, int64_t M, int64_t N, int64_t K, int64_t lda, int majorA,
                    int64_t ldb, int majorB, gb_gemm_plan* pl, const InType* in_override = nullptr) {
  const InType in = in_override ? *in_override : in16(dtype);
  gb_status st = validate_sizes(M, N, K, lda, majorA, ldb, majorB, in.bytes);
  if (st != GB_OK) return st;
  if (dtype != GB_F16 && dtype != GB_BF16) return GB_ERR_INVALID_ARG;
  if (variant != kVariantSingle && variant != kVariantNarrow && !is_pair(variant)) return GB_ERR_INVALID_ARG;
  const bool pair = is_pair(variant);
  const int64_t tile_m = pair ? gb::Cfg<true>::kTileM : gb::Cfg<false>::kTileM;
  if (in.mx && variant == kVariantNarrow) return GB_ERR_INVALID_ARG;
  if (variant == kVariantPair224 && (in.mx || majorB != GB_K_MAJOR)) return GB_ERR_INVALID_ARG;
  if ((variant == kVariantPair512 || variant == kVariantPair448) && in.mx) return GB_ERR_INVALID_ARG;
  if (variant == kVariantPair448 && majorB != GB_K_MAJOR) return GB_ERR_INVALID_ARG;
  const int64_t tile_n = tile_n_of(variant, in);
  // B rows one copy stages: one CTA's share of one MMA's columns
  const int64_t rows_b = pair ? mma_n_of(variant, in) / 2 : mma_n_of(variant, in);
  std::memset(pl, 0, sizeof(*pl));
  pl->variant = variant;
  pl->tile_m = tile_m;
  pl->tile_n = tile_n;
  pl->tile_k = in.bk();
  if (M == 0 || N == 0) return GB_OK;
  try {
    // D (and C): (M,N):(N,1) divided into (tile_m, tile_n) tiles -> ((tile),(grid))
    la::Layout mD = la::make_layout({M, N}, {N, 1});
    la::Layout zD = la::zipped_divide(mD, la::tiler_of({tile_m, tile_n}));
    auto grid_shape = la::flatten(zD.mode(1).shape);
    auto grid_stride = la::flatten(zD.mode(1).stride);
    auto elem_stride = la::flatten(mD.stride);
    pl->m_tiles = grid_shape[0];
    pl->n_tiles = grid_shape[1];
    pl->d_grid_stride[0] = grid_stride[0];
    pl->d_grid_stride[1] = grid_stride[1];
    pl->d_elem_stride[0] = elem_stride[0];
    pl->d_elem_stride[1] = elem_stride[1];
    pl->vector_epilogue = (pl->d_elem_stride[1] == 1 && N % 8 == 0) ? 1 : 0;
    if (K > 0) {
      OperandPlan a, b;
      if ((st = plan_operand(M, K, lda, majorA, tile_m, gb::kRowsA, &a, in)) != GB_OK) return st;
      // B's copy box covers one CTA's rows of one 256-column MMA
      if ((st = plan_operand(N, K, ldb, majorB, tile_n, rows_b, &b, in)) != GB_OK) return st;
      if (a.grid_rows != pl->m_tiles || b.grid_rows != pl->n_tiles || a.k_blocks != b.k_blocks)
        return GB_ERR_INVALID_ARG;
      pl->k_blocks = a.k_blocks;
      for (int i = 0; i < 2; ++i) {
        pl->a_dim[i] = a.dim[i];
        pl->a_box[i] = a.box[i];
        pl->b_dim[i] = b.dim[i];
        pl->b_box[i] = b.box[i];
      }
      pl->a_row_bytes = a.row_bytes;
      pl->a_boxes = a.boxes;
      pl->b_row_bytes = b.row_bytes;
      pl->b_boxes = b.boxes;
    }
    const int64_t tiles = pl->m_tiles * pl->n_tiles;
    if (tiles > (int64_t(1) << 31) - 1) return GB_ERR_INVALID_ARG;
  } catch (const la::Error&) {
    return GB_ERR_INVALID_ARG;
  }
  pl->instr_desc = make_idesc(in, majorA, majorB, static_cast<int>(tile_m), static_cast<int>(mma_n_of(variant, in)));
  return GB_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

gb_status encode_map(CUtensorMap* map, const void* base, const int64_t dim[2], int64_t row_bytes,
                     const int64_t box[2], int dtype, bool f8 = false, bool swizzle = true) {
  auto fn = encode_fn();
  if (!fn) return GB_ERR_LAUNCH;
  cuuint64_t gdim[2] = {static_cast<cuuint64_t>(dim[0]), static_cast<cuuint64_t>(dim[1])};
  cuuint64_t gstride[1] = {static_cast<cuuint64_t>(row_bytes)};
  cuuint32_t bdim[2] = {static_cast<cuuint32_t>(box[0]), static_cast<cuuint32_t>(box[1])};
  cuuint32_t estride[2] = {1, 1};
  const CUtensorMapDataType t = f8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                  : (dtype == GB_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                      : CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
  CUresult r = fn(map, t,
                  2, const_cast<void*>(base), gdim, gstride, bdim, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GB_OK : GB_ERR_LAUNCH;
}

// Stage-deep map of a K-major operand described by the two-dimensional (K, rows) geometry of
// plan_operand: the K mode divided by the k-block, (K):(1) -> (bk, K/bk):(1, bk), as in the
// zipped_divide of the operand by (rows, bk), gives copy dimensions (bk, rows, k-blocks) with
// byte strides (row_bytes, bk * bytes); the box takes `depth` k-blocks at once.  The map
// covers the K / bk whole k-blocks only (rounded down), so no row reads past its own K
// elements; a tail k-block goes through the two-dimensional map.
gb_status encode_map_kblocks(CUtensorMap* map, const void* base, const int64_t dim[2], int64_t row_bytes,
                             const int64_t box[2], int64_t depth, int dtype, bool f8) {
  auto fn = encode_fn();
  if (!fn) return GB_ERR_LAUNCH;
  const int64_t bk = box[0], bytes = f8 ? 1 : 2;
  if (dim[0] < bk) return GB_ERR_INVALID_ARG;
  cuuint64_t gdim[3] = {static_cast<cuuint64_t>(bk), static_cast<cuuint64_t>(dim[1]),
                        static_cast<cuuint64_t>(dim[0] / bk)};
  cuuint64_t gstride[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(bk * bytes)};
  cuuint32_t bdim[3] = {static_cast<cuuint32_t>(bk), static_cast<cuuint32_t>(box[1]),
                        static_cast<cuuint32_t>(depth)};
  cuuint32_t estride[3] = {1, 1, 1};
  const CUtensorMapDataType t = f8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                  : (dtype == GB_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                      : CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
  CUresult r = fn(map, t, 3, const_cast<void*>(base), gdim, gstride, bdim, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GB_OK : GB_ERR_LAUNCH;
}

// Stage-deep map of an MN-major operand described by plan_operand's (rows, K) geometry (rows
// contiguous, K rows `row_bytes` apart).  Dividing the row mode by 64 (one 128-byte swizzle
// span) and the K mode by the k-block gives (64, chunks):(1, 64) and (bk, K/bk):(ld, bk ld);
// ordered as the stage holds them, the copy dimensions are (64 MN elements, bk K rows,
// MN chunks, k-blocks) with byte strides (row_bytes, 128, bk row_bytes).  The box takes
// box_rows / 64 chunks and `depth` k-blocks.  Used only when rows are a multiple of 64; the
// map covers the K / bk whole k-blocks (rounded down), so no copy reads an element outside the
// operand, and a tail k-block goes through the two-dimensional map.
gb_status encode_map_mn_kblocks(CUtensorMap* map, const void* base, const int64_t dim[2], int64_t row_bytes,
                                int64_t box_rows, int64_t bk, int64_t depth, int dtype) {
  auto fn = encode_fn();
  if (!fn) return GB_ERR_LAUNCH;
  const int64_t span = gb::kSwz;
  if (dim[0] % span != 0 || dim[1] < bk || box_rows % span != 0) return GB_ERR_INVALID_ARG;
  cuuint64_t gdim[4] = {static_cast<cuuint64_t>(span), static_cast<cuuint64_t>(bk),
                        static_cast<cuuint64_t>(dim[0] / span), static_cast<cuuint64_t>(dim[1] / bk)};
  cuuint64_t gstride[3] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(span * 2),
                           static_cast<cuuint64_t>(bk * row_bytes)};
  cuuint32_t bdim[4] = {static_cast<cuuint32_t>(span), static_cast<cuuint32_t>(bk),
                        static_cast<cuuint32_t>(box_rows / span), static_cast<cuuint32_t>(depth)};
  cuuint32_t estride[4] = {1, 1, 1, 1};
  const CUtensorMapDataType t = dtype == GB_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUresult r = fn(map, t, 4, const_cast<void*>(base), gdim, gstride, bdim, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GB_OK : GB_ERR_LAUNCH;
}

// Tensor map of a row-major 16-bit M x N matrix (C or D, leading dimension N) for the
// tile-store epilogue: dimensions (N, M), 32 x 32 boxes in the 64-byte swizzle.  A store
// writes only the box's elements inside (N, M); a load zero-fills the rest.
gb_status encode_tile_map(CUtensorMap* map, const void* base, int64_t M, int64_t N, int dtype) {
  auto fn = encode_fn();
  if (!fn) return GB_ERR_LAUNCH;
  cuuint64_t gdim[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M)};
  cuuint64_t gstride[1] = {static_cast<cuuint64_t>(N * 2)};
  cuuint32_t bdim[2] = {32, 32};
  cuuint32_t estride[2] = {1, 1};
  const CUtensorMapDataType t = dtype == GB_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUresult r = fn(map, t, 2, const_cast<void*>(base), gdim, gstride, bdim, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GB_OK : GB_ERR_LAUNCH;
}

// Whether the kernel instance of (variant, input kind) has shared memory for the tile-store
// epilogue's staging tiles.
bool epi_tma_fits(int variant, int kind) {
  using namespace gb;
  if (variant == kVariantNarrow)
    return kind == kIn8 ? Cfg<false, kIn8, kShapeNarrow>::kEpiTma : Cfg<false, kIn16, kShapeNarrow>::kEpiTma;
  if (variant == kVariantPair224)
    return kind == kIn8 ? Cfg<true, kIn8, kShapeN224>::kEpiTma : Cfg<true, kIn16, kShapeN224>::kEpiTma;
  if (variant == kVariantPair512)
    return kind == kIn8 ? Cfg<true, kIn8, kShapeW512>::kEpiTma : Cfg<true, kIn16, kShapeW512>::kEpiTma;
  if (variant == kVariantPair448)
    return kind == kIn8 ? Cfg<true, kIn8, kShapeW448>::kEpiTma : Cfg<true, kIn16, kShapeW448>::kEpiTma;
  if (is_pair(variant))
    return kind == kInMx ? Cfg<true, kInMx>::kEpiTma
                         : (kind == kIn8 ? Cfg<true, kIn8>::kEpiTma : Cfg<true, kIn16>::kEpiTma);
  return kind == kInMx ? Cfg<false, kInMx>::kEpiTma
                       : (kind == kIn8 ? Cfg<false, kIn8>::kEpiTma : Cfg<false, kIn16>::kEpiTma);
}

// K-blocks one pipeline stage of the kernel instance of (variant, input kind) holds: the
// stage-blocks of the schedule (and of the stream-K units) are counted in these.
int stage_kblocks(int variant, int kind) {
  using namespace gb;
  if (variant == kVariantNarrow)
    return kind == kIn8 ? Cfg<false, kIn8, kShapeNarrow>::kKB : Cfg<false, kIn16, kShapeNarrow>::kKB;
  if (variant == kVariantPair224)
    return kind == kIn8 ? Cfg<true, kIn8, kShapeN224>::kKB : Cfg<true, kIn16, kShapeN224>::kKB;
  if (variant == kVariantPair512)
    return kind == kIn8 ? Cfg<true, kIn8, kShapeW512>::kKB : Cfg<true, kIn16, kShapeW512>::kKB;
  if (variant == kVariantPair448)
    return kind == kIn8 ? Cfg<true, kIn8, kShapeW448>::kKB : Cfg<true, kIn16, kShapeW448>::kKB;
  if (is_pair(variant))
    return kind == kInMx ? Cfg<true, kInMx>::kKB : (kind == kIn8 ? Cfg<true, kIn8>::kKB : Cfg<true, kIn16>::kKB);
  return kind == kInMx ? Cfg<false, kInMx>::kKB : (kind == kIn8 ? Cfg<false, kIn8>::kKB : Cfg<false, kIn16>::kKB);
}

gb_status device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GB_ERR_UNSUPPORTED_ARCH;
  if (dev < 0 || dev >= 128) return GB_ERR_UNSUPPORTED_ARCH;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceState& d = g_dev[dev];
  if (!d.probed) {
    if (cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return GB_ERR_UNSUPPORTED_ARCH;
    if (d.major == 10 && d.minor == 3 &&
        (cudaGetSymbolAddress(reinterpret_cast<void**>(&d.status), gb::g_status) != cudaSuccess || !d.status))
      return GB_ERR_CUDA;
    d.probed = true;
  }
  if (d.major != 10 || d.minor != 3) return GB_ERR_UNSUPPORTED_ARCH;
  *out = &d;
  return GB_OK;
}

void fill_params(const DeviceState* dev, const gb_gemm_plan& pl, int64_t M, int64_t N, int64_t K, float alpha, int majorA,
                 int majorB, float beta, const void* C, void* D, Params* p) {
  std::memset(p, 0, sizeof(*p));
  p->M = static_cast<int32_t>(M);
  p->N = static_cast<int32_t>(N);
  p->K = static_cast<int32_t>(K);
  p->m_tiles = static_cast<int32_t>(pl.m_tiles);
  p->n_tiles = static_cast<int32_t>(pl.n_tiles);
  p->k_blocks = static_cast<int32_t>(pl.k_blocks);
  p->num_tiles = static_cast<int32_t>(pl.m_tiles * pl.n_tiles);   // work items: output tiles
  p->group_m = is_pair(pl.variant) ? 8 : 16;
  const int kkb = stage_kblocks(pl.variant, gb::kIn16);
  p->nsb = static_cast<int32_t>((pl.k_blocks + kkb - 1) / kkb);
  p->dp_tiles = p->num_tiles;   // data-parallel unless the caller sets up stream-K
  p->bk_elems = 64;             // 16-bit inputs; 8-bit inputs set 128
  p->majorA = majorA;
  p->majorB = majorB;
  p->alpha = alpha;
  p->beta = beta;
  p->C = static_cast<const uint16_t*>(C);
  p->D = static_cast<uint16_t*>(D);
  p->d_grid_m = pl.d_grid_stride[0];
  p->d_grid_n = pl.d_grid_stride[1];
  p->d_row = pl.d_elem_stride[0];
  p->d_col = pl.d_elem_stride[1];
  p->idesc = pl.instr_desc;
  p->vec_ok = pl.vector_epilogue;
  p->has_c = beta != 0.0f ? 1 : 0;
  std::lock_guard<std::mutex> lk(g_mu);
  p->timeout_ns = g_timeout_ns;
  p->skip_kb = g_skip_kb;
  p->status = dev->status;
}


// Dispatch on the output type, the input kind and the pair kernels (the 224-column pair takes
// 16-bit and FP8 inputs).  prepare_*_any run with g_dev_mu held.
template <bool kBF16>
gb_status prepare_single_any(int kin, bool narrow, DeviceState* dev) {
  using namespace gb;
  if (narrow)
    return kin == kIn8 ? prepare_single<kBF16, kIn8, kShapeNarrow>(dev) : prepare_single<kBF16, kIn16, kShapeNarrow>(dev);
  if (kin == kInMx) return prepare_single<kBF16, kInMx, kShapeStd>(dev);
  return kin == kIn8 ? prepare_single<kBF16, kIn8, kShapeStd>(dev) : prepare_single<kBF16, kIn16, kShapeStd>(dev);
}

template <bool kBF16>
gb_status prepare_pair_any(int kin, int shape, DeviceState* dev) {
  using namespace gb;
  if (shape == kShapeN224)
    return kin == kIn8 ? prepare_pair<kBF16, kIn8, kShapeN224>(dev) : prepare_pair<kBF16, kIn16, kShapeN224>(dev);
  if (shape == kShapeW512)
    return kin == kIn8 ? prepare_pair<kBF16, kIn8, kShapeW512>(dev) : prepare_pair<kBF16, kIn16, kShapeW512>(dev);
  if (shape == kShapeW448)
    return kin == kIn8 ? prepare_pair<kBF16, kIn8, kShapeW448>(dev) : prepare_pair<kBF16, kIn16, kShapeW448>(dev);
  if (kin == kInMx) return prepare_pair<kBF16, kInMx, kShapeStd>(dev);
  return kin == kIn8 ? prepare_pair<kBF16, kIn8, kShapeStd>(dev) : prepare_pair<kBF16, kIn16, kShapeStd>(dev);
}

template <bool kBF16>
gb_status launch_any(bool pair, int kin, int shape, bool narrow, const Maps& m, const Params& p, int G,
                     cudaStream_t s) {
  if (!pair) {
    if (narrow)
      return kin == gb::kIn8 ? launch_single<kBF16, gb::kIn8, gb::kShapeNarrow>(m, p, G, s)
                             : launch_single<kBF16, gb::kIn16, gb::kShapeNarrow>(m, p, G, s);
    if (kin == gb::kInMx) return launch_single<kBF16, gb::kInMx, gb::kShapeStd>(m, p, G, s);
    return kin == gb::kIn8 ? launch_single<kBF16, gb::kIn8, gb::kShapeStd>(m, p, G, s)
                           : launch_single<kBF16, gb::kIn16, gb::kShapeStd>(m, p, G, s);
  }
  if (shape == gb::kShapeN224)
    return kin == gb::kIn8 ? launch_pair<kBF16, gb::kIn8, gb::kShapeN224>(m, p, G, s)
                           : launch_pair<kBF16, gb::kIn16, gb::kShapeN224>(m, p, G, s);
  if (shape == gb::kShapeW512)
    return kin == gb::kIn8 ? launch_pair<kBF16, gb::kIn8, gb::kShapeW512>(m, p, G, s)
                           : launch_pair<kBF16, gb::kIn16, gb::kShapeW512>(m, p, G, s);
  if (shape == gb::kShapeW448)
    return kin == gb::kIn8 ? launch_pair<kBF16, gb::kIn8, gb::kShapeW448>(m, p, G, s)
                           : launch_pair<kBF16, gb::kIn16, gb::kShapeW448>(m, p, G, s);
  if (kin == gb::kInMx) return launch_pair<kBF16, gb::kInMx, gb::kShapeStd>(m, p, G, s);
  return kin == gb::kIn8 ? launch_pair<kBF16, gb::kIn8, gb::kShapeStd>(m, p, G, s)
                         : launch_pair<kBF16, gb::kIn16, gb::kShapeStd>(m, p, G, s);
}

// Workspace layout: one 32-bit flag per CTA (padded to 256 B), then one 128 x 256 fp32
// partial per CTA.  Every slot a grid on this device can use fits (one per SM).
int64_t workspace_bytes_for(int sms) {
  const int64_t flags = ((static_cast<int64_t>(sms) * 4 + 255) / 256) * 256;
  return flags + static_cast<int64_t>(sms) * gb::kSlotFloats * 4;
}

// Plans and tensor maps of recent calls.  Building them (the layout algebra and four map
// encodings) costs tens of microseconds on the host, more than a small GEMM takes on the
// GPU; a repeated call with the same operands and shape reuses them.
struct PlanKey {
  int device, dtype, kind, a_fmt, b_fmt, variant, majorA, majorB;
  int64_t M, N, K, lda, ldb;
  const void *A, *B, *sfa, *sfb, *C, *D;
  bool epi_tma;
  bool operator==(const PlanKey& o) const {
    return device == o.device && dtype == o.dtype && kind == o.kind && a_fmt == o.a_fmt && b_fmt == o.b_fmt &&
           variant == o.variant && majorA == o.majorA && majorB == o.majorB && M == o.M && N == o.N &&
           K == o.K && lda == o.lda && ldb == o.ldb && A == o.A && B == o.B && sfa == o.sfa && sfb == o.sfb &&
           C == o.C && D == o.D && epi_tma == o.epi_tma;
  }
};
struct PlanEntry {
  bool valid = false;
  PlanKey key;
  gb_gemm_plan pl;
  Maps maps;
};
constexpr int kPlanCacheSize = 16;
PlanEntry g_plan_cache[kPlanCacheSize];
int g_plan_next = 0;

bool plan_cache_get(const PlanKey& k, gb_gemm_plan* pl, Maps* maps) {
  std::lock_guard<std::mutex> lk(g_mu);
  for (const PlanEntry& e : g_plan_cache)
    if (e.valid && e.key == k) {
      *pl = e.pl;
      *maps = e.maps;
      return true;
    }
  return false;
}

void plan_cache_put(const PlanKey& k, const gb_gemm_plan& pl, const Maps& maps) {
  std::lock_guard<std::mutex> lk(g_mu);
  PlanEntry& e = g_plan_cache[g_plan_next];
  g_plan_next = (g_plan_next + 1) % kPlanCacheSize;
  e.valid = true;
  e.key = k;
  e.pl = pl;
  e.maps = maps;
}

gb_status gemm_entry(int dtype, int64_t M, int64_t N, int64_t K, float alpha, const void* A, int64_t lda,
                     int majorA, const void* B, int64_t ldb, int majorB, float beta, const void* C, void* D,
                     void* workspace, size_t workspace_size, void* stream, const gb_epilogue* epi = nullptr,
                     const InType* in_f8 = nullptr, const void* sfa = nullptr, const void* sfb = nullptr) {
  // dtype names the 16-bit type of C, D and the bias; the inputs share it unless in_f8 names
  // 8-bit input formats (with packed scale factors sfa / sfb when block-scaled)
  const InType in = in_f8 ? *in_f8 : in16(dtype);
  gb_status st = validate_sizes(M, N, K, lda, majorA, ldb, majorB, in.bytes);
  if (st != GB_OK) return st;
  if (dtype != GB_F16 && dtype != GB_BF16) return GB_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return GB_OK;
  if (D == nullptr) return GB_ERR_INVALID_ARG;
  if (beta != 0.0f && C == nullptr) return GB_ERR_INVALID_ARG;
  if (K > 0 && (A == nullptr || B == nullptr)) return GB_ERR_INVALID_ARG;
  if (!aligned16(D) || (C && !aligned16(C))) return GB_ERR_MISALIGNED;
  if (K > 0 && (!aligned16(A) || !aligned16(B))) return GB_ERR_MISALIGNED;
  if (K > 0 && in.mx) {
    if (sfa == nullptr || sfb == nullptr) return GB_ERR_INVALID_ARG;
    if (!aligned16(sfa) || !aligned16(sfb)) return GB_ERR_MISALIGNED;
  }
  if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return GB_ERR_MISALIGNED;
  if (epi) {
    if (epi->activation < GB_ACT_NONE || epi->activation > GB_ACT_GELU) return GB_ERR_INVALID_ARG;
    if (epi->out_format < GB_OUT_INPUT_TYPE || epi->out_format > GB_OUT_E5M2) return GB_ERR_INVALID_ARG;
    if (epi->out_format != GB_OUT_INPUT_TYPE && !(epi->out_scale > 0.0f && epi->out_scale < 3.0e38f))
      return GB_ERR_INVALID_ARG;
    if (epi->amax && (reinterpret_cast<uintptr_t>(epi->amax) & 3u) != 0) return GB_ERR_MISALIGNED;
    if (epi->bias && (reinterpret_cast<uintptr_t>(epi->bias) & 1u) != 0) return GB_ERR_MISALIGNED;
  }
  DeviceState* dev;
  if ((st = device_state(&dev)) != GB_OK) return st;
  if (workspace && static_cast<int64_t>(workspace_size) < workspace_bytes_for(dev->sms))
    return GB_ERR_INVALID_ARG;
  const bool heavy_epilogue = epi && (epi->bias != nullptr || epi->activation != GB_ACT_NONE ||
                                      epi->amax != nullptr || epi->out_format != GB_OUT_INPUT_TYPE);
  const int variant = choose_variant(M, N, K, in, majorA, lda, majorB, ldb, dev->sms, heavy_epilogue);
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return GB_ERR_UNSUPPORTED_ARCH;

  // tile-store epilogue: 16-bit D stored by 32 x 32 tensor copies (row-major, N % 8 == 0; C
  // read the same way); other outputs use per-thread stores
  const bool epi_tma = (N % 8 == 0) && (!epi || epi->out_format == GB_OUT_INPUT_TYPE) &&
                       epi_tma_fits(variant, in.kind());
  const void* c_key = epi_tma && beta != 0.0f ? C : nullptr;
  const PlanKey key{device, dtype, in.kind(), in.a_fmt, in.b_fmt, variant, majorA, majorB, M, N, K, lda, ldb,
                    K > 0 ? A : nullptr, K > 0 ? B : nullptr, in.mx ? sfa : nullptr, in.mx ? sfb : nullptr,
                    c_key, epi_tma ? D : nullptr, epi_tma};
  gb_gemm_plan pl;
  Maps maps;
  if (!plan_cache_get(key, &pl, &maps)) {
    if ((st = make_plan(dtype, variant, M, N, K, lda, majorA, ldb, majorB, &pl, &in)) != GB_OK) return st;
    std::memset(&maps, 0, sizeof(maps));
    if (K > 0) {
      // CTA pairs copy a whole stage (kKB k-blocks) of an operand with one
      // copy when K is a multiple of the k-block (and, MN-major, the operand's rows a multiple
      // of 64): fewer, larger copies keep the per-SM copy rate up (each copy costs a fixed
      // overhead).  Other operands use two-dimensional copies per k-block.
      const int64_t depth = stage_kblocks(pl.variant, in.kind());
      // whole k-blocks the stage-deep maps cover; a K tail is copied per k-block (tail maps)
      const int64_t kb_full = K / in.bk();
      const bool stage_boxes = is_pair(pl.variant) && depth > 1 && kb_full >= 1;
      maps.kb_full = static_cast<int32_t>(stage_boxes ? kb_full : pl.k_blocks);
      if (stage_boxes && majorA == GB_K_MAJOR) {
        if ((st = encode_map_kblocks(&maps.a, A, pl.a_dim, pl.a_row_bytes, pl.a_box, depth, dtype, in.f8)) != GB_OK)
          return st;
        maps.kb_boxes |= 1;
      } else if (stage_boxes && !in.f8 && M % gb::kSwz == 0) {
        if ((st = encode_map_mn_kblocks(&maps.a, A, pl.a_dim, pl.a_row_bytes, gb::kRowsA, in.bk(), depth, dtype)) !=
            GB_OK)
          return st;
        maps.kb_boxes |= 1;
      } else if ((st = encode_map(&maps.a, A, pl.a_dim, pl.a_row_bytes, pl.a_box, dtype, in.f8)) != GB_OK) {
        return st;
      }
      if (stage_boxes && majorB == GB_K_MAJOR) {
        if ((st = encode_map_kblocks(&maps.b, B, pl.b_dim, pl.b_row_bytes, pl.b_box, depth, dtype, in.f8)) != GB_OK)
          return st;
        maps.kb_boxes |= 2;
      } else if (stage_boxes && !in.f8 && N % gb::kSwz == 0) {
        if ((st = encode_map_mn_kblocks(&maps.b, B, pl.b_dim, pl.b_row_bytes, gb::Cfg<true>::kRowsBSub, in.bk(), depth,
                                        dtype)) != GB_OK)
          return st;
        maps.kb_boxes |= 2;
      } else if ((st = encode_map(&maps.b, B, pl.b_dim, pl.b_row_bytes, pl.b_box, dtype, in.f8)) != GB_OK) {
        return st;
      }
      if (maps.kb_full < pl.k_blocks) {
        if ((maps.kb_boxes & 1) &&
            (st = encode_map(&maps.at, A, pl.a_dim, pl.a_row_bytes, pl.a_box, dtype, in.f8)) != GB_OK)
          return st;
        if ((maps.kb_boxes & 2) &&
            (st = encode_map(&maps.bt, B, pl.b_dim, pl.b_row_bytes, pl.b_box, dtype, in.f8)) != GB_OK)
          return st;
      }
      if (in.mx) {
        // packed scales seen as rows of 256 bytes: a 512-byte atom of A per (128 rows,
        // k-block), two atoms of B per (224 columns, k-block); one copy takes a stage's kKB
        // consecutive k-blocks
        const int64_t kkb = stage_kblocks(pl.variant, gb::kInMx);
        const int64_t a_rows = 2 * ((M + 127) / 128) * pl.k_blocks;
        const int64_t b_rows = 4 * pl.n_tiles * pl.k_blocks;
        const int64_t a_dim[2] = {256, a_rows}, b_dim[2] = {256, b_rows};
        const int64_t a_box[2] = {256, 2 * kkb}, b_box[2] = {256, 4 * kkb};
        if ((st = encode_map(&maps.sfa, sfa, a_dim, 256, a_box, dtype, true, false)) != GB_OK) return st;
        if ((st = encode_map(&maps.sfb, sfb, b_dim, 256, b_box, dtype, true, false)) != GB_OK) return st;
      }
    }
    if (epi_tma && pl.vector_epilogue) {
      if ((st = encode_tile_map(&maps.d, D, M, N, dtype)) != GB_OK) return st;
      if (c_key && (st = encode_tile_map(&maps.c, C, M, N, dtype)) != GB_OK) return st;
      maps.epi_tma = 1;
    }
    plan_cache_put(key, pl, maps);
  }
  Params p;
  fill_params(dev, pl, M, N, K, alpha, majorA, majorB, beta, C, D, &p);
  p.bk_elems = in.bk();
  p.kb_boxes = maps.kb_boxes;
  p.kb_full = K > 0 ? maps.kb_full : 0;
  p.epi_tma = maps.epi_tma;
  if (epi) {
    p.fused = 1;
    p.bias = static_cast<const uint16_t*>(epi->bias);
    p.act = epi->activation;
    p.amax = epi->amax;
    p.out_fmt = epi->out_format;
    p.out_scale = epi->out_scale;
    p.vec8_ok = (pl.d_elem_stride[1] == 1 && N % 16 == 0) ? 1 : 0;
  }
  const bool pair = is_pair(pl.variant);
  const int shape = pl.variant == kVariantPair224 ? gb::kShapeN224
                    : (pl.variant == kVariantPair512 ? gb::kShapeW512
                                                     : (pl.variant == kVariantPair448 ? gb::kShapeW448 : gb::kShapeStd));
  const bool bf = dtype == GB_BF16;
  const bool narrow = pl.variant == kVariantNarrow;
  int slots;   // CTAs (clusters) that can run at once
  {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (pair)
      st = bf ? prepare_pair_any<true>(in.kind(), shape, dev) : prepare_pair_any<false>(in.kind(), shape, dev);
    else
      st = bf ? prepare_single_any<true>(in.kind(), narrow, dev) : prepare_single_any<false>(in.kind(), narrow, dev);
    if (st != GB_OK) return st;
    slots = pair ? dev->pair_clusters[gb::pair_shape_index(shape)] : dev->sms;
  }

  // schedule: stream-K needs a workspace and some K; by default it is used when the tiles
  // leave a ragged last wave (or fewer tiles than CTAs)
  int sched;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    sched = g_force_schedule;
  }
  const int kkb = stage_kblocks(pl.variant, in.kind());
  p.nsb = static_cast<int32_t>((pl.k_blocks + kkb - 1) / kkb);
  bool sk = workspace != nullptr && p.nsb > 0 && sched != 1;
  // default: only an under-filled GPU gains (fewer tiles than CTAs, the decode-like shapes);
  // a ragged last wave of a larger problem is cheaper than the partial-tile hand-offs (the
  // 224-column pair tiles absorb most of it), and a K too short to give every CTA two
  // stage-blocks costs more in hand-offs than it spreads
  if (sk && sched == 0)
    sk = p.num_tiles < slots && static_cast<int64_t>(p.num_tiles) * p.nsb >= 2 * static_cast<int64_t>(slots);
  int G;
  if (sk) {
    G = slots;
    const int full = p.num_tiles / G;
    p.dp_tiles = full >= 2 ? (full - 1) * G : 0;
    {
      std::lock_guard<std::mutex> lk(g_dev_mu);
      if (++dev->epoch == 0) dev->epoch = 1;
      p.epoch = dev->epoch;
    }
    p.ws_flags = static_cast<uint32_t*>(workspace);
    p.ws_part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                         ((static_cast<int64_t>(dev->sms) * 4 + 255) / 256) * 256);
  } else {
    G = std::min(p.num_tiles, slots);
    p.dp_tiles = p.num_tiles;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return bf ? launch_any<true>(pair, in.kind(), shape, narrow, maps, p, G, s)
            : launch_any<false>(pair, in.kind(), shape, narrow, maps, p, G, s);
}

}  // namespace

extern "C" {

gb_status gb_gemm_f16(int64_t M, int64_t N, int64_t K, float alpha, const void* A, int64_t lda, int majorA,
                      const void* B, int64_t ldb, int majorB, float beta, const void* C, void* D,
                      void* stream) {
  return gemm_entry(GB_F16, M, N, K, alpha, A, lda, majorA, B, ldb, majorB, beta, C, D, nullptr, 0, stream);
}

gb_status gb_gemm_bf16(int64_t M, int64_t N, int64_t K, float alpha, const void* A, int64_t lda, int majorA,
                       const void* B, int64_t ldb, int majorB, float beta, const void* C, void* D,
                       void* stream) {
  return gemm_entry(GB_BF16, M, N, K, alpha, A, lda, majorA, B, ldb, majorB, beta, C, D, nullptr, 0, stream);
}

gb_status gb_gemm_f16_ws(int64_t M, int64_t N, int64_t K, float alpha, const void* A, int64_t lda, int majorA,
                         const void* B, int64_t ldb, int majorB, float beta, const void* C, void* D,
                         void* workspace, size_t workspace_bytes, void* stream) {
  if (!workspace) return GB_ERR_INVALID_ARG;
  return gemm_entry(GB_F16, M, N, K, alpha, A, lda, majorA, B, ldb, majorB, beta, C, D, workspace,
                    workspace_bytes, stream);
}

gb_status gb_gemm_bf16_ws(int64_t M, int64_t N, int64_t K, float alpha, const void* A, int64_t lda, int majorA,
                          const void* B, int64_t ldb, int majorB, float beta, const void* C, void* D,
                          void* workspace, size_t workspace_bytes, void* stream) {
  if (!workspace) return GB_ERR_INVALID_ARG;
  return gemm_entry(GB_BF16, M, N, K, alpha, A, lda, majorA, B, ldb, majorB, beta, C, D, workspace,
                    workspace_bytes, stream);
}

gb_status gb_gemm_fp8(int a_format, int b_format, int out_dtype, int64_t M, int64_t N, int64_t K, float alpha,
                      const void* A, int64_t lda, const void* B, int64_t ldb, float beta, const void* C, void* D,
                      const gb_epilogue* epi, void* workspace, size_t workspace_bytes, void* stream) {
  if (a_format != GB_FP8_E4M3 && a_format != GB_FP8_E5M2) return GB_ERR_INVALID_ARG;
  if (b_format != GB_FP8_E4M3 && b_format != GB_FP8_E5M2) return GB_ERR_INVALID_ARG;
  if (out_dtype != GB_F16 && out_dtype != GB_BF16) return GB_ERR_INVALID_ARG;
  const InType in{a_format, b_format, true, 1};
  return gemm_entry(out_dtype, M, N, K, alpha, A, lda, GB_K_MAJOR, B, ldb, GB_K_MAJOR, beta, C, D, workspace,
                    workspace_bytes, stream, epi, &in);
}

gb_status gb_mx_scales_bytes(int operand, int64_t rows, int64_t K, size_t* bytes) {
  if (!bytes || rows < 0 || K < 0 || (operand != 0 && operand != 1)) return GB_ERR_INVALID_ARG;
  const int64_t kbs = (K + 127) / 128;
  const int64_t blocks = operand == 0 ? (rows + 127) / 128 : (rows + gb::kMxTileN - 1) / gb::kMxTileN;
  *bytes = static_cast<size_t>(blocks * kbs * (operand == 0 ? 512 : 1024));
  return GB_OK;
}

gb_status gb_mx_pack_scales(int operand, int64_t rows, int64_t K, const void* src, int64_t ld_src, void* dst,
                            void* stream) {
  size_t bytes = 0;
  gb_status st = gb_mx_scales_bytes(operand, rows, K, &bytes);
  if (st != GB_OK) return st;
  if (bytes == 0) return GB_OK;
  if (!src || !dst || ld_src < (K + 31) / 32) return GB_ERR_INVALID_ARG;
  DeviceState* dev;
  if ((st = device_state(&dev)) != GB_OK) return st;
  const int64_t total = static_cast<int64_t>(bytes);
  const int threads = 256;
  const int64_t blocks = (total + threads - 1) / threads;
  if (blocks > 0x7fffffff) return GB_ERR_INVALID_ARG;
  gb::mx_pack_kernel<<<static_cast<unsigned>(blocks), threads, 0, static_cast<cudaStream_t>(stream)>>>(
      operand, rows, K, static_cast<const uint8_t*>(src), ld_src, static_cast<uint8_t*>(dst), total);
  return cudaGetLastError() == cudaSuccess ? GB_OK : GB_ERR_LAUNCH;
}

gb_status gb_gemm_mxfp8(int a_format, int b_format, int out_dtype, int64_t M, int64_t N, int64_t K, float alpha,
                        const void* A, int64_t lda, const void* sfa, const void* B, int64_t ldb, const void* sfb,
                        float beta, const void* C, void* D, const gb_epilogue* epi, void* workspace,
                        size_t workspace_bytes, void* stream) {
  if (a_format != GB_FP8_E4M3 && a_format != GB_FP8_E5M2) return GB_ERR_INVALID_ARG;
  if (b_format != GB_FP8_E4M3 && b_format != GB_FP8_E5M2) return GB_ERR_INVALID_ARG;
  if (out_dtype != GB_F16 && out_dtype != GB_BF16) return GB_ERR_INVALID_ARG;
  const InType in{a_format, b_format, true, 1, true};
  return gemm_entry(out_dtype, M, N, K, alpha, A, lda, GB_K_MAJOR, B, ldb, GB_K_MAJOR, beta, C, D, workspace,
                    workspace_bytes, stream, epi, &in, sfa, sfb);
}

gb_status gb_gemm_ex(int dtype, int64_t M, int64_t N, int64_t K, float alpha, const void* A, int64_t lda,
                     int majorA, const void* B, int64_t ldb, int majorB, float beta, const void* C, void* D,
                     const gb_epilogue* epi, void* workspace, size_t workspace_bytes, void* stream) {
  if (dtype != GB_F16 && dtype != GB_BF16) return GB_ERR_INVALID_ARG;
  return gemm_entry(dtype, M, N, K, alpha, A, lda, majorA, B, ldb, majorB, beta, C, D, workspace,
                    workspace_bytes, stream, epi);
}

gb_status gb_gemm_workspace_bytes(size_t* bytes) {
  if (!bytes) return GB_ERR_INVALID_ARG;
  DeviceState* dev;
  gb_status st = device_state(&dev);
  if (st != GB_OK) return st;
  *bytes = static_cast<size_t>(workspace_bytes_for(dev->sms));
  return GB_OK;
}

gb_status gb_set_schedule(int schedule) {
  if (schedule < 0 || schedule > 2) return GB_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  g_force_schedule = schedule;
  return GB_OK;
}

gb_status gb_last_device_status(void* stream, uint32_t* detail) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return GB_ERR_CUDA;
  uint32_t v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, gb::g_status, sizeof(v)) != cudaSuccess) return GB_ERR_CUDA;
  if (v != 0 && cudaMemcpyToSymbol(gb::g_status, &zero, sizeof(zero)) != cudaSuccess) return GB_ERR_CUDA;
  if (detail) *detail = v;
  return v == 0 ? GB_OK : GB_ERR_TIMEOUT;
}

const char* gb_status_string(int status) {
  switch (status) {
    case GB_OK: return "ok";
    case GB_ERR_INVALID_ARG: return "invalid argument";
    case GB_ERR_MISALIGNED: return "misaligned operand";
    case GB_ERR_UNSUPPORTED_ARCH: return "unsupported architecture (needs compute capability 10.3)";
    case GB_ERR_LAUNCH: return "launch failed";
    case GB_ERR_TIMEOUT: return "device wait timed out";
    case GB_ERR_CUDA: return "CUDA runtime error";
    case GB_ERR_SCRATCH_LIMIT: return "device needs more scratch than the built-in array holds";
    default: return "unknown status";
  }
}

gb_status gb_gemm_make_plan(int dtype, int64_t M, int64_t N, int64_t K, int64_t lda, int majorA, int64_t ldb,
                            int majorB, gb_gemm_plan* plan) {
  if (!plan) return GB_ERR_INVALID_ARG;
  if (M < 0) return GB_ERR_INVALID_ARG;
  // the variant is chosen for this device's SM count; without a device (a plan made on a host
  // with no GPU), for 152 SMs
  int sms = 152, device = 0;
  if (cudaGetDevice(&device) == cudaSuccess) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) == cudaSuccess && n > 0) sms = n;
  }
  cudaGetLastError();
  return make_plan(dtype, choose_variant(M, N, K, in16(dtype), majorA, lda, majorB, ldb, sms), M, N, K, lda, majorA,
                   ldb, majorB, plan);
}

gb_status gb_set_wait_timeout_ns(uint64_t ns) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_timeout_ns = ns == 0 ? gb::kDefaultTimeoutNs : ns;
  return GB_OK;
}

gb_status gb_debug_skip_k_block(int64_t k_block) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_skip_kb = k_block < 0 ? -1 : k_block;
  return GB_OK;
}

gb_status gb_set_kernel_variant(int variant) {
  if (variant != 0 && variant != kVariantSingle && variant != kVariantNarrow && !is_pair(variant))
    return GB_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  g_force_variant = variant;
  return GB_OK;
}

gb_status gb_debug_epilogue_map(int variant, int64_t M, int64_t N, int64_t m_tile, int64_t n_tile, int64_t* out,
                                void* stream) {
  gb_gemm_plan pl;
  gb_status st = make_plan(GB_F16, variant, M, N, 0, 0, GB_K_MAJOR, 0, GB_K_MAJOR, &pl);
  if (st != GB_OK) return st;
  if (M == 0 || N == 0 || !out || m_tile < 0 || n_tile < 0 || m_tile >= pl.m_tiles || n_tile >= pl.n_tiles)
    return GB_ERR_INVALID_ARG;
  DeviceState* dev;
  if ((st = device_state(&dev)) != GB_OK) return st;
  Params p;
  fill_params(dev, pl, M, N, 0, 1.0f, 0, 0, 0.0f, nullptr, nullptr, &p);
  const int n = static_cast<int>(pl.tile_m * pl.tile_n);
  gb::epilogue_map_kernel<<<n / 256, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      p, static_cast<int32_t>(pl.tile_m), static_cast<int32_t>(pl.tile_n), static_cast<int32_t>(m_tile),
      static_cast<int32_t>(n_tile), out);
  return cudaGetLastError() == cudaSuccess ? GB_OK : GB_ERR_LAUNCH;
}

gb_status gb_debug_stage_bytes(int dtype, int which, int64_t M, int64_t N, int64_t K, const void* A,
                               int64_t lda, int majorA, const void* B, int64_t ldb, int majorB, int64_t tile,
                               int64_t k_block, void* out, void* stream) {
  gb_gemm_plan pl;
  gb_status st = make_plan(dtype, kVariantSingle, M, N, K, lda, majorA, ldb, majorB, &pl);
  if (st != GB_OK) return st;
  if (M == 0 || N == 0 || K == 0 || !out || (which != 0 && which != 1)) return GB_ERR_INVALID_ARG;
  const void* base = which == 0 ? A : B;
  if (!base || !aligned16(base) || !aligned16(out)) return GB_ERR_MISALIGNED;
  const int64_t ntiles = which == 0 ? pl.m_tiles : pl.n_tiles;
  if (tile < 0 || tile >= ntiles || k_block < 0 || k_block >= pl.k_blocks) return GB_ERR_INVALID_ARG;
  DeviceState* dev;
  if ((st = device_state(&dev)) != GB_OK) return st;
  CUtensorMap tm;
  st = which == 0 ? encode_map(&tm, A, pl.a_dim, pl.a_row_bytes, pl.a_box, dtype)
                  : encode_map(&tm, B, pl.b_dim, pl.b_row_bytes, pl.b_box, dtype);
  if (st != GB_OK) return st;
  Params p;
  fill_params(dev, pl, M, N, K, 1.0f, majorA, majorB, 0.0f, nullptr, nullptr, &p);
  const int smem = 1024 + gb::Cfg<false>::kStageBytes + gb::kCtlBytes;
  {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (!dev->dbg_attr) {
      if (cudaFuncSetAttribute(gb::stage_bytes_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
          cudaSuccess)
        return GB_ERR_LAUNCH;
      dev->dbg_attr = true;
    }
  }
  gb::stage_bytes_kernel<<<1, 32, smem, static_cast<cudaStream_t>(stream)>>>(
      tm, p, which, static_cast<int32_t>(tile), static_cast<int32_t>(k_block), static_cast<uint4*>(out));
  return cudaGetLastError() == cudaSuccess ? GB_OK : GB_ERR_LAUNCH;
}

}  // extern "C"

// ====================================================================== allocation-free entry
// For callers that may not allocate device memory: the stream-K scratch of
// gb_gemm_noalloc is this array, sized for devices of up to kNoAllocMaxSms SMs.  It is
// zero at module load; its flag region is cleared once more at set-up.
namespace {
constexpr int kNoAllocMaxSms = 160;
constexpr int64_t kNoAllocFlagBytes = ((static_cast<int64_t>(kNoAllocMaxSms) * 4 + 255) / 256) * 256;
constexpr int64_t kNoAllocBytes =
    kNoAllocFlagBytes + static_cast<int64_t>(kNoAllocMaxSms) * gb::kSlotFloats * 4;
void* g_noalloc_ptr[128] = {};   // device address of the array, per device, after set-up
}  // namespace

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

extern "C" gb_status gb_gemm_noalloc(int dtype, int64_t M, int64_t N, int64_t K, float alpha,
                                     const void* A, int64_t lda, int majorA, const void* B,
                                     int64_t ldb, int majorB, float beta, const void* C, void* D,
                                     void* stream) {
  if (dtype != GB_F16 && dtype != GB_BF16) return GB_ERR_INVALID_ARG;
  DeviceState* dev;
  gb_status st = device_state(&dev);
  if (st != GB_OK) return st;
  if (workspace_bytes_for(dev->sms) > kNoAllocBytes) return GB_ERR_SCRATCH_LIMIT;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= 128) return GB_ERR_CUDA;
  void* scratch;
  {
    // set-up, once per device, with that device current: host code cannot use the array's
    // name as an address, so ask the runtime for it
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_noalloc_ptr[device] == nullptr) {
      void* ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) return GB_ERR_CUDA;
      // the hand-off flags start at zero (no launch number): the array is zero when the module
      // loads, and is cleared once more here, in stream order before this call's kernel
      const size_t flag_bytes =
          static_cast<size_t>(workspace_bytes_for(dev->sms) - dev->sms * int64_t(gb::kSlotFloats) * 4);
      if (cudaMemsetAsync(ptr, 0, flag_bytes, static_cast<cudaStream_t>(stream)) != cudaSuccess) return GB_ERR_CUDA;
      g_noalloc_ptr[device] = ptr;
    }
    scratch = g_noalloc_ptr[device];
  }
  return gemm_entry(dtype, M, N, K, alpha, A, lda, majorA, B, ldb, majorB, beta, C, D, scratch,
                    static_cast<size_t>(kNoAllocBytes), stream);
}
