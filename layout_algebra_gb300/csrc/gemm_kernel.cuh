// Device side of the persistent tcgen05 GEMM: configuration, shared-memory control
// block, bounded waits, the copy / MMA / epilogue roles and the kernel template, plus
// the host launchers' declarations.  Kernel instances are compiled in separate
// translation units (gemm_inst.cu) so that the build runs in parallel.
#pragma once

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
#include "ptx.cuh"

namespace gb {

constexpr int kBN = 256;             // N of one MMA instruction (and the single variant's tile)
constexpr int kWideTileN = 512;      // output tile columns of the wide CTA-pair shape
constexpr int kWide448TileN = 448;   // ... and of its 2 x 224-column form (K-major B)
constexpr int kBK = 64;              // one 128-byte swizzle row of 16-bit elements
constexpr int kRowsA = 128;          // A rows staged per CTA (one MMA's M per SM)
constexpr int kUmmaK = 16;           // K of one kind::f16 MMA
constexpr int kSwz = 64;             // elements per 128-byte swizzle span
constexpr int kChunkBytes = kSwz * kBK * 2;   // one 64-wide MN-major box: 64 K-rows x 128 B
constexpr int kTmemCols = 512;       // all of Tensor Memory: accumulators of 512 fp32 columns
constexpr int kCtlBytes = 1024;
constexpr int kMaxStages = 8;
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;

// The kernel variants share all code:
//  single (kPair = false): one CTA per 128 x 256 tile, 4 stages of A 128x64 + B 256x64, two
//         256-column accumulators in TMEM (the epilogue of one tile overlaps the main loop of
//         the next); narrow single-CTA tiles of 128 x 64 for outputs with few columns;
//  pair   (kPair = true):  a cluster of two CTAs on two SMs per 256 x 256 (or 256 x 224) tile;
//         the even CTA issues tcgen05.mma.cta_group::2 (M = 256) reading both CTAs' shared
//         memory, and each CTA's TMEM holds its own 128 rows of the accumulator.  Each CTA
//         stages its 128 A rows and its half of the tile's B rows, two k-blocks per stage.
//  wide pair (kShapeW512, kShapeW448): the pair with 256 x 512 (or 256 x 448) tiles: each
//         k-block of A feeds two MMAs of 256 (224) columns, so a CTA copies 48 KiB per 2 x 128 x 256 x 64 MMA work instead of
//         32 KiB per half of it (a third fewer copied bytes per flop, which is what bounds the
//         pair's main loop).  The accumulator then fills TMEM: the epilogue of a tile does not
//         overlap the next tile's main loop, so eight epilogue warps (two per TMEM lane
//         quarter) share it, storing D through staging tiles and reading C into registers.
// Input kinds: 16-bit (fp16/bf16, kind::f16), FP8 (kind::f8f6f4) and block-scaled FP8
// (kind::mxf8f6f4 with one E8M0 scale per 32 K elements of each row of A and column of B).
enum : int { kIn16 = 0, kIn8 = 1, kInMx = 2 };

// Block-scaled FP8 uses 224-column tiles: two accumulators (at TMEM columns 0 and 256) and,
// in the 32 columns behind each, two slots of scale factors (4 columns for A's 128 rows, 8
// for B's columns), so the epilogue still overlaps the next tile.
constexpr int kMxTileN = 224;
constexpr int kMxSfBytes = 512 + 1024;   // one k-block's scales: A's atom, then B's two atoms

// Kernel shapes: the standard tiles, narrow single-CTA tiles (128 x 64) for problems with few
// output columns, CTA-pair tiles of 256 x 224 (for problems whose 256-column tiles leave a
// ragged last wave) and the wide CTA-pair tiles of 256 x 512 and 256 x 448.  No shape loads a
// tile into several CTAs at once (no copy multicast).
enum : int { kShapeStd = 0, kShapeNarrow = 1, kShapeN224 = 2, kShapeW512 = 3, kShapeW448 = 4 };
constexpr int kNarrowTileN = 64;

template <bool kPair, int kIn = kIn16, int kShape = kShapeStd>
struct Cfg {
  static constexpr bool kMx = kIn == kInMx;
  static constexpr bool kNarrow = kShape == kShapeNarrow;
  static constexpr bool kN224 = kShape == kShapeN224;
  static constexpr bool kW512 = kShape == kShapeW512;
  static constexpr bool kW448 = kShape == kShapeW448;
  static constexpr int kTileM = kPair ? 256 : 128;
  static constexpr int kTileN =
      kNarrow ? kNarrowTileN
              : ((kMx || kN224) ? kMxTileN : (kW512 ? kWideTileN : (kW448 ? kWide448TileN : kBN)));
  static constexpr int kNSub = kW448 ? 2 : (kTileN > kBN ? kTileN / kBN : 1);   // MMAs per K step (along N)
  static constexpr int kMmaN = kTileN / kNSub;                     // N of one MMA
  static constexpr int kRowsBSub = kPair ? kMmaN / 2 : kMmaN;     // B rows a CTA stages per MMA
  static constexpr int kRowsB = kRowsBSub * kNSub;                // B rows a CTA stages per k-block
  static constexpr int kAccBufs = (kMx || kTmemCols / kTileN >= 2) ? 2 : 1;   // accumulators in TMEM
  static constexpr int kAccStride = (kMx || kN224) ? 256 : kTileN;   // TMEM columns between them
  static constexpr int kKB = (kPair && kNSub == 1) ? 2 : 1;       // k-blocks per stage
  // narrow tiles: 24 KiB k-blocks, eight in flight
  // 448-column pair tiles: five 44 KiB stages, the epilogue staging entirely in borrowed stages
  static constexpr int kStages = kNarrow ? 8 : ((kPair && kNSub == 1) ? 3 : (kW448 ? 5 : 4));
  static constexpr bool kEpiOwn = !kW448;   // staging tiles of its own beside the stages
  static constexpr int kEpiWarps = kAccBufs == 1 ? 8 : 4;
  static constexpr int kThreads = 64 + 32 * kEpiWarps;            // producer, MMA, epilogue warps
  static constexpr int kAHalf = kRowsA * kBK * 2;                // one k-block of A (bytes)
  static constexpr int kBSub = kRowsBSub * kBK * 2;              // one k-block of one MMA's B rows
  static constexpr int kBHalf = kRowsB * kBK * 2;                // one k-block of B (bytes)
  static constexpr int kSfBytes = kMx ? kMxSfBytes : 0;          // one k-block's scale factors
  static constexpr int kAStage = kAHalf * kKB;
  static constexpr int kBStage = kBHalf * kKB;
  static constexpr int kSfOff = kAStage + kBStage;               // scale factors after A and B
  // stage bases stay 1024-byte aligned (the swizzle atom)
  static constexpr int kStageBytes = ((kSfOff + kSfBytes * kKB) + 1023) / 1024 * 1024;
  // Tile-store epilogue: per epilogue warp two 32 x 32 staging tiles of D (16-bit, 64-byte
  // rows) written back by tensor copies and, with two accumulators, two of C read in the same
  // way (kEpiCTma); with one accumulator (eight epilogue warps) C is copied into the D staging
  // tiles themselves (or into borrowed stages, below), which halves the staging.  Used when it
  // fits.
  static constexpr int kEpiBufBytes = 32 * 64;
  static constexpr bool kEpiCTma = kAccBufs == 2;
  static constexpr int kEpiBufsPerWarp = kEpiCTma ? 4 : 2;
  static constexpr int kEpiStageBytesFull = kEpiOwn ? kEpiWarps * kEpiBufsPerWarp * kEpiBufBytes : 0;
  static constexpr bool kEpiTma =
      1024 + kStages * kStageBytes + kEpiStageBytesFull + kCtlBytes <= 227 * 1024;
  static constexpr int kEpiStageBytes = kEpiTma ? kEpiStageBytesFull : 0;
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kEpiStageBytes + kCtlBytes;
  static constexpr uint32_t kAccEmptyArrivals = kEpiWarps * (kPair ? 2 : 1);
  // Wide pair forms: during a tile's epilogue the two ring stages that held its last two
  // k-blocks are idle (the next tile's copies go into the other two first), so each warp
  // borrows kRingBufs staging tiles in each of them: with its own two, every run of the tile
  // (up to kEpiNB) has a staging tile of its own and C is copied in several runs ahead.
  // (448 columns: no staging of its own; the warps' tiles are packed across both borrowed
  // stages, kRingTiles per stage)
  static constexpr int kRingFit = kStageBytes / (kEpiWarps * kEpiBufBytes);
  static constexpr int kRingBufs = (kW512 || kW448) ? (kRingFit < 3 ? kRingFit : 3) : 0;
  static constexpr int kRingTiles = kStageBytes / kEpiBufBytes;
  static constexpr int kEpiNB = kEpiOwn ? 2 + 2 * kRingBufs : (2 * kRingTiles) / kEpiWarps;
  static constexpr int kSlotFloats = kRowsA * kTileN;       // one CTA's stream-K partial
  static_assert(kSmemBytes <= 227 * 1024, "shared-memory budget per CTA");
  static_assert(kStages <= kMaxStages, "control block");
  static_assert(kAccBufs >= 1 && kAccBufs <= 2 && kTileN % kNSub == 0, "TMEM accumulators");
  static_assert(!kMx || (kTileN <= 224 && kTileN % 32 == 0 && kBSub % 1024 == 0), "MX tile");
  static_assert(!kNarrow || (!kPair && !kMx), "narrow tiles: single CTA, 16-bit or FP8 inputs");
  static_assert(!kN224 || (kPair && !kMx), "224-column tiles: CTA pair, 16-bit or FP8 inputs");
  static_assert(!kW512 || (kPair && !kMx && kAccBufs == 1), "512-column tiles: CTA pair, 16-bit or FP8 inputs");
  static_assert(!kW448 || (kPair && !kMx && kAccBufs == 1 && kMmaN == kMxTileN && kBSub % 1024 == 0),
                "448-column tiles: CTA pair, two 224-column MMAs, 16-bit or FP8 inputs");
};
static_assert(kBK == kSwz, "a K-major stage row is exactly one swizzle span");

struct Params {
  int32_t M, N, K;
  int32_t m_tiles, n_tiles, k_blocks, num_tiles, group_m;
  int32_t majorA, majorB;     // 0: K-major, 1: MN-major
  float alpha, beta;
  const uint16_t* C;
  uint16_t* D;
  int64_t d_grid_m, d_grid_n; // D/C offset per tile step (grid mode of the divide)
  int64_t d_row, d_col;       // D/C offset per element step (tile mode of the divide)
  uint32_t idesc;
  int32_t vec_ok, has_c;
  uint64_t timeout_ns;
  int64_t skip_kb;
  // stream-K schedule: each CTA (pair) first runs data-parallel tiles t = c, c + G, ... <
  // dp_tiles, then an even, contiguous share of the remaining (tile, stage-block) units.
  int32_t nsb;                // stage-blocks per tile
  int32_t dp_tiles;           // tiles run whole; == num_tiles when stream-K is off
  uint32_t epoch;             // launch number, written to the partial-ready flags
  float* ws_part;             // per CTA slot: one 128 x 256 fp32 partial accumulator
  uint32_t* ws_flags;         // per CTA slot: epoch of the last partial written
  // fused epilogue ("CUTLASS, in depth" — "Epilogue fusion"): v = alpha*acc + beta*c,
  // v += bias[column], v = act(v), amax = max |v|, D = v (16-bit) or sat_fp8(v * out_scale)
  int32_t fused;              // 0: plain alpha/beta epilogue
  const uint16_t* bias;       // N values of the input type, or null
  int32_t act;                // 0 none, 1 ReLU, 2 GELU (erf form)
  float* amax;                // device float receiving max |v| (by atomic max), or null
  int32_t out_fmt;            // 0 same 16-bit type as the inputs, 1 FP8 E4M3, 2 FP8 E5M2
  float out_scale;
  int32_t vec8_ok;            // 16-byte FP8 stores legal (N % 16 == 0)
  int32_t bk_elems;           // K elements of one k-block: 64 (16-bit inputs), 128 (8-bit)
  uint32_t* status;           // device status word: first failing wait, 0 if none
  // bit 0 (A), bit 1 (B): one copy moves all kKB k-blocks of the operand's stage (CTA pair,
  // K a multiple of the k-block).  K-major: a three-dimensional map (k-block elements, rows,
  // k-blocks); MN-major (rows a multiple of 64): four-dimensional (64 MN elements, K rows of
  // a k-block, 64-wide MN chunks, k-blocks).  Otherwise one two-dimensional copy per k-block.
  int32_t kb_boxes;
  // k-blocks the stage-deep maps cover (K / bk rounded down): a stage reaching past them
  // (the tail of a K that is not a multiple of the k-block) is copied per k-block through
  // the two-dimensional tail maps instead; == k_blocks when K is a multiple
  int32_t kb_full;
  // 1: the epilogue stages each 32 x 32 run of D in shared memory and writes it with a
  // tensor copy (tmD), and reads C the same way (tmC); 16-bit D, row-major, N % 8 == 0
  int32_t epi_tma;
};

// Largest stream-K slot of any variant (floats): sizes the workspace, and is the slot pitch of
// every variant.
constexpr int kSlotFloats = kRowsA * kWideTileN;

struct Ctl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t drain;
  uint64_t part_done;         // epilogue warps finished writing a stream-K partial
  uint64_t fix_done;          // epilogue warps finished reading other CTAs' partials
  uint32_t tmem_base;
  int32_t abort;
  uint32_t* status;           // copy of Params::status for the wait helpers
  uint64_t c_full[8][8];      // tile-store epilogue: C staging tile landed (per warp, buffer)
  uint64_t epi_ring;          // epilogue warps done with the ring stages they borrowed
};
static_assert(sizeof(Ctl) <= kCtlBytes, "control block");
static_assert(kCtlBytes % 8 == 0, "control block alignment");

enum : uint32_t {
  kSiteEmpty = 1,     // copy stage waiting for a free ring slot
  kSiteFull = 2,      // MMA waiting for a k-block to land
  kSiteAccEmpty = 3,  // MMA waiting for the epilogue to free an accumulator
  kSiteAccFull = 4,   // epilogue waiting for a finished accumulator
  kSiteDrain = 5,     // abort path: waiting for own operations in flight
  kSiteTail = 6,      // copy stage waiting for the last releases before exit
  kSiteFixup = 7,     // tile owner waiting for another CTA's stream-K partial
  kSiteEpiC = 8,      // epilogue waiting for a C tile copied into its staging buffer
  kSiteRing = 9,      // copy stage waiting for the epilogue to return borrowed ring stages
};

// The epilogue borrows ring stages (wide pair forms, with C: its copies then run several runs
// ahead; 448-column tiles always, having no staging of their own): every tile is whole (no
// stream-K) and has at least kStages stage-blocks, so the copy stage reaches the borrowed stages
// only with stage-block kStages - 2 of the next tile, and waits there for their return.
// (Without C the two staging tiles of a 512-column tile's warp suffice; the hold-off of the next
// tile's copies would cost more than it saves.)
template <class C>
__device__ __forceinline__ bool ring_epilogue(const Params& p) {
  return C::kRingBufs > 0 && C::kEpiTma && p.epi_tma != 0 && (p.has_c != 0 || !C::kEpiOwn) &&
         p.dp_tiles == p.num_tiles && p.nsb >= C::kStages;
}

// Record the first failing wait, and stop this CTA (and its peer, in a pair).
template <bool kPair>
__device__ __forceinline__ void raise_status(Ctl* ctl, uint32_t site) {
  atomicCAS(ctl->status, 0u, site | (blockIdx.x << 8));
  *reinterpret_cast<volatile int32_t*>(&ctl->abort) = 1;
  if constexpr (kPair) {
    const uint32_t me = cluster_ctarank(), n = cluster_nctarank();
    for (uint32_t c = 0; c < n; ++c)
      if (c != me) st_cluster_u32(map_to_cta(smem_addr(&ctl->abort), c), 1u);
  }
}

__device__ __forceinline__ bool aborted(Ctl* ctl) {
  return *reinterpret_cast<volatile int32_t*>(&ctl->abort) != 0;
}

template <bool kCluster>
__device__ __forceinline__ bool probe(uint32_t bar, uint32_t parity) {
  if constexpr (kCluster)
    return mbar_try_wait_cluster(bar, parity);
  else
    return mbar_try_wait(bar, parity);
}

// Single-thread bounded wait; gives up on the abort flag or the time limit.  kCluster
// selects a cluster-scope acquire: needed only where the arrivals are plain thread
// arrivals from the peer CTA; barriers completed by copies or tcgen05.commit are
// waited at CTA scope.
template <bool kPair, bool kCluster = false>
__device__ __noinline__ bool wait_one_slow(uint32_t bar, uint32_t parity, Ctl* ctl, uint64_t limit,
                                           uint32_t site) {
  if (probe<kCluster>(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t n = 1;; ++n) {
    if (probe<kCluster>(bar, parity)) return true;
    if ((n & 7) == 0) {
      if (aborted(ctl)) return false;
      if (global_timer_ns() - t0 > limit) {
        raise_status<kPair>(ctl, site);
        return false;
      }
    }
  }
}

// The common case (already complete) stays inline: one probe, no call.  Measured: the
// per-stage hand-off cost of the call alone was ~5 % of an 8192^3 GEMM.
template <bool kPair, bool kCluster = false>
__device__ __forceinline__ bool wait_one(uint32_t bar, uint32_t parity, Ctl* ctl, uint64_t limit,
                                         uint32_t site) {
  if (probe<kCluster>(bar, parity)) return true;
  return wait_one_slow<kPair, kCluster>(bar, parity, ctl, limit, site);
}

// Bounded wait that ignores the abort flag (used to drain own work after an abort).
static __device__ __noinline__ bool wait_drain(uint32_t bar, uint32_t parity, uint64_t limit, uint32_t* status) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > limit) {
      atomicCAS(status, 0u, kSiteDrain | (blockIdx.x << 8));
      return false;
    }
  }
  return true;
}

// Warp-collective bounded wait with a warp-uniform outcome.
template <bool kPair>
__device__ __noinline__ bool wait_warp(uint32_t bar, uint32_t parity, Ctl* ctl, uint64_t limit,
                                       uint32_t site) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t n = 0;; ++n) {
    const bool ok = probe<false>(bar, parity);
    if (__all_sync(0xffffffffu, ok)) return true;
    if ((n & 7) == 7) {
      int stop = 0;
      if ((threadIdx.x & 31) == 0) {
        if (aborted(ctl)) {
          stop = 1;
        } else if (global_timer_ns() - t0 > limit) {
          raise_status<kPair>(ctl, site);
          stop = 1;
        }
      }
      if (__shfl_sync(0xffffffffu, stop, 0)) return false;
    }
  }
}

// Grouped raster order: runs of group_m M-tiles, walked down M first, then across N,
// so that CTAs working at the same time share A rows and B columns in L2 ("CUTLASS, in
// depth" — "Kernel schedules", rasterisation).  Odd groups walk N backwards, so a group
// starts on the B columns the previous one ended on (still in L2).
__device__ __forceinline__ void raster(int32_t t, int32_t m_tiles, int32_t n_tiles, int32_t group_m,
                                       int32_t& mt, int32_t& nt) {
  const int32_t per_group = group_m * n_tiles;
  const int32_t g = t / per_group;
  const int32_t first_m = g * group_m;
  const int32_t gm = min(m_tiles - first_m, group_m);
  const int32_t local = t - g * per_group;
  mt = first_m + local % gm;
  nt = local / gm;
  if (g & 1) nt = n_tiles - 1 - nt;
}

__device__ __forceinline__ void tile_coords(const Params& p, int32_t t, int32_t& mt, int32_t& nt) {
  raster(t, p.m_tiles, p.n_tiles, p.group_m, mt, nt);
}

// One unit of work: stage-blocks [sb0, sb1) of tile `tile`.
struct Item {
  int32_t tile, sb0, sb1;
};

// The work list of one CTA (or pair), walked identically by the copy, MMA and epilogue
// roles.  Stream-K part: the U = (num_tiles - dp_tiles) * nsb remaining units are cut
// into G contiguous ranges [c*U/G, (c+1)*U/G); an item never crosses a tile boundary.
struct Sched {
  int32_t dp_next;
  int64_t u, u_end;
  __device__ __forceinline__ void init(const Params& p, uint32_t c, uint32_t G) {
    dp_next = static_cast<int32_t>(c);
    const int64_t U = static_cast<int64_t>(p.num_tiles - p.dp_tiles) * p.nsb;
    u = U * c / G;
    u_end = U * (c + 1) / G;
  }
  __device__ __forceinline__ bool next(const Params& p, uint32_t G, Item& it) {
    if (dp_next < p.dp_tiles) {
      it.tile = dp_next;
      it.sb0 = 0;
      it.sb1 = p.nsb;
      dp_next += static_cast<int32_t>(G);
      return true;
    }
    if (u >= u_end) return false;
    const int64_t gu = static_cast<int64_t>(p.dp_tiles) * p.nsb + u;
    it.tile = static_cast<int32_t>(gu / p.nsb);
    it.sb0 = static_cast<int32_t>(gu % p.nsb);
    const int64_t span = u_end - u, room = p.nsb - it.sb0;
    it.sb1 = it.sb0 + static_cast<int32_t>(span < room ? span : room);
    u += it.sb1 - it.sb0;
    return true;
  }
};

// The CTA (pair) whose stream-K range holds unit index `gu` (counted over all tiles).
__device__ __forceinline__ uint32_t sk_owner_of(const Params& p, uint32_t G, int64_t gu) {
  const int64_t U = static_cast<int64_t>(p.num_tiles - p.dp_tiles) * p.nsb;
  const int64_t v = gu - static_cast<int64_t>(p.dp_tiles) * p.nsb;
  return static_cast<uint32_t>(((v + 1) * G + U - 1) / U - 1);
}

// True when CTA (pair) c's stream-K range holds at least one unit (with fewer units than
// CTAs some ranges are empty, and those CTAs hand nothing over).
__device__ __forceinline__ bool sk_has_units(const Params& p, uint32_t G, uint32_t c) {
  const int64_t U = static_cast<int64_t>(p.num_tiles - p.dp_tiles) * p.nsb;
  return U * (c + 1) / G > U * c / G;
}

// C/D offset of in-tile element (r, c) of tile (mt, nt): the divided layout evaluated.
__device__ __forceinline__ int64_t d_offset(const Params& p, int32_t mt, int32_t nt, int32_t r,
                                            int32_t c) {
  return mt * p.d_grid_m + nt * p.d_grid_n + r * p.d_row + c * p.d_col;
}

// Copies of one k-block of one operand, `rows` rows starting at row0.  K-major: one box of
// 64 (K) x rows.  MN-major: rows/64 boxes of 64 (M or N) x 64 (K), 8 KiB each, back to back.
template <bool kPair>
__device__ __forceinline__ void issue_operand(int major, const void* tm, uint32_t dst, uint32_t bar,
                                              int32_t row0, int rows, int32_t kb, int32_t bk_elems) {
  if (major == 0) {
    // a K-major k-block is one 128-byte swizzle row per operand row: 64 16-bit or 128
    // 8-bit elements
    if constexpr (kPair)
      tma_load_2d_pair(dst, tm, bar, kb * bk_elems, row0);
    else
      tma_load_2d(dst, tm, bar, kb * bk_elems, row0);
  } else {
    for (int j = 0; j < rows / kSwz; ++j) {
      if constexpr (kPair)
        tma_load_2d_pair(dst + j * kChunkBytes, tm, bar, row0 + j * kSwz, kb * kBK);
      else
        tma_load_2d(dst + j * kChunkBytes, tm, bar, row0 + j * kSwz, kb * kBK);
    }
  }
}

// Shared-memory descriptor of the k-th K=16 slice of a stage operand.
//  K-major, 128-byte swizzle: rows of 128 B, 8-row atoms 1024 B apart (stride offset);
//    the leading offset is unused; the k-th slice starts 32 B further along the row.
//  MN-major, 128-byte swizzle: 64-element MN chunks one box (8 KiB) apart (leading
//    offset), 8-row K groups 1024 B apart (stride offset); the k-th slice starts 16 rows
//    (2 KiB) further down.
__device__ __forceinline__ uint64_t operand_desc(uint32_t base, int major, int k) {
  if (major == 0) return smem_desc_sw128(base + k * (kUmmaK * 2), 16, 1024);
  return smem_desc_sw128(base + k * (kUmmaK * 128), kChunkBytes, 1024);
}

template <bool kPair, int kIn, int kShape>
__device__ void run_producer(const Params& p, const void* tmA, const void* tmB, const void* tmSFA,
                             const void* tmSFB, const void* tmAt, const void* tmBt, uint8_t* smem, Ctl* ctl,
                             uint32_t rank, uint32_t cluster, uint32_t nclusters) {
  using C = Cfg<kPair, kIn, kShape>;
  const uint32_t prank = rank & 1u;   // rank in the pair; the even CTA leads
  // stage-deep copies: CTA pairs, one MMA per k-block along N
  constexpr bool kStageBoxes = kPair && C::kNSub == 1 && C::kKB > 1;
  int stage = 0;
  uint32_t phase = 0;
  int64_t gkb = 0;
  uint32_t issued = 0, issued_parity = 0;
  bool ok = true;
  const bool ring = ring_epilogue<C>(p);
  int32_t it = 0;
  Sched sched;
  sched.init(p, cluster, nclusters);
  Item item;
  for (; ok && sched.next(p, nclusters, item); ++it) {
    int32_t mt, nt;
    tile_coords(p, item.tile, mt, nt);
    const int32_t a_row0 = mt * C::kTileM + static_cast<int32_t>(prank) * kRowsA;
    const int32_t b_row0 = nt * C::kTileN + static_cast<int32_t>(prank) * C::kRowsBSub;
    for (int32_t sb = item.sb0; sb < item.sb1; ++sb, ++gkb) {
      // the previous tile's epilogue holds the stages of its last two k-blocks, which this
      // tile's stage-blocks kStages - 2 and kStages - 1 are about to reuse
      if (ring && it > 0 && sb == item.sb0 + C::kStages - 2 &&
          !wait_one<kPair>(smem_addr(&ctl->epi_ring), static_cast<uint32_t>((it - 1) & 1), ctl, p.timeout_ns,
                           kSiteRing)) {
        ok = false;
        break;
      }
      if (!wait_one<kPair>(smem_addr(&ctl->empty[stage]), phase ^ 1u, ctl, p.timeout_ns, kSiteEmpty)) {
        ok = false;
        break;
      }
      if (gkb != p.skip_kb) {
        const uint32_t full = smem_addr(&ctl->full[stage]);
        // in a pair both CTAs' copies are counted on the even CTA's barrier
        const uint32_t full_tgt = kPair ? map_to_cta(full, 0) : full;
        const uint32_t sa = smem_addr(smem + stage * C::kStageBytes);
        // the last stage of a tile may hold fewer k-blocks: copy and count only those (a
        // stage-deep copy always lands whole, its k-blocks past K zero-filled)
        const int nkb = min(C::kKB, p.k_blocks - sb * C::kKB);
        bool a3 = false, b3 = false;
        // operands with stage-deep maps copy a stage reaching past the maps' k-blocks (a K
        // tail) per k-block through their two-dimensional tail maps
        const void* tmA1 = tmA;
        const void* tmB1 = tmB;
        if constexpr (kStageBoxes) {
          const bool whole = sb * C::kKB + C::kKB <= p.kb_full || p.kb_full == p.k_blocks;
          a3 = whole && (p.kb_boxes & 1) != 0;
          b3 = whole && (p.kb_boxes & 2) != 0;
          if (p.kb_boxes & 1) tmA1 = tmAt;
          if (p.kb_boxes & 2) tmB1 = tmBt;
        }
        if (!kPair || prank == 0) {
          // scale factors always arrive for the whole stage (one copy per operand)
          const uint32_t tx = (C::kAHalf * (a3 ? C::kKB : nkb) + C::kBHalf * (b3 ? C::kKB : nkb) +
                               C::kSfBytes * C::kKB) * (kPair ? 2u : 1u);
          mbar_arrive_expect_tx(full, tx);
        }
        if constexpr (kStageBoxes) {
          if (a3) {
            if (p.majorA == 0)
              tma_load_3d_pair(sa, tmA, full_tgt, 0, a_row0, sb * C::kKB);
            else
              tma_load_4d_pair(sa, tmA, full_tgt, 0, 0, a_row0 / kSwz, sb * C::kKB);
          }
          if (b3) {
            if (p.majorB == 0)
              tma_load_3d_pair(sa + C::kAStage, tmB, full_tgt, 0, b_row0, sb * C::kKB);
            else
              tma_load_4d_pair(sa + C::kAStage, tmB, full_tgt, 0, 0, b_row0 / kSwz, sb * C::kKB);
          }
        }
        for (int h = 0; h < nkb; ++h) {
          const int32_t kb = sb * C::kKB + h;
          if (!a3)
            issue_operand<kPair>(p.majorA, tmA1, sa + h * C::kAHalf, full_tgt, a_row0, kRowsA, kb,
                                 p.bk_elems);
          if (!b3) {
            // per MMA along N: this CTA's rows of that MMA's 256 tile columns
#pragma unroll
            for (int j = 0; j < C::kNSub; ++j)
              issue_operand<kPair>(p.majorB, tmB1, sa + C::kAStage + h * C::kBHalf + j * C::kBSub,
                                   full_tgt, b_row0 + j * C::kMmaN, C::kRowsBSub, kb, p.bk_elems);
          }
        }
        if constexpr (C::kMx) {
          // scale factors, packed in 512-byte atoms (two 256-byte rows of the scale maps) that
          // are consecutive in k-blocks: one copy of A's kKB atoms of this CTA's 128 rows, then
          // one of B's 2 kKB atoms of the tile's columns (every CTA of a pair holds all of
          // them); past a tile's last k-block the copy reads unused atoms (or zero fill)
          const uint32_t sf = sa + C::kSfOff;
          const int32_t kb0 = sb * C::kKB;
          const int32_t rb = a_row0 / kRowsA;
          const int32_t ya = 2 * (rb * p.k_blocks + kb0), yb = 4 * (nt * p.k_blocks + kb0);
          if constexpr (kPair) {
            tma_load_2d_pair(sf, tmSFA, full_tgt, 0, ya);
            tma_load_2d_pair(sf + C::kKB * 512, tmSFB, full_tgt, 0, yb);
          } else {
            tma_load_2d(sf, tmSFA, full_tgt, 0, ya);
            tma_load_2d(sf + C::kKB * 512, tmSFB, full_tgt, 0, yb);
          }
        }
        issued |= 1u << stage;
        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
      } else {
        issued &= ~(1u << stage);
      }
      if (++stage == C::kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }
  if (ok) {
    // The consumer releases stages through asynchronous arrivals; wait for the last
    // kStages releases so that none lands after this CTA's shared memory is gone.
    for (int i = 0; i < C::kStages; ++i) {
      if (!wait_one<kPair>(smem_addr(&ctl->empty[stage]), phase ^ 1u, ctl, p.timeout_ns, kSiteTail)) break;
      if (++stage == C::kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
  } else if (!kPair || prank == 0) {
    for (int s = 0; s < C::kStages; ++s)
      if (issued & (1u << s))
        wait_drain(smem_addr(&ctl->full[s]), (issued_parity >> s) & 1u, p.timeout_ns, p.status);
  } else {
    // the odd CTA's copies complete on the even CTA's barrier, which it cannot observe;
    // a stage of 64 KiB lands in microseconds
    __nanosleep(200000);
  }
}

template <bool kPair, int kIn, int kShape>
__device__ void run_mma(const Params& p, uint8_t* smem, Ctl* ctl, uint32_t tmem_base, uint32_t rank,
                        uint32_t cluster, uint32_t nclusters) {
  using C = Cfg<kPair, kIn, kShape>;
  uint32_t kbc = 0;                        // k-blocks issued: selects the scale-factor slot
  if (kPair && (rank & 1u) != 0) return;   // the even CTA issues for the pair
  // a stage is free, and an accumulator full, for both CTAs of the pair at once
  constexpr uint16_t kPairMask = 0x3;
  int stage = 0;
  uint32_t phase = 0;
  bool ok = true, issued_any = false;
  int32_t it = 0;
  Sched sched;
  sched.init(p, cluster, nclusters);
  Item item;
  for (; ok && sched.next(p, nclusters, item); ++it) {
    const int buf = C::kAccBufs == 2 ? (it & 1) : 0;
    const uint32_t use = C::kAccBufs == 2 ? ((it >> 1) & 1) : (it & 1);
    if (!wait_one<kPair, kPair>(smem_addr(&ctl->acc_empty[buf]), use ^ 1u, ctl, p.timeout_ns,
                                kSiteAccEmpty)) {
      ok = false;
      break;
    }
    tc_fence_after_sync();
    const uint32_t d_tmem = tmem_base + buf * C::kAccStride;
    for (int32_t sbk = item.sb0; sbk < item.sb1; ++sbk) {
      if (!wait_one<kPair>(smem_addr(&ctl->full[stage]), phase, ctl, p.timeout_ns, kSiteFull)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const uint32_t sa = smem_addr(smem + stage * C::kStageBytes);
      const uint32_t sb = sa + C::kAStage;
      const int nkb = min(C::kKB, p.k_blocks - sbk * C::kKB);
      // descriptors differ only in the start-address field (bits 0-13, bytes >> 4), which
      // never carries for shared-memory addresses: build one per operand, then add offsets
      const uint64_t da0 = operand_desc(sa, p.majorA, 0), db0 = operand_desc(sb, p.majorB, 0);
      const uint32_t ka = p.majorA == 0 ? (kUmmaK * 2) >> 4 : (kUmmaK * 128) >> 4;
      const uint32_t kb_ = p.majorB == 0 ? (kUmmaK * 2) >> 4 : (kUmmaK * 128) >> 4;
      for (int h = 0; h < nkb; ++h) {
        uint32_t sfa = 0, sfb = 0;
        if constexpr (C::kMx) {
          // this k-block's scale factors into a TMEM slot behind an accumulator (four slots of
          // 12 columns, two in the 32 columns behind each accumulator, rotate; copies and MMAs
          // of one thread execute in issue order)
          const uint32_t slot = tmem_base + C::kTileN + (kbc & 1u) * C::kAccStride + ((kbc >> 1) & 1u) * 16u;
          // the stage holds A's kKB atoms, then B's kKB atom pairs
          const uint32_t sfa_s = sa + C::kSfOff + h * 512;
          const uint32_t sfb_s = sa + C::kSfOff + C::kKB * 512 + h * 1024;
          sfa = slot;
          sfb = slot + 4;
          if constexpr (kPair) {
            tc_cp_32x128b_x4_pair(sfa, smem_desc_plain(sfa_s, 0, 128));
            tc_cp_32x128b_x4_pair(sfb, smem_desc_plain(sfb_s, 0, 128));
            tc_cp_32x128b_x4_pair(sfb + 4, smem_desc_plain(sfb_s + 512, 0, 128));
          } else {
            tc_cp_32x128b_x4(sfa, smem_desc_plain(sfa_s, 0, 128));
            tc_cp_32x128b_x4(sfb, smem_desc_plain(sfb_s, 0, 128));
            tc_cp_32x128b_x4(sfb + 4, smem_desc_plain(sfb_s + 512, 0, 128));
          }
        }
        ++kbc;
#pragma unroll
        for (int k = 0; k < kBK / kUmmaK; ++k) {
          const uint64_t da = da0 + ((h * C::kAHalf) >> 4) + k * ka;
          const uint32_t acc = (sbk != item.sb0 || h != 0 || k != 0) ? 1u : 0u;
          // one instruction covers 32 bytes of K (16 16-bit or 32 8-bit elements) and up to
          // 256 columns; the N sub-tiles share the A slice
#pragma unroll
          for (int j = 0; j < C::kNSub; ++j) {
            const uint64_t db = db0 + ((h * C::kBHalf + j * C::kBSub) >> 4) + k * kb_;
            const uint32_t dt = d_tmem + j * C::kMmaN;
            if constexpr (C::kMx) {
              // the k-th 32-element slice takes scale byte k of each 32-bit scale cell
              const uint32_t id = p.idesc | (static_cast<uint32_t>(k) << 29) | (static_cast<uint32_t>(k) << 4);
              if constexpr (kPair)
                tc_mma_mx_pair(dt, da, db, id, sfa, sfb, acc);
              else
                tc_mma_mx(dt, da, db, id, sfa, sfb, acc);
            } else if constexpr (kPair && kIn == kIn8) {
              tc_mma_f8_pair(dt, da, db, p.idesc, acc);
            } else if constexpr (kPair) {
              tc_mma_f16_pair(dt, da, db, p.idesc, acc);
            } else if constexpr (kIn == kIn8) {
              tc_mma_f8(dt, da, db, p.idesc, acc);
            } else {
              tc_mma_f16(dt, da, db, p.idesc, acc);
            }
          }
        }
      }
      issued_any = true;
      if constexpr (kPair)
        tc_commit_pair_mc(smem_addr(&ctl->empty[stage]), kPairMask);
      else
        tc_commit(smem_addr(&ctl->empty[stage]));
      if (++stage == C::kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (!ok) break;
    const uint32_t af = smem_addr(&ctl->acc_full[buf]);
    if (p.k_blocks == 0) {
      mbar_arrive(af);
      if constexpr (kPair) mbar_arrive_cluster(map_to_cta(af, rank + 1));
    } else {
      if constexpr (kPair)
        tc_commit_pair_mc(af, kPairMask);
      else
        tc_commit(af);
    }
  }
  if (!ok && issued_any) {
    if constexpr (kPair)
      tc_commit_pair(smem_addr(&ctl->drain));
    else
      tc_commit(smem_addr(&ctl->drain));
    wait_drain(smem_addr(&ctl->drain), 0u, p.timeout_ns, p.status);
    __nanosleep(20000);   // let the arrivals of earlier commits land
  }
}

template <bool kBF16>
__device__ __forceinline__ float to_f32(uint16_t b) {
  if constexpr (kBF16)
    return __bfloat162float(__ushort_as_bfloat16(b));
  else
    return __half2float(__ushort_as_half(b));
}

template <bool kBF16>
__device__ __forceinline__ uint16_t from_f32(float v) {
  if constexpr (kBF16)
    return __bfloat16_as_ushort(__float2bfloat16_rn(v));
  else
    return __half_as_ushort(__float2half_rn(v));
}

// Two values rounded to nearest even and packed, lo in the low 16 bits: one paired
// conversion instruction (the same rounding as from_f32 on each value).
template <bool kBF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (kBF16) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
  } else {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
}

// beta * c added to v from 32 C values held as four 16-byte words.
template <bool kBF16>
__device__ __forceinline__ void add_c_words(const Params& p, const uint4 (&cw)[4], float (&v)[32]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t w[4] = {cw[j].x, cw[j].y, cw[j].z, cw[j].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      v[8 * j + 2 * e] = fmaf(p.beta, to_f32<kBF16>(static_cast<uint16_t>(w[e] & 0xffffu)), v[8 * j + 2 * e]);
      v[8 * j + 2 * e + 1] = fmaf(p.beta, to_f32<kBF16>(static_cast<uint16_t>(w[e] >> 16)), v[8 * j + 2 * e + 1]);
    }
  }
}

// 32 consecutive outputs of one row: v = alpha*acc (+ beta*c) in fp32.
template <bool kBF16>
__device__ __forceinline__ void epilogue_values(const Params& p, int64_t off, bool have_cw, const uint4 (&cw)[4],
                                                const uint32_t (&acc)[32],
                                                int valid, float (&v)[32]) {
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = p.alpha * __uint_as_float(acc[i]);
  if (!p.has_c) return;
  if (have_cw) {
    // 32 C values loaded ahead as four 16-byte words
    add_c_words<kBF16>(p, cw, v);
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i < valid) v[i] = fmaf(p.beta, to_f32<kBF16>(p.C[off + i * p.d_col]), v[i]);
  }
}

// Round v to the 16-bit output type and store it (16-byte stores when legal).
template <bool kBF16>
__device__ __forceinline__ void store_16(const Params& p, int64_t off, const float (&v)[32], int valid) {
  if (p.vec_ok && valid == 32) {
    uint4* dst = reinterpret_cast<uint4*>(p.D + off);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint4 u;
      u.x = pack2<kBF16>(v[8 * j + 0], v[8 * j + 1]);
      u.y = pack2<kBF16>(v[8 * j + 2], v[8 * j + 3]);
      u.z = pack2<kBF16>(v[8 * j + 4], v[8 * j + 5]);
      u.w = pack2<kBF16>(v[8 * j + 6], v[8 * j + 7]);
      dst[j] = u;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i < valid) p.D[off + i * p.d_col] = from_f32<kBF16>(v[i]);
  }
}

// v * out_scale to FP8 with saturation to the largest finite value (round to nearest even).
__device__ __forceinline__ uint32_t to_fp8(float x, int fmt) {
  return fmt == 1 ? static_cast<uint32_t>(__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3))
                  : static_cast<uint32_t>(__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E5M2));
}

__device__ __forceinline__ void store_fp8(const Params& p, int64_t off, const float (&v)[32], int valid) {
  uint8_t* d8 = reinterpret_cast<uint8_t*>(p.D);
  if (p.vec8_ok && valid == 32) {
    uint4* dst = reinterpret_cast<uint4*>(d8 + off);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int b = 16 * j + 4 * e;
        w[e] = to_fp8(v[b] * p.out_scale, p.out_fmt) | (to_fp8(v[b + 1] * p.out_scale, p.out_fmt) << 8) |
               (to_fp8(v[b + 2] * p.out_scale, p.out_fmt) << 16) |
               (to_fp8(v[b + 3] * p.out_scale, p.out_fmt) << 24);
      }
      dst[j] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i < valid) d8[off + i * p.d_col] = static_cast<uint8_t>(to_fp8(v[i] * p.out_scale, p.out_fmt));
  }
}

// The fused nodes on 32 consecutive outputs of one row (columns col0 .. col0+31): bias,
// activation, amax of the first `valid`.
template <bool kBF16>
__device__ __forceinline__ void fused_nodes(const Params& p, int valid, int64_t col0, float& amax, float (&v)[32]) {
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    if (p.bias != nullptr && i < valid) v[i] += to_f32<kBF16>(__ldg(p.bias + col0 + i));
    if (p.act == 1) v[i] = fmaxf(v[i], 0.0f);
    if (p.act == 2) v[i] = 0.5f * v[i] * (1.0f + erff(v[i] * 0.70710678118654752f));
    if (i < valid) amax = fmaxf(amax, fabsf(v[i]));
  }
}

// The epilogue of 32 consecutive outputs of one row, stored by this thread.
template <bool kBF16>
__device__ __forceinline__ void store_run(const Params& p, int64_t off, bool have_cw, const uint4 (&cw)[4],
                                          const uint32_t (&acc)[32], int valid, int64_t col0, float& amax) {
  float v[32];
  epilogue_values<kBF16>(p, off, have_cw, cw, acc, valid, v);
  if (p.fused) fused_nodes<kBF16>(p, valid, col0, amax, v);
  if (p.out_fmt == 0)
    store_16<kBF16>(p, off, v, valid);
  else
    store_fp8(p, off, v, valid);
}

// Staging tiles of the tile-store epilogue: 32 rows of 64 bytes (32 16-bit values), in the
// 64-byte swizzle of tensor copies: the 16-byte chunk j of row r sits at chunk
// j ^ ((r >> 1) & 3), so a warp writing (or reading) one row per lane spreads each 16-byte
// access over all banks.
__device__ __forceinline__ uint32_t stage64_offset(int row, int chunk) {
  return static_cast<uint32_t>(row * 64 + ((chunk ^ ((row >> 1) & 3)) << 4));
}

// Stream-K workspace slot of CTA (cluster c, rank r): a 128 x 256 fp32 partial stored
// column-major ([column][row]) so that a warp's 32 rows form one 128-byte access.
template <bool kPair>
__device__ __forceinline__ float* part_slot(const Params& p, uint32_t c, uint32_t rank) {
  return p.ws_part + (static_cast<int64_t>(c) * (kPair ? 2 : 1) + rank) * kSlotFloats;
}

template <bool kPair>
__device__ __forceinline__ uint32_t* part_flag(const Params& p, uint32_t c, uint32_t rank) {
  return p.ws_flags + static_cast<int64_t>(c) * (kPair ? 2 : 1) + rank;
}

// Warp-collective bounded wait until the partial-ready flags of the CTAs (pairs) c_lo..c_hi
// that hold stream-K units carry this launch's epoch.  The flags are spread over the lanes
// (lane l watches c_lo + l, c_lo + l + 32, ...), so one poll has all of them in flight
// instead of one round trip per flag; each lane's acquire load orders, and the warp barrier
// then passes on to every lane, the contributors' partials before the reads that follow.
template <bool kPair>
__device__ __noinline__ bool wait_flags(const Params& p, uint32_t G, uint32_t c_lo, uint32_t c_hi, uint32_t rank,
                                        Ctl* ctl) {
  const uint32_t lane = threadIdx.x & 31;
  uint32_t c = c_lo + lane;   // this lane's next flag still to be seen set
  uint64_t t0 = 0;
  for (uint32_t n = 0;; ++n) {
    // a flag seen set stays set for this launch (only this owner clears it, afterwards)
    while (c <= c_hi &&
           (!sk_has_units(p, G, c) || ld_acquire_gpu(part_flag<kPair>(p, c, rank)) == p.epoch))
      c += 32;
    if (__all_sync(0xffffffffu, c > c_hi)) break;
    if ((n & 63) == 63) {
      int stop = 0;
      if (lane == 0) {
        if (aborted(ctl)) {
          stop = 1;
        } else {
          const uint64_t now = global_timer_ns();
          if (t0 == 0) {
            t0 = now;
          } else if (now - t0 > p.timeout_ns) {
            raise_status<kPair>(ctl, kSiteFixup);
            stop = 1;
          }
        }
      }
      if (__shfl_sync(0xffffffffu, stop, 0)) return false;
    }
  }
  __syncwarp();
  return true;
}

// The next CTA (pair) at or after c, up to c_hi, whose stream-K range holds units (c_hi + 1
// if none).
__device__ __forceinline__ uint32_t next_contributor(const Params& p, uint32_t G, uint32_t c, uint32_t c_hi) {
  while (c <= c_hi && !sk_has_units(p, G, c)) ++c;
  return c;
}

// One 32-column run of the tile-store epilogue for this warp's 32 rows: C from its staging
// tile (tload_c: copied in two runs ahead into tiles of its own; cd_c: copied one run ahead into
// the D staging tile this run then writes), alpha/beta and the fused nodes, the 16-bit row
// written to the D staging tile, one tensor copy of the 32 x 32 tile to D (clipped at M and N),
// and the next C copy issued.  Returns false if a wait gave up.
template <bool kBF16, bool kPair>
__device__ __forceinline__ bool tile_store_run(const Params& p, Ctl* ctl, const uint32_t (&acc)[32], int ew,
                                               int lane, uint32_t stg, uint32_t& gr, uint32_t& c_phase,
                                               uint32_t& c_pending, bool tload_c, int run, int nruns, int32_t x0,
                                               int32_t y0, int valid, int64_t col0, float& amax, const void* tmC,
                                               const void* tmD, bool cd_c) {
  constexpr uint32_t kBuf = 32 * 64;
  const uint32_t b = gr & 1u;
  const uint32_t sd = stg + b * kBuf, sc = stg + (2 + b) * kBuf;
  float v[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = p.alpha * __uint_as_float(acc[i]);
  if (cd_c) {
    // this run's C tile, copied into the D staging tile before (every lane reads its row before
    // D is written there)
    if (!wait_warp<kPair>(smem_addr(&ctl->c_full[ew][b]), (c_phase >> b) & 1u, ctl, p.timeout_ns, kSiteEpiC))
      return false;
    c_phase ^= 1u << b;
    c_pending &= ~(1u << b);
    uint4 cw[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) cw[j] = ld_shared_u4(sd + stage64_offset(lane, j));
    add_c_words<kBF16>(p, cw, v);
    __syncwarp();
  }
  if (tload_c) {
    if (!wait_warp<kPair>(smem_addr(&ctl->c_full[ew][b]), (c_phase >> b) & 1u, ctl, p.timeout_ns, kSiteEpiC))
      return false;
    c_phase ^= 1u << b;
    c_pending &= ~(1u << b);
    uint4 cw[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) cw[j] = ld_shared_u4(sc + stage64_offset(lane, j));
    add_c_words<kBF16>(p, cw, v);
  }
  if (p.fused) fused_nodes<kBF16>(p, valid, col0, amax, v);
  // the copy that last read this D staging tile (two runs back) must be done with it
  if (lane == 0) bulk_wait_group_read<1>();
  __syncwarp();
#pragma unroll
  for (int j = 0; j < 4; ++j)
    st_shared_u4(sd + stage64_offset(lane, j),
                 make_uint4(pack2<kBF16>(v[8 * j + 0], v[8 * j + 1]), pack2<kBF16>(v[8 * j + 2], v[8 * j + 3]),
                            pack2<kBF16>(v[8 * j + 4], v[8 * j + 5]), pack2<kBF16>(v[8 * j + 6], v[8 * j + 7])));
  fence_proxy_async_smem();
  __syncwarp();
  const bool refill = tload_c && run + 2 < nruns;
  const bool next_c = cd_c && run + 1 < nruns;
  if (lane == 0) {
    tma_store_2d(tmD, sd, x0 + 32 * run, y0);
    bulk_commit_group();
    // this C tile is consumed (every lane passed the __syncwarp above): refill it with the
    // run two further on
    if (refill) {
      const uint32_t bar = smem_addr(&ctl->c_full[ew][b]);
      mbar_arrive_expect_tx(bar, kBuf);
      tma_load_2d(sc, tmC, bar, x0 + 32 * (run + 2), y0);
    }
    // the next run's C goes into the other D staging tile once the store of the run before
    // this one has read it
    if (next_c) {
      bulk_wait_group_read<1>();
      const uint32_t bar = smem_addr(&ctl->c_full[ew][b ^ 1u]);
      mbar_arrive_expect_tx(bar, kBuf);
      tma_load_2d(stg + (b ^ 1u) * kBuf, tmC, bar, x0 + 32 * (run + 1), y0);
    }
  }
  if (refill) c_pending |= 1u << b;
  if (next_c) c_pending |= 1u << (b ^ 1u);
  ++gr;
  return true;
}

// One 32-column run of the wide pair forms' epilogue with borrowed ring stages: run `run` of
// the tile uses staging tile b = run % NB (address buf(b)), whose C copy (if any) was issued
// several runs earlier; D is written over C in that tile and stored by one tensor copy; then
// the C copy of run + NB - 1 is issued into the tile of the run before this one once that
// run's store has read it.  Returns false if a wait gave up.
template <bool kBF16, bool kPair, int kNB, class BufAddr>
__device__ __forceinline__ bool ring_store_run(const Params& p, Ctl* ctl, const uint32_t (&acc)[32], int ew,
                                               int lane, const BufAddr& buf, uint32_t& c_phase,
                                               uint32_t& c_pending, int run, int nruns, int32_t x0, int32_t y0,
                                               int valid, int64_t col0, float& amax, const void* tmC,
                                               const void* tmD) {
  constexpr uint32_t kBuf = 32 * 64;
  const uint32_t b = static_cast<uint32_t>(run % kNB);
  const uint32_t sd = buf(b);
  float v[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = p.alpha * __uint_as_float(acc[i]);
  if (p.has_c) {
    if (!wait_warp<kPair>(smem_addr(&ctl->c_full[ew][b]), (c_phase >> b) & 1u, ctl, p.timeout_ns, kSiteEpiC))
      return false;
    c_phase ^= 1u << b;
    c_pending &= ~(1u << b);
    uint4 cw[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) cw[j] = ld_shared_u4(sd + stage64_offset(lane, j));
    add_c_words<kBF16>(p, cw, v);
    __syncwarp();
  } else if (run >= kNB) {
    // the store of run - NB, which read this staging tile, must be done with it
    if (lane == 0) bulk_wait_group_read<kNB - 1>();
    __syncwarp();
  }
  if (p.fused) fused_nodes<kBF16>(p, valid, col0, amax, v);
#pragma unroll
  for (int j = 0; j < 4; ++j)
    st_shared_u4(sd + stage64_offset(lane, j),
                 make_uint4(pack2<kBF16>(v[8 * j + 0], v[8 * j + 1]), pack2<kBF16>(v[8 * j + 2], v[8 * j + 3]),
                            pack2<kBF16>(v[8 * j + 4], v[8 * j + 5]), pack2<kBF16>(v[8 * j + 6], v[8 * j + 7])));
  fence_proxy_async_smem();
  __syncwarp();
  const int ahead = run + kNB - 1;
  const bool next_c = p.has_c && run >= 1 && ahead < nruns;
  if (lane == 0) {
    tma_store_2d(tmD, sd, x0 + 32 * run, y0);
    bulk_commit_group();
    if (next_c) {
      const uint32_t nb = static_cast<uint32_t>(ahead % kNB);
      bulk_wait_group_read<1>();   // the store of run - 1 has read tile nb
      const uint32_t bar = smem_addr(&ctl->c_full[ew][nb]);
      mbar_arrive_expect_tx(bar, kBuf);
      tma_load_2d(buf(nb), tmC, bar, x0 + 32 * ahead, y0);
    }
  }
  if (next_c) c_pending |= 1u << (ahead % kNB);
  return true;
}

template <bool kBF16, bool kPair, int kIn, int kShape>
__device__ void run_epilogue(const Params& p, Ctl* ctl, uint32_t tmem_base, int warp, int lane,
                             uint32_t rank, uint32_t cluster, uint32_t nclusters, uint8_t* epi_smem,
                             const void* tmC, const void* tmD) {
  using C = Cfg<kPair, kIn, kShape>;
  const uint32_t prank = rank & 1u;
  const int q = warp & 3;            // a warp may read TMEM lanes 32*(warp%4) .. +31
  const int lrow = q * 32 + lane;    // accumulator row in this CTA = TMEM lane
  // with eight epilogue warps two share a lane quarter and split the columns
  constexpr int kCols = C::kTileN / (C::kEpiWarps / 4);
  const int ew = warp - 2;           // epilogue warp index
  const int cbeg = (ew >> 2) * kCols;
  const int r = static_cast<int>(prank) * kRowsA + lrow;   // row within the tile
  constexpr int kRuns = kCols / 32;
  // Tile-store epilogue (p.epi_tma): this warp's staging tiles D0, D1, C0, C1 and the
  // barriers its C copies complete on.  Runs alternate between the two buffers by a count
  // kept across tiles (gr), so a buffer is rewritten only once the copy that last read it
  // (two runs earlier) has finished reading.
  // without staging of its own, the tile-store epilogue needs the borrowed stages
  const bool tma = C::kEpiTma && p.epi_tma != 0 && (C::kEpiOwn || ring_epilogue<C>(p));
  const uint32_t stg = smem_addr(epi_smem) + static_cast<uint32_t>(ew) * C::kEpiBufsPerWarp * C::kEpiBufBytes;
  // stream-K owner: this lane's column of this warp's share of the stage ring, where the
  // other CTAs' partials of a run are gathered (kPartBatch CTAs x 32 columns x 32 rows fp32)
  constexpr int kRingBytes = C::kStages * C::kStageBytes;
  constexpr int kPartBatch = kRingBytes / (C::kEpiWarps * 4096) < 8 ? kRingBytes / (C::kEpiWarps * 4096) : 8;
  static_assert(kPartBatch >= 1, "the stage ring holds one run of partials per epilogue warp");
  const uint32_t part_buf = smem_addr(epi_smem) - static_cast<uint32_t>(kRingBytes) +
                            static_cast<uint32_t>(ew) * kPartBatch * 4096u + static_cast<uint32_t>(lane) * 4u;
  uint32_t gr = 0, c_phase = 0;
  uint32_t c_pending = 0;            // staging buffers with a C copy issued, not yet waited for
  // borrowed ring stages (wide pair forms): the stages of the tile's last two k-blocks, found
  // from the stage-blocks this CTA's copy stage has issued up to the end of the tile
  const bool ring_ok = ring_epilogue<C>(p);
  int64_t sb_done = 0;
  int32_t it = 0;
  float amax = 0.0f;                 // this thread's max |v| (fused epilogue)
  Sched sched;
  sched.init(p, cluster, nclusters);
  Item item;
  for (; sched.next(p, nclusters, item); ++it) {
    int32_t mt, nt;
    tile_coords(p, item.tile, mt, nt);
    const bool row_ok = static_cast<int64_t>(mt) * C::kTileM + r < p.M;
    const int32_t cols_left = p.N - nt * C::kTileN;
    const int64_t base = d_offset(p, mt, nt, r, 0);
    const int cend = min(cbeg + kCols, static_cast<int>(min(cols_left, C::kTileN)));
    const int nruns = cend > cbeg ? (cend - cbeg + 31) / 32 : 0;
    // stream-K roles: a contributor holds later k-units of a tile and hands its partial
    // over; the owner (which holds k = 0) adds every contributor's partial.
    const bool contributor = item.sb0 > 0;
    const bool owner_with_parts = item.sb0 == 0 && item.sb1 < p.nsb;
    // tile-store path: the 32-row slab of this warp starts at row y0, its runs at x0 + 32 run
    const bool tstore = tma && !contributor;
    const bool ring = tstore && ring_ok;                      // staging in borrowed ring stages
    const bool tload_c = tstore && p.has_c && C::kEpiCTma;   // C by tensor copy into staging
    const bool cd_c = tstore && p.has_c && !C::kEpiCTma && !ring;   // C by tensor copy into the D tiles
    sb_done += item.sb1 - item.sb0;
    const uint32_t ring_base = smem_addr(epi_smem) - static_cast<uint32_t>(kRingBytes);
    const int s_last = static_cast<int>((sb_done - 1) % C::kStages);
    const uint32_t slot_a = ring_base + static_cast<uint32_t>(((s_last + C::kStages - 1) % C::kStages) * C::kStageBytes);
    const uint32_t slot_b = ring_base + static_cast<uint32_t>(s_last * C::kStageBytes);
    // staging tile b of this warp: its own two, then kRingBufs in each borrowed stage
    auto ring_buf = [&](uint32_t b) -> uint32_t {
      if constexpr (!C::kEpiOwn) {
        // this warp's tiles packed across both stages, kRingTiles in each
        const uint32_t t = static_cast<uint32_t>(ew * C::kEpiNB) + b;
        return t < static_cast<uint32_t>(C::kRingTiles) ? slot_a + t * C::kEpiBufBytes
                                                         : slot_b + (t - C::kRingTiles) * C::kEpiBufBytes;
      }
      if (b < 2u) return stg + b * C::kEpiBufBytes;
      constexpr uint32_t kPer = C::kRingBufs > 0 ? C::kRingBufs : 1;
      const uint32_t i = b - 2u;
      const uint32_t slot = i < kPer ? slot_a : slot_b;
      return slot + (static_cast<uint32_t>(ew) * kPer + i % kPer) * C::kEpiBufBytes;
    };
    const int32_t y0 = mt * C::kTileM + static_cast<int32_t>(prank) * kRowsA + q * 32;
    const int32_t x0 = nt * C::kTileN + cbeg;
    // C in 16-byte words when rows are contiguous and aligned (vec_ok): the tile's C rows are
    // pulled into L2 and the first kAhead 32-column runs into registers while the main loop
    // still runs; each later run is loaded kAhead runs before its use.  On the tile-store path
    // the first C tiles are copied into staging tiles instead: two runs into C tiles of their
    // own (tload_c), or, with one accumulator (whose eight warps have no room for C tiles),
    // the first run into the D staging tile it will write (cd_c; each later run one run ahead).
    const bool cvec = !tstore && p.has_c && p.vec_ok && row_ok && item.sb0 == 0;
    // (one run ahead with one accumulator: its 320 threads have 168 registers each)
    constexpr int kAhead = C::kEpiCTma ? 2 : 1;
    uint4 cr[kAhead][4];
    // (not with borrowed staging: its C copies all go out when the accumulator is full, and a
    // prefetch into L2 during the main loop competes with the operand copies — measured without
    // it: ragged 5000x3000x4104 92.4 -> 90.4 us, 8192^3 with C unchanged)
    if ((cvec || cd_c) && row_ok && cend > cbeg)
      prefetch_l2_bulk(p.C + base + cbeg, static_cast<uint32_t>(((cend - cbeg) * 2 + 15) & ~15));
#pragma unroll
    for (int a = 0; a < kAhead; ++a)
      if (cvec && cbeg + 32 * a + 32 <= cend) {
        const uint4* src = reinterpret_cast<const uint4*>(p.C + base + cbeg + 32 * a);
#pragma unroll
        for (int j = 0; j < 4; ++j) cr[a][j] = __ldg(src + j);
      }
    if constexpr (C::kEpiTma) {
      if (tload_c && lane == 0) {
        for (int a = 0; a < 2 && a < nruns; ++a) {
          const uint32_t b = (gr + a) & 1u;
          const uint32_t bar = smem_addr(&ctl->c_full[ew][b]);
          mbar_arrive_expect_tx(bar, C::kEpiBufBytes);
          tma_load_2d(stg + (2 + b) * C::kEpiBufBytes, tmC, bar, x0 + 32 * a, y0);
        }
      }
      if (tload_c) c_pending |= (nruns > 0 ? 1u << (gr & 1u) : 0u) | (nruns > 1 ? 1u << ((gr + 1) & 1u) : 0u);
      if (cd_c && nruns > 0) {
        if (lane == 0) {
          // the D staging tile of the first run is free once the store two runs back has read it
          bulk_wait_group_read<1>();
          const uint32_t bar = smem_addr(&ctl->c_full[ew][gr & 1u]);
          mbar_arrive_expect_tx(bar, C::kEpiBufBytes);
          tma_load_2d(stg + (gr & 1u) * C::kEpiBufBytes, tmC, bar, x0, y0);
        }
        c_pending |= 1u << (gr & 1u);
      }
      if (C::kRingBufs > 0 && C::kEpiOwn && ring && p.has_c) {
        // the first two runs' C into this warp's own staging tiles (free: the previous tile's
        // stores have read them), while the main loop still runs
        if (lane == 0)
          for (int a = 0; a < 2 && a < nruns; ++a) {
            const uint32_t bar = smem_addr(&ctl->c_full[ew][a]);
            mbar_arrive_expect_tx(bar, C::kEpiBufBytes);
            tma_load_2d(ring_buf(static_cast<uint32_t>(a)), tmC, bar, x0 + 32 * a, y0);
          }
        c_pending |= (nruns > 0 ? 1u : 0u) | (nruns > 1 ? 2u : 0u);
      }
    }
    const int buf = C::kAccBufs == 2 ? (it & 1) : 0;
    const uint32_t use = C::kAccBufs == 2 ? ((it >> 1) & 1) : (it & 1);
    if (!wait_warp<kPair>(smem_addr(&ctl->acc_full[buf]), use, ctl, p.timeout_ns, kSiteAccFull)) break;
    tc_fence_after_sync();
    if (C::kRingBufs > 0 && ring && p.has_c) {
      // every MMA of this tile has completed, so the borrowed stages are free: the C of the
      // runs up to NB - 1 into them
      constexpr int kFirst = C::kEpiOwn ? 2 : 0;
      if (lane == 0)
        for (int a = kFirst; a < C::kEpiNB && a < nruns; ++a) {
          const uint32_t bar = smem_addr(&ctl->c_full[ew][a]);
          mbar_arrive_expect_tx(bar, C::kEpiBufBytes);
          tma_load_2d(ring_buf(static_cast<uint32_t>(a)), tmC, bar, x0 + 32 * a, y0);
        }
      for (int a = kFirst; a < C::kEpiNB && a < nruns; ++a) c_pending |= 1u << a;
    }
    uint32_t c_lo = 1, c_hi = 0;
    if (owner_with_parts) {
      c_lo = sk_owner_of(p, nclusters, static_cast<int64_t>(item.tile) * p.nsb + item.sb1);
      c_hi = sk_owner_of(p, nclusters, static_cast<int64_t>(item.tile + 1) * p.nsb - 1);
      if (!wait_flags<kPair>(p, nclusters, c_lo, c_hi, rank, ctl)) break;
    }
    float* mine = contributor ? part_slot<kPair>(p, cluster, rank) : nullptr;
    bool ok = true;
    // with one accumulator and C, it is released once this warp has read its last columns from
    // TMEM (the rest of that run works on registers), so the next tile's MMAs overlap that run
    // (measured: 1 % faster with C; without C, whose runs are short, 0.5-1.5 % slower)
    const bool early = C::kAccBufs == 1 && p.has_c != 0;
    bool released = false;
    auto release_acc = [&]() {
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        const uint32_t ae = smem_addr(&ctl->acc_empty[buf]);
        if constexpr (kPair)
          mbar_arrive_cluster(map_to_cta(ae, 0));
        else
          mbar_arrive(ae);
      }
      released = true;
    };
#pragma unroll
    for (int run = 0; run < kRuns; ++run) {
      const int c0 = cbeg + 32 * run;
      if (c0 < cend && ok) {
        uint32_t acc[32];
        if (p.k_blocks > 0) {
          tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * C::kAccStride + c0, acc);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) acc[i] = 0u;
        }
        if (early && c0 + 32 >= cend) release_acc();
        if (contributor) {
#pragma unroll
          for (int i = 0; i < 32; ++i) __stcg(mine + (c0 + i) * 128 + lrow, __uint_as_float(acc[i]));
        } else {
          // the other CTAs' partials of this run, added in CTA order: up to kPartBatch
          // CTAs' values are gathered at once (asynchronous copies, one round trip) into
          // this warp's part of the stage ring, which is idle here — a split tile is its
          // owner's last item, so every copy into the ring has landed and every MMA
          // reading it has completed
          uint32_t c = next_contributor(p, nclusters, c_lo, c_hi);
          while (c <= c_hi) {
            int n = 0;
            for (; n < kPartBatch && c <= c_hi; ++n) {
              const float* part = part_slot<kPair>(p, c, rank) + c0 * 128 + lrow;
#pragma unroll
              for (int i = 0; i < 32; ++i) cp_async_4(part_buf + (n * 32 + i) * 128, part + i * 128);
              c = next_contributor(p, nclusters, c + 1, c_hi);
            }
            cp_async_wait_all();   // this lane reads back only what it copied
            for (int k = 0; k < n; ++k)
#pragma unroll
              for (int i = 0; i < 32; ++i)
                acc[i] = __float_as_uint(__uint_as_float(acc[i]) + ld_shared_f32(part_buf + (k * 32 + i) * 128));
          }
          if (C::kRingBufs > 0 && ring)
            ok = ring_store_run<kBF16, kPair, (C::kEpiNB > 2 ? C::kEpiNB : 2)>(
                p, ctl, acc, ew, lane, ring_buf, c_phase, c_pending, run, nruns, x0, y0,
                row_ok ? min(32, cols_left - c0) : 0, static_cast<int64_t>(nt) * C::kTileN + c0, amax, tmC, tmD);
          else if (C::kEpiTma && tstore)
            ok = tile_store_run<kBF16, kPair>(p, ctl, acc, ew, lane, stg, gr, c_phase, c_pending, tload_c, run,
                                              nruns, x0, y0, row_ok ? min(32, cols_left - c0) : 0,
                                              static_cast<int64_t>(nt) * C::kTileN + c0, amax, tmC, tmD, cd_c);
          else if (row_ok)
            store_run<kBF16>(p, base + c0 * p.d_col, cvec && c0 + 32 <= cend, cr[0], acc,
                             min(32, cols_left - c0), static_cast<int64_t>(nt) * C::kTileN + c0, amax);
          // rotate the C registers (fixed indices keep them in registers) and load the run
          // kAhead further on into the last slot
#pragma unroll
          for (int a = 0; a + 1 < kAhead; ++a)
#pragma unroll
            for (int j = 0; j < 4; ++j) cr[a][j] = cr[a + 1][j];
          const int cn0 = c0 + 32 * kAhead;
          if (cvec && cn0 + 32 <= cend) {
            const uint4* src = reinterpret_cast<const uint4*>(p.C + base + cn0);
#pragma unroll
            for (int j = 0; j < 4; ++j) cr[kAhead - 1][j] = __ldg(src + j);
          }
        }
      }
    }
    if (!ok) break;
    if (contributor) fence_acq_rel_gpu();   // this thread's partial before the hand-off
    if (!released) release_acc();          // a warp with no columns in this tile
    if (C::kRingBufs > 0 && ring_ok) {
      // return the borrowed stages once every store of this tile has read its staging tile
      if (lane == 0) {
        bulk_wait_group_read<0>();
        mbar_arrive(smem_addr(&ctl->epi_ring));
      }
    }
    __syncwarp();
    if (lane == 0) {
      if (contributor) mbar_arrive(smem_addr(&ctl->part_done));
      if (owner_with_parts) mbar_arrive(smem_addr(&ctl->fix_done));
    }
    if (owner_with_parts && warp == 2) {
      // the partials this CTA added are consumed: clear their flags, so that a later launch
      // with the same launch number (a replayed CUDA graph) waits for fresh ones.  A CTA
      // owns at most one split tile per launch, so fix_done completes phase 0 once.
      if (!wait_warp<kPair>(smem_addr(&ctl->fix_done), 0u, ctl, p.timeout_ns, kSiteFixup)) break;
      // (relaxed stores: nothing reads these flags again in this launch, and the next launch
      // starts after this one has completed)
      if (lane == 0)
        for (uint32_t c = c_lo; c <= c_hi; ++c)
          if (sk_has_units(p, nclusters, c)) st_relaxed_gpu(part_flag<kPair>(p, c, rank), 0u);
      __syncwarp();
    }
    if (contributor && warp == 2) {
      // a CTA contributes at most one partial per launch: part_done completes phase 0 once
      // all epilogue warps have written theirs; then publish it at device scope
      if (!wait_warp<kPair>(smem_addr(&ctl->part_done), 0u, ctl, p.timeout_ns, kSiteFixup)) break;
      if (lane == 0) {
        fence_acq_rel_gpu();
        st_release_gpu(part_flag<kPair>(p, cluster, rank), p.epoch);
      }
      __syncwarp();
    }
  }
  if constexpr (C::kEpiTma) {
    // every tile store issued by this warp has written D, and every C copy into its staging
    // tiles (outstanding only after an abort) has landed, before the CTA finishes
    if (tma && lane == 0) {
      bulk_wait_group<0>();
      for (uint32_t b = 0; b < 8; ++b)
        if (c_pending & (1u << b))
          wait_drain(smem_addr(&ctl->c_full[ew][b]), (c_phase >> b) & 1u, p.timeout_ns, p.status);
    }
    __syncwarp();
  }
  if (p.fused && p.amax != nullptr) {
    // one atomic per warp; |v| >= 0, so the float order equals the integer order
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (lane == 0) atomicMax(reinterpret_cast<int*>(p.amax), __float_as_int(amax));
  }
}

__device__ __forceinline__ uint8_t* align_1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

template <bool kBF16, bool kPair, int kIn, int kShape = kShapeStd>
__global__ void __launch_bounds__(Cfg<kPair, kIn, kShape>::kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmSFA, const __grid_constant__ CUtensorMap tmSFB,
                const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmD,
                const __grid_constant__ CUtensorMap tmAt, const __grid_constant__ CUtensorMap tmBt,
                const Params p) {
  using C = Cfg<kPair, kIn, kShape>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_1024(smem_raw);
  uint8_t* epi_smem = smem + C::kStages * C::kStageBytes;   // tile-store staging (1024-aligned)
  Ctl* ctl = reinterpret_cast<Ctl*>(epi_smem + C::kEpiStageBytes);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;
  const uint32_t cluster = kPair ? cluster_id_x() : blockIdx.x;
  const uint32_t nclusters = kPair ? cluster_count_x() : gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(smem_addr(&ctl->full[s]), 1);
      mbar_init(smem_addr(&ctl->empty[s]), 1);   // one release (the pair's MMA commit)
    }
    for (int b = 0; b < C::kAccBufs; ++b) {
      mbar_init(smem_addr(&ctl->acc_full[b]), 1);
      mbar_init(smem_addr(&ctl->acc_empty[b]), C::kAccEmptyArrivals);
    }
    mbar_init(smem_addr(&ctl->drain), 1);
    mbar_init(smem_addr(&ctl->part_done), C::kEpiWarps);
    mbar_init(smem_addr(&ctl->fix_done), C::kEpiWarps);
    if constexpr (C::kEpiTma)
      for (int w = 0; w < C::kEpiWarps; ++w)
        for (int b = 0; b < 8; ++b) mbar_init(smem_addr(&ctl->c_full[w][b]), 1);
    mbar_init(smem_addr(&ctl->epi_ring), C::kEpiWarps);
    ctl->abort = 0;
    ctl->status = p.status;
    fence_barrier_init();
    if (p.k_blocks > 0) {
      prefetch_tensormap(&tmA);
      prefetch_tensormap(&tmB);
      if constexpr (C::kMx) {
        prefetch_tensormap(&tmSFA);
        prefetch_tensormap(&tmSFB);
      }
    }
    if (C::kEpiTma && p.epi_tma) {
      if (p.has_c) prefetch_tensormap(&tmC);
      prefetch_tensormap(&tmD);
    }
  }
  if (warp == 1) {
    if constexpr (kPair) {
      tmem_alloc_pair(smem_addr(&ctl->tmem_base), kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_addr(&ctl->tmem_base), kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if constexpr (kPair) cluster_sync();   // peer barriers initialised before any remote use
  tc_fence_after_sync();
  const uint32_t tmem_base = ctl->tmem_base;
  // launched with programmatic stream serialisation: the set-up above may overlap the end of
  // the previous kernel in the stream; nothing below touches global memory before it is done
  griddep_wait();
  griddep_launch_dependents();

  if (warp == 0) {
    if (lane == 0)
      run_producer<kPair, kIn, kShape>(p, &tmA, &tmB, &tmSFA, &tmSFB, &tmAt, &tmBt, smem, ctl, rank, cluster,
                                       nclusters);
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) run_mma<kPair, kIn, kShape>(p, smem, ctl, tmem_base, rank, cluster, nclusters);
    __syncwarp();
  } else {
    run_epilogue<kBF16, kPair, kIn, kShape>(p, ctl, tmem_base, warp, lane, rank, cluster, nclusters, epi_smem,
                                            &tmC, &tmD);
  }

  tc_fence_before_sync();
  __syncthreads();
  if constexpr (kPair) cluster_sync();   // no remote arrival or MMA targets a CTA that left
  if (warp == 1) {
    tc_fence_after_sync();
    if constexpr (kPair)
      tmem_dealloc_pair(tmem_base, kTmemCols);
    else
      tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ------------------------------------------------------------------ host launch side
// Index of a pair shape in DeviceState's per-shape arrays.
constexpr int pair_shape_index(int shape) {
  return shape == kShapeN224 ? 1 : (shape == kShapeW512 ? 2 : (shape == kShapeW448 ? 3 : 0));
}

// Per-device state the launchers keep (function attributes set, co-resident clusters).
// The host writes it only while holding its device-state lock (calls may come from several
// host threads); each field goes from its initial value to its final one once, except the
// stream-K launch counter.
struct DeviceState {
  bool probed = false;
  int major = 0, minor = 0, sms = 0;
  bool attr_single[2][3][2] = {};   // [bf16 out][input kind][narrow]
  bool attr_pair[2][3][4] = {};   // [bf16 out][input kind][pair shape: standard, 224, 512, 448 wide]
  int pair_clusters[4] = {};      // co-resident clusters per pair shape (0: not queried yet)
  uint32_t epoch = 0;      // stream-K launch counter (flags compare against it)
  bool dbg_attr = false;
  uint32_t* status = nullptr;   // device address of the status word
};

// The tensor maps of one call: A, B and, for block-scaled inputs, the packed scale factors.
struct Maps {
  CUtensorMap a, b, sfa, sfb;
  CUtensorMap c, d;   // tile-store epilogue: C and D as (N, M) tensors, 32 x 32 boxes
  CUtensorMap at, bt; // two-dimensional maps of A, B for the K tail when a, b are stage-deep
  int32_t kb_full;    // Params::kb_full
  int32_t epi_tma;    // Params::epi_tma: c (when C is read) and d are encoded
  int32_t kb_boxes;   // Params::kb_boxes: which of a, b are stage-deep (three-dimensional) maps
};

// Defined in gemm_launch.cuh; instances come from gemm_inst.cu.
// prepare_* set the function attributes (and, for pairs, count the co-resident clusters)
// once per device: call them with the device-state lock held.  launch_* touch no shared state.
template <bool kBF16, int kIn, int kShape>
gb_status prepare_single(DeviceState* dev);
template <bool kBF16, int kIn, int kShape>
gb_status launch_single(const Maps& m, const Params& p, int grid, cudaStream_t s);
template <bool kBF16, int kIn, int kShape>
gb_status prepare_pair(DeviceState* dev);
template <bool kBF16, int kIn, int kShape>
gb_status launch_pair(const Maps& m, const Params& p, int clusters, cudaStream_t s);

}  // namespace gb
