// The tcgen05 GEMM kernels: D[M,N] = A[M,K] * B[N,K]^T, fp32 accumulation in
// TMEM, bf16 output.
//
//  * gemm_ws_kernel   -- persistent, warp-specialised kernel (TMA producer
//                        warp, single-thread MMA issuer, one or two groups of
//                        four epilogue warps, a scale-factor warp for MXFP8
//                        with row-major scales or a scale-copy thread for
//                        tiled ones), one CTA (cta_group::1) or a CTA pair
//                        (cta_group::2); bf16 operands (128x256 / 256x256
//                        tiles), block-scaled MXFP8 operands with row-major
//                        scales (128x224 / 256x224) or tiled scales
//                        (128x256 / 256x256).  A short last round of tiles
//                        may run as column halves, or a cheap last column
//                        block's tiles as halves at the end of the deal; the
//                        fused epilogue can bring C in by TMA.  A plain build
//                        (PLAIN) leaves out the stream-K, fused-epilogue and
//                        C-by-TMA code for launches that need none of it.
//  * gemm_sync_kernel -- (gemm_sync.cuh) one 128x128 tile per CTA with synchronous thread
//                        copies into shared memory and one MMA batch per
//                        K-tile: the first rungs of the optimisation ladder,
//                        kept as a bisection reference.
//  * zero_fill_kernel -- (gemm_sync.cuh) D = 0 for an empty reduction (K = 0).
//
// Method: b200-gemm-optimization-ladder ("A1 -- The nine-level route",
// levels 1-8), b200-tma-pipeline-designer ("E -- Executable steps": tensor-map
// descriptor, single issuer, ready/free barriers, store drain, three-phase
// timeline) and b200-tmem-lifecycle-planner ("E -- Executable steps": column
// budget, TLane/TCol map, write/read paths and the lifecycle).
#pragma once

#include <cstdint>

#include "kernel_common.cuh"

namespace gb300 {

// BF16: bf16 operands.  MXF8: block-scaled E4M3 operands with row-major
// scale matrices, re-tiled on chip by a scale-factor warp.  MXF8T: the same
// with the scale matrices already in the tensor core's chunk layout in
// global memory ("tiled": 512-byte chunks of 128 rows x 4 scale blocks),
// loaded by TMA into each operand stage like A and B.
enum class Kind { BF16, MXF8, MXF8T };

struct GemmArgs {
  uint32_t M, N, K;
  uint32_t num_m_blocks;      // tiles along M (UMMA_M rows each)
  uint32_t num_n_blocks;      // tiles along N (UMMA_N columns each)
  uint32_t num_k_tiles;       // ceil(K / BK)
  uint32_t group_m;           // raster group (M-blocks swept together)
  void* D;                    // D base (direct-store epilogue)
  uint64_t ldd;               // D row pitch in elements
  unsigned long long* status; // device status word
  unsigned long long timeout_ns;
  uint32_t stall_iter;        // watchdog test hook: K-tile iteration whose loads are
                              // withheld (0xFFFFFFFF: none)
  // Schedule: the first dp_tiles tiles go whole to clusters round-robin; the
  // next sk_tiles tiles are cut into units of sk_unit K-tiles and the units
  // are dealt out in equal contiguous ranges to all clusters (stream-K).
  uint32_t dp_tiles;
  uint32_t sk_tiles;
  uint32_t sk_unit;
  // Tail split (data-parallel schedule only): the last half_tiles of the
  // dp_tiles whole tiles are cut into two column halves of UMMA_N / 2, each
  // a work item of its own, so a last round that would leave most clusters
  // idle takes about half a tile's time.
  uint32_t half_tiles;
  // Right-edge tiles last (plain bf16 launches whose last column block holds
  // at most UMMA_N / 2 live columns): the last column block's tiles come
  // after all others, and rounds are dealt in alternating directions, so the
  // cheap edge tiles fill the last round and land on the clusters that took
  // full tiles last.  edge_half: the edge tiles run as first column halves
  // (set with edge_last).  0 otherwise.
  uint32_t edge_last;
  uint32_t edge_half;
  float* ws_part;             // stream-K partial accumulators, one slot per cluster
  uint32_t* ws_flag;          // per (slot, CTA, epilogue warp) ready flags
  uint32_t epoch;             // this launch's flag value (never 0)
  // Fused epilogue: v = alpha acc + beta C + bias[col], act(v) (mode 0: none)
  uint32_t epi_mode;
  float alpha, beta;
  const void* C;
  uint64_t ldc;
  const void* bias;
  // C of the fused epilogue arrives by TMA (tmC) into the epilogue warp's
  // second staging buffer, one chunk ahead, instead of by per-thread loads
  // (bf16 C in the TMA-store kernels with 64-column chunks)
  uint32_t c_tma;
  // MXFP8 scale bytes read with plain loads (sf_gather != 0: a pitch or base
  // that TMA cannot take) instead of through the tmSFA / tmSFB tensor maps
  uint32_t sf_gather;
  const uint8_t* sfa;
  const uint8_t* sfb;
  uint64_t ldsfa, ldsfb;
};

// One piece of work for a cluster: K-tiles [k_begin, k_end) of a tile.
//   kind 0: the whole tile;  1: the first K-range of a split tile (this
//   cluster owns it: adds the later ranges' partials and stores D);
//   2: a later K-range (partial accumulator goes to this cluster's slot).
//   half 0: all UMMA_N columns of the tile; 1 / 2: its first / second
//   column half (tail split, kind 0 only).
struct WorkItem {
  uint32_t tile, k_begin, k_end, kind, half;
};

// First column of D and number of columns that work item w covers in its
// tile's column block nb.
__device__ __forceinline__ uint32_t item_n0(const WorkItem& w, uint32_t nb, uint32_t umma_n) {
  return nb * umma_n + (w.half == 2u ? umma_n / 2 : 0u);
}
__device__ __forceinline__ uint32_t item_cols(const WorkItem& w, uint32_t umma_n) {
  return w.half != 0u ? umma_n / 2 : umma_n;
}

__device__ __forceinline__ uint64_t sk_bound(uint64_t units, uint32_t c, uint32_t G) {
  return units * c / G;
}

// Block coordinates of tile t: the grouped raster of tile_coords, or, with
// edge_last (EDGE builds), that raster over all column blocks but the last,
// followed by the last column block's tiles in row order.
template <bool EDGE>
__device__ __forceinline__ void item_coords(const GemmArgs& a, uint32_t t, uint32_t& mb, uint32_t& nb) {
  if (EDGE && a.edge_last != 0) {
    const uint32_t nf = a.num_n_blocks - 1;
    const uint32_t e0 = a.num_m_blocks * nf;
    if (t >= e0) {
      mb = t - e0;
      nb = nf;
      return;
    }
    tile_coords(t, a.num_m_blocks, nf, a.group_m, mb, nb);
    return;
  }
  tile_coords(t, a.num_m_blocks, a.num_n_blocks, a.group_m, mb, nb);
}

// The wi-th work item of cluster c among G clusters; false past the last.
// Every role of every CTA calls this with the same arguments, so they all
// walk the same sequence.  SK = false: a kernel built without stream-K
// (launched only with sk_tiles == 0).  EDGE: a build that honours edge_last.
template <bool SK = true, bool EDGE = false>
__device__ __forceinline__ bool work_item(const GemmArgs& a, uint32_t c, uint32_t G, uint32_t KT,
                                          uint32_t wi, WorkItem& w) {
  if (EDGE && a.edge_last != 0) {
    // whole tiles only (no tail split, no stream-K): round wi deals tiles
    // wi G .. wi G + G - 1, to clusters 0 .. G-1 in even rounds and G-1 .. 0
    // in odd ones; the pair runs an edge tile as a first column half
    const uint32_t x = wi * G + ((wi & 1u) ? G - 1u - c : c);
    if (x >= a.dp_tiles) return false;
    w.tile = x;
    w.half = (a.edge_half != 0 && x >= a.num_m_blocks * (a.num_n_blocks - 1)) ? 1u : 0u;
    w.k_begin = 0;
    w.k_end = KT;
    w.kind = 0;
    return true;
  }
  // data-parallel items: the whole tiles, then two halves of each of the
  // last half_tiles tiles
  const uint32_t n_items = a.dp_tiles + a.half_tiles;
  const uint32_t n_dp = n_items > c ? (n_items - c + G - 1) / G : 0u;
  if (wi < n_dp) {
    const uint32_t x = c + wi * G;
    const uint32_t whole = a.dp_tiles - a.half_tiles;
    if (x < whole) {
      w.tile = x;
      w.half = 0;
    } else {
      w.tile = whole + (x - whole) / 2u;
      w.half = 1u + ((x - whole) & 1u);
    }
    w.k_begin = 0;
    w.k_end = KT;
    w.kind = 0;
    return true;
  }
  if (!SK || a.sk_tiles == 0) return false;
  const uint32_t KU = (KT + a.sk_unit - 1) / a.sk_unit;   // units per tile
  const uint64_t U = static_cast<uint64_t>(a.sk_tiles) * KU;
  const uint64_t u0 = sk_bound(U, c, G), u1 = sk_bound(U, c + 1, G);
  const uint64_t j = wi - n_dp;
  const uint64_t start = j == 0 ? u0 : (u0 / KU + j) * KU;
  if (start >= u1) return false;
  const uint64_t ts = start / KU;
  const uint64_t end = u1 < (ts + 1) * KU ? u1 : (ts + 1) * KU;
  const uint32_t ub = static_cast<uint32_t>(start - ts * KU);
  const uint32_t ue = static_cast<uint32_t>(end - ts * KU);
  w.tile = a.dp_tiles + static_cast<uint32_t>(ts);
  w.half = 0;
  w.k_begin = ub * a.sk_unit;
  w.k_end = min(KT, ue * a.sk_unit);
  w.kind = (ub == 0 && ue == KU) ? 0u : (ub == 0 ? 1u : 2u);
  return true;
}

// Number of clusters whose partials the owner of `tile` (kind 1 at cluster c)
// adds: c+1, c+2, ... up to the one holding the tile's last unit.  The host
// launches no more clusters than units, so every cluster's range is
// non-empty and the contributors are consecutive.
__device__ __forceinline__ uint32_t num_contributors(const GemmArgs& a, uint32_t c, uint32_t G,
                                                     uint32_t KT, uint32_t tile) {
  const uint32_t KU = (KT + a.sk_unit - 1) / a.sk_unit;
  const uint64_t U = static_cast<uint64_t>(a.sk_tiles) * KU;
  const uint64_t tile_end = static_cast<uint64_t>(tile - a.dp_tiles + 1) * KU;
  uint32_t n = 0;
  for (uint32_t cc = c + 1; cc < G && sk_bound(U, cc, G) < tile_end; ++cc) ++n;
  return n;
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_u32(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Bounded wait (lane 0) for a stream-K flag to reach `epoch`; warp-uniform result.
__device__ __forceinline__ bool wait_flag(const uint32_t* f, uint32_t epoch, const Watchdog& wd,
                                          uint32_t lane) {
  bool ok = true;
  if (lane == 0) {
    const uint64_t t0 = global_timer_ns();
    for (uint32_t n = 0;; ++n) {
      if (ld_acquire_u32(f) == epoch) break;
      if ((n & 31u) == 31u) {
        if (*wd.abort_flag) { ok = false; break; }
        if (global_timer_ns() - t0 > wd.timeout_ns) {
          *wd.abort_flag = 1u;
          report_error(wd.status, kDevTimeout, kSiteStreamKFlag);
          ok = false;
          break;
        }
      }
    }
  }
  return __shfl_sync(0xffffffffu, ok ? 1u : 0u, 0) != 0;
}

__host__ __device__ constexpr uint32_t align_up_u32(uint32_t x, uint32_t a) {
  return (x + a - 1) / a * a;
}

// Compile-time plan of one kernel configuration: tile shape, stage ring,
// TMEM column budget and shared-memory map.
//
//   bf16,  1 CTA : 128 x 256 tiles, two 256-column accumulators
//   bf16,  pair  : 256 x 256 cluster tiles, two 256-column accumulators
//   MXFP8, 1 CTA : 128 x 224 tiles, two 224-column accumulators + scale
//                  columns (2 x 224 + 12 <= 512)
//   MXFP8, pair  : 256 x 224 cluster tiles, two 224-column accumulators +
//                  scale columns (2 x 224 + 12 <= 512)
//   MXFP8 with tiled scales, 1 CTA / pair : 128 x 256 / 256 x 256 tiles, one
//                  256-column accumulator + scale columns (256 + 12 <= 512)
template <int CG, Kind KIND, bool TMA_STORE, bool EPI2 = false>
struct GemmCfg {
  static_assert(CG == 1 || CG == 2, "cta_group is 1 or 2");
  static constexpr bool MX = KIND != Kind::BF16;          // block-scaled E4M3
  static constexpr bool SF_TILED = KIND == Kind::MXF8T;   // scales by TMA, in the stages
  static constexpr bool SF_WARP = MX && !SF_TILED;        // scales re-tiled on chip

  // w0 TMA producer, w1 MMA issuer / TMEM owner, w2..5 epilogue and, for
  // MXFP8, w6: the scale-factor warp.  It re-tiles each stage's scale bytes as
  // soon as they land (their own barrier) and then arrives on the leader's
  // ready barrier, which keeps that work off the MMA issuer's path.  Kernels
  // with the masked-store epilogue and two accumulator buffers add a second
  // epilogue warpgroup after those (see EPI_WG).
  static constexpr uint32_t kSfWarp = 6;
  static constexpr uint32_t BLOCK_M = 128;    // D rows owned by one CTA (= TMEM lanes)
  static constexpr uint32_t UMMA_M = 128 * CG;
  // D columns per tile.  MXFP8 uses 224 so that two accumulators and the scale
  // columns fit in 512 TMEM columns (2 x 224 + 12): the epilogue of one tile
  // then overlaps the next tile's MMAs (measured +4% at 8192^3, +16% at
  // 8192x8192x4096 against one 256-column accumulator).
  // Tiled scales need no on-chip scale rings, and tile at N = 256: their
  // 128-row chunks then line up with whole tiles.
  static constexpr uint32_t UMMA_N = SF_WARP ? 224 : 256;
  static constexpr uint32_t B_ROWS = UMMA_N / CG;  // B rows staged by one CTA
  static constexpr uint32_t ELEM = MX ? 1 : 2;
  static constexpr uint32_t BK = 128 / ELEM;  // K elements per stage: one 128-byte row
  static constexpr uint32_t UMMA_K = 32 / ELEM;
  static constexpr uint32_t K_STEPS = BK / UMMA_K;
  static constexpr uint32_t A_BYTES = BLOCK_M * 128;
  static constexpr uint32_t B_BYTES = B_ROWS * 128;
  // Tiled scales: the K-tile's 512-byte chunk of this CTA's 128 A rows, then
  // one chunk per 128 B rows of the tile (every CTA holds the scales of all
  // the tile's B rows), behind A and B in the same stage.
  static constexpr uint32_t SFB_TILE_CHUNKS = SF_TILED ? UMMA_N / 128 : 0;
  static constexpr uint32_t SF_STAGE_BYTES = SF_TILED ? 512 * (1 + SFB_TILE_CHUNKS) : 0;
  static constexpr uint32_t OFF_B = A_BYTES;
  static constexpr uint32_t OFF_SF = A_BYTES + B_BYTES;
  static constexpr uint32_t STAGE_BYTES = align_up_u32(A_BYTES + B_BYTES + SF_STAGE_BYTES, 1024);
  // Bytes that land on a stage's ready barrier, per CTA: the A and B tiles.
  // Tiled scales have a ready barrier of their own per stage, and the
  // producer issues their loads first: the scale copies into TMEM then start
  // while the operand tiles are still arriving.
  static constexpr uint32_t AB_TX = A_BYTES + B_BYTES;
  static constexpr uint32_t FULL_ARRIVALS = 1;                    // the producer's expect_tx

  // MXFP8 scale factors travel in two rings of their own, one slot per group
  // of SF_GROUP = 4 K-tiles (one 16-byte TMA box row carries 4 K-tiles'
  // scales: 4 x 4 UE8M0 bytes):
  //   raw ring (RAW_SLOTS): the TMA boxes of this CTA's A rows and of all the
  //     tile's B rows.  The scale-factor warp loads them itself and reloads a
  //     slot as soon as it has re-tiled it, so scale bytes run ahead of the
  //     operand ring instead of arriving with it;
  //   re-tiled ring (T_SLOTS): one 32x16-byte chunk per 128 rows and K-tile,
  //     the layout tcgen05.cp ... 32x128b.warpx4 copies into TMEM; freed by
  //     the MMA issuer's commit after the group's last K-tile.  Its depth is
  //     the MMA issuer's look-ahead over scale factors.
  // Every CTA holds the scales of all UMMA_N B rows of the tile (its tensor
  // core multiplies by all of them) and of its own 128 A rows.
  static constexpr uint32_t SF_GROUP = 4;
  static constexpr uint32_t RAW_SLOTS = 2;
  static constexpr uint32_t T_SLOTS = CG == 2 || SF_TILED ? 4 : 2;
  static constexpr uint32_t SFB_ROWS = MX ? UMMA_N : 0;
  static constexpr uint32_t SFB_CHUNKS = (SFB_ROWS + 127) / 128;
  static constexpr uint32_t SFA_RAW = SF_WARP ? BLOCK_M * 16 : 0;
  static constexpr uint32_t SFB_RAW = SF_WARP ? SFB_ROWS * 16 : 0;
  static constexpr uint32_t SFA_T = SF_WARP ? 512 : 0;            // one chunk per K-tile
  static constexpr uint32_t SFB_T = SF_WARP ? SFB_CHUNKS * 512 : 0;
  static constexpr uint32_t T_PER_KT = SFA_T + SFB_T;
  static constexpr uint32_t OFF_SFA_RAW = 0;                      // within a raw slot
  static constexpr uint32_t OFF_SFB_RAW = SFA_RAW;
  static constexpr uint32_t RAW_SLOT_BYTES = SF_WARP ? align_up_u32(SFA_RAW + SFB_RAW, 1024) : 0;
  static constexpr uint32_t T_SLOT_BYTES = SF_WARP ? align_up_u32(SF_GROUP * T_PER_KT, 1024) : 0;
  static constexpr uint32_t SF_BYTES = RAW_SLOTS * RAW_SLOT_BYTES + T_SLOTS * T_SLOT_BYTES;
  static constexpr uint32_t SF_TX = SFA_RAW + SFB_RAW;            // per CTA and raw slot

  // TMEM: ACC_STAGES accumulators of UMMA_N fp32 columns, then the scale
  // factors (MXFP8: 4 columns for A, 4 per 128 B rows).  512 = whole TMEM.
  // Two 256-column accumulators leave no columns for scales, so the tiled-
  // scale kernels (N = 256) keep one.
  static constexpr uint32_t ACC_STAGES = SF_TILED ? 1 : 2;
  // Unroll factor of the MMA issuer's K-tile loop.
  // (the tiled-scale pair: 4, measured +4% over 2 at 8192^3)
  static constexpr int MMA_UNROLL = CG == 2 ? (SF_WARP ? 2 : 4) : 1;
  // Epilogue warpgroups (the ladder's multi-consumer level): with two, both
  // groups drain every tile, group g taking the 32-column chunks c with
  // c % 2 == g, so a tile's epilogue takes half as long.  Used where the
  // epilogue is the slow consumer -- the bf16 masked-store path, whose staging
  // costs 2 KB per warp and no operand stage.  (In the MXFP8 pair the extra
  // staging would cost a stage: 6 -> 5, measured 3% slower.)
  // EPI2 asks for the second group in an MXFP8 kernel as well (used for
  // launches that split tiles along K, whose epilogue also sums partial tiles).
  // The tiled-scale kernels (one accumulator) use two groups as well: their
  // epilogue hands the accumulator back as soon as it sits in registers, so a
  // faster drain shortens the MMA issuer's wait directly.
  static constexpr uint32_t EPI_WG =
      SF_TILED || (!TMA_STORE && ACC_STAGES == 2 && (!MX || EPI2)) ? 2 : 1;
  static constexpr uint32_t kEpiWg1Warp = SF_WARP ? 7 : 6;   // first warp of group 1
  // Tiled scales: one more warp after the epilogue groups issues the scale
  // copies (tcgen05.cp) into two alternating TMEM scale sets, so the MMA
  // thread issues only MMAs and commits.
  static constexpr uint32_t kCpWarp = kEpiWg1Warp + 4 * (EPI_WG - 1);
  static constexpr uint32_t kThreads = 32 * (kCpWarp + (SF_TILED ? 1 : 0));
  static constexpr uint32_t SF_TMEM_COL = ACC_STAGES * UMMA_N;
  static constexpr uint32_t SF_SET_COLS = MX ? 4 + 4 * SFB_CHUNKS : 0;   // one K-tile's scales
  static constexpr uint32_t TMEM_COLS = 512;

  // Epilogue staging for TMA stores: per epilogue warp, two buffers of 32
  // rows x TS_COLS bf16 columns -- 64 columns (128-byte rows, 128-byte
  // swizzle) where the tile width allows, else 32 (64-byte rows, 64-byte
  // swizzle: the MXFP8 tiles are 224 = 7 x 32 columns wide).
  // (The tiled-scale kernels use 32-column boxes too: half the staging, so
  // the pair keeps six operand stages with eight epilogue warps.)
  static constexpr uint32_t TS_COLS = UMMA_N % 64 == 0 && !SF_TILED ? 64 : 32;
  static_assert(!TMA_STORE || UMMA_N % TS_COLS == 0, "TMA-store chunks tile the accumulator");
  // The masked-store epilogue instead stages one 32x32 chunk per warp (2 KB)
  // and writes it back row by row, lanes across columns, so its global stores
  // are coalesced whatever the pitch.
  static constexpr uint32_t EPI_BUF_BYTES = 32 * TS_COLS * 2;
  // Staging buffers per epilogue warp: two (the next chunk's conversion
  // overlaps the previous chunk's store), one with two epilogue groups.
  static constexpr uint32_t EPI_BUFS = EPI_WG == 2 ? 1 : 2;
  static constexpr uint32_t CHUNK_BYTES = 32 * 64;
  static constexpr uint32_t EPI_BYTES =
      TMA_STORE ? 4 * EPI_WG * EPI_BUFS * EPI_BUF_BYTES : 4 * EPI_WG * CHUNK_BYTES;

  static constexpr uint32_t SMEM_LIMIT = 232448;  // 227 KB opt-in per CTA
  static constexpr uint32_t BAR_BYTES = SF_TILED ? 1024 : 512;
  static constexpr uint32_t ALIGN_SLACK = 1024;
  static constexpr uint32_t STAGES_FIT =
      (SMEM_LIMIT - ALIGN_SLACK - BAR_BYTES - EPI_BYTES - SF_BYTES) / STAGE_BYTES;
  static constexpr uint32_t STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
  static_assert(STAGES >= 2, "stage ring needs two slots");
  static constexpr uint32_t SMEM_BYTES =
      ALIGN_SLACK + STAGES * STAGE_BYTES + SF_BYTES + EPI_BYTES + BAR_BYTES;
  static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared memory budget");
  // Tiled scales: TMEM scale sets the copy thread rotates through (4 measured
  // 16% faster than 2: the copies of the next K-tiles no longer wait for the
  // MMAs just issued).  At most STAGES: the copy thread finds a set free by
  // waiting for the stage barrier phase of the K-tile SF_SETS back, and that
  // barrier must not have moved on to its next phase (K-tile SF_SETS back +
  // STAGES, whose copies this thread has not issued yet).
  static constexpr uint32_t SF_SETS = SF_TILED ? (STAGES < 4 ? STAGES : 4) : 1;
  static_assert(SF_SETS <= STAGES, "a scale set's free phase must be unambiguous");
  static_assert(SF_TMEM_COL + SF_SETS * SF_SET_COLS <= TMEM_COLS, "TMEM column budget");
  static_assert(!SF_TILED || T_SLOTS >= SF_SETS, "scale-set barriers");
  // Stream-K owner: each epilogue warp streams its contributors' partial
  // chunks (32 rows x 32 fp32 columns, 4 KB) through FIX_SLOTS slots of its
  // own, placed in the operand stages, which are idle once the CTA's last MMA
  // has completed.  32 slots in all (4 or 8 per warp: the depth measured the
  // same).
  static constexpr uint32_t FIX_SLOTS = 8 / EPI_WG;
  static constexpr uint32_t FIX_SLOT_BYTES = 32 * 32 * 4;
  static constexpr uint32_t FIX_TOTAL = 4 * EPI_WG * FIX_SLOTS;
  static_assert(FIX_TOTAL * FIX_SLOT_BYTES <= STAGES * STAGE_BYTES, "partial ring fits the stages");
  static_assert((2 * STAGES + RAW_SLOTS + 2 * T_SLOTS + 5) * 8 + 8 + FIX_TOTAL * 8 + 4 * 8 +
                        (SF_TILED ? STAGES * 8 : 0) <= BAR_BYTES,
                "barrier area");
};

// Re-tile one slot's scale bytes for tcgen05.cp ... 32x128b.warpx4.  The raw
// TMA box holds 16 bytes per row: the 4-byte words of 4 consecutive K-tiles
// (one UE8M0 per 32 k).  For K-tile j, row r's word moves to byte
// 16*(r%32) + 4*(r/32) of its 128-row chunk.  Lane l reads whole 16-byte rows
// l, l+32, l+64, l+96 and writes one 16-byte chunk row per K-tile, so both
// sides are bank-conflict free.  Rows past `rows` are written as zero.
template <uint32_t CHUNKS>
__device__ __forceinline__ void retile_scales(const uint8_t* raw, uint8_t* t_base, uint32_t t_stride,
                                              uint32_t t_off, uint32_t rows, uint32_t lane) {
  if constexpr (CHUNKS > 0) {   // (bf16 instantiations have no scales)
    const uint4* rw = reinterpret_cast<const uint4*>(raw);
#pragma unroll
    for (uint32_t h = 0; h < CHUNKS; ++h) {
      uint4 v[4];
#pragma unroll
      for (uint32_t q = 0; q < 4; ++q) {
        const uint32_t r = h * 128 + 32 * q + lane;
        v[q] = r < rows ? rw[r] : make_uint4(0, 0, 0, 0);
      }
      uint8_t* d0 = t_base + t_off + h * 512 + 16 * lane;
      *reinterpret_cast<uint4*>(d0) = make_uint4(v[0].x, v[1].x, v[2].x, v[3].x);
      *reinterpret_cast<uint4*>(d0 + t_stride) = make_uint4(v[0].y, v[1].y, v[2].y, v[3].y);
      *reinterpret_cast<uint4*>(d0 + 2 * t_stride) = make_uint4(v[0].z, v[1].z, v[2].z, v[3].z);
      *reinterpret_cast<uint4*>(d0 + 3 * t_stride) = make_uint4(v[0].w, v[1].w, v[2].w, v[3].w);
    }
  }
}

// Plain-load gather of one scale-factor group for scale pitches and bases
// that TMA cannot take: rows row0 .. row0 + ROWS - 1 of an R-row byte matrix
// with pitch ld, bytes kb0 .. kb0 + 15 of each row (one UE8M0 byte per 32 k,
// 4 K-tiles), written to `dst` in the layout the TMA box would give (16 bytes
// per row).  Rows >= R and bytes >= nblk are written as zero and never read.
// Lane l takes rows l, l + 32, ...; four rows' 64 byte loads are in flight at
// once (the scale bytes are small and L2-resident).
template <uint32_t ROWS>
__device__ __forceinline__ void gather_scale_rows(uint8_t* dst, const uint8_t* src, uint64_t ld,
                                                  uint32_t row0, uint32_t R, uint32_t kb0,
                                                  uint32_t nblk, uint32_t lane) {
  constexpr uint32_t PER_LANE = (ROWS + 31) / 32;
  const uint32_t nb = kb0 < nblk ? min(16u, nblk - kb0) : 0u;
#pragma unroll
  for (uint32_t i0 = 0; i0 < PER_LANE; i0 += 4) {
    uint32_t w[4][4];
#pragma unroll
    for (uint32_t j = 0; j < 4; ++j) {
      const uint32_t r = (i0 + j) * 32 + lane;
      const bool live = i0 + j < PER_LANE && r < ROWS && row0 + r < R;
      const uint8_t* p = src + static_cast<uint64_t>(row0 + r) * ld + kb0;
#pragma unroll
      for (uint32_t q = 0; q < 4; ++q) {
        uint32_t x = 0;
#pragma unroll
        for (uint32_t b = 0; b < 4; ++b)
          if (live && 4 * q + b < nb) x |= static_cast<uint32_t>(__ldg(p + 4 * q + b)) << (8 * b);
        w[j][q] = x;
      }
    }
#pragma unroll
    for (uint32_t j = 0; j < 4; ++j) {
      const uint32_t r = (i0 + j) * 32 + lane;
      if (i0 + j < PER_LANE && r < ROWS)
        *reinterpret_cast<uint4*>(dst + 16 * r) = make_uint4(w[j][0], w[j][1], w[j][2], w[j][3]);
    }
  }
}

template <int CG>
__device__ __forceinline__ void commit_to(uint32_t bar) {
  if constexpr (CG == 1)
    tc_commit(bar);
  else
    tc_commit_pair_multicast(bar, 0x3);  // the same barrier in both CTAs of the pair
}

// Bounded wait by lane 0, result broadcast to the warp; on success the other
// lanes also observe the completed phase (acquire) before touching its data.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const Watchdog& wd,
                                          uint32_t site, uint32_t lane) {
  bool ok = true;
  if (lane == 0) ok = wait_bounded(bar, parity, wd, site);
  ok = __shfl_sync(0xffffffffu, ok ? 1u : 0u, 0) != 0;
  if (ok && lane != 0) ok = wait_bounded(bar, parity, wd, site);
  return __all_sync(0xffffffffu, ok);
}

// Exit-path wait that ignores the abort flag (used to let this CTA's own
// asynchronous operations finish before shared memory / TMEM are released).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, const Watchdog& wd,
                                           uint32_t site) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t n = 0;; ++n) {
    if (mbar_try_wait(bar, parity)) return;
    if ((n & 31u) == 31u && global_timer_ns() - t0 > wd.timeout_ns) {
      report_error(wd.status, kDevTimeout, site);
      return;
    }
  }
}

// Direct epilogue store of one thread's 32 consecutive outputs of row `row`
// starting at column `col0`, masked against M/N; any pitch and alignment.
__device__ __forceinline__ void store_row32(uint16_t* D, uint64_t ldd, uint32_t M, uint32_t N,
                                            uint32_t row, uint32_t col0, const uint32_t (&v)[32]) {
  if (row >= M || col0 >= N) return;
  uint32_t p[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) p[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
  uint16_t* dst = D + static_cast<uint64_t>(row) * ldd + col0;
  const uint32_t n = min(32u, N - col0);
  const uintptr_t a = reinterpret_cast<uintptr_t>(dst);
  if (n == 32 && (a & 15) == 0) {
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int i = 0; i < 4; ++i) d4[i] = make_uint4(p[4 * i], p[4 * i + 1], p[4 * i + 2], p[4 * i + 3]);
  } else if ((a & 3) == 0) {
    uint32_t* d2 = reinterpret_cast<uint32_t*>(dst);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (2 * i + 1 < n) d2[i] = p[i];
      else if (2 * i < n) dst[2 * i] = static_cast<uint16_t>(p[i] & 0xFFFFu);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (2 * i < n) dst[2 * i] = static_cast<uint16_t>(p[i] & 0xFFFFu);
      if (2 * i + 1 < n) dst[2 * i + 1] = static_cast<uint16_t>(p[i] >> 16);
    }
  }
}

// Masked epilogue store of a 32x32 chunk held one row per thread (thread t:
// row row0+t, columns col0..col0+31 as fp32 bits): convert to bf16, stage in
// the warp's 2 KB buffer (16-byte pieces XOR-swizzled by row, conflict free),
// then write row by row with the warp spread over the columns, so each store
// instruction covers one contiguous row segment.  Any pitch and alignment;
// rows >= M and columns >= N are skipped.
__device__ __forceinline__ void store_chunk32_staged(uint8_t* buf, uint16_t* D, uint64_t ldd,
                                                     uint32_t M, uint32_t N, uint32_t row0,
                                                     uint32_t col0, const uint32_t (&v)[32],
                                                     uint32_t lane) {
#pragma unroll
  for (uint32_t j = 0; j < 4; ++j) {
    const uint4 piece = make_uint4(
        pack_bf16x2(__uint_as_float(v[8 * j + 0]), __uint_as_float(v[8 * j + 1])),
        pack_bf16x2(__uint_as_float(v[8 * j + 2]), __uint_as_float(v[8 * j + 3])),
        pack_bf16x2(__uint_as_float(v[8 * j + 4]), __uint_as_float(v[8 * j + 5])),
        pack_bf16x2(__uint_as_float(v[8 * j + 6]), __uint_as_float(v[8 * j + 7])));
    *reinterpret_cast<uint4*>(buf + lane * 64 + ((j ^ ((lane >> 1) & 3u)) << 4)) = piece;
  }
  __syncwarp();
  const uint32_t ncols = min(32u, N - col0);
  const uint32_t nrows = row0 < M ? min(32u, M - row0) : 0u;
  const bool vec = ncols == 32 && ((reinterpret_cast<uintptr_t>(D + col0) | (ldd * 2)) & 15) == 0;
  if (vec) {
    // 16 bytes per lane: lane l covers row 8*i + l/4, piece l%4
#pragma unroll
    for (uint32_t i = 0; i < 4; ++i) {
      const uint32_t r = 8 * i + (lane >> 2), j = lane & 3u;
      if (r < nrows) {
        const uint4 piece = *reinterpret_cast<const uint4*>(buf + r * 64 + ((j ^ ((r >> 1) & 3u)) << 4));
        *reinterpret_cast<uint4*>(D + static_cast<uint64_t>(row0 + r) * ldd + col0 + 8 * j) = piece;
      }
    }
  } else {
    // one bf16 per lane: lane l covers column l of each row
    const uint32_t j = lane >> 3, e = lane & 7u;
#pragma unroll 4
    for (uint32_t r = 0; r < nrows; ++r) {
      if (lane < ncols) {
        const uint16_t x = *reinterpret_cast<const uint16_t*>(buf + r * 64 + ((j ^ ((r >> 1) & 3u)) << 4) + 2 * e);
        D[static_cast<uint64_t>(row0 + r) * ldd + col0 + lane] = x;
      }
    }
  }
  __syncwarp();
}

// store_chunk32_staged for a chunk already converted to 16 packed bf16 pairs.
__device__ __forceinline__ void store_chunk32_packed(uint8_t* buf, uint16_t* D, uint64_t ldd,
                                                     uint32_t M, uint32_t N, uint32_t row0,
                                                     uint32_t col0, const uint32_t (&p)[16],
                                                     uint32_t lane) {
#pragma unroll
  for (uint32_t j = 0; j < 4; ++j)
    *reinterpret_cast<uint4*>(buf + lane * 64 + ((j ^ ((lane >> 1) & 3u)) << 4)) =
        make_uint4(p[4 * j], p[4 * j + 1], p[4 * j + 2], p[4 * j + 3]);
  __syncwarp();
  const uint32_t ncols = min(32u, N - col0);
  const uint32_t nrows = row0 < M ? min(32u, M - row0) : 0u;
  const bool vec = ncols == 32 && ((reinterpret_cast<uintptr_t>(D + col0) | (ldd * 2)) & 15) == 0;
  if (vec) {
#pragma unroll
    for (uint32_t i = 0; i < 4; ++i) {
      const uint32_t r = 8 * i + (lane >> 2), j = lane & 3u;
      if (r < nrows) {
        const uint4 piece = *reinterpret_cast<const uint4*>(buf + r * 64 + ((j ^ ((r >> 1) & 3u)) << 4));
        *reinterpret_cast<uint4*>(D + static_cast<uint64_t>(row0 + r) * ldd + col0 + 8 * j) = piece;
      }
    }
  } else {
    const uint32_t j = lane >> 3, e = lane & 7u;
#pragma unroll 4
    for (uint32_t r = 0; r < nrows; ++r) {
      if (lane < ncols) {
        const uint16_t x = *reinterpret_cast<const uint16_t*>(buf + r * 64 + ((j ^ ((r >> 1) & 3u)) << 4) + 2 * e);
        D[static_cast<uint64_t>(row0 + r) * ldd + col0 + lane] = x;
      }
    }
  }
  __syncwarp();
}

// ------------------------------------------------------------ fused epilogue

__device__ __forceinline__ float epi_act(float x, uint32_t act) {
  if (act == kActRelu) return x < 0.0f ? 0.0f : x;                        // NaN kept
  if (act == kActGelu) return 0.5f * x * (1.0f + erff(x * 0.70710678118654752f));
  return x;
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t h) { return __uint_as_float(h << 16); }

// 32 consecutive values starting at p (the first n valid, the rest 0) of
// fp32 or bf16 type, with 16-byte loads where the address allows.
template <bool F32>
__device__ __forceinline__ void load_row32(const void* p, uint32_t n, float (&x)[32]) {
  if constexpr (F32) {
    const float* q = static_cast<const float*>(p);
    if (n == 32 && (reinterpret_cast<uintptr_t>(q) & 15u) == 0) {
#pragma unroll
      for (uint32_t i = 0; i < 8; ++i) {
        const float4 t = __ldg(reinterpret_cast<const float4*>(q) + i);
        x[4 * i] = t.x; x[4 * i + 1] = t.y; x[4 * i + 2] = t.z; x[4 * i + 3] = t.w;
      }
    } else {
#pragma unroll
      for (uint32_t t = 0; t < 32; ++t) x[t] = t < n ? __ldg(q + t) : 0.0f;
    }
  } else {
    const uint16_t* q = static_cast<const uint16_t*>(p);
    if (n == 32 && (reinterpret_cast<uintptr_t>(q) & 15u) == 0) {
#pragma unroll
      for (uint32_t i = 0; i < 4; ++i) {
        const uint4 t = __ldg(reinterpret_cast<const uint4*>(q) + i);
        const uint32_t w[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
        for (uint32_t k = 0; k < 4; ++k) {
          x[8 * i + 2 * k] = bf16_bits_to_f32(w[k] & 0xFFFFu);
          x[8 * i + 2 * k + 1] = bf16_bits_to_f32(w[k] >> 16);
        }
      }
    } else {
#pragma unroll
      for (uint32_t t = 0; t < 32; ++t) x[t] = t < n ? bf16_bits_to_f32(__ldg(q + t)) : 0.0f;
    }
  }
}

// The fused epilogue on one thread's 32 accumulators: row `row`, columns
// col0 .. col0 + 31 (columns >= N and rows >= M read nothing):
// v = alpha * acc + beta * C[row, col] + bias[col], then the activation, in fp32.
// cpk: this row's 32 bf16 values of C already in registers (packed pairs,
// element 2t in the low half of word t), or nullptr to load them here.
__device__ __forceinline__ void epi_apply(uint32_t (&v)[32], const GemmArgs& a, uint32_t row,
                                          uint32_t col0, const uint32_t* cpk = nullptr) {
  const uint32_t mode = a.epi_mode;
  const uint32_t n = col0 < a.N ? min(32u, a.N - col0) : 0u;
  float x[32];
#pragma unroll
  for (uint32_t t = 0; t < 32; ++t) x[t] = __uint_as_float(v[t]);
  if (mode & kEpiAlpha) {
#pragma unroll
    for (uint32_t t = 0; t < 32; ++t) x[t] *= a.alpha;
  }
  if ((mode & kEpiC) && row < a.M && n > 0) {
    float c[32];
    if (cpk != nullptr) {
#pragma unroll
      for (uint32_t t = 0; t < 16; ++t) {
        c[2 * t] = bf16_bits_to_f32(cpk[t] & 0xFFFFu);
        c[2 * t + 1] = bf16_bits_to_f32(cpk[t] >> 16);
      }
    } else if (mode & kEpiOutF32)
      load_row32<true>(static_cast<const float*>(a.C) + static_cast<uint64_t>(row) * a.ldc + col0, n, c);
    else
      load_row32<false>(static_cast<const uint16_t*>(a.C) + static_cast<uint64_t>(row) * a.ldc + col0, n, c);
#pragma unroll
    for (uint32_t t = 0; t < 32; ++t) x[t] = fmaf(a.beta, c[t], x[t]);
  }
  if ((mode & kEpiBias) && n > 0) {
    float b[32];
    if (mode & kEpiBiasF32)
      load_row32<true>(static_cast<const float*>(a.bias) + col0, n, b);
    else
      load_row32<false>(static_cast<const uint16_t*>(a.bias) + col0, n, b);
#pragma unroll
    for (uint32_t t = 0; t < 32; ++t) x[t] += b[t];
  }
  const uint32_t act = (mode >> kEpiActShift) & 3u;
  if (act != 0) {
#pragma unroll
    for (uint32_t t = 0; t < 32; ++t) x[t] = epi_act(x[t], act);
  }
#pragma unroll
  for (uint32_t t = 0; t < 32; ++t) v[t] = __float_as_uint(x[t]);
}

// fp32 output: one thread's row segment of 32 values (one 128-byte line when
// aligned), masked against M and N.
__device__ __forceinline__ void store_row32_f32(float* D, uint64_t ldd, uint32_t M, uint32_t N,
                                                uint32_t row, uint32_t col0, const uint32_t (&v)[32]) {
  if (row >= M || col0 >= N) return;
  const uint32_t n = min(32u, N - col0);
  float* dp = D + static_cast<uint64_t>(row) * ldd + col0;
  if (n == 32 && (reinterpret_cast<uintptr_t>(dp) & 15u) == 0) {
#pragma unroll
    for (uint32_t i = 0; i < 8; ++i)
      reinterpret_cast<float4*>(dp)[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                                     __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
  } else {
#pragma unroll
    for (uint32_t t = 0; t < 32; ++t)
      if (t < n) dp[t] = __uint_as_float(v[t]);
  }
}

// PLAIN: a build for plain launches -- whole tiles (column halves included)
// and D = A B^T stored as bf16, with the stream-K, fused-epilogue and
// C-by-TMA code compiled out.  The smaller kernel measured 0.5-2% faster on
// bf16 and 2.5% on the tiled-scale MXFP8 pair than the general build running
// the same launches.
template <int CG, Kind KIND, bool TMA_STORE, bool EPI2 = false, bool PLAIN = false>
__global__ void __launch_bounds__(GemmCfg<CG, KIND, TMA_STORE, EPI2>::kThreads, 1)
    gemm_ws_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmD,
                   const __grid_constant__ CUtensorMap tmSFA,
                   const __grid_constant__ CUtensorMap tmSFB,
                   const __grid_constant__ CUtensorMap tmBh,
                   const __grid_constant__ CUtensorMap tmC, const GemmArgs args) {
  using C = GemmCfg<CG, KIND, TMA_STORE, EPI2>;
  // the launch's fused-epilogue mode and C-by-TMA flag (none in a plain build)
  constexpr bool EDGE = PLAIN && KIND == Kind::BF16;   // builds that honour edge_last
  const uint32_t epi_mode = PLAIN ? 0u : args.epi_mode;
  const uint32_t c_tma = PLAIN ? 0u : args.c_tma;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - raw);
  const uint32_t stage0 = base;
  const uint32_t sf0 = base + C::STAGES * C::STAGE_BYTES;
  const uint32_t epi0 = sf0 + C::SF_BYTES;
  const uint32_t bar0 = epi0 + C::EPI_BYTES;
  const auto full_bar = [&](uint32_t s) { return bar0 + 8 * s; };
  const auto empty_bar = [&](uint32_t s) { return bar0 + 8 * (C::STAGES + s); };
  constexpr uint32_t kSfBar0 = 2 * C::STAGES;
  const auto raw_full_bar = [&](uint32_t g) { return bar0 + 8 * (kSfBar0 + g); };
  constexpr uint32_t kTBar0 = kSfBar0 + C::RAW_SLOTS;
  const auto t_ready_bar = [&](uint32_t g) { return bar0 + 8 * (kTBar0 + g); };
  const auto t_empty_bar = [&](uint32_t g) { return bar0 + 8 * (kTBar0 + C::T_SLOTS + g); };
  constexpr uint32_t kAccBar0 = kTBar0 + 2 * C::T_SLOTS;
  const uint32_t raw0 = sf0;                                       // raw slots, then re-tiled slots
  const uint32_t t0 = sf0 + C::RAW_SLOTS * C::RAW_SLOT_BYTES;
  const auto accf_bar = [&](uint32_t b) { return bar0 + 8 * (kAccBar0 + b); };
  const auto acce_bar = [&](uint32_t b) { return bar0 + 8 * (kAccBar0 + 2 + b); };
  const uint32_t drain_bar = bar0 + 8 * (kAccBar0 + 4);
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + (bar0 - base) + 8 * (kAccBar0 + 5));
  constexpr uint32_t kFixBar0 = kAccBar0 + 6;
  // one barrier per epilogue warp of group 0: its TMA-loaded C chunk landed
  constexpr uint32_t kCBar0 = kFixBar0 + C::FIX_TOTAL;
  // tiled scales: one per stage, the stage's scale chunks landed
  constexpr uint32_t kSfStageBar0 = kCBar0 + 4;
  const auto sf_full_bar = [&](uint32_t s) { return bar0 + 8 * (kSfStageBar0 + s); };
  volatile uint32_t* const abort_flag = tmem_slot + 1;

  const uint32_t warp = warp_idx_sync();
  const uint32_t lane = lane_idx();
  const uint32_t rank = (CG == 2) ? cluster_cta_rank() : 0u;
  const bool leader = rank == 0;
  const uint32_t cluster_id = blockIdx.x / CG;
  const uint32_t num_clusters = gridDim.x / CG;
  const Watchdog wd{args.status, args.timeout_ns, abort_flag};

  // ---- set-up: descriptor prefetches and barriers (warp 0, the barriers one
  // per lane), TMEM allocation (warp 1) ----------------------------------------
  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      if (args.half_tiles != 0 || args.edge_half != 0) tma_prefetch_desc(&tmBh);
      if (c_tma != 0) tma_prefetch_desc(&tmC);
      if constexpr (TMA_STORE) tma_prefetch_desc(&tmD);
      if (C::MX && !args.sf_gather) {
        tma_prefetch_desc(&tmSFA);
        tma_prefetch_desc(&tmSFB);
      }
      *abort_flag = 0u;
    }
    // Arrival counts: the producer's expect_tx (ready barriers), one commit
    // (free, accumulator-full, drain, scale-slot-free barriers), one arrival
    // per transfer (fix-up ring, C chunks), and
    //   t_ready: every CTA's scale-factor warp once per group (tiled scales:
    //            the copy thread's commit);
    //   acc_empty: every epilogue warp of the pair.
    constexpr uint32_t kNumBars = kCBar0 + 4 + (C::SF_TILED ? C::STAGES : 0u);
    static_assert(kNumBars * 8 <= C::BAR_BYTES && C::FULL_ARRIVALS == 1, "barrier area");
    for (uint32_t i = lane; i < kNumBars; i += 32) {
      if (i == kAccBar0 + 5) continue;   // the TMEM address and the abort flag
      uint32_t count = 1;
      if (i >= kTBar0 && i < kTBar0 + C::T_SLOTS) count = C::SF_TILED ? 1u : static_cast<uint32_t>(CG);
      if (i >= kAccBar0 + 2 && i < kAccBar0 + 4) count = 4 * CG * C::EPI_WG;
      mbar_init(bar0 + 8 * i, count);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc<CG>(smem_addr(tmem_slot), C::TMEM_COLS);
    tmem_relinquish<CG>();
  }
  tc_fence_before_sync();
  __syncthreads();
  if constexpr (CG == 2) cluster_sync();
  tc_fence_after_sync();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

  const uint32_t KT = args.num_k_tiles;

  if (warp == 0) {
    // ==================== TMA producer: one elected thread ====================
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_last();
      uint32_t it = 0;
      bool ok = true;
      WorkItem w;
      for (uint32_t wi = 0; ok && work_item<!PLAIN, EDGE>(args, cluster_id, num_clusters, KT, wi, w); ++wi) {
        uint32_t mb, nb;
        item_coords<EDGE>(args, w.tile, mb, nb);
        const int32_t a_row = static_cast<int32_t>(mb * C::UMMA_M + rank * C::BLOCK_M);
        // this CTA's share of the item's B rows: B_ROWS, or half of them
        // for a column half (through the half-height box of tmBh)
        const uint32_t n0 = item_n0(w, nb, C::UMMA_N);
        const int32_t b_row = static_cast<int32_t>(n0 + rank * (item_cols(w, C::UMMA_N) / CG));
        const CUtensorMap* const mapB = w.half != 0 ? &tmBh : &tmB;
        const uint32_t tx = w.half != 0 ? C::AB_TX - C::B_BYTES / 2 : C::AB_TX;
        for (uint32_t kt = w.k_begin; kt < w.k_end; ++kt, ++it) {
          const uint32_t s = it % C::STAGES;
          const uint32_t round = it / C::STAGES;
          if (it == args.stall_iter) continue;   // watchdog test: this stage never fills
          // free barrier: the MMA that last read this slot has completed
          if (!wait_bounded(empty_bar(s), (round & 1u) ^ 1u, wd, kSiteProducerEmpty)) {
            ok = false;
            break;
          }
          const uint32_t sb = stage0 + s * C::STAGE_BYTES;
          const int32_t kx = static_cast<int32_t>(kt * C::BK);
          // Tiled scales: the K-tile's chunk of this CTA's A row block, then
          // those of the tile's B row blocks (one box each).
          const int32_t sfa_blk = static_cast<int32_t>(static_cast<uint32_t>(a_row) / 128u);
          const int32_t sfb_blk = static_cast<int32_t>(n0 / 128u);
          if constexpr (CG == 1) {
            if constexpr (C::SF_TILED) {
              mbar_arrive_expect_tx(sf_full_bar(s), C::SF_STAGE_BYTES);
              tma_load_3d(sb + C::OFF_SF, &tmSFA, sf_full_bar(s), 0, static_cast<int32_t>(kt), sfa_blk, pol);
              tma_load_3d(sb + C::OFF_SF + 512, &tmSFB, sf_full_bar(s), 0, static_cast<int32_t>(kt), sfb_blk,
                          pol);
            }
            mbar_arrive_expect_tx(full_bar(s), tx);
            tma_load_2d(sb, &tmA, full_bar(s), kx, a_row, pol);
            tma_load_2d(sb + C::OFF_B, mapB, full_bar(s), kx, b_row, pol);
          } else {
            // both CTAs' bytes land on the leader's barriers
            if constexpr (C::SF_TILED) {
              const uint32_t leader_sf = mapa_shared(sf_full_bar(s), 0);
              if (leader) mbar_arrive_expect_tx(sf_full_bar(s), CG * C::SF_STAGE_BYTES);
              tma_load_3d_pair(sb + C::OFF_SF, &tmSFA, leader_sf, 0, static_cast<int32_t>(kt), sfa_blk, pol);
              tma_load_3d_pair(sb + C::OFF_SF + 512, &tmSFB, leader_sf, 0, static_cast<int32_t>(kt), sfb_blk,
                               pol);
            }
            const uint32_t leader_full = mapa_shared(full_bar(s), 0);
            if (leader) mbar_arrive_expect_tx(full_bar(s), CG * tx);
            tma_load_2d_pair(sb, &tmA, leader_full, kx, a_row, pol);
            tma_load_2d_pair(sb + C::OFF_B, mapB, leader_full, kx, b_row, pol);
          }
        }
      }
      // Exit path after a give-up: let this CTA's issued loads land first.
      if (*abort_flag) {
        const uint32_t first = it > C::STAGES ? it - C::STAGES : 0u;
        if (leader)
          for (uint32_t i = first; i < it; ++i)
            if (i != args.stall_iter) {
              drain_wait(full_bar(i % C::STAGES), (i / C::STAGES) & 1u, wd, kSiteProducerDrain);
              if constexpr (C::SF_TILED)
                drain_wait(sf_full_bar(i % C::STAGES), (i / C::STAGES) & 1u, wd, kSiteProducerDrain);
            }
      }
    }
  } else if (warp == 1) {
    // ==================== MMA issuer: one thread of the leader CTA ==============
    // A single thread waits and issues: no warp-collective steps sit between
    // consecutive MMAs (an FP8 K-tile is only ~450 tensor cycles).
    if (leader && lane == 0) {
      uint32_t it = 0, j = 0, gi = 0;
      bool issued = false;
      WorkItem w;
      for (uint32_t wi = 0; work_item<!PLAIN, EDGE>(args, cluster_id, num_clusters, KT, wi, w); ++wi, ++j) {
        const uint32_t b = j % C::ACC_STAGES;
        const uint32_t around = j / C::ACC_STAGES;
        // accumulator b must have been drained by every epilogue warp
        if (!wait_bounded(acce_bar(b), (around & 1u) ^ 1u, wd, kSiteMmaAccEmpty)) break;
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + b * C::UMMA_N;
        // N of this item's MMAs: the item's columns; in the one-CTA bf16
        // kernels only those inside N, rounded up to the epilogue's chunk (a
        // tile at the right edge of D with 5 live columns multiplies 64, not
        // 256).  Not in the pair: there the MMA takes N / 2 B rows from each
        // CTA's stage, so its N is tied to the height of the B box the
        // producer loaded (UMMA_N / 2 rows, or a quarter for a column half).
        uint32_t n_mma = item_cols(w, C::UMMA_N);
        if constexpr (KIND == Kind::BF16 && CG == 1) {
          uint32_t mb, nb;
          item_coords<EDGE>(args, w.tile, mb, nb);
          const uint32_t n0 = item_n0(w, nb, C::UMMA_N);
          constexpr uint32_t kChunk = TMA_STORE ? C::TS_COLS : 32u;
          const uint32_t live_cols = args.N > n0 ? args.N - n0 : 0u;
          const uint32_t need = live_cols == 0 ? kChunk : (live_cols + kChunk - 1) / kChunk * kChunk;
          if (need < n_mma) n_mma = need;
        }
        bool ok = true;
        // Unrolled in the pair kernels (measured: +1-3% bf16 with 4, +2.4% MXFP8 with 2;
        // the one-CTA MXFP8 kernel measured slightly slower unrolled).
#pragma unroll(C::MMA_UNROLL)
        for (uint32_t kt = w.k_begin; kt < w.k_end; ++kt, ++it) {
          const uint32_t s = it % C::STAGES;
          const uint32_t round = it / C::STAGES;
          const uint32_t g = gi % C::T_SLOTS;
          if constexpr (C::SF_WARP) {
            // first K-tile of a scale-factor group: every CTA filled the slot
            if (kt % C::SF_GROUP == 0 &&
                !wait_bounded(t_ready_bar(g), (gi / C::T_SLOTS) & 1u, wd, kSiteMmaFull)) {
              ok = false;
              break;
            }
          }
          if (!wait_bounded(full_bar(s), round & 1u, wd, kSiteMmaFull)) {
            ok = false;
            break;
          }
          // tiled scales: the copy thread has written this K-tile's scale set
          if (C::SF_TILED &&
              !wait_bounded(t_ready_bar(it % C::SF_SETS), (it / C::SF_SETS) & 1u, wd, kSiteMmaFull)) {
            ok = false;
            break;
          }
          const uint32_t sb = stage0 + s * C::STAGE_BYTES;
          tc_fence_after_sync();
          const uint64_t adesc = smem_desc_sw128(sb);
          const uint64_t bdesc = smem_desc_sw128(sb + C::OFF_B);
          if constexpr (C::MX) {
            const uint32_t sfa_t = tmem_base + C::SF_TMEM_COL + (it % C::SF_SETS) * C::SF_SET_COLS;
            const uint32_t sfb_t = sfa_t + 4;
            if constexpr (C::SF_WARP) {
              // the K-tile's chunks in the re-tiled slot of its group
              const uint32_t tsrc = t0 + g * C::T_SLOT_BYTES + (kt % C::SF_GROUP) * C::T_PER_KT;
              tmem_cp_32x128b_warpx4<CG>(sfa_t, smem_desc_rows16(tsrc));
#pragma unroll
              for (uint32_t h = 0; h < C::SFB_CHUNKS; ++h)
                tmem_cp_32x128b_warpx4<CG>(sfb_t + 4 * h, smem_desc_rows16(tsrc + 512 * (1 + h)));
            }
#pragma unroll
            for (uint32_t k = 0; k < C::K_STEPS; ++k)
              mma_mxf8<CG>(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc_mxf8(C::UMMA_M, n_mma, k, k),
                           sfa_t, sfb_t, (kt != w.k_begin || k != 0u));
          } else {
            const uint32_t idesc = idesc_bf16(C::UMMA_M, n_mma);
#pragma unroll
            for (uint32_t k = 0; k < C::K_STEPS; ++k)
              mma_bf16<CG>(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc, (kt != w.k_begin || k != 0u));
          }
          commit_to<CG>(empty_bar(s));   // frees the stage once these MMAs finish
          if (C::SF_WARP && (kt % C::SF_GROUP == C::SF_GROUP - 1 || kt + 1 == w.k_end)) {
            commit_to<CG>(t_empty_bar(g));   // and the re-tiled scale slot
            ++gi;
          }
          issued = true;
        }
        if (!ok) break;
        commit_to<CG>(accf_bar(b));   // accumulator b complete
      }
      // Exit path: every tcgen05 op this thread issued completes before TMEM
      // is released.
      if (issued) {
        if constexpr (CG == 1)
          tc_commit(drain_bar);
        else
          tc_commit_pair_multicast(drain_bar, 0x1);
        drain_wait(drain_bar, 0, wd, kSiteMmaDrain);
      }
    }
  } else if (C::SF_TILED && warp == C::kCpWarp) {
    // ==================== scale copies: one thread of the leader CTA ==============
    // For each K-tile, once its stage's scale chunks have landed and the MMAs
    // of the K-tile SF_SETS back (which read the same scale set) have completed, copy its
    // scale chunks from the stage into scale set it % SF_SETS and commit to
    // that set's barrier.  tcgen05 operations of different threads are ordered only
    // through these commits and barrier waits.
    if (leader && lane == 0) {
      uint32_t it = 0;
      bool issued = false, ok = true;
      WorkItem w;
      for (uint32_t wi = 0; ok && work_item<!PLAIN, EDGE>(args, cluster_id, num_clusters, KT, wi, w); ++wi) {
        for (uint32_t kt = w.k_begin; kt < w.k_end; ++kt, ++it) {
          const uint32_t s = it % C::STAGES;
          if (!wait_bounded(sf_full_bar(s), (it / C::STAGES) & 1u, wd, kSiteSfFull)) { ok = false; break; }
          if (it >= C::SF_SETS) {
            const uint32_t p = it - C::SF_SETS;   // the K-tile whose MMAs read this set last
            if (!wait_bounded(empty_bar(p % C::STAGES), (p / C::STAGES) & 1u, wd, kSiteSfFull)) {
              ok = false;
              break;
            }
          }
          tc_fence_after_sync();
          const uint32_t sb = stage0 + s * C::STAGE_BYTES;
          const uint32_t sfa_t = tmem_base + C::SF_TMEM_COL + (it % C::SF_SETS) * C::SF_SET_COLS;
          tmem_cp_32x128b_warpx4<CG>(sfa_t, smem_desc_rows16(sb + C::OFF_SF));
#pragma unroll
          for (uint32_t h = 0; h < C::SFB_CHUNKS; ++h)
            tmem_cp_32x128b_warpx4<CG>(sfa_t + 4 + 4 * h, smem_desc_rows16(sb + C::OFF_SF + 512 * (1 + h)));
          if constexpr (CG == 1)
            tc_commit(t_ready_bar(it % C::SF_SETS));
          else
            tc_commit_pair_multicast(t_ready_bar(it % C::SF_SETS), 0x1);
          issued = true;
        }
      }
      // Exit path: this thread's copies complete before TMEM is released.
      if (issued) {
        if constexpr (CG == 1)
          tc_commit(t_empty_bar(0));
        else
          tc_commit_pair_multicast(t_empty_bar(0), 0x1);
        drain_wait(t_empty_bar(0), 0, wd, kSiteMmaDrain);
      }
    }
  } else if (C::SF_WARP && warp == C::kSfWarp) {
    // ==================== scale-factor warp (every CTA) ===========================
    // Load this CTA's scale bytes group by group (RAW_SLOTS groups ahead),
    // re-tile each landed group into the tcgen05.cp layout and report it to
    // the leader's slot-ready barrier (one arrival per CTA and group).  A
    // cursor walks (work item, group) in the MMA issuer's order; K ranges
    // start on group boundaries (stream-K units are whole groups).
    struct GroupCursor {
      uint32_t wi, q;
      WorkItem w;
      bool valid;
    };
    const auto cur_first = [&](GroupCursor& g) {
      g.wi = 0;
      g.q = 0;
      g.valid = work_item<!PLAIN, EDGE>(args, cluster_id, num_clusters, KT, 0, g.w);
    };
    const auto cur_next = [&](GroupCursor& g) {
      if (!g.valid) return;
      const uint32_t ng = (g.w.k_end - g.w.k_begin + C::SF_GROUP - 1) / C::SF_GROUP;
      if (++g.q < ng) return;
      g.q = 0;
      ++g.wi;
      g.valid = work_item<!PLAIN, EDGE>(args, cluster_id, num_clusters, KT, g.wi, g.w);
    };
    const uint64_t pol = l2_policy_evict_last();
    const uint32_t nblk = (args.K + 31u) / 32u;
    // Loads of one group into raw slot gi % RAW_SLOTS (called by the whole
    // warp): two TMA boxes issued by lane 0, or, for scale pitches TMA cannot
    // take, a plain-load gather by every lane into the same layout followed by
    // lane 0's arrival (the slot is then full when the barrier's phase ends,
    // as after the TMA bytes).
    const auto load_group = [&](const GroupCursor& g, uint32_t gi) {
      uint32_t mb, nb;
      item_coords<EDGE>(args, g.w.tile, mb, nb);
      const uint32_t r = gi % C::RAW_SLOTS;
      const uint32_t slot = raw0 + r * C::RAW_SLOT_BYTES;
      const uint32_t kb0 = (g.w.k_begin / C::SF_GROUP + g.q) * 16;
      const uint32_t a_row = mb * C::UMMA_M + rank * C::BLOCK_M;
      const uint32_t b_row = nb * C::UMMA_N;
      if (!args.sf_gather) {
        if (lane == 0) {
          mbar_arrive_expect_tx(raw_full_bar(r), C::SF_TX);
          tma_load_2d(slot + C::OFF_SFA_RAW, &tmSFA, raw_full_bar(r), static_cast<int32_t>(kb0),
                      static_cast<int32_t>(a_row), pol);
          tma_load_2d(slot + C::OFF_SFB_RAW, &tmSFB, raw_full_bar(r), static_cast<int32_t>(kb0),
                      static_cast<int32_t>(b_row), pol);
        }
      } else {
        uint8_t* const sp = base_ptr + (slot - base);
        gather_scale_rows<C::BLOCK_M>(sp + C::OFF_SFA_RAW, args.sfa, args.ldsfa, a_row, args.M,
                                      kb0, nblk, lane);
        gather_scale_rows<C::SFB_ROWS>(sp + C::OFF_SFB_RAW, args.sfb, args.ldsfb, b_row, args.N,
                                       kb0, nblk, lane);
        __syncwarp();
        if (lane == 0) mbar_arrive(raw_full_bar(r));
      }
    };
    GroupCursor lc, pc;   // load cursor (RAW_SLOTS ahead) and processing cursor
    cur_first(lc);
    cur_first(pc);
    uint32_t issued = 0;
    for (; issued < C::RAW_SLOTS && lc.valid; ++issued, cur_next(lc)) load_group(lc, issued);
    __syncwarp();
    uint32_t gi = 0;
    for (; pc.valid; ++gi, cur_next(pc)) {
      const uint32_t gr = gi % C::RAW_SLOTS;
      const uint32_t gt = gi % C::T_SLOTS;
      // the scale bytes have landed, and the MMAs that read this re-tiled slot
      // last time have completed
      if (!warp_wait(raw_full_bar(gr), (gi / C::RAW_SLOTS) & 1u, wd, kSiteSfFull, lane) ||
          !warp_wait(t_empty_bar(gt), ((gi / C::T_SLOTS) & 1u) ^ 1u, wd, kSiteSfFull, lane))
        break;
      const uint8_t* const rp = base_ptr + (raw0 + gr * C::RAW_SLOT_BYTES - base);
      uint8_t* const tp = base_ptr + (t0 + gt * C::T_SLOT_BYTES - base);
      retile_scales<1>(rp + C::OFF_SFA_RAW, tp, C::T_PER_KT, 0, C::BLOCK_M, lane);
      retile_scales<C::SFB_CHUNKS>(rp + C::OFF_SFB_RAW, tp, C::T_PER_KT, C::SFA_T, C::SFB_ROWS,
                                   lane);
      fence_proxy_async_smem();
      __syncwarp();   // every lane's reads of the raw slot are done
      if (lane == 0) {
        if constexpr (CG == 1)
          mbar_arrive(t_ready_bar(gt));
        else
          mbar_arrive_cluster(mapa_shared(t_ready_bar(gt), 0));
      }
      if (lc.valid) {   // refill this raw slot with the next group to load
        load_group(lc, issued);
        ++issued;
        cur_next(lc);
      }
      __syncwarp();
    }
    // Exit path after a give-up: let this warp's scale loads still in flight
    // land (a gathered slot's phase has already completed).
    if (lane == 0 && *abort_flag && !args.sf_gather)
      for (uint32_t i = gi; i < issued; ++i)
        drain_wait(raw_full_bar(i % C::RAW_SLOTS), (i / C::RAW_SLOTS) & 1u, wd, kSiteProducerDrain);
  } else if ((warp >= 2 && warp < 6) ||
             (C::EPI_WG == 2 && warp >= C::kEpiWg1Warp && warp < C::kEpiWg1Warp + 4)) {
    // ==================== epilogue: four warps per group, one TMEM lane quarter each ===
    constexpr uint32_t NG = C::EPI_WG;
    const uint32_t eg = warp < 6 ? 0u : 1u;  // epilogue group: the chunks c with c % NG == eg
    const uint32_t q = warp & 3u;            // TMEM lanes 32q .. 32q+31
    const uint32_t ew = eg == 0 ? warp - 2u : 4u + warp - C::kEpiWg1Warp;   // staging slot owner
    uint32_t j = 0, chunk_ctr = 0;
    bool ok = true;
    // the 32 x UMMA_N fp32 slice of a stream-K partial slot for this lane
    // quarter (chunk c of 32 columns at float offset 1024 c), and this warp's
    // flag in it (one per lane quarter and group: 8 words per CTA slot)
    const auto part_ptr = [&](uint32_t slot) {
      return args.ws_part + (static_cast<uint64_t>(slot * CG + rank) * 4 + q) * (32u * C::UMMA_N);
    };
    const auto flag_ptr = [&](uint32_t slot) {
      return args.ws_flag + ((slot * CG + rank) * 4 + q) * 2 + eg;
    };
    const uint32_t ring = (q * NG + eg) * C::FIX_SLOTS;   // this warp's fix-up slots
    // C by TMA (args.c_tma; kernels with one epilogue group and two 64-column
    // staging buffers per warp): chunk c of an item's C lands in the second
    // buffer; the first chunk is requested before the accumulator wait, each
    // next one as soon as the current one has been read into registers.
    constexpr bool kCTma = TMA_STORE && C::TS_COLS == 64 && C::EPI_BUFS == 2;
    const uint32_t cbuf = epi0 + (ew * C::EPI_BUFS + 1) * C::EPI_BUF_BYTES;
    const uint32_t c_bar = bar0 + 8 * (kCBar0 + (ew & 3u));
    const uint64_t pol_c = l2_policy_evict_first();
    uint32_t c_issued = 0, c_done = 0;
    const auto issue_c = [&](uint32_t r0, uint32_t col) {
      fence_proxy_async_smem();   // the lanes' reads of the buffer come first
      mbar_arrive_expect_tx(c_bar, C::EPI_BUF_BYTES);
      tma_load_2d(cbuf, &tmC, c_bar, static_cast<int32_t>(col), static_cast<int32_t>(r0), pol_c);
    };
    const auto fix_slot = [&](uint32_t r) { return stage0 + (ring + r) * C::FIX_SLOT_BYTES; };
    const auto fix_bar = [&](uint32_t r) { return bar0 + 8 * (kFixBar0 + ring + r); };
    // owner-side transfer stream: transfer n = this warp's (n / nc)-th chunk
    // (chunk (n / nc) NG + eg) of contributor cluster_id + 1 + (n % nc);
    // issued FIX_SLOTS ahead by lane 0
    uint32_t nc = 0, nfix = 0, fix_issued = 0, fix_done = 0;
    const auto issue_fix = [&](uint32_t n) {
      const uint32_t r = n % C::FIX_SLOTS;
      mbar_arrive_expect_tx(fix_bar(r), C::FIX_SLOT_BYTES);
      bulk_load_1d(fix_slot(r), part_ptr(cluster_id + 1 + n % nc) + ((n / nc) * NG + eg) * 1024u,
                   C::FIX_SLOT_BYTES, fix_bar(r));
    };
    // v += every contributor's partial of chunk c (c % NG == eg; contributor order)
    const auto add_partials = [&](uint32_t (&v)[32], uint32_t c) -> bool {
      for (uint32_t i = 0; i < nc; ++i) {
        const uint32_t n = (c / NG) * nc + i;
        const uint32_t r = n % C::FIX_SLOTS;
        if (!warp_wait(fix_bar(r), (n / C::FIX_SLOTS) & 1u, wd, kSiteStreamKFlag, lane)) return false;
        const float4* src = reinterpret_cast<const float4*>(base_ptr + (fix_slot(r) - base));
#pragma unroll
        for (uint32_t i4 = 0; i4 < 8; ++i4) {
          const float4 p = src[i4 * 32 + lane];
          v[4 * i4 + 0] = __float_as_uint(__uint_as_float(v[4 * i4 + 0]) + p.x);
          v[4 * i4 + 1] = __float_as_uint(__uint_as_float(v[4 * i4 + 1]) + p.y);
          v[4 * i4 + 2] = __float_as_uint(__uint_as_float(v[4 * i4 + 2]) + p.z);
          v[4 * i4 + 3] = __float_as_uint(__uint_as_float(v[4 * i4 + 3]) + p.w);
        }
        __syncwarp();   // every lane has read the slot
        ++fix_done;
        if (fix_issued < nfix) {
          if (lane == 0) issue_fix(fix_issued);
          ++fix_issued;
        }
      }
      return true;
    };
    WorkItem w;
    for (uint32_t wi = 0; ok && work_item<!PLAIN, EDGE>(args, cluster_id, num_clusters, KT, wi, w); ++wi, ++j) {
      const uint32_t b = j % C::ACC_STAGES;
      const uint32_t around = j / C::ACC_STAGES;
      if constexpr (kCTma) {
        if (c_tma != 0 && w.kind != 2) {
          uint32_t mb0, nb0;
          item_coords<EDGE>(args, w.tile, mb0, nb0);
          const uint32_t r0 = mb0 * C::UMMA_M + rank * C::BLOCK_M + q * 32;
          const uint32_t c0 = item_n0(w, nb0, C::UMMA_N);
          if (r0 < args.M && c0 < args.N) {
            if (lane == 0) issue_c(r0, c0);
            ++c_issued;
          }
        }
      }
      if (!warp_wait(accf_bar(b), around & 1u, wd, kSiteEpiAccFull, lane)) break;
      tc_fence_after_sync();
      uint32_t mb, nb;
      item_coords<EDGE>(args, w.tile, mb, nb);
      const uint32_t row0 = mb * C::UMMA_M + rank * C::BLOCK_M + q * 32;
      const uint32_t col_base = item_n0(w, nb, C::UMMA_N);
      const uint32_t t_addr = tmem_base + ((q * 32u) << 16) + b * C::UMMA_N;
      // 32-column chunks of this item inside N (none for a column half past N)
      const uint32_t item_nch = item_cols(w, C::UMMA_N) / 32u;
      const uint32_t live = col_base < args.N ? min(item_nch, (args.N - col_base + 31u) / 32u) : 0u;
      if constexpr (C::SF_TILED) {
        // One accumulator, handed back early: this group's 128 columns go to
        // registers as packed bf16 (4 chunks of 32, 64 words), the issuer is
        // told the accumulator is free, and only then are the values staged
        // and stored -- under the next tile's MMAs.  (The tiled-scale entry
        // point has no stream-K or fused epilogue: whole tiles, plain store.)
        // Chunks of group eg: the 32-column chunks eg, eg + 2, eg + 4, eg + 6.
        static_assert(C::UMMA_N == 256 && NG == 2 && C::TS_COLS == 32, "early release: 4 chunks of 32");
        const auto chunk = [&](uint32_t i) -> uint32_t { return 2 * i + eg; };
        uint32_t pk[4][16];
        const bool rows_live = row0 < args.M;
        if (rows_live) {
#pragma unroll
          for (uint32_t i = 0; i < 4; ++i) {
            if (chunk(i) < live) {
              uint32_t v[32];
              tmem_ld_32x32b_x32_sync(t_addr + chunk(i) * 32, v);
#pragma unroll
              for (uint32_t t = 0; t < 16; ++t)
                pk[i][t] = pack_bf16x2(__uint_as_float(v[2 * t]), __uint_as_float(v[2 * t + 1]));
            }
          }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) {
          if constexpr (CG == 1)
            mbar_arrive(acce_bar(b));
          else
            mbar_arrive_cluster(mapa_shared(acce_bar(b), 0));
        }
        if (rows_live) {
          if constexpr (TMA_STORE) {
#pragma unroll
            for (uint32_t i = 0; i < 4; ++i) {
              if (chunk(i) < live) {
                const uint32_t buf = epi0 + (ew * C::EPI_BUFS + (chunk_ctr % C::EPI_BUFS)) * C::EPI_BUF_BYTES;
                if (lane == 0) bulk_wait_group_read<C::EPI_BUFS - 1>();   // the buffer's last store has read it
                __syncwarp();
                uint8_t* rowp = base_ptr + (buf - base) + lane * 64;
#pragma unroll
                for (uint32_t j = 0; j < 4; ++j)
                  // 64-byte swizzle: 16-byte chunk j of row r sits at chunk j ^ ((r / 2) % 4)
                  *reinterpret_cast<uint4*>(rowp + ((j ^ ((lane >> 1) & 3u)) << 4)) =
                      make_uint4(pk[i][4 * j], pk[i][4 * j + 1], pk[i][4 * j + 2], pk[i][4 * j + 3]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                  tma_store_2d(&tmD, buf, static_cast<int32_t>(col_base + chunk(i) * 32), static_cast<int32_t>(row0));
                  bulk_commit_group();
                }
                ++chunk_ctr;
              }
            }
          } else {
#pragma unroll
            for (uint32_t i = 0; i < 4; ++i)
              if (chunk(i) < live)
                store_chunk32_packed(base_ptr + (epi0 - base) + ew * C::CHUNK_BYTES,
                                     static_cast<uint16_t*>(args.D), args.ldd, args.M, args.N, row0,
                                     col_base + chunk(i) * 32, pk[i], lane);
          }
        }
        continue;
      }
      if (w.kind == 2) {
        // a later K-range of a split tile: park the fp32 slice in this
        // cluster's slot (float4 index (chunk * 8 + i / 4) * 32 + lane, so each
        // store instruction writes 512 contiguous bytes), then raise the flag
        float* const part = part_ptr(cluster_id);
#pragma unroll 1
        for (uint32_t c = eg; c < live; c += NG) {
          uint32_t v[32];
          tmem_ld_32x32b_x32_sync(t_addr + c * 32, v);
          float4* dst = reinterpret_cast<float4*>(part + c * 1024);
#pragma unroll
          for (uint32_t i4 = 0; i4 < 8; ++i4)
            dst[i4 * 32 + lane] = make_float4(__uint_as_float(v[4 * i4]), __uint_as_float(v[4 * i4 + 1]),
                                              __uint_as_float(v[4 * i4 + 2]), __uint_as_float(v[4 * i4 + 3]));
        }
        __threadfence();
        __syncwarp();
        if (lane == 0) st_release_u32(flag_ptr(cluster_id), args.epoch);
      } else if (w.kind == 1) {
        // the first K-range: this CTA's last item, so its operand stages are
        // idle.  Wait for every later range's partial, then stream them in.
        nc = num_contributors(args, cluster_id, num_clusters, KT, w.tile);
        for (uint32_t i = 0; ok && i < nc; ++i) ok = wait_flag(flag_ptr(cluster_id + 1 + i), args.epoch, wd, lane);
        if (ok && row0 < args.M) {
          nfix = (live > eg ? (live - eg + NG - 1) / NG : 0u) * nc;
          const uint32_t first = min(nfix, C::FIX_SLOTS);
          if (lane == 0) {
            fence_proxy_async_global();
            for (uint32_t n = 0; n < first; ++n) issue_fix(n);
          }
          fix_issued = first;
        }
      }
      if (w.kind != 2 && ok && row0 < args.M) {
        if constexpr (TMA_STORE && C::TS_COLS == 32) {
          // 32-column chunks: one tcgen05.ld, one 32x32 box per chunk
#pragma unroll 1
          for (uint32_t c = 0; c < item_nch; ++c) {
            if (col_base + c * 32 >= args.N) break;
            uint32_t v[32];
            tmem_ld_32x32b_x32_sync(t_addr + c * 32, v);
            if (w.kind == 1 && !add_partials(v, c)) { ok = false; break; }
            if (epi_mode != 0) epi_apply(v, args, row0 + lane, col_base + c * 32);
            const uint32_t buf = epi0 + (ew * C::EPI_BUFS + (chunk_ctr % C::EPI_BUFS)) * C::EPI_BUF_BYTES;
            if (lane == 0) bulk_wait_group_read<C::EPI_BUFS - 1>();   // this buffer's last store has read it
            __syncwarp();
            uint8_t* rowp = base_ptr + (buf - base) + lane * 64;
#pragma unroll
            for (uint32_t i = 0; i < 4; ++i) {
              const uint4 val = make_uint4(pack_bf16x2(__uint_as_float(v[8 * i + 0]), __uint_as_float(v[8 * i + 1])),
                                           pack_bf16x2(__uint_as_float(v[8 * i + 2]), __uint_as_float(v[8 * i + 3])),
                                           pack_bf16x2(__uint_as_float(v[8 * i + 4]), __uint_as_float(v[8 * i + 5])),
                                           pack_bf16x2(__uint_as_float(v[8 * i + 6]), __uint_as_float(v[8 * i + 7])));
              // 64-byte swizzle: 16-byte chunk i of row r sits at chunk i ^ ((r / 2) % 4)
              *reinterpret_cast<uint4*>(rowp + ((i ^ ((lane >> 1) & 3u)) << 4)) = val;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmD, buf, static_cast<int32_t>(col_base + c * 32), static_cast<int32_t>(row0));
              bulk_commit_group();
            }
            ++chunk_ctr;
          }
        } else if constexpr (TMA_STORE) {
#pragma unroll 1
          for (uint32_t c = 0; c < item_nch / 2; ++c) {
            if (col_base + c * 64 >= args.N) break;
            uint32_t v0[32], v1[32];
            tmem_ld2_32x32b_x32_sync(t_addr + c * 64, t_addr + c * 64 + 32, v0, v1);
            if (w.kind == 1) {
              if (!add_partials(v0, 2 * c)) { ok = false; break; }
              if (2 * c + 1 < live && !add_partials(v1, 2 * c + 1)) { ok = false; break; }
            }
            const bool ctma = kCTma && c_tma != 0;
            uint32_t cw[32];   // this lane's row of the C chunk: bf16 pairs
            if (ctma) {
              if (!warp_wait(c_bar, c_done & 1u, wd, kSiteEpiC, lane)) { ok = false; break; }
              ++c_done;
              const uint8_t* crow = base_ptr + (cbuf - base) + lane * 128;
#pragma unroll
              for (uint32_t i = 0; i < 8; ++i) {
                // 128-byte swizzle, as for D: 16-byte chunk i of row r at chunk i ^ (r % 8)
                const uint4 t = *reinterpret_cast<const uint4*>(crow + ((i ^ (lane & 7u)) << 4));
                cw[4 * i] = t.x;
                cw[4 * i + 1] = t.y;
                cw[4 * i + 2] = t.z;
                cw[4 * i + 3] = t.w;
              }
              __syncwarp();   // every lane has read the buffer
              const uint32_t cn = col_base + (c + 1) * 64;
              if (c + 1 < item_nch / 2 && cn < args.N) {
                if (lane == 0) issue_c(row0, cn);
                ++c_issued;
              }
            }
            if (epi_mode != 0) {
              epi_apply(v0, args, row0 + lane, col_base + c * 64, ctma ? cw : nullptr);
              epi_apply(v1, args, row0 + lane, col_base + c * 64 + 32, ctma ? cw + 16 : nullptr);
            }
            // D staging: the rotating buffers, or the first one alone when
            // the second receives C
            const uint32_t buf = ctma ? epi0 + ew * C::EPI_BUFS * C::EPI_BUF_BYTES
                                      : epi0 + (ew * C::EPI_BUFS + (chunk_ctr % C::EPI_BUFS)) * C::EPI_BUF_BYTES;
            if (lane == 0) {   // the buffer's last store has read it
              if (ctma)
                bulk_wait_group_read<0>();
              else
                bulk_wait_group_read<C::EPI_BUFS - 1>();
            }
            __syncwarp();
            uint8_t* rowp = base_ptr + (buf - base) + lane * 128;
#pragma unroll
            for (uint32_t i = 0; i < 8; ++i) {
              uint4 val;
              if (i < 4) {
                val = make_uint4(pack_bf16x2(__uint_as_float(v0[8 * i + 0]), __uint_as_float(v0[8 * i + 1])),
                                 pack_bf16x2(__uint_as_float(v0[8 * i + 2]), __uint_as_float(v0[8 * i + 3])),
                                 pack_bf16x2(__uint_as_float(v0[8 * i + 4]), __uint_as_float(v0[8 * i + 5])),
                                 pack_bf16x2(__uint_as_float(v0[8 * i + 6]), __uint_as_float(v0[8 * i + 7])));
              } else {
                const uint32_t o = 8 * (i - 4);
                val = make_uint4(pack_bf16x2(__uint_as_float(v1[o + 0]), __uint_as_float(v1[o + 1])),
                                 pack_bf16x2(__uint_as_float(v1[o + 2]), __uint_as_float(v1[o + 3])),
                                 pack_bf16x2(__uint_as_float(v1[o + 4]), __uint_as_float(v1[o + 5])),
                                 pack_bf16x2(__uint_as_float(v1[o + 6]), __uint_as_float(v1[o + 7])));
              }
              // 128-byte swizzle: 16-byte chunk i of row r sits at chunk i ^ (r % 8)
              *reinterpret_cast<uint4*>(rowp + ((i ^ (lane & 7u)) << 4)) = val;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmD, buf, static_cast<int32_t>(col_base + c * 64), static_cast<int32_t>(row0));
              bulk_commit_group();
            }
            ++chunk_ctr;
          }
        } else {
          // One 32-column chunk at a time (this group's chunks eg, eg + NG, ...).
          // Each tcgen05.ld and its tcgen05.wait::ld form one asm statement:
          // the load writes its destination registers asynchronously, so no
          // other code may sit between the two.
          const auto finish_chunk = [&](uint32_t (&v)[32], uint32_t c) -> bool {
            if (w.kind == 1 && !add_partials(v, c)) return false;
            if (epi_mode != 0) epi_apply(v, args, row0 + lane, col_base + c * 32);
            if (epi_mode & kEpiOutF32)
              store_row32_f32(static_cast<float*>(args.D), args.ldd, args.M, args.N, row0 + lane,
                              col_base + c * 32, v);
            else
              store_chunk32_staged(base_ptr + (epi0 - base) + ew * C::CHUNK_BYTES,
                                   static_cast<uint16_t*>(args.D), args.ldd, args.M, args.N, row0,
                                   col_base + c * 32, v, lane);
            return true;
          };
#pragma unroll 1
          for (uint32_t c = eg; c < live; c += NG) {
            uint32_t v[32];
            tmem_ld_32x32b_x32_sync(t_addr + c * 32, v);
            if (!finish_chunk(v, c)) { ok = false; break; }
          }
        }
      }
      if (w.kind == 1 && ok) {
        // partials consumed: leave the flags at zero for the next launch
        __syncwarp();
        if (lane == 0)
          for (uint32_t i = 0; i < nc; ++i) *flag_ptr(cluster_id + 1 + i) = 0u;
      }
      // all TMEM reads of accumulator b by this warp are complete
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        if constexpr (CG == 1)
          mbar_arrive(acce_bar(b));
        else
          mbar_arrive_cluster(mapa_shared(acce_bar(b), 0));
      }
    }
    // Exit path after a give-up: let the partial transfers and a C chunk
    // still in flight land.
    if (lane == 0) {
      for (uint32_t n = fix_done; n < fix_issued; ++n)
        drain_wait(fix_bar(n % C::FIX_SLOTS), (n / C::FIX_SLOTS) & 1u, wd, kSiteStreamKFlag);
      if (c_issued > c_done) drain_wait(c_bar, c_done & 1u, wd, kSiteEpiC);
    }
    if constexpr (TMA_STORE) {
      if (lane == 0) bulk_wait_group<0>();
      __syncwarp();
    }
  }

  // ---- teardown: every role is done with TMEM and with the peer's barriers ----
  __syncwarp();   // reconverge the single-lane roles before the aligned barriers below
  tc_fence_before_sync();
  __syncthreads();
  if constexpr (CG == 2) cluster_sync();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc<CG>(tmem_base, C::TMEM_COLS);
  }
}

}  // namespace gb300
