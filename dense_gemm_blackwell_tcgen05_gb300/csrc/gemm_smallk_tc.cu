// Small-K bf16 GEMM on the tensor core (GEMM_VARIANT_SMALLK_TC; K <= 16):
// two tcgen05.mma (M = 128, N = 128, K = 16) per 128x256 output tile, then a
// tcgen05.ld epilogue that is a stream of aligned 16-byte stores.  For so few
// products per output the GEMM is a write of D, so the kernel is built to
// keep the stores going:
//
//  * Persistent, one CTA per SM, with two TMEM accumulators and two operand
//    stages: four loader warps fill a stage, one thread issues the tile's
//    MMAs, and eight epilogue warps drain the other accumulator meanwhile.
//  * The loader threads copy each operand row's first 16 k (two 16-byte
//    chunks, zero past K) into the 128-byte-swizzled K-major layout the MMA
//    reads (the layout of the ladder's synchronous kernel); the MMA's single
//    K = 16 step reads exactly those two chunks.  A swizzled TMA box would
//    have to be 64 columns wide and zero-fill 56 of them per row, which the
//    TMA engine does far more slowly than it loads.
//  * A tile's 128 rows are the rows of one residue class mod 8 (rows r,
//    r + 8, r + 16, ...).  Such rows all start the same number e of elements
//    past a 16-byte line, whatever the pitch, so the tile's column origin is
//    shifted back by e: each row's 32-column runs then sit on whole 16-byte
//    lines and leave as 16-byte pieces, eight rows per store instruction
//    (staged through shared memory); only the matrix's left and right edges
//    take 2-byte stores.
//
// Accumulation is the tensor core's fp32 (order unspecified, as in the other
// tcgen05 kernels), rounded once to bf16 (RNE).
#include <cuda_runtime.h>

#include <cstdint>

#include "gemm_gb300.h"
#include "gemm_host.h"
#include "gemm_kernels.cuh"   // bounded waits, store_chunk32_packed

namespace gb300 {
namespace {

constexpr uint32_t kTcRows = 128;       // tile rows (MMA M, TMEM lanes)
constexpr uint32_t kTcCols = 256;       // tile columns (two MMAs of N = 128)
constexpr uint32_t kTcMaxK = 16;
// warps: 0-3 loaders, 4 MMA issuer, 5-8 and 9-12 the two epilogue groups
constexpr uint32_t kTcLoadWarps = 4;
constexpr uint32_t kTcMmaWarp = 4;
constexpr uint32_t kTcEpiWarp0 = 5;
constexpr uint32_t kTcThreads = 32 * 13;
// 128-row operand blocks in the 128-byte-swizzled layout: A, then B's two
// 128-row halves.  Only the first two 16-byte chunks of each 128-byte row
// are written and read (k < 16).
constexpr uint32_t kTcBlock = 128 * 128;      // 16 KB
constexpr uint32_t kTcStage = 3 * kTcBlock;   // 48 KB
constexpr uint32_t kTcStages = 2;
// Epilogue staging: one 32x32 bf16 chunk (2 KB) per epilogue warp.
constexpr uint32_t kTcStageOff = kTcStages * kTcStage;
constexpr uint32_t kTcSmemBytes = kTcStageOff + 8 * 2048 + 1024;   // + alignment slack

struct SmallKTcArgs {
  const uint16_t* A;
  const uint16_t* B;
  uint16_t* D;
  uint32_t M, N, K;
  uint64_t lda, ldb, ldd;
  uint32_t class_rows[8];     // rows in residue class r (rows r, r + 8, ...)
  uint32_t groups;            // 128-row groups of the largest class
  uint32_t strips;            // 256-column strips
  unsigned long long* status;
  unsigned long long timeout_ns;
};

// Chunk c (k = 8c .. 8c + 7) of a row, zero past K or for a missing row.
__device__ __forceinline__ uint4 row_chunk(const uint16_t* row, uint32_t c, uint32_t K, bool ok) {
  const uint32_t k = 8 * c;
  if (!ok || k >= K) return make_uint4(0, 0, 0, 0);
  if (k + 8 <= K) return __ldg(reinterpret_cast<const uint4*>(row + k));   // rows 16-byte aligned
  uint32_t h[8];
#pragma unroll
  for (uint32_t i = 0; i < 8; ++i) h[i] = k + i < K ? __ldg(row + k + i) : 0u;
  return make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16), h[6] | (h[7] << 16));
}

// The t-th tile (in 0 .. strips * 8 * groups): strip, residue class and
// 128-row group; false when that class has no such group (an empty tile,
// skipped the same way by every role).
__device__ __forceinline__ bool tile_of(const SmallKTcArgs& a, uint32_t t, uint32_t& strip,
                                        uint32_t& r8, uint32_t& g) {
  strip = t % a.strips;
  const uint32_t rest = t / a.strips;
  r8 = rest % 8;
  g = rest / 8;
  return g * kTcRows < a.class_rows[r8];
}

// Elements from class r8's rows to the previous 16-byte line: the same for
// every row r8 + 8 j, since 8 j ldd elements are whole lines.
__device__ __forceinline__ int64_t tile_col0(const SmallKTcArgs& a, uint32_t strip, uint32_t r8) {
  const uint32_t e = static_cast<uint32_t>(
      (reinterpret_cast<uintptr_t>(a.D + static_cast<uint64_t>(r8) * a.ldd) >> 1) & 7u);
  return static_cast<int64_t>(strip) * kTcCols - e;
}

__global__ void __launch_bounds__(kTcThreads, 1) gemm_smallk_tc_kernel(const __grid_constant__ SmallKTcArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_dyn[];
  __shared__ __align__(8) uint64_t bars[10];
  __shared__ uint32_t tmem_slot;
  __shared__ uint32_t abort_word;
  const uint32_t tid = threadIdx.x;
  const uint32_t warp = warp_idx_sync();
  const uint32_t lane = lane_idx();
  const uint32_t base = (smem_addr(smem_dyn) + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_dyn + (base - smem_addr(smem_dyn));
  const uint32_t bar0 = smem_addr(&bars[0]);
  const auto full_bar = [&](uint32_t s) { return bar0 + 8 * s; };          // loaders -> MMA
  const auto free_bar = [&](uint32_t s) { return bar0 + 8 * (2 + s); };    // MMA done reading a stage
  const auto accf_bar = [&](uint32_t b) { return bar0 + 8 * (4 + b); };    // accumulator b complete
  const auto acce_bar = [&](uint32_t b) { return bar0 + 8 * (6 + b); };    // accumulator b drained
  const uint32_t drain_bar = bar0 + 8 * 8;
  const Watchdog wd{a.status, a.timeout_ns, &abort_word};
  const uint32_t tiles = a.strips * 8 * a.groups;

  if (tid == 0) {
    for (uint32_t s = 0; s < kTcStages; ++s) {
      mbar_init(full_bar(s), kTcLoadWarps);   // one arrival per loader warp
      mbar_init(free_bar(s), 1);              // the MMA thread's commit
    }
    for (uint32_t b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1);              // the MMA thread's commit
      mbar_init(acce_bar(b), 8);              // every epilogue warp
    }
    mbar_init(drain_bar, 1);
    abort_word = 0;
    fence_mbar_init();
  }
  if (warp == kTcMmaWarp) {
    tmem_alloc<1>(smem_addr(&tmem_slot), 2 * kTcCols);
    tmem_relinquish<1>();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(&tmem_slot);

  if (warp < kTcLoadWarps) {
    // ==================== loaders: 128 threads, one A row and two B rows each
    const uint32_t lt = tid;   // 0 .. 127
    const uint32_t sw0 = lt * 128 + ((0u ^ (lt & 7u)) << 4), sw1 = lt * 128 + ((1u ^ (lt & 7u)) << 4);
    uint32_t i = 0;
    for (uint32_t t = blockIdx.x; t < tiles; t += gridDim.x) {
      uint32_t strip, r8, g;
      if (!tile_of(a, t, strip, r8, g)) continue;
      const uint32_t s = i % kTcStages;
      if (!warp_wait(free_bar(s), ((i / kTcStages) & 1u) ^ 1u, wd, kSiteProducerEmpty, lane)) break;
      const int64_t col0 = tile_col0(a, strip, r8);
      const uint32_t j = g * kTcRows + lt;   // A row r8 + 8 j
      const uint16_t* arow = a.A + (static_cast<uint64_t>(r8) + 8ull * j) * a.lda;
      const int64_t bc0 = col0 + lt, bc1 = col0 + 128 + lt;
      const bool ok0 = bc0 >= 0 && bc0 < a.N, ok1 = bc1 >= 0 && bc1 < a.N;
      const uint16_t* b0 = a.B + (ok0 ? bc0 : 0) * static_cast<int64_t>(a.ldb);
      const uint16_t* b1 = a.B + (ok1 ? bc1 : 0) * static_cast<int64_t>(a.ldb);
      const uint4 va0 = row_chunk(arow, 0, a.K, j < a.class_rows[r8]);
      const uint4 va1 = row_chunk(arow, 1, a.K, j < a.class_rows[r8]);
      const uint4 vb00 = row_chunk(b0, 0, a.K, ok0), vb01 = row_chunk(b0, 1, a.K, ok0);
      const uint4 vb10 = row_chunk(b1, 0, a.K, ok1), vb11 = row_chunk(b1, 1, a.K, ok1);
      uint8_t* const st = base_ptr + s * kTcStage;
      *reinterpret_cast<uint4*>(st + sw0) = va0;
      *reinterpret_cast<uint4*>(st + sw1) = va1;
      *reinterpret_cast<uint4*>(st + kTcBlock + sw0) = vb00;
      *reinterpret_cast<uint4*>(st + kTcBlock + sw1) = vb01;
      *reinterpret_cast<uint4*>(st + 2 * kTcBlock + sw0) = vb10;
      *reinterpret_cast<uint4*>(st + 2 * kTcBlock + sw1) = vb11;
      fence_proxy_async_smem();   // generic writes, read by the tensor core
      __syncwarp();
      if (lane == 0) mbar_arrive(full_bar(s));
      ++i;
    }
  } else if (warp == kTcMmaWarp) {
    // ==================== MMA issuer: one thread
    if (lane == 0) {
      uint32_t i = 0;
      bool issued = false;
      for (uint32_t t = blockIdx.x; t < tiles; t += gridDim.x) {
        uint32_t strip, r8, g;
        if (!tile_of(a, t, strip, r8, g)) continue;
        const uint32_t s = i % kTcStages, b = i % 2;
        if (!wait_bounded(full_bar(s), (i / kTcStages) & 1u, wd, kSiteMmaFull) ||
            !wait_bounded(acce_bar(b), ((i / 2) & 1u) ^ 1u, wd, kSiteMmaAccEmpty))
          break;
        tc_fence_after_sync();
        const uint32_t sb = base + s * kTcStage;
        for (uint32_t h = 0; h < 2; ++h)
          mma_bf16<1>(tmem + b * kTcCols + 128 * h, smem_desc_sw128(sb),
                      smem_desc_sw128(sb + (1 + h) * kTcBlock), idesc_bf16(kTcRows, 128), 0u);
        tc_commit(free_bar(s));
        tc_commit(accf_bar(b));
        issued = true;
        ++i;
      }
      if (issued) {   // every tcgen05 op of this thread completes before TMEM is released
        tc_commit(drain_bar);
        drain_wait(drain_bar, 0, wd, kSiteMmaDrain);
      }
    }
  } else {
    // ==================== epilogue: two groups of four warps, one TMEM lane quarter each
    const uint32_t ew = warp - kTcEpiWarp0;   // 0 .. 7
    const uint32_t eg = ew / 4, q = warp & 3u;
    uint8_t* const stage = base_ptr + kTcStageOff + ew * 2048;
    uint32_t i = 0;
    for (uint32_t t = blockIdx.x; t < tiles; t += gridDim.x) {
      uint32_t strip, r8, g;
      if (!tile_of(a, t, strip, r8, g)) continue;
      const uint32_t b = i % 2;
      if (!warp_wait(accf_bar(b), (i / 2) & 1u, wd, kSiteEpiAccFull, lane)) break;
      tc_fence_after_sync();
      const int64_t col0 = tile_col0(a, strip, r8);
      const uint32_t rows = a.class_rows[r8];
      const uint32_t jr0 = g * kTcRows + q * 32;   // this warp's first class row
      const uint32_t jr = jr0 + lane;
      uint16_t* const dclass = a.D + static_cast<uint64_t>(r8) * a.ldd;   // pitch 8 ldd
      uint16_t* const drow = dclass + 8ull * jr * a.ldd;
#pragma unroll 1
      for (uint32_t c = eg; c < kTcCols / 32; c += 2) {
        uint32_t v[32];
        tmem_ld_32x32b_x32_sync(tmem + b * kTcCols + ((q * 32u) << 16) + c * 32, v);
        const int64_t cc = col0 + 32 * c;   // first column of this run (warp-uniform)
        if (cc >= static_cast<int64_t>(a.N) || cc + 32 <= 0 || jr0 >= rows) continue;
        uint32_t p[16];
#pragma unroll
        for (uint32_t u = 0; u < 16; ++u) p[u] = pack_bf16x2(__uint_as_float(v[2 * u]), __uint_as_float(v[2 * u + 1]));
        if (cc >= 0 && cc + 32 <= static_cast<int64_t>(a.N)) {
          store_chunk32_packed(stage, dclass, 8 * a.ldd, rows, a.N, jr0, static_cast<uint32_t>(cc), p, lane);
        } else if (jr < rows) {
          // the matrix's left or right edge: one 2-byte store per column inside
          uint16_t* const dst = drow + cc;
#pragma unroll
          for (uint32_t u = 0; u < 32; ++u)
            if (cc + u >= 0 && cc + u < static_cast<int64_t>(a.N))
              dst[u] = static_cast<uint16_t>(u % 2 ? p[u / 2] >> 16 : p[u / 2] & 0xFFFFu);
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(acce_bar(b));
      ++i;
    }
  }
  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kTcMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc<1>(tmem, 2 * kTcCols);
  }
}

}  // namespace

int launch_bf16_smallk_tc(const Problem& p, const LaunchCtx& ctx, cudaStream_t stream) {
  if (p.K == 0 || p.K > kTcMaxK) return GEMM_ERR_INVALID_ARG;
  static bool prepared[128] = {false};
  if (ctx.device < 0 || ctx.device >= 128) return GEMM_ERR_UNSUPPORTED_DEVICE;
  if (!prepared[ctx.device]) {
    if (const cudaError_t e = cudaFuncSetAttribute(gemm_smallk_tc_kernel,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(kTcSmemBytes));
        e != cudaSuccess) {
      note_cuda_error(e);
      cudaGetLastError();
      return GEMM_ERR_LAUNCH;
    }
    prepared[ctx.device] = true;
  }
  SmallKTcArgs a;
  a.A = static_cast<const uint16_t*>(p.A);
  a.B = static_cast<const uint16_t*>(p.B);
  a.D = static_cast<uint16_t*>(p.D);
  a.M = p.M;
  a.N = p.N;
  a.K = p.K;
  a.lda = p.lda;
  a.ldb = p.ldb;
  a.ldd = p.ldd;
  a.status = ctx.status;
  a.timeout_ns = ctx.timeout_ns;
  for (uint32_t r = 0; r < 8; ++r) a.class_rows[r] = p.M > r ? (p.M - r + 7) / 8 : 0u;
  a.groups = (a.class_rows[0] + kTcRows - 1) / kTcRows;
  // a tile's columns start up to 7 before its strip, so strips cover N + 7
  const uint64_t strips = (static_cast<uint64_t>(p.N) + 7 + kTcCols - 1) / kTcCols;
  const uint64_t tiles = strips * 8 * a.groups;
  if (tiles > 0xFFFFFFFFull) return GEMM_ERR_INVALID_ARG;
  a.strips = static_cast<uint32_t>(strips);
  const uint64_t grid = tiles < static_cast<uint64_t>(ctx.num_sms) ? tiles : ctx.num_sms;
  gemm_smallk_tc_kernel<<<static_cast<unsigned>(grid), kTcThreads, kTcSmemBytes, stream>>>(a);
  if (const cudaError_t e = cudaGetLastError(); e != cudaSuccess) {
    note_cuda_error(e);
    return GEMM_ERR_LAUNCH;
  }
  return GEMM_OK;
}

}  // namespace gb300
