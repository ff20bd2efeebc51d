// Small-K bf16 GEMM on the tensor core (GEMM_VARIANT_SMALLK_TC; K <= 16):
// two tcgen05.mma (M = 128, N = 128, K = 16) per 128x256 output tile, then a
// tcgen05.ld epilogue that is a stream of aligned 16-byte stores.  For so few
// products per output the GEMM is a write of D; this kernel loads only the
// operand bytes that exist and keeps every store aligned:
//
//  * The CTA's threads copy each operand row's first 16 k (two 16-byte
//    chunks, zero past K) into the 128-byte-swizzled K-major layout the MMA
//    reads (the layout of the ladder's synchronous kernel); the MMA's single
//    K = 16 step reads exactly those two chunks.  A swizzled TMA box would
//    have to be 64 columns wide and zero-fill 56 of them per row, which the
//    TMA engine does far more slowly than it loads.
//  * A tile's 128 rows are the rows of one residue class mod 8 (rows r,
//    r + 8, r + 16, ...).  Such rows all start the same number e of elements
//    past a 16-byte line, whatever the pitch, so the tile's column origin is
//    shifted back by e: every thread's 32-column run then sits on whole
//    16-byte lines of its row and is written with four 16-byte stores; only
//    the matrix's left and right edges take 2-byte stores.
//
// Accumulation is the tensor core's fp32 (order unspecified, as in the other
// tcgen05 kernels), rounded once to bf16 (RNE).
#include <cuda_runtime.h>

#include <cstdint>

#include "gemm_gb300.h"
#include "gemm_host.h"
#include "gemm_kernels.cuh"   // bounded waits (warp_wait, drain_wait)

namespace gb300 {
namespace {

constexpr uint32_t kTcRows = 128;       // tile rows (MMA M, TMEM lanes)
constexpr uint32_t kTcCols = 256;       // tile columns (two MMAs of N = 128; TMEM columns)
constexpr uint32_t kTcThreads = 128;    // four warps: one TMEM lane quarter each
constexpr uint32_t kTcMaxK = 16;
// 128-row operand blocks in the 128-byte-swizzled layout: A, then B's two
// 128-row halves.  Only the first two 16-byte chunks of each 128-byte row
// are written and read (k < 16).
constexpr uint32_t kTcBlock = 128 * 128;      // 16 KB
constexpr uint32_t kTcOperandBytes = 3 * kTcBlock;
// Epilogue staging: one 32x32 bf16 chunk (2 KB) per warp, so that stores
// leave as 16-byte pieces, eight rows per instruction.
constexpr uint32_t kTcStageBytes = 4 * 2048;
// Dynamic shared memory asked for per CTA: the operands plus alignment
// slack, sized so that at most two CTAs share an SM, which is what their
// 2 x 256 TMEM columns allow without an allocation ever waiting.
constexpr uint32_t kTcSmemBytes = 96 * 1024;
static_assert(kTcOperandBytes + kTcStageBytes + 1024 <= kTcSmemBytes, "operand blocks fit");

struct SmallKTcArgs {
  const uint16_t* A;
  const uint16_t* B;
  uint16_t* D;
  uint32_t M, N, K;
  uint64_t lda, ldb, ldd;
  uint32_t class_rows[8];     // rows in residue class r (rows r, r + 8, ...)
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

__global__ void __launch_bounds__(kTcThreads) gemm_smallk_tc_kernel(const __grid_constant__ SmallKTcArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_dyn[];
  __shared__ __align__(8) uint64_t bar_mma;
  __shared__ uint32_t tmem_slot;
  __shared__ uint32_t abort_word;
  const uint32_t tid = threadIdx.x;
  const uint32_t warp = warp_idx_sync();
  const uint32_t lane = lane_idx();
  const uint32_t r8 = blockIdx.y % 8;
  const uint32_t rows = a.class_rows[r8];
  if (blockIdx.y / 8 * kTcRows >= rows) return;   // no tile of this class for this CTA (uniform)
  const uint32_t base = (smem_addr(smem_dyn) + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_dyn + (base - smem_addr(smem_dyn));
  // elements from this class's rows to the previous 16-byte line: the same
  // for every row r8 + 8 j, since 8 j ldd elements are whole lines
  const uint32_t e = static_cast<uint32_t>(
      (reinterpret_cast<uintptr_t>(a.D + static_cast<uint64_t>(r8) * a.ldd) >> 1) & 7u);
  const int64_t col0 = static_cast<int64_t>(blockIdx.x) * kTcCols - e;   // tile column origin
  const Watchdog wd{a.status, a.timeout_ns, &abort_word};

  if (tid == 0) {
    mbar_init(smem_addr(&bar_mma), 1);
    abort_word = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc<1>(smem_addr(&tmem_slot), kTcCols);
    tmem_relinquish<1>();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(&tmem_slot);
  // this thread's operand rows: tile row tid of A, tile rows tid and 128 + tid of B
  const int64_t bc0 = col0 + tid, bc1 = col0 + 128 + tid;
  const uint4 b00 = row_chunk(a.B + bc0 * static_cast<int64_t>(a.ldb), 0, a.K, bc0 >= 0 && bc0 < a.N);
  const uint4 b01 = row_chunk(a.B + bc0 * static_cast<int64_t>(a.ldb), 1, a.K, bc0 >= 0 && bc0 < a.N);
  const uint4 b10 = row_chunk(a.B + bc1 * static_cast<int64_t>(a.ldb), 0, a.K, bc1 >= 0 && bc1 < a.N);
  const uint4 b11 = row_chunk(a.B + bc1 * static_cast<int64_t>(a.ldb), 1, a.K, bc1 >= 0 && bc1 < a.N);
  // 128-byte swizzle: 16-byte chunk c of row r at r * 128 + ((c ^ (r % 8)) << 4)
  const uint32_t sw0 = tid * 128 + ((0u ^ (tid & 7u)) << 4), sw1 = tid * 128 + ((1u ^ (tid & 7u)) << 4);
  *reinterpret_cast<uint4*>(base_ptr + kTcBlock + sw0) = b00;
  *reinterpret_cast<uint4*>(base_ptr + kTcBlock + sw1) = b01;
  *reinterpret_cast<uint4*>(base_ptr + 2 * kTcBlock + sw0) = b10;
  *reinterpret_cast<uint4*>(base_ptr + 2 * kTcBlock + sw1) = b11;

  bool ok = true, committed = false;
  uint32_t iter = 0;
  for (uint32_t g = blockIdx.y / 8; ok && g * kTcRows < rows; g += gridDim.y / 8, ++iter) {
    const uint32_t j = g * kTcRows + tid;   // this thread's row of the class (A row r8 + 8 j)
    const uint16_t* arow = a.A + (static_cast<uint64_t>(r8) + 8ull * j) * a.lda;
    *reinterpret_cast<uint4*>(base_ptr + sw0) = row_chunk(arow, 0, a.K, j < rows);
    *reinterpret_cast<uint4*>(base_ptr + sw1) = row_chunk(arow, 1, a.K, j < rows);
    fence_proxy_async_smem();   // generic writes, read by the tensor core
    tc_fence_before_sync();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after_sync();
      for (uint32_t h = 0; h < 2; ++h)
        mma_bf16<1>(tmem + 128 * h, smem_desc_sw128(base), smem_desc_sw128(base + (1 + h) * kTcBlock),
                    idesc_bf16(kTcRows, 128), 0u);
      tc_commit(smem_addr(&bar_mma));
      committed = true;
    }
    __syncwarp();
    ok = warp_wait(smem_addr(&bar_mma), iter & 1u, wd, kSiteEpiAccFull, lane);
    ok = __syncthreads_and(ok);
    tc_fence_after_sync();
    if (ok) {
      // thread = TMEM lane = tile row: D row r8 + 8 (128 g + warp * 32 + lane)
      const uint32_t jr = g * kTcRows + warp * 32 + lane;
      const bool row_ok = jr < rows;
      uint16_t* const drow = a.D + (static_cast<uint64_t>(r8) + 8ull * jr) * a.ldd;
      // the class's rows as a matrix of pitch 8 ldd (a multiple of 16 bytes)
      uint16_t* const dclass = a.D + static_cast<uint64_t>(r8) * a.ldd;
      uint8_t* const stage = base_ptr + kTcOperandBytes + warp * 2048;
#pragma unroll 1
      for (uint32_t c = 0; c < kTcCols / 32; ++c) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tmem + ((warp * 32u) << 16) + c * 32, v);
        tmem_wait_ld();
        const int64_t cc = col0 + 32 * c;   // first column of this run (warp-uniform)
        if (cc >= static_cast<int64_t>(a.N) || cc + 32 <= 0) continue;
        uint32_t p[16];
#pragma unroll
        for (uint32_t t = 0; t < 16; ++t) p[t] = pack_bf16x2(__uint_as_float(v[2 * t]), __uint_as_float(v[2 * t + 1]));
        if (cc >= 0 && cc + 32 <= static_cast<int64_t>(a.N)) {
          // whole run inside D: staged, then 16-byte pieces of eight rows per
          // store instruction (each row's run starts on a 16-byte line)
          store_chunk32_packed(stage, dclass, 8 * a.ldd, rows, a.N, g * kTcRows + warp * 32,
                               static_cast<uint32_t>(cc), p, lane);
        } else if (row_ok) {
          uint16_t* const dst = drow + cc;
          // the matrix's left or right edge: one 2-byte store per column inside
#pragma unroll
          for (uint32_t t = 0; t < 32; ++t)
            if (cc + t >= 0 && cc + t < static_cast<int64_t>(a.N))
              dst[t] = static_cast<uint16_t>(t % 2 ? p[t / 2] >> 16 : p[t / 2] & 0xFFFFu);
        }
      }
    } else if (tid == 0 && committed) {
      drain_wait(smem_addr(&bar_mma), iter & 1u, wd, kSiteMmaDrain);   // the committed MMAs complete first
    }
    committed = false;
    // every TMEM read and shared-memory operand read of this tile done before
    // the next tile's A rows and MMAs
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc<1>(tmem, kTcCols);
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
  const uint32_t groups = (a.class_rows[0] + kTcRows - 1) / kTcRows;
  // a tile's columns start up to 7 before its strip, so strips cover N + 7
  const uint64_t strips = (static_cast<uint64_t>(p.N) + 7 + kTcCols - 1) / kTcCols;
  if (strips > 0x7FFFFFFFull) return GEMM_ERR_INVALID_ARG;
  const uint32_t gy = 8u * (groups < 8191u ? groups : 8191u);
  gemm_smallk_tc_kernel<<<dim3(static_cast<unsigned>(strips), gy), kTcThreads, kTcSmemBytes, stream>>>(a);
  if (const cudaError_t e = cudaGetLastError(); e != cudaSuccess) {
    note_cuda_error(e);
    return GEMM_ERR_LAUNCH;
  }
  return GEMM_OK;
}

}  // namespace gb300
