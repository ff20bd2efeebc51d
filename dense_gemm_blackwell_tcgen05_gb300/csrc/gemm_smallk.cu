// Small-K bf16 GEMM on the CUDA cores (GEMM_VARIANT_SMALLK; the automatic
// choice for K <= 16).  With so few products per output the operation is a
// write of D, HBM-bound at about 8 flops per byte: the tensor-core path would
// move a mostly zero-filled 64-wide K box per tile for 16 or fewer real
// columns and wait on it, so this kernel skips staging through TMEM and
// spends its time on coalesced stores instead.
//
// A block covers 64 rows x 256 columns of D with 8 warps.  A lane owns CPL = 4
// consecutive columns (8 measured slower: fewer resident blocks and, on odd
// pitches, twice the 2-byte stores) and keeps their K values
// of B in registers for the whole block; a warp covers 32 CPL columns and
// walks its share of the block's rows.  A's rows are staged in shared memory
// (fp32) and read as broadcasts.  Per row a warp writes 32 CPL * 2 contiguous
// bytes, in 16-, 8-, 4- or 2-byte pieces as the row's address allows.  K is
// rounded up to a compile-time 4, 8 or 16 (zero-padded).  Sums are fp32 FMAs
// in k order, rounded once to bf16 (RNE).  The kernel is bound by instruction
// issue rather than HBM on the ragged shapes: per output about K FMAs plus a
// share of a row's broadcast loads, conversion and store.
#include <cuda_runtime.h>

#include <cstdint>

#include "gemm_gb300.h"
#include "gemm_host.h"
#include "kernel_common.cuh"

namespace gb300 {
namespace {

constexpr uint32_t kRows = 64;        // D rows per block
constexpr uint32_t kCols = 256;       // D columns per block
constexpr uint32_t kMaxK = 16;
constexpr uint32_t kThreadsSmallK = 256;

struct SmallKArgs {
  const uint16_t* A;
  const uint16_t* B;
  uint16_t* D;
  uint32_t M, N, K;
  uint64_t lda, ldb, ldd;
};

__device__ __forceinline__ float bf16f(uint32_t h) { return __uint_as_float(h << 16); }

// The first K (<= KK) values of a row as fp32, zero-padded to KK.  Nothing at
// k >= K is read (the last row of a buffer may end at K): 16-byte loads cover
// the full groups of 8 (a row starts 16-byte aligned: base aligned and pitch a
// multiple of 8 elements), single loads the rest.
template <uint32_t KK>
__device__ __forceinline__ void load_row(const uint16_t* p, uint32_t K, float (&x)[KK]) {
#pragma unroll
  for (uint32_t h = 0; h < (KK + 7) / 8; ++h) {
    if (8 * (h + 1) <= KK && K >= 8 * (h + 1)) {
      const uint4 w = *reinterpret_cast<const uint4*>(p + 8 * h);
      const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (uint32_t i = 0; i < 4; ++i) {
        x[8 * h + 2 * i] = bf16f(u[i] & 0xFFFFu);
        x[8 * h + 2 * i + 1] = bf16f(u[i] >> 16);
      }
    } else {
#pragma unroll
      for (uint32_t i = 0; i < 8; ++i) {
        const uint32_t k = 8 * h + i;
        if (k < KK) x[k] = k < K ? bf16f(p[k]) : 0.0f;
      }
    }
  }
}

// Four consecutive outputs (packed bf16 pairs p01, p23) at dp, n of them
// valid, in the widest pieces the address allows.
__device__ __forceinline__ void store4(uint16_t* dp, uint32_t p01, uint32_t p23, uint32_t n) {
  const uintptr_t al = reinterpret_cast<uintptr_t>(dp);
  if (n == 4 && (al & 7u) == 0) {
    *reinterpret_cast<uint2*>(dp) = make_uint2(p01, p23);
  } else if ((al & 3u) == 0) {
    if (n >= 2) *reinterpret_cast<uint32_t*>(dp) = p01;
    else dp[0] = static_cast<uint16_t>(p01 & 0xFFFFu);
    if (n == 4) *reinterpret_cast<uint32_t*>(dp + 2) = p23;
    else if (n == 3) dp[2] = static_cast<uint16_t>(p23 & 0xFFFFu);
  } else {
    dp[0] = static_cast<uint16_t>(p01 & 0xFFFFu);
    if (n > 1) dp[1] = static_cast<uint16_t>(p01 >> 16);
    if (n > 2) dp[2] = static_cast<uint16_t>(p23 & 0xFFFFu);
    if (n > 3) dp[3] = static_cast<uint16_t>(p23 >> 16);
  }
}

template <uint32_t KK, uint32_t CPL>
__global__ void __launch_bounds__(kThreadsSmallK) gemm_smallk_kernel(const SmallKArgs a) {
  constexpr uint32_t kWarpCols = 32 * CPL;
  constexpr uint32_t kWarpsPerRow = kCols / kWarpCols;           // 2 (CPL 4) or 1 (CPL 8)
  constexpr uint32_t kRowsPerWarp = kRows * kWarpsPerRow / 8;    // 16 or 8
  __shared__ __align__(16) float sA[kRows][KK];
  const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
  const uint32_t c = blockIdx.x * kCols + kWarpCols * (warp % kWarpsPerRow) + CPL * lane;
  const uint32_t r_base = kRowsPerWarp * (warp / kWarpsPerRow);
  // B values of columns c .. c + CPL - 1, kept in registers (zero past N)
  float b[CPL][KK];
#pragma unroll
  for (uint32_t t = 0; t < CPL; ++t) {
    if (c + t < a.N) {
      load_row<KK>(a.B + static_cast<uint64_t>(c + t) * a.ldb, a.K, b[t]);
    } else {
#pragma unroll
      for (uint32_t k = 0; k < KK; ++k) b[t][k] = 0.0f;
    }
  }
  for (uint32_t rt = blockIdx.y; rt * kRows < a.M; rt += gridDim.y) {
    const uint32_t row0 = rt * kRows;
    __syncthreads();   // the previous row tile's reads of sA are done
    if (threadIdx.x < kRows) {
      float x[KK];
      const uint32_t row = row0 + threadIdx.x;
      if (row < a.M) {
        load_row<KK>(a.A + static_cast<uint64_t>(row) * a.lda, a.K, x);
      } else {
#pragma unroll
        for (uint32_t k = 0; k < KK; ++k) x[k] = 0.0f;
      }
#pragma unroll
      for (uint32_t k = 0; k < KK; k += 4)
        *reinterpret_cast<float4*>(&sA[threadIdx.x][k]) = make_float4(x[k], x[k + 1], x[k + 2], x[k + 3]);
    }
    __syncthreads();
    if (c >= a.N || row0 + r_base >= a.M) continue;
    const uint32_t nvalid = min(CPL, a.N - c);
    const uint32_t nrows = min(kRowsPerWarp, a.M - (row0 + r_base));
    uint16_t* dp = a.D + static_cast<uint64_t>(row0 + r_base) * a.ldd + c;
#pragma unroll 2
    for (uint32_t r = 0; r < nrows; ++r, dp += a.ldd) {
      float x[CPL];
#pragma unroll
      for (uint32_t t = 0; t < CPL; ++t) x[t] = 0.0f;
#pragma unroll
      for (uint32_t k = 0; k < KK; k += 4) {
        const float4 av = *reinterpret_cast<const float4*>(&sA[r_base + r][k]);   // broadcast
        const float ak[4] = {av.x, av.y, av.z, av.w};
#pragma unroll
        for (uint32_t i = 0; i < 4; ++i)
#pragma unroll
          for (uint32_t t = 0; t < CPL; ++t) x[t] = fmaf(ak[i], b[t][k + i], x[t]);
      }
      uint32_t pk[CPL / 2];
#pragma unroll
      for (uint32_t t = 0; t < CPL / 2; ++t) pk[t] = pack_bf16x2(x[2 * t], x[2 * t + 1]);
      if (CPL == 8 && nvalid == 8 && (reinterpret_cast<uintptr_t>(dp) & 15u) == 0) {
        *reinterpret_cast<uint4*>(dp) = make_uint4(pk[0], pk[1], pk[2 % (CPL / 2)], pk[3 % (CPL / 2)]);
      } else {
#pragma unroll
        for (uint32_t g = 0; g < CPL / 4; ++g)
          if (4 * g < nvalid) store4(dp + 4 * g, pk[2 * g], pk[2 * g + 1], min(4u, nvalid - 4 * g));
      }
    }
  }
}

}  // namespace

uint32_t smallk_max_k() { return kMaxK; }

int launch_bf16_smallk(const Problem& p, cudaStream_t stream) {
  if (p.K == 0 || p.K > kMaxK) return GEMM_ERR_INVALID_ARG;
  SmallKArgs a;
  a.A = static_cast<const uint16_t*>(p.A);
  a.B = static_cast<const uint16_t*>(p.B);
  a.D = static_cast<uint16_t*>(p.D);
  a.M = p.M;
  a.N = p.N;
  a.K = p.K;
  a.lda = p.lda;
  a.ldb = p.ldb;
  a.ldd = p.ldd;
  const uint64_t col_tiles = (static_cast<uint64_t>(p.N) + kCols - 1) / kCols;
  const uint64_t row_tiles = (static_cast<uint64_t>(p.M) + kRows - 1) / kRows;
  if (col_tiles > 0x7FFFFFFFull) return GEMM_ERR_INVALID_ARG;
  const dim3 grid(static_cast<unsigned>(col_tiles),
                  static_cast<unsigned>(row_tiles < 65535 ? row_tiles : 65535));
  if (p.K <= 4)
    gemm_smallk_kernel<4, 4><<<grid, kThreadsSmallK, 0, stream>>>(a);
  else if (p.K <= 8)
    gemm_smallk_kernel<8, 4><<<grid, kThreadsSmallK, 0, stream>>>(a);
  else
    gemm_smallk_kernel<16, 4><<<grid, kThreadsSmallK, 0, stream>>>(a);
  if (const cudaError_t e = cudaGetLastError(); e != cudaSuccess) {
    note_cuda_error(e);
    return GEMM_ERR_LAUNCH;
  }
  return GEMM_OK;
}

}  // namespace gb300
