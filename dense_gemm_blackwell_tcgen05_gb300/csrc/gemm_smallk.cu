// Small-K bf16 GEMM on the CUDA cores (GEMM_VARIANT_SMALLK; the automatic
// choice for K <= 16).  With so few products per output the operation is a
// write of D at about K flops per output byte: the tensor-core path would move
// a mostly zero-filled 64-wide K box per tile for 16 or fewer real columns and
// then drain a whole TMEM accumulator per tile, so this kernel keeps
// everything in registers and spends its time on wide, aligned stores.
//
// Layout of the work.  A block of 8 warps owns one strip of 32 * CPL columns
// of D (CPL = 8 consecutive columns per lane, 4 for K > 8) and row tiles of
// kTileRows rows (grid-stride over the tiles).  A row tile's A values are
// staged once in shared memory as fp32 pairs (a, a) and read back as
// broadcasts.  Warp w computes rows w, w + 8, ... of the tile: per row a lane
// forms its CPL sums with packed fp32 FMAs (two columns per instruction) in
// k order, rounds them once to bf16 (RNE) and stores them as one 2*CPL-byte
// piece.
//
// Stores.  A warp's rows all start the same number e of elements past a
// 2*CPL-byte boundary (the rows are 8 apart and CPL divides 8), whatever the
// pitch.  So each warp's strip is shifted back by its own e columns: every
// lane's CPL columns then sit on one aligned 2*CPL-byte piece in every row
// it writes, and the only narrower stores are at the matrix's left and right
// edges (2 bytes per column there).  Each lane keeps the K values of B for
// its columns in registers for the whole block.  Nothing outside row x
// [0, N) is written and nothing at k >= K is read.
#include <cuda_runtime.h>

#include <cstdint>

#include "gemm_gb300.h"
#include "gemm_host.h"
#include "kernel_common.cuh"

namespace gb300 {
namespace {

constexpr uint32_t kTileRows = 128;   // rows of A staged per tile
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
      const uint4 w = __ldg(reinterpret_cast<const uint4*>(p + 8 * h));
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
        if (k < KK) x[k] = k < K ? bf16f(__ldg(p + k)) : 0.0f;
      }
    }
  }
}

template <uint32_t KK, uint32_t CPL>
__global__ void __launch_bounds__(kThreadsSmallK, 2) gemm_smallk_kernel(const SmallKArgs a) {
  constexpr uint32_t W = CPL / 2;            // packed words per lane and row
  constexpr uint32_t kStrip = 32 * CPL;      // columns of a warp's strip
  // A row tile as fp32 pairs (a, a): one 16-byte broadcast load feeds two
  // packed FMAs
  __shared__ __align__(16) float2 sA[kTileRows][KK];
  const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
  // This warp's rows (warp, warp + 8, ... of every tile) all start the same
  // number e of elements past a 2*CPL-byte boundary: tiles start at multiples
  // of 8 rows, and CPL divides 8.  Shifting the warp's strip back by e
  // columns puts every lane's CPL columns on such a boundary in every row.
  const uint32_t e = static_cast<uint32_t>(
      (reinterpret_cast<uintptr_t>(a.D + static_cast<uint64_t>(warp) * a.ldd) >> 1) & (CPL - 1u));
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * kStrip - e + CPL * lane;   // first column
  const bool lane_full = c0 >= 0 && c0 + CPL <= a.N;
  const bool lane_any = c0 + CPL > 0 && c0 < static_cast<int64_t>(a.N);
  // The block's B strip -- the kStrip + CPL - 1 columns its warps' shifted
  // strips cover -- staged once in shared memory as raw bf16 rows of KK
  // values (16-byte chunks; one padding slot per 8 columns, so that lanes
  // reading columns 8 apart hit different banks).  Every warp reads its
  // columns from here: the block loads each B row from L2 once instead of
  // once per warp.  Values at k >= K and columns outside [0, N) are zero,
  // and nothing at k >= K is read.
  constexpr uint32_t kBCols = kStrip + CPL - 1;
  constexpr uint32_t kChunks = (KK + 7) / 8;
  __shared__ __align__(16) uint4 sB[kBCols + kBCols / 8 + 1][kChunks];
  const int64_t bbase = static_cast<int64_t>(blockIdx.x) * kStrip - (CPL - 1);
  for (uint32_t i = threadIdx.x; i < kBCols; i += kThreadsSmallK) {
    const int64_t c = bbase + i;
    const bool in = c >= 0 && c < static_cast<int64_t>(a.N);
#pragma unroll
    for (uint32_t h = 0; h < kChunks; ++h) {
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      const uint16_t* src = a.B + static_cast<uint64_t>(in ? c : 0) * a.ldb + 8 * h;
      if (in && a.K >= 8 * (h + 1)) {
        // a whole chunk inside K: one 16-byte load (rows start 16-byte aligned)
        v = __ldg(reinterpret_cast<const uint4*>(src));
      } else if (in && 8 * h < a.K) {
        // the chunk K ends in: only its values below K are read
        uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (uint32_t q = 0; q < 8; ++q)
          if (8 * h + q < a.K) w[q / 2] |= static_cast<uint32_t>(__ldg(src + q)) << (16 * (q % 2));
        v = make_uint4(w[0], w[1], w[2], w[3]);
      }
      sB[i + i / 8][h] = v;
    }
  }
  __syncthreads();
  // B values of columns c0 .. c0 + CPL - 1 in registers as column pairs
  float2 b[W][KK];
  {
    float x[CPL][KK];
#pragma unroll
    for (uint32_t t = 0; t < CPL; ++t) {
      const uint32_t i = static_cast<uint32_t>(c0 + t - bbase);
#pragma unroll
      for (uint32_t h = 0; h < kChunks; ++h) {
        const uint4 v = sB[i + i / 8][h];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (uint32_t q = 0; q < 4; ++q) {
          if (8 * h + 2 * q < KK) x[t][8 * h + 2 * q] = bf16f(w[q] & 0xFFFFu);
          if (8 * h + 2 * q + 1 < KK) x[t][8 * h + 2 * q + 1] = bf16f(w[q] >> 16);
        }
      }
    }
#pragma unroll
    for (uint32_t p = 0; p < W; ++p)
#pragma unroll
      for (uint32_t k = 0; k < KK; ++k) b[p][k] = make_float2(x[2 * p][k], x[2 * p + 1][k]);
  }
  for (uint32_t rt = blockIdx.y; rt * kTileRows < a.M; rt += gridDim.y) {
    const uint32_t row0 = rt * kTileRows;
    const uint32_t nrows = min(kTileRows, a.M - row0);
    __syncthreads();   // the previous row tile's reads of sA are done
    if (threadIdx.x < nrows) {
      float x[KK];
      load_row<KK>(a.A + static_cast<uint64_t>(row0 + threadIdx.x) * a.lda, a.K, x);
#pragma unroll
      for (uint32_t k = 0; k < KK; k += 2)
        *reinterpret_cast<float4*>(&sA[threadIdx.x][k]) = make_float4(x[k], x[k], x[k + 1], x[k + 1]);
    }
    __syncthreads();
#pragma unroll 2
    for (uint32_t r = warp; r < nrows; r += 8) {
      float2 acc[W];
#pragma unroll
      for (uint32_t p = 0; p < W; ++p) acc[p] = make_float2(0.0f, 0.0f);
#pragma unroll
      for (uint32_t k = 0; k < KK; k += 2) {
        const float4 av = *reinterpret_cast<const float4*>(&sA[r][k]);   // (a_k, a_k, a_k+1, a_k+1)
#pragma unroll
        for (uint32_t p = 0; p < W; ++p)
          acc[p] = __ffma2_rn(make_float2(av.x, av.y), b[p][k], acc[p]);
#pragma unroll
        for (uint32_t p = 0; p < W; ++p)
          acc[p] = __ffma2_rn(make_float2(av.z, av.w), b[p][k + 1], acc[p]);
      }
      uint32_t v[W];
#pragma unroll
      for (uint32_t p = 0; p < W; ++p) v[p] = pack_bf16x2(acc[p].x, acc[p].y);
      // 2*CPL-byte aligned: the row's start is e elements past a boundary
      uint16_t* const dst = a.D + static_cast<int64_t>(row0 + r) * static_cast<int64_t>(a.ldd) + c0;
      if (lane_full) {
        if constexpr (W == 4)
          *reinterpret_cast<uint4*>(dst) = make_uint4(v[0], v[1], v[2], v[3]);
        else
          *reinterpret_cast<uint2*>(dst) = make_uint2(v[0], v[1]);
      } else if (lane_any) {
        // the matrix's left or right edge: one 2-byte store per column inside
#pragma unroll
        for (uint32_t t = 0; t < CPL; ++t)
          if (c0 + t >= 0 && c0 + t < a.N)
            dst[t] = static_cast<uint16_t>(t % 2 ? v[t / 2] >> 16 : v[t / 2] & 0xFFFFu);
      }
    }
  }
}

}  // namespace

uint32_t smallk_max_k() { return kMaxK; }

int launch_bf16_smallk(const Problem& p, int num_sms, cudaStream_t stream) {
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
  const uint32_t cpl = p.K <= 8 ? 8u : 4u;
  // a warp's strip starts up to cpl - 1 columns before the block's, so the
  // strips must cover N + cpl - 1 columns
  const uint64_t strips = (static_cast<uint64_t>(p.N) + cpl - 1 + 32 * cpl - 1) / (32 * cpl);
  const uint64_t row_tiles = (static_cast<uint64_t>(p.M) + kTileRows - 1) / kTileRows;
  if (strips > 0x7FFFFFFFull) return GEMM_ERR_INVALID_ARG;
  // one wave of two blocks per SM; each block walks its strip's row tiles
  const uint64_t target = 2ull * static_cast<uint64_t>(num_sms > 0 ? num_sms : 1);
  uint64_t gy = (target + strips - 1) / strips;
  if (gy > row_tiles) gy = row_tiles;
  if (gy > 65535) gy = 65535;
  if (gy < 1) gy = 1;
  const dim3 grid(static_cast<unsigned>(strips), static_cast<unsigned>(gy));
  if (p.K <= 4)
    gemm_smallk_kernel<4, 8><<<grid, kThreadsSmallK, 0, stream>>>(a);
  else if (p.K <= 8)
    gemm_smallk_kernel<8, 8><<<grid, kThreadsSmallK, 0, stream>>>(a);
  else
    gemm_smallk_kernel<16, 4><<<grid, kThreadsSmallK, 0, stream>>>(a);
  if (const cudaError_t e = cudaGetLastError(); e != cudaSuccess) {
    note_cuda_error(e);
    return GEMM_ERR_LAUNCH;
  }
  return GEMM_OK;
}

}  // namespace gb300
