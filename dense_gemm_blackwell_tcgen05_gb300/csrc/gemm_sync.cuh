// Ladder levels 1-3 (one tile per CTA, synchronous copies) and the K = 0
// fill.  Included by exactly one translation unit.
#pragma once

#include <cstdint>

#include "gemm_kernels.cuh"

namespace gb300 {

// ----------------------------------------------------------------------------
// Ladder levels 1-3: one 128x128 output tile per CTA, synchronous copies.
// 128 threads copy the A and B K-tiles (64 bf16 = 128 bytes per row) from
// global memory into the 128-byte-swizzled K-major layout, one thread issues
// four K=16 MMAs (M=128, N=128) and commits to an mbarrier that every thread
// waits on before the slot is overwritten; the accumulator is read back with
// tcgen05.ld and stored with masks.
// ----------------------------------------------------------------------------
struct SyncArgs {
  const uint16_t* A;
  const uint16_t* B;
  uint16_t* D;
  uint32_t M, N, K;
  uint64_t lda, ldb, ldd;
  unsigned long long* status;
  unsigned long long timeout_ns;
};

__device__ __forceinline__ uint4 load_row_chunk8(const uint16_t* src_row, uint32_t k, uint32_t K,
                                                 bool row_ok) {
  if (!row_ok || k >= K) return make_uint4(0, 0, 0, 0);
  if (k + 8 <= K) return *reinterpret_cast<const uint4*>(src_row + k);
  uint16_t h[8];
#pragma unroll
  for (uint32_t i = 0; i < 8; ++i) h[i] = (k + i < K) ? src_row[k + i] : uint16_t(0);
  return make_uint4(h[0] | (uint32_t(h[1]) << 16), h[2] | (uint32_t(h[3]) << 16),
                    h[4] | (uint32_t(h[5]) << 16), h[6] | (uint32_t(h[7]) << 16));
}

__global__ void __launch_bounds__(128, 1) gemm_sync_kernel(const SyncArgs args) {
  __shared__ __align__(1024) uint8_t sA[128 * 128];
  __shared__ __align__(1024) uint8_t sB[128 * 128];
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tmem_slot;
  __shared__ uint32_t abort_word;
  const uint32_t tid = threadIdx.x;
  const uint32_t warp = warp_idx_sync();
  const uint32_t lane = lane_idx();
  const uint32_t m0 = blockIdx.y * 128, n0 = blockIdx.x * 128;
  const Watchdog wd{args.status, args.timeout_ns, &abort_word};
  if (tid == 0) {
    mbar_init(smem_addr(&bar), 1);
    abort_word = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc<1>(smem_addr(&tmem_slot), 128);
    tmem_relinquish<1>();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(&tmem_slot);
  const uint32_t num_kt = (args.K + 63) / 64;
  bool ok = true;
  uint32_t kt = 0;
  for (; kt < num_kt && ok; ++kt) {
    // 128 rows x 8 chunks of 16 bytes per operand, 8 chunks per thread
#pragma unroll 1
    for (uint32_t idx = tid; idx < 1024; idx += 128) {
      const uint32_t r = idx >> 3, c = idx & 7u;
      const uint32_t k = kt * 64 + c * 8;
      const uint32_t sw = (r * 128) + ((c ^ (r & 7u)) << 4);
      *reinterpret_cast<uint4*>(sA + sw) =
          load_row_chunk8(args.A + static_cast<uint64_t>(m0 + r) * args.lda, k, args.K, m0 + r < args.M);
      *reinterpret_cast<uint4*>(sB + sw) =
          load_row_chunk8(args.B + static_cast<uint64_t>(n0 + r) * args.ldb, k, args.K, n0 + r < args.N);
    }
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after_sync();
      const uint64_t adesc = smem_desc_sw128(smem_addr(sA));
      const uint64_t bdesc = smem_desc_sw128(smem_addr(sB));
#pragma unroll
      for (uint32_t k = 0; k < 4; ++k)
        mma_bf16<1>(tmem, adesc + 2 * k, bdesc + 2 * k, idesc_bf16(128, 128), (kt | k) != 0u);
      tc_commit(smem_addr(&bar));
    }
    __syncwarp();
    ok = warp_wait(smem_addr(&bar), kt & 1u, wd, kSiteSyncMma, lane);
    ok = __syncthreads_and(ok);
    tc_fence_after_sync();
    if (!ok && tid == 0) drain_wait(smem_addr(&bar), kt & 1u, wd, kSiteMmaDrain);
  }
  if (ok) {
    const uint32_t row = m0 + warp * 32 + lane;
#pragma unroll 1
    for (uint32_t c = 0; c < 4; ++c) {
      uint32_t v[32];
      tmem_ld_32x32b_x32_sync(tmem + ((warp * 32u) << 16) + c * 32, v);
      if (num_kt == 0) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0u;
      }
      store_row32(args.D, args.ldd, args.M, args.N, row, n0 + c * 32, v);
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc<1>(tmem, 128);
  }
}

// D = 0 (the empty sum), any pitch.
__global__ void zero_fill_kernel(uint16_t* D, uint32_t M, uint32_t N, uint64_t ldd) {
  const uint64_t total = static_cast<uint64_t>(M) * N;
  for (uint64_t i = blockIdx.x * static_cast<uint64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<uint64_t>(gridDim.x) * blockDim.x) {
    const uint64_t r = i / N, c = i - r * N;
    D[r * ldd + c] = 0;
  }
}

}  // namespace gb300
