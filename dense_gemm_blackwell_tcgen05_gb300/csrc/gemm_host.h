// Host-side plumbing shared by the translation units of the library (not
// part of the public ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace gb300 {

struct Problem {
  uint32_t M, N, K;
  uint64_t lda, ldb, ldd, ldsfa, ldsfb;
  const void* A;
  const void* B;
  const void* SFA;
  const void* SFB;
  void* D;
  uint32_t stall_iter = 0xFFFFFFFFu;   // watchdog test hook (see gemm_debug_stall_next_launch)
  void* workspace = nullptr;           // stream-K partials + flags (nullptr: data-parallel only)
  uint64_t workspace_bytes = 0;
};

// Stream-K workspace per CTA: 4 epilogue warps x 32 rows x tile_n fp32, plus
// 4 flags; the library sizes it for every SM of the device.
inline uint64_t streamk_bytes_per_cta(uint32_t tile_n) {
  return 4ull * 32ull * tile_n * 4ull + 4ull * 4ull;
}

struct LaunchCtx {
  int device;
  int num_sms;
  unsigned long long* status;      // device address of the status word
  unsigned long long timeout_ns;
};

struct Maps {
  CUtensorMap A;
  CUtensorMap B;
  CUtensorMap D;
  CUtensorMap SFA;
  CUtensorMap SFB;
};

// Records the CUDA error behind a GEMM_ERR_LAUNCH for gemm_last_cuda_error().
void note_cuda_error(cudaError_t e);
// Records the calling thread's last persistent-kernel schedule (gemm_last_schedule).
void note_schedule(uint32_t clusters, uint32_t cg, uint32_t dp_tiles, uint32_t sk_tiles,
                   uint32_t sk_unit);

// Encodes a 2-D tiled tensor map (rows of `inner` elements, pitch in bytes).
// Returns false when the driver rejects it.
bool encode_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner,
                   uint64_t rows, uint64_t pitch_bytes, uint32_t box_inner, uint32_t box_rows,
                   CUtensorMapSwizzle swizzle);

// Kernel launchers; each returns a gemm_status_t value.
int launch_bf16_ws(int cg, bool tma_store, const Problem& p, const LaunchCtx& ctx,
                   cudaStream_t stream);
int launch_bf16_sync(const Problem& p, const LaunchCtx& ctx, cudaStream_t stream);
int launch_mxf8_ws(int cg, bool tma_store, const Problem& p, const LaunchCtx& ctx,
                   cudaStream_t stream);
int launch_zero_fill(const Problem& p, cudaStream_t stream);
int launch_mxfp8_quantize(const float* X, uint32_t rows, uint32_t K, uint64_t ldx, uint8_t* Q,
                          uint64_t ldq, uint8_t* SF, uint64_t ldsf, int num_sms,
                          cudaStream_t stream);

// Compile-time plans for gemm_kernel_plan().
struct KernelPlan {
  int stages, smem_bytes, tmem_cols, threads, cluster, tile_m, tile_n;
};
bool plan_bf16(int cg, bool tma_store, KernelPlan* out);
bool plan_mxf8(int cg, bool tma_store, KernelPlan* out);

}  // namespace gb300
