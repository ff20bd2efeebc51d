// gemm_bf16_streamk_noalloc: the bf16 stream-K GEMM with its scratch in a
// fixed, statically sized device buffer instead of a caller workspace.
//
// Who this is for: callers that must not allocate device memory at the point
// where they multiply.  Examples are code running inside a memory allocator's
// own out-of-memory or defragmentation path (an allocation there would
// re-enter the allocator) and a serving loop that reserves all of its device
// memory at start-up and may not grow afterwards.  Such callers cannot create
// the workspace gemm_bf16_streamk wants, so this entry point owns one.
//
// Nothing here allocates: the scratch is a file-scope __device__ array that
// the CUDA loader places with the module.  Its device address is fetched once
// per device (cudaGetSymbolAddress, with that device current) on the first
// call for the device, and that call also clears the buffer with a
// cudaMemsetAsync on the caller's stream, ordered before its own kernel.
// Later calls need no clearing: a completed split launch leaves its flag words
// at zero, and one that gave up on a watchdog timeout leaves flag values of
// its own launch, which no later launch waits for (the flag value is a
// process-wide launch sequence number).
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "gemm_gb300.h"
#include "gemm_host.h"

namespace {

// 24 MiB: partial tiles and flags for up to 191 resident CTAs of the bf16
// kernels (128 rows x 256 fp32 columns + 32 flag bytes per CTA); a GB300 runs
// at most 152.
constexpr uint64_t kScratchBytes = 24ull << 20;

__device__ __align__(256) unsigned char g_streamk_scratch[kScratchBytes];

constexpr int kMaxDevices = 128;
std::mutex g_mu;
void* g_ptr[kMaxDevices] = {};

// Device address of the scratch for the current device, set up on first use:
// the symbol lookup and a clear of the whole buffer on `stream` (the stream-K
// flags must start at zero; the partial slots need no initial value but
// clearing all of it is as cheap).  The clear is queued on the caller's
// stream, so the kernel that follows on that stream runs after it whatever the
// stream's flags.  Returns a gemm_status_t.
int scratch_for_current_device(cudaStream_t stream, void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return GEMM_ERR_UNSUPPORTED_DEVICE;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_ptr[dev] == nullptr) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_streamk_scratch);
    if (e == cudaSuccess) e = cudaMemsetAsync(p, 0, kScratchBytes, stream);
    if (e != cudaSuccess) {
      gb300::note_cuda_error(e);
      cudaGetLastError();
      return GEMM_ERR_LAUNCH;
    }
    g_ptr[dev] = p;
  }
  *out = g_ptr[dev];
  return GEMM_OK;
}

}  // namespace

extern "C" int gemm_bf16_streamk_noalloc(int variant, const void* A, const void* B, void* D,
                                         int64_t M, int64_t N, int64_t K, int64_t lda,
                                         int64_t ldb, int64_t ldd, cudaStream_t stream) {
  // Variants are checked here so that a bad one never reaches the set-up.
  const int base = variant & 0xFF;
  if ((variant & ~(0xFF | GEMM_VARIANT_DIRECT_STORE)) != 0 || base > GEMM_VARIANT_2CTA)
    return GEMM_ERR_INVALID_ARG;
  const int64_t need = gemm_streamk_workspace_bytes(0, variant);
  if (need < 0) return static_cast<int>(need);
  if (static_cast<uint64_t>(need) > kScratchBytes) return GEMM_ERR_INVALID_ARG;
  void* scratch = nullptr;
  if (const int rc = scratch_for_current_device(stream, &scratch); rc != GEMM_OK) return rc;
  return gemm_bf16_streamk(variant, A, B, D, M, N, K, lda, ldb, ldd, scratch,
                           static_cast<int64_t>(kScratchBytes), stream);
}
