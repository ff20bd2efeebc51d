// Device-side pieces shared by the GEMM kernels: the status word protocol,
// bounded mbarrier waits (the watchdog) and the persistent tile order.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace gb300 {

// Status word layout (64-bit, first error wins via atomicCAS from 0):
//   bits 56-63 error code, bits 48-55 site, bits 0-31 linear CTA index.
enum DeviceError : uint32_t { kDevOk = 0, kDevTimeout = 5 };

enum WaitSite : uint32_t {
  kSiteProducerEmpty = 1,   // producer waiting for a stage to be freed
  kSiteMmaFull = 2,         // MMA waiting for a stage's TMA bytes
  kSiteMmaAccEmpty = 3,     // MMA waiting for the epilogue to drain TMEM
  kSiteEpiAccFull = 4,      // epilogue waiting for the accumulator
  kSiteMmaDrain = 5,        // MMA issuer draining its own tcgen05 ops at exit
  kSiteProducerDrain = 6,   // producer draining its own TMA loads at exit
  kSiteSyncMma = 7,         // single-tile kernel waiting for its MMA
  kSiteSfFull = 8,          // scale-factor warp waiting for its scale bytes
  kSiteStreamKFlag = 9,     // stream-K owner waiting for a partial accumulator
  kSiteEpiC = 10,           // epilogue waiting for a TMA-loaded tile of C
};

// Fused-epilogue mode word (0: the plain bf16 store of the accumulator).
constexpr uint32_t kEpiOutF32 = 1u;    // D (and C) hold fp32
constexpr uint32_t kEpiC = 2u;         // + beta * C
constexpr uint32_t kEpiBias = 4u;      // + bias[column]
constexpr uint32_t kEpiBiasF32 = 8u;   // bias holds fp32 (else bf16)
constexpr uint32_t kEpiAlpha = 16u;    // alpha != 1
constexpr uint32_t kEpiActShift = 8u;  // activation code in bits 8..9
constexpr uint32_t kActRelu = 1u;
constexpr uint32_t kActGelu = 2u;

struct Watchdog {
  unsigned long long* status;       // library-owned device status word
  unsigned long long timeout_ns;    // per-wait limit
  volatile uint32_t* abort_flag;    // per-CTA shared flag: set once any wait gave up
};

__device__ __forceinline__ void report_error(unsigned long long* status, uint32_t code,
                                             uint32_t site) {
  const uint32_t cta = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
  const unsigned long long word = (static_cast<unsigned long long>(code) << 56) |
                                  (static_cast<unsigned long long>(site & 0xFF) << 48) | cta;
  atomicCAS(status, 0ull, word);
}

// Wait for the phase of `bar` with parity `parity` to complete, giving up
// after `wd.timeout_ns` (or as soon as another role of this CTA gave up).
// Returns false on give-up; the caller then takes its teardown path.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const Watchdog& wd,
                                             uint32_t site) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 31u) == 0) {
      if (*wd.abort_flag) return false;
      if (global_timer_ns() - t0 > wd.timeout_ns) {
        *wd.abort_flag = 1u;
        report_error(wd.status, kDevTimeout, site);
        return false;
      }
    }
  }
}

// Grouped raster over output tiles: `group` consecutive M-blocks are swept
// together along N so that CTAs resident at the same time share A and B
// panels in L2.  Tile t -> (mb, nb).
__device__ __forceinline__ void tile_coords(uint32_t t, uint32_t num_m, uint32_t num_n,
                                            uint32_t group, uint32_t& mb, uint32_t& nb) {
  const uint32_t span = group * num_n;
  const uint32_t g = t / span;
  const uint32_t first = g * group;
  const uint32_t gs = min(num_m - first, group);
  const uint32_t r = t - g * span;
  mb = first + r % gs;
  nb = r / gs;
}

}  // namespace gb300
