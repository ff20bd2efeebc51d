// MXFP8 quantisation on the GPU: float32 rows -> E4M3 codes + one UE8M0 scale
// per 32 consecutive k, the encoding the block-scaled GEMM consumes
// (b200-tmem-lifecycle-planner, "A1 -- Case 2: block-scaled MMA": block-scaled
// operands travel with their scale factors).  The per-block rule:
//   amax = largest |x| over the block's finite values
//   e    = smallest integer with amax <= 448 * 2^e, clamped to [-127, 127]
//          (amax = 0 gives e = -127); scale byte = e + 127
//   q    = round-to-nearest-even E4M3 of x * 2^-e (exact power-of-two scaling;
//          |x * 2^-e| <= 448 by construction); NaN / +-Inf -> E4M3 NaN.
// HBM-bound: 4 bytes read and ~1.03 bytes written per element.  The scale
// bytes go to a row-major matrix, or to the tiled layout of gemm_mxfp8_tiled
// (512-byte chunks of 128 rows x 4 blocks), whose padding is written as zero.
#include <cuda_runtime.h>

#include <cstdint>

#include "gemm_gb300.h"
#include "gemm_host.h"

namespace gb300 {
namespace {

struct QuantArgs {
  const float* X;
  uint8_t* Q;
  uint8_t* SF;
  uint32_t rows, K;
  uint64_t ldx, ldq, ldsf;
  uint32_t units_per_row;   // ceil(K / kUnit)
  bool vec_in, vec_out;     // 16-byte loads / 4-byte stores are aligned everywhere
  uint32_t groups;          // tiled layout: ceil(nblk / 4) block groups per row block
};

// Byte offset of the scale of (row, block b) in the SF buffer: row-major
// with pitch ldsf, or the tiled layout (ldsf unused).
template <bool TILED>
__device__ __forceinline__ uint64_t sf_offset(const QuantArgs& a, uint32_t row, uint32_t b) {
  if constexpr (!TILED) return static_cast<uint64_t>(row) * a.ldsf + b;
  return 512ull * (static_cast<uint64_t>(row / 128) * a.groups + b / 4) + 16 * (row % 32) +
         4 * ((row % 128) / 32) + b % 4;
}

// Elements per warp iteration (32 blocks of 32): eight 16-byte loads in flight
// per lane; 512 measured 5% slower, 2048 slower still.
constexpr uint32_t kUnit = 1024;

// Smallest e with amax <= 448 * 2^e for a finite amax >= 0, from its bits:
// amax = (1 + f) 2^(E-127) with 448 = 1.75 * 2^8, so e = E - 135 + (f > 0.75).
__device__ __forceinline__ int scale_exponent(float amax) {
  const uint32_t b = __float_as_uint(amax);
  const int E = static_cast<int>((b >> 23) & 0xFFu);
  int e = E - 135 + ((b & 0x7FFFFFu) > 0x600000u ? 1 : 0);
  e = e < -127 ? -127 : e;
  e = e > 127 ? 127 : e;
  return e;
}

__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t encode_one(float x, float scale) {
  if (!isfinite(x)) return (__float_as_uint(x) >> 24 & 0x80u) | 0x7Fu;
  return e4m3x2(x * scale, 0.0f) & 0xFFu;
}

template <bool TILED>
__global__ void __launch_bounds__(256) mxfp8_quantize_kernel(const QuantArgs a) {
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t warp_global = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const uint32_t warps = (gridDim.x * blockDim.x) >> 5;
  const uint64_t units = static_cast<uint64_t>(a.rows) * a.units_per_row;
  for (uint64_t u = warp_global; u < units; u += warps) {
    const uint32_t row = static_cast<uint32_t>(u / a.units_per_row);
    const uint32_t k0 = static_cast<uint32_t>(u % a.units_per_row) * kUnit;
    const float* xr = a.X + row * a.ldx;
    // lane l holds elements k0 + 128 j + 4 l .. +3, j = 0..7 (block 4 j + l / 8)
    float x[8][4];
#pragma unroll
    for (uint32_t j = 0; j < 8; ++j) {
      const uint32_t k = k0 + 128 * j + 4 * lane;
      if (a.vec_in && k + 4 <= a.K) {
        const float4 v = __ldcs(reinterpret_cast<const float4*>(xr + k));   // read once
        x[j][0] = v.x; x[j][1] = v.y; x[j][2] = v.z; x[j][3] = v.w;
      } else {
#pragma unroll
        for (uint32_t t = 0; t < 4; ++t) x[j][t] = (k + t < a.K) ? xr[k + t] : 0.0f;
      }
    }
#pragma unroll
    for (uint32_t j = 0; j < 8; ++j) {
      const uint32_t kb = k0 + 128 * j + 32 * (lane >> 3);   // first k of this lane's block
      float m = 0.0f;
      bool fin = true;   // this lane's four values are all finite
#pragma unroll
      for (uint32_t t = 0; t < 4; ++t) {
        const float ax = fabsf(x[j][t]);
        if (ax <= 3.402823466e38f) {   // finite values only
          if (ax > m) m = ax;
        } else {
          fin = false;
        }
      }
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
      if (kb >= a.K) {   // whole block past K (all lanes took part in the shuffles)
        // tiled layout: the last group's blocks past K hold zero
        if (TILED && (lane & 7u) == 0 && kb / 32 < 4 * a.groups) a.SF[sf_offset<TILED>(a, row, kb / 32)] = 0;
        continue;
      }
      const int e = scale_exponent(m);
      const float scale = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);   // 2^-e, e <= 126
      const uint32_t k = k0 + 128 * j + 4 * lane;
      // two values per conversion; a NaN or an infinity (E4M3 NaN, sign kept,
      // where the saturating conversion would give 448) one at a time
      uint32_t q = 0;
      if (fin) {
        q = e4m3x2(x[j][0] * scale, x[j][1] * scale) | (e4m3x2(x[j][2] * scale, x[j][3] * scale) << 16);
      } else {
#pragma unroll
        for (uint32_t t = 0; t < 4; ++t) q |= encode_one(x[j][t], scale) << (8 * t);
      }
      uint8_t* qr = a.Q + row * a.ldq;
      if (a.vec_out && k + 4 <= a.K) {
        __stcs(reinterpret_cast<unsigned int*>(qr + k), q);   // written once
      } else {
#pragma unroll
        for (uint32_t t = 0; t < 4; ++t)
          if (k + t < a.K) qr[k + t] = static_cast<uint8_t>(q >> (8 * t));
      }
      if ((lane & 7u) == 0) a.SF[sf_offset<TILED>(a, row, kb / 32)] = static_cast<uint8_t>(e + 127);
    }
  }
  if constexpr (TILED) {
    // rows past the last real row of the last row block: zero scales
    const uint32_t pad_rows = (a.rows + 127) / 128 * 128 - a.rows;
    const uint64_t pad = static_cast<uint64_t>(pad_rows) * 4 * a.groups;
    for (uint64_t i = blockIdx.x * blockDim.x + threadIdx.x; i < pad; i += gridDim.x * blockDim.x)
      a.SF[sf_offset<TILED>(a, a.rows + static_cast<uint32_t>(i / (4 * a.groups)),
                            static_cast<uint32_t>(i % (4 * a.groups)))] = 0;
  }
}

}  // namespace

int launch_mxfp8_quantize(const float* X, uint32_t rows, uint32_t K, uint64_t ldx, uint8_t* Q,
                          uint64_t ldq, uint8_t* SF, uint64_t ldsf, bool tiled, int num_sms,
                          cudaStream_t stream) {
  QuantArgs a;
  a.X = X;
  a.Q = Q;
  a.SF = SF;
  a.rows = rows;
  a.K = K;
  a.ldx = ldx;
  a.ldq = ldq;
  a.ldsf = ldsf;
  a.units_per_row = (K + kUnit - 1) / kUnit;
  a.groups = ((K + 31) / 32 + 3) / 4;
  a.vec_in = (reinterpret_cast<uintptr_t>(X) & 15u) == 0 && (ldx % 4) == 0;
  a.vec_out = (reinterpret_cast<uintptr_t>(Q) & 3u) == 0 && (ldq % 4) == 0;
  const uint64_t units = static_cast<uint64_t>(rows) * a.units_per_row;
  const uint64_t want = (units + 7) / 8;                      // 8 warps per block
  const uint64_t cap = static_cast<uint64_t>(num_sms) * 8;    // 8 blocks (64 warps) per SM
  const unsigned blocks = static_cast<unsigned>(want < cap ? want : cap);
  if (tiled)
    mxfp8_quantize_kernel<true><<<blocks, 256, 0, stream>>>(a);
  else
    mxfp8_quantize_kernel<false><<<blocks, 256, 0, stream>>>(a);
  if (const cudaError_t e = cudaGetLastError(); e != cudaSuccess) {
    note_cuda_error(e);
    return GEMM_ERR_LAUNCH;
  }
  return GEMM_OK;
}

}  // namespace gb300
