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
  // fused epilogue (epi_mode bits in kernel_common.cuh; 0 = plain bf16 store)
  uint32_t epi_mode = 0;
  float alpha = 1.0f, beta = 0.0f;
  const void* C = nullptr;
  uint64_t ldc = 0;
  const void* bias = nullptr;
};

// Stream-K workspace per CTA: 4 lane quarters x 32 rows x tile_n fp32, plus
// 8 flags (one per lane quarter and epilogue group); the library sizes it for
// every SM of the device.
constexpr uint64_t kStreamKFlagBytes = 8ull * 4ull;
inline uint64_t streamk_bytes_per_cta(uint32_t tile_n) {
  return 4ull * 32ull * tile_n * 4ull + kStreamKFlagBytes;
}

// Stream-K schedule choice (host only).  Units are K-tiles of the kernel's
// MMA time (about 0.37 us for every kernel here): a tile costs KT; a split
// launch pays a fixed cost (contributor partial written, flag seen, owner
// fix-up set up: about 11 us measured) plus about 3 us per contributor whose
// 128 KB fp32 partial the owner streams in (the partial traffic moves at
// about 45 GB/s per SM).  Constants fitted to per-CTA timelines on GB300.
struct StreamKPlan {
  uint32_t dp_tiles;   // tiles computed whole, round-robin over `clusters`
  uint32_t sk_tiles;   // tiles after them, cut along K
  uint32_t clusters;   // clusters launched
};

enum StreamKMode { kStreamKAuto = 0, kStreamKAlways = 1, kStreamKNever = 2 };
int streamk_mode();

// Tail split of the data-parallel schedule: how many of `tiles` whole tiles
// (the last ones) to cut into two column halves over `resident` clusters --
// the tiles of the last, partial round, when their halves fit in one round
// (0 when switched off with gemm_set_tail_split).
uint32_t plan_tail_split(uint64_t tiles, uint64_t resident);

// The flag value of the next split launch: one process-wide sequence shared by
// every kernel configuration, never 0.  A flag word left behind by a launch
// that gave up (watchdog timeout) holds an earlier launch's value, which no
// later launch waits for, so a workspace needs zeroing only once, before its
// first use.
uint32_t next_streamk_epoch();

inline StreamKPlan plan_streamk(uint64_t tiles, uint64_t resident, uint32_t kt, uint32_t unit,
                                int mode) {
  constexpr double kFixed = 30.0, kPerContributor = 8.0, kMinGain = 0.05;
  const uint64_t ku = (kt + unit - 1) / unit;   // units per tile
  const uint64_t waves = tiles / resident, rem = tiles % resident;
  StreamKPlan dp{static_cast<uint32_t>(tiles), 0u,
                 static_cast<uint32_t>(tiles < resident ? tiles : resident)};
  if (mode == kStreamKNever || rem == 0 || ku < 2) return dp;
  const double t_dp = static_cast<double>(waves + 1) * kt;
  if (waves >= 1) {
    // the partial wave plus one full wave, dealt over every resident cluster:
    // each range spans more than one tile, so a tile has one contributor
    const uint64_t sk = rem + resident;
    StreamKPlan p{static_cast<uint32_t>(tiles - sk), static_cast<uint32_t>(sk),
                  static_cast<uint32_t>(resident)};
    const double t_sk = static_cast<double>(waves - 1) * kt +
                        static_cast<double>((sk * ku + resident - 1) / resident) * unit + kFixed +
                        kPerContributor;
    return (mode == kStreamKAlways || t_sk < (1.0 - kMinGain) * t_dp) ? p : dp;
  }
  // fewer tiles than clusters: all tiles split; choose how many clusters
  // (at most one per unit, so that no cluster's range is empty)
  const uint64_t units = tiles * ku;
  const uint64_t cap = units < resident ? units : resident;
  StreamKPlan best = dp;
  double t_best = 1e300;
  for (uint64_t g = tiles + 1; g <= cap; ++g) {
    const uint64_t per = (units + g - 1) / g;                  // units per cluster
    const uint64_t contributors = (ku + per - 1) / per;        // later ranges touching a tile
    const double t = static_cast<double>(per) * unit + kFixed + kPerContributor * contributors;
    if (t < t_best || mode == kStreamKAlways) {
      t_best = t;
      best = StreamKPlan{0u, static_cast<uint32_t>(tiles), static_cast<uint32_t>(g)};
      if (mode == kStreamKAlways) best.clusters = static_cast<uint32_t>(cap);
    }
  }
  if (best.sk_tiles == 0) return dp;
  return (mode == kStreamKAlways || t_best < (1.0 - kMinGain) * t_dp) ? best : dp;
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
  CUtensorMap Bh;   // B with a half-height box, for column-half work items
  CUtensorMap C;    // the fused epilogue's C in D's staging boxes (when loaded by TMA)
};

// Records the CUDA error behind a GEMM_ERR_LAUNCH for gemm_last_cuda_error().
void note_cuda_error(cudaError_t e);
// Records the calling thread's last persistent-kernel schedule (gemm_last_schedule).
void note_schedule(uint32_t clusters, uint32_t cg, uint32_t dp_tiles, uint32_t sk_tiles,
                   uint32_t sk_unit, uint32_t half_tiles, uint32_t edge_last);
// Whether plain bf16 launches may deal right-edge tiles last (gemm_set_edge_last).
bool edge_last_enabled();

// Encodes a 2-D tiled tensor map (rows of `inner` elements, pitch in bytes).
// Returns false when the driver rejects it.
bool encode_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner,
                   uint64_t rows, uint64_t pitch_bytes, uint32_t box_inner, uint32_t box_rows,
                   CUtensorMapSwizzle swizzle);
// Encodes a 3-D tiled tensor map without swizzle: extents dims[0..2]
// (elements), strides of dimensions 1 and 2 in bytes, box extents box[0..2].
bool encode_map_3d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                   const uint64_t (&dims)[3], const uint64_t (&strides)[2], const uint32_t (&box)[3]);

// Kernel launchers; each returns a gemm_status_t value.
int launch_bf16_ws(int cg, bool tma_store, const Problem& p, const LaunchCtx& ctx,
                   cudaStream_t stream);
int launch_bf16_sync(const Problem& p, const LaunchCtx& ctx, cudaStream_t stream);
// Tiles a bf16 launch on `p` (one CTA or a pair) would split along K with its
// workspace under the current stream-K mode; 0 for the data-parallel schedule.
int bf16_streamk_split_tiles(int cg, const Problem& p, const LaunchCtx& ctx, uint32_t* sk_tiles);
int launch_mxf8_ws(int cg, bool tma_store, const Problem& p, const LaunchCtx& ctx,
                   cudaStream_t stream);
// MXFP8 with scale matrices in the tiled layout (gemm_mxfp8_tiled).
int launch_mxf8t_ws(int cg, bool tma_store, const Problem& p, const LaunchCtx& ctx,
                    cudaStream_t stream);
int launch_zero_fill(const Problem& p, cudaStream_t stream);
// CUDA-core kernel for 1 <= K <= smallk_max_k() (plain bf16 store only).
int launch_bf16_smallk(const Problem& p, int num_sms, cudaStream_t stream);
uint32_t smallk_max_k();
// Tensor-core kernel for 1 <= K <= 16 (plain bf16 store only).
int launch_bf16_smallk_tc(const Problem& p, const LaunchCtx& ctx, cudaStream_t stream);
// K == 0 with a fused epilogue: D = act(alpha * 0 + beta * C + bias).
int launch_epilogue_only(const Problem& p, int num_sms, cudaStream_t stream);
int launch_mxfp8_quantize(const float* X, uint32_t rows, uint32_t K, uint64_t ldx, uint8_t* Q,
                          uint64_t ldq, uint8_t* SF, uint64_t ldsf, bool tiled, int num_sms,
                          cudaStream_t stream);

// Compile-time plans for gemm_kernel_plan().
struct KernelPlan {
  int stages, smem_bytes, tmem_cols, threads, cluster, tile_m, tile_n;
};
bool plan_bf16(int cg, bool tma_store, KernelPlan* out);
bool plan_mxf8(int cg, bool tma_store, KernelPlan* out);
bool plan_mxf8t(int cg, bool tma_store, KernelPlan* out);

}  // namespace gb300
