// Host-side launcher of gemm_ws_kernel: encodes the tensor maps, sizes the
// persistent grid from the SM count (or the number of co-resident clusters)
// and launches with the cluster dimension of the configuration.
#pragma once

#include <atomic>
#include <cstring>
#include <mutex>

#include "gemm_gb300.h"
#include "gemm_host.h"
#include "gemm_kernels.cuh"

namespace gb300 {

// The builds of gemm_ws_kernel<CG, KIND, TMA_STORE, EPI2> the library keeps:
// the plain one (PLAIN = true) for bf16 and the tiled-scale MXFP8 kernels,
// the general one for bf16 and the row-major-scale MXFP8 kernels (the
// tiled-scale entry point never splits tiles along K or fuses an epilogue).
// Not the general one-CTA bf16 TMA-store build: the launches that would need
// it (a fused epilogue on one CTA; a stream-K split) take the masked-store
// kernel, because that build faulted on one fused shape whose cause is not
// known.
template <int CG, Kind KIND, bool TMA_STORE, bool EPI2>
struct WsBuilds {
  static constexpr bool kPlain = KIND != Kind::MXF8 && !EPI2;
  static constexpr bool kGeneral = KIND != Kind::MXF8T && !(KIND == Kind::BF16 && CG == 1 && TMA_STORE);
  static_assert(kPlain || kGeneral, "at least one build");
};

// The kernel a launch runs: the plain build when the launch needs nothing it
// leaves out, else the general one; nullptr when this configuration keeps no
// build that fits (not reachable from the API).  Only the kept builds are
// named, so only they are instantiated.
template <int CG, Kind KIND, bool TMA_STORE, bool EPI2>
auto ws_kernel_for(bool plain) {
  using Bld = WsBuilds<CG, KIND, TMA_STORE, EPI2>;
  decltype(&gemm_ws_kernel<CG, KIND, TMA_STORE, EPI2, false>) k = nullptr;
  if constexpr (Bld::kPlain) {
    if (plain) k = gemm_ws_kernel<CG, KIND, TMA_STORE, EPI2, true>;
  }
  if constexpr (Bld::kGeneral) {
    if (k == nullptr) k = gemm_ws_kernel<CG, KIND, TMA_STORE, EPI2, false>;
  }
  return k;
}

// One-time, per device: opt the builds of gemm_ws_kernel<CG, KIND, TMA_STORE>
// into the large shared-memory carve-out and (pairs) find how many clusters
// can be resident at once.  *resident: the clusters a launch may use.
template <int CG, Kind KIND, bool TMA_STORE, bool EPI2 = false>
int ws_resident(const LaunchCtx& ctx, uint64_t* resident) {
  using C = GemmCfg<CG, KIND, TMA_STORE, EPI2>;
  using Bld = WsBuilds<CG, KIND, TMA_STORE, EPI2>;
  static std::mutex mu;
  static int prepared[128] = {0};
  static int max_clusters[128] = {0};
  if (ctx.device < 0 || ctx.device >= 128) return GEMM_ERR_UNSUPPORTED_DEVICE;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (!prepared[ctx.device]) {
      for (int build = 0; build < 2; ++build) {
        if (build == 0 ? !Bld::kPlain : !Bld::kGeneral) continue;
        auto k = ws_kernel_for<CG, KIND, TMA_STORE, EPI2>(build == 0);
        if (const cudaError_t e = cudaFuncSetAttribute(
                k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(C::SMEM_BYTES));
            e != cudaSuccess) {
          note_cuda_error(e);
          cudaGetLastError();
          return GEMM_ERR_LAUNCH;
        }
        if constexpr (CG == 2) {
          if (cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 0) !=
              cudaSuccess)
            cudaGetLastError();
        }
      }
      if constexpr (CG == 2) {
        cudaLaunchConfig_t q = {};
        q.gridDim = dim3(2 * ctx.num_sms);
        q.blockDim = dim3(C::kThreads);
        q.dynamicSmemBytes = C::SMEM_BYTES;
        cudaLaunchAttribute qa[1];
        qa[0].id = cudaLaunchAttributeClusterDimension;
        qa[0].val.clusterDim.x = CG;
        qa[0].val.clusterDim.y = 1;
        qa[0].val.clusterDim.z = 1;
        q.attrs = qa;
        q.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, ws_kernel_for<CG, KIND, TMA_STORE, EPI2>(Bld::kPlain), &q) !=
                cudaSuccess ||
            n <= 0) {
          cudaGetLastError();
          n = ctx.num_sms / 2;
        }
        max_clusters[ctx.device] = n;
      }
      prepared[ctx.device] = 1;
    }
  }
  *resident = CG == 2 ? static_cast<uint64_t>(max_clusters[ctx.device])
                      : static_cast<uint64_t>(ctx.num_sms);
  return GEMM_OK;
}

// The number of tiles a launch of gemm_ws_kernel<CG, KIND, TMA_STORE> on `p`
// would split along K (0: the data-parallel schedule).
template <int CG, Kind KIND, bool TMA_STORE, bool EPI2 = false>
int ws_streamk_split_tiles(const Problem& p, const LaunchCtx& ctx, uint32_t* sk_tiles) {
  using C = GemmCfg<CG, KIND, TMA_STORE, EPI2>;
  *sk_tiles = 0;
  if (p.workspace == nullptr) return GEMM_OK;
  uint64_t resident = 0;
  if (const int rc = ws_resident<CG, KIND, TMA_STORE, EPI2>(ctx, &resident); rc != GEMM_OK) return rc;
  const uint64_t tiles = static_cast<uint64_t>((p.M + C::UMMA_M - 1) / C::UMMA_M) *
                         ((p.N + C::UMMA_N - 1) / C::UMMA_N);
  const uint32_t kt = (p.K + C::BK - 1) / C::BK;
  *sk_tiles = plan_streamk(tiles, resident, kt, C::SF_WARP ? C::SF_GROUP : 1u, streamk_mode()).sk_tiles;
  return GEMM_OK;
}

template <int CG, Kind KIND, bool TMA_STORE, bool EPI2 = false>
int launch_ws_impl(const Problem& p, const LaunchCtx& ctx, cudaStream_t stream) {
  using C = GemmCfg<CG, KIND, TMA_STORE, EPI2>;
  uint64_t resident = 0;
  if (const int rc = ws_resident<CG, KIND, TMA_STORE, EPI2>(ctx, &resident); rc != GEMM_OK) return rc;

  Maps maps;
  std::memset(&maps, 0, sizeof maps);
  const CUtensorMapDataType dt =
      C::MX ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (!encode_map_2d(&maps.A, dt, p.A, p.K, p.M, p.lda * C::ELEM, C::BK, C::BLOCK_M,
                     CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_map_2d(&maps.B, dt, p.B, p.K, p.N, p.ldb * C::ELEM, C::BK, C::B_ROWS,
                     CU_TENSOR_MAP_SWIZZLE_128B))
    return GEMM_ERR_LAUNCH;
  if constexpr (TMA_STORE) {
    if (!encode_map_2d(&maps.D, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.D, p.N, p.M, p.ldd * 2, C::TS_COLS,
                       32, C::TS_COLS == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B))
      return GEMM_ERR_LAUNCH;
  }
  // Scale bytes travel by TMA when both matrices are 16-byte aligned with
  // pitches that are multiples of 16 bytes (TMA's rules); otherwise the
  // scale-factor warp gathers them with plain loads.
  const bool sf_gather =
      C::SF_WARP && (((reinterpret_cast<uintptr_t>(p.SFA) | reinterpret_cast<uintptr_t>(p.SFB)) & 15u) != 0 ||
                     p.ldsfa % 16 != 0 || p.ldsfb % 16 != 0);
  if constexpr (C::SF_TILED) {
    // the tiled scale matrices as 512-byte chunks (128 words of 32 bits),
    // indexed (K-tile, row block): one box is a K-tile's chunk of one row
    // block for A, of the tile's SFB_TILE_CHUNKS row blocks for B (chunks of
    // consecutive row blocks lie KT chunks apart)
    const uint64_t kt = (p.K + C::BK - 1) / C::BK;
    const uint64_t sa_dims[3] = {128, kt, (p.M + 127) / 128};
    const uint64_t sb_dims[3] = {128, kt, (p.N + 127) / 128};
    const uint64_t strides[2] = {512, kt * 512};
    const uint32_t sa_box[3] = {128, 1, 1};
    const uint32_t sb_box[3] = {128, 1, C::SFB_TILE_CHUNKS};
    if (!encode_map_3d(&maps.SFA, CU_TENSOR_MAP_DATA_TYPE_UINT32, p.SFA, sa_dims, strides, sa_box) ||
        !encode_map_3d(&maps.SFB, CU_TENSOR_MAP_DATA_TYPE_UINT32, p.SFB, sb_dims, strides, sb_box))
      return GEMM_ERR_LAUNCH;
  } else if (C::MX && !sf_gather) {
    const uint64_t nblk = (p.K + 31) / 32;
    if (!encode_map_2d(&maps.SFA, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.SFA, nblk, p.M, p.ldsfa, 16,
                       C::BLOCK_M, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_map_2d(&maps.SFB, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.SFB, nblk, p.N, p.ldsfb, 16,
                       C::SFB_ROWS, CU_TENSOR_MAP_SWIZZLE_NONE))
      return GEMM_ERR_LAUNCH;
  }

  GemmArgs a;
  a.M = p.M;
  a.N = p.N;
  a.K = p.K;
  a.num_m_blocks = (p.M + C::UMMA_M - 1) / C::UMMA_M;
  a.num_n_blocks = (p.N + C::UMMA_N - 1) / C::UMMA_N;
  a.num_k_tiles = (p.K + C::BK - 1) / C::BK;
  a.group_m = CG == 2 ? 8u : 16u;
  a.D = p.D;
  a.ldd = p.ldd;
  a.status = ctx.status;
  a.timeout_ns = ctx.timeout_ns;
  a.stall_iter = p.stall_iter;
  a.ws_part = nullptr;
  a.ws_flag = nullptr;
  a.epoch = 0;
  a.epi_mode = p.epi_mode;
  a.alpha = p.alpha;
  a.beta = p.beta;
  a.C = p.C;
  a.ldc = p.ldc;
  a.bias = p.bias;
  // C by TMA: bf16 C (bf16 output) in the TMA-store kernels with 64-column
  // staging chunks, when TMA can address it (16-byte base and pitch)
  a.c_tma = 0;
  if constexpr (TMA_STORE && C::TS_COLS == 64 && C::EPI_BUFS == 2) {
    if ((p.epi_mode & kEpiC) && !(p.epi_mode & kEpiOutF32) && p.C != nullptr &&
        (reinterpret_cast<uintptr_t>(p.C) & 15u) == 0 && (p.ldc * 2) % 16 == 0) {
      if (!encode_map_2d(&maps.C, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.C, p.N, p.M, p.ldc * 2,
                         C::TS_COLS, 32, CU_TENSOR_MAP_SWIZZLE_128B))
        return GEMM_ERR_LAUNCH;
      a.c_tma = 1;
    }
  }
  a.sf_gather = sf_gather ? 1u : 0u;
  a.sfa = static_cast<const uint8_t*>(p.SFA);
  a.sfb = static_cast<const uint8_t*>(p.SFB);
  a.ldsfa = p.ldsfa;
  a.ldsfb = p.ldsfb;

  const uint64_t tiles = static_cast<uint64_t>(a.num_m_blocks) * a.num_n_blocks;
  // Schedule.  Data-parallel: whole tiles round-robin over min(tiles, resident)
  // clusters.  Stream-K (only with a caller workspace, and only where the
  // cost model in plan_streamk predicts a gain, unless forced): the tiles of
  // the last partial wave plus one full wave, or all tiles when there are
  // fewer than clusters, are cut into units of sk_unit K-tiles dealt out in
  // equal contiguous ranges.
  a.dp_tiles = static_cast<uint32_t>(tiles);
  a.sk_tiles = 0;
  a.sk_unit = C::SF_WARP ? C::SF_GROUP : 1u;
  uint64_t clusters = tiles < resident ? tiles : resident;
  if (p.workspace != nullptr) {
    const uint64_t need = resident * CG * streamk_bytes_per_cta(C::UMMA_N);
    if (p.workspace_bytes < need || (reinterpret_cast<uintptr_t>(p.workspace) & 15u) != 0)
      return GEMM_ERR_INVALID_ARG;
    const StreamKPlan sp = plan_streamk(tiles, resident, a.num_k_tiles, a.sk_unit, streamk_mode());
    if (sp.sk_tiles != 0) {
      a.dp_tiles = sp.dp_tiles;
      a.sk_tiles = sp.sk_tiles;
      clusters = sp.clusters;
      // flags first (kStreamKFlagBytes per CTA slot), then the partial slots
      a.ws_flag = static_cast<uint32_t*>(p.workspace);
      a.ws_part = reinterpret_cast<float*>(static_cast<uint8_t*>(p.workspace) +
                                           resident * CG * kStreamKFlagBytes);
      a.epoch = next_streamk_epoch();
    }
  }
  // Tail split: a data-parallel launch cuts the tiles of a last, partial round
  // into column halves when those fit in one round (not in the kernels whose
  // scale-factor warp loads B scales by whole tiles).
  a.half_tiles = 0;
  if constexpr (!C::SF_WARP) {
    if (a.sk_tiles == 0) {
      a.half_tiles = plan_tail_split(tiles, resident);
      const uint64_t items = tiles + a.half_tiles;
      clusters = items < resident ? items : resident;
    }
  }
  // Right-edge tiles last (plain bf16 launches whose last column block holds
  // at most UMMA_N / 2 live columns): those tiles run as first column halves
  // and end the deal, instead of a tail split.
  a.edge_last = 0;
  a.edge_half = 0;
  if constexpr (KIND == Kind::BF16) {
    const uint32_t rem = p.N % C::UMMA_N;
    if (a.sk_tiles == 0 && a.epi_mode == 0 && a.c_tma == 0 && rem != 0 && rem <= C::UMMA_N / 2 &&
        a.num_n_blocks >= 2 && edge_last_enabled()) {
      a.edge_last = 1;
      a.edge_half = 1;
      a.half_tiles = 0;
      clusters = tiles < resident ? tiles : resident;
    }
  }
  if ((a.half_tiles != 0 || a.edge_half != 0) &&
      !encode_map_2d(&maps.Bh, dt, p.B, p.K, p.N, p.ldb * C::ELEM, C::BK, C::B_ROWS / 2,
                     CU_TENSOR_MAP_SWIZZLE_128B))
    return GEMM_ERR_LAUNCH;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  if constexpr (CG == 2) {
    cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters));
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  } else {
    cfg.gridDim = dim3(static_cast<unsigned>(clusters));
  }
  note_schedule(static_cast<uint32_t>(clusters), CG, a.dp_tiles, a.sk_tiles, a.sk_unit, a.half_tiles,
                a.edge_last);
  const auto kern =
      ws_kernel_for<CG, KIND, TMA_STORE, EPI2>(a.sk_tiles == 0 && a.epi_mode == 0 && a.c_tma == 0);
  if (kern == nullptr) return GEMM_ERR_INVALID_ARG;
  const cudaError_t err =
      cudaLaunchKernelEx(&cfg, kern, maps.A, maps.B, maps.D, maps.SFA, maps.SFB, maps.Bh, maps.C, a);
  if (err != cudaSuccess) {
    note_cuda_error(err);
    cudaGetLastError();
    return GEMM_ERR_LAUNCH;
  }
  return GEMM_OK;
}

template <int CG, Kind KIND, bool TMA_STORE, bool EPI2 = false>
void fill_plan(KernelPlan* out) {
  using C = GemmCfg<CG, KIND, TMA_STORE, EPI2>;
  out->stages = C::STAGES;
  out->smem_bytes = C::SMEM_BYTES;
  out->tmem_cols = C::TMEM_COLS;
  out->threads = C::kThreads;
  out->cluster = CG;
  out->tile_m = C::UMMA_M;
  out->tile_n = C::UMMA_N;
}

}  // namespace gb300
