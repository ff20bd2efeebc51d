// bf16 kernels of the library: the persistent warp-specialised tcgen05
// kernel (one CTA or a CTA pair, TMA-store or masked-store epilogue), the
// synchronous single-tile reference rung and the K = 0 fill.
#include "gemm_sync.cuh"
#include "launch_ws.cuh"

namespace gb300 {

int launch_bf16_ws(int cg, bool tma_store, const Problem& p, const LaunchCtx& ctx,
                   cudaStream_t stream) {
  if (cg == 1)
    return tma_store ? launch_ws_impl<1, Kind::BF16, true>(p, ctx, stream)
                     : launch_ws_impl<1, Kind::BF16, false>(p, ctx, stream);
  if (cg == 2)
    return tma_store ? launch_ws_impl<2, Kind::BF16, true>(p, ctx, stream)
                     : launch_ws_impl<2, Kind::BF16, false>(p, ctx, stream);
  return GEMM_ERR_INVALID_ARG;
}

int bf16_streamk_split_tiles(int cg, const Problem& p, const LaunchCtx& ctx, uint32_t* sk_tiles) {
  if (cg == 1) return ws_streamk_split_tiles<1, Kind::BF16, false>(p, ctx, sk_tiles);
  if (cg == 2) return ws_streamk_split_tiles<2, Kind::BF16, false>(p, ctx, sk_tiles);
  return GEMM_ERR_INVALID_ARG;
}

bool plan_bf16(int cg, bool tma_store, KernelPlan* out) {
  if (cg == 1) {
    tma_store ? fill_plan<1, Kind::BF16, true>(out) : fill_plan<1, Kind::BF16, false>(out);
    return true;
  }
  if (cg == 2) {
    tma_store ? fill_plan<2, Kind::BF16, true>(out) : fill_plan<2, Kind::BF16, false>(out);
    return true;
  }
  if (cg == 3) {
    *out = KernelPlan{1, 0, 128, 128, 1, 128, 128};
    return true;
  }
  if (cg == 4) {   // small-K CUDA-core kernel: 128-row tiles of A (fp32) in shared memory
    *out = KernelPlan{0, 128 * 16 * 4, 0, 256, 1, 128, 256};
    return true;
  }
  return false;
}

int launch_bf16_sync(const Problem& p, const LaunchCtx& ctx, cudaStream_t stream) {
  SyncArgs a;
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
  const dim3 grid((p.N + 127) / 128, (p.M + 127) / 128);
  if (grid.y > 65535u) return GEMM_ERR_INVALID_ARG;
  // ~32 KB static + 15 KB unused dynamic shared memory (+1 KB reserved per
  // CTA, under the 48 KB no-opt-in limit): at most four CTAs per SM, so their
  // 128-column TMEM allocations (4 x 128 = 512 columns) never contend.
  gemm_sync_kernel<<<grid, 128, 15 * 1024, stream>>>(a);
  if (const cudaError_t e = cudaGetLastError(); e != cudaSuccess) {
    note_cuda_error(e);
    return GEMM_ERR_LAUNCH;
  }
  return GEMM_OK;
}

int launch_zero_fill(const Problem& p, cudaStream_t stream) {
  zero_fill_kernel<<<1024, 256, 0, stream>>>(static_cast<uint16_t*>(p.D), p.M, p.N, p.ldd);
  if (const cudaError_t e = cudaGetLastError(); e != cudaSuccess) {
    note_cuda_error(e);
    return GEMM_ERR_LAUNCH;
  }
  return GEMM_OK;
}

}  // namespace gb300
