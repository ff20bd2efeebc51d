// Block-scaled MXFP8 kernels of the library (E4M3 operands, one UE8M0 scale
// per 32 k carried into TMEM by tcgen05.cp): the single-CTA kernel and the
// cta_group::2 pair kernel.  Both use 224-column tiles (two accumulators and
// the scale columns fit in 512 TMEM columns); their TMA-store epilogue works
// in 32-column boxes (224 = 7 x 32), the masked-store one in 32x32 chunks.
// Split stream-K launches of the single-CTA kernel use its masked-store
// variant with a second epilogue group.
#include "launch_ws.cuh"

namespace gb300 {

int launch_mxf8_ws(int cg, bool tma_store, const Problem& p, const LaunchCtx& ctx,
                   cudaStream_t stream) {
  if (cg == 1) {
    // A launch that splits tiles along K also sums partial tiles in its
    // epilogue warps: the masked-store variant with a second epilogue group
    // shares that work between eight warps (as for bf16).
    uint32_t sk_tiles = 0;
    if (const int rc = ws_streamk_split_tiles<1, Kind::MXF8, false>(p, ctx, &sk_tiles); rc != GEMM_OK)
      return rc;
    if (sk_tiles != 0) return launch_ws_impl<1, Kind::MXF8, false, true>(p, ctx, stream);
    return tma_store ? launch_ws_impl<1, Kind::MXF8, true>(p, ctx, stream)
                     : launch_ws_impl<1, Kind::MXF8, false>(p, ctx, stream);
  }
  if (cg == 2)
    return tma_store ? launch_ws_impl<2, Kind::MXF8, true>(p, ctx, stream)
                     : launch_ws_impl<2, Kind::MXF8, false>(p, ctx, stream);
  return GEMM_ERR_INVALID_ARG;
}

bool plan_mxf8(int cg, bool tma_store, KernelPlan* out) {
  if (cg == 1) {
    tma_store ? fill_plan<1, Kind::MXF8, true>(out) : fill_plan<1, Kind::MXF8, false>(out);
    return true;
  }
  if (cg == 2) {
    tma_store ? fill_plan<2, Kind::MXF8, true>(out) : fill_plan<2, Kind::MXF8, false>(out);
    return true;
  }
  return false;
}

int launch_mxf8t_ws(int cg, bool tma_store, const Problem& p, const LaunchCtx& ctx,
                    cudaStream_t stream) {
  if (cg == 1)
    return tma_store ? launch_ws_impl<1, Kind::MXF8T, true>(p, ctx, stream)
                     : launch_ws_impl<1, Kind::MXF8T, false>(p, ctx, stream);
  if (cg == 2)
    return tma_store ? launch_ws_impl<2, Kind::MXF8T, true>(p, ctx, stream)
                     : launch_ws_impl<2, Kind::MXF8T, false>(p, ctx, stream);
  return GEMM_ERR_INVALID_ARG;
}

bool plan_mxf8t(int cg, bool tma_store, KernelPlan* out) {
  if (cg == 1) {
    tma_store ? fill_plan<1, Kind::MXF8T, true>(out) : fill_plan<1, Kind::MXF8T, false>(out);
    return true;
  }
  if (cg == 2) {
    tma_store ? fill_plan<2, Kind::MXF8T, true>(out) : fill_plan<2, Kind::MXF8T, false>(out);
    return true;
  }
  return false;
}

}  // namespace gb300
