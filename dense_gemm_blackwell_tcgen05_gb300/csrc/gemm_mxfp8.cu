// Block-scaled MXFP8 kernels of the library (E4M3 operands, one UE8M0 scale
// per 32 k carried into TMEM by tcgen05.cp).
#include "launch_ws.cuh"

namespace gb300 {

int launch_mxf8_ws(bool tma_store, const Problem& p, const LaunchCtx& ctx, cudaStream_t stream) {
  return tma_store ? launch_ws_impl<1, Kind::MXF8, true>(p, ctx, stream)
                   : launch_ws_impl<1, Kind::MXF8, false>(p, ctx, stream);
}

bool plan_mxf8(bool tma_store, KernelPlan* out) {
  tma_store ? fill_plan<1, Kind::MXF8, true>(out) : fill_plan<1, Kind::MXF8, false>(out);
  return true;
}

}  // namespace gb300
