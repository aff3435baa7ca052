// mnw_gemm_warp_dep.cu -- the warp-MMA kernel instances that take part in a
// gate/up -> down tile dependency (see WarpDep in mnw_internal.h), compiled
// apart from the others so that the two translation units build in parallel.
#include "mnw_gemm_warp.cuh"

namespace mnw {
namespace warpmma {

#define MNW_WARP_DEP_DEFINE(WF, AM, GU, NT, DEP) \
  template cudaError_t launch<WF, AM, GU, NT, DEP>(const CUtensorMap*, const Args&, size_t, int, cudaStream_t);
MNW_WARP_DEP_INSTANCES(MNW_WARP_DEP_DEFINE)
#undef MNW_WARP_DEP_DEFINE

}  // namespace warpmma
}  // namespace mnw
