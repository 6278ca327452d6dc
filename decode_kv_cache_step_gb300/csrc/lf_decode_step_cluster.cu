// Instantiations of the decode-step kernel whose unit runs as one
// thread-block cluster (one-wave grids): a 2-stage TMA ring at three CTAs
// per SM, or a kDeepStages ring at one CTA per SM that keeps every tile of a
// short chunk in flight at once when the grid has at most one CTA per SM.
#include "lf_step_kernel.cuh"

namespace lf {
namespace {

template <int D, int G>
cudaError_t launch_cluster_dg(const CUtensorMap& tmK, const CUtensorMap& tmV, const StepParams& p,
                              int units, cudaStream_t stream, int stages, bool score, bool pdl) {
    if (stages == kDeepStages)
        return score ? launch_t<D, G, kDeepStages, true, true>(tmK, tmV, p, units, stream, pdl)
                     : launch_t<D, G, kDeepStages, false, true>(tmK, tmV, p, units, stream, pdl);
    return score ? launch_t<D, G, 2, true, true>(tmK, tmV, p, units, stream, pdl)
                 : launch_t<D, G, 2, false, true>(tmK, tmV, p, units, stream, pdl);
}

}  // namespace

cudaError_t launch_decode_step_cluster(int D, int G, int stages, bool score,
                                       const CUtensorMap& tmK, const CUtensorMap& tmV,
                                       const StepParams& p, int units, cudaStream_t stream,
                                       bool pdl) {
#define LF_STEP_CASE(DD, GG) \
    if (D == DD && G == GG)  \
        return launch_cluster_dg<DD, GG>(tmK, tmV, p, units, stream, stages, score, pdl);
    LF_STEP_CASE(64, 1) LF_STEP_CASE(64, 2) LF_STEP_CASE(64, 4) LF_STEP_CASE(64, 8)
    LF_STEP_CASE(128, 1) LF_STEP_CASE(128, 2) LF_STEP_CASE(128, 4) LF_STEP_CASE(128, 8)
#undef LF_STEP_CASE
    return cudaErrorInvalidValue;
}

}  // namespace lf
