// Instantiations of the decode-step kernel whose unit runs as one
// thread-block cluster (grids whose clusters are all resident at once): a
// 2-stage TMA ring at three CTAs per SM, or a kDeepStages ring at one CTA per
// SM that keeps every tile of a short chunk in flight at once. Also the
// cluster-residency query the launch plan relies on.
#include <atomic>

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

template <int D, int G>
int clusters_dg(int stages, bool score, int csize) {
    if (stages == kDeepStages)
        return score ? max_active_clusters_t<D, G, kDeepStages, true>(csize)
                     : max_active_clusters_t<D, G, kDeepStages, false>(csize);
    return score ? max_active_clusters_t<D, G, 2, true>(csize)
                 : max_active_clusters_t<D, G, 2, false>(csize);
}

}  // namespace

int max_active_clusters(int D, int G, int stages, bool score, int csize) {
    if (csize < 1 || csize > kMaxClusterChunks) return 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    // One query per device and instance (the answer is fixed for a process);
    // an entry holds the count + 1, 0 while unknown.
    constexpr int kDevs = 16;
    static std::atomic<int> cache[kDevs][2][4][2][2][kMaxClusterChunks + 1];
    const int gi = G == 1 ? 0 : (G == 2 ? 1 : (G == 4 ? 2 : 3));
    std::atomic<int>* c = dev < kDevs ? &cache[dev][D == 128 ? 1 : 0][gi]
                                              [stages == kDeepStages ? 1 : 0][score ? 1 : 0][csize]
                                      : nullptr;
    if (c) {
        const int v = c->load(std::memory_order_relaxed);
        if (v > 0) return v - 1;
    }
    int n = 0;
#define LF_STEP_CASE(DD, GG) \
    if (D == DD && G == GG) n = clusters_dg<DD, GG>(stages, score, csize);
    LF_STEP_CASE(64, 1) LF_STEP_CASE(64, 2) LF_STEP_CASE(64, 4) LF_STEP_CASE(64, 8)
    LF_STEP_CASE(128, 1) LF_STEP_CASE(128, 2) LF_STEP_CASE(128, 4) LF_STEP_CASE(128, 8)
#undef LF_STEP_CASE
    if (c) c->store(n + 1, std::memory_order_relaxed);
    return n;
}

int deep_term_slots(int D, int G) {
#define LF_STEP_CASE(DD, GG) \
    if (D == DD && G == GG) return StepAlloc<DD, GG, kDeepStages, true>::kTermSlots;
    LF_STEP_CASE(64, 1) LF_STEP_CASE(64, 2) LF_STEP_CASE(64, 4) LF_STEP_CASE(64, 8)
    LF_STEP_CASE(128, 1) LF_STEP_CASE(128, 2) LF_STEP_CASE(128, 4) LF_STEP_CASE(128, 8)
#undef LF_STEP_CASE
    return 0;
}

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
