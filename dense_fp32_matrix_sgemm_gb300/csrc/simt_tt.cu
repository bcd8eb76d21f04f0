// SIMT SGEMM instantiation: transA = true, transB = true.
#include "simt_launch.cuh"

namespace sgemm {
cudaError_t launch_simt_tt(const GemmArgs &a, bool vec, cudaStream_t s) {
    return simt::launch_pair<true, true>(a, vec, s);
}
cudaError_t launch_simt_streamk_tt(const GemmArgs &a, bool vec, const StreamKPlan &pl, void *ws,
                                    cudaStream_t s) {
    return simt::launch_streamk_pair<true, true>(a, vec, pl, ws, s);
}
}  // namespace sgemm
