// SIMT SGEMM instantiation: transA = true, transB = false.
#include "simt_launch.cuh"

namespace sgemm {
cudaError_t launch_simt_tn(const GemmArgs &a, bool vec, cudaStream_t s) {
    return simt::launch_pair<true, false>(a, vec, s);
}
cudaError_t launch_simt_streamk_tn(const GemmArgs &a, bool vec, const StreamKPlan &pl, void *ws,
                                    cudaStream_t s) {
    return simt::launch_streamk_pair<true, false>(a, vec, pl, ws, s);
}
}  // namespace sgemm
