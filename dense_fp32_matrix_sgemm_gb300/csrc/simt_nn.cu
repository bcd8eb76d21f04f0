// SIMT SGEMM instantiation: transA = false, transB = false.
#include "simt_launch.cuh"

namespace sgemm {
cudaError_t launch_simt_nn(const GemmArgs &a, bool vec, cudaStream_t s) {
    return simt::launch_pair<false, false>(a, vec, s);
}
}  // namespace sgemm
