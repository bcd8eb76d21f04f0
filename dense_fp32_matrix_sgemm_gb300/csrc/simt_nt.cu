// SIMT SGEMM instantiation: transA = false, transB = true.
#include "simt_launch.cuh"

namespace sgemm {
cudaError_t launch_simt_nt(const GemmArgs &a, bool vec, cudaStream_t s) {
    return simt::launch_pair<false, true>(a, vec, s);
}
}  // namespace sgemm
