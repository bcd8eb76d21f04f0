// Host-side access to the driver's tensor-map encoder (cuTensorMapEncodeTiled),
// looked up once through the runtime so the library links no libcuda.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

namespace sgemm {

// The encoder, or null when the driver does not provide it (defined in
// tf32x3.cu).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

}  // namespace sgemm
