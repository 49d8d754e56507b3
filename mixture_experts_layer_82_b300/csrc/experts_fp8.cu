// FP8 E4M3 grouped expert GEMMs (fine-grained scales).  Not built yet: the
// FP8 kind is rejected by the host checks until this kernel exists.
#include "common.cuh"
#include "kernels.h"

namespace moe {

cudaError_t launch_experts_fp8(const ExpertsArgs&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace moe
