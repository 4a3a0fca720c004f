// Placeholder until the tcgen05 GEMM lands: bf16-coded operands are rejected.
#include "internal.h"

namespace convrot {

cudaError_t launch_gemm_tc(const GemmArgs &, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace convrot
