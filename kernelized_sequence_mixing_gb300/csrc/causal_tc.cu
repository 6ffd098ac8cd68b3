// Causal linear attention on tcgen05 tensor cores (bf16 operands, fp32
// accumulation in tensor memory).  Not yet implemented: every shape falls
// back to the CUDA-core kernel.
#include "kernels.h"

namespace linattn {

cudaError_t launch_causal_tc(const Problem &, const Gammas &, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace linattn
