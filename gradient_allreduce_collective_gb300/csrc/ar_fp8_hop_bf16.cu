// ar_fp8_hop_bf16.cu — per-hop FP8 allreduce kernels for bf16 inputs (see ar_fp8_hop_impl.cuh).
#include "ar_fp8_hop_impl.cuh"

namespace gar {
cudaError_t launch_fp8_hop_bf16(int out_dtype, int op, const Fp8HopArgs& a, cudaStream_t stream) {
  return launch_hop_in<DT_BF16>(out_dtype, op, a, stream);
}
}  // namespace gar
