// ar_reduce_bf16.cu — reduction kernels for one element type (see ar_reduce_impl.cuh).
#include "ar_reduce_impl.cuh"

namespace gar {
cudaError_t launch_reduce_bf16(int op, int mode, const ReduceArgs& a, cudaStream_t stream) {
  return launch_reduce_dt<DT_BF16>(op, mode, a, stream);
}
}  // namespace gar
