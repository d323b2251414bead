// ar_reduce_f32.cu — reduction kernels for one element type (see ar_reduce_impl.cuh).
#include "ar_reduce_impl.cuh"

namespace gar {
cudaError_t launch_reduce_f32(int op, int mode, const ReduceArgs& a, cudaStream_t stream) {
  return launch_reduce_dt<DT_F32>(op, mode, a, stream);
}
}  // namespace gar
