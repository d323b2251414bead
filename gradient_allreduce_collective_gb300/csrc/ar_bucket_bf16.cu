// ar_bucket_bf16.cu — bucket allreduce kernels for one element type (see ar_bucket_impl.cuh).
#include "ar_bucket_impl.cuh"

namespace gar {
cudaError_t launch_bucket_bf16(int op, int mode, const BucketArgs& a, cudaStream_t stream) {
  return launch_bucket_dt<DT_BF16>(op, mode, a, stream);
}
}  // namespace gar
