// ar_fp8_fused_f16.cu — fused FP8 allreduce kernels for f16 inputs (see ar_fp8_fused_impl.cuh).
#include "ar_fp8_fused_impl.cuh"

namespace gar {
cudaError_t launch_fp8_fused_f16(int out_dtype, int op, int mode, bool vec, const Fp8FusedArgs& a,
                                 cudaStream_t stream) {
  if (out_dtype == DT_F16) return launch_fused_io<DT_F16, DT_F16>(op, mode, vec, a, stream);
  if (out_dtype == DT_BF16) return launch_fused_io<DT_F16, DT_BF16>(op, mode, vec, a, stream);
  return cudaErrorInvalidValue;  // 16-bit inputs need 16-bit outputs
}
}  // namespace gar
