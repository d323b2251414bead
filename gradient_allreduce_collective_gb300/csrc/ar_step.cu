// ar_step.cu — one reduce-scatter step of the stepwise executors (sm_103a).
//
// The stepwise executors run the pages' algorithms literally, one launch per
// step: the ring's N-1 reduce-scatter and N-1 all-gather steps ("AllReduce
// （オールリデュース）" glossary, §Ring-AllReduceの仕組み; "AllReduce" astro-wiki,
// §Ring AllReduce) and the recursive halving / doubling exchange (glossary
// algorithm table, "Recursive Halving-Doubling"; astro-wiki, §其他 AllReduce
// 算法). A reduce-scatter step combines, for every rank, the partial it
// receives with its own values into its own buffer; this kernel does that for
// all ranks of one step at once (all-gather steps are plain copies). Results
// equal the one-pass kernels' bit for bit: the combine is commutative and the
// grouping (the expression tree) is the same.
#include <cstdint>

#include "ar_device.cuh"

namespace gar {

// storage bits of an unfinished partial (binary32 sums are kept as binary32)
template <class Acc> __device__ __forceinline__ uint32_t partial_bits(Acc v) {
  if constexpr (std::is_same_v<Acc, float>) return __float_as_uint(v);
  else return v;
}

template <int DT, int OP>
__global__ void __launch_bounds__(kThreads) k_step_combine(const __grid_constant__ StepArgs A) {
  using R = Red<DT, OP>;
  constexpr int B = Fmt<DT>::bytes;
  constexpr int V = 16 / B;
  const uint32_t total = A.tile_start[A.ntasks];
  for (uint32_t tile = blockIdx.x; tile < total; tile += gridDim.x) {
    int lo = 0, hi = A.ntasks - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (A.tile_start[mid] <= tile) lo = mid;
      else hi = mid - 1;
    }
    const int t = lo;
    const uint64_t item = (uint64_t)(tile - A.tile_start[t]) * kThreads + threadIdx.x;
    const uint64_t len = A.len[t];
    if (A.vec && (item + 1) * V <= len) {
      const uint4 x = __ldcs(reinterpret_cast<const uint4*>(A.a[t]) + item);
      const uint4 y = __ldcs(reinterpret_cast<const uint4*>(A.b[t]) + item);
      uint4 o = make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int k = 0; k < V; ++k) {
        typename R::Acc v = R::comb(R::init(get_lane<B>(x, k)), R::init(get_lane<B>(y, k)));
        set_lane<B>(o, k, A.finish ? R::fin(v, A.nranks) : partial_bits(v));
      }
      __stcs(reinterpret_cast<uint4*>(A.dst[t]) + item, o);
    } else {
      const uint64_t e0 = A.vec ? item * V : item;
      const uint64_t e1 = A.vec ? (e0 + V < len ? e0 + V : len) : (e0 + 1 < len ? e0 + 1 : len);
      for (uint64_t e = e0; e < e1; ++e) {
        const uint32_t xa = reinterpret_cast<const uint32_t*>(A.a[t])[e];
        const uint32_t xb = reinterpret_cast<const uint32_t*>(A.b[t])[e];
        typename R::Acc v = R::comb(R::init(xa), R::init(xb));
        reinterpret_cast<uint32_t*>(A.dst[t])[e] = A.finish ? R::fin(v, A.nranks) : partial_bits(v);
      }
    }
  }
}

template <int DT, int OP> cudaError_t launch_step_t(const StepArgs& a, cudaStream_t s) {
  const uint32_t total = a.tile_start[a.ntasks];
  if (total == 0) return cudaSuccess;
  k_step_combine<DT, OP><<<total, kThreads, 0, s>>>(a);  // one block per tile
  return cudaGetLastError();
}

template <int DT> cudaError_t launch_step_dt(int op, const StepArgs& a, cudaStream_t s) {
  switch (op) {
    case OP_SUM: return launch_step_t<DT, OP_SUM>(a, s);
    case OP_AVG: return launch_step_t<DT, OP_AVG>(a, s);
    case OP_MIN: return launch_step_t<DT, OP_MIN>(a, s);
    case OP_MAX: return launch_step_t<DT, OP_MAX>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

// 4-byte element types only: partial sums are kept in the ranks' output
// buffers, in the element type itself
cudaError_t launch_step_combine(int dtype, int op, const StepArgs& a, cudaStream_t stream) {
  switch (dtype) {
    case DT_F32: return launch_step_dt<DT_F32>(op, a, stream);
    case DT_I32: return launch_step_dt<DT_I32>(op, a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gar
