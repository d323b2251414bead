// ar_bucket_impl.cuh — allreduce of a gradient bucket straight from its tensors.
//
// DDP packs many small gradients into one bucket per allreduce ("AllReduce
// （オールリデュース）" glossary, §パフォーマンスチューニング, bucketing). On one
// device the bucket need not exist: this kernel reads each rank's tensor t
// where it lives, folds every element in the order the bucket's allreduce
// would (its chunk is fixed by the element's offset in the bucket layout, so
// the ring start rank is the same as for the flattened bucket), and writes
// the result into every rank's output tensor t. The result is bit-identical
// to flatten -> allreduce -> unflatten while moving 2*N*B bytes instead of
// 6*N*B.
//
// One block handles one tile of kThreads items of one tensor (a block finds
// its tensor by binary search over tile_start, in parameter space); one
// thread handles one 16-byte vector (or one element on the element-wise
// path). Tensor offsets and chunk boundaries are multiples of the vector
// width, so a vector lies in one chunk; a tensor's last vector may be short
// and is then folded element by element.
#pragma once

#include <cstdint>

#include "ar_device.cuh"
#include "ar_reduce_impl.cuh"

namespace gar {

template <int DT, int OP, bool VEC> struct BucketLd {
  using R = Red<DT, OP>;
  using Acc = typename R::Acc;
  static constexpr int B = Fmt<DT>::bytes;
  static constexpr int V = VEC ? 16 / B : 1;
  using Raw = std::conditional_t<VEC, uint4, uint32_t>;

  const BucketArgs& A;
  int t;
  uint64_t idx;  // vector index (VEC) or element index within tensor t

  __device__ __forceinline__ Raw load(int r) const {
    const char* p = static_cast<const char*>(A.src[r * A.nt + t]);
    if constexpr (VEC) return __ldcs(reinterpret_cast<const uint4*>(p) + idx);
    else if constexpr (B == 4) return *(reinterpret_cast<const uint32_t*>(p) + idx);
    else return (uint32_t) * (reinterpret_cast<const uint16_t*>(p) + idx);
  }
  __device__ __forceinline__ void unpack(const Raw& raw, Acc (&a)[V]) const {
    if constexpr (VEC) {
#pragma unroll
      for (int k = 0; k < V; ++k) a[k] = R::init(get_lane<B>(raw, k));
    } else {
      a[0] = R::init(raw);
    }
  }
  __device__ __forceinline__ static Acc comb(Acc a, Acc b) { return R::comb(a, b); }
};

template <int DT, int OP, int MODE, int MAXN, bool VEC>
__device__ __forceinline__ void bucket_item(const BucketArgs& A, int t, uint64_t i, int c) {
  using Ld = BucketLd<DT, OP, VEC>;
  using R = typename Ld::R;
  constexpr int V = Ld::V;
  constexpr int B = Ld::B;
  const int N = A.nranks;
  const Ld ld{A, t, i};
  typename Ld::Acc acc[V];
  if constexpr (MODE == MODE_FUSED_TREE) {
    Fold<Ld>::template tree<MAXN>(ld, N, acc);
  } else {
    const int s = (c + 1 == N) ? 0 : c + 1;
    Fold<Ld>::template ring<MAXN>(ld, N, s, acc);
  }
  if constexpr (VEC) {
    uint4 out = make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int k = 0; k < V; ++k) set_lane<B>(out, k, R::fin(acc[k], N));
    for (int r = 0; r < N; ++r) __stcs(reinterpret_cast<uint4*>(A.dst[r * A.nt + t]) + i, out);
  } else {
    const uint32_t out = R::fin(acc[0], N);
    for (int r = 0; r < N; ++r) {
      char* p = static_cast<char*>(A.dst[r * A.nt + t]);
      if constexpr (B == 4) *(reinterpret_cast<uint32_t*>(p) + i) = out;
      else *(reinterpret_cast<uint16_t*>(p) + i) = (uint16_t)out;
    }
  }
}

template <int DT, int OP, int MODE, int MAXN>
__global__ void __launch_bounds__(kThreads) k_bucket_reduce(const __grid_constant__ BucketArgs A) {
  pdl_begin();
  constexpr int V = 16 / Fmt<DT>::bytes;
  const uint32_t total = A.tile_start[A.nt];
  for (uint32_t tile = blockIdx.x; tile < total; tile += gridDim.x) {
    int lo = 0, hi = A.nt - 1;  // the tensor whose tiles contain this one
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (A.tile_start[mid] <= tile) lo = mid;
      else hi = mid - 1;
    }
    const int t = lo;
    const uint64_t item = (uint64_t)(tile - A.tile_start[t]) * kThreads + threadIdx.x;
    const uint64_t cnt = A.count[t];
    if (A.vec) {
      const uint64_t e0 = item * V;
      if (e0 >= cnt) continue;
      const int c = (int)((A.offset[t] + e0) / A.L);
      if (e0 + V <= cnt) {
        bucket_item<DT, OP, MODE, MAXN, true>(A, t, item, c);
      } else {
        for (uint64_t e = e0; e < cnt; ++e) bucket_item<DT, OP, MODE, MAXN, false>(A, t, e, c);
      }
    } else {
      if (item >= cnt) continue;
      bucket_item<DT, OP, MODE, MAXN, false>(A, t, item, (int)((A.offset[t] + item) / A.L));
    }
  }
}

template <int DT, int OP, int MODE>
cudaError_t launch_bucket_t(const BucketArgs& a, cudaStream_t stream) {
  const uint32_t total = a.tile_start[a.nt];
  if (total == 0) return cudaSuccess;
  const unsigned grid = total < 0x7FFFFFFFu ? total : 0x7FFFFFFFu;  // one block per tile
  return a.nranks <= 8 ? launch_pdl(k_bucket_reduce<DT, OP, MODE, 8>, dim3(grid), 0, stream, a)
                       : launch_pdl(k_bucket_reduce<DT, OP, MODE, kMaxRanks>, dim3(grid), 0, stream, a);
}

template <int DT> cudaError_t launch_bucket_dt(int op, int mode, const BucketArgs& a, cudaStream_t s) {
#define GAR_BMODES(OPV)                                                               \
  return mode == MODE_FUSED_TREE ? launch_bucket_t<DT, OPV, MODE_FUSED_TREE>(a, s)    \
                                 : launch_bucket_t<DT, OPV, MODE_FUSED_RING>(a, s);
  switch (op) {
    case OP_SUM: GAR_BMODES(OP_SUM)
    case OP_AVG: GAR_BMODES(OP_AVG)
    case OP_MIN: GAR_BMODES(OP_MIN)
    case OP_MAX: GAR_BMODES(OP_MAX)
    default: return cudaErrorInvalidValue;
  }
#undef GAR_BMODES
}

}  // namespace gar
