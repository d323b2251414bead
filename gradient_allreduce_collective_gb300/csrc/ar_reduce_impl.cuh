// ar_reduce_impl.cuh — the reduction kernel (reduce-scatter, fused ring,
// fused tree), instantiated per element type in ar_reduce_<type>.cu.
//
// One thread owns one 16-byte vector position (or one element on the
// unaligned path): it loads the N ranks' vectors (8 in flight), folds them in
// the fixed order, finishes (AVG divide, rounding) and stores to the chunk
// owner (MODE_RS) or to all N outputs (fused modes). The grid has one thread
// per position; the grid-stride loop only matters beyond the largest grid,
// and then tracks the chunk incrementally. Chunk boundaries are multiples of
// the vector width, so a vector never straddles two chunks and its fold start
// rank is constant. HBM-bound: N*16 bytes read and 16 or N*16 bytes
// written per vector, ~(N-1)/4 flops per 16 bytes read.
#pragma once

#include "ar_device.cuh"

namespace gar {

template <int DT, int OP, bool VEC> struct PlainLd {
  using R = Red<DT, OP>;
  using Acc = typename R::Acc;
  static constexpr int B = Fmt<DT>::bytes;
  static constexpr int V = VEC ? 16 / B : 1;
  using Raw = std::conditional_t<VEC, uint4, uint32_t>;

  const ReduceArgs& A;
  uint64_t idx;  // vector index (VEC) or element index

  __device__ __forceinline__ Raw load(int r) const {
    const char* p = static_cast<const char*>(A.src[r]);
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

  __device__ __forceinline__ static void store(void* base, uint64_t i, const Raw& v) {
    char* p = static_cast<char*>(base);
    if constexpr (VEC) __stcs(reinterpret_cast<uint4*>(p) + i, v);
    else if constexpr (B == 4) *(reinterpret_cast<uint32_t*>(p) + i) = v;
    else *(reinterpret_cast<uint16_t*>(p) + i) = (uint16_t)v;
  }
};

// Reduce item `i` (vector or element index) that lies in chunk c at offset `ci`.
template <int DT, int OP, int MODE, int MAXN, bool VEC>
__device__ __forceinline__ void reduce_item(const ReduceArgs& A, uint64_t i, int c, uint64_t ci) {
  using Ld = PlainLd<DT, OP, VEC>;
  using R = typename Ld::R;
  constexpr int V = Ld::V;
  const int N = A.nranks;
  const Ld ld{A, i};
  typename Ld::Acc acc[V];
  if constexpr (MODE == MODE_FUSED_TREE) {
    Fold<Ld>::template tree<MAXN>(ld, N, acc);
  } else {
    const int s = (c + 1 == N) ? 0 : c + 1;  // chunk c starts at rank c+1
    Fold<Ld>::template ring<MAXN>(ld, N, s, acc);
  }
  typename Ld::Raw out;
  if constexpr (VEC) {
    out = make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int k = 0; k < V; ++k) set_lane<Ld::B>(out, k, R::fin(acc[k], N));
  } else {
    out = R::fin(acc[0], N);
  }
  if constexpr (MODE == MODE_RS) {
    Ld::store(A.dst[c], ci, out);
  } else {
    for (int r = 0; r < N; ++r) Ld::store(A.dst[r], i, out);
  }
}

template <int DT, int OP, int MODE, int MAXN, bool VEC>
__device__ __forceinline__ void reduce_range(const ReduceArgs& A, uint64_t t0, uint64_t nt, uint64_t items,
                                             uint64_t Litems) {
  if (t0 >= items) return;
  int c = (int)(t0 / Litems);
  uint64_t cbeg = (uint64_t)c * Litems, cend = cbeg + Litems;
  for (uint64_t i = t0; i < items; i += nt) {
    while (i >= cend) {
      ++c;
      cbeg = cend;
      cend += Litems;
    }
    reduce_item<DT, OP, MODE, MAXN, VEC>(A, i, c, i - cbeg);
  }
}

template <int DT, int OP, int MODE, int MAXN>
__global__ void __launch_bounds__(kThreads) k_reduce(const __grid_constant__ ReduceArgs A) {
  pdl_begin();
  const uint64_t t0 = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const uint64_t nt = (uint64_t)gridDim.x * blockDim.x;
  if (A.vec) {
    constexpr int V = 16 / Fmt<DT>::bytes;
    const uint64_t nvec = A.count / V;
    reduce_range<DT, OP, MODE, MAXN, true>(A, t0, nt, nvec, A.L / V);
    // the last few elements (count not a multiple of V) lie in the last chunk
    const uint64_t done = nvec * V;
    if (t0 < A.count - done) {
      const uint64_t e = done + t0;
      const int c = (int)(e / A.L);
      reduce_item<DT, OP, MODE, MAXN, false>(A, e, c, e - (uint64_t)c * A.L);
    }
  } else {
    reduce_range<DT, OP, MODE, MAXN, false>(A, t0, nt, A.count, A.L);
  }
}

template <int DT, int OP, int MODE, int MAXN>
cudaError_t launch_reduce_n(const ReduceArgs& a, cudaStream_t stream) {
  const uint64_t items = a.vec ? a.count / (16 / Fmt<DT>::bytes) : a.count;
  return launch_pdl(k_reduce<DT, OP, MODE, MAXN>, dim3(grid_for(items > 0 ? items : a.count)), 0, stream, a);
}

template <int DT, int OP, int MODE>
cudaError_t launch_reduce_t(const ReduceArgs& a, cudaStream_t stream) {
  return a.nranks <= 8 ? launch_reduce_n<DT, OP, MODE, 8>(a, stream) : launch_reduce_n<DT, OP, MODE, kMaxRanks>(a, stream);
}

template <int DT>
cudaError_t launch_reduce_dt(int op, int mode, const ReduceArgs& a, cudaStream_t stream) {
#define GAR_MODES(OPV)                                                                   \
  switch (mode) {                                                                        \
    case MODE_RS: return launch_reduce_t<DT, OPV, MODE_RS>(a, stream);                   \
    case MODE_FUSED_RING: return launch_reduce_t<DT, OPV, MODE_FUSED_RING>(a, stream);   \
    case MODE_FUSED_TREE: return launch_reduce_t<DT, OPV, MODE_FUSED_TREE>(a, stream);   \
    default: return cudaErrorInvalidValue;                                               \
  }
  switch (op) {
    case OP_SUM: GAR_MODES(OP_SUM)
    case OP_AVG: GAR_MODES(OP_AVG)
    case OP_MIN: GAR_MODES(OP_MIN)
    case OP_MAX: GAR_MODES(OP_MAX)
    default: return cudaErrorInvalidValue;
  }
#undef GAR_MODES
}

}  // namespace gar
