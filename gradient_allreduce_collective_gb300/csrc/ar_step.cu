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
  pdl_begin();
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
  return launch_pdl(k_step_combine<DT, OP>, dim3(total), 0, s, a);  // one block per tile
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

// ---------------------------------------------------------------- 16-bit types
//
// The same step for bf16 and fp16 with binary32 partials, so that the
// stepwise orders round once, at the end, exactly as the one-pass kernels:
// operand a (b) is a 16-bit input or, when A32 (B32), a partial word (the
// binary32 sum for SUM/AVG, the selected element's bits for MIN/MAX); the
// result is a partial word or, when FIN, the finished 16-bit value. An item
// is 4 consecutive elements (8 bytes of 16-bit values, 16 bytes of partials).

template <int DT, int OP>
__device__ __forceinline__ typename Red<DT, OP>::Acc acc_of_partial(uint32_t w) {
  if constexpr (std::is_same_v<typename Red<DT, OP>::Acc, float>) return __uint_as_float(w);
  else return w;
}

template <int DT, int OP, bool WIDE>
__device__ __forceinline__ void load4(const void* base, uint64_t item, typename Red<DT, OP>::Acc (&v)[4]) {
  using R = Red<DT, OP>;
  if constexpr (WIDE) {
    const uint4 w = __ldcs(reinterpret_cast<const uint4*>(base) + item);
    v[0] = acc_of_partial<DT, OP>(w.x);
    v[1] = acc_of_partial<DT, OP>(w.y);
    v[2] = acc_of_partial<DT, OP>(w.z);
    v[3] = acc_of_partial<DT, OP>(w.w);
  } else {
    const uint2 w = __ldcs(reinterpret_cast<const uint2*>(base) + item);
    v[0] = R::init(w.x & 0xFFFFu);
    v[1] = R::init(w.x >> 16);
    v[2] = R::init(w.y & 0xFFFFu);
    v[3] = R::init(w.y >> 16);
  }
}

template <int DT, int OP, bool WIDE>
__device__ __forceinline__ typename Red<DT, OP>::Acc load1(const void* base, uint64_t e) {
  if constexpr (WIDE) return acc_of_partial<DT, OP>(reinterpret_cast<const uint32_t*>(base)[e]);
  else return Red<DT, OP>::init(reinterpret_cast<const uint16_t*>(base)[e]);
}

template <int DT, int OP, bool A32, bool B32, bool FIN>
__global__ void __launch_bounds__(kThreads) k_step_combine16(const __grid_constant__ StepArgs A) {
  pdl_begin();
  using R = Red<DT, OP>;
  using Acc = typename R::Acc;
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
    const uint64_t e0 = item * 4;
    if (e0 >= len) continue;
    if (A.vec && e0 + 4 <= len) {
      Acc x[4], y[4];
      load4<DT, OP, A32>(A.a[t], item, x);
      load4<DT, OP, B32>(A.b[t], item, y);
      uint32_t o[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const Acc v = R::comb(x[k], y[k]);
        o[k] = FIN ? R::fin(v, A.nranks) : partial_bits(v);
      }
      if constexpr (FIN)
        __stcs(reinterpret_cast<uint2*>(A.dst[t]) + item, make_uint2(o[0] | (o[1] << 16), o[2] | (o[3] << 16)));
      else
        __stcs(reinterpret_cast<uint4*>(A.dst[t]) + item, make_uint4(o[0], o[1], o[2], o[3]));
    } else {
      const uint64_t e1 = e0 + 4 < len ? e0 + 4 : len;
      for (uint64_t e = e0; e < e1; ++e) {
        const Acc v = R::comb(load1<DT, OP, A32>(A.a[t], e), load1<DT, OP, B32>(A.b[t], e));
        if constexpr (FIN) reinterpret_cast<uint16_t*>(A.dst[t])[e] = (uint16_t)R::fin(v, A.nranks);
        else reinterpret_cast<uint32_t*>(A.dst[t])[e] = partial_bits(v);
      }
    }
  }
}

template <int DT, int OP, bool A32, bool B32>
cudaError_t launch_step16_ab(bool fin, const StepArgs& a, cudaStream_t s) {
  const uint32_t total = a.tile_start[a.ntasks];
  if (total == 0) return cudaSuccess;
  return fin ? launch_pdl(k_step_combine16<DT, OP, A32, B32, true>, dim3(total), 0, s, a)
             : launch_pdl(k_step_combine16<DT, OP, A32, B32, false>, dim3(total), 0, s, a);
}

template <int DT, int OP>
cudaError_t launch_step16_op(bool a32, bool b32, bool fin, const StepArgs& a, cudaStream_t s) {
  if (a32) return b32 ? launch_step16_ab<DT, OP, true, true>(fin, a, s) : launch_step16_ab<DT, OP, true, false>(fin, a, s);
  return b32 ? launch_step16_ab<DT, OP, false, true>(fin, a, s) : launch_step16_ab<DT, OP, false, false>(fin, a, s);
}

template <int DT>
cudaError_t launch_step16_dt(int op, bool a32, bool b32, bool fin, const StepArgs& a, cudaStream_t s) {
  switch (op) {
    case OP_SUM: return launch_step16_op<DT, OP_SUM>(a32, b32, fin, a, s);
    case OP_AVG: return launch_step16_op<DT, OP_AVG>(a32, b32, fin, a, s);
    case OP_MIN: return launch_step16_op<DT, OP_MIN>(a32, b32, fin, a, s);
    case OP_MAX: return launch_step16_op<DT, OP_MAX>(a32, b32, fin, a, s);
    default: return cudaErrorInvalidValue;
  }
}

// items: tile_start counts tiles of kThreads items of 4 elements each
cudaError_t launch_step_combine16(int dtype, int op, bool a32, bool b32, const StepArgs& a, cudaStream_t stream) {
  switch (dtype) {
    case DT_BF16: return launch_step16_dt<DT_BF16>(op, a32, b32, a.finish != 0, a, stream);
    case DT_F16: return launch_step16_dt<DT_F16>(op, a32, b32, a.finish != 0, a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gar
