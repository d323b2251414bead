// ar_fp8.cu — FP8 (E4M3) gradient compression for the allreduce (sm_103a).
//
// FP8 on the wire halves the bytes of FP16 ("AllReduce（オールリデュース）"
// glossary, §NCCLにおけるAllReduce and §勾配圧縮技術) at the cost of quantise /
// dequantise work and a scale exchange ("All-Reduce・All-Gather・All-to-All
// とは？" vasteelab, §data typeと圧縮は品質だけの問題ではない). Each rank is
// quantised once, before the reduction, per block of 128 consecutive
// elements: amax = max|x| (binary32), s = amax / 448, q = E4M3(x / s) with
// round-to-nearest-even and saturation; amax = 0 gives s = 0, q = 0.
//
//  k_fp8_quant_vec     one group of 128/V lanes per block (16 lanes of 8 bf16
//                      or fp16, 32 lanes of 4 fp32): 16-byte loads, amax by
//                      xor shuffles inside the group, V code bytes per lane.
//  k_fp8_quant_scalar  one warp per block, for a short last block or inputs
//                      that are not 16-byte aligned.
//  k_fp8_reduce        dequantise float(q) * s (one binary32 multiply),
//                      fold in ring or tree order in binary32, SUM or AVG,
//                      round once to the output type, store to the chunk
//                      owner or to all N outputs.
#include <cstdint>

#include "ar_fp8_common.cuh"

namespace gar {

// Blocks handled by one lane group per launch row: every lane issues the loads
// of kQuantUnroll blocks before any arithmetic, so 8 x 16 bytes are in flight
// (2.120 against 2.150 ms per materialised step with 4 on GB300).
constexpr int kQuantUnroll = 8;

template <int DT>
__device__ __forceinline__ void fp8_quant_vec_body(const Fp8QuantArgs& A) {
  pdl_begin();
  constexpr int B = Fmt<DT>::bytes, V = 16 / B, G = kFp8Block / V, BPW = 32 / G;
  const int r = blockIdx.y;
  const uint64_t nfull = A.count / kFp8Block;
  const int lane = threadIdx.x & 31, g = lane / G, gl = lane % G;
  const uint64_t warp = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const uint64_t b0 = warp * (uint64_t)(kQuantUnroll * BPW);
  if (b0 >= nfull) return;  // warp-uniform
  const char* src = static_cast<const char*>(A.src[r]);
  uint4 raw[kQuantUnroll];
#pragma unroll
  for (int u = 0; u < kQuantUnroll; ++u) {
    const uint64_t b = b0 + (uint64_t)(u * BPW + g);
    raw[u] = (b < nfull) ? __ldcs(reinterpret_cast<const uint4*>(src + (b * kFp8Block + (uint64_t)gl * V) * B))
                         : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int u = 0; u < kQuantUnroll; ++u) {
    const uint64_t b = b0 + (uint64_t)(u * BPW + g);
    float x[V];
    float amax = 0.0f;
#pragma unroll
    for (int k = 0; k < V; ++k) {
      x[k] = to_f32<DT>(get_lane<B>(raw[u], k));
      amax = fmax_nan(amax, fabsf(x[k]));
    }
    amax = group_amax<G>(amax);
    const float s = scale_of(amax);
    uint32_t word[V / 4];
    quantise_lane<V>(x, amax, s, word);
    if (b < nfull) {
      uint8_t* qp = A.q[r] + b * kFp8Block + (uint64_t)gl * V;
      if constexpr (V == 8) __stcs(reinterpret_cast<uint2*>(qp), make_uint2(word[0], word[1]));
      else __stcs(reinterpret_cast<unsigned int*>(qp), word[0]);
      if (gl == 0) A.s[r][b] = s;
    }
  }
}

template <int DT>
__global__ void __launch_bounds__(kThreads) k_fp8_quant_vec(const __grid_constant__ Fp8QuantArgs A) {
  fp8_quant_vec_body<DT>(A);
}

// 16-bit inputs at 5 resident blocks per SM (48 registers, a 16-byte spill,
// against 4 blocks at 63): materialised step 2.013 -> 1.987 ms. The binary32
// input kernel already fits 5 blocks at 49 registers and keeps k_fp8_quant_vec.
template <int DT>
__global__ void __launch_bounds__(kThreads, 5) k_fp8_quant_vec16(const __grid_constant__ Fp8QuantArgs A) {
  fp8_quant_vec_body<DT>(A);
}

template <int DT>
__global__ void __launch_bounds__(kThreads) k_fp8_quant_scalar(const __grid_constant__ Fp8QuantArgs A) {
  pdl_begin();
  constexpr int B = Fmt<DT>::bytes;
  const uint64_t nblocks = (A.count + kFp8Block - 1) / kFp8Block;
  const uint64_t nb = nblocks - A.first_block;
  const uint64_t tasks = (uint64_t)A.nranks * nb;
  const int lane = threadIdx.x & 31;
  const uint64_t warp0 = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const uint64_t nwarps = ((uint64_t)gridDim.x * blockDim.x) >> 5;
  for (uint64_t w = warp0; w < tasks; w += nwarps) {
    const int r = (int)(w / nb);
    const uint64_t b = A.first_block + (w - (uint64_t)r * nb);
    const uint64_t lo = b * kFp8Block;
    const char* src = static_cast<const char*>(A.src[r]);
    float x[4];
    float amax = 0.0f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint64_t e = lo + lane + 32 * k;
      uint32_t bits = 0;
      if (e < A.count) {
        if constexpr (B == 4) bits = *reinterpret_cast<const uint32_t*>(src + e * 4);
        else bits = *reinterpret_cast<const uint16_t*>(src + e * 2);
      }
      x[k] = to_f32<DT>(bits);
      amax = fmax_nan(amax, fabsf(x[k]));
    }
    amax = group_amax<32>(amax);
    const float s = scale_of(amax);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint64_t e = lo + lane + 32 * k;
      if (e < A.count) A.q[r][e] = (uint8_t)((amax == 0.0f) ? 0u : f32_to_e4m3(__fdiv_rn(x[k], s)));
    }
    if (lane == 0) A.s[r][b] = s;
  }
}

template <int DT> cudaError_t launch_fp8_quant_dt(bool vec, const Fp8QuantArgs& a, cudaStream_t stream) {
  constexpr int BPW = 32 / (kFp8Block / (16 / Fmt<DT>::bytes));
  const uint64_t nblocks = (a.count + kFp8Block - 1) / kFp8Block;
  Fp8QuantArgs b = a;
  if (vec) {
    const uint64_t nfull = a.count / kFp8Block;
    if (nfull > 0) {
      const uint64_t warps = (nfull + kQuantUnroll * BPW - 1) / (kQuantUnroll * BPW);
      const dim3 grid(grid_for(warps * 32), (unsigned)a.nranks);
      const cudaError_t e = Fmt<DT>::bytes == 2 ? launch_pdl(k_fp8_quant_vec16<DT>, grid, 0, stream, a)
                                                : launch_pdl(k_fp8_quant_vec<DT>, grid, 0, stream, a);
      if (e != cudaSuccess) return e;
    }
    b.first_block = nfull;
  } else {
    b.first_block = 0;
  }
  if (b.first_block < nblocks) {
    const uint64_t warps = (uint64_t)a.nranks * (nblocks - b.first_block);
    return launch_pdl(k_fp8_quant_scalar<DT>, dim3(grid_for(warps * 32)), 0, stream, b);
  }
  return cudaSuccess;
}

cudaError_t launch_fp8_quant(int in_dtype, bool vec, const Fp8QuantArgs& a, cudaStream_t stream) {
  switch (in_dtype) {
    case DT_F32: return launch_fp8_quant_dt<DT_F32>(vec, a, stream);
    case DT_F16: return launch_fp8_quant_dt<DT_F16>(vec, a, stream);
    case DT_BF16: return launch_fp8_quant_dt<DT_BF16>(vec, a, stream);
    default: return cudaErrorInvalidValue;
  }
}

// ---------------------------------------------------------------- dequantise + reduce

template <int VV> struct Fp8Ld {
  static constexpr int V = VV;
  // every rank's codes and scale (12 bytes each at V = 8) loaded before the
  // fold: one round trip for up to 16 ranks (2.165 against 2.239 ms per
  // materialised step of 16 x 134,217,728 bf16 with batches of 8 on GB300)
  static constexpr int kBatch = 16;
  static constexpr bool kPairAdd = true;  // comb is a binary32 add: pairs may use the packed add
  using Acc = float;
  struct Raw {
    uint32_t q[(V + 3) / 4];
    float s;
  };
  const Fp8ReduceArgs& A;
  uint64_t e0;  // first element of the item

  __device__ __forceinline__ Raw load(int r) const {
    Raw w;
    const uint8_t* qp = A.q[r] + e0;
    if constexpr (V == 8) {
      const uint2 t = __ldcs(reinterpret_cast<const uint2*>(qp));
      w.q[0] = t.x;
      w.q[1] = t.y;
    } else if constexpr (V == 4) {
      w.q[0] = __ldcs(reinterpret_cast<const unsigned int*>(qp));
    } else {
      w.q[0] = *qp;
    }
    w.s = __ldg(A.s[r] + (e0 / kFp8Block));
    return w;
  }
  __device__ __forceinline__ void unpack(const Raw& w, Acc (&a)[V]) const {
    dequantise_lane<V>(w.q, w.s, a);
  }
  __device__ __forceinline__ static Acc comb(Acc a, Acc b) { return __fadd_rn(a, b); }
};

template <int ODT, int OP, int MODE, int MAXN, bool VEC>
__device__ __forceinline__ void fp8_item(const Fp8ReduceArgs& A, uint64_t i, int c, uint64_t ci) {
  constexpr int B = Fmt<ODT>::bytes;
  constexpr int V = VEC ? 16 / B : 1;
  using Ld = Fp8Ld<V>;
  const int N = A.nranks;
  const Ld ld{A, i * V};
  float acc[V];
  if constexpr (MODE == MODE_FUSED_TREE) {
    Fold<Ld>::template tree<MAXN>(ld, N, acc);
  } else {
    const int s = (c + 1 == N) ? 0 : c + 1;
    Fold<Ld>::template ring<MAXN>(ld, N, s, acc);
  }
  uint32_t bits[V];
#pragma unroll
  for (int k = 0; k < V; ++k) bits[k] = from_f32<ODT>(OP == OP_AVG ? avg_div(acc[k], N) : acc[k]);
  if constexpr (VEC) {
    uint4 out = make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int k = 0; k < V; ++k) set_lane<B>(out, k, bits[k]);
    if constexpr (MODE == MODE_RS) {
      __stcs(reinterpret_cast<uint4*>(A.dst[c]) + ci, out);
    } else {
      for (int r = 0; r < N; ++r) __stcs(reinterpret_cast<uint4*>(A.dst[r]) + i, out);
    }
  } else {
    auto put = [&](void* base, uint64_t j) {
      if constexpr (B == 4) reinterpret_cast<uint32_t*>(base)[j] = bits[0];
      else reinterpret_cast<uint16_t*>(base)[j] = (uint16_t)bits[0];
    };
    if constexpr (MODE == MODE_RS) {
      put(A.dst[c], ci);
    } else {
      for (int r = 0; r < N; ++r) put(A.dst[r], i);
    }
  }
}

template <int ODT, int OP, int MODE, int MAXN, bool VEC>
__device__ __forceinline__ void fp8_range(const Fp8ReduceArgs& A, uint64_t t0, uint64_t nt, uint64_t items,
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
    fp8_item<ODT, OP, MODE, MAXN, VEC>(A, i, c, i - cbeg);
  }
}

template <int ODT, int OP, int MODE, int MAXN>
__device__ __forceinline__ void fp8_reduce_body(const Fp8ReduceArgs& A) {
  pdl_begin();
  const uint64_t t0 = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const uint64_t nt = (uint64_t)gridDim.x * blockDim.x;
  if (A.vec) {
    constexpr int V = 16 / Fmt<ODT>::bytes;
    const uint64_t items = A.count / V;
    fp8_range<ODT, OP, MODE, MAXN, true>(A, t0, nt, items, A.L / V);
    const uint64_t done = items * V;
    if (t0 < A.count - done) {
      const uint64_t e = done + t0;
      const int c = (int)(e / A.L);
      fp8_item<ODT, OP, MODE, MAXN, false>(A, e, c, e - (uint64_t)c * A.L);
    }
  } else {
    fp8_range<ODT, OP, MODE, MAXN, false>(A, t0, nt, A.count, A.L);
  }
}

template <int ODT, int OP, int MODE, int MAXN>
__global__ void __launch_bounds__(kThreads) k_fp8_reduce(const __grid_constant__ Fp8ReduceArgs A) {
  fp8_reduce_body<ODT, OP, MODE, MAXN>(A);
}

// The ring-order sum into a 16-bit output, up to 16 ranks, at 3 resident
// blocks per SM: it fits 80 registers (a 16-24 byte spill) and keeps more of
// its loads in flight than k_fp8_reduce's 2 blocks at 91 registers (measured
// 4-9 % faster at 4, 8 and 16 ranks). AVG and binary32 outputs spill more
// and measured 2-5 % slower this way, so they keep k_fp8_reduce.
template <int ODT, int OP, int MAXN>
__global__ void __launch_bounds__(kThreads, 3) k_fp8_reduce_sum16(const __grid_constant__ Fp8ReduceArgs A) {
  fp8_reduce_body<ODT, OP, MODE_FUSED_RING, MAXN>(A);
}

template <int ODT, int OP, int MODE, int MAXN>
cudaError_t launch_fp8_reduce_n(const Fp8ReduceArgs& a, cudaStream_t stream) {
  const uint64_t items = a.vec ? a.count / (16 / Fmt<ODT>::bytes) : a.count;
  const dim3 grid(grid_for(items > 0 ? items : a.count));
  if constexpr (MODE == MODE_FUSED_RING && MAXN <= 16 && OP != OP_AVG && Fmt<ODT>::bytes == 2)
    return launch_pdl(k_fp8_reduce_sum16<ODT, OP, MAXN>, grid, 0, stream, a);
  else
    return launch_pdl(k_fp8_reduce<ODT, OP, MODE, MAXN>, grid, 0, stream, a);
}

template <int ODT, int OP>
cudaError_t launch_fp8_reduce_op(int mode, const Fp8ReduceArgs& a, cudaStream_t stream) {
  // compile-time rank bound: 8, 16 (two batches of loads, unrolled) or 64
  const int tier = a.nranks <= 8 ? 0 : (a.nranks <= 16 ? 1 : 2);
#define GAR_TIERS(MODEV)                                                                          \
  return tier == 0 ? launch_fp8_reduce_n<ODT, OP, MODEV, 8>(a, stream)                          \
       : tier == 1 ? launch_fp8_reduce_n<ODT, OP, MODEV, 16>(a, stream)                         \
                   : launch_fp8_reduce_n<ODT, OP, MODEV, kMaxRanks>(a, stream);
  switch (mode) {
    case MODE_RS: GAR_TIERS(MODE_RS)
    case MODE_FUSED_RING: GAR_TIERS(MODE_FUSED_RING)
    case MODE_FUSED_TREE: GAR_TIERS(MODE_FUSED_TREE)
    default: return cudaErrorInvalidValue;
  }
#undef GAR_TIERS
}

template <int ODT> cudaError_t launch_fp8_reduce_dt(int op, int mode, const Fp8ReduceArgs& a, cudaStream_t s) {
  switch (op) {
    case OP_SUM: return launch_fp8_reduce_op<ODT, OP_SUM>(mode, a, s);
    case OP_AVG: return launch_fp8_reduce_op<ODT, OP_AVG>(mode, a, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_fp8_reduce(int out_dtype, int op, int mode, const Fp8ReduceArgs& a, cudaStream_t stream) {
  switch (out_dtype) {
    case DT_F32: return launch_fp8_reduce_dt<DT_F32>(op, mode, a, stream);
    case DT_F16: return launch_fp8_reduce_dt<DT_F16>(op, mode, a, stream);
    case DT_BF16: return launch_fp8_reduce_dt<DT_BF16>(op, mode, a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gar
