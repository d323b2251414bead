// ar_fp8_fused_impl.cuh — FP8-compressed allreduce with the quantisation fused into
// the reduction (sm_103a).
//
// Same numbers as the materialised path (ar_fp8.cu): each rank's 128-element
// blocks are quantised once (amax, s = amax/448, q = E4M3(x/s)), dequantised
// (float(q)*s) and folded in binary32 in ring or tree order. Here the codes
// never leave registers: a lane group loads a rank's block, finds its amax by
// shuffles, quantises, dequantises and accumulates, rank after rank; the
// result is written once to every rank. On one device this moves 2*N*M bytes
// instead of the materialised path's 2*N*M + 2*N*(M/2 + M/64): the wire
// format is what a multi-device ring would exchange, and its rounding is kept
// exactly.
//
//  k_fp8_fused_vec   16-byte loads, one lane group per block (16 lanes for
//                    bf16/fp16, 32 for fp32); a warp whose elements all lie in
//                    one ring chunk shares one start rank, so the fold needs no
//                    per-rank storage. Warps that straddle a chunk boundary are
//                    left to the element-wise kernel.
//  k_fp8_fused_elem  one warp per block, elements lane + 32k: every rank's
//                    dequantised values first, then each element folded in its
//                    own chunk's order (straddling warps, the short last block,
//                    unaligned buffers).
#pragma once

#include <cstdint>

#include "ar_fp8_common.cuh"

namespace gar {

// Loader for the fold: a rank's "value" is its dequantised block slice, which
// needs the block's amax, so unpack() shuffles across the lane group; Fold
// calls it for every rank in the same (warp-uniform) order.
template <int IDT> struct Fp8FusedLd {
  static constexpr int B = Fmt<IDT>::bytes;
  static constexpr int V = 16 / B;
  static constexpr int G = kFp8Block / V;
  static constexpr bool kPairAdd = true;  // comb is a binary32 add: pairs may use the packed add
  using Acc = float;
  using Raw = uint4;

  const Fp8FusedArgs& A;
  uint64_t e0;  // lane's first element
  bool valid;

  __device__ __forceinline__ Raw load(int r) const {
    return valid ? __ldcs(reinterpret_cast<const uint4*>(static_cast<const char*>(A.src[r]) + e0 * B))
                 : make_uint4(0, 0, 0, 0);
  }
  __device__ __forceinline__ void unpack(const Raw& raw, Acc (&d)[V]) const {
    float x[V];
    float amax = 0.0f;
#pragma unroll
    for (int k = 0; k < V; ++k) {
      x[k] = to_f32<IDT>(get_lane<B>(raw, k));
      amax = fmaxf(amax, fabsf(x[k]));
    }
    amax = group_amax<G>(amax);
    const float s = scale_of(amax);
    qdq_lane<V>(x, amax, s, d);
  }
  __device__ __forceinline__ static Acc comb(Acc a, Acc b) { return __fadd_rn(a, b); }
};

template <int IDT, int ODT, int OP, int MODE, int MAXN>
__global__ void __launch_bounds__(kThreads, MODE == MODE_FUSED_TREE ? 1 : 4) k_fp8_fused_vec(const __grid_constant__ Fp8FusedArgs A) {
  using Ld = Fp8FusedLd<IDT>;
  constexpr int V = Ld::V, G = Ld::G, BPW = 32 / G, OB = Fmt<ODT>::bytes;
  const int N = A.nranks;
  const uint64_t nfull = A.count / kFp8Block;
  const uint64_t warp = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31, g = lane / G, gl = lane % G;
  const uint64_t wb0 = warp * BPW;
  if (wb0 >= nfull) return;  // warp-uniform
  const uint64_t wb1 = (wb0 + BPW < nfull) ? wb0 + BPW : nfull;
  const uint64_t b = wb0 + (uint64_t)g;
  const Ld ld{A, b * kFp8Block + (uint64_t)gl * V, b < nfull};
  float acc[V];
  if constexpr (MODE == MODE_FUSED_TREE) {
    Fold<Ld>::template tree<MAXN>(ld, N, acc);
  } else {
    const uint64_t c_lo = (wb0 * kFp8Block) / A.L, c_hi = (wb1 * kFp8Block - 1) / A.L;
    if (c_lo != c_hi) return;  // straddles a chunk boundary: the element-wise kernel's
    const int s = ((int)c_lo + 1 == N) ? 0 : (int)c_lo + 1;
    Fold<Ld>::template ring<MAXN>(ld, N, s, acc);
  }
  if (!ld.valid) return;
  uint32_t bits[V];
#pragma unroll
  for (int k = 0; k < V; ++k) bits[k] = from_f32<ODT>(OP == OP_AVG ? __fdiv_rn(acc[k], (float)N) : acc[k]);
  if constexpr (V * OB == 16) {
    uint4 out = make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int k = 0; k < V; ++k) set_lane<OB>(out, k, bits[k]);
    for (int r = 0; r < N; ++r) __stcs(reinterpret_cast<uint4*>(static_cast<char*>(A.dst[r]) + ld.e0 * OB), out);
  } else {  // 4 fp32 inputs -> 4 x 16-bit outputs
    const uint2 out = make_uint2((bits[0] & 0xFFFFu) | (bits[1] << 16), (bits[2] & 0xFFFFu) | (bits[3] << 16));
    for (int r = 0; r < N; ++r) __stcs(reinterpret_cast<uint2*>(static_cast<char*>(A.dst[r]) + ld.e0 * OB), out);
  }
}

template <int IDT, int ODT, int OP, int MODE, int MAXN>
__global__ void __launch_bounds__(kThreads) k_fp8_fused_elem(const __grid_constant__ Fp8FusedArgs A) {
  constexpr int IB = Fmt<IDT>::bytes, OB = Fmt<ODT>::bytes;
  const int N = A.nranks;
  const uint64_t nblocks = (A.count + kFp8Block - 1) / kFp8Block;
  const uint64_t tasks = (uint64_t)A.nlist + (nblocks - A.first_block);
  const int lane = threadIdx.x & 31;
  const uint64_t warp0 = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const uint64_t nwarps = ((uint64_t)gridDim.x * blockDim.x) >> 5;
  for (uint64_t w = warp0; w < tasks; w += nwarps) {  // warp-uniform
    const uint64_t b = (w < (uint64_t)A.nlist) ? A.list[w] : A.first_block + (w - A.nlist);
    const uint64_t lo = b * kFp8Block;
    float d[MAXN][4];
    for (int r = 0; r < N; ++r) {
      const char* src = static_cast<const char*>(A.src[r]);
      float x[4];
      float amax = 0.0f;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint64_t e = lo + lane + 32 * k;
        uint32_t bits = 0;
        if (e < A.count) {
          if constexpr (IB == 4) bits = *reinterpret_cast<const uint32_t*>(src + e * 4);
          else bits = *reinterpret_cast<const uint16_t*>(src + e * 2);
        }
        x[k] = to_f32<IDT>(bits);
        amax = fmaxf(amax, fabsf(x[k]));
      }
      amax = group_amax<32>(amax);
      const float s = scale_of(amax);
      float t[4];
      qdq_lane<4>(x, amax, s, t);
#pragma unroll
      for (int k = 0; k < 4; ++k) d[r][k] = t[k];
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint64_t e = lo + lane + 32 * k;
      if (e >= A.count) continue;
      float acc;
      if constexpr (MODE == MODE_FUSED_TREE) {
        float v[MAXN];
        for (int r = 0; r < N; ++r) v[r] = d[r][k];
        for (int dd = N / 2; dd >= 1; dd >>= 1)
          for (int r = 0; r < dd; ++r) v[r] = __fadd_rn(v[r], v[r + dd]);
        acc = v[0];
      } else {
        const int c = (int)(e / A.L);
        int r = (c + 1 == N) ? 0 : c + 1;
        acc = d[r][k];
        for (int j = 1; j < N; ++j) {
          r = (r + 1 == N) ? 0 : r + 1;
          acc = __fadd_rn(acc, d[r][k]);
        }
      }
      const uint32_t out = from_f32<ODT>(OP == OP_AVG ? __fdiv_rn(acc, (float)N) : acc);
      for (int r = 0; r < N; ++r) {
        char* p = static_cast<char*>(A.dst[r]);
        if constexpr (OB == 4) *reinterpret_cast<uint32_t*>(p + e * 4) = out;
        else *reinterpret_cast<uint16_t*>(p + e * 2) = (uint16_t)out;
      }
    }
  }
}

template <int IDT, int ODT, int OP, int MODE, int MAXN>
cudaError_t launch_fused_n(bool vec, const Fp8FusedArgs& a, cudaStream_t stream) {
  constexpr int V = 16 / Fmt<IDT>::bytes, BPW = 32 / (kFp8Block / V);
  if (vec) {
    const uint64_t nfull = a.count / kFp8Block;
    if (nfull > 0) {
      const uint64_t warps = (nfull + BPW - 1) / BPW;
      k_fp8_fused_vec<IDT, ODT, OP, MODE, MAXN><<<grid_for(warps * 32), kThreads, 0, stream>>>(a);
      const cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
  }
  const uint64_t nblocks = (a.count + kFp8Block - 1) / kFp8Block;
  const uint64_t tasks = (uint64_t)a.nlist + (nblocks - a.first_block);
  if (tasks == 0) return cudaSuccess;
  k_fp8_fused_elem<IDT, ODT, OP, MODE, MAXN><<<grid_for(tasks * 32), kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

template <int IDT, int ODT, int OP>
cudaError_t launch_fused_op(int mode, bool vec, const Fp8FusedArgs& a, cudaStream_t s) {
  const int tier = a.nranks <= 8 ? 0 : (a.nranks <= 16 ? 1 : 2);
#define GAR_FT(MODEV)                                                                  \
  return tier == 0 ? launch_fused_n<IDT, ODT, OP, MODEV, 8>(vec, a, s)                 \
       : tier == 1 ? launch_fused_n<IDT, ODT, OP, MODEV, 16>(vec, a, s)                \
                   : launch_fused_n<IDT, ODT, OP, MODEV, kMaxRanks>(vec, a, s);
  if (mode == MODE_FUSED_TREE) { GAR_FT(MODE_FUSED_TREE) }
  GAR_FT(MODE_FUSED_RING)
#undef GAR_FT
}

template <int IDT, int ODT>
cudaError_t launch_fused_io(int op, int mode, bool vec, const Fp8FusedArgs& a, cudaStream_t s) {
  if (op == OP_AVG) return launch_fused_op<IDT, ODT, OP_AVG>(mode, vec, a, s);
  if (op == OP_SUM) return launch_fused_op<IDT, ODT, OP_SUM>(mode, vec, a, s);
  return cudaErrorInvalidValue;
}

}  // namespace gar
