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
//  k_fp8_fused_pair  ring order, bf16/fp16 inputs: a warp per two blocks,
//                    lane l holding elements 4l..4l+3 of each; block amax by a
//                    warp max-reduction; every rank's pair quantised on the
//                    call-free division-free path (the general path redoes a
//                    warp whose scales leave its range), so that successive
//                    ranks' quantisations overlap.
//  k_fp8_fused_vec   16-byte loads, one lane group per block (16 lanes for
//                    bf16/fp16, 32 for fp32); the tree order, and fp32 inputs.
//                    In both vector kernels a warp whose elements all lie in
//                    one ring chunk shares one start rank, so the fold needs no
//                    per-rank storage; warps that straddle a chunk boundary
//                    are left to the element-wise kernel.
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
      amax = fmax_nan(amax, fabsf(x[k]));
    }
    amax = group_amax<G>(amax);
    const float s = scale_of(amax);
    qdq_lane<V>(x, amax, s, d);
  }
  __device__ __forceinline__ static Acc comb(Acc a, Acc b) { return __fadd_rn(a, b); }
};

template <int IDT, int ODT, int OP, int MODE, int MAXN>
__global__ void __launch_bounds__(kThreads, MODE == MODE_FUSED_TREE ? 1 : 4) k_fp8_fused_vec(const __grid_constant__ Fp8FusedArgs A) {
  pdl_begin();
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
  for (int k = 0; k < V; ++k) bits[k] = from_f32<ODT>(OP == OP_AVG ? avg_div(acc[k], N) : acc[k]);
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

// Ring order, 16-bit inputs: the same two blocks per warp as
// k_fp8_fused_vec, laid out as in the per-hop kernel: lane l holds elements
// 4l..4l+3 of each block, each block's amax is one warp max-reduction, and
// every rank's two blocks are quantised on the division-free path with no
// branch or call, so that the quantisations of successive ranks (independent
// of the running sum) overlap. If some block's scale lies outside
// [2^-90, 2^90] the warp folds its blocks again on the general path.
template <int IDT>
__device__ __forceinline__ void fused_pair_load(const Fp8FusedArgs& A, int r, uint64_t ea, bool vb, uint2& a,
                                                uint2& b) {
  const uint16_t* src = static_cast<const uint16_t*>(A.src[r]);
  a = __ldcs(reinterpret_cast<const uint2*>(src + ea));
  b = vb ? __ldcs(reinterpret_cast<const uint2*>(src + ea + kFp8Block)) : make_uint2(0, 0);
}

template <int IDT>
__device__ __forceinline__ void unpack4x16(uint2 v, float (&x)[4]) {
  x[0] = to_f32<IDT>(v.x & 0xFFFFu);
  x[1] = to_f32<IDT>(v.x >> 16);
  x[2] = to_f32<IDT>(v.y & 0xFFFFu);
  x[3] = to_f32<IDT>(v.y >> 16);
}

// dequantised values of one rank's two blocks; FAST: the division-free path,
// returning false if a scale is outside its range
template <bool FAST>
__device__ __forceinline__ bool qdq_two(const float (&xa)[4], const float (&xb)[4], float (&da)[4],
                                        float (&db)[4]) {
  float ma = 0.0f, mb = 0.0f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    ma = fmax_nan(ma, fabsf(xa[k]));
    mb = fmax_nan(mb, fabsf(xb[k]));
  }
  ma = group_amax<32>(ma);
  mb = group_amax<32>(mb);
  if constexpr (FAST) {
    const float sa = scale_fast(ma), sb = scale_fast(mb);
    qdq_fast_z<4>(xa, ma, sa, da);
    qdq_fast_z<4>(xb, mb, sb, db);
    return (ma == 0.0f || scale_in_range(sa)) && (mb == 0.0f || scale_in_range(sb));
  } else {
    qdq_lane<4>(xa, ma, scale_of(ma), da);
    qdq_lane<4>(xb, mb, scale_of(mb), db);
    return true;
  }
}

// ring-order fold of every rank's dequantised pair of blocks, starting at
// rank s; ranks loaded eight at a time before they are folded
template <int IDT, int MAXN, bool FAST>
__device__ __forceinline__ bool fused_pair_ring(const Fp8FusedArgs& A, uint64_t ea, bool vb, int s,
                                                float (&pa)[4], float (&pb)[4]) {
  const int N = A.nranks;
  bool ok = true;
#pragma unroll 1
  for (int b0 = 0; b0 < MAXN; b0 += 8) {
    if (b0 >= N) break;
    uint2 ra[8], rb[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      if (b0 + m < N) {
        int r = s + b0 + m;
        r = (r >= N) ? r - N : r;
        fused_pair_load<IDT>(A, r, ea, vb, ra[m], rb[m]);
      }
    }
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      if (b0 + m < N) {
        float xa[4], xb[4], da[4], db[4];
        unpack4x16<IDT>(ra[m], xa);
        unpack4x16<IDT>(rb[m], xb);
        if (FAST) ok &= qdq_two<true>(xa, xb, da, db);
        else qdq_two<false>(xa, xb, da, db);
        if (b0 + m == 0) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            pa[k] = da[k];
            pb[k] = db[k];
          }
        } else {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            pa[k] = __fadd_rn(pa[k], da[k]);
            pb[k] = __fadd_rn(pb[k], db[k]);
          }
        }
      }
    }
  }
  return ok;
}

template <int IDT, int MAXN>
static __device__ __noinline__ void fused_pair_ring_general(const Fp8FusedArgs& A, uint64_t ea, bool vb, int s,
                                                            float (&pa)[4], float (&pb)[4]) {
  fused_pair_ring<IDT, MAXN, false>(A, ea, vb, s, pa, pb);
}

constexpr int kFusedPairBlocksPerSm = 3;

template <int IDT, int ODT, int OP, int MAXN>
__global__ void __launch_bounds__(kThreads, kFusedPairBlocksPerSm) k_fp8_fused_pair(const __grid_constant__ Fp8FusedArgs A) {
  pdl_begin();
  static_assert(Fmt<IDT>::bytes == 2, "16-bit inputs");
  const int N = A.nranks;
  const uint64_t nfull = A.count / kFp8Block;
  const uint64_t warp = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t wb0 = warp * 2;
  if (wb0 >= nfull) return;  // warp-uniform
  const uint64_t wb1 = (wb0 + 2 < nfull) ? wb0 + 2 : nfull;
  const uint64_t c_lo = (wb0 * kFp8Block) / A.L, c_hi = (wb1 * kFp8Block - 1) / A.L;
  if (c_lo != c_hi) return;  // straddles a chunk boundary: the element-wise kernel's
  const int s = ((int)c_lo + 1 == N) ? 0 : (int)c_lo + 1;
  const bool vb = wb0 + 1 < nfull;  // the second block is whole
  const uint64_t ea = wb0 * kFp8Block + 4 * lane;
  float pa[4], pb[4];
  if (!fused_pair_ring<IDT, MAXN, true>(A, ea, vb, s, pa, pb)) fused_pair_ring_general<IDT, MAXN>(A, ea, vb, s, pa, pb);
  uint32_t ba[4], bb[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    ba[k] = from_f32<ODT>(OP == OP_AVG ? avg_div(pa[k], N) : pa[k]);
    bb[k] = from_f32<ODT>(OP == OP_AVG ? avg_div(pb[k], N) : pb[k]);
  }
  for (int r = 0; r < N; ++r) {
    char* dst = static_cast<char*>(A.dst[r]);
    if constexpr (Fmt<ODT>::bytes == 4) {
      __stcs(reinterpret_cast<uint4*>(dst + ea * 4), make_uint4(ba[0], ba[1], ba[2], ba[3]));
      if (vb) __stcs(reinterpret_cast<uint4*>(dst + (ea + kFp8Block) * 4), make_uint4(bb[0], bb[1], bb[2], bb[3]));
    } else {
      __stcs(reinterpret_cast<uint2*>(dst + ea * 2), make_uint2(ba[0] | (ba[1] << 16), ba[2] | (ba[3] << 16)));
      if (vb) __stcs(reinterpret_cast<uint2*>(dst + (ea + kFp8Block) * 2), make_uint2(bb[0] | (bb[1] << 16), bb[2] | (bb[3] << 16)));
    }
  }
}

template <int IDT, int ODT, int OP, int MODE, int MAXN>
__global__ void __launch_bounds__(kThreads) k_fp8_fused_elem(const __grid_constant__ Fp8FusedArgs A) {
  pdl_begin();
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
        amax = fmax_nan(amax, fabsf(x[k]));
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
      const uint32_t out = from_f32<ODT>(OP == OP_AVG ? avg_div(acc, N) : acc);
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
      cudaError_t e;
      if constexpr (MODE == MODE_FUSED_RING && Fmt<IDT>::bytes == 2)
        e = launch_pdl(k_fp8_fused_pair<IDT, ODT, OP, MAXN>, dim3(grid_for(warps * 32)), 0, stream, a);
      else
        e = launch_pdl(k_fp8_fused_vec<IDT, ODT, OP, MODE, MAXN>, dim3(grid_for(warps * 32)), 0, stream, a);
      if (e != cudaSuccess) return e;
    }
  }
  const uint64_t nblocks = (a.count + kFp8Block - 1) / kFp8Block;
  const uint64_t tasks = (uint64_t)a.nlist + (nblocks - a.first_block);
  if (tasks == 0) return cudaSuccess;
  return launch_pdl(k_fp8_fused_elem<IDT, ODT, OP, MODE, MAXN>, dim3(grid_for(tasks * 32)), 0, stream, a);
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
