// ar_fp8_hop_impl.cuh — FP8 re-quantised on every hop of the ring (sm_103a).
//
// A ring that compresses its traffic sends each partial sum in FP8 ("AllReduce
// （オールリデュース）" glossary, §NCCLにおけるAllReduce: FP8 AllReduce; "All-
// Reduce・All-Gather・All-to-All とは？" vasteelab, §data typeと圧縮: reducing
// partial results at low precision changes the numerical error). Chunk c
// starts at rank c+1; at every hop the running partial of each 128-element
// block (counted from the chunk's start) is quantised (s = amax/448, E4M3
// nearest even, saturating), dequantised, and the next rank's value is added
// in binary32; the finished chunk is quantised once more for the all-gather
// and every rank stores the same dequantised values in the output type.
//
// One warp per pair of consecutive blocks of a chunk: lane l holds elements
// 4l..4l+3 of each when every buffer is aligned for 4-element vectors (one
// load and one store per rank, lane and block), and each hop quantises the
// two partials as two independent chains on the division-free path (the
// block amax a warp max-reduction, s = amax/448 by a multiply and a
// correction, RN(1/s) inline, the quotient by Markstein's steps), with no
// branch or call inside the fold, so that the scheduler interleaves them. A
// pair with a scale outside [2^-90, 2^90] on some hop is redone block by
// block on the general path, which also takes a chunk's odd or short last
// block and unaligned buffers (elements l, l+32, l+64, l+96 per lane). The
// ranks' values are loaded in batches of eight ranks (four for binary32
// inputs) before they are folded.
#pragma once

#include <cstdint>

#include "ar_fp8_common.cuh"

namespace gar {

// quantise-dequantise a warp's 128-element block held 4 values per lane
__device__ __forceinline__ void qdq_block(float (&p)[4]) {
  float amax = 0.0f;
#pragma unroll
  for (int k = 0; k < 4; ++k) amax = fmax_nan(amax, fabsf(p[k]));
  amax = group_amax<32>(amax);
  const float s = scale_of(amax);
  const float x[4] = {p[0], p[1], p[2], p[3]};
  qdq_lane<4>(x, amax, s, p);
}

// the same for two blocks at once, on the division-free path only: two
// independent chains without branches, so that the scheduler can interleave
// them. A block whose amax is 0 gives zeros as qdq_block does; false if a
// block's scale lies outside [2^-90, 2^90] (subnormal, huge or infinite
// amax), whose values are then meaningless and the caller redoes the pair on
// the general path.
__device__ __forceinline__ bool qdq_block_pair(float (&pa)[4], float (&pb)[4]) {
  float ma = 0.0f, mb = 0.0f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    ma = fmax_nan(ma, fabsf(pa[k]));
    mb = fmax_nan(mb, fabsf(pb[k]));
  }
  ma = group_amax<32>(ma);
  mb = group_amax<32>(mb);
  const float sa = scale_fast(ma), sb = scale_fast(mb);
  const float xa[4] = {pa[0], pa[1], pa[2], pa[3]}, xb[4] = {pb[0], pb[1], pb[2], pb[3]};
  qdq_fast_z<4>(xa, ma, sa, pa);
  qdq_fast_z<4>(xb, mb, sb, pb);
  return (ma == 0.0f || scale_in_range(sa)) && (mb == 0.0f || scale_in_range(sb));
}

// four consecutive elements starting at e (e a multiple of 4, base aligned)
template <int DT> struct Vec4 {
  using Raw = std::conditional_t<Fmt<DT>::bytes == 4, uint4, uint2>;
  static __device__ __forceinline__ Raw load(const void* base, uint64_t e) {
    return __ldcs(reinterpret_cast<const Raw*>(static_cast<const char*>(base) + e * Fmt<DT>::bytes));
  }
  static __device__ __forceinline__ void unpack(const Raw& v, float (&x)[4]) {
    if constexpr (Fmt<DT>::bytes == 4) {
      x[0] = to_f32<DT>(v.x);
      x[1] = to_f32<DT>(v.y);
      x[2] = to_f32<DT>(v.z);
      x[3] = to_f32<DT>(v.w);
    } else {
      x[0] = to_f32<DT>(v.x & 0xFFFFu);
      x[1] = to_f32<DT>(v.x >> 16);
      x[2] = to_f32<DT>(v.y & 0xFFFFu);
      x[3] = to_f32<DT>(v.y >> 16);
    }
  }
};

template <int DT> __device__ __forceinline__ void load4(const void* base, uint64_t e, float (&x)[4]) {
  Vec4<DT>::unpack(Vec4<DT>::load(base, e), x);
}

template <int DT> __device__ __forceinline__ void store4(void* base, uint64_t e, const uint32_t (&b)[4]) {
  if constexpr (Fmt<DT>::bytes == 4) {
    __stcs(reinterpret_cast<uint4*>(static_cast<uint32_t*>(base) + e), make_uint4(b[0], b[1], b[2], b[3]));
  } else {
    __stcs(reinterpret_cast<uint2*>(static_cast<uint16_t*>(base) + e),
           make_uint2((b[0] & 0xFFFFu) | (b[1] << 16), (b[2] & 0xFFFFu) | (b[3] << 16)));
  }
}

template <int DT> __device__ __forceinline__ float load_elem(const void* base, uint64_t e) {
  if constexpr (Fmt<DT>::bytes == 4) return to_f32<DT>(*(static_cast<const uint32_t*>(base) + e));
  else return to_f32<DT>(*(static_cast<const uint16_t*>(base) + e));
}

// The block [lo, hi) of a chunk whose fold starts at rank s0, on its own
// (a chunk's short last block, an odd last block, unaligned buffers).
template <int IDT, int ODT, int OP, int MAXN, bool VEC>
__device__ __forceinline__ void hop_block(const Fp8HopArgs& A, uint64_t lo, uint64_t hi, int s0, int lane) {
  const int N = A.nranks;
  const bool full = VEC && hi - lo == kFp8Block;  // warp-uniform
  bool valid[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) valid[k] = full || lo + lane + 32 * k < hi;
  float p[4];
#pragma unroll 1
  for (int b0 = 0; b0 < MAXN; b0 += 8) {
    if (b0 >= N) break;
    float x[8][4];
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      if (b0 + m < N) {
        int r = s0 + b0 + m;
        r = (r >= N) ? r - N : r;
        if (full) {
          load4<IDT>(A.src[r], lo + 4 * lane, x[m]);
        } else {
#pragma unroll
          for (int k = 0; k < 4; ++k) x[m][k] = valid[k] ? load_elem<IDT>(A.src[r], lo + lane + 32 * k) : 0.0f;
        }
      }
    }
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      if (b0 + m < N) {
        if (b0 + m == 0) {
#pragma unroll
          for (int k = 0; k < 4; ++k) p[k] = x[m][k];
        } else {
          qdq_block(p);  // the partial goes over the wire in FP8
#pragma unroll
          for (int k = 0; k < 4; ++k) p[k] = __fadd_rn(p[k], x[m][k]);
        }
      }
    }
  }
  if constexpr (OP == OP_AVG) {
#pragma unroll
    for (int k = 0; k < 4; ++k) p[k] = avg_div(p[k], N);
  }
  qdq_block(p);  // the finished chunk, as the all-gather sends it
  if (full) {
    uint32_t bits[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) bits[k] = from_f32<ODT>(p[k]);
    for (int r = 0; r < N; ++r) store4<ODT>(A.dst[r], lo + 4 * lane, bits);
    return;
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    if (!valid[k]) continue;
    const uint32_t bits = from_f32<ODT>(p[k]);
    const uint64_t e = lo + lane + 32 * k;
    for (int r = 0; r < N; ++r) {
      if constexpr (Fmt<ODT>::bytes == 4) *(static_cast<uint32_t*>(A.dst[r]) + e) = bits;
      else *(static_cast<uint16_t*>(A.dst[r]) + e) = (uint16_t)bits;
    }
  }
}

constexpr int kHopBatch16 = 8;  // ranks loaded before they are folded, 16-bit inputs

// hop_block out of line: the pairs' rare general path and the chunks' tails,
// so that the division and reciprocal calls of the general quantiser shape
// the register allocation of neither the pairs' loop nor the kernel's
template <int IDT, int ODT, int OP, int MAXN, bool VEC>
static __device__ __noinline__ void hop_block_general(const Fp8HopArgs& A, uint64_t lo, uint64_t hi, int s0,
                                                      int lane) {
  hop_block<IDT, ODT, OP, MAXN, VEC>(A, lo, hi, s0, lane);
}

// Two whole aligned blocks [lo, lo + 256) of one chunk: lane l holds elements
// 4l..4l+3 of each; the ranks' raw vectors are loaded in batches (8 ranks of
// 16-bit inputs, 4 of binary32) before they are folded.
template <int IDT, int ODT, int OP, int MAXN>
__device__ __forceinline__ void hop_pair(const Fp8HopArgs& A, uint64_t lo, int s0, int lane) {
  using V4 = Vec4<IDT>;
  constexpr int BATCH = Fmt<IDT>::bytes == 4 ? 4 : kHopBatch16;
  const int N = A.nranks;
  const uint64_t ea = lo + 4 * lane, eb = ea + kFp8Block;
  float pa[4], pb[4];
  bool ok = true;  // warp-uniform
#pragma unroll 1
  for (int b0 = 0; b0 < MAXN; b0 += BATCH) {
    if (b0 >= N) break;
    typename V4::Raw xa[BATCH], xb[BATCH];
#pragma unroll
    for (int m = 0; m < BATCH; ++m) {
      if (b0 + m < N) {
        int r = s0 + b0 + m;
        r = (r >= N) ? r - N : r;
        xa[m] = V4::load(A.src[r], ea);
        xb[m] = V4::load(A.src[r], eb);
      }
    }
#pragma unroll
    for (int m = 0; m < BATCH; ++m) {
      if (b0 + m < N) {
        float fa[4], fb[4];
        V4::unpack(xa[m], fa);
        V4::unpack(xb[m], fb);
        if (b0 + m == 0) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            pa[k] = fa[k];
            pb[k] = fb[k];
          }
        } else {
          ok &= qdq_block_pair(pa, pb);  // the partials go over the wire in FP8
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            pa[k] = __fadd_rn(pa[k], fa[k]);
            pb[k] = __fadd_rn(pb[k], fb[k]);
          }
        }
      }
    }
  }
  if constexpr (OP == OP_AVG) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      pa[k] = avg_div(pa[k], N);
      pb[k] = avg_div(pb[k], N);
    }
  }
  ok &= qdq_block_pair(pa, pb);  // the finished chunk, as the all-gather sends it
  if (!ok) {
    hop_block_general<IDT, ODT, OP, MAXN, true>(A, lo, lo + kFp8Block, s0, lane);
    hop_block_general<IDT, ODT, OP, MAXN, true>(A, lo + kFp8Block, lo + 2 * kFp8Block, s0, lane);
    return;
  }
  uint32_t ba[4], bb[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    ba[k] = from_f32<ODT>(pa[k]);
    bb[k] = from_f32<ODT>(pb[k]);
  }
  for (int r = 0; r < N; ++r) {
    store4<ODT>(A.dst[r], ea, ba);
    store4<ODT>(A.dst[r], eb, bb);
  }
}

constexpr int kHopBlocksPerSm = 3;

// One warp per pair of blocks (blocks 2j and 2j+1 of a chunk, counted from
// its start), the resident grid's warps looping over the pairs.
template <int IDT, int ODT, int OP, int MAXN, bool VEC>
__global__ void __launch_bounds__(kThreads, kHopBlocksPerSm) k_fp8_hop(const __grid_constant__ Fp8HopArgs A) {
  pdl_begin();
  const int N = A.nranks;
  const int lane = threadIdx.x & 31;
  const uint64_t npairs = (A.nbc + 1) / 2;
  const uint64_t tasks = (uint64_t)N * npairs;
  const uint64_t warp0 = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const uint64_t nwarps = ((uint64_t)gridDim.x * blockDim.x) >> 5;
  for (uint64_t t = warp0; t < tasks; t += nwarps) {  // warp-uniform
    const int c = (int)(t / npairs);
    const uint64_t clo = (uint64_t)c * A.L;
    const uint64_t chi = (clo + A.L < A.count) ? clo + A.L : A.count;
    const uint64_t lo = clo + (t - (uint64_t)c * npairs) * (2 * kFp8Block);
    if (clo >= A.count || lo >= chi) continue;
    const int s0 = (c + 1 == N) ? 0 : c + 1;
    if (VEC && lo + 2 * kFp8Block <= chi) {
      hop_pair<IDT, ODT, OP, MAXN>(A, lo, s0, lane);
      continue;
    }
    const uint64_t mid = (lo + kFp8Block < chi) ? lo + kFp8Block : chi;
    hop_block_general<IDT, ODT, OP, MAXN, VEC>(A, lo, mid, s0, lane);
    if (mid < chi)
      hop_block_general<IDT, ODT, OP, MAXN, VEC>(A, mid, (mid + kFp8Block < chi) ? mid + kFp8Block : chi, s0, lane);
  }
}

template <int IDT, int ODT, int OP>
cudaError_t launch_hop_op(const Fp8HopArgs& a, cudaStream_t s) {
  const uint64_t tasks = (uint64_t)a.nranks * ((a.nbc + 1) / 2);
  if (tasks == 0) return cudaSuccess;
  // a resident grid (kHopBlocksPerSm blocks per SM), each warp looping over
  // pairs of blocks: measured faster than one warp per pair (1.42 against
  // 1.46 ms for 16 x 134,217,728 bf16)
  int sms = 0;
  const cudaError_t e = sm_count(&sms);
  if (e != cudaSuccess) return e;
  const uint64_t resident = (uint64_t)sms * kHopBlocksPerSm;
  const unsigned grid = grid_for(tasks * 32) < resident ? grid_for(tasks * 32) : (unsigned)resident;
  // 4-element vectors when every buffer allows them (block starts are
  // multiples of 4 elements: chunk lengths are multiples of 16 bytes of the
  // output type)
  bool vec = true;
  for (int r = 0; r < a.nranks; ++r)
    vec = vec && reinterpret_cast<uintptr_t>(a.src[r]) % (4 * Fmt<IDT>::bytes) == 0 &&
          reinterpret_cast<uintptr_t>(a.dst[r]) % (4 * Fmt<ODT>::bytes) == 0;
#define GAR_HOP(MAXNV)                                                                 \
  return vec ? launch_pdl(k_fp8_hop<IDT, ODT, OP, MAXNV, true>, dim3(grid), 0, s, a) \
             : launch_pdl(k_fp8_hop<IDT, ODT, OP, MAXNV, false>, dim3(grid), 0, s, a);
  if (a.nranks <= 8) {
    GAR_HOP(8)
  } else if (a.nranks <= 16) {
    GAR_HOP(16)
  } else {
    GAR_HOP(kMaxRanks)
  }
#undef GAR_HOP
}

template <int IDT, int ODT> cudaError_t launch_hop_io(int op, const Fp8HopArgs& a, cudaStream_t s) {
  if (op == OP_SUM) return launch_hop_op<IDT, ODT, OP_SUM>(a, s);
  if (op == OP_AVG) return launch_hop_op<IDT, ODT, OP_AVG>(a, s);
  return cudaErrorInvalidValue;
}

template <int IDT> cudaError_t launch_hop_in(int out_dtype, int op, const Fp8HopArgs& a, cudaStream_t s) {
  switch (out_dtype) {
    case DT_F32: return launch_hop_io<IDT, DT_F32>(op, a, s);
    case DT_F16: return launch_hop_io<IDT, DT_F16>(op, a, s);
    case DT_BF16: return launch_hop_io<IDT, DT_BF16>(op, a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gar
