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
// One warp per block: lane l holds elements 4l..4l+3 of a whole block when
// every buffer is aligned for 4-element vectors (one load and one store per
// rank and lane), otherwise elements l, l+32, l+64, l+96; the block amax of
// each hop is a warp-wide xor reduction; the ranks' values are loaded in
// batches of eight ranks before they are folded.
#pragma once

#include <cstdint>

#include "ar_fp8_common.cuh"

namespace gar {

// quantise-dequantise a warp's 128-element block held 4 values per lane
__device__ __forceinline__ void qdq_block(float (&p)[4]) {
  float amax = 0.0f;
#pragma unroll
  for (int k = 0; k < 4; ++k) amax = fmaxf(amax, fabsf(p[k]));
  amax = group_amax<32>(amax);
  const float s = scale_of(amax);
  const float x[4] = {p[0], p[1], p[2], p[3]};
  qdq_lane<4>(x, amax, s, p);
}

// four consecutive elements starting at e (e a multiple of 4, base aligned)
template <int DT> __device__ __forceinline__ void load4(const void* base, uint64_t e, float (&x)[4]) {
  if constexpr (Fmt<DT>::bytes == 4) {
    const uint4 v = __ldcs(reinterpret_cast<const uint4*>(static_cast<const uint32_t*>(base) + e));
    x[0] = to_f32<DT>(v.x);
    x[1] = to_f32<DT>(v.y);
    x[2] = to_f32<DT>(v.z);
    x[3] = to_f32<DT>(v.w);
  } else {
    const uint2 v = __ldcs(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(base) + e));
    x[0] = to_f32<DT>(v.x & 0xFFFFu);
    x[1] = to_f32<DT>(v.x >> 16);
    x[2] = to_f32<DT>(v.y & 0xFFFFu);
    x[3] = to_f32<DT>(v.y >> 16);
  }
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

template <int IDT, int ODT, int OP, int MAXN, bool VEC>
__global__ void __launch_bounds__(kThreads, 4) k_fp8_hop(const __grid_constant__ Fp8HopArgs A) {
  const int N = A.nranks;
  const int lane = threadIdx.x & 31;
  const uint64_t tasks = (uint64_t)N * A.nbc;
  const uint64_t warp0 = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const uint64_t nwarps = ((uint64_t)gridDim.x * blockDim.x) >> 5;
  for (uint64_t t = warp0; t < tasks; t += nwarps) {  // warp-uniform
    const int c = (int)(t / A.nbc);
    const uint64_t j = t - (uint64_t)c * A.nbc;
    const uint64_t clo = (uint64_t)c * A.L;
    const uint64_t chi = (clo + A.L < A.count) ? clo + A.L : A.count;
    const uint64_t lo = clo + j * kFp8Block;
    if (clo >= A.count || lo >= chi) continue;
    const uint64_t hi = (lo + kFp8Block < chi) ? lo + kFp8Block : chi;
    const bool full = VEC && hi - lo == kFp8Block;  // warp-uniform
    bool valid[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) valid[k] = full || lo + lane + 32 * k < hi;
    const int s0 = (c + 1 == N) ? 0 : c + 1;
    if (VEC) {
      // this lane's vectors of the warp's next block, every rank, into L2:
      // their loads then wait on L2 rather than DRAM
      const uint64_t tn = t + nwarps;
      if (tn < tasks) {
        const int cn = (int)(tn / A.nbc);
        const uint64_t lon = (uint64_t)cn * A.L + (tn - (uint64_t)cn * A.nbc) * kFp8Block;
        if (lon + kFp8Block <= A.count) {
          for (int r = 0; r < N; ++r)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(static_cast<const char*>(A.src[r]) +
                                                            (lon + 4 * lane) * Fmt<IDT>::bytes));
        }
      }
    }
    float p[4];
#pragma unroll
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
            if (b0 + 8 + m < N) {  // the same lane's vector of the rank eight places later, into L2
              int r2 = r + 8;
              r2 = (r2 >= N) ? r2 - N : r2;
              asm volatile("prefetch.global.L2 [%0];" ::"l"(static_cast<const char*>(A.src[r2]) +
                                                              (lo + 4 * lane) * Fmt<IDT>::bytes));
            }
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
      for (int k = 0; k < 4; ++k) p[k] = __fdiv_rn(p[k], (float)N);
    }
    qdq_block(p);  // the finished chunk, as the all-gather sends it
    if (full) {
      uint32_t bits[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) bits[k] = from_f32<ODT>(p[k]);
      for (int r = 0; r < N; ++r) store4<ODT>(A.dst[r], lo + 4 * lane, bits);
      continue;
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
}

template <int IDT, int ODT, int OP>
cudaError_t launch_hop_op(const Fp8HopArgs& a, cudaStream_t s) {
  const uint64_t tasks = (uint64_t)a.nranks * a.nbc;
  if (tasks == 0) return cudaSuccess;
  // a resident grid (4 blocks of 8 warps per SM), each warp looping over
  // blocks, so that it can prefetch its next block while folding this one
  const uint64_t resident = 152ull * 4;
  const unsigned grid = grid_for(tasks * 32) < resident ? grid_for(tasks * 32) : (unsigned)resident;
  // 4-element vectors when every buffer allows them (block starts are
  // multiples of 4 elements: chunk lengths are multiples of 16 bytes of the
  // output type)
  bool vec = true;
  for (int r = 0; r < a.nranks; ++r)
    vec = vec && reinterpret_cast<uintptr_t>(a.src[r]) % (4 * Fmt<IDT>::bytes) == 0 &&
          reinterpret_cast<uintptr_t>(a.dst[r]) % (4 * Fmt<ODT>::bytes) == 0;
#define GAR_HOP(MAXNV)                                                        \
  if (vec) k_fp8_hop<IDT, ODT, OP, MAXNV, true><<<grid, kThreads, 0, s>>>(a); \
  else k_fp8_hop<IDT, ODT, OP, MAXNV, false><<<grid, kThreads, 0, s>>>(a);
  if (a.nranks <= 8) {
    GAR_HOP(8)
  } else if (a.nranks <= 16) {
    GAR_HOP(16)
  } else {
    GAR_HOP(kMaxRanks)
  }
#undef GAR_HOP
  return cudaGetLastError();
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
