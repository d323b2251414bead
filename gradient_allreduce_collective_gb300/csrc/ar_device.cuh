// ar_device.cuh — device building blocks for the allreduce kernels (sm_103a).
//
// Element formats, the element-wise operator, and the two fold orders:
//   ring: the chunk-c element is folded x_{c+1}, x_{c+2}, ..., x_{c+N} (mod N)
//     — the order a ring reduce-scatter produces when GPU i sends its partial
//     to GPU i+1, which adds it to its own chunk ("AllReduce（オールリデュース）"
//     glossary, §Ring-AllReduceの仕組み; "AllReduce" astro-wiki, §Ring AllReduce
//     阶段一); chunk c finishes at rank c.
//   tree: recursive halving, v_r = v_r (+) v_{r+d} for d = N/2, ..., 1
//     (glossary algorithm table, "Recursive Halving-Doubling").
// Both orders are fixed per element, so every kernel that uses the same order
// produces bit-identical results whatever its grid or vector width.
#pragma once

#include <cstdint>
#include <type_traits>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "ar_internal.h"

namespace gar {

// ---------------------------------------------------------------- formats

template <int DT> struct Fmt;
template <> struct Fmt<DT_F32> {
  static constexpr int bytes = 4;
  static constexpr uint32_t sign = 0x80000000u, mag = 0x7FFFFFFFu, inf = 0x7F800000u, qnan = 0x7FC00000u,
                            all = 0xFFFFFFFFu;
};
template <> struct Fmt<DT_BF16> {
  static constexpr int bytes = 2;
  static constexpr uint32_t sign = 0x8000u, mag = 0x7FFFu, inf = 0x7F80u, qnan = 0x7FC0u, all = 0xFFFFu;
};
template <> struct Fmt<DT_F16> {
  static constexpr int bytes = 2;
  static constexpr uint32_t sign = 0x8000u, mag = 0x7FFFu, inf = 0x7C00u, qnan = 0x7E00u, all = 0xFFFFu;
};
template <> struct Fmt<DT_I32> {
  static constexpr int bytes = 4;
};

// exact widening of a storage pattern to binary32
template <int DT> __device__ __forceinline__ float to_f32(uint32_t b) {
  if constexpr (DT == DT_F32) return __uint_as_float(b);
  else if constexpr (DT == DT_BF16) return __uint_as_float(b << 16);
  else return __half2float(__ushort_as_half((unsigned short)b));
}

// binary32 -> storage pattern, round to nearest even (hardware conversion)
template <int DT> __device__ __forceinline__ uint32_t from_f32(float x) {
  if constexpr (DT == DT_F32) return __float_as_uint(x);
  else if constexpr (DT == DT_BF16) return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x));
  else return (uint32_t)__half_as_ushort(__float2half_rn(x));
}

template <int DT> __device__ __forceinline__ bool is_nan_bits(uint32_t b) {
  return (b & Fmt<DT>::mag) > Fmt<DT>::inf;
}

// total-order key: -0 below +0, negatives reversed; NaN handled by the caller
template <int DT> __device__ __forceinline__ uint32_t order_key(uint32_t b) {
  return (b & Fmt<DT>::sign) ? (~b & Fmt<DT>::all) : (b | Fmt<DT>::sign);
}

// x / n of the AVG operator, the correctly rounded binary32 quotient. For n a
// power of two, 1/n is exact and x * (1/n) rounds the same real number x/n
// once, so one multiply gives the division's bits (subnormal results
// included); other n take the IEEE division.
__device__ __forceinline__ float avg_div(float x, int n) {
  if ((n & (n - 1)) == 0) return __fmul_rn(x, __int_as_float((128 - __ffs(n)) << 23));
  return __fdiv_rn(x, (float)n);
}

// ---------------------------------------------------------------- operator
//
// Sum, min, max and average are the element-wise operators of the "All-reduce"
// page (wikiprompt, definition); average sums and divides the finished sum by
// N once ("AllReduce" astro-wiki, §在 DDP 中的角色). Floating sums run in
// binary32 (bf16/fp16 widen exactly, round once at the end); int32 sums wrap;
// MIN/MAX select one input exactly (or the canonical NaN).

template <int DT, int OP> struct Red {
  static constexpr bool kInt = (DT == DT_I32);
  static constexpr bool kSel = (OP == OP_MIN || OP == OP_MAX);
  using Acc = std::conditional_t<(!kInt && !kSel), float, uint32_t>;

  __device__ __forceinline__ static Acc init(uint32_t bits) {
    if constexpr (!kInt && !kSel) return to_f32<DT>(bits);
    else return bits;
  }

  __device__ __forceinline__ static Acc comb(Acc a, Acc b) {
    if constexpr (kSel) {
      if constexpr (kInt) {
        const int32_t x = (int32_t)a, y = (int32_t)b;
        if constexpr (OP == OP_MIN) return (y < x) ? b : a;
        else return (y > x) ? b : a;
      } else {
        if (is_nan_bits<DT>(a) || is_nan_bits<DT>(b)) return Fmt<DT>::qnan;
        if constexpr (OP == OP_MIN) return (order_key<DT>(b) < order_key<DT>(a)) ? b : a;
        else return (order_key<DT>(b) > order_key<DT>(a)) ? b : a;
      }
    } else if constexpr (kInt) {
      return a + b;  // modulo 2^32
    } else {
      return __fadd_rn(a, b);
    }
  }

  __device__ __forceinline__ static uint32_t fin(Acc a, int n) {
    if constexpr (kSel) {
      if constexpr (!kInt) {
        if (is_nan_bits<DT>(a)) return Fmt<DT>::qnan;
      }
      return a;
    } else if constexpr (kInt) {
      if constexpr (OP == OP_AVG) return (uint32_t)((int32_t)a / n);
      else return a;
    } else {
      if constexpr (OP == OP_AVG) return from_f32<DT>(avg_div(a, n));
      else return from_f32<DT>(a);
    }
  }
};

// ---------------------------------------------------------------- lanes of a 16-byte vector

template <int BYTES> __device__ __forceinline__ uint32_t get_lane(const uint4& v, int k) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  if constexpr (BYTES == 4) return w[k];
  else return (w[k >> 1] >> ((k & 1) * 16)) & 0xFFFFu;
}

template <int BYTES> __device__ __forceinline__ void set_lane(uint4& v, int k, uint32_t b) {
  uint32_t w[4] = {v.x, v.y, v.z, v.w};
  if constexpr (BYTES == 4) {
    w[k] = b;
  } else {
    const int sh = (k & 1) * 16;
    w[k >> 1] = (w[k >> 1] & ~(0xFFFFu << sh)) | ((b & 0xFFFFu) << sh);
  }
  v = make_uint4(w[0], w[1], w[2], w[3]);
}

// ---------------------------------------------------------------- fold orders
//
// A loader `Ld` gives, for one item (a vector of V elements, or one element),
//   Raw  load(int r)                 — issue the loads of rank r's values
//   void unpack(const Raw&, Acc(&)[V]) — turn them into accumulator lanes
//   Acc  comb(Acc, Acc)              — the operator
// Loads of up to 8 ranks are issued before any combine so that 8 x 16 bytes
// per thread are in flight.

// A loader may declare `static constexpr bool kPairAdd = true` when its comb
// is the binary32 add; pairs of lanes then use the packed add, whose
// components are rounded exactly as two scalar adds.
template <class Ld, class = void> struct PairAdd { static constexpr bool value = false; };
template <class Ld> struct PairAdd<Ld, std::void_t<decltype(Ld::kPairAdd)>> {
  static constexpr bool value = Ld::kPairAdd;
};

// A loader may declare `static constexpr int kBatch`: how many ranks' loads
// the ring order issues before folding them (8 unless it says otherwise).
template <class Ld, class = void> struct LoadBatch { static constexpr int value = 8; };
template <class Ld> struct LoadBatch<Ld, std::void_t<decltype(Ld::kBatch)>> {
  static constexpr int value = Ld::kBatch;
};

template <class Ld> struct Fold {
  using Acc = typename Ld::Acc;
  using Raw = typename Ld::Raw;
  static constexpr int V = Ld::V;
  static constexpr int kB = LoadBatch<Ld>::value;

  __device__ __forceinline__ static void comb_into(Acc (&a)[V], const Acc (&b)[V]) {
    if constexpr (PairAdd<Ld>::value && V % 2 == 0) {
#pragma unroll
      for (int k = 0; k < V; k += 2) {
        const float2 p = __fadd2_rn(make_float2(a[k], a[k + 1]), make_float2(b[k], b[k + 1]));
        a[k] = p.x;
        a[k + 1] = p.y;
      }
    } else {
#pragma unroll
      for (int k = 0; k < V; ++k) a[k] = Ld::comb(a[k], b[k]);
    }
  }

  // ring order starting at rank s (0 <= s < N): acc = x_s (+) x_{s+1} (+) ...
  // MAXN: compile-time bound on N (it drops the code for further batches);
  // the loads of kB ranks are issued before they are folded.
  template <int MAXN>
  __device__ __forceinline__ static void ring(const Ld& ld, int N, int s, Acc (&acc)[V]) {
    {
      Raw raw[kB];
#pragma unroll
      for (int j = 0; j < kB; ++j) {
        if (j < N) {
          int r = s + j;
          r = (r >= N) ? r - N : r;
          raw[j] = ld.load(r);
        }
      }
      ld.unpack(raw[0], acc);
#pragma unroll
      for (int j = 1; j < kB; ++j) {
        if (j < N) {
          Acc x[V];
          ld.unpack(raw[j], x);
          comb_into(acc, x);
        }
      }
    }
    if constexpr (MAXN > kB) {
#pragma unroll
      for (int b0 = kB; b0 < MAXN; b0 += kB) {
        if (b0 >= N) break;
        Raw raw[kB];
#pragma unroll
        for (int j = 0; j < kB; ++j) {
          if (b0 + j < N) {
            int r = s + b0 + j;
            r = (r >= N) ? r - N : r;
            raw[j] = ld.load(r);
          }
        }
#pragma unroll
        for (int j = 0; j < kB; ++j) {
          if (b0 + j < N) {
            Acc x[V];
            ld.unpack(raw[j], x);
            comb_into(acc, x);
          }
        }
      }
    }
  }

  // one recursive-halving step over n (power of two, <= 8) partial values
  __device__ __forceinline__ static void halve(Acc (&v)[8][V], int n) {
    if (4 < n) {
#pragma unroll
      for (int q = 0; q < 4; ++q) comb_into(v[q], v[q + 4]);
    }
    if (2 < n) {
#pragma unroll
      for (int q = 0; q < 2; ++q) comb_into(v[q], v[q + 2]);
    }
    if (1 < n) comb_into(v[0], v[1]);
  }

  // recursive halving over ranks base + m*stride, m = 0..n-1 (n <= 8, power of two)
  __device__ __forceinline__ static void tree8(const Ld& ld, int base, int stride, int n, Acc (&out)[V]) {
    Raw raw[8];
#pragma unroll
    for (int m = 0; m < 8; ++m)
      if (m < n) raw[m] = ld.load(base + m * stride);
    Acc v[8][V];
#pragma unroll
    for (int m = 0; m < 8; ++m)
      if (m < n) ld.unpack(raw[m], v[m]);
    halve(v, n);
#pragma unroll
    for (int k = 0; k < V; ++k) out[k] = v[0][k];
  }

  // Recursive halving over N ranks (N a power of two, <= 64). For N > 8 the
  // first three halving steps (distances N/2, N/4, N/8) act on the ranks
  // r + m*(N/8), m = 0..7, separately for each r < N/8; the remaining steps
  // halve those N/8 partial results. The expression tree is the same.
  template <int MAXN>
  __device__ __forceinline__ static void tree(const Ld& ld, int N, Acc (&acc)[V]) {
    if (MAXN <= 8 || N <= 8) {
      tree8(ld, 0, 1, N, acc);
      return;
    }
    const int nb = N >> 3;
    Acc part[8][V];
#pragma unroll
    for (int r = 0; r < (MAXN >= 64 ? 8 : MAXN / 8); ++r)
      if (r < nb) tree8(ld, r, nb, 8, part[r]);
    halve(part, nb);
#pragma unroll
    for (int k = 0; k < V; ++k) acc[k] = part[0][k];
  }
};

}  // namespace gar
