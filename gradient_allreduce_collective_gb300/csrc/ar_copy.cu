// ar_copy.cu — pure data-movement kernels (sm_103a):
//
//  k_gather     ring all-gather: each finished chunk is read once and written
//               to every other rank ("AllReduce（オールリデュース）" glossary,
//               §Ring-AllReduceの仕組み, AllGather phase; "AllReduce" astro-wiki,
//               §阶段二: receivers overwrite their copy). The ring's N-1
//               forwarding steps carry the same bytes to the same places, so on
//               one device a chunk goes straight from its owner to all ranks:
//               M read + (N-1)*M written instead of 2(N-1)*M moved.
//  k_multicopy  batched gather/scatter of gradient tensors into or out of a
//               flat bucket (glossary §パフォーマンスチューニング, bucketing).
//
// Both are HBM-bound copies with 16-byte streaming loads and stores.
#include <cstdint>

#include "ar_internal.h"

namespace gar {

template <int U> struct Unit;
template <> struct Unit<16> { using T = uint4; };
template <> struct Unit<4> { using T = uint32_t; };
template <> struct Unit<2> { using T = uint16_t; };
template <> struct Unit<1> { using T = uint8_t; };

template <int U> __device__ __forceinline__ typename Unit<U>::T ld_unit(const void* p) {
  if constexpr (U == 16) return __ldcs(static_cast<const uint4*>(p));
  else return *static_cast<const typename Unit<U>::T*>(p);
}
template <int U> __device__ __forceinline__ void st_unit(void* p, typename Unit<U>::T v) {
  if constexpr (U == 16) __stcs(static_cast<uint4*>(p), v);
  else *static_cast<typename Unit<U>::T*>(p) = v;
}

template <int U>
__global__ void __launch_bounds__(kThreads) k_gather(const __grid_constant__ GatherArgs A) {
  pdl_begin();
  const uint64_t t0 = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const uint64_t nt = (uint64_t)gridDim.x * blockDim.x;
  const int N = A.nranks;
  if (t0 < A.units) {
    int c = (int)(t0 / A.Lu);
    uint64_t cbeg = (uint64_t)c * A.Lu, cend = cbeg + A.Lu;
    for (uint64_t i = t0; i < A.units; i += nt) {
      while (i >= cend) {
        ++c;
        cbeg = cend;
        cend += A.Lu;
      }
      const auto v = ld_unit<U>(static_cast<const char*>(A.src[c]) + (i - cbeg) * U);
      const bool skip_own = (A.skip_mask >> c) & 1u;
      for (int q = 0; q < N; ++q) {
        if (q == c && skip_own) continue;
        st_unit<U>(static_cast<char*>(A.dst[q]) + i * U, v);
      }
    }
  }
  // byte tail after the last whole unit (all in one chunk)
  if (t0 < A.tail_bytes) {
    const uint64_t b = A.units * U + t0;
    const int c = (int)(b / A.Lb);
    const uint8_t v = *(static_cast<const uint8_t*>(A.src[c]) + (b - (uint64_t)c * A.Lb));
    const bool skip_own = (A.skip_mask >> c) & 1u;
    for (int q = 0; q < N; ++q) {
      if (q == c && skip_own) continue;
      *(static_cast<uint8_t*>(A.dst[q]) + b) = v;
    }
  }
}

template <int U> cudaError_t launch_gather_u(const GatherArgs& a, cudaStream_t stream) {
  const uint64_t items = a.units > a.tail_bytes ? a.units : a.tail_bytes;
  return launch_pdl(k_gather<U>, dim3(grid_for(items)), 0, stream, a);
}

cudaError_t launch_gather(int unit_bytes, const GatherArgs& a, cudaStream_t stream) {
  switch (unit_bytes) {
    case 16: return launch_gather_u<16>(a, stream);
    case 4: return launch_gather_u<4>(a, stream);
    case 2: return launch_gather_u<2>(a, stream);
    case 1: return launch_gather_u<1>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

// One block copies one kCopyTile-byte tile at a time; 4 x 16 bytes in flight per thread.
__global__ void __launch_bounds__(kThreads) k_multicopy(const __grid_constant__ MultiCopyArgs A) {
  pdl_begin();
  const uint32_t total = A.tile_start[A.nitems];
  for (uint32_t t = blockIdx.x; t < total; t += gridDim.x) {
    int lo = 0, hi = A.nitems - 1;  // last item whose first tile is <= t
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (A.tile_start[mid] <= t) lo = mid;
      else hi = mid - 1;
    }
    const CopyItem& it = A.item[lo];
    const uint64_t off = (uint64_t)(t - A.tile_start[lo]) * kCopyTile;
    const uint64_t end = (off + kCopyTile < it.bytes) ? off + kCopyTile : it.bytes;
    const char* s = static_cast<const char*>(it.src);
    char* d = static_cast<char*>(it.dst);
    if ((((uintptr_t)s | (uintptr_t)d) & 15u) == 0) {
      const uint64_t vend = off + ((end - off) & ~(uint64_t)15);
      constexpr int kUnroll = kCopyTile / (kThreads * 16);
      uint4 v[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const uint64_t b = off + ((uint64_t)u * kThreads + threadIdx.x) * 16;
        if (b < vend) v[u] = __ldcs(reinterpret_cast<const uint4*>(s + b));
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const uint64_t b = off + ((uint64_t)u * kThreads + threadIdx.x) * 16;
        if (b < vend) __stcs(reinterpret_cast<uint4*>(d + b), v[u]);
      }
      for (uint64_t b = vend + threadIdx.x; b < end; b += kThreads) d[b] = s[b];
    } else {
      for (uint64_t b = off + threadIdx.x; b < end; b += kThreads) d[b] = s[b];
    }
  }
}

cudaError_t launch_multicopy(const MultiCopyArgs& a, cudaStream_t stream) {
  const uint32_t total = a.tile_start[a.nitems];
  if (total == 0) return cudaSuccess;
  // one block per tile
  const unsigned grid = total < 0x7FFFFFFFu ? total : 0x7FFFFFFFu;
  return launch_pdl(k_multicopy, dim3(grid), 0, stream, a);
}

}  // namespace gar
