// ar_topk.cu — Top-K gradient sparsification with error feedback, and the
// allreduce of the resulting sparse vectors (sm_103a).
//
// "AllReduce（オールリデュース）" glossary, §勾配圧縮技術: only the top K% of the
// gradient is communicated and error feedback compensates what is dropped;
// "All-reduce" (wikiprompt), §优化技术: top-k also has to send the indices.
// Per rank: a = g + e (binary32; e is the residual kept from the previous
// step), keep the k largest |a| (ties: lower index first), emit (index,
// value) pairs in ascending index order, and leave e = a with the kept
// entries zeroed.
//
// Exact selection without sorting: the key T of the k-th largest magnitude
// comes from a three-digit radix select over the 31 magnitude bits (11 + 10
// + 10 bits). Pass 1 reads g and e once, writes a, and histograms the first
// digit. Pass 2 reads a once more, histograms the second digit among the keys
// in the first digit's bin, and compacts every key at or above that bin (all
// that can still be kept) in index order into the tile's slots. Pass 3, the
// count of keys above and equal to T per tile, and the emission read only
// the slots; if some tile's keys do not fit its slots they read the data
// instead (same results). The block of each pass that finishes last picks
// the digit or scans the per-tile counts, so the state never leaves the
// device and no launch is spent on it. Keys above T are all kept; of the keys
// equal to T, the first (k - #above) in index order. All ranks of a call
// share each launch (grid.y = rank): six launches per call.
//
// On large calls the previous call's T, kept in the workspace, makes the
// common case cheaper without changing any result: pass 1 also compacts the
// values at or above T times a margin into the slots, and when at least k of
// them fit, pass 2 reads the slots instead of the data (or, when T's first
// digit held, has nothing left to do: pass 1 found the second digit too).
// Pass 3 then compacts each tile's slots to the keys at or above the
// two-digit prefix and, from a short list of the keys equal to it, derives
// the per-tile counts itself, so the count pass only reads its flag.
//
// The sparse allreduce (SUM, AVG) densifies each output tile from every
// rank's pairs in shared memory and folds it in the dense order, so only the
// N replicas are written; MIN and MAX go through dense copies and the dense
// allreduce.
#include <algorithm>
#include <cstdint>
#include <string>
#include <vector>

#include "ar.h"
#include "ar_device.cuh"
#include "ar_topk_internal.h"
#include "ar_trace.h"

namespace gar {

void set_last_error(const std::string& msg);

namespace {

constexpr int kHistBlocksPerSm = 8;
constexpr int kSplitBlocksPerSm = 3;  // the register budget of k_topk_split
constexpr int kPass1BlocksPerSm = 5;  // k_topk_pass1 keeps 8 float4 loads in flight per thread
constexpr int kSpecBlocksPerSm = 3;   // k_topk_pass1_spec keeps 16 float4 loads in flight per lane

__device__ __forceinline__ uint32_t mag_key(float a) { return __float_as_uint(a) & 0x7FFFFFFFu; }

// Programmatic dependent launch: every kernel here is launched by launch_pdl
// and begins with pdl_begin (ar_internal.h), or with pdl_wait.

// Only the wait: the kernel's dependents launch as its blocks exit. For a
// grid of many waves whose dependents would otherwise hold SM resources,
// waiting, while its last waves still need them.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

constexpr int kWarps = kThreads / 32;  // tiles per block in the slot-reading passes

struct RankWs {
  uint32_t* hist;
  TopkState* st;
  uint32_t* n_gt;
  uint32_t* n_eq;
  uint32_t* eq_before;
  uint32_t* out_off;
  uint32_t* n_s;
  uint32_t* masks;
  uint32_t* slots;
};

__device__ __forceinline__ RankWs rank_ws(const TopkArgs& A, int r) {
  uint32_t* base = A.ws + (uint64_t)r * A.ws_words;
  RankWs w;
  w.hist = base;
  w.st = reinterpret_cast<TopkState*>(base + kTopkHistWords);
  w.n_gt = base + kTopkHistWords + kTopkStateWords;
  w.n_eq = w.n_gt + A.nb;
  w.eq_before = w.n_eq + A.nb;
  w.out_off = w.eq_before + A.nb;
  w.n_s = w.out_off + A.nb;
  w.masks = w.n_s + A.nb;
  w.slots = w.masks + A.nb * kThreads * kTopkRuns;
  return w;
}

// slot indices and values of one tile
__device__ __forceinline__ uint32_t* slot_idx(const RankWs& w, uint64_t tile, uint32_t S) {
  return w.slots + tile * 2ull * S;
}
__device__ __forceinline__ float* slot_val(const RankWs& w, uint64_t tile, uint32_t S) {
  return reinterpret_cast<float*>(w.slots + tile * 2ull * S + S);
}

// exclusive scan over the block of one value per thread; *total = block sum
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* total) {
  __shared__ uint32_t warp_sums[kThreads / 32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[w] = x;
  __syncthreads();
  if (w == 0) {
    uint32_t s = lane < kThreads / 32 ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < kThreads / 32) warp_sums[lane] = s;
  }
  __syncthreads();
  const uint32_t before = (w > 0 ? warp_sums[w - 1] : 0) + x - v;
  if (total) *total = warp_sums[kThreads / 32 - 1];
  __syncthreads();
  return before;
}

// Called by every thread of a block after its global writes for this pass:
// true in the block that finishes last among the gridDim.x blocks of its
// rank. The barrier orders the block's writes before thread 0's fence and
// ticket (the fence is cumulative over what the barrier made visible to it).
// No block waits for another.
__device__ __forceinline__ bool last_block(uint32_t* ticket) {
  __shared__ bool s_last;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(ticket, 1u) == gridDim.x - 1;
    if (s_last) __threadfence();
  }
  __syncthreads();
  return s_last;
}

// The last block of a radix pass: the highest digit whose count from the top
// reaches `need` (a block-wide scan over BINS bins, highest first); fold it
// into the prefix and clear the bins for the next pass.
template <int BINS>
__device__ void find_digit(uint32_t* hist, int shift, TopkState* st) {
  constexpr int R = BINS / kThreads;
  const int top = BINS - threadIdx.x * R;  // this thread: bins [top - R, top)
  const uint32_t need = st->need;
  uint32_t h[R];
  uint32_t local = 0;
#pragma unroll
  for (int j = 0; j < R; ++j) {
    h[j] = __ldcg(hist + top - 1 - j);
    local += h[j];
  }
  const uint32_t above0 = block_exclusive_scan(local, nullptr);
  if (above0 < need && above0 + local >= need) {  // exactly one thread
    uint32_t above = above0;
    int pick = top - R;
#pragma unroll
    for (int j = 0; j < R; ++j) {
      if (above + h[j] >= need) {
        pick = top - 1 - j;
        break;
      }
      above += h[j];
    }
    st->prefix |= (uint32_t)pick << shift;
    st->mask |= (uint32_t)(BINS - 1) << shift;
    st->need = need - above;
    st->gt += above;
  }
#pragma unroll
  for (int j = 0; j < R; ++j) hist[top - 1 - j] = 0;
}

__global__ void __launch_bounds__(kThreads) k_topk_init(const __grid_constant__ TopkArgs A) {
  pdl_begin();
  const RankWs w = rank_ws(A, blockIdx.y);
  for (int i = threadIdx.x; i < kTopkHistWords; i += blockDim.x) w.hist[i] = 0;
  if (threadIdx.x == 0) {
    w.st->prefix = 0;
    w.st->mask = 0;
    w.st->need = A.k;
    w.st->gt = 0;
    for (int p = 0; p < 4; ++p) w.st->ticket[p] = 0;
    w.st->overflow = 0;
    w.st->spec_ok = 0;  // the hint and t_prev are left as the previous call set them
    w.st->spec_overflow = 0;
    w.st->spec_count = 0;
    w.st->pre2 = 0;
    w.st->mcount = 0;
    w.st->counted = 0;
  }
  if (A.nb > 0)  // pass 1's second-digit histogram
    for (int i = threadIdx.x; i < 1024; i += blockDim.x) w.masks[i] = 0;
}

__device__ __forceinline__ float4 add4(float4 x, float4 y) {
  return make_float4(__fadd_rn(x.x, y.x), __fadd_rn(x.y, y.y), __fadd_rn(x.z, y.z), __fadd_rn(x.w, y.w));
}

// Pass 1: a = g + e into e, histogram of bits 30..20 of |a|, then (last
// block, if k > 0) the first digit.
template <bool VEC>
__global__ void __launch_bounds__(kThreads, kPass1BlocksPerSm) k_topk_pass1(const __grid_constant__ TopkArgs A) {
  pdl_begin();
  __shared__ uint32_t sh[2048];
  const int r = blockIdx.y;
  const RankWs w = rank_ws(A, r);
  const float* __restrict__ g = A.g[r];
  float* __restrict__ e = A.e[r];
  const uint64_t count = A.count;
  for (int i = threadIdx.x; i < 2048; i += blockDim.x) sh[i] = 0;
  __syncthreads();
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  const uint64_t t0 = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
  uint64_t done = 0;
  if (VEC) {
    const uint64_t n4 = count / 4;
    const float4* g4 = reinterpret_cast<const float4*>(g);
    float4* e4 = reinterpret_cast<float4*>(e);
    uint64_t q = t0;
    // four float4 of g and of e in flight per thread (128 bytes)
    for (; q + 3 * stride < n4; q += 4 * stride) {
      float4 x[4], y[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        x[u] = __ldcs(g4 + q + u * stride);
        y[u] = e4[q + u * stride];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float4 s4 = add4(x[u], y[u]);
        e4[q + u * stride] = s4;
        atomicAdd(&sh[mag_key(s4.x) >> 20], 1u);
        atomicAdd(&sh[mag_key(s4.y) >> 20], 1u);
        atomicAdd(&sh[mag_key(s4.z) >> 20], 1u);
        atomicAdd(&sh[mag_key(s4.w) >> 20], 1u);
      }
    }
    for (; q < n4; q += stride) {
      const float4 s4 = add4(__ldcs(g4 + q), e4[q]);
      e4[q] = s4;
      atomicAdd(&sh[mag_key(s4.x) >> 20], 1u);
      atomicAdd(&sh[mag_key(s4.y) >> 20], 1u);
      atomicAdd(&sh[mag_key(s4.z) >> 20], 1u);
      atomicAdd(&sh[mag_key(s4.w) >> 20], 1u);
    }
    done = n4 * 4;
  }
  for (uint64_t i = done + t0; i < count; i += stride) {
    const float s = __fadd_rn(g[i], e[i]);
    e[i] = s;
    atomicAdd(&sh[mag_key(s) >> 20], 1u);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 2048; i += blockDim.x)
    if (sh[i]) atomicAdd(&w.hist[i], sh[i]);
  if (A.k == 0) return;  // nothing to select
  if (last_block(&w.st->ticket[0])) find_digit<2048>(w.hist, 20, w.st);
}

// Pass 1 with speculative candidate slots (every buffer 16-byte aligned and
// enough tiles for a warp each): as k_topk_pass1, and each warp walks whole
// tiles of kTopkBlock values in index order, compacting the values whose key
// is at or above the hint into the tile's slots, in the layout the split
// pass fills. A warp takes 512 values at a time, lane l the float4 at
// offsets 128 q + 4 l (q = 0..3), so index order is q-major; the four
// per-q candidate counts of a lane are scanned across the warp as one word
// of 8-bit fields. The last block finds the first digit and decides whether
// the slots hold every key that can be kept: at least k keys at or above the
// hint (then T is at or above it, and so is every key kept) and no tile
// overflowing.
constexpr int kSpecSeg = 512;  // values of a warp in one segment

// The candidates (bit 4q + j of m: value (q, j) of the segment) of one lane
// to the slots from position p on, in index order; lb = the index of the
// lane's value (0, 0). CHECKED: positions at or past S are counted, not written.
template <bool CHECKED>
__device__ __forceinline__ void spec_emit(uint32_t m, uint32_t exc, uint32_t tot, uint32_t before,
                                          uint32_t lb, const float (&v)[4][4], uint32_t S,
                                          uint32_t* __restrict__ si, float* __restrict__ sv) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t p = before + ((exc >> (8 * q)) & 0xFFu);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if ((m >> (4 * q + j)) & 1u) {
        if (!CHECKED || p < S) {
          si[p] = lb + 128 * q + j;
          sv[p] = v[q][j];
        }
        ++p;
      }
    }
    before += (tot >> (8 * q)) & 0xFFu;
  }
}

// The speculative pass 1's block histogram, one count per key: bins 0..2047
// by bits 30..20, except that a key in the guessed first-digit bin d1g counts
// in bin 2048 + bits 19..10 instead (bin d1g is their sum).
__shared__ uint32_t s_spec_h[3072];

// Two 512-value segments of a tile from e0 on (lane l: the float4 at offsets
// 128 q + 4 l of each); rem = count - e0. FULL: both lie inside the data.
// The indices of values inside the data fit 32 bits (count does).
template <bool FULL>
__device__ __forceinline__ void spec_round(const float* __restrict__ g, float* __restrict__ e, uint32_t e0,
                                           uint32_t rem, uint32_t tau, uint32_t S, uint32_t* __restrict__ si,
                                           float* __restrict__ sv, uint32_t d1g, uint32_t& pos, int lane) {
  float v[2][4][4];
  if (FULL) {
    float4 x[8], y[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      x[q] = __ldcs(reinterpret_cast<const float4*>(g + e0 + 128 * q) + lane);
      y[q] = reinterpret_cast<const float4*>(e + e0 + 128 * q)[lane];
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 s4 = add4(x[q], y[q]);
      reinterpret_cast<float4*>(e + e0 + 128 * q)[lane] = s4;
      v[q >> 2][q & 3][0] = s4.x;
      v[q >> 2][q & 3][1] = s4.y;
      v[q >> 2][q & 3][2] = s4.z;
      v[q >> 2][q & 3][3] = s4.w;
    }
  } else {
#pragma unroll
    for (int q = 0; q < 8; ++q)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t o = 128 * q + 4 * lane + j;
        v[q >> 2][q & 3][j] = 0.0f;
        if (o < rem) {
          v[q >> 2][q & 3][j] = __fadd_rn(g[e0 + o], e[e0 + o]);
          e[e0 + o] = v[q >> 2][q & 3][j];
        }
      }
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {  // the two segments in index order
    const uint32_t lb = e0 + kSpecSeg * h + 4 * lane;
    uint32_t m = 0;  // bit 4q + j: value (h, q, j) is a candidate
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const bool in = FULL || (uint32_t)(kSpecSeg * h + 4 * lane + 128 * q + j) < rem;
        const uint32_t key = mag_key(v[h][q][j]);
        const uint32_t hi = key >> 20;
        if (in) atomicAdd(&s_spec_h[hi == d1g ? 2048u + ((key >> 10) & 1023u) : hi], 1u);
        if (in && key >= tau) m |= 1u << (4 * q + j);
      }
    const uint32_t c = (uint32_t)__popc(m & 0xFu) | ((uint32_t)__popc(m & 0xF0u) << 8) |
                       ((uint32_t)__popc(m & 0xF00u) << 16) | ((uint32_t)__popc(m & 0xF000u) << 24);
    uint32_t inc = c;  // no field overflows: at most 128 each
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t t = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += t;
    }
    const uint32_t tot = __shfl_sync(0xffffffffu, inc, 31), exc = inc - c;
    const uint32_t seg = (tot & 0xFFu) + ((tot >> 8) & 0xFFu) + ((tot >> 16) & 0xFFu) + (tot >> 24);
    if (pos + seg <= S)  // the same for the whole warp
      spec_emit<false>(m, exc, tot, pos, lb, v[h], S, si, sv);
    else
      spec_emit<true>(m, exc, tot, pos, lb, v[h], S, si, sv);
    pos += seg;
  }
}

__global__ void __launch_bounds__(kThreads, kSpecBlocksPerSm) k_topk_pass1_spec(const __grid_constant__ TopkArgs A) {
  pdl_begin();
  const int r = blockIdx.y;
  const RankWs w = rank_ws(A, r);
  const float* __restrict__ g = A.g[r];
  float* __restrict__ e = A.e[r];
  const uint32_t count = (uint32_t)A.count;
  const uint32_t tau = w.st->hint;
  const uint32_t d1g = w.st->t_prev >> 20;  // the first digit guessed
  const uint32_t S = A.slots;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < 3072; i += blockDim.x) s_spec_h[i] = 0;
  __syncthreads();
  // tiles interleaved over the blocks (tile = warp * gridDim.x + block), so
  // that every block, and so every SM, gets an equal share
  for (uint64_t tile = (uint64_t)wid * gridDim.x + blockIdx.x; tile < A.nb; tile += (uint64_t)gridDim.x * kWarps) {
    uint32_t* __restrict__ si = slot_idx(w, tile, S);
    float* __restrict__ sv = slot_val(w, tile, S);
    uint32_t pos = 0;
    const uint32_t t0 = (uint32_t)tile * kTopkBlock;
    if ((uint64_t)t0 + kTopkBlock <= count) {  // a whole tile: no bounds checks
      for (uint32_t e0 = t0; e0 < t0 + kTopkBlock; e0 += 2 * kSpecSeg)
        spec_round<true>(g, e, e0, 0u, tau, S, si, sv, d1g, pos, lane);
    } else {
      for (uint64_t e0 = t0; e0 < count; e0 += 2 * kSpecSeg) {
        const uint32_t rem = (uint32_t)(count - e0);
        if (rem >= 2 * kSpecSeg)
          spec_round<true>(g, e, (uint32_t)e0, rem, tau, S, si, sv, d1g, pos, lane);
        else
          spec_round<false>(g, e, (uint32_t)e0, rem, tau, S, si, sv, d1g, pos, lane);
      }
    }
    if (lane == 0) {
      w.n_s[tile] = pos;
      if (pos > S) atomicOr(&w.st->spec_overflow, 1u);
      if (pos) atomicAdd(&w.st->spec_count, pos);
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 2048; i += blockDim.x)
    if (s_spec_h[i]) atomicAdd(&w.hist[i], s_spec_h[i]);
  if (d1g < 2048) {  // a garbage t_prev gives a bin no key falls in
    uint32_t part = 0;
    for (int i = threadIdx.x; i < 1024; i += blockDim.x) {
      const uint32_t c = s_spec_h[2048 + i];
      part += c;
      if (c) atomicAdd(&w.masks[i], c);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if ((threadIdx.x & 31) == 0 && part) atomicAdd(&w.hist[d1g], part);
  }
  if (A.k == 0) return;
  if (last_block(&w.st->ticket[0])) {
    find_digit<2048>(w.hist, 20, w.st);
    __shared__ uint32_t s_pre2;
    __syncthreads();
    if (threadIdx.x == 0) {
      const bool ok = __ldcg(&w.st->spec_count) >= A.k && __ldcg(&w.st->spec_overflow) == 0;
      w.st->spec_ok = ok ? 1u : 0u;
      s_pre2 = (ok && (w.st->prefix >> 20) == d1g) ? 1u : 0u;
      w.st->pre2 = s_pre2;
    }
    __syncthreads();
    // the guessed bin is the first digit: the second digit from pass 1's own
    // histogram of that bin (the split pass would count the same keys)
    if (s_pre2) find_digit<1024>(w.masks, 10, w.st);
  }
}

// kTopkElems consecutive values starting at `base` (zero past the end)
template <bool VEC>
__device__ __forceinline__ void load_run(const float* __restrict__ a, uint64_t base, uint64_t count,
                                         float (&v)[kTopkElems]) {
  if (VEC && base + kTopkElems <= count) {
    const float4* p = reinterpret_cast<const float4*>(a + base);
#pragma unroll
    for (int q = 0; q < kTopkElems / 4; ++q) {
      const float4 x = p[q];
      v[4 * q] = x.x;
      v[4 * q + 1] = x.y;
      v[4 * q + 2] = x.z;
      v[4 * q + 3] = x.w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < kTopkElems; ++j) v[j] = base + j < count ? a[base + j] : 0.0f;
  }
}

__device__ __forceinline__ uint64_t run_base(uint64_t tile, int u) {
  return tile * kTopkBlock + (uint64_t)(u * kThreads + threadIdx.x) * kTopkElems;
}

// bit j set if value j of the run (inside the data) has a key >= lo
__device__ __forceinline__ uint32_t ge_mask(const float (&v)[kTopkElems], uint64_t base, uint64_t count,
                                            uint32_t lo) {
  uint32_t m = 0;
  const bool full = base + kTopkElems <= count;
#pragma unroll
  for (int j = 0; j < kTopkElems; ++j)
    if (mag_key(v[j]) >= lo && (full || base + j < count)) m |= 1u << j;
  return m;
}

// Slot positions of a tile's four runs per thread, in index order (all runs
// of u = 0, then u = 1, ...), with one barrier: each warp scans its lanes'
// counts with shuffles (runs 0 and 1, and 2 and 3, packed as two 16-bit
// fields), publishes its four totals, and every thread adds up the totals of
// the earlier runs and of the earlier warps. `tot` is a per-block buffer of
// 2 x kWarps x 4 words used alternately by consecutive tiles (`parity`), so a
// warp may start writing the next tile's totals while a slower one still
// reads this tile's. Returns the tile's total in *n.
__device__ __forceinline__ void run_positions(const uint32_t (&m)[kTopkRuns], uint32_t* tot, int parity,
                                              uint32_t (&pos)[kTopkRuns], uint32_t* n) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const uint32_t mine01 = (uint32_t)__popc(m[0]) | ((uint32_t)__popc(m[1]) << 16);
  const uint32_t mine23 = (uint32_t)__popc(m[2]) | ((uint32_t)__popc(m[3]) << 16);
  uint32_t s01 = mine01, s23 = mine23;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t a = __shfl_up_sync(0xffffffffu, s01, o), b = __shfl_up_sync(0xffffffffu, s23, o);
    if (lane >= o) {
      s01 += a;
      s23 += b;
    }
  }
  uint32_t* t = tot + parity * (kWarps * 4);
  if (lane == 31) {  // the warp's totals per run (at most 512 each: no field overflows)
    t[wid * 4 + 0] = s01 & 0xFFFFu;
    t[wid * 4 + 1] = s01 >> 16;
    t[wid * 4 + 2] = s23 & 0xFFFFu;
    t[wid * 4 + 3] = s23 >> 16;
  }
  __syncthreads();
  uint32_t run_tot[kTopkRuns] = {0, 0, 0, 0}, before[kTopkRuns] = {0, 0, 0, 0};
#pragma unroll
  for (int w2 = 0; w2 < kWarps; ++w2) {
#pragma unroll
    for (int u = 0; u < kTopkRuns; ++u) {
      const uint32_t v = t[w2 * 4 + u];
      run_tot[u] += v;
      if (w2 < wid) before[u] += v;
    }
  }
  const uint32_t ex01 = s01 - mine01, ex23 = s23 - mine23;
  pos[0] = before[0] + (ex01 & 0xFFFFu);
  pos[1] = run_tot[0] + before[1] + (ex01 >> 16);
  pos[2] = run_tot[0] + run_tot[1] + before[2] + (ex23 & 0xFFFFu);
  pos[3] = run_tot[0] + run_tot[1] + run_tot[2] + before[3] + (ex23 >> 16);
  *n = run_tot[0] + run_tot[1] + run_tot[2] + run_tot[3];
}

// Pass 2, a resident grid looping over the tiles: each tile's keys at or
// above the first digit's bin (every key that can still be kept) compacted in
// index order into the tile's slots, and the histogram of bits 19..10 of the
// keys inside that bin; then (last block) the second digit. The sparse work
// runs over the set bits of each run's mask, re-reading those few values
// from the cache.
template <bool VEC>
__global__ void __launch_bounds__(kThreads) k_topk_split(const __grid_constant__ TopkArgs A) {
  pdl_begin();
  __shared__ uint32_t sh[1024];
  __shared__ uint32_t tot[2 * kWarps * 4];
  int parity = 0;
  const int r = blockIdx.y;
  const RankWs w = rank_ws(A, r);
  if (w.st->pre2) return;  // pass 1 found the second digit (the same for the whole block)
  const uint64_t count = A.count;
  const float* __restrict__ a = A.e[r];
  const uint32_t S = A.slots;
  for (int i = threadIdx.x; i < 1024; i += blockDim.x) sh[i] = 0;
  const uint32_t d1 = w.st->prefix >> 20;
  const uint32_t lo = d1 << 20;
  __syncthreads();
  if (w.st->spec_ok) {
    // pass 1 left every candidate in the slots: only the histogram of bits
    // 19..10 of the keys in the first digit's bin, from the slots (a warp per
    // tile, eight slot loads in flight per lane)
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    for (uint64_t tile = (uint64_t)blockIdx.x * kWarps + wid; tile < A.nb; tile += (uint64_t)gridDim.x * kWarps) {
      const float* sv = slot_val(w, tile, S);
      const uint32_t n = w.n_s[tile];
      for (uint32_t c0 = 0; c0 < n; c0 += 32 * 8) {
        uint32_t key[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint32_t c = c0 + 32 * u + lane;
          key[u] = c < n ? mag_key(sv[c]) : 0u;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (c0 + 32 * u + lane < n && (key[u] >> 20) == d1) atomicAdd(&sh[(key[u] >> 10) & 1023u], 1u);
      }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 1024; i += blockDim.x)
      if (sh[i]) atomicAdd(&w.hist[i], sh[i]);
    if (last_block(&w.st->ticket[1])) find_digit<1024>(w.hist, 10, w.st);
    return;
  }
  // highest tiles first: pass 1 wrote them last, so some are still in L2
  for (uint64_t step = blockIdx.x; step < A.nb; step += gridDim.x) {
    const uint64_t tile = A.nb - 1 - step;
    uint32_t m[kTopkRuns];
    if (VEC && (tile + 1) * kTopkBlock <= count) {
      // a whole tile: no bounds checks (the same for every thread of the block)
      const float4* p = reinterpret_cast<const float4*>(a + tile * kTopkBlock);
      float4 x[kTopkRuns][kTopkElems / 4];
#pragma unroll
      for (int u = 0; u < kTopkRuns; ++u)
#pragma unroll
        for (int q = 0; q < kTopkElems / 4; ++q) x[u][q] = p[(u * kThreads + threadIdx.x) * (kTopkElems / 4) + q];
#pragma unroll
      for (int u = 0; u < kTopkRuns; ++u) {
        uint32_t b = 0;
#pragma unroll
        for (int q = 0; q < kTopkElems / 4; ++q) {
          if (mag_key(x[u][q].x) >= lo) b |= 1u << (4 * q);
          if (mag_key(x[u][q].y) >= lo) b |= 2u << (4 * q);
          if (mag_key(x[u][q].z) >= lo) b |= 4u << (4 * q);
          if (mag_key(x[u][q].w) >= lo) b |= 8u << (4 * q);
        }
        m[u] = b;
      }
    } else {
      float v[kTopkRuns][kTopkElems];
#pragma unroll
      for (int u = 0; u < kTopkRuns; ++u) load_run<VEC>(a, run_base(tile, u), count, v[u]);
#pragma unroll
      for (int u = 0; u < kTopkRuns; ++u) m[u] = ge_mask(v[u], run_base(tile, u), count, lo);
    }
    uint32_t pos[kTopkRuns], ntile;
    run_positions(m, tot, parity, pos, &ntile);
    parity ^= 1;
    uint32_t* __restrict__ si = slot_idx(w, tile, S);
    float* __restrict__ sv = slot_val(w, tile, S);
#pragma unroll
    for (int u = 0; u < kTopkRuns; ++u) {
      const uint64_t base = run_base(tile, u);
      uint32_t bits = m[u];
      uint32_t p = pos[u];
      while (bits) {
        const int j = __ffs(bits) - 1;
        bits &= bits - 1;
        const float x = a[base + j];
        const uint32_t key = mag_key(x);
        if ((key >> 20) == d1) atomicAdd(&sh[(key >> 10) & 1023u], 1u);
        if (p < S) {
          si[p] = (uint32_t)(base + j);
          sv[p] = x;
        }
        ++p;
      }
    }
    if (threadIdx.x == 0) {
      w.n_s[tile] = ntile;
      if (ntile > S) atomicOr(&w.st->overflow, 1u);
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 1024; i += blockDim.x)
    if (sh[i]) atomicAdd(&w.hist[i], sh[i]);
  if (last_block(&w.st->ticket[1])) find_digit<1024>(w.hist, 10, w.st);
}

template <bool GLOBAL>
__device__ void scan_tiles(const RankWs& w, uint64_t nb, const uint32_t* gt, const uint32_t* eq);

// Pass 3: histogram of bits 9..0 among the keys that match the prefix, read
// from the slots (or, after an overflow, from the data); then (last block)
// the last digit, which completes T. From the slots, each tile's run is also
// compacted in place to the keys at or above the prefix (every key that can
// still be kept: about the tile's share of k), in index order, so that the
// count and the emission read only those; and the keys equal to the prefix
// in its 21 bits (few) are listed, so that the last block, once T is known,
// derives each tile's counts of keys above and equal to T from its run
// length and the list, and scans them: the count pass then has nothing to do.
template <bool VEC>
__global__ void __launch_bounds__(kThreads) k_topk_pass3(const __grid_constant__ TopkArgs A) {
  pdl_begin();
  __shared__ uint32_t sh[1024];
  const int r = blockIdx.y;
  const RankWs w = rank_ws(A, r);
  for (int i = threadIdx.x; i < 1024; i += blockDim.x) sh[i] = 0;
  __syncthreads();
  const uint32_t mask = w.st->mask, prefix = w.st->prefix;
  auto add = [&](float x) {
    const uint32_t key = mag_key(x);
    if ((key & mask) == prefix) atomicAdd(&sh[key & 1023u], 1u);
  };
  if (!w.st->overflow) {
    // one warp per tile, kP3 slots (index and value) loaded per lane before
    // any is written back: a kept entry moves to the count of kept entries
    // before it, never past an entry not yet loaded
    constexpr int kP3 = 16;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const uint32_t lt = (1u << lane) - 1u;
    const uint32_t cap = topk_match_cap(A.nb);
    uint32_t* list = w.masks + 1024;
    const float* er = A.e[r];
    for (uint64_t tile = (uint64_t)blockIdx.x * kWarps + wid; tile < A.nb; tile += (uint64_t)gridDim.x * kWarps) {
      uint32_t* si = slot_idx(w, tile, A.slots);
      float* sv = slot_val(w, tile, A.slots);
      const uint32_t n = w.n_s[tile];
      uint32_t kept = 0;
      for (uint32_t c0 = 0; c0 < n; c0 += 32 * kP3) {
        float x[kP3];
        uint32_t ii[kP3];
#pragma unroll
        for (int u = 0; u < kP3; ++u) {
          const uint32_t c = c0 + 32 * u + lane;
          x[u] = c < n ? sv[c] : 0.0f;
          ii[u] = c < n ? si[c] : 0u;
        }
        __syncwarp();
#pragma unroll
        for (int u = 0; u < kP3; ++u) {
          const uint32_t key = mag_key(x[u]);
          const bool in = c0 + 32 * u + lane < n;
          if (in && (key & mask) == prefix) {
            atomicAdd(&sh[key & 1023u], 1u);
            const uint32_t m = atomicAdd(&w.st->mcount, 1u);
            if (m < cap) {
              list[2 * m] = ii[u];
              list[2 * m + 1] = key;
            }
          }
          const bool keep = in && key >= prefix;
          const uint32_t bal = __ballot_sync(0xffffffffu, keep);
          if (keep) {
            const uint32_t p = kept + (uint32_t)__popc(bal & lt);
            si[p] = ii[u];
            sv[p] = x[u];
            // the emission zeroes this residual: bring its sector into L2 now
            asm volatile("prefetch.global.L2 [%0];" ::"l"(er + ii[u]));
          }
          kept += (uint32_t)__popc(bal);
        }
        __syncwarp();
      }
      if (lane == 0) w.n_s[tile] = kept;
    }
  } else {
    const float* __restrict__ a = A.e[r];
    const uint64_t count = A.count;
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    const uint64_t t0 = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    uint64_t done = 0;
    if (VEC) {
      const uint64_t n4 = count / 4;
      const float4* a4 = reinterpret_cast<const float4*>(a);
      for (uint64_t q = t0; q < n4; q += stride) {
        const float4 x = a4[q];
        add(x.x);
        add(x.y);
        add(x.z);
        add(x.w);
      }
      done = n4 * 4;
    }
    for (uint64_t i = done + t0; i < count; i += stride) add(a[i]);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 1024; i += blockDim.x)
    if (sh[i]) atomicAdd(&w.hist[i], sh[i]);
  if (last_block(&w.st->ticket[2])) {
    find_digit<1024>(w.hist, 0, w.st);
    __syncthreads();
    if (threadIdx.x == 0) {
      // the margin for the next call: wider after too few candidates,
      // narrower after a run of calls whose candidates served
      uint32_t level = w.st->margin & 0xFFu, run = w.st->margin >> 8;
      if (level >= (uint32_t)kTopkHintLevels) level = kTopkHintStart, run = 0;
      if (w.st->spec_ok) {
        if (++run >= kTopkTightenRun) {
          run = level > 0 ? 0 : kTopkTightenRun;
          if (level > 0) --level;
        }
      } else {
        run = 0;
        if (w.st->spec_count < A.k && level + 1 < (uint32_t)kTopkHintLevels) ++level;
      }
      w.st->margin = level | run << 8;
      // the next call's hint: T's magnitude scaled down by the margin (for
      // an infinity or a NaN, the infinity's key); and T itself
      const uint32_t T = w.st->prefix;
      w.st->hint =
          T >= 0x7F800000u ? 0x7F800000u : __float_as_uint(__fmul_rn(__uint_as_float(T), topk_hint_scale(level)));
      w.st->t_prev = T;
    }
    __syncthreads();
    const uint32_t m = __ldcg(&w.st->mcount);
    if (!w.st->overflow && m <= topk_match_cap(A.nb)) {  // the same for the whole block
      // each run holds the tile's keys at or above the prefix: all above T
      // but the listed ones at or below it. Up to 512 tiles the counts stay
      // in this block's shared memory (the histogram is done with).
      const uint32_t T = w.st->prefix;
      const bool smem = A.nb <= 512;
      uint32_t* gt = smem ? sh : w.n_gt;
      uint32_t* eq = smem ? sh + 512 : w.n_eq;
      for (uint64_t t = threadIdx.x; t < A.nb; t += blockDim.x) {
        gt[t] = __ldcg(w.n_s + t);
        eq[t] = 0;
      }
      __syncthreads();
      const uint32_t* list = w.masks + 1024;
      for (uint32_t i = threadIdx.x; i < m; i += blockDim.x) {
        const uint32_t key = __ldcg(list + 2 * i + 1);
        const uint64_t t = __ldcg(list + 2 * i) / kTopkBlock;
        if (key <= T) atomicSub(gt + t, 1u);
        if (key == T) atomicAdd(eq + t, 1u);
      }
      __syncthreads();
      if (smem)
        scan_tiles<false>(w, A.nb, gt, eq);
      else
        scan_tiles<true>(w, A.nb, gt, eq);
      if (threadIdx.x == 0) w.st->counted = 1;
    }
  }
}

// run mask: bit j set if value j's key is above T, bit 16 + j if it equals T
__device__ __forceinline__ uint32_t run_mask(const float (&v)[kTopkElems], uint64_t base, uint64_t count,
                                             uint32_t T) {
  static_assert(kTopkElems == 16, "one 32-bit mask word per run");
  uint32_t m = 0;
#pragma unroll
  for (int j = 0; j < kTopkElems; ++j) {
    if (base + j < count) {
      const uint32_t key = mag_key(v[j]);
      m |= (key > T ? 1u : 0u) << j;
      m |= (key == T ? 1u : 0u) << (16 + j);
    }
  }
  return m;
}

// keys above T (low 16 bits) and equal to T (high 16 bits) of a run mask
__device__ __forceinline__ uint32_t mask_counts(uint32_t m) {
  return (uint32_t)__popc(m & 0xFFFFu) | ((uint32_t)__popc(m >> 16) << 16);
}

// The count pass's last block: eq_before[b] = keys equal to T in earlier
// tiles; out_off[b] = kept elements in earlier tiles, where tile b keeps all
// its keys above T and min(eq[b], max(0, need - eq_before[b])) of its keys
// equal to T, gt[b] and eq[b] being its keys above and equal to T (global
// arrays read through L2, or shared memory). Each thread scans a contiguous
// run of tiles.
template <bool GLOBAL>
__device__ void scan_tiles(const RankWs& w, uint64_t nb, const uint32_t* gt, const uint32_t* eq) {
  auto ld = [](const uint32_t* p) { return GLOBAL ? __ldcg(p) : *p; };
  const uint32_t need = w.st->need;
  const uint64_t m = (nb + kThreads - 1) / kThreads;
  const uint64_t lo = (uint64_t)threadIdx.x * m < nb ? (uint64_t)threadIdx.x * m : nb;
  const uint64_t hi = lo + m < nb ? lo + m : nb;
  uint32_t se = 0;
  for (uint64_t b = lo; b < hi; ++b) se += ld(eq + b);
  const uint32_t eq0 = block_exclusive_scan(se, nullptr);
  auto take_of = [&](uint64_t b, uint32_t eqb) {
    const uint32_t e = ld(eq + b);
    const uint32_t rest = need > eqb ? need - eqb : 0u;
    return ld(gt + b) + (e < rest ? e : rest);
  };
  uint32_t st = 0;
  uint32_t eqb = eq0;
  for (uint64_t b = lo; b < hi; ++b) {
    st += take_of(b, eqb);
    eqb += ld(eq + b);
  }
  uint32_t off = block_exclusive_scan(st, nullptr);
  eqb = eq0;
  for (uint64_t b = lo; b < hi; ++b) {
    const uint32_t t = take_of(b, eqb);
    w.eq_before[b] = eqb;
    w.out_off[b] = off;
    off += t;
    eqb += ld(eq + b);
  }
}

// Keys above T and equal to T per tile, unless pass 3 derived them. From the
// slots: one warp per tile. After an overflow: the block takes its kWarps
// tiles one after another from the data, writing the run masks. The last
// block scans all tiles' counts.
template <bool VEC>
__global__ void __launch_bounds__(kThreads) k_topk_count(const __grid_constant__ TopkArgs A) {
  pdl_begin();
  const int r = blockIdx.y;
  const RankWs w = rank_ws(A, r);
  if (w.st->counted) return;  // pass 3 did it (the same for the whole block)
  const uint32_t T = w.st->prefix;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  if (!w.st->overflow) {
    const uint64_t tile = (uint64_t)blockIdx.x * kWarps + wid;
    if (tile < A.nb) {
      const float* sv = slot_val(w, tile, A.slots);
      const uint32_t n = w.n_s[tile];
      uint32_t gt = 0, eq = 0;
      for (uint32_t c0 = 0; c0 < n; c0 += 32 * 8) {  // eight slot loads in flight per lane
        uint32_t key[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint32_t c = c0 + 32 * u + lane;
          key[u] = c < n ? mag_key(sv[c]) : 0u;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const bool in = c0 + 32 * u + lane < n;
          gt += in && key[u] > T;
          eq += in && key[u] == T;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        gt += __shfl_xor_sync(0xffffffffu, gt, o);
        eq += __shfl_xor_sync(0xffffffffu, eq, o);
      }
      if (lane == 0) {
        w.n_gt[tile] = gt;
        w.n_eq[tile] = eq;
      }
    }
  } else {
    for (int t = 0; t < kWarps; ++t) {
      const uint64_t tile = (uint64_t)blockIdx.x * kWarps + t;
      if (tile >= A.nb) break;  // uniform across the block
      float v[kTopkRuns][kTopkElems];
#pragma unroll
      for (int u = 0; u < kTopkRuns; ++u) load_run<VEC>(A.e[r], run_base(tile, u), A.count, v[u]);
      uint32_t c = 0;
#pragma unroll
      for (int u = 0; u < kTopkRuns; ++u) {
        const uint32_t m = run_mask(v[u], run_base(tile, u), A.count, T);
        w.masks[tile * kThreads * kTopkRuns + u * kThreads + threadIdx.x] = m;
        c += mask_counts(m);
      }
      uint32_t tot;
      block_exclusive_scan(c, &tot);  // no field overflows: at most kTopkBlock = 16384 each
      if (threadIdx.x == 0) {
        w.n_gt[tile] = tot & 0xFFFFu;
        w.n_eq[tile] = tot >> 16;
      }
    }
  }
  if (last_block(&w.st->ticket[3])) scan_tiles<true>(w, A.nb, w.n_gt, w.n_eq);
}

// Emission from the slots, one warp per tile: the slots are in index order,
// so the kept ones (above T, or equal to T while their rank among all keys
// equal to T is below `need`) are written in order with warp ballots.
__device__ void emit_slots(const TopkArgs& A, const RankWs& w, int r) {
  const int lane = threadIdx.x & 31;
  const uint64_t tile = (uint64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (tile >= A.nb) return;
  const uint32_t T = w.st->prefix, need = w.st->need;
  const uint32_t* si = slot_idx(w, tile, A.slots);
  const float* sv = slot_val(w, tile, A.slots);
  const uint32_t n = w.n_s[tile];
  uint32_t eq_run = w.eq_before[tile], pos_run = w.out_off[tile];
  float* __restrict__ e = A.e[r];
  uint32_t* __restrict__ idx = A.idx[r];
  float* __restrict__ val = A.val[r];
  const uint32_t lt = (1u << lane) - 1u;
  constexpr int U = 8;  // rounds of 32 slots whose loads are issued together
  for (uint32_t c0 = 0; c0 < n; c0 += 32 * U) {
    float x[U];
    uint32_t ii[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint32_t c = c0 + 32 * u + lane;
      x[u] = c < n ? sv[c] : 0.0f;
      ii[u] = c < n ? si[c] : 0u;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint32_t c = c0 + 32 * u + lane;
      const uint32_t key = mag_key(x[u]);
      const bool eq = c < n && key == T;
      const uint32_t eq_bal = __ballot_sync(0xffffffffu, eq);
      const bool keep = c < n && (key > T || (eq && eq_run + (uint32_t)__popc(eq_bal & lt) < need));
      const uint32_t keep_bal = __ballot_sync(0xffffffffu, keep);
      const uint32_t p = pos_run + (uint32_t)__popc(keep_bal & lt);
      if (keep && p < A.k) {  // p < k always holds; the test keeps every write inside idx and val
        idx[p] = ii[u];
        val[p] = x[u];
        e[ii[u]] = 0.0f;
      }
      eq_run += (uint32_t)__popc(eq_bal);
      pos_run += (uint32_t)__popc(keep_bal);
    }
  }
}

// Emission from the run masks (after an overflow), one tile: values are
// read where a key is kept. Called by the whole block.
__device__ void emit_masks(const TopkArgs& A, const RankWs& w, int r, uint64_t tile) {
  uint32_t m[kTopkRuns];
#pragma unroll
  for (int u = 0; u < kTopkRuns; ++u) m[u] = w.masks[tile * kThreads * kTopkRuns + u * kThreads + threadIdx.x];
  const uint32_t need = w.st->need;
  const uint32_t eq_block = w.eq_before[tile];
  const uint32_t off_block = w.out_off[tile];
  // runs in index order: all of u = 0, then u = 1, ...; ex[u] = the counts of
  // the tile's runs before run (u, this thread)
  uint32_t ex[kTopkRuns];
  uint32_t carry = 0;
#pragma unroll
  for (int u = 0; u < kTopkRuns; ++u) {
    uint32_t tot;
    ex[u] = carry + block_exclusive_scan(mask_counts(m[u]), &tot);
    carry += tot;
  }
  float* __restrict__ a = A.e[r];
  uint32_t* __restrict__ idx = A.idx[r];
  float* __restrict__ val = A.val[r];
#pragma unroll
  for (int u = 0; u < kTopkRuns; ++u) {
    if (m[u] == 0) continue;
    // kept before this run: every key above T in earlier runs of the tile,
    // and the keys equal to T whose rank among all equal keys is below `need`
    const uint32_t eq_in_tile = ex[u] >> 16;
    const uint32_t eq_kept = need > eq_block ? min(eq_in_tile, need - eq_block) : 0u;
    uint32_t pos = off_block + (ex[u] & 0xFFFFu) + eq_kept;
    uint32_t eq_rank = eq_block + eq_in_tile;
    uint32_t keep = m[u] & 0xFFFFu;
#pragma unroll
    for (int j = 0; j < kTopkElems; ++j) {
      if ((m[u] >> (16 + j)) & 1u) {
        if (eq_rank < need) keep |= 1u << j;
        ++eq_rank;
      }
    }
    const uint64_t base = run_base(tile, u);
    while (keep) {
      const int j = __ffs(keep) - 1;
      keep &= keep - 1;
      if (pos >= A.k) break;  // never taken; keeps every write inside idx and val
      idx[pos] = (uint32_t)(base + j);
      val[pos] = a[base + j];
      a[base + j] = 0.0f;
      ++pos;
    }
  }
}

// Kept elements to (index, value) in index order; zero their residual. Each
// block covers kWarps tiles.
__global__ void __launch_bounds__(kThreads) k_topk_emit(const __grid_constant__ TopkArgs A) {
  pdl_begin();
  const int r = blockIdx.y;
  const RankWs w = rank_ws(A, r);
  if (!w.st->overflow) {
    emit_slots(A, w, r);
  } else {
    for (int t = 0; t < kWarps; ++t) {
      const uint64_t tile = (uint64_t)blockIdx.x * kWarps + t;
      if (tile >= A.nb) break;  // uniform across the block
      emit_masks(A, w, r, tile);
    }
  }
}

// recv[r][idx_r[j]] = val_r[j] for every rank (outputs already zeroed)
__global__ void __launch_bounds__(kThreads) k_sparse_scatter(const __grid_constant__ ScatterArgs A) {
  pdl_begin();
  const uint32_t total = A.tile_start[A.nranks];
  for (uint32_t tile = blockIdx.x; tile < total; tile += gridDim.x) {
    int lo = 0, hi = A.nranks - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (A.tile_start[mid] <= tile) lo = mid;
      else hi = mid - 1;
    }
    const uint64_t j = (uint64_t)(tile - A.tile_start[lo]) * kThreads + threadIdx.x;
    if (j < A.nnz[lo]) {
      const uint32_t ix = A.idx[lo][j];
      if (ix < A.count) A.dst[lo][ix] = A.val[lo][j];
    }
  }
}

// Tile starts of the sparse fold: for each pair position p of rank r
// (0 <= p <= nnz), starts[t] = p for the tiles t after the tile of pair p - 1
// up to the tile of pair p (pairs with an index >= count, and p = nnz, count
// as tile ntiles). A thread takes four consecutive positions, its five index
// loads issued together. With ascending indices every entry is written once;
// otherwise the fold clamps what it reads.
constexpr int kBoundsPerThread = 4;

__global__ void __launch_bounds__(kThreads) k_sparse_bounds(const __grid_constant__ SparseArgs A) {
  pdl_begin();
  const int r = blockIdx.y;
  const uint64_t nnz = A.nnz[r];
  const uint64_t p0 = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) * kBoundsPerThread;
  if (p0 > nnz) return;
  const uint32_t* __restrict__ ix = A.idx[r];
  // tiles of pairs p0 - 1 .. p0 + 3 (-1 before the first pair, ntiles past the last)
  int64_t tl[kBoundsPerThread + 1];
#pragma unroll
  for (int u = 0; u <= kBoundsPerThread; ++u) {
    const uint64_t q = p0 + u - 1;  // wraps to 2^64 - 1 for p0 = 0, u = 0
    uint32_t i = 0;
    if (q < nnz) i = ix[q];
    tl[u] = (u == 0 && p0 == 0) ? -1
          : (q >= nnz || i >= A.count) ? (int64_t)A.ntiles : (int64_t)(i / A.tile);
  }
  uint32_t* st = A.starts + (uint64_t)r * (A.ntiles + 1);
#pragma unroll
  for (int u = 0; u < kBoundsPerThread; ++u) {
    const uint64_t p = p0 + u;
    if (p > nnz) break;
    for (int64_t t = tl[u] + 1; t <= tl[u + 1]; ++t) st[t] = (uint32_t)p;
  }
}

// resident blocks of k_sparse_fold (24 KiB of shared memory each): the ring
// order fits 32 registers, eight blocks of 256 threads; the recursive
// halving 48 (a 12-byte spill, measured faster than 64 registers at 4 blocks)
template <bool TREE> constexpr int kSparseBlocksPerSm = TREE ? 5 : 8;

// One tile per block: every rank's pairs of the tile scattered into shared
// memory (zeros elsewhere), folded per element in the ring order of its
// chunk (or recursive halving), divided by N for AVG, and stored to all N
// outputs. The dense allreduce of the densified vectors gives the same bits.
template <bool TREE>
__global__ void __launch_bounds__(kThreads, kSparseBlocksPerSm<TREE>) k_sparse_fold(const __grid_constant__ SparseArgs A) {
  pdl_wait();  // seven waves: the next call's kernels launch as its last blocks exit
  extern __shared__ float sm[];  // nranks x tile
  const int N = A.nranks;
  const uint32_t T = A.tile;
  const uint64_t t = blockIdx.x;
  const uint64_t i0 = t * T;
  const uint32_t len = (uint32_t)(A.count - i0 < T ? A.count - i0 : T);
  // one warp per rank, so that the ranks' short lists are read concurrently;
  // the first rank's tile bounds are requested before the zeroing
  const int lane = threadIdx.x & 31;
  const int wr = threadIdx.x >> 5;
  uint32_t b0 = 0, b1 = 0;
  if (wr < N) {
    const uint32_t* st = A.starts + (uint64_t)wr * (A.ntiles + 1);
    b0 = st[t];
    b1 = st[t + 1];
  }
  float4* sm4 = reinterpret_cast<float4*>(sm);
  for (uint32_t q = threadIdx.x; q < (uint32_t)N * T / 4; q += blockDim.x) sm4[q] = make_float4(0.f, 0.f, 0.f, 0.f);
  __syncthreads();
  for (int r = wr; r < N; r += kWarps) {
    if (r != wr) {
      const uint32_t* st = A.starts + (uint64_t)r * (A.ntiles + 1);
      b0 = st[t];
      b1 = st[t + 1];
    }
    const uint64_t nnz = A.nnz[r];
    const uint64_t s = b0 < nnz ? b0 : nnz;
    const uint64_t e = b1 < nnz ? (b1 > s ? b1 : s) : nnz;
    const uint32_t* __restrict__ ix = A.idx[r];
    const float* __restrict__ vx = A.val[r];
    for (uint64_t p = s + lane; p < e; p += 32) {
      const uint64_t d = (uint64_t)ix[p] - i0;
      if (d < len) sm[(uint32_t)r * T + (uint32_t)d] = vx[p];
    }
  }
  __syncthreads();
  // four consecutive elements per thread: one chunk (L is a multiple of 4)
  const float4* s4 = reinterpret_cast<const float4*>(sm);
  float4* w4 = reinterpret_cast<float4*>(sm);
  const uint32_t T4 = T / 4;
  for (uint32_t q = threadIdx.x; q * 4 < len; q += blockDim.x) {
    const uint64_t i = i0 + 4ull * q;
    float4 acc;
    if (TREE) {
      for (int d = N >> 1; d >= 1; d >>= 1)
        for (int r = 0; r < d; ++r) {
          const float4 x = s4[(uint32_t)r * T4 + q], y = s4[(uint32_t)(r + d) * T4 + q];
          w4[(uint32_t)r * T4 + q] =
              make_float4(__fadd_rn(x.x, y.x), __fadd_rn(x.y, y.y), __fadd_rn(x.z, y.z), __fadd_rn(x.w, y.w));
        }
      acc = s4[q];
    } else {
      const uint32_t c = (uint32_t)i / (uint32_t)A.L;  // indices fit 32 bits
      int r = (int)c + 1 >= N ? (int)c + 1 - N : (int)c + 1;
      acc = s4[(uint32_t)r * T4 + q];
      for (int j = 1; j < N; ++j) {
        r = r + 1 == N ? 0 : r + 1;
        const float4 y = s4[(uint32_t)r * T4 + q];
        acc = make_float4(__fadd_rn(acc.x, y.x), __fadd_rn(acc.y, y.y), __fadd_rn(acc.z, y.z), __fadd_rn(acc.w, y.w));
      }
    }
    if (A.avg) acc = make_float4(avg_div(acc.x, N), avg_div(acc.y, N), avg_div(acc.z, N), avg_div(acc.w, N));
    if (A.vec && 4 * q + 4 <= len) {
      for (int r = 0; r < N; ++r) __stcs(reinterpret_cast<float4*>(A.dst[r] + i), acc);
    } else {
      const float o[4] = {acc.x, acc.y, acc.z, acc.w};
      for (int r = 0; r < N; ++r)
        for (uint32_t l = 0; l < 4 && 4 * q + l < len; ++l) A.dst[r][i + l] = o[l];
    }
  }
}

template <bool VEC>
cudaError_t launch_topk_t(const TopkArgs& a, cudaStream_t s) {
  int sms = 0;
  cudaError_t err = sm_count(&sms);
  if (err != cudaSuccess) return err;
  const dim3 one(1, a.nranks);
  err = launch_pdl(k_topk_init, one, 0, s, a);
  if (err != cudaSuccess) return err;
  // histogram passes over the data: a resident grid looping over it, so that
  // each block flushes its shared histogram once
  const uint64_t items = VEC ? (a.count + 3) / 4 : a.count;
  unsigned per_rank = (unsigned)(sms * kHistBlocksPerSm / a.nranks);
  if (per_rank < 1) per_rank = 1;
  const unsigned hx = grid_for(items) < per_rank ? grid_for(items) : per_rank;
  const dim3 hgrid(hx, a.nranks);
  unsigned p1 = (unsigned)(sms * kPass1BlocksPerSm / a.nranks);
  if (p1 < 1) p1 = 1;
  const unsigned p1x = grid_for(items) < p1 ? grid_for(items) : p1;
  // the speculative pass 1 takes a warp per tile: used when the tiles of all
  // ranks keep at least 16 warps per SM busy
  if (VEC && a.k > 0 && a.nb * (uint64_t)a.nranks >= (uint64_t)sms * 16) {
    unsigned sbx = (unsigned)(sms * kSpecBlocksPerSm / a.nranks);
    if (sbx < 1) sbx = 1;
    err = launch_pdl(k_topk_pass1_spec, dim3(sbx, a.nranks), 0, s, a);
  } else {
    err = launch_pdl(k_topk_pass1<VEC>, dim3(p1x, a.nranks), 0, s, a);
  }
  if (err != cudaSuccess) return err;
  if (a.k == 0) return cudaSuccess;  // nothing kept: e = a
  unsigned sx = (unsigned)(sms * kSplitBlocksPerSm / a.nranks);
  if (sx < 1) sx = 1;
  if (sx > a.nb) sx = (unsigned)a.nb;
  if ((err = launch_pdl(k_topk_split<VEC>, dim3(sx, a.nranks), 0, s, a)) != cudaSuccess) return err;
  if ((err = launch_pdl(k_topk_pass3<VEC>, hgrid, 0, s, a)) != cudaSuccess) return err;
  const dim3 wgrid((unsigned)((a.nb + kWarps - 1) / kWarps), a.nranks);
  if ((err = launch_pdl(k_topk_count<VEC>, wgrid, 0, s, a)) != cudaSuccess) return err;
  return launch_pdl(k_topk_emit, wgrid, 0, s, a);
}

}  // namespace

cudaError_t launch_topk(const TopkArgs& a, bool vec, cudaStream_t stream) {
  return vec ? launch_topk_t<true>(a, stream) : launch_topk_t<false>(a, stream);
}

cudaError_t launch_sparse_fold(const SparseArgs& a, uint64_t max_nnz, cudaStream_t stream) {
  const cudaError_t err = launch_pdl(
      k_sparse_bounds, dim3(grid_for((max_nnz + kBoundsPerThread) / kBoundsPerThread), a.nranks), 0, stream, a);
  if (err != cudaSuccess) return err;
  const size_t smem = (size_t)a.nranks * a.tile * sizeof(float);
  return a.tree ? launch_pdl(k_sparse_fold<true>, dim3(a.ntiles), smem, stream, a)
                : launch_pdl(k_sparse_fold<false>, dim3(a.ntiles), smem, stream, a);
}

cudaError_t launch_sparse_scatter(const ScatterArgs& a, cudaStream_t stream) {
  const uint32_t total = a.tile_start[a.nranks];
  if (total == 0) return cudaSuccess;
  k_sparse_scatter<<<total, kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace gar

// ---------------------------------------------------------------------------
// C ABI
// ---------------------------------------------------------------------------
namespace {

ar_status_t tk_fail(ar_status_t st, const std::string& msg) {
  gar::set_last_error(msg);
  return st;
}
// a CUDA error, reported here and taken off the runtime's last-error slot
ar_status_t tk_cuda_fail(const char* what, cudaError_t e) {
  (void)cudaGetLastError();
  return tk_fail(AR_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}
ar_status_t tk_ok() {
  gar::set_last_error("");
  return AR_SUCCESS;
}
uintptr_t tk_addr(const void* p) { return reinterpret_cast<uintptr_t>(p); }

struct Rng {
  uintptr_t lo, hi;
};
// true if any two of the ranges overlap
bool any_overlap(std::vector<Rng> v) {
  std::vector<Rng> s;
  for (const Rng& x : v)
    if (x.hi > x.lo) s.push_back(x);
  std::sort(s.begin(), s.end(), [](const Rng& a, const Rng& b) { return a.lo < b.lo; });
  for (size_t i = 1; i < s.size(); ++i)
    if (s[i].lo < s[i - 1].hi) return true;
  return false;
}

}  // namespace

extern "C" {

size_t ar_topk_workspace_bytes(int nranks, size_t count, size_t k) {
  if (nranks < 1 || nranks > AR_MAX_RANKS || count > 0xFFFFFFFFull || k > count) return 0;
  return (size_t)nranks * gar::topk_rank_words(count, k) * 4;
}

ar_status_t ar_topk_compress(const float* const* grads, float* const* residuals, int nranks, size_t count, size_t k,
                             uint32_t* const* idx, float* const* val, void* workspace, size_t ws_bytes,
                             ar_stream_t stream) {
  AR_TRACE("ar_topk_compress");
  if (!grads || !residuals || !idx || !val) return tk_fail(AR_ERR_INVALID_ARGUMENT, "null buffer array");
  if (nranks < 1 || nranks > AR_MAX_RANKS) return tk_fail(AR_ERR_INVALID_ARGUMENT, "nranks must be in 1..64");
  if (count > 0xFFFFFFFFull) return tk_fail(AR_ERR_INVALID_ARGUMENT, "count must fit 32-bit indices");
  if (k > count) return tk_fail(AR_ERR_INVALID_ARGUMENT, "k exceeds count");
  if (count == 0) return tk_ok();
  const size_t need = ar_topk_workspace_bytes(nranks, count, k);
  if (!workspace) return tk_fail(AR_ERR_INVALID_ARGUMENT, "null workspace");
  if (tk_addr(workspace) % 16) return tk_fail(AR_ERR_INVALID_ARGUMENT, "workspace must be 16-byte aligned");
  if (ws_bytes < need) return tk_fail(AR_ERR_INVALID_ARGUMENT, "workspace too small");
  const size_t b = count * 4, kb = k * 4;
  std::vector<Rng> outs = {{tk_addr(workspace), tk_addr(workspace) + need}};
  gar::TopkArgs a{};
  bool vec = true;
  for (int r = 0; r < nranks; ++r) {
    if (!grads[r] || !residuals[r] || (k > 0 && (!idx[r] || !val[r])))
      return tk_fail(AR_ERR_INVALID_ARGUMENT, "null buffer of rank " + std::to_string(r));
    if (tk_addr(grads[r]) % 4 || tk_addr(residuals[r]) % 4 || tk_addr(idx[r]) % 4 || tk_addr(val[r]) % 4)
      return tk_fail(AR_ERR_INVALID_ARGUMENT, "buffer not aligned to its element size");
    vec = vec && tk_addr(grads[r]) % 16 == 0 && tk_addr(residuals[r]) % 16 == 0;
    outs.push_back({tk_addr(residuals[r]), tk_addr(residuals[r]) + b});
    outs.push_back({tk_addr(idx[r]), tk_addr(idx[r]) + kb});
    outs.push_back({tk_addr(val[r]), tk_addr(val[r]) + kb});
    a.g[r] = grads[r];
    a.e[r] = residuals[r];
    a.idx[r] = idx[r];
    a.val[r] = val[r];
  }
  // outputs are disjoint from each other and from every input (inputs may overlap each other)
  if (any_overlap(outs)) return tk_fail(AR_ERR_ALIAS, "buffers overlap");
  for (int r = 0; r < nranks; ++r) {
    std::vector<Rng> v = outs;
    v.push_back({tk_addr(grads[r]), tk_addr(grads[r]) + b});
    if (any_overlap(v)) return tk_fail(AR_ERR_ALIAS, "buffers overlap");
  }
  a.ws = static_cast<uint32_t*>(workspace);
  a.ws_words = gar::topk_rank_words(count, k);
  a.slots = gar::topk_slots(count, k);
  a.count = count;
  a.nb = gar::topk_blocks(count);
  a.k = (uint32_t)k;
  a.nranks = nranks;
  const cudaError_t e = gar::launch_topk(a, vec, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return tk_cuda_fail("top-k launch", e);
  return tk_ok();
}

size_t ar_sparse_workspace_bytes(int nranks, size_t count) {
  if (nranks < 1 || nranks > AR_MAX_RANKS || count > 0xFFFFFFFFull) return 0;
  return ((size_t)nranks * (gar::sparse_ntiles(count, nranks) + 1) * 4 + 255) / 256 * 256;
}

ar_status_t ar_sparse_allreduce(const uint32_t* const* idx, const float* const* val, const size_t* nnz, int nranks,
                                size_t count, ar_op_t op, ar_algo_t algo, float* const* recvbufs, void* workspace,
                                size_t ws_bytes, ar_stream_t stream) {
  AR_TRACE("ar_sparse_allreduce");
  if (!idx || !val || !nnz || !recvbufs) return tk_fail(AR_ERR_INVALID_ARGUMENT, "null array");
  if (nranks < 1 || nranks > AR_MAX_RANKS) return tk_fail(AR_ERR_INVALID_ARGUMENT, "nranks must be in 1..64");
  if (op < AR_SUM || op > AR_MAX) return tk_fail(AR_ERR_INVALID_ARGUMENT, "unknown op");
  if (algo < AR_ALGO_RING || algo > AR_ALGO_AUTO) return tk_fail(AR_ERR_INVALID_ARGUMENT, "unknown algo");
  if ((algo == AR_ALGO_TREE || algo == AR_ALGO_STEP_TREE) && (nranks & (nranks - 1)))
    return tk_fail(AR_ERR_UNSUPPORTED, "TREE needs nranks to be a power of two");
  if (count > 0xFFFFFFFFull) return tk_fail(AR_ERR_INVALID_ARGUMENT, "count must fit 32-bit indices");
  if (count == 0) return tk_ok();
  const bool fold = op == AR_SUM || op == AR_AVG;
  const size_t need = ar_sparse_workspace_bytes(nranks, count);
  if (fold) {
    if (!workspace) return tk_fail(AR_ERR_INVALID_ARGUMENT, "null workspace");
    if (tk_addr(workspace) % 16) return tk_fail(AR_ERR_INVALID_ARGUMENT, "workspace must be 16-byte aligned");
    if (ws_bytes < need) return tk_fail(AR_ERR_INVALID_ARGUMENT, "workspace too small");
  }
  const size_t b = count * 4;
  uint64_t tiles = 0, max_nnz = 0;
  gar::ScatterArgs a{};
  gar::SparseArgs f{};
  a.nranks = f.nranks = nranks;
  a.count = f.count = count;
  std::vector<Rng> outs;
  if (fold) outs.push_back({tk_addr(workspace), tk_addr(workspace) + need});
  for (int r = 0; r < nranks; ++r) {
    if (nnz[r] > count) return tk_fail(AR_ERR_INVALID_ARGUMENT, "nnz exceeds count");
    if (!recvbufs[r] || (nnz[r] > 0 && (!idx[r] || !val[r])))
      return tk_fail(AR_ERR_INVALID_ARGUMENT, "null buffer of rank " + std::to_string(r));
    if (tk_addr(recvbufs[r]) % 4 || tk_addr(idx[r]) % 4 || tk_addr(val[r]) % 4)
      return tk_fail(AR_ERR_INVALID_ARGUMENT, "buffer not aligned to its element size");
    outs.push_back({tk_addr(recvbufs[r]), tk_addr(recvbufs[r]) + b});
    a.idx[r] = f.idx[r] = idx[r];
    a.val[r] = f.val[r] = val[r];
    a.dst[r] = f.dst[r] = recvbufs[r];
    a.nnz[r] = f.nnz[r] = nnz[r];
    a.tile_start[r] = (uint32_t)tiles;
    tiles += (nnz[r] + gar::kThreads - 1) / gar::kThreads;
    if (nnz[r] > max_nnz) max_nnz = nnz[r];
  }
  a.tile_start[nranks] = (uint32_t)tiles;
  if (any_overlap(outs)) return tk_fail(AR_ERR_ALIAS, "buffers overlap");
  for (int r = 0; r < nranks; ++r) {
    std::vector<Rng> v = outs;
    v.push_back({tk_addr(idx[r]), tk_addr(idx[r]) + nnz[r] * 4});
    if (any_overlap(v)) return tk_fail(AR_ERR_ALIAS, "buffers overlap");
    v.back() = {tk_addr(val[r]), tk_addr(val[r]) + nnz[r] * 4};
    if (any_overlap(v)) return tk_fail(AR_ERR_ALIAS, "buffers overlap");
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (fold) {
    // one pass: densify each tile in shared memory, fold, store N replicas
    f.starts = static_cast<uint32_t*>(workspace);
    f.tile = gar::sparse_tile(nranks);
    f.ntiles = (uint32_t)gar::sparse_ntiles(count, nranks);
    f.L = (count / (size_t)nranks + (count % (size_t)nranks != 0) + 3) / 4 * 4;  // ar_allreduce's F32 chunk
    f.avg = op == AR_AVG;
    f.tree = algo == AR_ALGO_TREE || algo == AR_ALGO_STEP_TREE;
    f.vec = 1;
    for (int r = 0; r < nranks; ++r) f.vec = f.vec && tk_addr(recvbufs[r]) % 16 == 0;
    const cudaError_t e = gar::launch_sparse_fold(f, max_nnz, s);
    if (e != cudaSuccess) return tk_cuda_fail("sparse fold launch", e);
    return tk_ok();
  }
  // MIN / MAX: the dense forms in the outputs, then the dense allreduce in place
  for (int r = 0; r < nranks; ++r) {
    const cudaError_t e = cudaMemsetAsync(recvbufs[r], 0, b, s);
    if (e != cudaSuccess) return tk_cuda_fail("zeroing the outputs", e);
  }
  const cudaError_t e = gar::launch_sparse_scatter(a, s);
  if (e != cudaSuccess) return tk_cuda_fail("sparse scatter launch", e);
  std::vector<const void*> in(recvbufs, recvbufs + nranks);
  std::vector<void*> out(recvbufs, recvbufs + nranks);
  return ar_allreduce(in.data(), out.data(), nranks, count, AR_F32, op, algo, stream);
}

}  // extern "C"
