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
// comes from a three-pass radix select over the 31 magnitude bits — a
// histogram of bits 30..20 (fused with a = g + e), then of bits 19..10 and
// 9..0 among the keys that match the prefix found so far; after each
// histogram a one-thread kernel picks the digit, so the state never leaves
// the device. Keys above T are all kept; of the keys equal to T, the first
// (k - #above) in index order are kept: per-block counts, a one-block scan
// over the blocks, and block-wide scans give every kept element its slot.
#include <cstdint>
#include <string>
#include <vector>

#include "ar.h"
#include "ar_topk_internal.h"

namespace gar {

void set_last_error(const std::string& msg);

namespace {

constexpr int kTopkElems = 16;                     // elements per thread in count / emit
constexpr int kTopkBlock = kThreads * kTopkElems;  // elements per block in count / emit
constexpr int kHistBlocksPerSm = 8;
constexpr int kSms = 152;

__device__ __forceinline__ uint32_t mag_key(float a) { return __float_as_uint(a) & 0x7FFFFFFFu; }

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

// a = g + e into e, and the histogram of bits 30..20 of |a| (pass 1)
template <bool VEC>
__global__ void __launch_bounds__(kThreads) k_topk_add_hist(const float* __restrict__ g, float* __restrict__ e,
                                                            uint64_t count, uint32_t* __restrict__ hist) {
  __shared__ uint32_t sh[2048];
  for (int i = threadIdx.x; i < 2048; i += blockDim.x) sh[i] = 0;
  __syncthreads();
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  uint64_t done = 0;
  if (VEC) {
    const uint64_t n4 = count / 4;
    const float4* g4 = reinterpret_cast<const float4*>(g);
    float4* e4 = reinterpret_cast<float4*>(e);
    for (uint64_t q = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; q < n4; q += stride) {
      const float4 x = __ldcs(g4 + q);
      const float4 y = e4[q];
      float4 s;
      s.x = __fadd_rn(x.x, y.x);
      s.y = __fadd_rn(x.y, y.y);
      s.z = __fadd_rn(x.z, y.z);
      s.w = __fadd_rn(x.w, y.w);
      e4[q] = s;
      atomicAdd(&sh[mag_key(s.x) >> 20], 1u);
      atomicAdd(&sh[mag_key(s.y) >> 20], 1u);
      atomicAdd(&sh[mag_key(s.z) >> 20], 1u);
      atomicAdd(&sh[mag_key(s.w) >> 20], 1u);
    }
    done = n4 * 4;
  }
  for (uint64_t i = done + (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count; i += stride) {
    const float s = __fadd_rn(g[i], e[i]);
    e[i] = s;
    atomicAdd(&sh[mag_key(s) >> 20], 1u);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 2048; i += blockDim.x)
    if (sh[i]) atomicAdd(&hist[i], sh[i]);
}

// histogram of the 10-bit digit at `shift` among keys whose fixed bits match
template <bool VEC>
__global__ void __launch_bounds__(kThreads) k_topk_hist(const float* __restrict__ a, uint64_t count,
                                                        const TopkState* __restrict__ st, int shift,
                                                        uint32_t* __restrict__ hist) {
  __shared__ uint32_t sh[1024];
  for (int i = threadIdx.x; i < 1024; i += blockDim.x) sh[i] = 0;
  __syncthreads();
  const uint32_t mask = st->mask, prefix = st->prefix;
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  uint64_t done = 0;
  if (VEC) {
    const uint64_t n4 = count / 4;
    const float4* a4 = reinterpret_cast<const float4*>(a);
    for (uint64_t q = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; q < n4; q += stride) {
      const float4 x = a4[q];
      const uint32_t k0 = mag_key(x.x), k1 = mag_key(x.y), k2 = mag_key(x.z), k3 = mag_key(x.w);
      if ((k0 & mask) == prefix) atomicAdd(&sh[(k0 >> shift) & 1023u], 1u);
      if ((k1 & mask) == prefix) atomicAdd(&sh[(k1 >> shift) & 1023u], 1u);
      if ((k2 & mask) == prefix) atomicAdd(&sh[(k2 >> shift) & 1023u], 1u);
      if ((k3 & mask) == prefix) atomicAdd(&sh[(k3 >> shift) & 1023u], 1u);
    }
    done = n4 * 4;
  }
  for (uint64_t i = done + (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count; i += stride) {
    const uint32_t key = mag_key(a[i]);
    if ((key & mask) == prefix) atomicAdd(&sh[(key >> shift) & 1023u], 1u);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 1024; i += blockDim.x)
    if (sh[i]) atomicAdd(&hist[i], sh[i]);
}

// One thread: the highest digit whose count from the top reaches `need`;
// fold it into the prefix and clear the histogram for the next pass.
__global__ void k_topk_find(uint32_t* __restrict__ hist, int bins, int shift, TopkState* __restrict__ st) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  uint64_t above = 0;
  int b = bins - 1;
  for (; b > 0; --b) {
    if (above + hist[b] >= st->need) break;
    above += hist[b];
  }
  st->prefix |= (uint32_t)b << shift;
  st->mask |= (uint32_t)(bins - 1) << shift;
  st->need -= (uint32_t)above;
  st->gt += (uint32_t)above;
  for (int i = 0; i < bins; ++i) hist[i] = 0;
}

__global__ void k_topk_init(TopkState* st, uint32_t k) {
  if (threadIdx.x == 0 && blockIdx.x == 0) {
    st->prefix = 0;
    st->mask = 0;
    st->need = k;
    st->gt = 0;
  }
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

// per block of kTopkBlock elements: keys above T and keys equal to T
template <bool VEC>
__global__ void __launch_bounds__(kThreads) k_topk_count(const float* __restrict__ a, uint64_t count,
                                                         const TopkState* __restrict__ st, uint32_t* __restrict__ n_gt,
                                                         uint32_t* __restrict__ n_eq) {
  const uint32_t T = st->prefix;
  const uint64_t base = (uint64_t)blockIdx.x * kTopkBlock + (uint64_t)threadIdx.x * kTopkElems;
  float v[kTopkElems];
  load_run<VEC>(a, base, count, v);
  uint32_t gt = 0, eq = 0;
#pragma unroll
  for (int j = 0; j < kTopkElems; ++j) {
    if (base + j < count) {
      const uint32_t key = mag_key(v[j]);
      gt += key > T;
      eq += key == T;
    }
  }
  // gt and eq fit 16 bits each (at most kTopkBlock per block): one scan
  uint32_t tot;
  block_exclusive_scan(gt | (eq << 16), &tot);
  if (threadIdx.x == 0) {
    n_gt[blockIdx.x] = tot & 0xFFFFu;
    n_eq[blockIdx.x] = tot >> 16;
  }
}

// One block: eq_before[b] = keys equal to T in earlier blocks; out_off[b] =
// kept elements in earlier blocks, where block b keeps all its keys above T
// and min(n_eq[b], max(0, need - eq_before[b])) of its keys equal to T.
__global__ void __launch_bounds__(kThreads) k_topk_scan(const uint32_t* __restrict__ n_gt,
                                                        const uint32_t* __restrict__ n_eq, uint32_t nb,
                                                        const TopkState* __restrict__ st,
                                                        uint32_t* __restrict__ eq_before,
                                                        uint32_t* __restrict__ out_off) {
  const uint32_t need = st->need;
  uint32_t carry_eq = 0, carry_out = 0;
  for (uint32_t start = 0; start < nb; start += kThreads) {
    const uint32_t b = start + threadIdx.x;
    const uint32_t e = b < nb ? n_eq[b] : 0;
    uint32_t tot_e;
    const uint32_t ex_e = block_exclusive_scan(e, &tot_e) + carry_eq;
    uint32_t take = 0;
    if (b < nb) {
      const uint32_t rest = need > ex_e ? need - ex_e : 0;
      take = n_gt[b] + (e < rest ? e : rest);
      eq_before[b] = ex_e;
    }
    uint32_t tot_o;
    const uint32_t ex_o = block_exclusive_scan(take, &tot_o) + carry_out;
    if (b < nb) out_off[b] = ex_o;
    carry_eq += tot_e;
    carry_out += tot_o;
  }
}

// Kept elements to (index, value) in index order; zero their residual.
template <bool VEC>
__global__ void __launch_bounds__(kThreads) k_topk_emit(float* __restrict__ a, uint64_t count,
                                                        const TopkState* __restrict__ st,
                                                        const uint32_t* __restrict__ eq_before,
                                                        const uint32_t* __restrict__ out_off,
                                                        uint32_t* __restrict__ idx, float* __restrict__ val) {
  const uint32_t T = st->prefix, need = st->need;
  const uint64_t base = (uint64_t)blockIdx.x * kTopkBlock + (uint64_t)threadIdx.x * kTopkElems;
  float v[kTopkElems];
  load_run<VEC>(a, base, count, v);
  uint32_t gt = 0, eq = 0;
#pragma unroll
  for (int j = 0; j < kTopkElems; ++j) {
    if (base + j < count) {
      const uint32_t key = mag_key(v[j]);
      gt += key > T;
      eq += key == T;
    }
  }
  // the block's keys above T and equal to T before this thread's run
  const uint32_t ex = block_exclusive_scan(gt | (eq << 16), nullptr);
  uint32_t eq_rank = eq_before[blockIdx.x] + (ex >> 16);
  const uint32_t eq_in_block_before = ex >> 16;
  const uint32_t eq_block_before = eq_before[blockIdx.x];
  // kept before this thread in the block: all keys above T, plus the keys
  // equal to T whose rank among all equal keys is below `need`
  const uint32_t eq_kept_before =
      need > eq_block_before ? min(eq_in_block_before, need - eq_block_before) : 0u;
  uint32_t pos = out_off[blockIdx.x] + (ex & 0xFFFFu) + eq_kept_before;
  if (gt == 0 && eq == 0) return;
#pragma unroll
  for (int j = 0; j < kTopkElems; ++j) {
    const uint64_t i = base + j;
    if (i >= count) continue;
    const uint32_t key = mag_key(v[j]);
    bool keep = key > T;
    if (key == T) {
      keep = eq_rank < need;
      ++eq_rank;
    }
    if (keep) {
      idx[pos] = (uint32_t)i;
      val[pos] = v[j];
      a[i] = 0.0f;
      ++pos;
    }
  }
}

// recv[r][idx_r[j]] = val_r[j] for every rank (outputs already zeroed)
__global__ void __launch_bounds__(kThreads) k_sparse_scatter(const __grid_constant__ ScatterArgs A) {
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

}  // namespace

size_t topk_workspace_bytes(uint64_t count) {
  const uint64_t nb = (count + kTopkBlock - 1) / kTopkBlock;
  const uint64_t words = 2048 + 16 + 4 * nb;
  return (size_t)((words * 4 + 255) / 256 * 256);
}

cudaError_t launch_topk(const float* grad, float* residual, uint64_t count, uint64_t k, uint32_t* idx, float* val,
                        void* ws, cudaStream_t s) {
  uint32_t* hist = static_cast<uint32_t*>(ws);
  TopkState* st = reinterpret_cast<TopkState*>(hist + 2048);
  const uint64_t nb = (count + kTopkBlock - 1) / kTopkBlock;
  uint32_t* n_gt = hist + 2048 + 16;
  uint32_t* n_eq = n_gt + nb;
  uint32_t* eq_before = n_eq + nb;
  uint32_t* out_off = eq_before + nb;
  const bool vec = (reinterpret_cast<uintptr_t>(grad) % 16 == 0) && (reinterpret_cast<uintptr_t>(residual) % 16 == 0);
  // histogram kernels: a resident grid looping over the data, so that each
  // block's shared histogram is flushed once
  const uint64_t items = vec ? (count + 3) / 4 : count;
  const unsigned cap = kSms * kHistBlocksPerSm;
  const unsigned hgrid = grid_for(items) < cap ? grid_for(items) : cap;
  cudaError_t e = cudaMemsetAsync(hist, 0, 2048 * sizeof(uint32_t), s);
  if (e != cudaSuccess) return e;
  k_topk_init<<<1, 32, 0, s>>>(st, (uint32_t)k);
  if (vec) k_topk_add_hist<true><<<hgrid, kThreads, 0, s>>>(grad, residual, count, hist);
  else k_topk_add_hist<false><<<hgrid, kThreads, 0, s>>>(grad, residual, count, hist);
  if (k == 0) return cudaGetLastError();  // nothing kept: e = a
  k_topk_find<<<1, 32, 0, s>>>(hist, 2048, 20, st);
  for (int shift = 10; shift >= 0; shift -= 10) {
    if (vec) k_topk_hist<true><<<hgrid, kThreads, 0, s>>>(residual, count, st, shift, hist);
    else k_topk_hist<false><<<hgrid, kThreads, 0, s>>>(residual, count, st, shift, hist);
    k_topk_find<<<1, 32, 0, s>>>(hist, 1024, shift, st);
  }
  if (vec) k_topk_count<true><<<(unsigned)nb, kThreads, 0, s>>>(residual, count, st, n_gt, n_eq);
  else k_topk_count<false><<<(unsigned)nb, kThreads, 0, s>>>(residual, count, st, n_gt, n_eq);
  k_topk_scan<<<1, kThreads, 0, s>>>(n_gt, n_eq, (uint32_t)nb, st, eq_before, out_off);
  if (vec) k_topk_emit<true><<<(unsigned)nb, kThreads, 0, s>>>(residual, count, st, eq_before, out_off, idx, val);
  else k_topk_emit<false><<<(unsigned)nb, kThreads, 0, s>>>(residual, count, st, eq_before, out_off, idx, val);
  return cudaGetLastError();
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
ar_status_t tk_ok() {
  gar::set_last_error("");
  return AR_SUCCESS;
}
uintptr_t tk_addr(const void* p) { return reinterpret_cast<uintptr_t>(p); }
bool tk_overlap(const void* a, size_t na, const void* b, size_t nb) {
  return na && nb && tk_addr(a) < tk_addr(b) + nb && tk_addr(b) < tk_addr(a) + na;
}

}  // namespace

extern "C" {

size_t ar_topk_workspace_bytes(size_t count) {
  if (count > 0xFFFFFFFFull) return 0;
  return gar::topk_workspace_bytes(count);
}

ar_status_t ar_topk_compress(const float* grad, float* residual, size_t count, size_t k, uint32_t* idx, float* val,
                             void* workspace, size_t ws_bytes, ar_stream_t stream) {
  if (count > 0xFFFFFFFFull) return tk_fail(AR_ERR_INVALID_ARGUMENT, "count must fit 32-bit indices");
  if (k > count) return tk_fail(AR_ERR_INVALID_ARGUMENT, "k exceeds count");
  if (count == 0) return tk_ok();
  if (!grad || !residual || !workspace || (k > 0 && (!idx || !val)))
    return tk_fail(AR_ERR_INVALID_ARGUMENT, "null pointer");
  if (tk_addr(grad) % 4 || tk_addr(residual) % 4 || tk_addr(idx) % 4 || tk_addr(val) % 4)
    return tk_fail(AR_ERR_INVALID_ARGUMENT, "buffer not aligned to its element size");
  if (tk_addr(workspace) % 16) return tk_fail(AR_ERR_INVALID_ARGUMENT, "workspace must be 16-byte aligned");
  const size_t need = gar::topk_workspace_bytes(count);
  if (ws_bytes < need) return tk_fail(AR_ERR_INVALID_ARGUMENT, "workspace too small");
  const size_t b = count * 4, kb = k * 4;
  // grad is read only; residual, idx, val and the workspace are written
  const void* outs[4] = {residual, idx, val, workspace};
  const size_t out_bytes[4] = {b, kb, kb, need};
  for (int i = 0; i < 4; ++i) {
    if (tk_overlap(grad, b, outs[i], out_bytes[i])) return tk_fail(AR_ERR_ALIAS, "buffers overlap");
    for (int j = i + 1; j < 4; ++j)
      if (tk_overlap(outs[i], out_bytes[i], outs[j], out_bytes[j])) return tk_fail(AR_ERR_ALIAS, "buffers overlap");
  }
  const cudaError_t e = gar::launch_topk(grad, residual, count, k, idx, val, workspace,
                                         reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return tk_fail(AR_ERR_CUDA, std::string("top-k launch: ") + cudaGetErrorString(e));
  return tk_ok();
}

ar_status_t ar_sparse_allreduce(const uint32_t* const* idx, const float* const* val, const size_t* nnz, int nranks,
                                size_t count, ar_op_t op, ar_algo_t algo, float* const* recvbufs, ar_stream_t stream) {
  if (!idx || !val || !nnz || !recvbufs) return tk_fail(AR_ERR_INVALID_ARGUMENT, "null array");
  if (nranks < 1 || nranks > AR_MAX_RANKS) return tk_fail(AR_ERR_INVALID_ARGUMENT, "nranks must be in 1..64");
  if (op < AR_SUM || op > AR_MAX) return tk_fail(AR_ERR_INVALID_ARGUMENT, "unknown op");
  if (algo < AR_ALGO_RING || algo > AR_ALGO_AUTO) return tk_fail(AR_ERR_INVALID_ARGUMENT, "unknown algo");
  if ((algo == AR_ALGO_TREE || algo == AR_ALGO_STEP_TREE) && (nranks & (nranks - 1)))
    return tk_fail(AR_ERR_UNSUPPORTED, "TREE needs nranks to be a power of two");
  if (count > 0xFFFFFFFFull) return tk_fail(AR_ERR_INVALID_ARGUMENT, "count must fit 32-bit indices");
  if (count == 0) return tk_ok();
  const size_t b = count * 4;
  uint64_t tiles = 0;
  gar::ScatterArgs a{};
  a.nranks = nranks;
  a.count = count;
  for (int r = 0; r < nranks; ++r) {
    if (nnz[r] > count) return tk_fail(AR_ERR_INVALID_ARGUMENT, "nnz exceeds count");
    if (!recvbufs[r] || (nnz[r] > 0 && (!idx[r] || !val[r])))
      return tk_fail(AR_ERR_INVALID_ARGUMENT, "null buffer of rank " + std::to_string(r));
    if (tk_addr(recvbufs[r]) % 4 || tk_addr(idx[r]) % 4 || tk_addr(val[r]) % 4)
      return tk_fail(AR_ERR_INVALID_ARGUMENT, "buffer not aligned to its element size");
    for (int q = 0; q < nranks; ++q) {
      if (q != r && tk_overlap(recvbufs[r], b, recvbufs[q], b)) return tk_fail(AR_ERR_ALIAS, "buffers overlap");
      if (tk_overlap(recvbufs[r], b, idx[q], nnz[q] * 4) || tk_overlap(recvbufs[r], b, val[q], nnz[q] * 4))
        return tk_fail(AR_ERR_ALIAS, "buffers overlap");
    }
    a.idx[r] = idx[r];
    a.val[r] = val[r];
    a.dst[r] = recvbufs[r];
    a.nnz[r] = nnz[r];
    a.tile_start[r] = (uint32_t)tiles;
    tiles += (nnz[r] + gar::kThreads - 1) / gar::kThreads;
  }
  a.tile_start[nranks] = (uint32_t)tiles;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  for (int r = 0; r < nranks; ++r) {
    const cudaError_t e = cudaMemsetAsync(recvbufs[r], 0, b, s);
    if (e != cudaSuccess) return tk_fail(AR_ERR_CUDA, std::string("zeroing the outputs: ") + cudaGetErrorString(e));
  }
  const cudaError_t e = gar::launch_sparse_scatter(a, s);
  if (e != cudaSuccess) return tk_fail(AR_ERR_CUDA, std::string("sparse scatter launch: ") + cudaGetErrorString(e));
  // the dense forms now sit in the outputs: allreduce them in place
  std::vector<const void*> in(recvbufs, recvbufs + nranks);
  std::vector<void*> out(recvbufs, recvbufs + nranks);
  return ar_allreduce(in.data(), out.data(), nranks, count, AR_F32, op, algo, stream);
}

}  // extern "C"
