// ar_api.cpp — the C ABI declared in include/ar.h: argument validation,
// aliasing rules, the chunk plan, the bucket plan, and packing of the
// by-value kernel argument blocks. Everything here runs on the host; nothing
// allocates device memory or synchronises.
#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <string>
#include <vector>

#include <cuda_runtime.h>

#include "ar.h"
#include "ar_internal.h"
#include "ar_trace.h"

namespace gar {

// in ar_reduce_<type>.cu
cudaError_t launch_reduce_f32(int op, int mode, const ReduceArgs& a, cudaStream_t stream);
cudaError_t launch_reduce_f16(int op, int mode, const ReduceArgs& a, cudaStream_t stream);
cudaError_t launch_reduce_bf16(int op, int mode, const ReduceArgs& a, cudaStream_t stream);
cudaError_t launch_reduce_i32(int op, int mode, const ReduceArgs& a, cudaStream_t stream);

cudaError_t launch_reduce(int dtype, int op, int mode, const ReduceArgs& a, cudaStream_t stream) {
  switch (dtype) {
    case DT_F32: return launch_reduce_f32(op, mode, a, stream);
    case DT_F16: return launch_reduce_f16(op, mode, a, stream);
    case DT_BF16: return launch_reduce_bf16(op, mode, a, stream);
    case DT_I32: return launch_reduce_i32(op, mode, a, stream);
    default: return cudaErrorInvalidValue;
  }
}

// in ar_bucket_<type>.cu
cudaError_t launch_bucket_f32(int op, int mode, const BucketArgs& a, cudaStream_t stream);
cudaError_t launch_bucket_f16(int op, int mode, const BucketArgs& a, cudaStream_t stream);
cudaError_t launch_bucket_bf16(int op, int mode, const BucketArgs& a, cudaStream_t stream);
cudaError_t launch_bucket_i32(int op, int mode, const BucketArgs& a, cudaStream_t stream);

// in ar_fp8_fused_<input type>.cu
cudaError_t launch_fp8_fused_bf16(int out_dtype, int op, int mode, bool vec, const Fp8FusedArgs& a,
                                  cudaStream_t stream);
cudaError_t launch_fp8_fused_f16(int out_dtype, int op, int mode, bool vec, const Fp8FusedArgs& a,
                                 cudaStream_t stream);
cudaError_t launch_fp8_fused_f32(int out_dtype, int op, int mode, bool vec, const Fp8FusedArgs& a,
                                 cudaStream_t stream);

cudaError_t launch_fp8_fused(int in_dtype, int out_dtype, int op, int mode, bool vec, const Fp8FusedArgs& a,
                             cudaStream_t stream) {
  switch (in_dtype) {
    case DT_BF16: return launch_fp8_fused_bf16(out_dtype, op, mode, vec, a, stream);
    case DT_F16: return launch_fp8_fused_f16(out_dtype, op, mode, vec, a, stream);
    case DT_F32: return launch_fp8_fused_f32(out_dtype, op, mode, vec, a, stream);
    default: return cudaErrorInvalidValue;
  }
}

// in ar_fp8_hop_<input type>.cu
cudaError_t launch_fp8_hop_bf16(int out_dtype, int op, const Fp8HopArgs& a, cudaStream_t stream);
cudaError_t launch_fp8_hop_f16(int out_dtype, int op, const Fp8HopArgs& a, cudaStream_t stream);
cudaError_t launch_fp8_hop_f32(int out_dtype, int op, const Fp8HopArgs& a, cudaStream_t stream);

cudaError_t launch_fp8_hop(int in_dtype, int out_dtype, int op, const Fp8HopArgs& a, cudaStream_t stream) {
  switch (in_dtype) {
    case DT_BF16: return launch_fp8_hop_bf16(out_dtype, op, a, stream);
    case DT_F16: return launch_fp8_hop_f16(out_dtype, op, a, stream);
    case DT_F32: return launch_fp8_hop_f32(out_dtype, op, a, stream);
    default: return cudaErrorInvalidValue;
  }
}

namespace {
constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];  // 0: not read yet
}  // namespace

cudaError_t sm_count(int* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < kMaxDevices) {
    const int c = g_sm_count[dev].load(std::memory_order_relaxed);
    if (c > 0) {
      *out = c;
      return cudaSuccess;
    }
  }
  int c = 0;
  e = cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  if (c < 1) c = 1;
  if (dev >= 0 && dev < kMaxDevices) g_sm_count[dev].store(c, std::memory_order_relaxed);
  *out = c;
  return cudaSuccess;
}

cudaError_t launch_bucket_reduce(int dtype, int op, int mode, const BucketArgs& a, cudaStream_t stream) {
  switch (dtype) {
    case DT_F32: return launch_bucket_f32(op, mode, a, stream);
    case DT_F16: return launch_bucket_f16(op, mode, a, stream);
    case DT_BF16: return launch_bucket_bf16(op, mode, a, stream);
    case DT_I32: return launch_bucket_i32(op, mode, a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gar

namespace {

using namespace gar;

thread_local std::string g_last_error;

ar_status_t fail(ar_status_t st, const std::string& msg) {
  g_last_error = msg;
  return st;
}

ar_status_t ok() {
  g_last_error.clear();
  return AR_SUCCESS;
}

// A CUDA error is reported once, through this library's status and message:
// it is also taken off the runtime's per-thread last-error slot, so that a
// later check elsewhere (a framework's own launch check) does not report it
// again.
ar_status_t cuda_fail(cudaError_t e, const char* what) {
  (void)cudaGetLastError();
  return fail(AR_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

size_t elem_size(int dt) {
  switch (dt) {
    case AR_F32: case AR_I32: return 4;
    case AR_F16: case AR_BF16: return 2;
    default: return 0;
  }
}

bool valid_op(int op) { return op >= AR_SUM && op <= AR_MAX; }
bool valid_algo(int a) { return a >= AR_ALGO_RING && a <= AR_ALGO_TREE; }
bool valid_any_algo(int a) { return a >= AR_ALGO_RING && a <= AR_ALGO_AUTO; }

// The one-pass orders for entry points that have no stepwise form: AUTO is
// the fused order; the stepwise values are refused.
ar_status_t basic_algo(ar_algo_t* algo) {
  if (*algo == AR_ALGO_AUTO) *algo = AR_ALGO_FUSED;
  if (*algo == AR_ALGO_STEP_RING || *algo == AR_ALGO_STEP_TREE)
    return fail(AR_ERR_UNSUPPORTED, "stepwise orders exist for ar_allreduce only");
  if (!valid_algo(*algo)) return fail(AR_ERR_INVALID_ARGUMENT, "unknown algo");
  return AR_SUCCESS;
}
bool pow2(int n) { return n >= 1 && (n & (n - 1)) == 0; }
uintptr_t addr(const void* p) { return reinterpret_cast<uintptr_t>(p); }
bool aligned(const void* p, size_t a) { return (addr(p) % a) == 0; }

// chunk length (elements): ceil(count / N) rounded up to a multiple of `vec` elements
size_t chunk_len(size_t count, int n, size_t vec) {
  const size_t q = count / (size_t)n + (count % (size_t)n != 0);
  return (q + vec - 1) / vec * vec;
}

// Overlap rules. Inputs may overlap each other (read only). An output may not
// overlap another output, nor an input, except output o and input `pair_in[o]`
// when the output starts exactly `pair_off[o]` bytes into that input (the
// documented in-place forms). pair_in[o] = -1: no in-place form.
struct Span {
  uintptr_t lo, hi;
  bool out;
  int idx;
};

bool overlap_ok(const std::vector<Span>& spans, const std::vector<int>& pair_in,
                const std::vector<uintptr_t>& pair_off) {
  std::vector<Span> s;
  s.reserve(spans.size());
  for (const Span& x : spans)
    if (x.hi > x.lo) s.push_back(x);
  std::sort(s.begin(), s.end(), [](const Span& a, const Span& b) { return a.lo < b.lo; });
  for (size_t i = 0; i < s.size(); ++i) {
    for (size_t j = i + 1; j < s.size() && s[j].lo < s[i].hi; ++j) {
      const Span& a = s[i];
      const Span& b = s[j];
      if (!a.out && !b.out) continue;
      if (a.out && b.out) return false;
      const Span& o = a.out ? a : b;
      const Span& in = a.out ? b : a;
      if (pair_in.empty() || pair_in[o.idx] != in.idx || o.lo != in.lo + pair_off[o.idx]) return false;
    }
  }
  return true;
}

ar_status_t check_ptrs(const void* const* p, int n, size_t es, const char* what) {
  for (int r = 0; r < n; ++r) {
    if (!p[r]) return fail(AR_ERR_INVALID_ARGUMENT, std::string(what) + "[" + std::to_string(r) + "] is null");
    if (!aligned(p[r], es))
      return fail(AR_ERR_INVALID_ARGUMENT,
                  std::string(what) + "[" + std::to_string(r) + "] is not aligned to the element size");
  }
  return AR_SUCCESS;
}

bool all_aligned16(const void* const* p, int n) {
  for (int r = 0; r < n; ++r)
    if (!aligned(p[r], 16)) return false;
  return true;
}

ar_status_t common_checks(const void* const* send, void* const* recv, int n, int dtype) {
  if (!send || !recv) return fail(AR_ERR_INVALID_ARGUMENT, "null buffer array");
  if (n < 1 || n > AR_MAX_RANKS) return fail(AR_ERR_INVALID_ARGUMENT, "nranks must be in 1..64");
  if (elem_size(dtype) == 0) return fail(AR_ERR_INVALID_ARGUMENT, "unknown dtype");
  return AR_SUCCESS;
}

// Ring all-gather of chunk c (owned by rank c, already in recv[c]) to every
// other rank; `es` bytes per element, chunk length L elements.
ar_status_t ring_gather(void* const* recv, int n, size_t count, size_t L, size_t es, bool vec, cudaStream_t s) {
  if (n == 1) return AR_SUCCESS;
  GatherArgs g{};
  g.nranks = n;
  g.skip_mask = (n == 64) ? ~0ull : ((1ull << n) - 1);
  for (int c = 0; c < n; ++c) {
    const size_t off = (size_t)c * L < count ? (size_t)c * L * es : 0;
    g.src[c] = static_cast<const char*>(recv[c]) + off;
    g.dst[c] = recv[c];
  }
  int unit;
  if (vec) {
    unit = 16;
    g.units = count * es / 16;
    g.Lu = L * es / 16;
    g.tail_bytes = count * es % 16;
    g.Lb = L * es;
  } else {
    unit = (int)es;
    g.units = count;
    g.Lu = L;
  }
  const cudaError_t e = launch_gather(unit, g, s);
  return e == cudaSuccess ? AR_SUCCESS : cuda_fail(e, "all-gather launch");
}

// All-gather steps of the stepwise executors: batched copies of N ranges.
ar_status_t step_copies(const std::vector<CopyItem>& items, cudaStream_t s) {
  MultiCopyArgs a{};
  uint64_t tiles = 0;
  for (const CopyItem& it : items) {
    if (it.bytes == 0) continue;
    a.item[a.nitems] = it;
    a.tile_start[a.nitems] = (uint32_t)tiles;
    tiles += (it.bytes + kCopyTile - 1) / kCopyTile;
    a.nitems += 1;
  }
  a.tile_start[a.nitems] = (uint32_t)tiles;
  const cudaError_t e = launch_multicopy(a, s);
  return e == cudaSuccess ? AR_SUCCESS : cuda_fail(e, "all-gather step launch");
}

struct StepTask {
  const void* a;
  const void* b;
  void* dst;
  uint64_t len;
};

ar_status_t step_combine(int dtype, int op, int nranks, bool finish, bool vec, const std::vector<StepTask>& tasks,
                         cudaStream_t s) {
  StepArgs a{};
  a.nranks = nranks;
  a.finish = finish ? 1 : 0;
  a.vec = vec ? 1 : 0;
  uint64_t tiles = 0;
  for (const StepTask& t : tasks) {
    if (t.len == 0) continue;
    const int k = a.ntasks++;
    a.a[k] = t.a;
    a.b[k] = t.b;
    a.dst[k] = t.dst;
    a.len[k] = t.len;
    a.tile_start[k] = (uint32_t)tiles;
    const uint64_t items = vec ? (t.len + 3) / 4 : t.len;
    tiles += (items + kThreads - 1) / kThreads;
  }
  a.tile_start[a.ntasks] = (uint32_t)tiles;
  const cudaError_t e = launch_step_combine(dtype, op, a, s);
  return e == cudaSuccess ? AR_SUCCESS : cuda_fail(e, "reduce-scatter step launch");
}

const char* at(const void* p, uint64_t elems) { return static_cast<const char*>(p) + elems * 4; }
char* at(void* p, uint64_t elems) { return static_cast<char*>(p) + elems * 4; }

// Ring, literally: step s, rank r sends its partial of chunk (r-s-1) mod N to
// r+1, which adds it to its own values of that chunk (the sender's partial is
// its input at step 0); then N-1 forwarding steps. 4-byte elements.
ar_status_t step_ring(const void* const* send, void* const* recv, int n, size_t count, int dtype, int op,
                      bool vec, cudaStream_t s) {
  const size_t L = chunk_len(count, n, 4);
  auto lo_of = [&](int c) { return std::min((size_t)c * L, count); };
  auto hi_of = [&](int c) { return std::min((size_t)(c + 1) * L, count); };
  for (int st = 0; st < n - 1; ++st) {
    std::vector<StepTask> tasks;
    for (int r = 0; r < n; ++r) {
      const int c = ((r - st - 1) % n + n) % n, d = (r + 1) % n;
      const size_t lo = lo_of(c), hi = hi_of(c);
      tasks.push_back({at(st == 0 ? send[r] : (const void*)recv[r], lo), at(send[d], lo), at(recv[d], lo), hi - lo});
    }
    if (ar_status_t e = step_combine(dtype, op, n, st == n - 2, vec, tasks, s); e != AR_SUCCESS) return e;
  }
  for (int st = 0; st < n - 1; ++st) {
    std::vector<CopyItem> items;
    for (int r = 0; r < n; ++r) {
      const int c = ((r - st) % n + n) % n, d = (r + 1) % n;
      const size_t lo = lo_of(c), hi = hi_of(c);
      items.push_back({at(recv[r], lo), at(recv[d], lo), (hi - lo) * 4});
    }
    if (ar_status_t e = step_copies(items, s); e != AR_SUCCESS) return e;
  }
  return AR_SUCCESS;
}

// Recursive halving reduce-scatter then recursive doubling all-gather: at
// distance d = N/2, N/4, ..., 1 partners r and r^d split their common segment
// (first half rounded up to 16 bytes) and each combines the half it keeps.
ar_status_t step_tree(const void* const* send, void* const* recv, int n, size_t count, int dtype, int op,
                      bool vec, cudaStream_t s) {
  int levels = 0;
  while ((1 << levels) < n) ++levels;
  std::vector<std::vector<std::pair<size_t, size_t>>> seg(levels + 1,
                                                          std::vector<std::pair<size_t, size_t>>(n));
  for (int r = 0; r < n; ++r) seg[0][r] = {0, count};
  for (int i = 0; i < levels; ++i) {
    const int d = n >> (i + 1);
    std::vector<StepTask> tasks;
    for (int r = 0; r < n; ++r) {
      const size_t lo = seg[i][r].first, hi = seg[i][r].second;
      const size_t half = ((hi - lo + 1) / 2 + 3) / 4 * 4;
      const size_t mid = std::min(lo + half, hi);
      seg[i + 1][r] = (r & d) ? std::make_pair(mid, hi) : std::make_pair(lo, mid);
      const int p = r ^ d;
      const size_t klo = seg[i + 1][r].first, khi = seg[i + 1][r].second;
      tasks.push_back({at(i == 0 ? send[r] : (const void*)recv[r], klo), at(i == 0 ? send[p] : (const void*)recv[p], klo),
                       at(recv[r], klo), khi - klo});
    }
    if (ar_status_t e = step_combine(dtype, op, n, i == levels - 1, vec, tasks, s); e != AR_SUCCESS) return e;
  }
  for (int i = levels - 1; i >= 0; --i) {
    const int d = n >> (i + 1);
    std::vector<CopyItem> items;
    for (int r = 0; r < n; ++r) {
      const size_t lo = seg[i + 1][r].first, hi = seg[i + 1][r].second;
      items.push_back({at(recv[r], lo), at(recv[r ^ d], lo), (hi - lo) * 4});
    }
    if (ar_status_t e = step_copies(items, s); e != AR_SUCCESS) return e;
  }
  return AR_SUCCESS;
}

// --- 16-bit element types: partial sums in binary32, in a workspace of one
// count-long partial array per rank (P[r]); the last reduce-scatter step
// writes the finished 16-bit values into the outputs, whose all-gather steps
// are the 16-bit copies above.

const char* at2(const void* p, uint64_t elems) { return static_cast<const char*>(p) + elems * 2; }
char* at2(void* p, uint64_t elems) { return static_cast<char*>(p) + elems * 2; }

ar_status_t step_combine16(int dtype, int op, int nranks, bool a32, bool b32, bool finish, bool vec,
                           const std::vector<StepTask>& tasks, cudaStream_t s) {
  StepArgs a{};
  a.nranks = nranks;
  a.finish = finish ? 1 : 0;
  a.vec = vec ? 1 : 0;
  uint64_t tiles = 0;
  for (const StepTask& t : tasks) {
    if (t.len == 0) continue;
    const int k = a.ntasks++;
    a.a[k] = t.a;
    a.b[k] = t.b;
    a.dst[k] = t.dst;
    a.len[k] = t.len;
    a.tile_start[k] = (uint32_t)tiles;
    tiles += ((t.len + 3) / 4 + kThreads - 1) / kThreads;
  }
  a.tile_start[a.ntasks] = (uint32_t)tiles;
  const cudaError_t e = launch_step_combine16(dtype, op, a32, b32, a, s);
  return e == cudaSuccess ? AR_SUCCESS : cuda_fail(e, "reduce-scatter step launch");
}

// Ring, literally, as step_ring: step st, rank r's partial of chunk
// (r-st-1) mod N (its input at step 0, else P[r]) plus rank r+1's input goes
// to P[r+1] (or, on the last step, finished into the output of r+1). Within
// a step rank d writes one chunk of P[d] while rank d+1 reads another.
ar_status_t step_ring16(const void* const* send, void* const* recv, char* const* P, int n, size_t count, int dtype,
                        int op, bool vec, cudaStream_t s) {
  const size_t L = chunk_len(count, n, 8);
  auto lo_of = [&](int c) { return std::min((size_t)c * L, count); };
  auto hi_of = [&](int c) { return std::min((size_t)(c + 1) * L, count); };
  for (int st = 0; st < n - 1; ++st) {
    const bool last = st == n - 2;
    std::vector<StepTask> tasks;
    for (int r = 0; r < n; ++r) {
      const int c = ((r - st - 1) % n + n) % n, d = (r + 1) % n;
      const size_t lo = lo_of(c), hi = hi_of(c);
      tasks.push_back({st == 0 ? at2(send[r], lo) : at(P[r], lo), at2(send[d], lo),
                       last ? static_cast<void*>(at2(recv[d], lo)) : static_cast<void*>(at(P[d], lo)), hi - lo});
    }
    if (ar_status_t e = step_combine16(dtype, op, n, st > 0, false, last, vec, tasks, s); e != AR_SUCCESS) return e;
  }
  for (int st = 0; st < n - 1; ++st) {
    std::vector<CopyItem> items;
    for (int r = 0; r < n; ++r) {
      const int c = ((r - st) % n + n) % n, d = (r + 1) % n;
      const size_t lo = lo_of(c), hi = hi_of(c);
      items.push_back({at2(recv[r], lo), at2(recv[d], lo), (hi - lo) * 2});
    }
    if (ar_status_t e = step_copies(items, s); e != AR_SUCCESS) return e;
  }
  return AR_SUCCESS;
}

// Recursive halving / doubling, as step_tree: at each level partners keep
// the two halves of their common segment; the partials of a level live in
// P, each rank writing the half it keeps while its partner reads the other.
ar_status_t step_tree16(const void* const* send, void* const* recv, char* const* P, int n, size_t count, int dtype,
                        int op, bool vec, cudaStream_t s) {
  int levels = 0;
  while ((1 << levels) < n) ++levels;
  std::vector<std::vector<std::pair<size_t, size_t>>> seg(levels + 1,
                                                          std::vector<std::pair<size_t, size_t>>(n));
  for (int r = 0; r < n; ++r) seg[0][r] = {0, count};
  for (int i = 0; i < levels; ++i) {
    const int d = n >> (i + 1);
    const bool last = i == levels - 1;
    std::vector<StepTask> tasks;
    for (int r = 0; r < n; ++r) {
      const size_t lo = seg[i][r].first, hi = seg[i][r].second;
      const size_t half = ((hi - lo + 1) / 2 + 3) / 4 * 4;
      const size_t mid = std::min(lo + half, hi);
      seg[i + 1][r] = (r & d) ? std::make_pair(mid, hi) : std::make_pair(lo, mid);
      const int p = r ^ d;
      const size_t klo = seg[i + 1][r].first, khi = seg[i + 1][r].second;
      tasks.push_back({i == 0 ? at2(send[r], klo) : at(P[r], klo), i == 0 ? at2(send[p], klo) : at(P[p], klo),
                       last ? static_cast<void*>(at2(recv[r], klo)) : static_cast<void*>(at(P[r], klo)),
                       khi - klo});
    }
    if (ar_status_t e = step_combine16(dtype, op, n, i > 0, i > 0, last, vec, tasks, s); e != AR_SUCCESS) return e;
  }
  for (int i = levels - 1; i >= 0; --i) {
    const int d = n >> (i + 1);
    std::vector<CopyItem> items;
    for (int r = 0; r < n; ++r) {
      const size_t lo = seg[i + 1][r].first, hi = seg[i + 1][r].second;
      items.push_back({at2(recv[r], lo), at2(recv[r ^ d], lo), (hi - lo) * 2});
    }
    if (ar_status_t e = step_copies(items, s); e != AR_SUCCESS) return e;
  }
  return AR_SUCCESS;
}

size_t stepwise_rank_bytes(size_t count) { return (count * 4 + 255) / 256 * 256; }

}  // namespace

extern "C" {

const char* ar_version(void) { return "gradient-allreduce-gb300 0.1.0 (sm_103a)"; }

const char* ar_status_string(ar_status_t st) {
  switch (st) {
    case AR_SUCCESS: return "success";
    case AR_ERR_INVALID_ARGUMENT: return "invalid argument";
    case AR_ERR_UNSUPPORTED: return "unsupported combination";
    case AR_ERR_ALIAS: return "buffers overlap";
    case AR_ERR_CUDA: return "CUDA error";
    case AR_ERR_TIMEOUT: return "timed out";
    case AR_ERR_MISMATCH: return "collective calls do not match";
    default: return "unknown status";
  }
}

const char* ar_last_error(void) { return g_last_error.c_str(); }

ar_status_t ar_allreduce(const void* const* sendbufs, void* const* recvbufs, int nranks, size_t count,
                         ar_dtype_t dtype, ar_op_t op, ar_algo_t algo, ar_stream_t stream) {
  AR_TRACE("ar_allreduce");
  ar_status_t st = common_checks(sendbufs, recvbufs, nranks, dtype);
  if (st != AR_SUCCESS) return st;
  if (!valid_op(op)) return fail(AR_ERR_INVALID_ARGUMENT, "unknown op");
  if (!valid_any_algo(algo)) return fail(AR_ERR_INVALID_ARGUMENT, "unknown algo");
  if (algo == AR_ALGO_AUTO) algo = AR_ALGO_FUSED;  // fastest one-pass order at every size on one device
  if ((algo == AR_ALGO_TREE || algo == AR_ALGO_STEP_TREE) && !pow2(nranks))
    return fail(AR_ERR_UNSUPPORTED, "TREE needs nranks to be a power of two");
  const size_t es = elem_size(dtype);
  const bool stepwise = algo == AR_ALGO_STEP_RING || algo == AR_ALGO_STEP_TREE;
  if (stepwise && es != 4)
    return fail(AR_ERR_UNSUPPORTED,
                "stepwise orders of 16-bit types keep binary32 partials in a workspace: use ar_allreduce_stepwise");
  if (count == 0) return ok();
  if (count > SIZE_MAX / es / 2) return fail(AR_ERR_INVALID_ARGUMENT, "count too large");
  if ((st = check_ptrs(sendbufs, nranks, es, "sendbufs")) != AR_SUCCESS) return st;
  if ((st = check_ptrs(recvbufs, nranks, es, "recvbufs")) != AR_SUCCESS) return st;
  const size_t bytes = count * es;
  std::vector<Span> spans;
  spans.reserve(2 * (size_t)nranks);
  std::vector<int> pair_in(nranks);
  std::vector<uintptr_t> pair_off(nranks, 0);
  for (int r = 0; r < nranks; ++r) {
    spans.push_back({addr(sendbufs[r]), addr(sendbufs[r]) + bytes, false, r});
    spans.push_back({addr(recvbufs[r]), addr(recvbufs[r]) + bytes, true, r});
    pair_in[r] = r;  // in place: recvbufs[r] == sendbufs[r]
  }
  if (!overlap_ok(spans, pair_in, pair_off)) return fail(AR_ERR_ALIAS, "buffers overlap");

  const size_t L = chunk_len(count, nranks, 16 / es);
  const bool vec = all_aligned16(sendbufs, nranks) && all_aligned16(recvbufs, nranks);
  ReduceArgs a{};
  a.nranks = nranks;
  a.count = count;
  a.L = L;
  a.vec = vec ? 1 : 0;
  for (int r = 0; r < nranks; ++r) a.src[r] = sendbufs[r];
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (stepwise && nranks > 1) {
    st = algo == AR_ALGO_STEP_RING ? step_ring(sendbufs, recvbufs, nranks, count, dtype, op, vec, s)
                                   : step_tree(sendbufs, recvbufs, nranks, count, dtype, op, vec, s);
    return st == AR_SUCCESS ? ok() : st;
  }
  if (algo == AR_ALGO_RING) {
    for (int c = 0; c < nranks; ++c)
      a.dst[c] = static_cast<char*>(recvbufs[c]) + ((size_t)c * L < count ? (size_t)c * L * es : 0);
    const cudaError_t e = launch_reduce(dtype, op, MODE_RS, a, s);
    if (e != cudaSuccess) return cuda_fail(e, "reduce-scatter launch");
    if ((st = ring_gather(recvbufs, nranks, count, L, es, vec, s)) != AR_SUCCESS) return st;
    return ok();
  }
  for (int r = 0; r < nranks; ++r) a.dst[r] = recvbufs[r];
  const cudaError_t e = launch_reduce(dtype, op, algo == AR_ALGO_TREE ? MODE_FUSED_TREE : MODE_FUSED_RING, a, s);
  if (e != cudaSuccess) return cuda_fail(e, "allreduce launch");
  return ok();
}

size_t ar_stepwise_workspace_bytes(int nranks, size_t count, ar_dtype_t dtype) {
  if (nranks < 1 || nranks > AR_MAX_RANKS || elem_size(dtype) != 2 || count > SIZE_MAX / 8 / AR_MAX_RANKS) return 0;
  return (size_t)nranks * stepwise_rank_bytes(count);
}

ar_status_t ar_allreduce_stepwise(const void* const* sendbufs, void* const* recvbufs, int nranks, size_t count,
                                  ar_dtype_t dtype, ar_op_t op, ar_algo_t algo, void* workspace, size_t ws_bytes,
                                  ar_stream_t stream) {
  AR_TRACE("ar_allreduce_stepwise");
  ar_status_t st = common_checks(sendbufs, recvbufs, nranks, dtype);
  if (st != AR_SUCCESS) return st;
  if (!valid_op(op)) return fail(AR_ERR_INVALID_ARGUMENT, "unknown op");
  if (algo != AR_ALGO_STEP_RING && algo != AR_ALGO_STEP_TREE)
    return fail(AR_ERR_INVALID_ARGUMENT, "ar_allreduce_stepwise takes STEP_RING or STEP_TREE");
  if (algo == AR_ALGO_STEP_TREE && !pow2(nranks))
    return fail(AR_ERR_UNSUPPORTED, "TREE needs nranks to be a power of two");
  const size_t es = elem_size(dtype);
  if (es == 4)  // partials in the element type, in the outputs: no workspace
    return ar_allreduce(sendbufs, recvbufs, nranks, count, dtype, op, algo, stream);
  if (count == 0) return ok();
  if (count > SIZE_MAX / 8 / AR_MAX_RANKS) return fail(AR_ERR_INVALID_ARGUMENT, "count too large");
  if (nranks == 1)  // nothing to combine: the one-pass kernel copies (and finishes) the input
    return ar_allreduce(sendbufs, recvbufs, nranks, count, dtype, op, AR_ALGO_FUSED, stream);
  const size_t need = ar_stepwise_workspace_bytes(nranks, count, dtype);
  if (!workspace) return fail(AR_ERR_INVALID_ARGUMENT, "null workspace");
  if (ws_bytes < need) return fail(AR_ERR_INVALID_ARGUMENT, "workspace too small");
  if (!aligned(workspace, 16)) return fail(AR_ERR_INVALID_ARGUMENT, "workspace must be 16-byte aligned");
  if ((st = check_ptrs(sendbufs, nranks, es, "sendbufs")) != AR_SUCCESS) return st;
  if ((st = check_ptrs(recvbufs, nranks, es, "recvbufs")) != AR_SUCCESS) return st;
  const size_t bytes = count * es;
  std::vector<Span> spans;
  std::vector<int> pair_in(nranks + 1, -1);
  std::vector<uintptr_t> pair_off(nranks + 1, 0);
  for (int r = 0; r < nranks; ++r) {
    spans.push_back({addr(sendbufs[r]), addr(sendbufs[r]) + bytes, false, r});
    spans.push_back({addr(recvbufs[r]), addr(recvbufs[r]) + bytes, true, r});
    pair_in[r] = r;  // in place: recvbufs[r] == sendbufs[r]
  }
  spans.push_back({addr(workspace), addr(workspace) + need, true, nranks});
  if (!overlap_ok(spans, pair_in, pair_off)) return fail(AR_ERR_ALIAS, "buffers overlap");
  std::vector<char*> P(nranks);
  for (int r = 0; r < nranks; ++r) P[r] = static_cast<char*>(workspace) + (size_t)r * stepwise_rank_bytes(count);
  const bool vec = all_aligned16(sendbufs, nranks) && all_aligned16(recvbufs, nranks);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  st = algo == AR_ALGO_STEP_RING ? step_ring16(sendbufs, recvbufs, P.data(), nranks, count, dtype, op, vec, s)
                                 : step_tree16(sendbufs, recvbufs, P.data(), nranks, count, dtype, op, vec, s);
  return st == AR_SUCCESS ? ok() : st;
}

ar_status_t ar_allreduce_slice(const void* const* sendbufs, void* const* recvbufs, int nranks, size_t count,
                               size_t first, size_t n, ar_dtype_t dtype, ar_op_t op, ar_algo_t algo,
                               ar_stream_t stream) {
  AR_TRACE("ar_allreduce_slice");
  ar_status_t st = common_checks(sendbufs, recvbufs, nranks, dtype);
  if (st != AR_SUCCESS) return st;
  if (!valid_op(op)) return fail(AR_ERR_INVALID_ARGUMENT, "unknown op");
  if (!valid_any_algo(algo)) return fail(AR_ERR_INVALID_ARGUMENT, "unknown algo");
  // the stepwise executors give the ring and tree orders' bits; a slice takes those orders one pass at a time
  if (algo == AR_ALGO_AUTO || algo == AR_ALGO_RING || algo == AR_ALGO_STEP_RING) algo = AR_ALGO_FUSED;
  if (algo == AR_ALGO_STEP_TREE) algo = AR_ALGO_TREE;
  if (algo == AR_ALGO_TREE && !pow2(nranks)) return fail(AR_ERR_UNSUPPORTED, "TREE needs nranks to be a power of two");
  const size_t es = elem_size(dtype);
  if (count > SIZE_MAX / es / 2) return fail(AR_ERR_INVALID_ARGUMENT, "count too large");
  if (first > count || n > count - first) return fail(AR_ERR_INVALID_ARGUMENT, "slice outside the problem");
  if (n == 0) return ok();
  if ((st = check_ptrs(sendbufs, nranks, es, "sendbufs")) != AR_SUCCESS) return st;
  if ((st = check_ptrs(recvbufs, nranks, es, "recvbufs")) != AR_SUCCESS) return st;
  std::vector<Span> spans;
  std::vector<int> pair_in(nranks);
  std::vector<uintptr_t> pair_off(nranks, 0);
  for (int r = 0; r < nranks; ++r) {
    spans.push_back({addr(sendbufs[r]), addr(sendbufs[r]) + n * es, false, r});
    spans.push_back({addr(recvbufs[r]), addr(recvbufs[r]) + n * es, true, r});
    pair_in[r] = r;  // in place: recvbufs[r] == sendbufs[r]
  }
  if (!overlap_ok(spans, pair_in, pair_off)) return fail(AR_ERR_ALIAS, "buffers overlap");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t V = 16 / es;
  auto launch_piece = [&](size_t lo, size_t len, int rot, size_t Lp, int mode) -> ar_status_t {
    // elements [lo, lo + len) of the slice in local chunks of Lp elements,
    // local chunk c folded from the rank after c + rot (rank pointers
    // rotated by rot)
    ReduceArgs a{};
    a.nranks = nranks;
    a.count = len;
    a.L = Lp;
    bool vec = true;
    for (int r = 0; r < nranks; ++r) {
      const int q = (r + rot) % nranks;
      a.src[r] = static_cast<const char*>(sendbufs[q]) + lo * es;
      a.dst[r] = static_cast<char*>(recvbufs[q]) + lo * es;
      vec = vec && aligned(a.src[r], 16) && aligned(a.dst[r], 16);
    }
    a.vec = vec ? 1 : 0;
    const cudaError_t e = launch_reduce(dtype, op, mode, a, s);
    return e == cudaSuccess ? AR_SUCCESS : cuda_fail(e, "slice allreduce launch");
  };
  if (algo == AR_ALGO_TREE) {  // the tree order does not depend on the chunk plan
    st = launch_piece(0, n, 0, (n + V - 1) / V * V, MODE_FUSED_TREE);
    return st == AR_SUCCESS ? ok() : st;
  }
  // ring order: chunk c of the whole problem folds from rank c + 1. The part
  // of the slice before its first chunk boundary is one launch rotated by its
  // chunk; from that boundary on, the problem's own chunk length with the
  // rotation by the boundary's chunk index gives every later chunk its start
  // rank: two launches at most.
  const size_t L = chunk_len(count, nranks, V);
  size_t g = first;
  if (g % L != 0) {
    const size_t c = g / L;
    const size_t end = std::min(first + n, (c + 1) * L);
    if ((st = launch_piece(0, end - g, (int)(c % (size_t)nranks), (end - g + V - 1) / V * V, MODE_FUSED_RING)) !=
        AR_SUCCESS)
      return st;
    g = end;
  }
  if (g < first + n) {
    if ((st = launch_piece(g - first, first + n - g, (int)((g / L) % (size_t)nranks), L, MODE_FUSED_RING)) !=
        AR_SUCCESS)
      return st;
  }
  return ok();
}

ar_status_t ar_reduce_scatter(const void* const* sendbufs, void* const* recvbufs, int nranks, size_t recvcount,
                              ar_dtype_t dtype, ar_op_t op, ar_stream_t stream) {
  AR_TRACE("ar_reduce_scatter");
  ar_status_t st = common_checks(sendbufs, recvbufs, nranks, dtype);
  if (st != AR_SUCCESS) return st;
  if (!valid_op(op)) return fail(AR_ERR_INVALID_ARGUMENT, "unknown op");
  if (recvcount == 0) return ok();
  const size_t es = elem_size(dtype);
  if (recvcount > SIZE_MAX / es / (size_t)nranks / 2) return fail(AR_ERR_INVALID_ARGUMENT, "count too large");
  if ((st = check_ptrs(sendbufs, nranks, es, "sendbufs")) != AR_SUCCESS) return st;
  if ((st = check_ptrs(recvbufs, nranks, es, "recvbufs")) != AR_SUCCESS) return st;
  const size_t rb = recvcount * es;
  std::vector<Span> spans;
  std::vector<int> pair_in(nranks);
  std::vector<uintptr_t> pair_off(nranks);
  for (int r = 0; r < nranks; ++r) {
    spans.push_back({addr(sendbufs[r]), addr(sendbufs[r]) + rb * (size_t)nranks, false, r});
    spans.push_back({addr(recvbufs[r]), addr(recvbufs[r]) + rb, true, r});
    pair_in[r] = r;  // in place: recvbufs[c] == sendbufs[c] + c*recvcount
    pair_off[r] = (uintptr_t)r * rb;
  }
  if (!overlap_ok(spans, pair_in, pair_off)) return fail(AR_ERR_ALIAS, "buffers overlap");
  ReduceArgs a{};
  a.nranks = nranks;
  a.count = recvcount * (size_t)nranks;
  a.L = recvcount;
  a.vec = (all_aligned16(sendbufs, nranks) && all_aligned16(recvbufs, nranks) && rb % 16 == 0) ? 1 : 0;
  for (int r = 0; r < nranks; ++r) {
    a.src[r] = sendbufs[r];
    a.dst[r] = recvbufs[r];
  }
  const cudaError_t e = launch_reduce(dtype, op, MODE_RS, a, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok() : cuda_fail(e, "reduce-scatter launch");
}

ar_status_t ar_all_gather(const void* const* sendbufs, void* const* recvbufs, int nranks, size_t sendcount,
                          ar_dtype_t dtype, ar_stream_t stream) {
  AR_TRACE("ar_all_gather");
  ar_status_t st = common_checks(sendbufs, recvbufs, nranks, dtype);
  if (st != AR_SUCCESS) return st;
  if (sendcount == 0) return ok();
  const size_t es = elem_size(dtype);
  if (sendcount > SIZE_MAX / es / (size_t)nranks / 2) return fail(AR_ERR_INVALID_ARGUMENT, "count too large");
  if ((st = check_ptrs(sendbufs, nranks, es, "sendbufs")) != AR_SUCCESS) return st;
  if ((st = check_ptrs(recvbufs, nranks, es, "recvbufs")) != AR_SUCCESS) return st;
  const size_t sb = sendcount * es;
  std::vector<Span> spans;
  // in place: sendbufs[r] == recvbufs[r] + r*sendcount (the input lies inside the output)
  std::vector<int> pair_in;
  std::vector<uintptr_t> pair_off;
  GatherArgs g{};
  g.nranks = nranks;
  for (int r = 0; r < nranks; ++r) {
    const bool inplace = addr(sendbufs[r]) == addr(recvbufs[r]) + (uintptr_t)r * sb;
    if (inplace) g.skip_mask |= 1ull << r;
    else spans.push_back({addr(sendbufs[r]), addr(sendbufs[r]) + sb, false, r});
    spans.push_back({addr(recvbufs[r]), addr(recvbufs[r]) + sb * (size_t)nranks, true, r});
    g.src[r] = sendbufs[r];
    g.dst[r] = recvbufs[r];
  }
  if (!overlap_ok(spans, pair_in, pair_off)) return fail(AR_ERR_ALIAS, "buffers overlap");
  int unit;
  if (all_aligned16(sendbufs, nranks) && all_aligned16(recvbufs, nranks) && sb % 16 == 0) {
    unit = 16;
    g.units = sb * (size_t)nranks / 16;
    g.Lu = sb / 16;
  } else {
    unit = (int)es;
    g.units = sendcount * (size_t)nranks;
    g.Lu = sendcount;
  }
  const cudaError_t e = launch_gather(unit, g, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok() : cuda_fail(e, "all-gather launch");
}

ar_status_t ar_bucket_plan(const size_t* counts, int ntensors, ar_dtype_t dtype, size_t cap_bytes, int* bucket_of,
                           size_t* offset_of, size_t* bucket_counts, int* nbuckets) {
  if (ntensors < 0) return fail(AR_ERR_INVALID_ARGUMENT, "ntensors < 0");
  if (!nbuckets || (ntensors > 0 && (!counts || !bucket_of || !offset_of || !bucket_counts)))
    return fail(AR_ERR_INVALID_ARGUMENT, "null pointer");
  const size_t es = elem_size(dtype);
  if (es == 0) return fail(AR_ERR_INVALID_ARGUMENT, "unknown dtype");
  const size_t vec = 16 / es;
  size_t fill = 0;  // elements used in the open bucket
  int nb = 0;
  bool open = false;
  for (int t = ntensors - 1; t >= 0; --t) {  // gradients are ready from the last layer backwards
    if (counts[t] > SIZE_MAX / es / 4) return fail(AR_ERR_INVALID_ARGUMENT, "tensor too large");
    size_t start = (fill + vec - 1) / vec * vec;
    if (open && (start + counts[t]) * es > cap_bytes) {
      bucket_counts[nb++] = fill;
      start = 0;
    }
    bucket_of[t] = nb;
    offset_of[t] = start;
    fill = start + counts[t];
    open = true;
  }
  if (open) bucket_counts[nb++] = fill;
  *nbuckets = nb;
  return ok();
}

}  // extern "C"

namespace {

// Flatten (to_bucket = true) or unflatten: batched range copies.
ar_status_t bucket_copy(const void* const* srcs_or_null, void* const* dsts_or_null, const void* bucket_src,
                        void* bucket_dst, const size_t* counts, const size_t* offsets, int ntensors, int dtype,
                        cudaStream_t s) {
  const bool flatten = bucket_dst != nullptr;
  const size_t es = elem_size(dtype);
  if (es == 0) return fail(AR_ERR_INVALID_ARGUMENT, "unknown dtype");
  if (ntensors < 0) return fail(AR_ERR_INVALID_ARGUMENT, "ntensors < 0");
  if (ntensors == 0) return ok();
  if (!counts || !offsets) return fail(AR_ERR_INVALID_ARGUMENT, "null counts/offsets");
  const void* const* tens_in = srcs_or_null;
  void* const* tens_out = dsts_or_null;
  if (flatten ? !tens_in : !tens_out) return fail(AR_ERR_INVALID_ARGUMENT, "null tensor array");
  const char* bucket = flatten ? static_cast<const char*>(bucket_dst) : static_cast<const char*>(bucket_src);
  if (!bucket) return fail(AR_ERR_INVALID_ARGUMENT, "null bucket");
  if (!aligned(bucket, es)) return fail(AR_ERR_INVALID_ARGUMENT, "bucket is not aligned to the element size");
  std::vector<Span> spans;
  spans.reserve(2 * (size_t)ntensors);
  for (int t = 0; t < ntensors; ++t) {
    if (counts[t] == 0) continue;
    const void* tp = flatten ? tens_in[t] : tens_out[t];
    if (!tp) return fail(AR_ERR_INVALID_ARGUMENT, "tensor " + std::to_string(t) + " is null");
    if (!aligned(tp, es))
      return fail(AR_ERR_INVALID_ARGUMENT, "tensor " + std::to_string(t) + " is not aligned to the element size");
    if (counts[t] > SIZE_MAX / es / 4 || offsets[t] > SIZE_MAX / es / 4)
      return fail(AR_ERR_INVALID_ARGUMENT, "tensor too large");
    const uintptr_t b = addr(bucket) + offsets[t] * es, n = counts[t] * es;
    spans.push_back({addr(tp), addr(tp) + n, !flatten, t});
    spans.push_back({b, b + n, flatten, t});
  }
  if (!overlap_ok(spans, {}, {})) return fail(AR_ERR_ALIAS, "buffers overlap");
  MultiCopyArgs a{};
  auto flush = [&]() -> ar_status_t {
    if (a.nitems == 0) return AR_SUCCESS;
    const cudaError_t e = launch_multicopy(a, s);
    a.nitems = 0;
    return e == cudaSuccess ? AR_SUCCESS : cuda_fail(e, "bucket copy launch");
  };
  uint64_t tiles = 0;
  for (int t = 0; t < ntensors; ++t) {
    if (counts[t] == 0) continue;
    const uint64_t n = counts[t] * es;
    const uint64_t nt = (n + kCopyTile - 1) / kCopyTile;
    if (a.nitems == kMaxCopyItems || tiles + nt > 0xFFFFFFFFull) {
      if (ar_status_t st = flush(); st != AR_SUCCESS) return st;
      tiles = 0;
    }
    char* b = const_cast<char*>(bucket) + offsets[t] * es;
    CopyItem& it = a.item[a.nitems];
    it.src = flatten ? tens_in[t] : b;
    it.dst = flatten ? static_cast<void*>(b) : tens_out[t];
    it.bytes = n;
    a.tile_start[a.nitems] = (uint32_t)tiles;
    tiles += nt;
    a.nitems += 1;
    a.tile_start[a.nitems] = (uint32_t)tiles;
  }
  if (ar_status_t st = flush(); st != AR_SUCCESS) return st;
  return ok();
}

}  // namespace

extern "C" {

ar_status_t ar_bucket_flatten(const void* const* tensors, const size_t* counts, const size_t* offsets, int ntensors,
                              ar_dtype_t dtype, void* bucket, ar_stream_t stream) {
  AR_TRACE("ar_bucket_flatten");
  if (!bucket && ntensors > 0) return fail(AR_ERR_INVALID_ARGUMENT, "null bucket");
  return bucket_copy(tensors, nullptr, nullptr, bucket, counts, offsets, ntensors, dtype,
                     reinterpret_cast<cudaStream_t>(stream));
}

ar_status_t ar_bucket_unflatten(const void* bucket, void* const* tensors, const size_t* counts, const size_t* offsets,
                                int ntensors, ar_dtype_t dtype, ar_stream_t stream) {
  AR_TRACE("ar_bucket_unflatten");
  if (!bucket && ntensors > 0) return fail(AR_ERR_INVALID_ARGUMENT, "null bucket");
  return bucket_copy(nullptr, tensors, bucket, nullptr, counts, offsets, ntensors, dtype,
                     reinterpret_cast<cudaStream_t>(stream));
}

ar_status_t ar_bucket_allreduce(const void* const* tensors, void* const* out_tensors, int nranks, int ntensors,
                                const size_t* counts, const size_t* offsets, size_t bucket_count, ar_dtype_t dtype,
                                ar_op_t op, ar_algo_t algo, ar_stream_t stream) {
  AR_TRACE("ar_bucket_allreduce");
  ar_status_t st = common_checks(tensors, out_tensors, nranks, dtype);
  if (st != AR_SUCCESS) return st;
  if (!valid_op(op)) return fail(AR_ERR_INVALID_ARGUMENT, "unknown op");
  if ((st = basic_algo(&algo)) != AR_SUCCESS) return st;
  if (algo == AR_ALGO_TREE && !pow2(nranks))
    return fail(AR_ERR_UNSUPPORTED, "TREE needs nranks to be a power of two");
  if (ntensors < 0) return fail(AR_ERR_INVALID_ARGUMENT, "ntensors < 0");
  if (ntensors == 0 || bucket_count == 0) return ok();
  if (!counts || !offsets) return fail(AR_ERR_INVALID_ARGUMENT, "null counts/offsets");
  const size_t es = elem_size(dtype);
  if (bucket_count > SIZE_MAX / es / 4) return fail(AR_ERR_INVALID_ARGUMENT, "bucket too large");
  const size_t vecw = 16 / es;
  bool vec = true;
  std::vector<Span> spans;
  spans.reserve(2 * (size_t)nranks * (size_t)ntensors);
  std::vector<int> pair_in;
  std::vector<uintptr_t> pair_off;
  for (int t = 0; t < ntensors; ++t) {
    if (counts[t] == 0) continue;
    if (offsets[t] > bucket_count || counts[t] > bucket_count - offsets[t])
      return fail(AR_ERR_INVALID_ARGUMENT, "tensor " + std::to_string(t) + " lies outside the bucket");
    if (offsets[t] % vecw) vec = false;
    for (int r = 0; r < nranks; ++r) {
      const void* in = tensors[(size_t)r * ntensors + t];
      void* out = out_tensors[(size_t)r * ntensors + t];
      if (!in || !out) return fail(AR_ERR_INVALID_ARGUMENT, "null tensor pointer");
      if (!aligned(in, es) || !aligned(out, es))
        return fail(AR_ERR_INVALID_ARGUMENT, "tensor not aligned to the element size");
      if (!aligned(in, 16) || !aligned(out, 16)) vec = false;
      const int id = (int)pair_in.size();
      const uintptr_t n = counts[t] * es;
      spans.push_back({addr(in), addr(in) + n, false, id});
      spans.push_back({addr(out), addr(out) + n, true, id});
      pair_in.push_back(id);  // in place: out == in for the same rank and tensor
      pair_off.push_back(0);
    }
  }
  if (!overlap_ok(spans, pair_in, pair_off)) return fail(AR_ERR_ALIAS, "buffers overlap");
  const size_t L = chunk_len(bucket_count, nranks, vecw);
  const int mode = algo == AR_ALGO_TREE ? MODE_FUSED_TREE : MODE_FUSED_RING;
  const int per_launch = std::min(kBucketTensors, kBucketPtrs / nranks);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  BucketArgs a{};
  a.nranks = nranks;
  a.L = L;
  a.vec = vec ? 1 : 0;
  uint64_t tiles = 0;
  auto flush = [&]() -> ar_status_t {
    if (a.nt == 0) return AR_SUCCESS;
    // pointer slots are rank-major over the tensors of this launch
    const cudaError_t e = launch_bucket_reduce(dtype, op, mode, a, s);
    a.nt = 0;
    tiles = 0;
    return e == cudaSuccess ? AR_SUCCESS : cuda_fail(e, "bucket allreduce launch");
  };
  std::vector<int> batch;
  auto pack = [&]() -> ar_status_t {
    const int nt = (int)batch.size();
    a.nt = nt;
    tiles = 0;
    for (int j = 0; j < nt; ++j) {
      const int t = batch[j];
      a.count[j] = counts[t];
      a.offset[j] = offsets[t];
      a.tile_start[j] = (uint32_t)tiles;
      const uint64_t items = vec ? (counts[t] + vecw - 1) / vecw : counts[t];
      tiles += (items + kThreads - 1) / kThreads;
      for (int r = 0; r < nranks; ++r) {
        a.src[r * nt + j] = tensors[(size_t)r * ntensors + t];
        a.dst[r * nt + j] = out_tensors[(size_t)r * ntensors + t];
      }
    }
    a.tile_start[nt] = (uint32_t)tiles;
    batch.clear();
    return flush();
  };
  uint64_t batch_tiles = 0;
  for (int t = 0; t < ntensors; ++t) {
    if (counts[t] == 0) continue;
    const uint64_t items = vec ? (counts[t] + vecw - 1) / vecw : counts[t];
    const uint64_t nt_tiles = (items + kThreads - 1) / kThreads;
    if ((int)batch.size() == per_launch || batch_tiles + nt_tiles > 0x7FFFFFFFull) {
      if ((st = pack()) != AR_SUCCESS) return st;
      batch_tiles = 0;
    }
    batch.push_back(t);
    batch_tiles += nt_tiles;
  }
  if (!batch.empty() && (st = pack()) != AR_SUCCESS) return st;
  return ok();
}

size_t ar_fp8_workspace_bytes(int nranks, size_t count) {
  if (nranks < 1 || nranks > AR_MAX_RANKS || count > (SIZE_MAX >> 8) / AR_MAX_RANKS) return 0;
  const size_t qs = (count + 255) / 256 * 256;
  const size_t nblocks = (count + AR_FP8_BLOCK - 1) / AR_FP8_BLOCK;
  const size_t ss = (nblocks + 63) / 64 * 64 * sizeof(float);
  return (size_t)nranks * (qs + ss);
}

ar_status_t ar_quantize_fp8_blocks(const void* in, ar_dtype_t in_dtype, size_t count, uint8_t* q, float* scales,
                                   ar_stream_t stream) {
  AR_TRACE("ar_quantize_fp8_blocks");
  if (in_dtype != AR_F32 && in_dtype != AR_F16 && in_dtype != AR_BF16)
    return fail(AR_ERR_INVALID_ARGUMENT, "in_dtype must be F32, F16 or BF16");
  if (count == 0) return ok();
  if (!in || !q || !scales) return fail(AR_ERR_INVALID_ARGUMENT, "null pointer");
  const size_t es = elem_size(in_dtype);
  if (count > SIZE_MAX / es / 4) return fail(AR_ERR_INVALID_ARGUMENT, "count too large");
  if (!aligned(in, es) || !aligned(scales, 4))
    return fail(AR_ERR_INVALID_ARGUMENT, "buffer not aligned to its element size");
  const size_t nblocks = (count + AR_FP8_BLOCK - 1) / AR_FP8_BLOCK;
  std::vector<Span> spans = {{addr(in), addr(in) + count * es, false, 0},
                             {addr(q), addr(q) + count, true, 0},
                             {addr(scales), addr(scales) + nblocks * 4, true, 1}};
  if (!overlap_ok(spans, {}, {})) return fail(AR_ERR_ALIAS, "buffers overlap");
  Fp8QuantArgs a{};
  a.src[0] = in;
  a.q[0] = q;
  a.s[0] = scales;
  a.count = count;
  a.nranks = 1;
  const bool vec = aligned(in, 16) && aligned(q, 8);
  const cudaError_t e = launch_fp8_quant(in_dtype, vec, a, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok() : cuda_fail(e, "quantise launch");
}

}  // extern "C"

namespace gar {

// The checks of ar_allreduce_fp8 that come before its workspace: buffer
// arrays, rank count, types, op and order (AUTO resolves to the fused order).
ar_status_t fp8_arg_checks(const void* const* sendbufs, void* const* recvbufs, int nranks, ar_dtype_t in_dtype,
                           ar_dtype_t out_dtype, ar_op_t op, ar_algo_t* algo) {
  ar_status_t st = common_checks(sendbufs, recvbufs, nranks, in_dtype);
  if (st != AR_SUCCESS) return st;
  if (in_dtype == AR_I32) return fail(AR_ERR_UNSUPPORTED, "FP8 path needs a floating input type");
  if (elem_size(out_dtype) == 0) return fail(AR_ERR_INVALID_ARGUMENT, "unknown out_dtype");
  if (out_dtype == AR_I32) return fail(AR_ERR_UNSUPPORTED, "FP8 path needs a floating output type");
  if (!valid_op(op)) return fail(AR_ERR_INVALID_ARGUMENT, "unknown op");
  if (op != AR_SUM && op != AR_AVG) return fail(AR_ERR_UNSUPPORTED, "FP8 path supports SUM and AVG");
  if ((st = basic_algo(algo)) != AR_SUCCESS) return st;
  if (*algo == AR_ALGO_TREE && !pow2(nranks))
    return fail(AR_ERR_UNSUPPORTED, "TREE needs nranks to be a power of two");
  return AR_SUCCESS;
}

}  // namespace gar

extern "C" {

ar_status_t ar_allreduce_fp8(const void* const* sendbufs, void* const* recvbufs, int nranks, size_t count,
                             ar_dtype_t in_dtype, ar_dtype_t out_dtype, ar_op_t op, ar_algo_t algo, void* workspace,
                             size_t ws_bytes, ar_stream_t stream) {
  AR_TRACE("ar_allreduce_fp8");
  ar_status_t st = gar::fp8_arg_checks(sendbufs, recvbufs, nranks, in_dtype, out_dtype, op, &algo);
  if (st != AR_SUCCESS) return st;
  if (count == 0) return ok();
  const size_t need = ar_fp8_workspace_bytes(nranks, count);
  if (need == 0) return fail(AR_ERR_INVALID_ARGUMENT, "count too large");
  if (!workspace) return fail(AR_ERR_INVALID_ARGUMENT, "null workspace");
  if (ws_bytes < need) return fail(AR_ERR_INVALID_ARGUMENT, "workspace too small");
  if (!aligned(workspace, 16)) return fail(AR_ERR_INVALID_ARGUMENT, "workspace must be 16-byte aligned");
  const size_t ies = elem_size(in_dtype), oes = elem_size(out_dtype);
  if ((st = check_ptrs(sendbufs, nranks, ies, "sendbufs")) != AR_SUCCESS) return st;
  if ((st = check_ptrs(recvbufs, nranks, oes, "recvbufs")) != AR_SUCCESS) return st;
  std::vector<Span> spans;
  for (int r = 0; r < nranks; ++r) {
    spans.push_back({addr(sendbufs[r]), addr(sendbufs[r]) + count * ies, false, r});
    spans.push_back({addr(recvbufs[r]), addr(recvbufs[r]) + count * oes, true, r});
  }
  spans.push_back({addr(workspace), addr(workspace) + need, true, nranks});
  if (!overlap_ok(spans, {}, {})) return fail(AR_ERR_ALIAS, "buffers overlap");

  const size_t qs = (count + 255) / 256 * 256;
  const size_t ss = ((count + AR_FP8_BLOCK - 1) / AR_FP8_BLOCK + 63) / 64 * 64 * sizeof(float);
  char* ws = static_cast<char*>(workspace);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  Fp8QuantArgs qa{};
  qa.nranks = nranks;
  qa.count = count;
  for (int r = 0; r < nranks; ++r) {
    qa.src[r] = sendbufs[r];
    qa.q[r] = reinterpret_cast<uint8_t*>(ws + (size_t)r * qs);
    qa.s[r] = reinterpret_cast<float*>(ws + (size_t)nranks * qs + (size_t)r * ss);
  }
  cudaError_t e = launch_fp8_quant(in_dtype, all_aligned16(sendbufs, nranks), qa, s);
  if (e != cudaSuccess) return cuda_fail(e, "quantise launch");

  const size_t L = chunk_len(count, nranks, 16 / oes);
  const bool vec = all_aligned16(recvbufs, nranks);
  Fp8ReduceArgs ra{};
  ra.nranks = nranks;
  ra.count = count;
  ra.L = L;
  ra.vec = vec ? 1 : 0;
  for (int r = 0; r < nranks; ++r) {
    ra.q[r] = qa.q[r];
    ra.s[r] = qa.s[r];
  }
  if (algo == AR_ALGO_RING) {
    for (int c = 0; c < nranks; ++c)
      ra.dst[c] = static_cast<char*>(recvbufs[c]) + ((size_t)c * L < count ? (size_t)c * L * oes : 0);
    e = launch_fp8_reduce(out_dtype, op, MODE_RS, ra, s);
    if (e != cudaSuccess) return cuda_fail(e, "fp8 reduce-scatter launch");
    if ((st = ring_gather(recvbufs, nranks, count, L, oes, vec, s)) != AR_SUCCESS) return st;
    return ok();
  }
  for (int r = 0; r < nranks; ++r) ra.dst[r] = recvbufs[r];
  e = launch_fp8_reduce(out_dtype, op, algo == AR_ALGO_TREE ? MODE_FUSED_TREE : MODE_FUSED_RING, ra, s);
  return e == cudaSuccess ? ok() : cuda_fail(e, "fp8 allreduce launch");
}


ar_status_t ar_allreduce_fp8_hops(const void* const* sendbufs, void* const* recvbufs, int nranks, size_t count,
                                  ar_dtype_t in_dtype, ar_dtype_t out_dtype, ar_op_t op, ar_stream_t stream) {
  AR_TRACE("ar_allreduce_fp8_hops");
  ar_status_t st = common_checks(sendbufs, recvbufs, nranks, in_dtype);
  if (st != AR_SUCCESS) return st;
  if (in_dtype == AR_I32) return fail(AR_ERR_UNSUPPORTED, "FP8 path needs a floating input type");
  if (elem_size(out_dtype) == 0) return fail(AR_ERR_INVALID_ARGUMENT, "unknown out_dtype");
  if (out_dtype == AR_I32) return fail(AR_ERR_UNSUPPORTED, "FP8 path needs a floating output type");
  if (!valid_op(op)) return fail(AR_ERR_INVALID_ARGUMENT, "unknown op");
  if (op != AR_SUM && op != AR_AVG) return fail(AR_ERR_UNSUPPORTED, "FP8 path supports SUM and AVG");
  if (count == 0) return ok();
  const size_t ies = elem_size(in_dtype), oes = elem_size(out_dtype);
  if (count > SIZE_MAX / 8 / (size_t)nranks) return fail(AR_ERR_INVALID_ARGUMENT, "count too large");
  if ((st = check_ptrs(sendbufs, nranks, ies, "sendbufs")) != AR_SUCCESS) return st;
  if ((st = check_ptrs(recvbufs, nranks, oes, "recvbufs")) != AR_SUCCESS) return st;
  std::vector<Span> spans;
  for (int r = 0; r < nranks; ++r) {
    spans.push_back({addr(sendbufs[r]), addr(sendbufs[r]) + count * ies, false, r});
    spans.push_back({addr(recvbufs[r]), addr(recvbufs[r]) + count * oes, true, r});
  }
  if (!overlap_ok(spans, {}, {})) return fail(AR_ERR_ALIAS, "buffers overlap");
  Fp8HopArgs a{};
  a.nranks = nranks;
  a.count = count;
  a.L = chunk_len(count, nranks, 16 / oes);
  a.nbc = (a.L + AR_FP8_BLOCK - 1) / AR_FP8_BLOCK;
  for (int r = 0; r < nranks; ++r) {
    a.src[r] = sendbufs[r];
    a.dst[r] = recvbufs[r];
  }
  const cudaError_t e = launch_fp8_hop(in_dtype, out_dtype, op, a, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok() : cuda_fail(e, "per-hop fp8 allreduce launch");
}

ar_status_t ar_allreduce_fp8_fused(const void* const* sendbufs, void* const* recvbufs, int nranks, size_t count,
                                   ar_dtype_t in_dtype, ar_dtype_t out_dtype, ar_op_t op, ar_algo_t algo,
                                   ar_stream_t stream) {
  AR_TRACE("ar_allreduce_fp8_fused");
  ar_status_t st = common_checks(sendbufs, recvbufs, nranks, in_dtype);
  if (st != AR_SUCCESS) return st;
  if (in_dtype == AR_I32) return fail(AR_ERR_UNSUPPORTED, "FP8 path needs a floating input type");
  if (elem_size(out_dtype) == 0) return fail(AR_ERR_INVALID_ARGUMENT, "unknown out_dtype");
  if (out_dtype == AR_I32) return fail(AR_ERR_UNSUPPORTED, "FP8 path needs a floating output type");
  if (elem_size(in_dtype) == 2 && elem_size(out_dtype) == 4)
    return fail(AR_ERR_UNSUPPORTED, "fused FP8 path: 16-bit inputs need a 16-bit output type");
  if (!valid_op(op)) return fail(AR_ERR_INVALID_ARGUMENT, "unknown op");
  if (op != AR_SUM && op != AR_AVG) return fail(AR_ERR_UNSUPPORTED, "FP8 path supports SUM and AVG");
  if ((st = basic_algo(&algo)) != AR_SUCCESS) return st;
  if (algo == AR_ALGO_TREE && !pow2(nranks))
    return fail(AR_ERR_UNSUPPORTED, "TREE needs nranks to be a power of two");
  if (count == 0) return ok();
  const size_t ies = elem_size(in_dtype), oes = elem_size(out_dtype);
  if (count > SIZE_MAX / 8 / (size_t)nranks) return fail(AR_ERR_INVALID_ARGUMENT, "count too large");
  if ((st = check_ptrs(sendbufs, nranks, ies, "sendbufs")) != AR_SUCCESS) return st;
  if ((st = check_ptrs(recvbufs, nranks, oes, "recvbufs")) != AR_SUCCESS) return st;
  std::vector<Span> spans;
  for (int r = 0; r < nranks; ++r) {
    spans.push_back({addr(sendbufs[r]), addr(sendbufs[r]) + count * ies, false, r});
    spans.push_back({addr(recvbufs[r]), addr(recvbufs[r]) + count * oes, true, r});
  }
  if (!overlap_ok(spans, {}, {})) return fail(AR_ERR_ALIAS, "buffers overlap");

  Fp8FusedArgs a{};
  a.nranks = nranks;
  a.count = count;
  a.L = chunk_len(count, nranks, 16 / oes);
  for (int r = 0; r < nranks; ++r) {
    a.src[r] = sendbufs[r];
    a.dst[r] = recvbufs[r];
  }
  const bool vec = all_aligned16(sendbufs, nranks) && all_aligned16(recvbufs, nranks);
  const uint64_t nfull = count / AR_FP8_BLOCK;
  const int mode = algo == AR_ALGO_TREE ? MODE_FUSED_TREE : MODE_FUSED_RING;
  if (!vec) {
    a.first_block = 0;  // every block on the element-wise kernel
  } else {
    a.first_block = nfull;  // the short last block, if any
    if (mode == MODE_FUSED_RING) {
      // a warp of the vector kernel covers BPW blocks and needs them in one
      // chunk; list the blocks of each warp that a chunk boundary cuts
      const uint64_t bpw = 32 / (AR_FP8_BLOCK * ies / 16);
      uint64_t last_w = UINT64_MAX;
      for (int c = 1; c < nranks; ++c) {
        const uint64_t e = (uint64_t)c * a.L;
        if (e >= nfull * AR_FP8_BLOCK) break;
        const uint64_t w = e / AR_FP8_BLOCK / bpw;
        if (e == w * bpw * AR_FP8_BLOCK || w == last_w) continue;
        last_w = w;
        for (uint64_t b = w * bpw; b < (w + 1) * bpw && b < nfull; ++b) {
          if (a.nlist == kFusedList) return fail(AR_ERR_UNSUPPORTED, "too many chunk boundaries");
          a.list[a.nlist++] = b;
        }
      }
    }
  }
  const cudaError_t e = launch_fp8_fused(in_dtype, out_dtype, op, mode, vec, a, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok() : cuda_fail(e, "fused fp8 allreduce launch");
}

}  // extern "C"

namespace gar {
// Lets other translation units of the library report an error through
// ar_last_error() for the calling thread.
void set_last_error(const std::string& msg) { g_last_error = msg; }
}  // namespace gar
