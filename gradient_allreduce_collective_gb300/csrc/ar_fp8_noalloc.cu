// ar_fp8_noalloc.cu — the FP8-compressed allreduce for callers that cannot
// allocate device memory.
//
// ar_allreduce_fp8 needs a caller-provided workspace for the quantised codes
// and block scales. Some callers have no way to provide one: code that runs
// where the allocator may not be called (inside a custom allocator or memory
// pool's own callbacks, under a framework that forbids allocation on its
// hot path, or a C host without access to the CUDA allocation API at all).
// This entry point instead uses a fixed workspace that lives in the library
// itself, as a file-scope __device__ array.
//
// Host code only sees a host-side stand-in for that array's name, never its
// device address; the address is fetched with cudaGetSymbolAddress once per
// device (on the first call made while that device is current) and cached.
#include <atomic>
#include <string>

#include <cuda_runtime.h>

#include "ar.h"
#include "ar_internal.h"

namespace gar {
void set_last_error(const std::string& msg);
}

namespace {

// Shared by every call on a device; held for as long as the library stays
// loaded. Every byte a call reads from it is written earlier in the same call
// (codes and scales of every block of every rank), so nothing needs clearing.
static __device__ __align__(256) unsigned char g_fp8_static_ws[AR_FP8_STATIC_WS_BYTES];

std::atomic<void*> g_ws_addr[gar::kMaxRanks];  // device address per device id

ar_status_t ws_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    gar::set_last_error(std::string("cudaGetDevice: ") + cudaGetErrorString(e));
    return AR_ERR_CUDA;
  }
  if (dev < 0 || dev >= gar::kMaxRanks) {
    gar::set_last_error("device index beyond the static workspace table");
    return AR_ERR_UNSUPPORTED;
  }
  void* p = g_ws_addr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    e = cudaGetSymbolAddress(&p, g_fp8_static_ws);
    if (e != cudaSuccess || p == nullptr) {
      gar::set_last_error(std::string("cudaGetSymbolAddress of the static FP8 workspace: ") +
                          cudaGetErrorString(e));
      return AR_ERR_CUDA;
    }
    g_ws_addr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return AR_SUCCESS;
}

}  // namespace

extern "C" ar_status_t ar_allreduce_fp8_noalloc(const void* const* sendbufs, void* const* recvbufs, int nranks,
                                                size_t count, ar_dtype_t in_dtype, ar_dtype_t out_dtype, ar_op_t op,
                                                ar_algo_t algo, ar_stream_t stream) {
  if (count == 0 || nranks < 1 || nranks > AR_MAX_RANKS) {
    // nothing to place in the workspace; the regular entry point handles the
    // argument checks and the empty call
    return ar_allreduce_fp8(sendbufs, recvbufs, nranks, count, in_dtype, out_dtype, op, algo, nullptr, 0, stream);
  }
  const size_t need = ar_fp8_workspace_bytes(nranks, count);
  if (need == 0 || need > (size_t)AR_FP8_STATIC_WS_BYTES) {
    gar::set_last_error("the static FP8 workspace holds " + std::to_string((size_t)AR_FP8_STATIC_WS_BYTES) +
                        " bytes; this call needs " + std::to_string(need) +
                        " (ar_fp8_workspace_bytes); use ar_allreduce_fp8 with a caller workspace");
    return AR_ERR_INVALID_ARGUMENT;
  }
  void* ws = nullptr;
  const ar_status_t st = ws_address(&ws);
  if (st != AR_SUCCESS) return st;
  return ar_allreduce_fp8(sendbufs, recvbufs, nranks, count, in_dtype, out_dtype, op, algo, ws,
                          (size_t)AR_FP8_STATIC_WS_BYTES, stream);
}
