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
// device address; the address is fetched with cudaGetSymbolAddress on the
// first call made in each CUDA context (in practice once per device: the
// device's primary context) and cached together with that context's ID. A
// call in a new context — after cudaDeviceReset, or from a thread whose
// current context was created later — fetches it again, so a stale address
// is never passed to a kernel.
#include <cuda.h>  // context types only; the driver functions are reached through the runtime
#include <mutex>
#include <string>

#include <cuda_runtime.h>

#include "ar.h"
#include "ar_internal.h"

namespace gar {
void set_last_error(const std::string& msg);
ar_status_t fp8_arg_checks(const void* const* sendbufs, void* const* recvbufs, int nranks, ar_dtype_t in_dtype,
                           ar_dtype_t out_dtype, ar_op_t op, ar_algo_t* algo);
}

namespace {

// Shared by every call on a device; held for as long as the library stays
// loaded. Every byte a call reads from it is written earlier in the same call
// (codes and scales of every block of every rank), so nothing needs clearing.
static __device__ __align__(256) unsigned char g_fp8_static_ws[AR_FP8_STATIC_WS_BYTES];

constexpr int kMaxDevices = 64;

struct DeviceWs {
  std::mutex m;
  bool valid = false;  // addr belongs to the context ctx_id
  unsigned long long ctx_id = 0;
  void* addr = nullptr;
};
DeviceWs g_ws[kMaxDevices];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// The driver's cuCtxGetCurrent and cuCtxGetId (CUDA 12.0 ABI), looked up once
// through the runtime so the library does not link the driver library.
struct DriverFns {
  CtxGetCurrentFn get_current = nullptr;
  CtxGetIdFn get_id = nullptr;
};

const DriverFns& driver_fns() {
  static const DriverFns fns = [] {
    DriverFns f;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.get_id = reinterpret_cast<CtxGetIdFn>(p);
    return f;
  }();
  return fns;
}

ar_status_t cuda_error(const char* what, cudaError_t e) {
  (void)cudaGetLastError();  // reported here, not again by a later check elsewhere
  gar::set_last_error(std::string(what) + ": " + cudaGetErrorString(e));
  return AR_ERR_CUDA;
}

// Device address of the array in the calling thread's current context.
ar_status_t ws_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_error("cudaGetDevice", e);
  if (dev < 0 || dev >= kMaxDevices) {
    gar::set_last_error("device index beyond the static workspace table");
    return AR_ERR_UNSUPPORTED;
  }
  // makes the device's primary context current on this thread if no context is
  e = cudaSetDevice(dev);
  if (e != cudaSuccess) return cuda_error("cudaSetDevice", e);
  const DriverFns& fns = driver_fns();
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!fns.get_current || !fns.get_id || fns.get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
      fns.get_id(ctx, &id) != CUDA_SUCCESS) {
    gar::set_last_error("cannot identify the current CUDA context (cuCtxGetCurrent / cuCtxGetId)");
    return AR_ERR_CUDA;
  }
  DeviceWs& w = g_ws[dev];
  std::lock_guard<std::mutex> lock(w.m);
  if (!w.valid || w.ctx_id != id) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_fp8_static_ws);
    if (e != cudaSuccess || p == nullptr)
      return cuda_error("cudaGetSymbolAddress of the static FP8 workspace", e);
    w.addr = p;
    w.ctx_id = id;
    w.valid = true;
  }
  *out = w.addr;
  return AR_SUCCESS;
}

}  // namespace

extern "C" ar_status_t ar_allreduce_fp8_noalloc(const void* const* sendbufs, void* const* recvbufs, int nranks,
                                                size_t count, ar_dtype_t in_dtype, ar_dtype_t out_dtype, ar_op_t op,
                                                ar_algo_t algo, ar_stream_t stream) {
  ar_algo_t a = algo;
  const ar_status_t chk = gar::fp8_arg_checks(sendbufs, recvbufs, nranks, in_dtype, out_dtype, op, &a);
  if (chk != AR_SUCCESS) return chk;
  if (count == 0)  // nothing to place in the workspace: the regular entry point's empty call
    return ar_allreduce_fp8(sendbufs, recvbufs, nranks, count, in_dtype, out_dtype, op, algo, nullptr, 0, stream);
  const size_t need = ar_fp8_workspace_bytes(nranks, count);
  if (need == 0) {
    gar::set_last_error("count too large");
    return AR_ERR_INVALID_ARGUMENT;
  }
  if (need > (size_t)AR_FP8_STATIC_WS_BYTES) {
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
