// aq_noalloc.cu -- aq_linear_noalloc: the reconstruction linear for callers that are not
// allowed to allocate device memory.
//
// aq_linear needs a small scratch area (t = V^T x, and for more than 64 tokens a
// transposed copy of V) that its caller normally allocates. Some callers cannot do that:
// a plugin inside an inference runtime that owns all device memory and hands plugins
// only their input and output buffers, a serving loop that forbids allocation after
// start-up (cudaMalloc can synchronise the device and fragments a fixed memory budget),
// or code running where no allocator is reachable at all. For them the scratch lives in
// one fixed array compiled into this library.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdio.h>

#include <mutex>

#include "aq.h"
#include "aq_internal.h"

// The scratch area. Every GPU on which this library is used holds these bytes until the
// process exits. All calls on a device share it; it keeps whatever the last call wrote.
// Being a static device array it starts at zero, which is what the workspace's sync part
// (its first AQ_WORKSPACE_SYNC_BYTES) needs; every completed call leaves that part zero.
static __device__ __align__(256) unsigned char aq_noalloc_scratch[AQ_NOALLOC_WORKSPACE_BYTES];

namespace aq {
// The workspace a call cannot run without (aq_linear_workspace_bytes adds room for optional
// split-K partial sums, which the scratch holds as far as it goes).
size_t linear_workspace_min_bytes(const aq_theta* th, int32_t n_theta, int64_t M);
}  // namespace aq

namespace {

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

// The current context, through the driver entry point (the runtime exposes no handle of
// its own). A context torn down and created again -- cudaDeviceReset, for one -- reloads
// this library's device code, and the array's address may then differ.
CUcontext current_context() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  CUcontext c = nullptr;
  if (fn && fn(&c) != CUDA_SUCCESS) c = nullptr;
  return c;
}

std::mutex g_scratch_mu;
// device address of aq_noalloc_scratch per device index, and the context it was looked up in
void* g_scratch_ptr[64] = {};
CUcontext g_scratch_ctx[64] = {};

// In host code the array's name is only a host-side stand-in; the kernels need its
// device address, which is looked up with the device current: once per device, and again
// whenever the device's current context is no longer the one of the last lookup.
aq_status scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    char msg[256];
    snprintf(msg, sizeof msg, "aq_linear_noalloc: cudaGetDevice failed: %s", cudaGetErrorString(e));
    return static_cast<aq_status>(aq::set_last_error(AQ_ERR_CUDA, msg));
  }
  if (dev < 0 || dev >= 64)
    return static_cast<aq_status>(aq::set_last_error(AQ_ERR_UNSUPPORTED, "aq_linear_noalloc: device index out of range"));
  const CUcontext ctx = current_context();
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr || ctx != g_scratch_ctx[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, aq_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      char msg[256];
      snprintf(msg, sizeof msg, "aq_linear_noalloc: cudaGetSymbolAddress of the scratch array failed: %s",
               cudaGetErrorString(e));
      return static_cast<aq_status>(aq::set_last_error(AQ_ERR_CUDA, msg));
    }
    g_scratch_ptr[dev] = p;
    g_scratch_ctx[dev] = current_context();
  }
  *out = g_scratch_ptr[dev];
  return AQ_OK;
}

}  // namespace

extern "C" aq_status aq_linear_noalloc(const aq_theta* th, const void* x, int64_t M, int64_t ldx, void* y,
                                       int64_t ldy, void* stream) {
  if (!th) return static_cast<aq_status>(aq::set_last_error(AQ_ERR_INVALID_ARG, "aq_linear_noalloc: theta is NULL"));
  const size_t need = aq::linear_workspace_min_bytes(th, 1, M);
  if (need == static_cast<size_t>(-1))  // invalid sizes: let aq_linear's validation name them
    return aq_linear(th, x, M, ldx, y, ldy, nullptr, 0, stream);
  if (need > static_cast<size_t>(AQ_NOALLOC_WORKSPACE_BYTES)) {
    char msg[256];
    snprintf(msg, sizeof msg,
             "aq_linear_noalloc: M=%lld, r=%d, in=%d needs %zu bytes of scratch, more than the %u bytes "
             "built into the library; use aq_linear with a caller-provided workspace",
             (long long)M, th->r, th->in, need, (unsigned)AQ_NOALLOC_WORKSPACE_BYTES);
    return static_cast<aq_status>(aq::set_last_error(AQ_ERR_WORKSPACE, msg));
  }
  // A call that needs no scratch may still split K into slices whose partial sums live in
  // it (r = 0 prefill calls with few output tiles): hand it the array whenever a full-size
  // workspace would be nonzero.
  if (need == 0 && aq_linear_workspace_bytes(th, 1, M) == 0) return aq_linear(th, x, M, ldx, y, ldy, nullptr, 0, stream);
  void* scratch = nullptr;
  aq_status st = scratch_address(&scratch);
  if (st != AQ_OK) return st;
  return aq_linear(th, x, M, ldx, y, ldy, scratch, AQ_NOALLOC_WORKSPACE_BYTES, stream);
}

extern "C" aq_status aq_noalloc_scratch_read(void* dst, size_t offset, size_t bytes, void* stream) {
  if (!dst || offset > AQ_NOALLOC_WORKSPACE_BYTES || bytes > AQ_NOALLOC_WORKSPACE_BYTES - offset)
    return static_cast<aq_status>(
        aq::set_last_error(AQ_ERR_INVALID_ARG, "aq_noalloc_scratch_read: range outside the scratch array"));
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyFromSymbolAsync(dst, aq_noalloc_scratch, bytes, offset, cudaMemcpyDefault, cs);
  if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
  if (e != cudaSuccess) {
    char msg[256];
    snprintf(msg, sizeof msg, "aq_noalloc_scratch_read: %s", cudaGetErrorString(e));
    return static_cast<aq_status>(aq::set_last_error(AQ_ERR_CUDA, msg));
  }
  return AQ_OK;
}
