// noalloc.cu -- a decode entry point for callers that cannot allocate device
// memory.
//
// mla_decode_run needs a caller-provided workspace.  Some callers have no way
// to obtain one: a custom operator inside a serving engine that owns every
// byte of device memory through its own pool and hands an operator only its
// input and output buffers, or code that runs while a stream is being
// captured into a CUDA graph under a capture mode that forbids new
// allocations.  For them this file keeps a fixed-size scratch buffer in
// statically allocated device memory, which exists from module load until the
// process exits, and runs the planner and the four decode steps on it.
//
// Nothing here calls cudaMalloc, cudaFree or any allocating library routine.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/mla_decode.h"
#include "host_checks.h"

namespace {

// 32 MiB per device that loads the library.  Enough for decode batches with up
// to 32 query rows per sequence (T * H), e.g. 64 sequences x 16 heads needs
// about 13 MiB; larger batches are rejected.
constexpr size_t kStaticScratchBytes = static_cast<size_t>(32) << 20;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;

// Per device: the context the address was looked up in (by its
// process-unique id) and the address itself.
struct ScratchEntry {
  unsigned long long ctx_id;
  void* ptr;
};
ScratchEntry g_scratch[kMaxDevices];
std::mutex g_scratch_mu;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
CtxGetCurrentFn g_ctx_current = nullptr;
CtxGetIdFn g_ctx_id = nullptr;
std::once_flag g_ctx_once;

template <typename Fn>
Fn driver_fn(const char* name) {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q{};
  if (cudaGetDriverEntryPointByVersion(name, &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    return reinterpret_cast<Fn>(fn);
  cudaGetLastError();
  return nullptr;
}

// Process-unique id of the calling thread's current context (0 on failure).
unsigned long long current_context_id() {
  std::call_once(g_ctx_once, []() {
    g_ctx_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
    g_ctx_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  });
  if (!g_ctx_current || !g_ctx_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (g_ctx_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of this device's copy of the scratch array.  In host code the
// array's name is only a host-side stand-in, so the address is looked up with
// the device current, once per device and context: a new context (after
// cudaDeviceReset, for example) loads the module anew and the array may sit
// elsewhere, so a changed context id triggers a fresh lookup.
int scratch_for_current_device(void** ptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return MLA_DECODE_CUDA_ERROR;
  }
  // Makes the device's primary context current if no runtime call has yet
  // (the context is what the cached address belongs to).
  if (cudaSetDevice(dev) != cudaSuccess) {
    cudaGetLastError();
    return MLA_DECODE_CUDA_ERROR;
  }
  const unsigned long long id = current_context_id();
  if (id == 0) return MLA_DECODE_CUDA_ERROR;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  ScratchEntry& e = g_scratch[dev];
  if (e.ptr == nullptr || e.ctx_id != id) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return MLA_DECODE_CUDA_ERROR;
    }
    e.ptr = p;
    e.ctx_id = id;
  }
  *ptr = e.ptr;
  return MLA_DECODE_OK;
}

}  // namespace

extern "C" int mla_decode_run_static_scratch(const mla_decode_dims* dims, const void* q,
                                             const void* kv_cache, const int32_t* block_table,
                                             const int32_t* seq_lens, const void* w_uk,
                                             const void* w_uv, float softmax_scale, void* out,
                                             float* lse, void* stream) {
  // Every argument first, so that a host-detected error enqueues nothing (and
  // leaves a call still in flight on the shared array untouched).
  int rc = mla::check_run_inputs(dims, q, kv_cache, block_table, seq_lens, w_uk, w_uv, false,
                                 nullptr, nullptr, softmax_scale, out, lse);
  if (rc != MLA_DECODE_OK) return rc;
  size_t need = 0;
  rc = mla_decode_workspace_size(dims, &need);
  if (rc != MLA_DECODE_OK) return rc;
  if (need > kStaticScratchBytes) return MLA_DECODE_WORKSPACE_TOO_SMALL;
  void* ws = nullptr;
  rc = scratch_for_current_device(&ws);
  if (rc != MLA_DECODE_OK) return rc;
  // The plan clears the status word; every other region the steps read is
  // written earlier in the same call, so the previous call's contents do not
  // matter.
  rc = mla_decode_plan(dims, seq_lens, ws, kStaticScratchBytes, stream);
  if (rc != MLA_DECODE_OK) return rc;
  return mla_decode_run(dims, q, kv_cache, block_table, seq_lens, w_uk, w_uv, softmax_scale, out,
                        lse, ws, kStaticScratchBytes, stream);
}
