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
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/mla_decode.h"

namespace {

// 32 MiB per device that loads the library.  Enough for decode batches with up
// to 32 query rows per sequence (T * H), e.g. 64 sequences x 16 heads needs
// about 13 MiB; larger batches are rejected.
constexpr size_t kStaticScratchBytes = static_cast<size_t>(32) << 20;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of this device's copy of the scratch array.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device, with that device current.
int scratch_for_current_device(void** ptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return MLA_DECODE_CUDA_ERROR;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return MLA_DECODE_CUDA_ERROR;
    }
    g_scratch_ptr[dev] = p;
  }
  *ptr = g_scratch_ptr[dev];
  return MLA_DECODE_OK;
}

}  // namespace

extern "C" int mla_decode_run_static_scratch(const mla_decode_dims* dims, const void* q,
                                             const void* kv_cache, const int32_t* block_table,
                                             const int32_t* seq_lens, const void* w_uk,
                                             const void* w_uv, float softmax_scale, void* out,
                                             float* lse, void* stream) {
  size_t need = 0;
  int rc = mla_decode_workspace_size(dims, &need);
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
