// api.cu -- the C ABI declared in include/mla_decode.h: argument validation,
// workspace layout, TMA descriptor encoding and kernel launches.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/mla_decode.h"
#include "common.cuh"
#include "host_checks.h"
#include "ptx.cuh"

namespace mla {
cudaError_t launch_plan(const int32_t* seq_lens, int B, int T, int max_pages, int R,
                        int32_t* status, PlanHeader* header, int32_t* range_b, int32_t* range_p,
                        int32_t* seq_first, int32_t* seq_nsplit, int32_t* seq_slot,
                        int32_t* seq_len_eff, int32_t* prefix, cudaStream_t stream);
int bmm_token_tile(int BT, bool absorb);
cudaError_t launch_absorb(const CUtensorMap& tm_wuk, const CUtensorMap& tm_q,
                          const CUtensorMap* tm_qlat, const CUtensorMap* tm_qlo, int BT, int H,
                          const __nv_bfloat16* q, __nv_bfloat16* qlat, uint8_t* qlo,
                          int32_t* status, cudaStream_t st, const uint8_t* wuk8,
                          const float* wuk_scale, int sm_count);
cudaError_t launch_up_project(const CUtensorMap& tm_wuv, const CUtensorMap& tm_olat, int BT,
                              int H, __nv_bfloat16* out, int32_t* status, cudaStream_t st,
                              const uint8_t* wuv8, const float* wuv_scale, bool one_wave);
int decode_tiles(int T, int H);
int decode_q_box_rows(int T, int H);
cudaError_t decode_default_ranges(int T, int H, int sm_count, int* ranges);
cudaError_t launch_decode(const CUtensorMap& tm_q, const CUtensorMap& tm_c, int sm_count,
                          const int32_t* block_table, const int32_t* seq_len_eff,
                          const PlanHeader* header, void* ws, const int32_t* seq_first,
                          const int32_t* seq_nsplit, const int32_t* seq_slot,
                          __nv_bfloat16* olat, float* lse,
                          int32_t* status, int B, int T, int H, int max_pages,
                          int num_pages, float scale, cudaStream_t st);
cudaError_t launch_up_project_rows(const CUtensorMap& tm_wuv, const CUtensorMap& tm_olat,
                                   const CUtensorMap& tm_qlo, const CUtensorMap& tm_out, int BT,
                                   int T, int H, const int32_t* seq_nsplit, float* lse,
                                   float scale, int32_t* status, const float* wuv_scale,
                                   int sm_count, cudaStream_t st);
cudaError_t launch_combine(const int32_t* seq_nsplit, const int32_t* seq_slot, const void* ws,
                           const PlanHeader* header, const uint8_t* qlo,
                           __nv_bfloat16* olat, float* lse, int B, int T, int H, float scale,
                           int splits_per_seq, int split_ranges, int32_t* status,
                           cudaStream_t st);
int combine_up_tile();
cudaError_t launch_combine_up(const CUtensorMap& tm_wuv, int B, int T, int H, const void* ws,
                              const PlanHeader* header, const int32_t* seq_nsplit,
                              const int32_t* seq_slot, const uint8_t* qlo,
                              const __nv_bfloat16* olat, float* lse, float scale,
                              __nv_bfloat16* out, int32_t* status, int splits_per_seq,
                              const float* wuv_scale, cudaStream_t st);
}  // namespace mla

namespace {

// One thread waits, through the same bounded wait as every pipeline barrier
// of the library, on an mbarrier that nothing ever arrives on.  The wait gives
// up after its time limit, records TIMEOUT in *status and the kernel exits.
__global__ void wait_timeout_kernel(int32_t* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mla::mbar_init(mla::smem_u32(&bar), 1);
    abort_flag = 0;
    mla::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mla::mbar_wait(mla::smem_u32(&bar), 0, &abort_flag, status);
}

}  // namespace

using namespace mla;

namespace {

constexpr int kMaxDevices = 64;
int g_sm_count[kMaxDevices];
std::once_flag g_sm_once[kMaxDevices];

int sm_count(int* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return MLA_DECODE_CUDA_ERROR;
  }
  std::call_once(g_sm_once[dev], [dev]() {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) n = 0;
    g_sm_count[dev] = n;
  });
  if (g_sm_count[dev] <= 0) {
    cudaGetLastError();
    return MLA_DECODE_CUDA_ERROR;
  }
  *out = g_sm_count[dev];
  return MLA_DECODE_OK;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;

EncodeTiledFn encoder() {
  std::call_once(g_encode_once, []() {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    else
      cudaGetLastError();
  });
  return g_encode;
}

// 2-D tensor map of bf16 (or, with elem_bytes = 1, byte) elements: `rows` x
// `cols` (row stride `row_stride` elements), box = box_cols x box_rows,
// 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint64_t row_stride,
              uint32_t box_cols, uint32_t box_rows, bool stream_hint, int elem_bytes = 2,
              bool swizzle = true) {
  EncodeTiledFn enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {row_stride * elem_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, elem_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                      : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                   2, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                   stream_hint ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B
                               : CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int cuda_rc(cudaError_t e) {
  if (e == cudaSuccess) return MLA_DECODE_OK;
  cudaGetLastError();
  return MLA_DECODE_CUDA_ERROR;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_dims(const mla_decode_dims* d) {
  if (!d) return MLA_DECODE_INVALID_ARG;
  if (d->qk_nope != kNope || d->qk_rope != kRope || d->kv_lora != kLora ||
      d->v_head != kVHead || d->page_size != kPage)
    return MLA_DECODE_UNSUPPORTED;
  if (d->q_len < 1 || d->q_len > kMaxQLen) return MLA_DECODE_UNSUPPORTED;
  if (d->num_heads < 16 || d->num_heads > 128 || d->num_heads % 16 != 0)
    return MLA_DECODE_UNSUPPORTED;
  if (d->batch < 1 || d->batch > 65535) return MLA_DECODE_INVALID_ARG;
  if (d->num_pages < 1 || d->max_pages_per_seq < 1) return MLA_DECODE_INVALID_ARG;
  // Row coordinates of the cache tensor map and key indices are int32.
  if (static_cast<int64_t>(d->num_pages) * kPage > INT32_MAX) return MLA_DECODE_INVALID_ARG;
  if (static_cast<int64_t>(d->max_pages_per_seq) * kPage > INT32_MAX / 2)
    return MLA_DECODE_INVALID_ARG;
  if (static_cast<int64_t>(d->batch) * d->q_len * d->num_heads > INT32_MAX / kDqk)
    return MLA_DECODE_INVALID_ARG;
  return MLA_DECODE_OK;
}

// Default number of work ranges: one per co-resident decode CTA group (a
// group = the CTAs covering all query rows of a sequence), or, when those
// groups would leave SMs idle, enough for every SM to take the same number of
// (range, tile set) tasks (decode_default_ranges).  Cached per device and
// (q_len, heads).
int g_groups[kMaxDevices][kMaxQLen + 1][9];
std::mutex g_groups_mu;

int default_ranges(const mla_decode_dims* d, int* R) {
  int sms = 0;
  int rc = sm_count(&sms);
  if (rc) return rc;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cuda_rc(cudaErrorUnknown);
  const int hi = d->num_heads / 16;
  std::lock_guard<std::mutex> lock(g_groups_mu);
  int& slot = g_groups[dev][d->q_len][hi];
  if (slot <= 0) {
    int ranges = 0;
    if (decode_default_ranges(d->q_len, d->num_heads, sms, &ranges) != cudaSuccess)
      return cuda_rc(cudaErrorUnknown);
    slot = ranges;
  }
  *R = slot;
  return MLA_DECODE_OK;
}

// Fixed-offset part of the layout (valid for every R).  The regions sized by
// the plan's R were checked against the workspace size when the plan was
// built; kernels locate them from the R recorded in the plan header.
int layout_for(const mla_decode_dims* d, size_t bytes, WsLayout* L) {
  *L = make_layout(d->batch, d->q_len, d->num_heads, 1);
  if (bytes < L->total) return MLA_DECODE_WORKSPACE_TOO_SMALL;
  return MLA_DECODE_OK;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}


}  // namespace

namespace mla {

bool softmax_scale_ok(float scale) { return std::isfinite(scale) && scale > 0.0f; }

int check_run_inputs(const mla_decode_dims* d, const void* q, const void* kv_cache,
                     const int32_t* block_table, const int32_t* seq_lens, const void* w_uk,
                     const void* w_uv, bool fp8, const float* uk_scale, const float* uv_scale,
                     float scale, const void* out, const float* lse) {
  int rc = check_dims(d);
  if (rc) return rc;
  auto aligned4 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; };
  if (!softmax_scale_ok(scale)) return MLA_DECODE_INVALID_ARG;
  if (!q || !kv_cache || !block_table || !seq_lens || !w_uk || !w_uv || !out || !lse ||
      !aligned16(q) || !aligned16(kv_cache) || !aligned16(w_uk) || !aligned16(w_uv) ||
      !aligned16(out) || !aligned4(block_table) || !aligned4(seq_lens) || !aligned4(lse))
    return MLA_DECODE_INVALID_ARG;
  if (fp8 && (!uk_scale || !uv_scale || !aligned4(uk_scale) || !aligned4(uv_scale)))
    return MLA_DECODE_INVALID_ARG;
  return MLA_DECODE_OK;
}

}  // namespace mla

extern "C" {

const char* mla_decode_status_string(int s) {
  switch (s) {
    case MLA_DECODE_OK: return "ok";
    case MLA_DECODE_INVALID_ARG: return "invalid argument (null or misaligned pointer, bad size)";
    case MLA_DECODE_UNSUPPORTED: return "unsupported configuration (dims or q_len)";
    case MLA_DECODE_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MLA_DECODE_CUDA_ERROR: return "CUDA error";
    case MLA_DECODE_DEVICE_BOUNDS: return "block_table entry or seq_len out of range";
    case MLA_DECODE_TIMEOUT: return "device-side wait timed out";
    default: return "unknown status";
  }
}


int mla_decode_selftest_wait_timeout(int32_t* status, void* stream) {
  if (!status || (reinterpret_cast<uintptr_t>(status) & 3u)) return MLA_DECODE_INVALID_ARG;
  wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status);
  return cuda_rc(cudaGetLastError());
}

int mla_decode_workspace_size_ex(const mla_decode_dims* d, int32_t num_ranges, size_t* bytes) {
  int rc = check_dims(d);
  if (rc) return rc;
  if (!bytes || num_ranges < 0 || num_ranges > 65536) return MLA_DECODE_INVALID_ARG;
  int R = num_ranges;
  if (R == 0) {
    rc = default_ranges(d, &R);
    if (rc) return rc;
  }
  *bytes = make_layout(d->batch, d->q_len, d->num_heads, R).total;
  return MLA_DECODE_OK;
}

int mla_decode_workspace_size(const mla_decode_dims* d, size_t* bytes) {
  return mla_decode_workspace_size_ex(d, 0, bytes);
}

}  // extern "C"

extern "C" {

int mla_decode_plan_ex(const mla_decode_dims* d, const int32_t* seq_lens, int32_t num_ranges,
                       void* ws, size_t ws_bytes, void* stream) {
  int rc = check_dims(d);
  if (rc) return rc;
  if (!seq_lens || !ws || !aligned16(ws) || num_ranges < 0 || num_ranges > 65536)
    return MLA_DECODE_INVALID_ARG;
  int R = num_ranges;
  if (R == 0) {
    rc = default_ranges(d, &R);
    if (rc) return rc;
  }
  const WsLayout L = make_layout(d->batch, d->q_len, d->num_heads, R);
  if (ws_bytes < L.total) return MLA_DECODE_WORKSPACE_TOO_SMALL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return cuda_rc(launch_plan(seq_lens, d->batch, d->q_len, d->max_pages_per_seq, R,
                             at<int32_t>(ws, L.status), at<PlanHeader>(ws, L.header),
                             at<int32_t>(ws, L.range_b), at<int32_t>(ws, L.range_p),
                             at<int32_t>(ws, L.seq_first), at<int32_t>(ws, L.seq_nsplit),
                             at<int32_t>(ws, L.seq_slot), at<int32_t>(ws, L.seq_len_eff),
                             at<int32_t>(ws, L.prefix), st));
}

int mla_decode_plan(const mla_decode_dims* d, const int32_t* seq_lens, void* ws, size_t ws_bytes,
                    void* stream) {
  return mla_decode_plan_ex(d, seq_lens, 0, ws, ws_bytes, stream);
}

// Steps a2 and a5 with bf16 weights (w_*) or FP8 weights (w8_* with block
// scales); exactly one of the two is given.
static int absorb_impl(const mla_decode_dims* d, const void* q, const void* w_uk,
                       const uint8_t* w8, const float* w8_scale, void* ws, size_t ws_bytes,
                       void* stream) {
  int rc = check_dims(d);
  if (rc) return rc;
  const void* w = w8 ? static_cast<const void*>(w8) : w_uk;
  if (!q || !w || !ws || !aligned16(q) || !aligned16(w) || !aligned16(ws) ||
      (w8 && (!w8_scale || (reinterpret_cast<uintptr_t>(w8_scale) & 3u))))
    return MLA_DECODE_INVALID_ARG;
  WsLayout L;
  rc = layout_for(d, ws_bytes, &L);
  if (rc) return rc;
  const int BT = d->batch * d->q_len, H = d->num_heads;
  CUtensorMap tm_q, tm_w;
  // 128 tokens or more: the untransposed absorb kernel,
  // which stores q_lat and q_lo by TMA as 2-D views [tokens, heads x row]
  // and reads 128-token boxes of q.
  const bool rows = BT >= 128;
  if (!make_map(&tm_q, q, BT, static_cast<uint64_t>(H) * kDq, static_cast<uint64_t>(H) * kDq,
                kBoxCols, rows ? 128 : bmm_token_tile(BT, true), false))
    return MLA_DECODE_CUDA_ERROR;
  // FP8 weights: 128-byte boxes of 128 m values x 64 k rows.
  if (!(w8 ? make_map(&tm_w, w8, static_cast<uint64_t>(H) * kNope, kLora, kLora, 128, 64, false, 1)
           : make_map(&tm_w, w_uk, static_cast<uint64_t>(H) * kNope, kLora, kLora, kBoxCols, 64,
                      false)))
    return MLA_DECODE_CUDA_ERROR;
  CUtensorMap tm_hi, tm_lo;
  if (rows && !(make_map(&tm_hi, at<void>(ws, L.qlat), BT, static_cast<uint64_t>(H) * kDqk,
                         static_cast<uint64_t>(H) * kDqk, kBoxCols, 128, false) &&
                make_map(&tm_lo, at<void>(ws, L.qlo), BT, static_cast<uint64_t>(H) * kLora,
                         static_cast<uint64_t>(H) * kLora, 128, 128, false, 1)))
    return MLA_DECODE_CUDA_ERROR;
  int sms = 0;
  rc = sm_count(&sms);
  if (rc) return rc;
  return cuda_rc(launch_absorb(tm_w, tm_q, rows ? &tm_hi : nullptr, rows ? &tm_lo : nullptr, BT,
                               H, static_cast<const __nv_bfloat16*>(q),
                               at<__nv_bfloat16>(ws, L.qlat), at<uint8_t>(ws, L.qlo),
                               at<int32_t>(ws, L.status), static_cast<cudaStream_t>(stream), w8,
                               w8_scale, sms));
}

static int up_project_impl(const mla_decode_dims* d, const void* w_uv, const uint8_t* w8,
                           const float* w8_scale, void* out, void* ws, size_t ws_bytes,
                           void* stream) {
  int rc = check_dims(d);
  if (rc) return rc;
  const void* w = w8 ? static_cast<const void*>(w8) : w_uv;
  if (!w || !out || !ws || !aligned16(w) || !aligned16(out) || !aligned16(ws) ||
      (w8 && (!w8_scale || (reinterpret_cast<uintptr_t>(w8_scale) & 3u))))
    return MLA_DECODE_INVALID_ARG;
  WsLayout L;
  rc = layout_for(d, ws_bytes, &L);
  if (rc) return rc;
  const int BT = d->batch * d->q_len, H = d->num_heads;
  CUtensorMap tm_o, tm_w;
  if (!make_map(&tm_o, at<void>(ws, L.olat), BT, static_cast<uint64_t>(H) * kLora,
                static_cast<uint64_t>(H) * kLora, kBoxCols, bmm_token_tile(BT, false), false))
    return MLA_DECODE_CUDA_ERROR;
  if (!(w8 ? make_map(&tm_w, w8, static_cast<uint64_t>(H) * kLora, kVHead, kVHead, 128, 64, false,
                      1)
           : make_map(&tm_w, w_uv, static_cast<uint64_t>(H) * kLora, kVHead, kVHead, kBoxCols, 64,
                      false)))
    return MLA_DECODE_CUDA_ERROR;
  int sms = 0;
  rc = sm_count(&sms);
  if (rc) return rc;
  const int nt = bmm_token_tile(BT, false);
  const bool one_wave = static_cast<int64_t>((BT + nt - 1) / nt) * H <= sms;
  return cuda_rc(launch_up_project(tm_w, tm_o, BT, H, static_cast<__nv_bfloat16*>(out),
                                   at<int32_t>(ws, L.status), static_cast<cudaStream_t>(stream),
                                   w8, w8_scale, one_wave));
}

// Whether a whole run takes the up-projection that also corrects the lse of
// unsplit sequences (then the combine merges split sequences only): 128
// tokens or more, in more (128-token tile, head) units than there are SMs.
// Measured: 512 tokens x 128 heads (512 units), step 319.3 -> 314.8 us; 128
// tokens x 128 heads (128 units on 152 SMs, one per SM), 235.4 -> 236.8 us,
// and still 227.6 -> 231.2 us once the split-only combine staged bf16
// partials.
static int run_uses_up_rows(const mla_decode_dims* d, bool* rows) {
  int sms = 0;
  const int rc = sm_count(&sms);
  if (rc) return rc;
  const int BT = d->batch * d->q_len;
  *rows = BT >= 128 && static_cast<int64_t>((BT + 127) / 128) * d->num_heads > sms;
  return MLA_DECODE_OK;
}

// The up-projection of such a run: untransposed, and it also adds the
// first-order LSE correction to the rows of unsplit sequences.  bf16 weights
// (w_uv) or FP8 weights (w8 with block scales).
static int up_project_rows_impl(const mla_decode_dims* d, const void* w_uv, const uint8_t* w8,
                                const float* w8_scale, float scale, void* out, float* lse,
                                void* ws, size_t ws_bytes, void* stream) {
  WsLayout L;
  int rc = layout_for(d, ws_bytes, &L);
  if (rc) return rc;
  const int BT = d->batch * d->q_len, H = d->num_heads;
  CUtensorMap tm_w, tm_o, tm_q, tm_out;
  if (!(w8 ? make_map(&tm_w, w8, static_cast<uint64_t>(H) * kLora, kVHead, kVHead, 128, 64,
                      false, 1)
           : make_map(&tm_w, w_uv, static_cast<uint64_t>(H) * kLora, kVHead, kVHead, kBoxCols,
                      64, false)) ||
      !make_map(&tm_o, at<void>(ws, L.olat), BT, static_cast<uint64_t>(H) * kLora,
                static_cast<uint64_t>(H) * kLora, kBoxCols, 128, false) ||
      !make_map(&tm_q, at<void>(ws, L.qlo), BT, static_cast<uint64_t>(H) * kLora,
                static_cast<uint64_t>(H) * kLora, 64, 128, false, 1, false) ||
      !make_map(&tm_out, out, BT, static_cast<uint64_t>(H) * kVHead,
                static_cast<uint64_t>(H) * kVHead, kBoxCols, 128, false))
    return MLA_DECODE_CUDA_ERROR;
  int sms = 0;
  rc = sm_count(&sms);
  if (rc) return rc;
  return cuda_rc(launch_up_project_rows(tm_w, tm_o, tm_q, tm_out, BT, d->q_len, H,
                                        at<int32_t>(ws, L.seq_nsplit), lse, scale,
                                        at<int32_t>(ws, L.status), w8 ? w8_scale : nullptr, sms,
                                        static_cast<cudaStream_t>(stream)));
}

int mla_decode_absorb(const mla_decode_dims* d, const void* q, const void* w_uk, void* ws,
                      size_t ws_bytes, void* stream) {
  if (!w_uk) return MLA_DECODE_INVALID_ARG;
  return absorb_impl(d, q, w_uk, nullptr, nullptr, ws, ws_bytes, stream);
}

int mla_decode_absorb_fp8w(const mla_decode_dims* d, const void* q, const uint8_t* w_uk_fp8,
                           const float* w_uk_scale, void* ws, size_t ws_bytes, void* stream) {
  if (!w_uk_fp8) return MLA_DECODE_INVALID_ARG;
  return absorb_impl(d, q, nullptr, w_uk_fp8, w_uk_scale, ws, ws_bytes, stream);
}

int mla_decode_attend(const mla_decode_dims* d, const void* kv_cache, const int32_t* block_table,
                      const int32_t* seq_lens, float scale, float* lse, void* ws, size_t ws_bytes,
                      void* stream) {
  int rc = check_dims(d);
  if (rc) return rc;
  if (!softmax_scale_ok(scale) || !kv_cache || !block_table || !seq_lens || !lse || !ws ||
      !aligned16(kv_cache) ||
      !aligned16(ws) || (reinterpret_cast<uintptr_t>(block_table) & 3u) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u))
    return MLA_DECODE_INVALID_ARG;
  WsLayout L;
  rc = layout_for(d, ws_bytes, &L);
  if (rc) return rc;
  const int TH = d->q_len * d->num_heads;
  const uint64_t rows = static_cast<uint64_t>(d->batch) * TH;
  CUtensorMap tm_q, tm_c;
  if (!make_map(&tm_q, at<void>(ws, L.qlat), rows, kDqk, kDqk, kBoxCols,
                decode_q_box_rows(d->q_len, d->num_heads), false) ||
      !make_map(&tm_c, kv_cache, static_cast<uint64_t>(d->num_pages) * kPage, kDqk, kDqk,
                kBoxCols, kPage, true))
    return MLA_DECODE_CUDA_ERROR;
  int sms = 0;
  rc = sm_count(&sms);
  if (rc) return rc;
  return cuda_rc(launch_decode(
      tm_q, tm_c, sms, block_table, at<int32_t>(ws, L.seq_len_eff), at<PlanHeader>(ws, L.header),
      ws, at<int32_t>(ws, L.seq_first), at<int32_t>(ws, L.seq_nsplit), at<int32_t>(ws, L.seq_slot),
      at<__nv_bfloat16>(ws, L.olat), lse,
      at<int32_t>(ws, L.status), d->batch, d->q_len, d->num_heads, d->max_pages_per_seq,
      d->num_pages, scale, static_cast<cudaStream_t>(stream)));
}

// The typical number of splits per sequence, which picks the merge variant of
// the combine: with fewer work ranges than sequences most rows are unsplit;
// otherwise a sequence is typically cut into about ranges / batch splits.
// (Only the speed depends on this guess: every variant computes the same.)
static int combine_variant(const mla_decode_dims* d, int* ranges, int* splits_per_seq) {
  const int rc = default_ranges(d, ranges);
  if (rc) return rc;
  *splits_per_seq = *ranges < d->batch ? 1 : (*ranges + d->batch - 1) / d->batch;
  return MLA_DECODE_OK;
}

// split_only: leave the rows of unsplit sequences alone (their LSE correction
// is then the up-projection's; see up_project_rows_impl).
static int combine_impl(const mla_decode_dims* d, float scale, float* lse, void* ws,
                        size_t ws_bytes, void* stream, bool split_only) {
  int rc = check_dims(d);
  if (rc) return rc;
  if (!softmax_scale_ok(scale) || !lse || !ws || !aligned16(ws) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u))
    return MLA_DECODE_INVALID_ARG;
  WsLayout L;
  rc = layout_for(d, ws_bytes, &L);
  if (rc) return rc;
  int ranges = 0, splits_per_seq = 0;
  rc = combine_variant(d, &ranges, &splits_per_seq);
  if (rc) return rc;
  return cuda_rc(launch_combine(at<int32_t>(ws, L.seq_nsplit), at<int32_t>(ws, L.seq_slot), ws,
                                at<PlanHeader>(ws, L.header), at<uint8_t>(ws, L.qlo),
                                at<__nv_bfloat16>(ws, L.olat), lse, d->batch, d->q_len,
                                d->num_heads, scale, splits_per_seq,
                                split_only ? (ranges > 1 ? ranges - 1 : 1) : 0,
                                at<int32_t>(ws, L.status), static_cast<cudaStream_t>(stream)));
}

// Whether a whole run merges the splits inside the up-projection
// (combine_up_kernel): fewer than 128 tokens, in 16-token tiles of every head
// that fit in one wave on the SMs.
static int run_uses_combine_up(const mla_decode_dims* d, bool* fused) {
  int sms = 0;
  const int rc = sm_count(&sms);
  if (rc) return rc;
  const int BT = d->batch * d->q_len, nt = combine_up_tile();
  *fused = BT < 128 && static_cast<int64_t>((BT + nt - 1) / nt) * d->num_heads <= sms;
  return MLA_DECODE_OK;
}

// Combine and up-projection of such a run in one launch, with bf16 weights
// (w_uv) or FP8 weights (w8 with block scales); out and lse equal those of the
// combine step followed by the up-projection step bit for bit.
static int combine_up_impl(const mla_decode_dims* d, const void* w_uv, const uint8_t* w8,
                           const float* w8_scale, float scale, void* out, float* lse, void* ws,
                           size_t ws_bytes, void* stream) {
  WsLayout L;
  int rc = layout_for(d, ws_bytes, &L);
  if (rc) return rc;
  int ranges = 0, splits_per_seq = 0;
  rc = combine_variant(d, &ranges, &splits_per_seq);
  if (rc) return rc;
  CUtensorMap tm_w;
  const uint64_t wrows = static_cast<uint64_t>(d->num_heads) * kLora;
  if (!(w8 ? make_map(&tm_w, w8, wrows, kVHead, kVHead, 128, 64, false, 1)
           : make_map(&tm_w, w_uv, wrows, kVHead, kVHead, kBoxCols, 64, false)))
    return MLA_DECODE_CUDA_ERROR;
  return cuda_rc(launch_combine_up(
      tm_w, d->batch, d->q_len, d->num_heads, ws, at<PlanHeader>(ws, L.header),
      at<int32_t>(ws, L.seq_nsplit), at<int32_t>(ws, L.seq_slot), at<uint8_t>(ws, L.qlo),
      at<__nv_bfloat16>(ws, L.olat), lse, scale, static_cast<__nv_bfloat16*>(out),
      at<int32_t>(ws, L.status), splits_per_seq, w8 ? w8_scale : nullptr,
      static_cast<cudaStream_t>(stream)));
}

int mla_decode_combine(const mla_decode_dims* d, float scale, float* lse, void* ws,
                       size_t ws_bytes, void* stream) {
  return combine_impl(d, scale, lse, ws, ws_bytes, stream, false);
}

int mla_decode_up_project(const mla_decode_dims* d, const void* w_uv, void* out, void* ws,
                          size_t ws_bytes, void* stream) {
  if (!w_uv) return MLA_DECODE_INVALID_ARG;
  return up_project_impl(d, w_uv, nullptr, nullptr, out, ws, ws_bytes, stream);
}

int mla_decode_up_project_fp8w(const mla_decode_dims* d, const uint8_t* w_uv_fp8,
                               const float* w_uv_scale, void* out, void* ws, size_t ws_bytes,
                               void* stream) {
  if (!w_uv_fp8) return MLA_DECODE_INVALID_ARG;
  return up_project_impl(d, nullptr, w_uv_fp8, w_uv_scale, out, ws, ws_bytes, stream);
}

// Every argument of a whole run, checked before its first launch so that a
// host-detected error leaves nothing enqueued.
static int check_run(const mla_decode_dims* d, const void* q, const void* kv_cache,
                     const int32_t* block_table, const int32_t* seq_lens, const void* w_uk,
                     const void* w_uv, bool fp8, const float* uk_scale, const float* uv_scale,
                     float scale, const void* out, const float* lse, const void* ws,
                     size_t ws_bytes) {
  int rc = check_run_inputs(d, q, kv_cache, block_table, seq_lens, w_uk, w_uv, fp8, uk_scale,
                            uv_scale, scale, out, lse);
  if (rc) return rc;
  if (!ws || !aligned16(ws)) return MLA_DECODE_INVALID_ARG;
  WsLayout L;
  return layout_for(d, ws_bytes, &L);
}

int mla_decode_run(const mla_decode_dims* d, const void* q, const void* kv_cache,
                   const int32_t* block_table, const int32_t* seq_lens, const void* w_uk,
                   const void* w_uv, float scale, void* out, float* lse, void* ws, size_t ws_bytes,
                   void* stream) {
  int rc = check_run(d, q, kv_cache, block_table, seq_lens, w_uk, w_uv, false, nullptr, nullptr,
                     scale, out, lse, ws, ws_bytes);
  if (rc) return rc;
  rc = mla_decode_absorb(d, q, w_uk, ws, ws_bytes, stream);
  if (rc) return rc;
  rc = mla_decode_attend(d, kv_cache, block_table, seq_lens, scale, lse, ws, ws_bytes, stream);
  if (rc) return rc;
  // Small batches: the combine's merges build the up-projection's operand in
  // shared memory (one launch, no o_lat round trip).
  bool fused = false;
  rc = run_uses_combine_up(d, &fused);
  if (rc) return rc;
  if (fused)
    return combine_up_impl(d, w_uv, nullptr, nullptr, scale, out, lse, ws, ws_bytes, stream);
  // Large batches: the combine merges split sequences only and the
  // up-projection corrects the lse of the others from the o_lat and q_lo
  // tiles it stages anyway (one read of each instead of two).
  bool rows = false;
  rc = run_uses_up_rows(d, &rows);
  if (rc) return rc;
  rc = combine_impl(d, scale, lse, ws, ws_bytes, stream, rows);
  if (rc) return rc;
  if (rows)
    return up_project_rows_impl(d, w_uv, nullptr, nullptr, scale, out, lse, ws, ws_bytes,
                                stream);
  return mla_decode_up_project(d, w_uv, out, ws, ws_bytes, stream);
}

int mla_decode_run_fp8w(const mla_decode_dims* d, const void* q, const void* kv_cache,
                        const int32_t* block_table, const int32_t* seq_lens,
                        const uint8_t* w_uk_fp8, const float* w_uk_scale,
                        const uint8_t* w_uv_fp8, const float* w_uv_scale, float scale, void* out,
                        float* lse, void* ws, size_t ws_bytes, void* stream) {
  int rc = check_run(d, q, kv_cache, block_table, seq_lens, w_uk_fp8, w_uv_fp8, true, w_uk_scale,
                     w_uv_scale, scale, out, lse, ws, ws_bytes);
  if (rc) return rc;
  rc = mla_decode_absorb_fp8w(d, q, w_uk_fp8, w_uk_scale, ws, ws_bytes, stream);
  if (rc) return rc;
  rc = mla_decode_attend(d, kv_cache, block_table, seq_lens, scale, lse, ws, ws_bytes, stream);
  if (rc) return rc;
  bool fused = false;  // as in mla_decode_run
  rc = run_uses_combine_up(d, &fused);
  if (rc) return rc;
  if (fused)
    return combine_up_impl(d, nullptr, w_uv_fp8, w_uv_scale, scale, out, lse, ws, ws_bytes,
                           stream);
  bool rows = false;
  rc = run_uses_up_rows(d, &rows);
  if (rc) return rc;
  rc = combine_impl(d, scale, lse, ws, ws_bytes, stream, rows);
  if (rc) return rc;
  if (rows)
    return up_project_rows_impl(d, nullptr, w_uv_fp8, w_uv_scale, scale, out, lse, ws, ws_bytes,
                                stream);
  return mla_decode_up_project_fp8w(d, w_uv_fp8, w_uv_scale, out, ws, ws_bytes, stream);
}

int mla_decode_kernels_per_run(const mla_decode_dims* d, int32_t fp8_weights,
                               int32_t* kernels) {
  int rc = check_dims(d);
  if (rc) return rc;
  if (!kernels) return MLA_DECODE_INVALID_ARG;
  (void)fp8_weights;  // both weight formats take the same arrangement
  bool fused = false;
  rc = run_uses_combine_up(d, &fused);
  if (rc) return rc;
  *kernels = fused ? 3 : 4;
  return MLA_DECODE_OK;
}

int mla_decode_workspace_offsets(const mla_decode_dims* d, int32_t num_ranges,
                                 int64_t* offsets, int32_t n) {
  int rc = check_dims(d);
  if (rc) return rc;
  if (!offsets || n < 4 || num_ranges < 0 || num_ranges > 65536) return MLA_DECODE_INVALID_ARG;
  int R = num_ranges;
  if (R == 0) {
    rc = default_ranges(d, &R);
    if (rc) return rc;
  }
  const WsLayout L = make_layout(d->batch, d->q_len, d->num_heads, R);
  offsets[0] = static_cast<int64_t>(L.qlat);
  offsets[1] = static_cast<int64_t>(L.qlo);
  offsets[2] = static_cast<int64_t>(L.olat);
  offsets[3] = static_cast<int64_t>(L.header);
  return MLA_DECODE_OK;
}

int mla_decode_check(const void* ws, void* stream) {
  if (!ws) return MLA_DECODE_INVALID_ARG;
  int32_t host = 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The status word sits at offset 0 of every layout.
  if (cudaMemcpyAsync(&host, ws, sizeof(int32_t), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return cuda_rc(cudaErrorUnknown);
  if (cudaStreamSynchronize(st) != cudaSuccess) return cuda_rc(cudaErrorUnknown);
  return host;
}

}  // extern "C"
