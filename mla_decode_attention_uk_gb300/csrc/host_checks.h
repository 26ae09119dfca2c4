// host_checks.h -- argument checks shared by the C ABI's entry points
// (host code only).
#pragma once
#include <cstddef>
#include <cstdint>

#include "../../include/mla_decode.h"

namespace mla {

// The softmax scale multiplies q_lat . c_j; the attention kernel takes the
// running maximum over unscaled scores, which is the maximum of the scaled
// ones only for a positive scale.  Finite and > 0, else INVALID_ARG.
bool softmax_scale_ok(float scale);

// Every caller-supplied argument of a whole decode run except the workspace:
// dims, the scale, and each pointer (non-null; 16-byte alignment for q, the
// cache, the weights and out; 4-byte for block_table, seq_lens, lse and the FP8
// block scales).  With fp8, w_uk / w_uv are the E4M3 codes and both scale
// arrays are required.  Returns an mla_decode_status; needs no device.
int check_run_inputs(const mla_decode_dims* d, const void* q, const void* kv_cache,
                     const int32_t* block_table, const int32_t* seq_lens, const void* w_uk,
                     const void* w_uv, bool fp8, const float* uk_scale, const float* uv_scale,
                     float softmax_scale, const void* out, const float* lse);

}  // namespace mla
