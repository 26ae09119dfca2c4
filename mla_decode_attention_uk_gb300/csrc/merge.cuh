// merge.cuh -- the row merge of step a4, shared by the combine kernel and the
// fused combine + up-projection for small batches, so both compute the same
// bits.
//
// A sequence cut into n key ranges has, per query row, n latent outputs o_s
// (each normalised over its own range) and their log-sum-exps lse_s.  Softmax
// over the union of the ranges is the lse-weighted mixture:
//   lse = ln sum_s exp(lse_s),   o = sum_s exp(lse_s - lse) o_s,
// the split-KV decomposition of the FlashAttention family that FlashMLA
// credits ("DeepSeek publica FlashMLA como codigo abierto").  Every row's lse
// (split or not) then gets the first-order correction scale * (q_lo . o): the
// attention step scored keys with the bf16 part of the absorbed query,
// q_lat = hi + q_lo, and d lse / d q_lat = scale * o.  q_lo arrives as E4M3 of
// q_lo * 2^10.  One warp per row.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "ptx.cuh"

namespace mla {

// Two E4M3 values (the low 16 bits of `bits`, first value in the low byte) of
// the scaled residual q_lo * 2^10, widened exactly to fp32.
__device__ __forceinline__ float2 qlo_pair(uint32_t bits) {
  const __nv_fp8x2_storage_t pr = static_cast<__nv_fp8x2_storage_t>(bits & 0xFFFFu);
  return __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(pr, __NV_E4M3)));
}
// The partial output row of split s (512 bf16), read where the attention
// step wrote it (the default source of merge_split_row).  uint2 = four bf16.
struct GlobalPartRows {
  __device__ const uint2* operator()(const __nv_bfloat16* opart, int slot0, int s, int TH,
                                     int r) const {
    return reinterpret_cast<const uint2*>(opart +
                                          (static_cast<size_t>(slot0 + s) * TH + r) * kLora);
  }
};
// Four bf16 (low half first) widened exactly to fp32.
__device__ __forceinline__ float4 bf16x4_to_float4(uint2 u) {
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

// One warp merges row r of split sequence b (ns splits, partial slots from
// slot0): lse and o over the splits, o as bf16 (sink(col, four bf16 of
// columns col .. col + 3), for col = (32 q + lane) * 4), and the lse with its
// first-order correction.  Rows of at most kFewN splits load every split's
// lse and partial output at once; others go through a split loop unrolled
// kUnroll times.  part_rows(opart, slot0, s, TH, r) gives split s's partial
// row (512 bf16 as 128 uint2): global memory, or a copy staged in shared
// memory; the arithmetic is the same either way.
template <int kUnroll, int kFewN, class Sink, class PartRows = GlobalPartRows>
__device__ __forceinline__ void merge_split_row(int b, int r, int lane, int ns, int slot0, int B,
                                                int T, int H, const uint8_t* __restrict__ ws,
                                                const PlanHeader* __restrict__ header,
                                                const uint8_t* __restrict__ qlo,
                                                float* __restrict__ lse_out, float scale,
                                                Sink&& sink, PartRows part_rows = PartRows()) {
  const int TH = T * H;
  const size_t row = static_cast<size_t>(b) * TH + r;
  uint32_t lo_raw[4];  // 4 E4M3 residuals per (q, lane): columns (32 q + lane) * 4 ..
#pragma unroll
  for (int q = 0; q < 4; ++q)
    lo_raw[q] = *reinterpret_cast<const uint32_t*>(qlo + row * kLora + (q * 32 + lane) * 4);
  griddep_wait();
  const WsLayout L = make_layout(B, T, H, header->num_ranges);
  const __nv_bfloat16* __restrict__ opart = reinterpret_cast<const __nv_bfloat16*>(ws + L.opart);
  const float* __restrict__ lpart = reinterpret_cast<const float*>(ws + L.lpart);

  float4 acc[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
  float lse;
  if (kFewN > 0 && ns <= kFewN) {
    // Every split's lse and partial output go out at once (one memory round
    // trip instead of one per split).
    constexpr int kN = kFewN > 0 ? kFewN : 1;
    float l[kN];
    float4 v[kN][4];
#pragma unroll
    for (int s = 0; s < kN; ++s) {
      l[s] = -INFINITY;
      if (s < ns) {
        const size_t srow = static_cast<size_t>(slot0 + s) * TH + r;
        l[s] = lpart[srow];
        const uint2* src = part_rows(opart, slot0, s, TH, r);
#pragma unroll
        for (int q = 0; q < 4; ++q) v[s][q] = bf16x4_to_float4(src[q * 32 + lane]);
      }
    }
    float m = l[0];
#pragma unroll
    for (int s = 1; s < kN; ++s) m = fmaxf(m, l[s]);
    float wsum = 0.0f;
#pragma unroll
    for (int s = 0; s < kN; ++s) wsum += (l[s] == -INFINITY) ? 0.0f : __expf(l[s] - m);
    lse = m + __logf(wsum);
#pragma unroll
    for (int s = 0; s < kN; ++s) {
      if (s < ns) {
        const float w = (l[s] == -INFINITY) ? 0.0f : __expf(l[s] - lse);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          acc[q].x += w * v[s][q].x;
          acc[q].y += w * v[s][q].y;
          acc[q].z += w * v[s][q].z;
          acc[q].w += w * v[s][q].w;
        }
      }
    }
  } else {
    // Lane s holds the lse of split s (32 splits per pass), so the loads go
    // out together and the max and sum are warp reductions.
    float m = -INFINITY;
    for (int s0 = 0; s0 < ns; s0 += 32) {
      const float l = s0 + lane < ns ? lpart[static_cast<size_t>(slot0 + s0 + lane) * TH + r]
                                     : -INFINITY;
      m = fmaxf(m, l);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float wsum = 0.0f;
    for (int s0 = 0; s0 < ns; s0 += 32) {
      const float l = s0 + lane < ns ? lpart[static_cast<size_t>(slot0 + s0 + lane) * TH + r]
                                     : -INFINITY;
      wsum += (l == -INFINITY) ? 0.0f : __expf(l - m);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
    lse = m + __logf(wsum);
    for (int s0 = 0; s0 < ns; s0 += 32) {
      const float l = s0 + lane < ns ? lpart[static_cast<size_t>(slot0 + s0 + lane) * TH + r]
                                     : -INFINITY;
      const float wl = (l == -INFINITY) ? 0.0f : __expf(l - lse);  // weight of split s0 + lane
      const int n = min(32, ns - s0);
#pragma unroll kUnroll
      for (int i = 0; i < n; ++i) {
        const float w = __shfl_sync(0xffffffffu, wl, i);
        const uint2* src = part_rows(opart, slot0, s0 + i, TH, r);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 v = bf16x4_to_float4(src[q * 32 + lane]);
          acc[q].x += w * v.x;
          acc[q].y += w * v.y;
          acc[q].z += w * v.z;
          acc[q].w += w * v.w;
        }
      }
    }
  }

  float corr = 0.0f;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int col = (q * 32 + lane) * 4;
    const float2 l01 = qlo_pair(lo_raw[q]);
    const float2 l23 = qlo_pair(lo_raw[q] >> 16);
    corr += l01.x * acc[q].x + l01.y * acc[q].y + l23.x * acc[q].z + l23.y * acc[q].w;
    __nv_bfloat162 o01 = __floats2bfloat162_rn(acc[q].x, acc[q].y);
    __nv_bfloat162 o23 = __floats2bfloat162_rn(acc[q].z, acc[q].w);
    uint2 packed;
    packed.x = *reinterpret_cast<uint32_t*>(&o01);
    packed.y = *reinterpret_cast<uint32_t*>(&o23);
    sink(col, packed);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) corr += __shfl_xor_sync(0xffffffffu, corr, o);
  if (lane == 0) lse_out[row] = lse + scale * kQloInvScale * corr;
}

// One warp corrects row `row` of an unsplit sequence: o_lat and lse were
// written by the attention step; lse += scale * (q_lo . o).  Lane l owns
// latent columns 16 l .. 16 l + 15 (sink(o0, o1): those columns' bf16 o, in
// two 16-byte halves).
template <class Sink>
__device__ __forceinline__ void correct_unsplit_row(size_t row, int lane,
                                                    const uint8_t* __restrict__ qlo,
                                                    const __nv_bfloat16* __restrict__ olat,
                                                    float* __restrict__ lse_out, float scale,
                                                    Sink&& sink) {
  const uint4* o4 = reinterpret_cast<const uint4*>(olat + row * kLora) + lane * 2;
  // This lane's 16 latent columns of q_lo: 16 E4M3 bytes.
  const uint4 lv = *(reinterpret_cast<const uint4*>(qlo + row * kLora) + lane);
  griddep_wait();
  // The row's lse goes out with the o_lat loads: one round trip, not two.
  const float lse_in = lane == 0 ? lse_out[row] : 0.0f;
  float corr = 0.0f;
  const uint32_t lw[4] = {lv.x, lv.y, lv.z, lv.w};
  uint4 ov[2];
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    ov[q] = o4[q];
    const uint32_t ow[4] = {ov[q].x, ov[q].y, ov[q].z, ov[q].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __nv_bfloat162 o2 = *reinterpret_cast<const __nv_bfloat162*>(&ow[e]);
      const float2 l2 = qlo_pair(lw[2 * q + (e >> 1)] >> (16 * (e & 1)));
      corr += l2.x * __low2float(o2) + l2.y * __high2float(o2);
    }
  }
  sink(ov[0], ov[1]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) corr += __shfl_xor_sync(0xffffffffu, corr, o);
  if (lane == 0) lse_out[row] = lse_in + scale * kQloInvScale * corr;
}

}  // namespace mla
