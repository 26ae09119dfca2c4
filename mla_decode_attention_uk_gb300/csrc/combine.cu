// combine.cu -- step a4: merge split-KV partial results by log-sum-exp and
// apply the first-order LSE correction (the row merge itself is in
// merge.cuh, shared with the fused combine + up-projection of small batches).
//
// One warp per query row; each lane owns 16 of the 512 latent columns and
// moves them with 16-byte vector loads.  Three instantiations, picked by the
// host from the typical split count:
//   - rows of at most two splits load all of them at once, more go through a
//     split loop that is not unrolled, when most rows are unsplit (64
//     registers, four CTAs per SM);
//   - rows of at most four splits at once, the loop unrolled by 4, when
//     sequences are cut into a few splits;
//   - the loop unrolled by 4 only, when sequences are cut into many splits.
// The merged o is stored as bf16 o_lat for the W_UV bmm.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "merge.cuh"
#include "ptx.cuh"

namespace mla {

namespace {

constexpr int kCombThreads = 256;

constexpr int kRowsPerCta = kCombThreads / 32;

// At least three CTAs per SM: the unrolled instantiations then get up to 85
// registers and do not spill (left to itself ptxas picks 64 and spills).
template <int kUnroll, int kFewN>
__global__ void __launch_bounds__(kCombThreads, 3)
combine_kernel(const int32_t* __restrict__ seq_nsplit, const int32_t* __restrict__ seq_slot,
               const uint8_t* __restrict__ ws, const PlanHeader* __restrict__ header, int B,
               int T, int H, const uint8_t* __restrict__ qlo,
               __nv_bfloat16* __restrict__ olat, float* __restrict__ lse_out, float scale) {
  // The plan and q_lo are complete when this kernel starts (the attention
  // step waited for them before letting it launch), so they are read before
  // waiting for the attention step itself.
  griddep_launch_dependents();
  const int TH = T * H;
  const int b = blockIdx.y;
  const int r = blockIdx.x * kRowsPerCta + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= TH) {
    griddep_wait();
    return;
  }
  const int ns = seq_nsplit[b];
  const size_t row = static_cast<size_t>(b) * TH + r;
  if (ns <= 1) {
    correct_unsplit_row(row, lane, qlo, olat, lse_out, scale, [](const uint4&, const uint4&) {});
    return;
  }
  const size_t row_o = static_cast<size_t>(b) * TH + r;
  merge_split_row<kUnroll, kFewN>(b, r, lane, ns, seq_slot[b], B, T, H, ws, header, qlo, lse_out,
                                  scale, [&](int col, const uint2& packed) {
                                    *reinterpret_cast<uint2*>(olat + row_o * kLora + col) = packed;
                                  });
}

// Split sequences only, for a run whose up-projection corrects the lse of the
// unsplit rows itself.  Sequence b is split exactly when a work range starts
// inside it, and the first such range is k = seq_first[b] + 1, so walking the
// ranges visits every split sequence once; the grid's y dimension strides
// over them.  (A kernel of its own: the loop around the merge would cost the
// other instantiations registers; its grid is small, so it may use as many
// as it needs.)
template <int kUnroll, int kFewN>
__global__ void __launch_bounds__(kCombThreads, 1)
combine_split_kernel(const int32_t* __restrict__ seq_nsplit,
                     const int32_t* __restrict__ seq_slot, const uint8_t* __restrict__ ws,
                     const PlanHeader* __restrict__ header, int B, int T, int H,
                     const uint8_t* __restrict__ qlo, __nv_bfloat16* __restrict__ olat,
                     float* __restrict__ lse_out, float scale) {
  // The plan is complete when this kernel starts (as in combine_kernel).
  griddep_launch_dependents();
  const int TH = T * H;
  const int r = blockIdx.x * kRowsPerCta + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r < TH) {
    const WsLayout L = make_layout(B, T, H, header->num_ranges);
    const int32_t* __restrict__ range_b = reinterpret_cast<const int32_t*>(ws + L.range_b);
    const int32_t* __restrict__ range_p = reinterpret_cast<const int32_t*>(ws + L.range_p);
    const int32_t* __restrict__ seq_first = reinterpret_cast<const int32_t*>(ws + L.seq_first);
    for (int k = blockIdx.y + 1; k < L.num_ranges; k += gridDim.y) {
      const int b = range_b[k];
      if (b >= B || range_p[k] == 0 || seq_first[b] + 1 != k) continue;
      const size_t row_o = static_cast<size_t>(b) * TH + r;
      merge_split_row<kUnroll, kFewN>(
          b, r, lane, seq_nsplit[b], seq_slot[b], B, T, H, ws, header, qlo, lse_out, scale,
          [&](int col, const uint2& packed) {
            *reinterpret_cast<uint2*>(olat + row_o * kLora + col) = packed;
          });
    }
  }
  griddep_wait();
}

}  // namespace

cudaError_t launch_combine(const int32_t* seq_nsplit, const int32_t* seq_slot, const void* ws,
                           const PlanHeader* header, const uint8_t* qlo,
                           __nv_bfloat16* olat, float* lse, int B, int T, int H, float scale,
                           int splits_per_seq, int split_ranges, cudaStream_t st) {
  // split_ranges > 0: split sequences only, the grid's y dimension striding
  // over that many work ranges (the planner's count or any other).
  const bool split_only = split_ranges > 0;
  dim3 grid((T * H + kRowsPerCta - 1) / kRowsPerCta, split_only ? split_ranges : B);
  // splits_per_seq: work ranges per sequence, rounded up (the host's guess of
  // the typical split count; only the speed depends on it).  A split-only
  // launch takes the same variant as the full combine would, so a split
  // row's o_lat is the same bit for bit either way.
  auto kern = splits_per_seq <= 1
                  ? (split_only ? combine_split_kernel<1, 2> : combine_kernel<1, 2>)
              : splits_per_seq <= 4
                  ? (split_only ? combine_split_kernel<4, 4> : combine_kernel<4, 4>)
                  : (split_only ? combine_split_kernel<4, 0> : combine_kernel<4, 0>);
  cudaError_t e = launch_pdl(kern, grid, dim3(kCombThreads), 0, st, seq_nsplit, seq_slot,
                             static_cast<const uint8_t*>(ws), header, B, T, H, qlo, olat, lse,
                             scale);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace mla
