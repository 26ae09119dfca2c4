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

// Bulk copy (no tensor map) of `bytes` from global to shared memory,
// completing on an mbarrier; both addresses and the size are multiples of 16
// bytes.
__device__ __forceinline__ void bulk_load_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

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
// over them and its x dimension over blocks of rows_blk rows.  A CTA that
// finds a split sequence brings the partial rows of its row block into
// shared memory with one bulk copy per split (the rows of one split are
// contiguous: rows_blk x 1 KB), so all of a block's partials are in flight at once
// instead of the few that one warp per row keeps in registers (measured:
// that form cost 11.7 us of a 512-token x 128-head step, latency-bound at
// one or two CTAs per SM).  Sequences with more splits than are staged read
// their partials from global memory; the merge arithmetic is the same either
// way.  (A kernel of its own: the loop around the merge would cost the other
// instantiations registers; its grid is small, so it may use what it
// needs: two CTAs per SM, one for the variant that keeps four splits'
// partials in registers.)


template <int kUnroll, int kFewN>
__global__ void __launch_bounds__(kCombThreads, kFewN == 4 ? 1 : 2)
combine_split_kernel(const int32_t* __restrict__ seq_nsplit,
                     const int32_t* __restrict__ seq_slot, const uint8_t* __restrict__ ws,
                     const PlanHeader* __restrict__ header, int B, int T, int H,
                     const uint8_t* __restrict__ qlo, __nv_bfloat16* __restrict__ olat,
                     float* __restrict__ lse_out, float scale, int stage_splits,
                     int rows_blk, int32_t* __restrict__ status) {
  extern __shared__ __align__(128) uint8_t stage_raw[];
  __shared__ __align__(8) uint64_t full_bar;
  __shared__ int abort_sh;
  // The plan is complete when this kernel starts (as in combine_kernel).
  griddep_launch_dependents();
  const int TH = T * H;
  const int r0 = blockIdx.x * rows_blk;
  const int nrows = min(rows_blk, TH - r0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&full_bar), 1);
    abort_sh = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const uint2* const stage = reinterpret_cast<const uint2*>(stage_raw);
  const WsLayout L = make_layout(B, T, H, header->num_ranges);
  const int32_t* __restrict__ range_b = reinterpret_cast<const int32_t*>(ws + L.range_b);
  const int32_t* __restrict__ range_p = reinterpret_cast<const int32_t*>(ws + L.range_p);
  const int32_t* __restrict__ seq_first = reinterpret_cast<const int32_t*>(ws + L.seq_first);
  uint32_t phase = 0;
  int issued = 0;  // bulk-copy rounds started by thread 0
  for (int k = blockIdx.y + 1; k < L.num_ranges && nrows > 0; k += gridDim.y) {
    if (abort_sh) break;  // a staging wait timed out (read after a barrier: uniform)
    const int b = range_b[k];
    if (b >= B || range_p[k] == 0 || seq_first[b] + 1 != k) continue;  // the same for the CTA
    const int ns = seq_nsplit[b], slot0 = seq_slot[b];
    const bool staged = ns <= stage_splits;
    bool ok = true;
    if (staged) {
      if (threadIdx.x == 0) {
        griddep_wait();  // the partials come from the attention step
        fence_proxy_async_smem();  // earlier reads of the staging area come first
        const __nv_bfloat16* opart = reinterpret_cast<const __nv_bfloat16*>(ws + L.opart);
        const uint32_t bytes = static_cast<uint32_t>(nrows) * kLora * 2;
        mbar_expect_tx(smem_u32(&full_bar), bytes * ns);
        for (int s = 0; s < ns; ++s)
          bulk_load_g2s(smem_u32(stage_raw) + s * rows_blk * kLora * 2,
                        opart + (static_cast<size_t>(slot0 + s) * TH + r0) * kLora, bytes,
                        smem_u32(&full_bar));
        ++issued;
      }
      ok = mbar_wait(smem_u32(&full_bar), phase, &abort_sh, status);
      phase ^= 1;
    }
    if (ok) {
      for (int rr = warp; rr < nrows; rr += kCombThreads / 32) {
        const int r = r0 + rr;
        const size_t row_o = static_cast<size_t>(b) * TH + r;
        auto sink = [&](int col, const uint2& packed) {
          *reinterpret_cast<uint2*>(olat + row_o * kLora + col) = packed;
        };
        if (staged) {
          merge_split_row<kUnroll, kFewN>(
              b, r, lane, ns, slot0, B, T, H, ws, header, qlo, lse_out, scale, sink,
              [&](const __nv_bfloat16*, int, int s, int, int) {
                return stage + (s * rows_blk + rr) * (kLora / 4);
              });
        } else {
          merge_split_row<kUnroll, kFewN>(b, r, lane, ns, slot0, B, T, H, ws, header, qlo,
                                          lse_out, scale, sink);
        }
      }
    }
    __syncthreads();  // the staging area is reused for the next sequence
  }
  // After a timeout, let a bulk copy still in flight land before exiting.
  if (threadIdx.x == 0 && abort_sh && issued > 0)
    mbar_wait_drain(smem_u32(&full_bar), (issued - 1) & 1, status);
  griddep_wait();
}

}  // namespace

cudaError_t launch_combine(const int32_t* seq_nsplit, const int32_t* seq_slot, const void* ws,
                           const PlanHeader* header, const uint8_t* qlo,
                           __nv_bfloat16* olat, float* lse, int B, int T, int H, float scale,
                           int splits_per_seq, int split_ranges, int32_t* status,
                           cudaStream_t st) {
  // splits_per_seq: work ranges per sequence, rounded up (the host's guess of
  // the typical split count; only the speed depends on it).  A split-only
  // launch takes the same merge variant as the full combine would, so a
  // split row's o_lat is the same bit for bit either way.
  cudaError_t e;
  if (split_ranges > 0) {
    // Split sequences only, the grid's y dimension striding over that many
    // work ranges (the planner's count or any other); partials of up to
    // stage_splits splits are staged in shared memory.
    // Blocks of 16 rows, or 32 when 16-row blocks over every range would
    // take more than two waves of CTAs (608 = two waves of two CTAs on each of
    // 152 SMs, the count this was tuned on; elsewhere only the speed
    // changes).  Measured: 1024 query rows x 18 ranges, step 487.0 -> 484.2
    // us with 32-row blocks; 256 x 37 (592 CTAs) lost 2.9 us with them.
    const int rows_blk = (T * H + 15) / 16 * split_ranges > 608 ? 32 : 16;
    const int stage_splits =
        (splits_per_seq <= 1 ? 2 : (splits_per_seq <= 4 ? 4 : 6)) * (32 / rows_blk);
    const int smem = stage_splits * rows_blk * kLora * 2;
    auto kern = splits_per_seq <= 1   ? combine_split_kernel<1, 2>
                : splits_per_seq <= 4 ? combine_split_kernel<4, 4>
                                      : combine_split_kernel<4, 0>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    dim3 grid((T * H + rows_blk - 1) / rows_blk, split_ranges);
    e = launch_pdl(kern, grid, dim3(kCombThreads), smem, st, seq_nsplit, seq_slot,
                   static_cast<const uint8_t*>(ws), header, B, T, H, qlo, olat, lse, scale,
                   stage_splits, rows_blk, status);
  } else {
    auto kern = splits_per_seq <= 1   ? combine_kernel<1, 2>
                : splits_per_seq <= 4 ? combine_kernel<4, 4>
                                      : combine_kernel<4, 0>;
    dim3 grid((T * H + kRowsPerCta - 1) / kRowsPerCta, B);
    e = launch_pdl(kern, grid, dim3(kCombThreads), 0, st, seq_nsplit, seq_slot,
                   static_cast<const uint8_t*>(ws), header, B, T, H, qlo, olat, lse, scale);
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace mla
