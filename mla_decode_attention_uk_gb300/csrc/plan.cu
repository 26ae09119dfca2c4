// plan.cu -- step a1: split-KV planner for variable-length decode batches.
//
// FlashMLA is described as optimised for serving variable-length sequences
// ("DeepSeek publica FlashMLA como codigo abierto", feature list).  This
// planner realises that with an equal-cost partition: every sequence b costs
// pages_b + kPieceCost units (pages to stream plus a fixed per-piece charge
// for loading the query tile and writing results), the costs are laid end to
// end, and the line is cut into num_ranges equal pieces.  Decode CTA group k
// streams range k; a sequence cut by a range boundary is split, and its pieces
// are merged by the LSE combine.  Runs as one CTA on the device so the plan
// needs no host synchronisation.
#include <cuda_runtime.h>

#include "common.cuh"
#include "ptx.cuh"

namespace mla {

namespace {

constexpr int kPlanThreads = 1024;
// Batches up to this size keep the cost prefix and page counts in shared
// memory, so the per-range binary searches do not chain global loads.
constexpr int kPlanSmemB = 4096;

// Inclusive block-wide scan of one int per thread (1024 threads).
__device__ int block_inclusive_scan(int v, int* warp_tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) warp_tot[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int w = warp_tot[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int n = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += n;
    }
    warp_tot[lane] = w;
  }
  __syncthreads();
  if (warp > 0) v += warp_tot[warp - 1];
  __syncthreads();
  return v;
}

__global__ void __launch_bounds__(kPlanThreads)
plan_kernel(const int32_t* __restrict__ seq_lens, int B, int T, int max_pages, int R,
            int32_t* __restrict__ status, PlanHeader* __restrict__ header,
            int32_t* __restrict__ range_b, int32_t* __restrict__ range_p,
            int32_t* __restrict__ seq_first, int32_t* __restrict__ seq_nsplit,
            int32_t* __restrict__ seq_slot, int32_t* __restrict__ seq_len_eff,
            int32_t* __restrict__ prefix /* [B+1] */) {
  __shared__ int warp_tot[32];
  __shared__ int carry;
  __shared__ int s_prefix[kPlanSmemB + 1];
  __shared__ int s_pages[kPlanSmemB];
  // Clear the status word once the previous step is done with it, then let
  // the absorb step start: it does not read the plan and overlaps this kernel.
  griddep_wait();
  if (threadIdx.x == 0) {
    *status = MLA_STATUS_OK;
    carry = 0;
  }
  __syncthreads();
  griddep_launch_dependents();
  const bool in_smem = B <= kPlanSmemB;
  int* pref = in_smem ? s_prefix : prefix;

  // Pass 1: sanitised lengths and the exclusive prefix of per-sequence cost.
  for (int base = 0; base < B; base += kPlanThreads) {
    const int b = base + threadIdx.x;
    int cost = 0;
    if (b < B) {
      int L = seq_lens[b];
      const int cap = max_pages * kPage;
      if (L < T || L > cap) {
        atomicCAS(status, 0, MLA_STATUS_BOUNDS);
        L = L < T ? T : cap;
      }
      seq_len_eff[b] = L;
      const int pages = (L + kPage - 1) / kPage;
      if (in_smem) s_pages[b] = pages;
      cost = pages + kPieceCost;
    }
    const int incl = block_inclusive_scan(cost, warp_tot);
    if (b < B) pref[b] = carry + incl - cost;
    __syncthreads();
    if (threadIdx.x == kPlanThreads - 1) carry += incl;
    __syncthreads();
  }
  const int total = carry;
  if (threadIdx.x == 0) pref[B] = total;
  const int per = (total + R - 1) / R > 0 ? (total + R - 1) / R : 1;
  __syncthreads();

  // Pass 2: start of every range, by binary search on the prefix.
  for (int k = threadIdx.x; k <= R; k += kPlanThreads) {
    long long x = static_cast<long long>(k) * per;
    int b = B, p = 0;
    if (k < R && x < total) {
      int lo = 0, hi = B - 1;  // largest b with prefix[b] <= x
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pref[mid] <= x) lo = mid; else hi = mid - 1;
      }
      b = lo;
      p = static_cast<int>(x - pref[b]);
      const int pages = in_smem ? s_pages[b] : (seq_len_eff[b] + kPage - 1) / kPage;
      if (p >= pages) { b += 1; p = 0; }
    }
    range_b[k] = b;
    range_p[k] = p;
  }

  // Pass 3: split counts and partial-slot bases.
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < B; base += kPlanThreads) {
    const int b = base + threadIdx.x;
    int ns = 0;
    if (b < B) {
      const int pages = in_smem ? s_pages[b] : (seq_len_eff[b] + kPage - 1) / kPage;
      const int kf = pref[b] / per;
      const int kl = (pref[b] + pages - 1) / per;
      ns = kl - kf + 1;
      seq_first[b] = kf;
      seq_nsplit[b] = ns;
    }
    const int contrib = ns > 1 ? ns : 0;
    const int incl = block_inclusive_scan(contrib, warp_tot);
    if (b < B) seq_slot[b] = ns > 1 ? carry + incl - contrib : -1;
    __syncthreads();
    if (threadIdx.x == kPlanThreads - 1) carry += incl;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    header->num_ranges = R;
    header->per = per;
    header->total_cost = total;
    header->num_slots = carry;
  }
}

}  // namespace

cudaError_t launch_plan(const int32_t* seq_lens, int B, int T, int max_pages, int R,
                        int32_t* status, PlanHeader* header, int32_t* range_b, int32_t* range_p,
                        int32_t* seq_first, int32_t* seq_nsplit, int32_t* seq_slot,
                        int32_t* seq_len_eff, int32_t* prefix, cudaStream_t stream) {
  cudaError_t e = launch_pdl(plan_kernel, dim3(1), dim3(kPlanThreads), 0, stream, seq_lens, B,
                             T, max_pages, R, status, header, range_b, range_p, seq_first,
                             seq_nsplit, seq_slot, seq_len_eff, prefix);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace mla
