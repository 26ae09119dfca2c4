// bmm.cu -- steps a2 and a5: the two per-head bf16 batched matmuls that
// replace materialised absorbed weights (vLLM PR #14770 "[Attention] MLA get
// rid of materialization", PR description: sequential bf16 matmuls with W_UK
// before attention and W_UV after it).
//
//   absorb (a2):      q_lat[tok, h, 0:512] = q_nope[tok, h, :] . W_UK[h]   (K = 128)
//                     q_lat[tok, h, 512:576] = q_pe[tok, h, :]
//   up-project (a5):  out[tok, h, :] = o_lat[tok, h, :] . W_UV[h]          (K = 512)
//
// Both run transposed on the tensor cores so the weight dimension fills the
// 128-row MMA and the (often small) token count is the N dimension (the
// absorb step with 128 tokens or more runs untransposed
// instead; see absorb_rows_kernel):
//   D[m, tok] = sum_k W[h][k][m] * X[tok, h, k]
// A = a 128-wide slice of W[h] (MN-major, staged by TMA with 128B swizzle),
// B = a token tile of X (K-major), D in TMEM (fp32), one CTA per
// (token tile, 128-wide m block, head).  Warp 0 issues TMA, warp 1 issues the
// MMAs, warp 2 owns TMEM; warps 0-3 move the accumulator out of TMEM and all
// warps store the tile.
//
// The absorb epilogue also writes the residual q_lat - bf16(q_lat), scaled by
// 2^10 and stored as FP8 E4M3, which the combine step uses to correct the
// log-sum-exp to first order; the
// q_pe columns of q_lat are copied by the warps not busy with TMA or MMAs
// while the MMAs run.
//
// FP8 weights (W8): the same PR description notes that the absorbed form has
// no FP8 bmm, so FP8 weights are decompressed to bf16 and the bmm runs in bf16.  Here
// the decompression happens inside the bmm: W is stored as FP8 E4M3 with one
// fp32 scale per 128 x 128 block.  FP8 kernels run 192 threads: warps 2-5
// keep a ring of raw 64 x 128 FP8 tiles filled by TMA (issued before the
// kernel waits for its predecessor: the weights do not depend on it), form
// W = bf16(fp32(w8) * scale) (fp32 product, round to nearest even) and write
// it straight into the swizzled shared-memory layout the MMA reads, while
// warp 0 brings the activation tile.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "merge.cuh"
#include "ptx.cuh"

namespace mla {

namespace {

constexpr int kBmmThreads = 128;    // bf16 weights
constexpr int kBmmThreadsW8 = 192;  // FP8 weights: two warps more (2-5 convert)
constexpr int kABytes = 2 * kBoxBytes;  // 128 m x 64 k, two 64-wide m boxes

enum class BmmMode { kAbsorb, kUpProject };

// FP8 weights: E4M3 bytes [H, K, M] (read through the W tensor map) and fp32
// scales [H, K/128, M/128].
struct Fp8Weights {
  const uint8_t* w;
  const float* scale;
  int M;
};

// Raw FP8 tiles kept in flight ahead of the converters: all of K = 128 for the
// absorb step, half of K = 512 for the up-projection.
__host__ __device__ constexpr int raw_tiles(BmmMode mode, bool w8) {
  return !w8 ? 0 : (mode == BmmMode::kAbsorb ? 2 : 4);
}
constexpr int kRawBytes = 64 * 128;  // one FP8 tile: 64 k rows x 128 m bytes

template <int NT, int STAGES, int RAWS>
struct BmmSmem {
  static constexpr int kBBytes = NT * 128;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kOutBytes = NT * 128 * 2;  // bf16 [NT tokens][128 m] staging tile
  static constexpr int kPipe = STAGES * kStageBytes;
  static constexpr int kIn = kPipe + RAWS * kRawBytes;  // raw FP8 ring after the stages
  static constexpr int kBody = kIn > 2 * kOutBytes ? kIn : 2 * kOutBytes;
  static constexpr int kTotal = kBody + 1024;  // + alignment slack
};

// Named barrier over `nthreads` threads that also returns the AND of `pred`
// over them, so the threads leave a loop together.
__device__ __forceinline__ bool named_bar_and(uint32_t id, uint32_t nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// One converter thread's share of a raw FP8 weight tile: k row kr, m (or n)
// columns 64 half .. 64 half + 63.  The raw tile arrives by TMA with 128B
// swizzle (16-byte chunk c of row r at chunk c ^ (r & 7)); the bf16 tile is
// written in the layout TMA gives a bf16 weight tile: two 64-column boxes
// (one per half), 128-byte rows, same swizzle.  The two halves of a row visit
// their chunks in opposite order (jj = j ^ 2 half), so a quarter-warp's
// 16-byte reads and writes fall on eight distinct chunk positions: no bank
// conflicts.
__device__ __forceinline__ void convert_fp8_row(uint32_t raw_tile, uint32_t bf16_tile, int kr,
                                                int half, float sc) {
  const uint32_t rrow = raw_tile + kr * 128;
  const uint32_t arow = bf16_tile + half * kBoxBytes + kr * 128;
#pragma unroll
  for (int j = 0; j < 4; ++j) {  // 16 weights per 16-byte chunk
    const int jj = j ^ (half << 1);
    const int qd = half * 4 + jj;
    const uint4 raw = ld_shared_v4(rrow + ((qd ^ (kr & 7)) << 4));
    const uint32_t rw[4] = {raw.x, raw.y, raw.z, raw.w};
    uint32_t ow[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {  // two E4M3 values -> one bf16 pair
      const __nv_fp8x2_storage_t pr =
          static_cast<__nv_fp8x2_storage_t>((rw[e >> 1] >> (16 * (e & 1))) & 0xFFFFu);
      const float2 f = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(pr, __NV_E4M3)));
      const __nv_bfloat162 bv = __floats2bfloat162_rn(f.x * sc, f.y * sc);
      ow[e] = *reinterpret_cast<const uint32_t*>(&bv);
    }
    const int c0 = 2 * jj;
    st_shared_v4(arow + ((c0 ^ (kr & 7)) << 4), ow[0], ow[1], ow[2], ow[3]);
    st_shared_v4(arow + (((c0 + 1) ^ (kr & 7)) << 4), ow[4], ow[5], ow[6], ow[7]);
  }
}

template <BmmMode MODE, int NT, int STAGES, bool W8>
__global__ void __launch_bounds__(W8 ? kBmmThreadsW8 : kBmmThreads)
bmm_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
           int BT, int H, int K, int Kx, const __nv_bfloat16* __restrict__ q,
           __nv_bfloat16* __restrict__ out_hi, uint8_t* __restrict__ out_lo,
           int32_t* __restrict__ status, Fp8Weights w8) {
  constexpr int RAWS = raw_tiles(MODE, W8);
  constexpr int kRing = RAWS > 0 ? RAWS : 1;  // ring length as a divisor
  extern __shared__ uint8_t smem_raw[];
  // full_bar: the stage's TMA bytes; conv_bar: the converters' bf16 weight
  // tile (W8); raw_bar: one raw FP8 tile's TMA bytes (W8).
  __shared__ __align__(8) uint64_t full_bar[STAGES], empty_bar[STAGES], done_bar,
      conv_bar[W8 ? STAGES : 1], raw_bar[W8 ? RAWS : 1];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;

  // Neither step waits for its predecessor up front.  The absorb step reads
  // only the caller's q and W_UK, so it overlaps the planner; it waits for
  // its predecessor just before exiting, so that its completion still implies
  // the planner's (the attention step relies on it).  The up-projection loads
  // its first weight tiles, then waits (producer thread) before loading o_lat.
  griddep_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tok0 = blockIdx.x * NT;
  const int m0 = blockIdx.y * 128;
  const int h = blockIdx.z;
  const int nk = K / 64;
  constexpr uint32_t kTmemCols = NT < 32 ? 32 : NT;
  using S = BmmSmem<NT, STAGES, RAWS>;

  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* const sbase_ptr = smem_raw + (sbase - smem_u32(smem_raw));

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
      if constexpr (W8) mbar_init(smem_u32(&conv_bar[s]), 1);
    }
    if constexpr (W8)
      for (int r = 0; r < RAWS; ++r) mbar_init(smem_u32(&raw_bar[r]), 1);
    mbar_init(smem_u32(&done_bar), 1);
    abort_sh = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_x);
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(&tmem_base_sh), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  if (warp == 0) {
    if (elect_one()) {
      int kc0 = 0, issued = 0;
      if constexpr (MODE == BmmMode::kUpProject) {
        kc0 = nk < STAGES ? nk : STAGES;
        for (int kc = 0; kc < kc0; ++kc) {
          const uint32_t a = sbase + kc * S::kStageBytes;
          const uint32_t fb = smem_u32(&full_bar[kc]);
          mbar_expect_tx(fb, W8 ? S::kBBytes : S::kStageBytes);
          if (!W8) {
            tma_load_2d(a, &tm_w, m0, h * K + kc * 64, fb);
            tma_load_2d(a + kBoxBytes, &tm_w, m0 + 64, h * K + kc * 64, fb);
          }
        }
        griddep_wait();  // o_lat comes from the step before
        for (int kc = 0; kc < kc0; ++kc) {
          const uint32_t b = sbase + kc * S::kStageBytes + kABytes;
          tma_load_2d(b, &tm_x, h * Kx + kc * 64, tok0, smem_u32(&full_bar[kc]));
        }
        issued = kc0;
      }
      for (int kc = kc0; kc < nk; ++kc) {
        const int s = kc % STAGES;
        if (kc >= STAGES &&
            !mbar_wait(smem_u32(&empty_bar[s]), ((kc / STAGES) - 1) & 1, &abort_sh, status))
          break;
        const uint32_t a = sbase + s * S::kStageBytes;
        const uint32_t b = a + kABytes;
        const uint32_t fb = smem_u32(&full_bar[s]);
        mbar_expect_tx(fb, W8 ? S::kBBytes : S::kStageBytes);
        if (!W8) {
          tma_load_2d(a, &tm_w, m0, h * K + kc * 64, fb);
          tma_load_2d(a + kBoxBytes, &tm_w, m0 + 64, h * K + kc * 64, fb);
        }
        tma_load_2d(b, &tm_x, h * Kx + kc * 64, tok0, fb);
        issued = kc + 1;
      }
      // Copies still in flight (only after a timeout) must land before the
      // CTA exits: wait for the last load of each stage.
      for (int j = issued > STAGES ? issued - STAGES : 0; j < issued; ++j)
        mbar_wait_drain(smem_u32(&full_bar[j % STAGES]), (j / STAGES) & 1, status);
    }
  } else if (W8 && warp >= 2 && warp < 6) {
    // FP8 weight converters: thread ct (0..127) owns m columns 64 half ..
    // 64 half + 63 of k row kr of each stage's 64 x 128 weight tile
    // (convert_fp8_row).
    const int ct = threadIdx.x - 64;
    const int kr = ct >> 1, half = ct & 1;
    const uint32_t raw0 = sbase + S::kPipe;
    int raw_issued = 0;
    if (ct == 0) {
      for (; raw_issued < RAWS && raw_issued < nk; ++raw_issued) {
        const uint32_t rb = smem_u32(&raw_bar[raw_issued]);
        mbar_expect_tx(rb, kRawBytes);
        tma_load_2d(raw0 + raw_issued * kRawBytes, &tm_w, m0, h * K + raw_issued * 64, rb);
      }
    }
    // The scales of this m block: one per 128 k rows (K / 128 <= 4).
    const float* scp = w8.scale + static_cast<size_t>(h) * (K / 128) * (w8.M / 128) + m0 / 128;
    float scl[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) scl[i] = i < K / 128 ? __ldg(scp + i * (w8.M / 128)) : 0.0f;
    int kc = 0;
    for (; kc < nk; ++kc) {
      const int s = kc % STAGES, r = kc % kRing;
      bool ok = true;
      if (kc >= STAGES)
        ok = mbar_wait(smem_u32(&empty_bar[s]), ((kc / STAGES) - 1) & 1, &abort_sh, status);
      if (ok) ok = mbar_wait(smem_u32(&raw_bar[r]), (kc / kRing) & 1, &abort_sh, status);
      if (!named_bar_and(1, 128, ok)) break;
      const int kb = kc >> 1;  // 128-row scale block of this 64-row tile
      const float sc = kb == 0 ? scl[0] : kb == 1 ? scl[1] : kb == 2 ? scl[2] : scl[3];
      convert_fp8_row(raw0 + r * kRawBytes, sbase + s * S::kStageBytes, kr, half, sc);
      // The bf16 tile goes to the tensor core and raw tile r back to TMA:
      // order these threads' shared-memory accesses before both.
      fence_proxy_async_smem();
      named_bar_sync(1, 128);
      if (ct == 0) {
        mbar_arrive(smem_u32(&conv_bar[s]));
        if (raw_issued < nk) {
          const uint32_t rb = smem_u32(&raw_bar[r]);
          mbar_expect_tx(rb, kRawBytes);
          tma_load_2d(raw0 + r * kRawBytes, &tm_w, m0, h * K + raw_issued * 64, rb);
          ++raw_issued;
        }
      }
    }
    // After a timeout, let the raw tiles still in flight land before exiting.
    if (ct == 0)
      for (int j = kc; j < raw_issued; ++j)
        mbar_wait_drain(smem_u32(&raw_bar[j % kRing]), (j / kRing) & 1, status);
  } else if (warp == 1) {
    if (elect_one()) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, NT, /*a_mn=*/true, /*b_mn=*/false);
      for (int kc = 0; kc < nk; ++kc) {
        const int s = kc % STAGES;
        if (!mbar_wait(smem_u32(&full_bar[s]), (kc / STAGES) & 1, &abort_sh, status)) break;
        if constexpr (W8)
          if (!mbar_wait(smem_u32(&conv_bar[s]), (kc / STAGES) & 1, &abort_sh, status)) break;
        tc_fence_after();
        const uint32_t a = sbase + s * S::kStageBytes;
        const uint32_t b = a + kABytes;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t ad = sdesc_sw128(a + kk * 2048, kBoxBytes, 1024);
          const uint64_t bd = sdesc_sw128(b + kk * 32, 16, 1024);
          umma_bf16(tmem, ad, bd, idesc, (kc | kk) != 0);
        }
        umma_commit(smem_u32(&empty_bar[s]));
      }
      umma_commit(smem_u32(&done_bar));
    }
  }
  __syncwarp();
  constexpr int kThreads = W8 ? kBmmThreadsW8 : kBmmThreads;

  if constexpr (MODE == BmmMode::kAbsorb) {
    // q_pe passes through unchanged into columns 512..575 of q_lat (8 chunks
    // of 16 B per token).  The helper warps (2 and up: idle, or done
    // converting) copy it while the MMAs run, all loads before the stores,
    // so the copy costs one memory round trip instead of one per chunk.
    if (blockIdx.y == 0 && warp >= 2) {
      constexpr int kHelpers = kThreads - 64;
      constexpr int kIters = (NT * 8 + kHelpers - 1) / kHelpers;
      const int nchunks = min(NT, BT - tok0) * 8;
      const int t0 = threadIdx.x - 64;
      uint4 v[kIters];
#pragma unroll
      for (int it = 0; it < kIters; ++it) {
        const int i = t0 + it * kHelpers;
        if (i < nchunks) {
          const size_t row = static_cast<size_t>(tok0 + (i >> 3)) * H + h;
          v[it] = *reinterpret_cast<const uint4*>(q + row * kDq + kNope + (i & 7) * 8);
        }
      }
#pragma unroll
      for (int it = 0; it < kIters; ++it) {
        const int i = t0 + it * kHelpers;
        if (i < nchunks) {
          const size_t row = static_cast<size_t>(tok0 + (i >> 3)) * H + h;
          *reinterpret_cast<uint4*>(out_hi + row * kDqk + kLora + (i & 7) * 8) = v[it];
        }
      }
    }
  }

  // Epilogue.  Thread (warp w < 4, lane i) owns feature m0 + 32 w + i: it
  // moves its accumulator column (one value per token) into a bf16
  // [token][128 m] tile in the now idle pipeline smem (and, absorbing, the
  // E4M3 residual into a byte tile), then all threads copy whole token rows
  // (256 + 128 bytes) to global memory with 16-byte stores.
  const bool have = mbar_wait(smem_u32(&done_bar), 0, &abort_sh, status);
  tc_fence_after();
  const int ml = warp * 32 + lane;
  __nv_bfloat16* const tile_hi = reinterpret_cast<__nv_bfloat16*>(sbase_ptr);
  uint8_t* const tile_lo = reinterpret_cast<uint8_t*>(tile_hi + NT * 128);
  const bool go = have && !abort_sh;
  if (go && warp < 4) {  // a warp reaches TMEM lanes 32 (warp % 4) .. + 31
    constexpr int kCols = NT >= 32 ? 32 : 16;  // tokens per TMEM load
#pragma unroll 1
    for (int c0 = 0; c0 < NT; c0 += kCols) {
      uint32_t r[kCols];
      const uint32_t ta = tmem + (static_cast<uint32_t>(warp * 32) << 16) + c0;
      if constexpr (kCols == 32)
        tmem_ld_x32(ta, r);
      else
        tmem_ld_x16(ta, r);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < kCols; ++j) {
        const float v = __uint_as_float(r[j]);
        const __nv_bfloat16 hv = __float2bfloat16_rn(v);
        tile_hi[(c0 + j) * 128 + ml] = hv;
        if constexpr (MODE == BmmMode::kAbsorb)
          tile_lo[(c0 + j) * 128 + ml] = static_cast<uint8_t>(__nv_cvt_float_to_fp8(
              (v - __bfloat162float(hv)) * kQloScale, __NV_SATFINITE, __NV_E4M3));
      }
    }
  }
  __syncthreads();
  if (go) {
    const int ntok = min(NT, BT - tok0);
    // 16 chunks of 16 B per token row.
    for (int i = threadIdx.x; i < ntok * 16; i += kThreads) {
      const int tl = i >> 4, ch = i & 15;
      const size_t row = static_cast<size_t>(tok0 + tl) * H + h;
      const uint4 vh = *reinterpret_cast<const uint4*>(tile_hi + tl * 128 + ch * 8);
      if constexpr (MODE == BmmMode::kAbsorb)
        *reinterpret_cast<uint4*>(out_hi + row * kDqk + m0 + ch * 8) = vh;
      else
        *reinterpret_cast<uint4*>(out_hi + row * kVHead + m0 + ch * 8) = vh;
    }
    if constexpr (MODE == BmmMode::kAbsorb) {
      // 8 chunks of 16 B (128 E4M3 residuals) per token row.
      for (int i = threadIdx.x; i < ntok * 8; i += kThreads) {
        const int tl = i >> 3, ch = i & 7;
        const size_t row = static_cast<size_t>(tok0 + tl) * H + h;
        *reinterpret_cast<uint4*>(out_lo + row * kLora + m0 + ch * 16) =
            *reinterpret_cast<const uint4*>(tile_lo + tl * 128 + ch * 16);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if constexpr (MODE == BmmMode::kAbsorb) griddep_wait();
}

// Absorb step for 128 tokens or more: the untransposed
// product D[tok, n] = sum_k X[tok, h, k] W_UK[h][k][n], one unit of work per
// (128-token tile, 128 latent columns, head), M = 128 tokens, N = 128, K = 128
// in two 64-deep stages.  A is the token tile of q_nope (K-major: the same TMA
// box the transposed kernel uses as B), B a 128-column slice of W_UK[h]
// (MN-major: two boxes of 64 columns).  An M = 128 accumulator holds token row
// i in TMEM lane i, so each epilogue thread owns one token: it converts its
// row (bf16 q_lat and the E4M3 residual) and writes it with 16-byte stores
// into 128B-swizzled staging tiles, and TMA tensor stores move whole
// 128-token boxes to global memory.  (Storing the rows from registers instead
// puts 32 rows in every warp store instruction: 44 -> 63 us for 512 tokens x
// 128 heads.)
//
// Persistent: one CTA per SM walks the units with a stride of the grid size,
// through a ring of TMA stages, two TMEM accumulators and two staging
// buffers, so the loads and MMAs of the next unit overlap the conversion and
// stores of the current one (one unit per short-lived CTA left the SMs waiting
// on memory: 16 % of warps active, DRAM at a third of its peak).  Its shared
// memory (193 KB) leaves room for the planner, which runs at the same time.
//   warp 0: TMA producer; warp 1: TMEM owner and MMA issuer; warps 2-9:
//   epilogue (TMEM lane quarter = warp % 4, two warps per quarter splitting
//   the columns, so each SM sub-partition has two to switch between), q_pe
//   pass-through and the tensor stores.
//
// FP8 weights (W8): each stage also holds the raw 64 k x 128 n FP8 tile,
// and warps 10-13 decompress it, W = bf16(fp32(w8) * scale), into the
// stage's B operand, which has exactly the layout of the transposed kernel's
// bf16 weight tile (two 64-column boxes of 64 k rows, 128B swizzle), so the
// same conversion applies.  One staging buffer keeps the shared memory
// (169 KB) clear of the planner's.
constexpr int kArEpiThreads = 256;                         // warps 2-9
constexpr int kArStages = 3;
constexpr int kArXBytes = 128 * 128;                       // 128 tokens x 64 k
constexpr int kArStageBytes = kArXBytes + 2 * kBoxBytes;   // + 64 k x 128 n: 32 KB
constexpr int kArHiBytes = 2 * 128 * 128;                  // 128 tokens x 128 n, bf16
constexpr int kArLoBytes = 128 * 128;                      // 128 tokens x 128 n, E4M3
constexpr int kArOutBytes = kArHiBytes + kArLoBytes;
template <bool W8>
struct RowsCfg {
  static constexpr int kThreads = 64 + kArEpiThreads + (W8 ? 128 : 0);
  static constexpr int kRawStage = W8 ? kRawBytes : 0;  // raw FP8 tile per stage
  static constexpr int kOutBufs = W8 ? 1 : 2;
  static constexpr int kSmem =
      kArStages * (kArStageBytes + kRawStage) + kOutBufs * kArOutBytes + 1024;
};

template <bool W8>
__global__ void __launch_bounds__(RowsCfg<W8>::kThreads, 1)
absorb_rows_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                   const __grid_constant__ CUtensorMap tm_hi,
                   const __grid_constant__ CUtensorMap tm_lo, int BT, int H,
                   const __nv_bfloat16* __restrict__ q, __nv_bfloat16* __restrict__ out_hi,
                   int32_t* __restrict__ status, const float* __restrict__ w8_scale) {
  using C = RowsCfg<W8>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kArStages], empty_bar[kArStages],
      conv_bar[W8 ? kArStages : 1], acc_full[2], acc_empty[2], drain_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;

  // Like the transposed absorb kernel: q and W_UK come from the caller, so
  // nothing is waited for up front; the wait for the predecessor (the
  // planner) comes just before exiting.
  griddep_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ntt = (BT + 127) / 128;
  const int units = ntt * (kLora / 128) * H;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t raw0 = sbase + kArStages * kArStageBytes;  // raw FP8 tiles (W8)
  const uint32_t sout = raw0 + kArStages * C::kRawStage;
  // Unit u: token tile u % ntt, latent block (u / ntt) % 4, head u / (4 ntt).
  auto coords = [&](int u, int& tok0, int& n0, int& h) {
    tok0 = (u % ntt) * 128;
    n0 = ((u / ntt) % (kLora / 128)) * 128;
    h = u / (ntt * (kLora / 128));
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kArStages; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
      if constexpr (W8) mbar_init(smem_u32(&conv_bar[s]), 1);
    }
    for (int j = 0; j < 2; ++j) {
      mbar_init(smem_u32(&acc_full[j]), 1);
      mbar_init(smem_u32(&acc_empty[j]), kArEpiThreads / 32);
    }
    mbar_init(smem_u32(&drain_bar), 1);
    abort_sh = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_hi);
    tma_prefetch_desc(&tm_lo);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_base_sh), 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  if (warp == 0) {
    if (elect_one()) {
      int g = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
        int tok0, n0, h;
        coords(u, tok0, n0, h);
        for (int kc = 0; kc < 2; ++kc, ++g) {
          const int s = g % kArStages;
          if (g >= kArStages &&
              !mbar_wait(smem_u32(&empty_bar[s]), ((g / kArStages) - 1) & 1, &abort_sh, status)) {
            ok = false;
            break;
          }
          const uint32_t x = sbase + s * kArStageBytes;
          const uint32_t fb = smem_u32(&full_bar[s]);
          mbar_expect_tx(fb, W8 ? kArXBytes + C::kRawStage : kArStageBytes);
          tma_load_2d(x, &tm_x, h * kDq + kc * 64, tok0, fb);
          if constexpr (W8) {
            tma_load_2d(raw0 + s * C::kRawStage, &tm_w, n0, h * kNope + kc * 64, fb);
          } else {
            tma_load_2d(x + kArXBytes, &tm_w, n0, h * kNope + kc * 64, fb);
            tma_load_2d(x + kArXBytes + kBoxBytes, &tm_w, n0 + 64, h * kNope + kc * 64, fb);
          }
        }
      }
      // Copies still in flight (only after a timeout) land before the CTA
      // exits: wait for the last load of each stage.
      for (int j = g > kArStages ? g - kArStages : 0; j < g; ++j)
        mbar_wait_drain(smem_u32(&full_bar[j % kArStages]), (j / kArStages) & 1, status);
    }
  } else if (warp == 1) {
    if (elect_one()) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, 128, /*a_mn=*/false, /*b_mn=*/true);
      int g = 0, i = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++i) {
        const int j = i & 1;
        if (i >= 2 &&
            !mbar_wait(smem_u32(&acc_empty[j]), ((i >> 1) - 1) & 1, &abort_sh, status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kc = 0; kc < 2; ++kc, ++g) {
          const int s = g % kArStages;
          if (!mbar_wait(smem_u32(&full_bar[s]), (g / kArStages) & 1, &abort_sh, status) ||
              (W8 && !mbar_wait(smem_u32(&conv_bar[s]), (g / kArStages) & 1, &abort_sh, status))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t x = sbase + s * kArStageBytes;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            // 16 k per MMA: 32 bytes along a token row of A, 16 rows of B.
            const uint64_t ad = sdesc_sw128(x + kk * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(x + kArXBytes + kk * 2048, kBoxBytes, 1024);
            umma_bf16(tmem + 128 * j, ad, bd, idesc, (kc | kk) != 0);
          }
          umma_commit(smem_u32(&empty_bar[s]));
        }
        if (!ok) break;
        umma_commit(smem_u32(&acc_full[j]));
      }
      // Drain this thread's MMAs before TMEM is released.
      umma_commit(smem_u32(&drain_bar));
      mbar_wait_drain(smem_u32(&drain_bar), 0, status);
    }
  } else if (W8 && warp >= 2 + kArEpiThreads / 32) {
    // FP8 converters (warps 10-13): thread ct owns k row ct / 2, columns
    // 64 (ct % 2) .. + 63 of each stage's weight tile.
    const int ct = threadIdx.x - 64 - kArEpiThreads;
    int g = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
      int tok0, n0, h;
      coords(u, tok0, n0, h);
      // W_UK scales [H, 1, 4]: one per 128 x 128 block.
      const float sc = __ldg(w8_scale + h * (kLora / 128) + n0 / 128);
      for (int kc = 0; kc < 2; ++kc, ++g) {
        const int s = g % kArStages;
        ok = mbar_wait(smem_u32(&full_bar[s]), (g / kArStages) & 1, &abort_sh, status);
        if (!named_bar_and(2, 128, ok)) {
          ok = false;
          break;
        }
        convert_fp8_row(raw0 + s * C::kRawStage, sbase + s * kArStageBytes + kArXBytes, ct >> 1,
                        ct & 1, sc);
        // The bf16 tile goes to the tensor core: order these threads' shared
        // memory writes before it.
        fence_proxy_async_smem();
        named_bar_sync(2, 128);
        if (ct == 0) mbar_arrive(smem_u32(&conv_bar[s]));
      }
    }
  } else {
    // Epilogue: thread (quarter q4 = warp % 4, lane) owns token row
    // r = 32 q4 + lane of each unit's tile (TMEM lane r); warps 2-5 take its
    // columns 0-63, warps 6-9 columns 64-127.  Per 32 columns: one TMEM load,
    // then 64 bytes of bf16 q_lat and 32 bytes of E4M3 residual
    // (q_lat - bf16(q_lat)) * 2^10 into the unit's staging buffer, whose
    // 128-byte rows hold 16-byte chunk c at c ^ (r & 7) (the 128B swizzle the
    // tensor stores expect; a warp's stores then hit eight distinct chunk
    // positions per eight rows).
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const int c0 = warp < 6 ? 0 : 2;      // first of this warp's two 32-column chunks
    const int et = threadIdx.x - 64;      // 0 .. kArEpiThreads - 1
    const uint32_t rsw = static_cast<uint32_t>(r & 7);
    constexpr int kPeIters = 128 * 8 / kArEpiThreads;
    int i = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++i) {
      int tok0, n0, h;
      coords(u, tok0, n0, h);
      const int j = i & 1;
      const uint32_t hi_t = sout + (i % C::kOutBufs) * kArOutBytes, lo_t = hi_t + kArHiBytes;
      // The first latent block's unit also passes q_pe through into columns
      // 512..575 of q_lat: loads now, stores once the tile is out.
      const bool pe = n0 == 0;
      uint4 pv[kPeIters];
      if (pe) {
#pragma unroll
        for (int it = 0; it < kPeIters; ++it) {
          const int idx = et + it * kArEpiThreads, tl = idx >> 3, ch = idx & 7;
          if (tok0 + tl < BT)
            pv[it] = *reinterpret_cast<const uint4*>(
                q + (static_cast<size_t>(tok0 + tl) * H + h) * kDq + kNope + ch * 8);
        }
      }
      const bool ok = mbar_wait(smem_u32(&acc_full[j]), (i >> 1) & 1, &abort_sh, status);
      // With two staging buffers, buffer j was last read by the tensor stores
      // of unit i - 2, and only those of unit i - 1 may still be reading;
      // with one, unit i - 1's must be done.
      if (et == 0) {
        if constexpr (C::kOutBufs == 2)
          tma_store_wait_read_all_but_last();
        else
          tma_store_wait_read();
      }
      if (!named_bar_and(1, kArEpiThreads, ok)) break;
      tc_fence_after();
#pragma unroll
      for (int c = c0; c < c0 + 2; ++c) {
        uint32_t v[32];
        tmem_ld_x32(tmem + 128 * j + (static_cast<uint32_t>(q4 * 32) << 16) + c * 32, v);
        tmem_wait_ld();
        uint32_t hw[16], lw[8];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float v0 = __uint_as_float(v[2 * e]), v1 = __uint_as_float(v[2 * e + 1]);
          const __nv_bfloat162 hv = __floats2bfloat162_rn(v0, v1);
          hw[e] = *reinterpret_cast<const uint32_t*>(&hv);
          const float2 hf = __bfloat1622float2(hv);
          // Two residuals per conversion, the first in the low byte.
          const uint32_t pair = __nv_cvt_float2_to_fp8x2(
              make_float2((v0 - hf.x) * kQloScale, (v1 - hf.y) * kQloScale), __NV_SATFINITE,
              __NV_E4M3);
          if (e & 1)
            lw[e >> 1] |= pair << 16;
          else
            lw[e >> 1] = pair;
        }
        // hi: box c / 2, chunks 4 (c % 2) .. + 3;  lo: chunks 2 c, 2 c + 1.
        const uint32_t hrow = hi_t + (c >> 1) * (128 * 128) + r * 128;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          st_shared_v4(hrow + (((4 * (c & 1) + k) ^ rsw) << 4), hw[4 * k], hw[4 * k + 1],
                       hw[4 * k + 2], hw[4 * k + 3]);
        const uint32_t lrow = lo_t + r * 128;
#pragma unroll
        for (int k = 0; k < 2; ++k)
          st_shared_v4(lrow + (((2 * c + k) ^ rsw) << 4), lw[4 * k], lw[4 * k + 1],
                       lw[4 * k + 2], lw[4 * k + 3]);
      }
      // The accumulator goes back to the MMA issuer, the staging tiles to the
      // tensor stores (rows past the last token are clipped by the maps).
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&acc_empty[j]));
      fence_proxy_async_smem();
      named_bar_sync(1, kArEpiThreads);
      if (et == 0) {
        tma_store_2d(&tm_hi, h * kDqk + n0, tok0, hi_t);
        tma_store_2d(&tm_hi, h * kDqk + n0 + 64, tok0, hi_t + 128 * 128);
        tma_store_2d(&tm_lo, h * kLora + n0, tok0, lo_t);
        tma_store_commit();
      }
      if (pe) {
#pragma unroll
        for (int it = 0; it < kPeIters; ++it) {
          const int idx = et + it * kArEpiThreads, tl = idx >> 3, ch = idx & 7;
          if (tok0 + tl < BT)
            *reinterpret_cast<uint4*>(out_hi + (static_cast<size_t>(tok0 + tl) * H + h) * kDqk +
                                      kLora + ch * 8) = pv[it];
        }
      }
    }
    // Shared memory must outlive the tensor stores' reads.
    if (et == 0) tma_store_wait_read();
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
  griddep_wait();
}

// Up-projection for 128 tokens or more (bf16 weights), with the first-order
// LSE correction of the rows of unsplit sequences folded in: the combine step
// then visits only split sequences' rows (merging their partials and
// correcting their lse), where it would otherwise re-read o_lat and q_lo of
// every row.  The product runs untransposed, D[tok, m] = sum_k
// o_lat[tok, h, k] W_UV[h][k][m], one unit per (128-token tile, head): M = 128
// tokens, N = 128, K = 512 in eight 64-deep stages.  Each stage brings by TMA
// the o_lat tile (A, K-major), a 64-row slice of W_UV[h] (B, MN-major: two
// 64-column boxes) and the q_lo tile of the same rows and columns (64 E4M3
// bytes per row), so the correction warps dot o with q_lo out of shared
// memory while the tensor core consumes the same stage; the stage is
// released once both are done with it.  Persistent: one CTA per SM walks the
// units.
//   warp 0: TMA producer; warp 1: TMEM owner and MMA issuer; warps 2-9:
//   correction (thread ct: token row ct % 128, column half ct / 128 of each
//   stage); warps 10-13: epilogue (TMEM lane quarter = warp % 4), out through
//   a 128B-swizzled staging tile and TMA tensor stores.
//
// FP8 weights (W8): each stage brings the raw 64 k x 128 m FP8 slice instead,
// and warps 14-17 decompress it into the B operand (convert_fp8_row: the same
// layout as the transposed kernel's bf16 weight tile); three stages.
constexpr int kUrCorrThreads = 256;
constexpr int kUrABytes = 128 * 128;                 // 128 tokens x 64 k, bf16
constexpr int kUrBBytes = 2 * kBoxBytes;             // 64 k x 128 m, bf16
constexpr int kUrQBytes = 128 * 64;                  // 128 tokens x 64 k, E4M3
constexpr int kUrOutBytes = 2 * 128 * 128;           // 128 tokens x 128 m, bf16
template <bool W8>
struct UpRowsCfg {
  static constexpr int kThreads = 64 + kUrCorrThreads + 128 + (W8 ? 128 : 0);
  static constexpr int kStages = W8 ? 3 : 4;
  static constexpr int kRawStage = W8 ? kRawBytes : 0;   // raw FP8 slice (W8)
  static constexpr int kStageBytes = kUrABytes + kUrBBytes + kUrQBytes + kRawStage;  // 40 / 48 KB
  // TMA bytes per stage: the B operand arrives raw (W8) or as bf16.
  static constexpr int kTxBytes = kUrABytes + kUrQBytes + (W8 ? kRawBytes : kUrBBytes);
  // One staging buffer: with two, dynamic and static shared memory would pass
  // the 227 KB a CTA may have.
  static constexpr int kSmem = kStages * kStageBytes + kUrOutBytes + 1024;
};

template <bool W8>
__global__ void __launch_bounds__(UpRowsCfg<W8>::kThreads, 1)
up_rows_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_o,
               const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_out,
               int BT, int T, int H, const int32_t* __restrict__ seq_nsplit,
               float* __restrict__ lse, float scale, int32_t* __restrict__ status,
               const float* __restrict__ w8_scale) {
  using C = UpRowsCfg<W8>;
  constexpr int kUrStages = C::kStages;
  constexpr int kUrStageBytes = C::kStageBytes;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kUrStages], empty_bar[kUrStages],
      conv_bar[W8 ? kUrStages : 1], acc_full[2], acc_empty[2], drain_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  __shared__ float corr_sh[2][2][128];  // [unit parity][column half][row]

  griddep_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ntt = (BT + 127) / 128;
  const int units = ntt * H;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sout = sbase + kUrStages * kUrStageBytes;
  // Unit u: token tile u % ntt, head u / ntt.
  constexpr int kNk = kLora / 64;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kUrStages; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      // The MMA issuer's commit and one arrival per correction warp.
      mbar_init(smem_u32(&empty_bar[s]), 1 + kUrCorrThreads / 32);
      if constexpr (W8) mbar_init(smem_u32(&conv_bar[s]), 1);
    }
    for (int j = 0; j < 2; ++j) {
      mbar_init(smem_u32(&acc_full[j]), 1);
      mbar_init(smem_u32(&acc_empty[j]), 4);
    }
    mbar_init(smem_u32(&drain_bar), 1);
    abort_sh = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_o);
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_out);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_base_sh), 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  // The stage's slice of W_UV: two bf16 boxes into the B operand, or the raw
  // FP8 slice (W8) next to the stage's other tiles.
  auto load_w = [&](uint32_t st, int h, int kc, uint32_t fb) {
    if constexpr (W8) {
      tma_load_2d(st + kUrABytes + kUrBBytes + kUrQBytes, &tm_w, 0, h * kLora + kc * 64, fb);
    } else {
      tma_load_2d(st + kUrABytes, &tm_w, 0, h * kLora + kc * 64, fb);
      tma_load_2d(st + kUrABytes + kBoxBytes, &tm_w, 64, h * kLora + kc * 64, fb);
    }
  };
  if (warp == 0) {
    if (elect_one()) {
      // The weight slices of the first stages do not depend on the previous
      // step: they load before the wait for it, o_lat and q_lo after.
      const int u0 = blockIdx.x;
      const int first = u0 < units ? (kNk < kUrStages ? kNk : kUrStages) : 0;
      for (int kc = 0; kc < first; ++kc) {
        const uint32_t st = sbase + kc * kUrStageBytes;
        const uint32_t fb = smem_u32(&full_bar[kc]);
        const int h = u0 / ntt;
        mbar_expect_tx(fb, C::kTxBytes);
        load_w(st, h, kc, fb);
      }
      griddep_wait();  // o_lat and q_lo come from the steps before
      int g = 0;
      bool ok = true;
      for (int u = u0; u < units && ok; u += gridDim.x) {
        const int tok0 = (u % ntt) * 128, h = u / ntt;
        for (int kc = 0; kc < kNk; ++kc, ++g) {
          const int s = g % kUrStages;
          const uint32_t st = sbase + s * kUrStageBytes;
          const uint32_t fb = smem_u32(&full_bar[s]);
          if (g >= first) {
            if (g >= kUrStages &&
                !mbar_wait(smem_u32(&empty_bar[s]), ((g / kUrStages) - 1) & 1, &abort_sh,
                           status)) {
              ok = false;
              break;
            }
            mbar_expect_tx(fb, C::kTxBytes);
            load_w(st, h, kc, fb);
          }
          tma_load_2d(st, &tm_o, h * kLora + kc * 64, tok0, fb);
          tma_load_2d(st + kUrABytes + kUrBBytes, &tm_q, h * kLora + kc * 64, tok0, fb);
        }
      }
      // Copies still in flight (only after a timeout) land before the CTA
      // exits: wait for the last load of each stage.
      for (int j = g > kUrStages ? g - kUrStages : 0; j < g; ++j)
        mbar_wait_drain(smem_u32(&full_bar[j % kUrStages]), (j / kUrStages) & 1, status);
    }
  } else if (warp == 1) {
    griddep_wait();
    if (elect_one()) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, 128, /*a_mn=*/false, /*b_mn=*/true);
      int g = 0, i = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++i) {
        const int j = i & 1;
        if (i >= 2 &&
            !mbar_wait(smem_u32(&acc_empty[j]), ((i >> 1) - 1) & 1, &abort_sh, status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kc = 0; kc < kNk; ++kc, ++g) {
          const int s = g % kUrStages;
          if (!mbar_wait(smem_u32(&full_bar[s]), (g / kUrStages) & 1, &abort_sh, status) ||
              (W8 && !mbar_wait(smem_u32(&conv_bar[s]), (g / kUrStages) & 1, &abort_sh, status))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = sbase + s * kUrStageBytes;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = sdesc_sw128(st + kk * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(st + kUrABytes + kk * 2048, kBoxBytes, 1024);
            umma_bf16(tmem + 128 * j, ad, bd, idesc, (kc | kk) != 0);
          }
          umma_commit(smem_u32(&empty_bar[s]));
        }
        if (!ok) break;
        umma_commit(smem_u32(&acc_full[j]));
      }
      umma_commit(smem_u32(&drain_bar));
      mbar_wait_drain(smem_u32(&drain_bar), 0, status);
    }
  } else if (warp < 2 + kUrCorrThreads / 32) {
    // Correction warps: thread ct owns token row r = ct % 128 of each unit
    // and columns 32 hf .. 32 hf + 31 (hf = ct / 128) of each 64-column
    // stage: 64 bytes of o (A rows are 128 bytes, 16-byte chunk c at
    // c ^ (r & 7)) and 32 bytes of q_lo (64-byte rows, unswizzled).
    griddep_wait();
    const int ct = threadIdx.x - 64;
    const int r = ct & 127, hf = ct >> 7;
    int g = 0, i = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++i) {
      const int tok0 = (u % ntt) * 128, h = u / ntt;
      const int tok = tok0 + r;
      const bool mine = tok < BT && seq_nsplit[tok / T] <= 1;  // unsplit rows only
      const size_t row = static_cast<size_t>(tok) * H + h;
      // The row's lse (from the attention step) loads now, under the stages,
      // rather than at the end of the unit where it would hold up the next.
      const float lse_in = (mine && hf == 0) ? lse[row] : 0.0f;
      float corr = 0.0f;
      for (int kc = 0; kc < kNk; ++kc, ++g) {
        const int s = g % kUrStages;
        ok = mbar_wait(smem_u32(&full_bar[s]), (g / kUrStages) & 1, &abort_sh, status);
        if (!ok) break;
        if (mine) {
          const uint32_t st = sbase + s * kUrStageBytes;
          const uint32_t arow = st + r * 128;
          const uint32_t qrow = st + kUrABytes + kUrBBytes + r * 64 + hf * 32;
          const uint4 q0 = ld_shared_v4(qrow), q1 = ld_shared_v4(qrow + 16);
          const uint32_t qw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint4 ov = ld_shared_v4(arow + (((4 * hf + c) ^ (r & 7)) << 4));
            const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const __nv_bfloat162 o2 = *reinterpret_cast<const __nv_bfloat162*>(&ow[e]);
              const float2 l2 = qlo_pair(qw[2 * c + (e >> 1)] >> (16 * (e & 1)));
              corr += l2.x * __low2float(o2) + l2.y * __high2float(o2);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty_bar[s]));
      }
      // The two column halves of a row meet in shared memory (one buffer per
      // unit parity, so one barrier per unit suffices).
      corr_sh[i & 1][hf][r] = corr;
      if (!named_bar_and(1, kUrCorrThreads, ok)) break;
      if (hf == 0 && mine)
        lse[row] = lse_in + scale * kQloInvScale * (corr_sh[i & 1][0][r] + corr_sh[i & 1][1][r]);
    }
  } else if (W8 && warp >= 2 + kUrCorrThreads / 32 + 4) {
    // FP8 converters (warps 14-17): thread ct owns k row ct / 2, columns
    // 64 (ct % 2) .. + 63 of each stage's weight slice.
    griddep_wait();
    const int ct = threadIdx.x - 64 - kUrCorrThreads - 128;
    int g = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
      const int h = u / ntt;
      for (int kc = 0; kc < kNk; ++kc, ++g) {
        const int s = g % kUrStages;
        ok = mbar_wait(smem_u32(&full_bar[s]), (g / kUrStages) & 1, &abort_sh, status);
        if (!named_bar_and(3, 128, ok)) {
          ok = false;
          break;
        }
        // W_UV scales [H, 4, 1]: one per 128 k rows.
        const float sc = __ldg(w8_scale + h * (kLora / 128) + kc / 2);
        const uint32_t st = sbase + s * kUrStageBytes;
        convert_fp8_row(st + kUrABytes + kUrBBytes + kUrQBytes, st + kUrABytes, ct >> 1, ct & 1,
                        sc);
        fence_proxy_async_smem();  // the bf16 slice goes to the tensor core
        named_bar_sync(3, 128);
        if (ct == 0) mbar_arrive(smem_u32(&conv_bar[s]));
      }
    }
  } else {
    // Epilogue: thread (quarter q4 = warp % 4, lane) owns token row
    // 32 q4 + lane of each unit (TMEM lane); out goes to the staging buffer
    // (two 64-column boxes, 128-byte rows, 16-byte chunk c at c ^ (row & 7))
    // and out by two tensor stores.
    griddep_wait();
    const int q4 = warp & 3;
    const int rr = q4 * 32 + lane;
    const int et = threadIdx.x - 64 - kUrCorrThreads;  // 0..127
    const uint32_t rsw = static_cast<uint32_t>(rr & 7);
    int i = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++i) {
      const int tok0 = (u % ntt) * 128, h = u / ntt;
      const int j = i & 1;
      const uint32_t ot = sout;
      const bool ok = mbar_wait(smem_u32(&acc_full[j]), (i >> 1) & 1, &abort_sh, status);
      // The staging buffer was last read by the tensor stores of unit i - 1.
      if (et == 0) tma_store_wait_read();
      if (!named_bar_and(2, 128, ok)) break;
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld_x32(tmem + 128 * j + (static_cast<uint32_t>(q4 * 32) << 16) + c * 32, v);
        tmem_wait_ld();
        uint32_t hw[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const __nv_bfloat162 hv =
              __floats2bfloat162_rn(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
          hw[e] = *reinterpret_cast<const uint32_t*>(&hv);
        }
        const uint32_t orow = ot + (c >> 1) * (128 * 128) + rr * 128;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          st_shared_v4(orow + (((4 * (c & 1) + k) ^ rsw) << 4), hw[4 * k], hw[4 * k + 1],
                       hw[4 * k + 2], hw[4 * k + 3]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&acc_empty[j]));
      fence_proxy_async_smem();
      named_bar_sync(2, 128);
      if (et == 0) {
        tma_store_2d(&tm_out, h * kVHead, tok0, ot);
        tma_store_2d(&tm_out, h * kVHead + 64, tok0, ot + 128 * 128);
        tma_store_commit();
      }
    }
    if (et == 0) tma_store_wait_read();
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}


// Combine and up-projection in one kernel, for small batches whose
// 16-token tiles of all heads fit in one wave: the up-projection's B operand
// (the tile's o rows, bf16) is built in shared memory by merge warps, one per
// token, with the combine's own routines (merge.cuh), so a merged row never
// goes through global memory (unsplit rows are read from o_lat as the
// attention step wrote them) and one kernel boundary of the step disappears.
// Rows of split sequences are merged from their partials, rows of unsplit
// ones copied from o_lat; either way the row's lse gets its first-order
// correction, and the result equals, bit for bit, the combine kernel followed
// by the up-projection.  The W_UV slices (A, all eight 64-deep K stages) load
// by TMA before the wait for the attention step.
//   warp 0: TMA producer; warp 1: MMA issuer; warp 2: TMEM owner; warps 0-3:
//   epilogue (as in bmm_kernel); warps 4-19: merge warps.
// FP8 weights (W8): the eight raw 64 k x 128 m FP8 slices load instead, and
// warps 20-23 decompress each into its bf16 stage (convert_fp8_row, the
// layout TMA gives the bf16 slices), so the result equals the bf16 weights'
// run on the decompressed weights bit for bit.
constexpr int kCuNT = 16;                            // tokens per tile
constexpr int kCuThreads = 128 + 32 * kCuNT;
constexpr int kCuChunkBytes = kCuNT * 128;           // one 64-deep K chunk of the B tile
constexpr int kCuSmem = 8 * kABytes + 8 * kCuChunkBytes + 1024;

template <bool W8>
struct CuCfg {
  static constexpr int kThreads = kCuThreads + (W8 ? 128 : 0);
  static constexpr int kSmem = kCuSmem + (W8 ? 8 * kRawBytes : 0);
};

template <int kUnroll, int kFewN, bool W8>
__global__ void __launch_bounds__(CuCfg<W8>::kThreads, 1)
combine_up_kernel(const __grid_constant__ CUtensorMap tm_w, int B, int T, int H,
                  const uint8_t* __restrict__ ws, const PlanHeader* __restrict__ header,
                  const int32_t* __restrict__ seq_nsplit, const int32_t* __restrict__ seq_slot,
                  const uint8_t* __restrict__ qlo, const __nv_bfloat16* __restrict__ olat,
                  float* __restrict__ lse, float scale, __nv_bfloat16* __restrict__ out,
                  int32_t* __restrict__ status, const float* __restrict__ w8_scale) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[8], conv_bar[W8 ? 8 : 1], b_ready, done_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;

  griddep_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int BT = B * T, TH = T * H;
  const int tok0 = blockIdx.x * kCuNT;
  const int h = blockIdx.y;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* const sbase_ptr = smem_raw + (sbase - smem_u32(smem_raw));
  const uint32_t btile = sbase + 8 * kABytes;
  const uint32_t rawbase = btile + 8 * kCuChunkBytes;  // W8: raw FP8 slices

  if (threadIdx.x == 0) {
    for (int s = 0; s < 8; ++s) mbar_init(smem_u32(&full_bar[s]), 1);
    if constexpr (W8)
      for (int s = 0; s < 8; ++s) mbar_init(smem_u32(&conv_bar[s]), 1);
    mbar_init(smem_u32(&b_ready), 1);
    mbar_init(smem_u32(&done_bar), 1);
    abort_sh = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_w);
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(&tmem_base_sh), 32);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  if (warp == 0) {
    if (elect_one()) {
      // W_UV does not depend on the attention step: all of K loads at once.
      for (int kc = 0; kc < 8; ++kc) {
        const uint32_t a = sbase + kc * kABytes;
        const uint32_t fb = smem_u32(&full_bar[kc]);
        if constexpr (W8) {
          mbar_expect_tx(fb, kRawBytes);
          tma_load_2d(rawbase + kc * kRawBytes, &tm_w, 0, h * kLora + kc * 64, fb);
        } else {
          mbar_expect_tx(fb, kABytes);
          tma_load_2d(a, &tm_w, 0, h * kLora + kc * 64, fb);
          tma_load_2d(a + kBoxBytes, &tm_w, 64, h * kLora + kc * 64, fb);
        }
      }
    }
  } else if (warp == 1) {
    if (elect_one()) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, kCuNT, /*a_mn=*/true, /*b_mn=*/false);
      if (mbar_wait(smem_u32(&b_ready), 0, &abort_sh, status)) {
        for (int kc = 0; kc < 8; ++kc) {
          if (!mbar_wait(smem_u32(&full_bar[kc]), 0, &abort_sh, status)) break;
          if (W8 && !mbar_wait(smem_u32(&conv_bar[kc]), 0, &abort_sh, status)) break;
          tc_fence_after();
          const uint32_t a = sbase + kc * kABytes;
          const uint32_t b = btile + kc * kCuChunkBytes;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = sdesc_sw128(a + kk * 2048, kBoxBytes, 1024);
            const uint64_t bd = sdesc_sw128(b + kk * 32, 16, 1024);
            umma_bf16(tmem, ad, bd, idesc, (kc | kk) != 0);
          }
        }
      }
      umma_commit(smem_u32(&done_bar));
    }
  } else if (W8 && warp >= 4 + kCuNT) {
    // FP8 converters: thread ct owns k row ct / 2, columns 64 (ct % 2) .. + 63
    // of each slice; W_UV's scales [H, 4, 1] hold one per 128 k rows.
    const int ct = threadIdx.x - kCuThreads;
    bool ok = true;
    for (int kc = 0; kc < 8; ++kc) {
      ok = mbar_wait(smem_u32(&full_bar[kc]), 0, &abort_sh, status);
      if (!named_bar_and(3, 128, ok)) break;
      const float sc = __ldg(w8_scale + h * (kLora / 128) + kc / 2);
      convert_fp8_row(rawbase + kc * kRawBytes, sbase + kc * kABytes, ct >> 1, ct & 1, sc);
      fence_proxy_async_smem();  // the bf16 slice goes to the tensor core
      named_bar_sync(3, 128);
      if (ct == 0) mbar_arrive(smem_u32(&conv_bar[kc]));
    }
  } else if (warp >= 4) {
    // Merge warp mw: token tok0 + mw, row mw of each K chunk of the B tile
    // (128-byte rows, 16-byte unit u at u ^ (mw & 7): the layout a TMA box of
    // the tile would have).
    const int mw = warp - 4;
    const int tok = tok0 + mw;
    if (tok < BT) {
      const int b = tok / T;
      const int r = (tok % T) * H + h;
      const size_t row = static_cast<size_t>(b) * TH + r;
      const uint32_t rbase = btile + mw * 128;
      const uint32_t rsw = static_cast<uint32_t>(mw & 7);
      const int ns = seq_nsplit[b];
      if (ns <= 1) {
        // Lane l holds latent columns 16 l .. 16 l + 15: chunk l / 4,
        // units 2 (l % 4) and 2 (l % 4) + 1.
        correct_unsplit_row(row, lane, qlo, olat, lse, scale,
                            [&](const uint4& o0, const uint4& o1) {
                              const uint32_t cb = rbase + (lane >> 2) * kCuChunkBytes;
                              const uint32_t u0 = 2u * (lane & 3);
                              st_shared_v4(cb + ((u0 ^ rsw) << 4), o0.x, o0.y, o0.z, o0.w);
                              st_shared_v4(cb + (((u0 + 1) ^ rsw) << 4), o1.x, o1.y, o1.z,
                                           o1.w);
                            });
      } else {
        // Four columns col .. col + 3 (8 bytes): chunk col / 64, unit
        // (col % 64) / 8, bytes (col % 8) * 2 into it.
        merge_split_row<kUnroll, kFewN>(
            b, r, lane, ns, seq_slot[b], B, T, H, ws, header, qlo, lse, scale,
            [&](int col, const uint2& packed) {
              const uint32_t u = static_cast<uint32_t>((col & 63) >> 3);
              st_shared_v2(rbase + (col >> 6) * kCuChunkBytes + ((u ^ rsw) << 4) + (col & 7) * 2,
                           packed.x, packed.y);
            });
      }
    } else {
      griddep_wait();
    }
    // The B tile goes to the tensor core once all merge warps wrote it.
    fence_proxy_async_smem();
    named_bar_sync(1, 32 * kCuNT);
    if (warp == 4 && lane == 0) mbar_arrive(smem_u32(&b_ready));
  }
  __syncwarp();

  // Epilogue (warps 0-3), as in bmm_kernel's up-projection: thread (warp w,
  // lane i) owns feature 32 w + i, stages a bf16 [token][128] tile in the idle
  // stage memory, then the four warps copy whole token rows out.
  if (warp < 4) {
    const bool have = mbar_wait(smem_u32(&done_bar), 0, &abort_sh, status);
    tc_fence_after();
    const int ml = warp * 32 + lane;
    __nv_bfloat16* const tile = reinterpret_cast<__nv_bfloat16*>(sbase_ptr);
    const bool go = __all_sync(0xffffffffu, have && !abort_sh);
    if (go) {
      uint32_t v[kCuNT];
      tmem_ld_x16(tmem + (static_cast<uint32_t>(warp * 32) << 16), v);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < kCuNT; ++j) tile[j * 128 + ml] = __float2bfloat16_rn(__uint_as_float(v[j]));
    }
    named_bar_sync(2, 128);
    if (go) {
      const int ntok = min(kCuNT, BT - tok0);
      for (int i = threadIdx.x; i < ntok * 16; i += 128) {
        const int tl = i >> 4, ch = i & 15;
        const size_t row = static_cast<size_t>(tok0 + tl) * H + h;
        *reinterpret_cast<uint4*>(out + row * kVHead + ch * 8) =
            *reinterpret_cast<const uint4*>(tile + tl * 128 + ch * 8);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  // After a timeout, let W_UV tiles still in flight land before exiting.
  if (warp == 0 && lane == 0 && abort_sh)
    for (int kc = 0; kc < 8; ++kc) mbar_wait_drain(smem_u32(&full_bar[kc]), 0, status);
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 32);
  }
}

template <BmmMode MODE, int NT, int kStagesAll = 0>
cudaError_t launch_bmm_nt(const CUtensorMap& tw, const CUtensorMap& tx, int BT, int H, int K,
                          int Kx, int Mtot, const __nv_bfloat16* q, __nv_bfloat16* hi,
                          uint8_t* lo, int32_t* status, cudaStream_t st,
                          Fp8Weights w8) {
  // Two stages for the absorb step (K = 128) and for 128-token tiles (64 KB of
  // stages, three CTAs per SM); four for the up-projection's smaller tiles,
  // or kStagesAll (all of K) when the caller asks for it.
  constexpr int STAGES =
      kStagesAll ? kStagesAll : ((MODE == BmmMode::kAbsorb || NT == 128) ? 2 : 4);
  auto kern = w8.w ? bmm_kernel<MODE, NT, STAGES, true> : bmm_kernel<MODE, NT, STAGES, false>;
  const int smem = w8.w ? BmmSmem<NT, STAGES, raw_tiles(MODE, true)>::kTotal
                        : BmmSmem<NT, STAGES, 0>::kTotal;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid((BT + NT - 1) / NT, Mtot / 128, H);
  e = launch_pdl(kern, grid, dim3(w8.w ? kBmmThreadsW8 : kBmmThreads), smem, st, tw, tx, BT, H, K, Kx, q, hi, lo,
                 status, w8);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <bool W8>
cudaError_t launch_absorb_rows(const CUtensorMap& tw, const CUtensorMap& tx,
                               const CUtensorMap& thi, const CUtensorMap& tlo, int BT, int H,
                               const __nv_bfloat16* q, __nv_bfloat16* hi, int32_t* status,
                               const float* w8_scale, int sm_count, cudaStream_t st) {
  using C = RowsCfg<W8>;
  cudaError_t e = cudaFuncSetAttribute(absorb_rows_kernel<W8>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  const int units = (BT + 127) / 128 * (kLora / 128) * H;
  e = launch_pdl(absorb_rows_kernel<W8>, dim3(units < sm_count ? units : sm_count),
                 dim3(C::kThreads), C::kSmem, st, tw, tx, thi, tlo, BT, H, q, hi, status,
                 w8_scale);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <bool W8>
cudaError_t launch_up_rows(const CUtensorMap& tw, const CUtensorMap& to, const CUtensorMap& tq,
                           const CUtensorMap& tout, int BT, int T, int H,
                           const int32_t* seq_nsplit, float* lse, float scale, int32_t* status,
                           const float* w8_scale, int sm_count, cudaStream_t st) {
  using C = UpRowsCfg<W8>;
  cudaError_t e = cudaFuncSetAttribute(up_rows_kernel<W8>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  const int units = (BT + 127) / 128 * H;
  e = launch_pdl(up_rows_kernel<W8>, dim3(units < sm_count ? units : sm_count),
                 dim3(C::kThreads), C::kSmem, st, tw, to, tq, tout, BT, T, H, seq_nsplit, lse,
                 scale, status, w8_scale);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int kUnroll, int kFewN, bool W8>
cudaError_t launch_cu(const CUtensorMap& tw, int B, int T, int H, const void* ws,
                      const PlanHeader* header, const int32_t* seq_nsplit,
                      const int32_t* seq_slot, const uint8_t* qlo, const __nv_bfloat16* olat,
                      float* lse, float scale, __nv_bfloat16* out, int32_t* status,
                      const float* w8_scale, cudaStream_t st) {
  using C = CuCfg<W8>;
  auto kern = combine_up_kernel<kUnroll, kFewN, W8>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  dim3 grid((B * T + kCuNT - 1) / kCuNT, H);
  e = launch_pdl(kern, grid, dim3(C::kThreads), C::kSmem, st, tw, B, T, H,
                 static_cast<const uint8_t*>(ws), header, seq_nsplit, seq_slot, qlo, olat, lse,
                 scale, out, status, w8_scale);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

// Token tile used for a given token count (also the TMA box height of X).
// The absorb step keeps 64-token tiles up to 128 tokens: one 128-token tile
// per head and m block would give 4 H CTAs at three per SM, just over one
// wave for 128 heads, where 64-token tiles run four per SM with half the
// epilogue each (measured: 14.3 -> 12.3 us for 128 tokens x 128 heads).  For
// more tokens the larger tiles win (fewer weight re-reads).
int bmm_token_tile(int BT, bool absorb) {
  if (BT <= 16) return 16;
  if (BT <= 32) return 32;
  if (BT <= 64 || (absorb && BT <= 128)) return 64;
  return 128;
}

cudaError_t launch_absorb(const CUtensorMap& tm_wuk, const CUtensorMap& tm_q,
                          const CUtensorMap* tm_qlat, const CUtensorMap* tm_qlo, int BT, int H,
                          const __nv_bfloat16* q, __nv_bfloat16* qlat, uint8_t* qlo,
                          int32_t* status, cudaStream_t st, const uint8_t* wuk8,
                          const float* wuk_scale, int sm_count) {
  const Fp8Weights w8{wuk8, wuk_scale, kLora};
  // 128 tokens or more (measured with bf16 weights, 128 tokens x 128 heads:
  // step 240.8 -> 238.5 us): the untransposed kernel, given output tensor
  // maps for q_lat and q_lo and 128-token boxes of q.
  if (tm_qlat && tm_qlo)
    return wuk8 ? launch_absorb_rows<true>(tm_wuk, tm_q, *tm_qlat, *tm_qlo, BT, H, q, qlat,
                                           status, wuk_scale, sm_count, st)
                : launch_absorb_rows<false>(tm_wuk, tm_q, *tm_qlat, *tm_qlo, BT, H, q, qlat,
                                            status, nullptr, sm_count, st);
  switch (bmm_token_tile(BT, true)) {
    case 16: return launch_bmm_nt<BmmMode::kAbsorb, 16>(tm_wuk, tm_q, BT, H, kNope, kDq, kLora, q, qlat, qlo, status, st, w8);
    case 32: return launch_bmm_nt<BmmMode::kAbsorb, 32>(tm_wuk, tm_q, BT, H, kNope, kDq, kLora, q, qlat, qlo, status, st, w8);
    case 64: return launch_bmm_nt<BmmMode::kAbsorb, 64>(tm_wuk, tm_q, BT, H, kNope, kDq, kLora, q, qlat, qlo, status, st, w8);
    default: return launch_bmm_nt<BmmMode::kAbsorb, 128>(tm_wuk, tm_q, BT, H, kNope, kDq, kLora, q, qlat, qlo, status, st, w8);
  }
}

cudaError_t launch_up_project(const CUtensorMap& tm_wuv, const CUtensorMap& tm_olat, int BT,
                              int H, __nv_bfloat16* out, int32_t* status, cudaStream_t st,
                              const uint8_t* wuv8, const float* wuv_scale, bool one_wave) {
  const Fp8Weights w8{wuv8, wuv_scale, kVHead};
  // When the whole grid runs in one wave, tiles of up to 64 tokens get a stage
  // for each of the eight 64-deep K steps (up to 225 KB of shared memory, one
  // CTA per SM): every o_lat tile loads at once after the wait, and FP8
  // weights are decompressed before o_lat is ready, behind the combine step.
  // 128-token tiles get six of the eight (192 KB; 225 KB with the FP8 raw
  // ring): 128 tokens x 128 heads, step 239.4 -> 237.9 us.
  if (one_wave) {
    switch (bmm_token_tile(BT, false)) {
      case 16: return launch_bmm_nt<BmmMode::kUpProject, 16, 8>(tm_wuv, tm_olat, BT, H, kLora, kLora, kVHead, nullptr, out, nullptr, status, st, w8);
      case 32: return launch_bmm_nt<BmmMode::kUpProject, 32, 8>(tm_wuv, tm_olat, BT, H, kLora, kLora, kVHead, nullptr, out, nullptr, status, st, w8);
      case 64: return launch_bmm_nt<BmmMode::kUpProject, 64, 8>(tm_wuv, tm_olat, BT, H, kLora, kLora, kVHead, nullptr, out, nullptr, status, st, w8);
      case 128: return launch_bmm_nt<BmmMode::kUpProject, 128, 6>(tm_wuv, tm_olat, BT, H, kLora, kLora, kVHead, nullptr, out, nullptr, status, st, w8);
      default: break;
    }
  }
  switch (bmm_token_tile(BT, false)) {
    case 16: return launch_bmm_nt<BmmMode::kUpProject, 16>(tm_wuv, tm_olat, BT, H, kLora, kLora, kVHead, nullptr, out, nullptr, status, st, w8);
    case 32: return launch_bmm_nt<BmmMode::kUpProject, 32>(tm_wuv, tm_olat, BT, H, kLora, kLora, kVHead, nullptr, out, nullptr, status, st, w8);
    case 64: return launch_bmm_nt<BmmMode::kUpProject, 64>(tm_wuv, tm_olat, BT, H, kLora, kLora, kVHead, nullptr, out, nullptr, status, st, w8);
    default: return launch_bmm_nt<BmmMode::kUpProject, 128>(tm_wuv, tm_olat, BT, H, kLora, kLora, kVHead, nullptr, out, nullptr, status, st, w8);
  }
}

cudaError_t launch_up_project_rows(const CUtensorMap& tm_wuv, const CUtensorMap& tm_olat,
                                   const CUtensorMap& tm_qlo, const CUtensorMap& tm_out, int BT,
                                   int T, int H, const int32_t* seq_nsplit, float* lse,
                                   float scale, int32_t* status, const float* wuv_scale,
                                   int sm_count, cudaStream_t st) {
  return wuv_scale ? launch_up_rows<true>(tm_wuv, tm_olat, tm_qlo, tm_out, BT, T, H, seq_nsplit,
                                          lse, scale, status, wuv_scale, sm_count, st)
                   : launch_up_rows<false>(tm_wuv, tm_olat, tm_qlo, tm_out, BT, T, H, seq_nsplit,
                                           lse, scale, status, nullptr, sm_count, st);
}

// Small one-wave batches: combine and up-projection in one kernel, with
// bf16 weights (tm_wuv over w_uv) or FP8 weights (tm_wuv over the FP8 codes,
// wuv_scale their block scales).  splits_per_seq picks the same merge
// variant as the combine step would.
int combine_up_tile() { return kCuNT; }
cudaError_t launch_combine_up(const CUtensorMap& tm_wuv, int B, int T, int H, const void* ws,
                              const PlanHeader* header, const int32_t* seq_nsplit,
                              const int32_t* seq_slot, const uint8_t* qlo,
                              const __nv_bfloat16* olat, float* lse, float scale,
                              __nv_bfloat16* out, int32_t* status, int splits_per_seq,
                              const float* wuv_scale, cudaStream_t st) {
#define MLA_CU_LAUNCH(U, F)                                                                      \
  (wuv_scale ? launch_cu<U, F, true>(tm_wuv, B, T, H, ws, header, seq_nsplit, seq_slot, qlo,    \
                                     olat, lse, scale, out, status, wuv_scale, st)             \
             : launch_cu<U, F, false>(tm_wuv, B, T, H, ws, header, seq_nsplit, seq_slot, qlo,   \
                                      olat, lse, scale, out, status, nullptr, st))
  if (splits_per_seq <= 1) return MLA_CU_LAUNCH(1, 2);
  if (splits_per_seq <= 4) return MLA_CU_LAUNCH(4, 4);
  return MLA_CU_LAUNCH(4, 0);
#undef MLA_CU_LAUNCH
}

}  // namespace mla
