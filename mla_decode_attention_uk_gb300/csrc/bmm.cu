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
// 128-row MMA and the (often small) token count is the N dimension:
//   D[m, tok] = sum_k W[h][k][m] * X[tok, h, k]
// A = a 128-wide slice of W[h] (MN-major, staged by TMA with 128B swizzle),
// B = a token tile of X (K-major), D in TMEM (fp32), one CTA per
// (token tile, 128-wide m block, head).  Warp 0 issues TMA, warp 1 issues the
// MMAs, warp 2 owns TMEM, and all four warps run the epilogue.
//
// The absorb epilogue also writes the bf16 residual q_lat - bf16(q_lat), which
// the attention step uses to correct its log-sum-exp to first order.
//
// FP8 weights (W8): the page says the absorbed form lacks an FP8 bmm, so the
// matrices involved are decompressed to bf16 and the bmm runs in bf16.  Here
// the decompression happens inside the bmm: W is stored as FP8 E4M3 with one
// fp32 scale per 128 x 128 block, warps 2-3 load each stage's 64 x 128 FP8
// tile, form W = bf16(fp32(w8) * scale) (fp32 product, round to nearest even)
// and write it straight into the swizzled shared-memory layout the MMA reads,
// while warp 0 brings the activation tile by TMA.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "ptx.cuh"

namespace mla {

namespace {

constexpr int kBmmThreads = 128;
constexpr int kABytes = 2 * kBoxBytes;  // 128 m x 64 k, two 64-wide m boxes

enum class BmmMode { kAbsorb, kUpProject };

// FP8 weights: E4M3 bytes [H, K, M] and fp32 scales [H, K/128, M/128].
struct Fp8Weights {
  const uint8_t* w;
  const float* scale;
  int M;
};

template <int NT, int STAGES>
struct BmmSmem {
  static constexpr int kBBytes = NT * 128;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kOutBytes = NT * 128 * 2;  // bf16 [NT tokens][128 m] staging tile
  static constexpr int kPipe = STAGES * kStageBytes;
  static constexpr int kBody = kPipe > 2 * kOutBytes ? kPipe : 2 * kOutBytes;
  static constexpr int kTotal = kBody + 1024;  // + alignment slack
};

template <BmmMode MODE, int NT, int STAGES, bool W8>
__global__ void __launch_bounds__(kBmmThreads)
bmm_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
           int BT, int H, int K, int Kx, const __nv_bfloat16* __restrict__ q,
           __nv_bfloat16* __restrict__ out_hi, __nv_bfloat16* __restrict__ out_lo,
           int32_t* __restrict__ status, Fp8Weights w8) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[STAGES], empty_bar[STAGES], done_bar;
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
  using S = BmmSmem<NT, STAGES>;

  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* const sbase_ptr = smem_raw + (sbase - smem_u32(smem_raw));

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      // FP8 weights: the TMA transaction and the converters' arrival.
      mbar_init(smem_u32(&full_bar[s]), W8 ? 2 : 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    mbar_init(smem_u32(&done_bar), 1);
    abort_sh = 0;
    fence_mbar_init();
    if (!W8) tma_prefetch_desc(&tm_w);
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
      int kc0 = 0;
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
      }
    }
  } else if (W8 && warp >= 2) {
    // FP8 weight converters: thread kr (0..63) owns k row kr of each stage's
    // 64 x 128 weight tile.  The tile's bf16 layout is the one TMA would have
    // produced: two 64-column m boxes, 128-byte rows, 16-byte chunks swizzled
    // by the row index (128B swizzle).
    const int kr = threadIdx.x - 64;
    for (int kc = 0; kc < nk; ++kc) {
      const int s = kc % STAGES;
      if (kc >= STAGES &&
          !mbar_wait(smem_u32(&empty_bar[s]), ((kc / STAGES) - 1) & 1, &abort_sh, status))
        break;
      const uint32_t a = sbase + s * S::kStageBytes;
      const size_t krow = static_cast<size_t>(h) * K + kc * 64 + kr;
      const uint4* src = reinterpret_cast<const uint4*>(w8.w + krow * w8.M + m0);
      const float sc =
          __ldg(w8.scale + (static_cast<size_t>(h) * (K / 128) + (kc * 64) / 128) * (w8.M / 128) +
                m0 / 128);
#pragma unroll
      for (int qd = 0; qd < 8; ++qd) {  // 16 weights (m) per 16-byte load
        const uint4 raw = __ldg(src + qd);
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
        const int box = qd >> 2, c0 = 2 * (qd & 3);
        const uint32_t row = a + box * kBoxBytes + kr * 128;
        st_shared_v4(row + ((c0 ^ (kr & 7)) << 4), ow[0], ow[1], ow[2], ow[3]);
        st_shared_v4(row + (((c0 + 1) ^ (kr & 7)) << 4), ow[4], ow[5], ow[6], ow[7]);
      }
      fence_proxy_async_smem();
      named_bar_sync(1, 64);
      if (kr == 0) mbar_arrive(smem_u32(&full_bar[s]));
    }
  } else if (warp == 1) {
    if (elect_one()) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, NT, /*a_mn=*/true, /*b_mn=*/false);
      for (int kc = 0; kc < nk; ++kc) {
        const int s = kc % STAGES;
        if (!mbar_wait(smem_u32(&full_bar[s]), (kc / STAGES) & 1, &abort_sh, status)) break;
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

  // Epilogue.  Thread (warp w, lane i) owns feature m0 + 32 w + i: it moves its
  // accumulator column (one value per token) into a bf16 [token][128 m] tile in
  // the now idle pipeline smem, then all threads copy whole 256-byte token rows
  // to global memory with 16-byte stores.
  const bool have = mbar_wait(smem_u32(&done_bar), 0, &abort_sh, status);
  tc_fence_after();
  const int ml = warp * 32 + lane;
  __nv_bfloat16* const tile_hi = reinterpret_cast<__nv_bfloat16*>(sbase_ptr);
  __nv_bfloat16* const tile_lo = tile_hi + NT * 128;
  const bool go = have && !abort_sh;
  if (go) {
#pragma unroll 1
    for (int c0 = 0; c0 < NT; c0 += 16) {
      uint32_t r[16];
      tmem_ld_x16(tmem + (static_cast<uint32_t>(warp * 32) << 16) + c0, r);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float v = __uint_as_float(r[j]);
        const __nv_bfloat16 hv = __float2bfloat16_rn(v);
        tile_hi[(c0 + j) * 128 + ml] = hv;
        if constexpr (MODE == BmmMode::kAbsorb)
          tile_lo[(c0 + j) * 128 + ml] = __float2bfloat16_rn(v - __bfloat162float(hv));
      }
    }
  }
  __syncthreads();
  if (go) {
    const int ntok = min(NT, BT - tok0);
    // 16 chunks of 16 B per token row; 128 threads cover 8 rows per pass.
    for (int i = threadIdx.x; i < ntok * 16; i += kBmmThreads) {
      const int tl = i >> 4, ch = i & 15;
      const size_t row = static_cast<size_t>(tok0 + tl) * H + h;
      const uint4 vh = *reinterpret_cast<const uint4*>(tile_hi + tl * 128 + ch * 8);
      if constexpr (MODE == BmmMode::kAbsorb) {
        *reinterpret_cast<uint4*>(out_hi + row * kDqk + m0 + ch * 8) = vh;
        const uint4 vl = *reinterpret_cast<const uint4*>(tile_lo + tl * 128 + ch * 8);
        *reinterpret_cast<uint4*>(out_lo + row * kLora + m0 + ch * 8) = vl;
      } else {
        *reinterpret_cast<uint4*>(out_hi + row * kVHead + m0 + ch * 8) = vh;
      }
    }
    if constexpr (MODE == BmmMode::kAbsorb) {
      // q_pe passes through unchanged into columns 512..575 (8 chunks of 16 B).
      if (blockIdx.y == 0) {
        for (int i = threadIdx.x; i < ntok * 8; i += kBmmThreads) {
          const int tl = i >> 3, ch = i & 7;
          const size_t row = static_cast<size_t>(tok0 + tl) * H + h;
          *reinterpret_cast<uint4*>(out_hi + row * kDqk + kLora + ch * 8) =
              *reinterpret_cast<const uint4*>(q + row * kDq + kNope + ch * 8);
        }
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

template <BmmMode MODE, int NT>
cudaError_t launch_bmm_nt(const CUtensorMap& tw, const CUtensorMap& tx, int BT, int H, int K,
                          int Kx, int Mtot, const __nv_bfloat16* q, __nv_bfloat16* hi,
                          __nv_bfloat16* lo, int32_t* status, cudaStream_t st,
                          Fp8Weights w8) {
  // Two stages for the absorb step (K = 128) and for 128-token tiles (64 KB of
  // stages, three CTAs per SM); four for the up-projection's smaller tiles.
  constexpr int STAGES = (MODE == BmmMode::kAbsorb || NT == 128) ? 2 : 4;
  auto kern = w8.w ? bmm_kernel<MODE, NT, STAGES, true> : bmm_kernel<MODE, NT, STAGES, false>;
  const int smem = BmmSmem<NT, STAGES>::kTotal;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid((BT + NT - 1) / NT, Mtot / 128, H);
  e = launch_pdl(kern, grid, dim3(kBmmThreads), smem, st, tw, tx, BT, H, K, Kx, q, hi, lo,
                 status, w8);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

// Token tile used for a given token count (also the TMA box height of X).
int bmm_token_tile(int BT) {
  if (BT <= 16) return 16;
  if (BT <= 32) return 32;
  if (BT <= 64) return 64;
  return 128;
}

cudaError_t launch_absorb(const CUtensorMap& tm_wuk, const CUtensorMap& tm_q, int BT, int H,
                          const __nv_bfloat16* q, __nv_bfloat16* qlat, __nv_bfloat16* qlo,
                          int32_t* status, cudaStream_t st, const uint8_t* wuk8,
                          const float* wuk_scale) {
  const Fp8Weights w8{wuk8, wuk_scale, kLora};
  switch (bmm_token_tile(BT)) {
    case 16: return launch_bmm_nt<BmmMode::kAbsorb, 16>(tm_wuk, tm_q, BT, H, kNope, kDq, kLora, q, qlat, qlo, status, st, w8);
    case 32: return launch_bmm_nt<BmmMode::kAbsorb, 32>(tm_wuk, tm_q, BT, H, kNope, kDq, kLora, q, qlat, qlo, status, st, w8);
    case 64: return launch_bmm_nt<BmmMode::kAbsorb, 64>(tm_wuk, tm_q, BT, H, kNope, kDq, kLora, q, qlat, qlo, status, st, w8);
    default: return launch_bmm_nt<BmmMode::kAbsorb, 128>(tm_wuk, tm_q, BT, H, kNope, kDq, kLora, q, qlat, qlo, status, st, w8);
  }
}

cudaError_t launch_up_project(const CUtensorMap& tm_wuv, const CUtensorMap& tm_olat, int BT,
                              int H, __nv_bfloat16* out, int32_t* status, cudaStream_t st,
                              const uint8_t* wuv8, const float* wuv_scale) {
  const Fp8Weights w8{wuv8, wuv_scale, kVHead};
  switch (bmm_token_tile(BT)) {
    case 16: return launch_bmm_nt<BmmMode::kUpProject, 16>(tm_wuv, tm_olat, BT, H, kLora, kLora, kVHead, nullptr, out, nullptr, status, st, w8);
    case 32: return launch_bmm_nt<BmmMode::kUpProject, 32>(tm_wuv, tm_olat, BT, H, kLora, kLora, kVHead, nullptr, out, nullptr, status, st, w8);
    case 64: return launch_bmm_nt<BmmMode::kUpProject, 64>(tm_wuv, tm_olat, BT, H, kLora, kLora, kVHead, nullptr, out, nullptr, status, st, w8);
    default: return launch_bmm_nt<BmmMode::kUpProject, 128>(tm_wuv, tm_olat, BT, H, kLora, kLora, kVHead, nullptr, out, nullptr, status, st, w8);
  }
}

}  // namespace mla
