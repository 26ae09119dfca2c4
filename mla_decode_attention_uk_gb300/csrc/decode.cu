// decode.cu -- step a3: split-KV latent attention over the paged latent cache.
//
// The method: every query head attends MQA-style to one shared latent cache
// row per token, c_j = [c_kv 512 || k_pe 64], with the query already absorbed
// into latent space (vLLM PR #14770 "[Attention] MLA get rid of
// materialization", PR description).  The cache is BF16 in 64-token pages
// ("DeepSeek publica FlashMLA como codigo abierto", feature list), gathered
// page by page through the block table.  Softmax is computed online, key
// range by key range, in the FlashAttention manner that page credits, and key
// ranges cut by the planner are merged later by their log-sum-exp.
//
// GB300 mapping (one CTA = 64 query rows of one sequence, one work range):
//   * TMA: the absorbed query tile (9 boxes of 64 x 64 bf16) and each 64-token
//     page (9 boxes) land in 128B-swizzled shared memory; two page slots.
//   * QK^T on tcgen05: S[row, key] = sum_576 Q[row] C[key]; M = 128 (rows
//     64..127 of the MMA are unused), N = 64 keys, fp32 in TMEM, two S buffers.
//   * Softmax (warps 4-5, one thread per query row, scores read from TMEM):
//     exp2 with a lazily updated running max (rescale only when the max grows
//     by more than 2^8), P written to shared memory as bf16.
//   * PV on tcgen05, transposed: O^T[latent, row] += C^T[latent, key] P^T[key, row]
//     with the page slot read MN-major as the A operand (M = 128 latent, four
//     MMAs for 512) and N = 64 rows; O^T lives in 256 TMEM columns.
//   * Epilogue (warps 4-7): O / l to bf16 o_lat plus lse for unsplit sequences
//     (with the first-order correction lse += scale * (q_lo . o) for the bf16
//     rounding of the absorbed query), or fp32 partials for split ones.
// Warp roles: 0 TMA producer, 1 MMA issuer, 2 TMEM owner, 3 idle, 4-7 softmax
// and epilogue.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "ptx.cuh"

namespace mla {

namespace {

constexpr int kDecThreads = 256;
constexpr int kQBytes = kBoxes * kBoxBytes;     // 72 KB
constexpr int kPageBytes = kBoxes * kBoxBytes;  // 72 KB
constexpr int kPTBytes = 64 * 128;              // P^T: 64 rows x 64 keys bf16
constexpr int kSmemQ = 0;
constexpr int kSmemSlot0 = kQBytes;
constexpr int kSmemPT = kQBytes + 2 * kPageBytes;
constexpr int kDecSmem = kSmemPT + kPTBytes + 1024;  // + alignment slack
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 128;                // O^T blocks at 128 + 64 m
constexpr float kRescaleThreshold = 8.0f;       // log2 units
constexpr float kLn2 = 0.6931471805599453f;

struct DecodeParams {
  const int32_t* block_table;
  const int32_t* seq_len_eff;
  const PlanHeader* header;
  uint8_t* ws;               // workspace base (R-dependent regions located from the header)
  const int32_t* range_b;    // filled in on the device
  const int32_t* range_p;
  const int32_t* seq_first;
  const int32_t* seq_nsplit;
  const int32_t* seq_slot;
  const __nv_bfloat16* qlo;  // [B*T*H, 512]
  __nv_bfloat16* olat;       // [B*T*H, 512]
  float* lse;                // [B*T*H]
  float* opart;              // [slots, T*H, 512]
  float* lpart;              // [slots, T*H]
  int32_t* status;
  int B, T, H, max_pages, num_pages, tiles, q_box_rows;
  float scale, scale_log2;
};

__device__ __forceinline__ bool bar_any(uint32_t id, uint32_t n, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}\n"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

// Walks the pieces (sequence, page range) of work range k.
struct PieceWalker {
  int b, p, b1, p1;
  __device__ PieceWalker(const DecodeParams& P, int k)
      : b(P.range_b[k]), p(P.range_p[k]), b1(P.range_b[k + 1]), p1(P.range_p[k + 1]) {}
  // Next piece: returns false when the range is exhausted.
  __device__ bool next(const DecodeParams& P, int& pb, int& pbeg, int& pend) {
    while (b < b1 || (b == b1 && p < p1)) {
      const int pages = (P.seq_len_eff[b] + kPage - 1) / kPage;
      const int e = (b == b1) ? p1 : pages;
      const int cb = b, cp = p;
      b += 1;
      p = 0;
      if (e > cp) {
        pb = cb;
        pbeg = cp;
        pend = e;
        return true;
      }
    }
    return false;
  }
};

__global__ void __launch_bounds__(kDecThreads, 1)
decode_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_c,
              DecodeParams P) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t q_full, q_free, slot_full[2], slot_empty[2], s_full[2],
      s_free[2], p_full, p_free, o_full, o_free, drain_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  __shared__ float alpha_sh[64];
  __shared__ float inv_l_sh[64];
  __shared__ float corr_sh[4][64];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x % P.tiles;
  const int k0 = blockIdx.x / P.tiles;
  const int G = gridDim.x / P.tiles;
  const int R = P.header->num_ranges;
  const int TH = P.T * P.H;
  {
    const WsLayout L = make_layout(P.B, P.T, P.H, R);
    P.range_b = reinterpret_cast<const int32_t*>(P.ws + L.range_b);
    P.range_p = reinterpret_cast<const int32_t*>(P.ws + L.range_p);
    P.lpart = reinterpret_cast<float*>(P.ws + L.lpart);
    P.opart = reinterpret_cast<float*>(P.ws + L.opart);
  }
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sQ = sbase + kSmemQ, sSlot0 = sbase + kSmemSlot0, sPT = sbase + kSmemPT;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&q_full), 1);
    mbar_init(smem_u32(&q_free), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&slot_full[i]), 1);
      mbar_init(smem_u32(&slot_empty[i]), 1);
      mbar_init(smem_u32(&s_full[i]), 1);
      mbar_init(smem_u32(&s_free[i]), 2);
    }
    mbar_init(smem_u32(&p_full), 4);
    mbar_init(smem_u32(&p_free), 1);
    mbar_init(smem_u32(&o_full), 1);
    mbar_init(smem_u32(&o_free), 4);
    mbar_init(smem_u32(&drain_bar), 1);
    abort_sh = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_c);
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
    // ------------------------------------------------------------ TMA producer
    if (elect_one()) {
      const uint64_t pol_stream = l2_policy_evict_first();
      const uint32_t q_bytes = static_cast<uint32_t>(P.q_box_rows) * 128u * kBoxes;
      int g = 0, pc = 0;
      bool ok = true;
      for (int k = k0; k < R && ok; k += G) {
        PieceWalker w(P, k);
        int b, pb, pe;
        while (ok && w.next(P, b, pb, pe)) {
          if (pc > 0 && !mbar_wait(smem_u32(&q_free), (pc - 1) & 1, &abort_sh, P.status)) {
            ok = false;
            break;
          }
          const int qrow = b * TH + tile * kTileRows;
          mbar_expect_tx(smem_u32(&q_full), q_bytes);
          for (int j = 0; j < kBoxes; ++j)
            tma_load_2d(sQ + j * kBoxBytes, &tm_q, j * kBoxCols, qrow, smem_u32(&q_full));
          for (int p = pb; p < pe; ++p, ++g) {
            const int s = g & 1;
            if (g >= 2 &&
                !mbar_wait(smem_u32(&slot_empty[s]), ((g >> 1) - 1) & 1, &abort_sh, P.status)) {
              ok = false;
              break;
            }
            int pg = __ldg(P.block_table + static_cast<size_t>(b) * P.max_pages + p);
            if (pg < 0 || pg >= P.num_pages) {
              atomicCAS(P.status, 0, MLA_STATUS_BOUNDS);
              pg = 0;
            }
            const uint32_t dst = sSlot0 + s * kPageBytes;
            mbar_expect_tx(smem_u32(&slot_full[s]), kPageBytes);
            for (int j = 0; j < kBoxes; ++j)
              tma_load_2d_hint(dst + j * kBoxBytes, &tm_c, j * kBoxCols, pg * kPage,
                               smem_u32(&slot_full[s]), pol_stream);
          }
          ++pc;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (elect_one()) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(128, 64, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(128, 64, true, false);
      int g = 0, pc = 0;
      bool ok = true;
      auto issue_pv = [&](int gg, bool first) -> bool {
        if (!mbar_wait(smem_u32(&p_full), gg & 1, &abort_sh, P.status)) return false;
        if (first && pc > 0 && !mbar_wait(smem_u32(&o_free), (pc - 1) & 1, &abort_sh, P.status))
          return false;
        tc_fence_after();
        const uint32_t slot = sSlot0 + (gg & 1) * kPageBytes;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = sdesc_sw128(slot + (2 * m) * kBoxBytes + kk * 2048, kBoxBytes, 1024);
            const uint64_t bd = sdesc_sw128(sPT + kk * 32, 16, 1024);
            umma_bf16(tmem + kTmemO + 64 * m, ad, bd, idesc_pv, !(first && kk == 0));
          }
        }
        umma_commit(smem_u32(&p_free));
        umma_commit(smem_u32(&slot_empty[gg & 1]));
        return true;
      };
      for (int k = k0; k < R && ok; k += G) {
        PieceWalker w(P, k);
        int b, pb, pe;
        while (ok && w.next(P, b, pb, pe)) {
          if (!mbar_wait(smem_u32(&q_full), pc & 1, &abort_sh, P.status)) {
            ok = false;
            break;
          }
          const int np = pe - pb;
          for (int i = 0; i < np; ++i, ++g) {
            const int s = g & 1;
            if (!mbar_wait(smem_u32(&slot_full[s]), (g >> 1) & 1, &abort_sh, P.status) ||
                (g >= 2 &&
                 !mbar_wait(smem_u32(&s_free[s]), ((g >> 1) - 1) & 1, &abort_sh, P.status))) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t slot = sSlot0 + s * kPageBytes;
#pragma unroll
            for (int j = 0; j < kBoxes; ++j) {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint64_t ad = sdesc_sw128(sQ + j * kBoxBytes + kk * 32, 16, 1024);
                const uint64_t bd = sdesc_sw128(slot + j * kBoxBytes + kk * 32, 16, 1024);
                umma_bf16(tmem + 64 * s, ad, bd, idesc_qk, (j | kk) != 0);
              }
            }
            umma_commit(smem_u32(&s_full[s]));
            if (i == np - 1) umma_commit(smem_u32(&q_free));
            if (i > 0 && !issue_pv(g - 1, i - 1 == 0)) {
              ok = false;
              break;
            }
          }
          if (!ok) break;
          if (!issue_pv(g - 1, np == 1)) {
            ok = false;
            break;
          }
          umma_commit(smem_u32(&o_full));
          ++pc;
        }
      }
      // Drain the tensor pipe before TMEM is released.
      umma_commit(smem_u32(&drain_bar));
      mbar_wait_drain(smem_u32(&drain_bar), 0, P.status);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax + epilogue
    const int wq = warp - 4;                    // TMEM lane quarter
    const int c = wq * 32 + lane;               // query row in tile (valid for wq < 2)
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const bool srow = wq < 2;
    int g = 0, pc = 0;
    bool fail = false;
    for (int k = k0; k < R && !fail; k += G) {
      PieceWalker w(P, k);
      int b, pb, pe;
      while (!fail && w.next(P, b, pb, pe)) {
        const int r = tile * kTileRows + c;     // row within the sequence's T*H rows
        const bool row_ok = srow && r < TH;
        const int L = P.seq_len_eff[b];
        const int n_row = row_ok ? L - P.T + r / P.H + 1 : 0;
        float m_used = -INFINITY, l = 0.0f;
        const int np = pe - pb;
        for (int i = 0; i < np; ++i, ++g) {
          const int s = g & 1;
          bool need = false;
          bool bad = false;
          if (srow) {
            if (!mbar_wait(smem_u32(&s_full[s]), (g >> 1) & 1, &abort_sh, P.status)) bad = true;
            bad = __any_sync(0xffffffffu, bad);  // tcgen05.ld below is warp-collective
            uint32_t v[64];
            if (!bad) {
              tc_fence_after();
              tmem_ld_x32(tmem + lane_off + 64 * s, v);
              tmem_ld_x32(tmem + lane_off + 64 * s + 32, v + 32);
              tmem_wait_ld();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&s_free[s]));
            if (!bad) {
              const int key0 = (pb + i) * kPage;
              float x[64];
              float pmax = -INFINITY;
#pragma unroll
              for (int j = 0; j < 64; ++j) {
                x[j] = (key0 + j < n_row) ? __uint_as_float(v[j]) * P.scale_log2 : -INFINITY;
                pmax = fmaxf(pmax, x[j]);
              }
              float alpha = 1.0f;
              if (pmax > m_used + kRescaleThreshold) {
                alpha = (m_used == -INFINITY) ? 0.0f : ex2_approx(m_used - pmax);
                m_used = pmax;
                need = i > 0;
              }
              uint32_t packed[32];
              float sum = 0.0f;
#pragma unroll
              for (int j = 0; j < 64; j += 2) {
                const float p0 = (x[j] == -INFINITY) ? 0.0f : ex2_approx(x[j] - m_used);
                const float p1 = (x[j + 1] == -INFINITY) ? 0.0f : ex2_approx(x[j + 1] - m_used);
                sum += p0 + p1;
                packed[j / 2] = pack_bf16x2(p0, p1);
              }
              l = l * alpha + sum;
              alpha_sh[c] = alpha;
              // The P^T buffer is free once the previous page's PV has finished.
              if (g >= 1 && !mbar_wait(smem_u32(&p_free), (g - 1) & 1, &abort_sh, P.status))
                bad = true;
              if (!bad) {
                const uint32_t rowaddr = sPT + c * 128;
#pragma unroll
                for (int q = 0; q < 8; ++q)
                  st_shared_v4(rowaddr + ((q ^ (c & 7)) << 4), packed[4 * q], packed[4 * q + 1],
                               packed[4 * q + 2], packed[4 * q + 3]);
                fence_proxy_async_smem();
              }
            }
          }
          if (bar_any(1, 128, bad)) { fail = true; break; }
          if (bar_any(1, 128, need)) {
            // Some row's running max moved: rescale its O^T column (all 4 quarters).
            tc_fence_after();
#pragma unroll 1
            for (int m = 0; m < 4; ++m) {
#pragma unroll 1
              for (int h2 = 0; h2 < 2; ++h2) {
                uint32_t v[32];
                const uint32_t ta = tmem + lane_off + kTmemO + 64 * m + 32 * h2;
                tmem_ld_x32(ta, v);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j)
                  v[j] = __float_as_uint(__uint_as_float(v[j]) * alpha_sh[32 * h2 + j]);
                tmem_st_x32(ta, v);
              }
            }
            tmem_wait_st();
            tc_fence_before();
            named_bar_sync(1, 128);  // alpha_sh is rewritten by the next page
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&p_full));
        }
        if (fail) break;

        // ---------------- epilogue for this piece
        bool bad = !mbar_wait(smem_u32(&o_full), pc & 1, &abort_sh, P.status);
        if (srow) {
          const bool has = row_ok && l > 0.0f;
          inv_l_sh[c] = has ? 1.0f / l : 0.0f;
        }
        if (bar_any(1, 128, bad)) { fail = true; break; }
        tc_fence_after();
        const int nsplit = P.seq_nsplit[b];
        const int split = k - P.seq_first[b];
        const size_t row_base = static_cast<size_t>(b) * TH + tile * kTileRows;
        const size_t part_base =
            nsplit > 1 ? (static_cast<size_t>(P.seq_slot[b] + split) * TH + tile * kTileRows) : 0;
        const int rows_here = min(kTileRows, TH - tile * kTileRows);
#pragma unroll 1
        for (int h2 = 0; h2 < 2; ++h2) {
          float corr[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) corr[j] = 0.0f;
#pragma unroll 1
          for (int m = 0; m < 4; ++m) {
            uint32_t v[32];
            tmem_ld_x32(tmem + lane_off + kTmemO + 64 * m + 32 * h2, v);
            tmem_wait_ld();
            const int lat = 128 * m + 32 * wq + lane;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int cc = 32 * h2 + j;
              if (cc < rows_here) {
                const float val = __uint_as_float(v[j]) * inv_l_sh[cc];
                if (nsplit > 1) {
                  P.opart[(part_base + cc) * kLora + lat] = val;
                } else {
                  const size_t o = (row_base + cc) * kLora + lat;
                  P.olat[o] = __float2bfloat16_rn(val);
                  corr[j] += __bfloat162float(P.qlo[o]) * val;
                }
              }
            }
          }
          if (nsplit <= 1) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              float t = corr[j];
#pragma unroll
              for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
              if (lane == j) corr_sh[wq][32 * h2 + j] = t;
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&o_free));
        named_bar_sync(1, 128);
        if (row_ok) {
          const float lse2 = (l > 0.0f) ? m_used + __log2f(l) : -INFINITY;
          if (nsplit > 1) {
            P.lpart[part_base + c] = lse2 * kLn2;
          } else {
            const float corr_tot = corr_sh[0][c] + corr_sh[1][c] + corr_sh[2][c] + corr_sh[3][c];
            P.lse[row_base + c] = lse2 * kLn2 + P.scale * corr_tot;
          }
        }
        named_bar_sync(1, 128);
        ++pc;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

int decode_tiles(int T, int H) { return (T * H + kTileRows - 1) / kTileRows; }
int decode_q_box_rows(int T, int H) {
  const int r = T * H;
  return r >= kTileRows ? kTileRows : ((r + 7) / 8) * 8;
}

cudaError_t launch_decode(const CUtensorMap& tm_q, const CUtensorMap& tm_c, int grid_ctas,
                          const int32_t* block_table, const int32_t* seq_len_eff,
                          const PlanHeader* header, void* ws, const int32_t* seq_first,
                          const int32_t* seq_nsplit, const int32_t* seq_slot,
                          const __nv_bfloat16* qlo, __nv_bfloat16* olat, float* lse,
                          int32_t* status, int B, int T, int H, int max_pages,
                          int num_pages, float scale, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kDecSmem);
  if (e != cudaSuccess) return e;
  DecodeParams P;
  P.block_table = block_table;
  P.seq_len_eff = seq_len_eff;
  P.header = header;
  P.ws = static_cast<uint8_t*>(ws);
  P.range_b = nullptr;
  P.range_p = nullptr;
  P.seq_first = seq_first;
  P.seq_nsplit = seq_nsplit;
  P.seq_slot = seq_slot;
  P.qlo = qlo;
  P.olat = olat;
  P.lse = lse;
  P.opart = nullptr;
  P.lpart = nullptr;
  P.status = status;
  P.B = B;
  P.T = T;
  P.H = H;
  P.max_pages = max_pages;
  P.num_pages = num_pages;
  P.tiles = decode_tiles(T, H);
  P.q_box_rows = decode_q_box_rows(T, H);
  P.scale = scale;
  P.scale_log2 = scale * 1.4426950408889634f;
  decode_kernel<<<grid_ctas, kDecThreads, kDecSmem, st>>>(tm_q, tm_c, P);
  return cudaGetLastError();
}

}  // namespace mla
