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
// GB300 mapping (one CTA = 64 query rows of one sequence at a time, over the
// work ranges it is dealt; see decode_shape for how CTAs are grouped):
//   * Keys stream page by page: the TMA producer gathers a 64-token page as 9
//     boxes of 64 x 64 bf16 (128B swizzle) into a ring of 72 KB slots (two fit
//     next to the query tile), looking the physical page up in the block
//     table.  Slots fill and empty box by box: QK^T starts on a page's first
//     boxes while the rest land, and the next page's boxes load as soon as
//     their release group of the slot is free.  When the query rows of a
//     sequence span several CTAs (tiles), those CTAs stream the same pages at
//     about the same time and the second read of a page is served by L2; they
//     are not coupled (a cluster sharing pages by multicast made every slot
//     refill wait for the slower CTA, which cost more than it saved).
//   * QK^T on tcgen05: S[row, key] = sum_576 Q[row] C[key]; M = 64 rows, N = 64
//     keys, fp32 in TMEM (an M = 64 accumulator puts 16 rows in each 32-lane
//     quarter), two S buffers.  A whole page per MMA keeps the shared-memory
//     reads of the query tile at one pass per 64 keys.
//   * Softmax (warps 4-7, 16 rows each, two threads per row holding the even
//     and odd keys): exp2 with a lazily updated running max (rescale only
//     when the max grows by more than 2^8), P written to shared memory as bf16.
//   * PV on tcgen05, transposed: O^T[latent, row] += C^T[latent, key] P^T[key, row]
//     with the page slot read MN-major as the A operand (M = 128 latent, four
//     MMAs for 512) and N = 64 rows; O^T lives in 256 TMEM columns.  P^T of a
//     page is written into that page's RoPE box (dead once QK^T is done), so
//     every page in flight has its own P^T buffer at no extra shared memory.
//   * Epilogue (warps 4-7): O / l to bf16 o_lat plus lse for unsplit sequences,
//     or bf16 partial outputs (fp32 lse) for split ones.
// Warp roles: 0 TMA producer, 1-2 QK^T issuers (K halves; warp 2 also owns
// TMEM), 3 and 8 PV issuers (latent halves), 4-7 softmax and epilogue.  The
// issuers work from precomputed descriptors, so one MMA costs an add and the
// issue itself.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "ptx.cuh"

namespace mla {

namespace {

constexpr int kDecThreads = 288;                   // 9 warps
constexpr int kChunk = 64;                         // keys per streamed chunk (one page)
constexpr int kChunkBox = kChunk * 128;            // one 64 x 64 bf16 box: 8 KB
constexpr int kSlotBytes = kBoxes * kChunkBox;     // 72 KB
constexpr int kMaxSlots = 4;
constexpr int kSBufs = 2;                          // S buffers, each two 64-column K halves
constexpr int kRopeBox = kBoxes - 1;               // box 8: the 64 RoPE columns, then P^T
constexpr int kFreeGroups = 5;                     // slot release groups (see slot_free)
// Box orders as nibble lists (first box in the lowest nibble).  The producer
// loads boxes in release order: PV blocks 0 and 2, then 1 and 3, then the
// RoPE box (it holds the page's P^T until PV is done).  Each QK^T issuer
// takes its boxes (0-4 / 5-8) in the same order.
constexpr uint64_t kLoadOrder = 0x876325410ull;    // 0, 1, 4, 5, 2, 3, 6, 7, 8
constexpr uint64_t kQkOrder0 = 0x32410ull;         // 0, 1, 4, 2, 3
constexpr uint64_t kQkOrder1 = 0x8765ull;          // 5, 6, 7, 8
__host__ __device__ constexpr int free_group(int box) { return box == kRopeBox ? 4 : box >> 1; }
constexpr int kPrefetchPages = 2;                  // L2 prefetch distance, in pages (at most)
constexpr int kDynSmemMax = 232448 - 2048;         // opt-in limit minus static smem budget
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 256;                   // O^T blocks at 256 + 64 m
constexpr float kRescaleThreshold = 8.0f;          // log2 units
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
  __nv_bfloat16* olat;       // [B*T*H, 512]
  float* lse;                // [B*T*H]
  __nv_bfloat16* opart;      // [slots, T*H, 512]
  float* lpart;              // [slots, T*H]
  int32_t* status;
  int B, T, H, max_pages, num_pages, q_box_rows, num_slots;
  int tpg, sets;             // tiles per CTA group; tile sets per sequence
  int pf_near;               // L2 prefetch one page ahead instead of kPrefetchPages
  float scale, scale_log2;
};

// max(a, b, c) in one instruction.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

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
  __device__ PieceWalker() : b(0), p(0), b1(0), p1(0) {}  // no pieces
  __device__ PieceWalker(const DecodeParams& P, int k)
      : b(P.range_b[k]), p(P.range_p[k]), b1(P.range_b[k + 1]), p1(P.range_p[k + 1]) {}
  // len: the piece's sequence length (seq_len_eff), read on the way.
  __device__ bool next(const DecodeParams& P, int& pb, int& pbeg, int& pend, int& len) {
    while (b < b1 || (b == b1 && p < p1)) {
      const int L = P.seq_len_eff[b];
      const int pages = (L + kPage - 1) / kPage;
      const int e = (b == b1) ? p1 : pages;
      const int cb = b, cp = p;
      b += 1;
      p = 0;
      if (e > cp) {
        pb = cb;
        pbeg = cp;
        pend = e;
        len = L;
        return true;
      }
    }
    return false;
  }
  __device__ bool next(const DecodeParams& P, int& pb, int& pbeg, int& pend) {
    int len;
    return next(P, pb, pbeg, pend, len);
  }
};

// Every piece of a CTA's tasks v = v0, v0 + stride, ... < nv in order (the
// order all roles walk), for a role that wants to find its next piece early.
struct PieceStream {
  int v, stride, nv, sets;
  PieceWalker w;
  __device__ PieceStream(const DecodeParams& P, int v0, int stride_, int nv_, int sets_)
      : v(v0), stride(stride_), nv(nv_), sets(sets_),
        w(v0 < nv_ ? PieceWalker(P, v0 / sets_) : PieceWalker()) {}
  __device__ bool next(const DecodeParams& P, int& task, int& pb, int& pbeg, int& pend,
                       int& len) {
    while (v < nv) {
      if (w.next(P, pb, pbeg, pend, len)) {
        task = v;
        return true;
      }
      v += stride;
      if (v < nv) w = PieceWalker(P, v / sets);
    }
    return false;
  }
};

// Chunks of a piece: one per page; chunk i covers keys key0(i) .. key0(i) + 63.
struct ChunkRange {
  int pbeg, nchunks;
  __device__ ChunkRange(int /*L*/, int pb, int pe) : pbeg(pb), nchunks(pe - pb) {}
  __device__ int page(int i) const { return pbeg + i; }
  __device__ int key0(int i) const { return (pbeg + i) * kPage; }
};

// kSets: a CTA group holds only some of a sequence's tiles (P.sets > 1).
// Without it the task loops below reduce at compile time to one range after
// another for a fixed tile (measured: the general loops cost 0.3 % of the
// attention time on shapes that do not need them).
template <bool kSets>
__global__ void __launch_bounds__(kDecThreads, 1)
decode_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_c,
              DecodeParams P) {
  extern __shared__ uint8_t smem_raw[];
  // Page slots are filled and released box by box: slot_full has one barrier
  // per box, so QK^T starts on the first boxes of a page while the rest are in
  // flight; slot_free has one per release group (latent boxes 2m, 2m+1 after
  // PV block m; the RoPE box, which holds the page's P^T once QK^T is done,
  // after both PV issuers), so the next page's boxes start loading as soon as
  // their group is free.  p_full / p_free (P^T written / PV done) follow the
  // slot of the page.
  __shared__ __align__(8) uint64_t q_full, q_free, slot_full[kMaxSlots][kBoxes],
      slot_free[kMaxSlots][kFreeGroups],
      s_full[kSBufs], s_free[kSBufs], p_full[kMaxSlots], p_free[kMaxSlots], o_full, o_free,
      drain_bar[4];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  __shared__ float alpha_sh[64];
  __shared__ __align__(16) float inv_l_sh[64];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Work: tasks v = (range k, tile set), v = k * sets + set, dealt round
  // robin to the CTA groups; a group's CTA ti takes tile set * tpg + ti.
  // Consecutive groups hold the tile sets of one range, so all tiles of a
  // range stream its pages at about the same time (the repeats come from
  // L2).  When the tiles of a sequence divide the SM count, sets = 1 and a
  // group holds every tile of its ranges.
  const int tpg = P.tpg;
  const int sets = kSets ? P.sets : 1;
  const int ti = blockIdx.x % tpg;
  const int gi = blockIdx.x / tpg;
  const int NG = gridDim.x / tpg;
  const int TH = P.T * P.H;
  const int NS = P.num_slots;
  const uint32_t q_box_bytes = static_cast<uint32_t>(P.q_box_rows) * 128u;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sQ = sbase;
  const uint32_t sSlot0 = sQ + kBoxes * q_box_bytes;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&q_full), 1);
    mbar_init(smem_u32(&q_free), 2);
    for (int i = 0; i < NS; ++i) {
      for (int j = 0; j < kBoxes; ++j) mbar_init(smem_u32(&slot_full[i][j]), 1);
      for (int r = 0; r < kFreeGroups; ++r)
        mbar_init(smem_u32(&slot_free[i][r]), r == free_group(kRopeBox) ? 2 : 1);
    }
    for (int i = 0; i < kSBufs; ++i) {
      mbar_init(smem_u32(&s_full[i]), 2);
      mbar_init(smem_u32(&s_free[i]), 4);
    }
    for (int i = 0; i < NS; ++i) {
      mbar_init(smem_u32(&p_full[i]), 1);
      mbar_init(smem_u32(&p_free[i]), 2);
    }
    mbar_init(smem_u32(&o_full), 2);
    mbar_init(smem_u32(&o_free), 4);
    for (int i = 0; i < 4; ++i) mbar_init(smem_u32(&drain_bar[i]), 1);
    abort_sh = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_c);
  }
  // Everything above overlaps the previous step's tail.  The plan, q_lat and
  // (on this SM) the tensor memory of the absorb step are only safe to use
  // once it has completed.
  griddep_wait();
  griddep_launch_dependents();
  const int R = P.header->num_ranges;
  {
    const WsLayout L = make_layout(P.B, P.T, P.H, R);
    P.range_b = reinterpret_cast<const int32_t*>(P.ws + L.range_b);
    P.range_p = reinterpret_cast<const int32_t*>(P.ws + L.range_p);
    P.lpart = reinterpret_cast<float*>(P.ws + L.lpart);
    P.opart = reinterpret_cast<__nv_bfloat16*>(P.ws + L.opart);
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
      const uint32_t q_bytes = q_box_bytes * kBoxes;
      int g = 0, pc = 0, nq = 0;  // nq: query-tile copies issued
      bool ok = true;
      for (int v = gi; v < R * sets && ok; v += NG) {
        const int k = v / sets, tile = (v % sets) * tpg + ti;
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
            tma_load_2d(sQ + j * q_box_bytes, &tm_q, j * kBoxCols, qrow, smem_u32(&q_full));
          ++nq;
          const ChunkRange cr(P.seq_len_eff[b], pb, pe);
          const int32_t* bt_row = P.block_table + static_cast<size_t>(b) * P.max_pages;
          // Pages are also prefetched into L2 ahead of their shared-memory
          // load, so a slot refill mostly hits L2 instead of waiting a full
          // HBM round trip: kPrefetchPages ahead, or one page when a
          // sequence's rows fit one CTA (P.pf_near; each page is then read
          // by one CTA only, and the nearer prefetch measured 1.9 % faster on
          // 16 heads, the farther one 0.2-0.6 % faster where two or more
          // tiles share each page).
          auto page_of = [&](int i) {
            int pg = __ldg(bt_row + cr.page(i));
            if (pg < 0 || pg >= P.num_pages) {
              atomicCAS(P.status, 0, MLA_STATUS_BOUNDS);
              pg = 0;
            }
            return pg;
          };
          // Block-table entries are read kLookAhead pages early so the
          // dependent global load stays off the slot-refill path.
          constexpr int kLookAhead = kPrefetchPages > 0 ? kPrefetchPages : 1;
          int ahead[kLookAhead];
#pragma unroll
          for (int a = 0; a < kLookAhead; ++a) {
            ahead[a] = a < cr.nchunks ? page_of(a) : 0;
            if (kPrefetchPages > 0 && a < cr.nchunks && (a == 0 || !P.pf_near))
              for (int j = 0; j < kBoxes; ++j)
                tma_prefetch_l2_2d(&tm_c, j * kBoxCols, ahead[a] * kPage);
          }
          for (int i = 0; i < cr.nchunks; ++i, ++g) {
            const int s = g % NS, u = g / NS;
            const int row = ahead[0] * kPage;
            const uint32_t dst = sSlot0 + s * kSlotBytes;
            // Each box is loaded as soon as its release group of the slot's
            // previous page is free.
            int t = 0;
            for (int prev = -1; t < kBoxes; ++t) {
              const int j = static_cast<int>((kLoadOrder >> (4 * t)) & 15);
              const int grp = free_group(j);
              if (u > 0 && grp != prev) {
                if (!mbar_wait(smem_u32(&slot_free[s][grp]), (u - 1) & 1, &abort_sh, P.status)) {
                  ok = false;
                  break;
                }
                prev = grp;
              }
              const uint32_t fb = smem_u32(&slot_full[s][j]);
              mbar_expect_tx(fb, kChunkBox);
              tma_load_2d(dst + j * kChunkBox, &tm_c, j * kBoxCols, row, fb);
            }
            if (!ok) {
              // Boxes of this page already in flight land before the CTA exits.
              for (int t2 = 0; t2 < t; ++t2)
                mbar_wait_drain(smem_u32(&slot_full[s][(kLoadOrder >> (4 * t2)) & 15]), u & 1,
                                P.status);
              break;
            }
            // Shift the look-ahead window and fetch (and L2-prefetch) the page
            // kLookAhead chunks ahead.
#pragma unroll
            for (int a = 0; a + 1 < kLookAhead; ++a) ahead[a] = ahead[a + 1];
            const int nxt = i + kLookAhead;
            ahead[kLookAhead - 1] = nxt < cr.nchunks ? page_of(nxt) : 0;
            // The page to prefetch: i + kLookAhead, or i + 1 (near).
            const int pf = P.pf_near ? i + 1 : nxt;
            if (kPrefetchPages > 0 && pf < cr.nchunks)
              for (int j = 0; j < kBoxes; ++j)
                tma_prefetch_l2_2d(&tm_c, j * kBoxCols,
                                   (P.pf_near ? ahead[0] : ahead[kLookAhead - 1]) * kPage);
          }
          ++pc;
        }
      }
      // After an abort the consumers may not have waited for every copy this
      // thread started; wait (bounded) for the last query tile and the last
      // page copy into each slot so that no copy lands after the CTA has exited.
      if (nq > 0) mbar_wait_drain(smem_u32(&q_full), (nq - 1) & 1, P.status);
      for (int s = 0; s < NS; ++s) {
        const int n = (g - s + NS - 1) / NS;  // copies issued into slot s
        if (n > 0)
          for (int j = 0; j < kBoxes; ++j)
            mbar_wait_drain(smem_u32(&slot_full[s][j]), (n - 1) & 1, P.status);
      }
    }
  }
  if ((warp >= 1 && warp <= 3) || warp == 8) {
    // ------------------------------------------------------------ MMA issuers
    // One issuing thread cannot keep the tensor pipe busy (each MMA costs it
    // ~50 cycles), so every page's MMAs are spread over four issuers whose
    // MMAs overlap: warps 1 and 2 issue the two K halves of QK^T into two
    // accumulators (the softmax adds them), warps 3 and 8 issue PV for latent
    // blocks 0-1 and 2-3 as soon as the softmax has written P.  Each issuer
    // commits its own MMAs, so the barriers they signal count two arrivals.
    if (elect_one()) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(64, kChunk, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(128, 64, true, false);
      // Descriptors differ only in the start-address field (bits 0-13, in
      // 16-byte units), so each MMA adds a small constant to a base.
      const uint64_t dq0 = sdesc_sw128(sQ, 16, 1024);
      const uint64_t dslot0 = sdesc_sw128(sSlot0, 16, 1024);
      const uint64_t dpv0 = sdesc_sw128(sSlot0, kChunkBox, 1024);
      const uint32_t qbox16 = q_box_bytes >> 4;
      const bool is_qk = warp == 1 || warp == 2;
      const int half = (warp == 1 || warp == 3) ? 0 : 1;  // K half (QK) / latent half (PV)
      const uint64_t qk_order = half == 0 ? kQkOrder0 : kQkOrder1;  // QK boxes
      const int qk_boxes = half == 0 ? 5 : 4;
      int g = 0, pc = 0;
      bool ok = true;
      for (int v = gi; v < R * sets && ok; v += NG) {
        PieceWalker w(P, v / sets);
        int b, pb, pe;
        while (ok && w.next(P, b, pb, pe)) {
          const ChunkRange cr(P.seq_len_eff[b], pb, pe);
          const int nc = cr.nchunks;
          if (is_qk) {
            if (!mbar_wait(smem_u32(&q_full), pc & 1, &abort_sh, P.status)) { ok = false; break; }
            for (int i = 0; i < nc; ++i, ++g) {
              const int s = g % NS, sb = g % kSBufs;
              if (g >= kSBufs && !mbar_wait(smem_u32(&s_free[sb]), ((g / kSBufs) - 1) & 1,
                                            &abort_sh, P.status)) {
                ok = false;
                break;
              }
              const uint64_t bd0 = dslot0 + static_cast<uint64_t>((s * kSlotBytes) >> 4);
              const uint32_t d = tmem + 128 * sb + 64 * half;
              for (int t = 0; t < qk_boxes && ok; ++t) {
                // Each box's MMAs go out as soon as that box has landed.
                const int j = static_cast<int>((qk_order >> (4 * t)) & 15);
                if (!mbar_wait(smem_u32(&slot_full[s][j]), (g / NS) & 1, &abort_sh, P.status)) {
                  ok = false;
                  break;
                }
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                  umma_bf16(d, dq0 + (j * qbox16 + kk * 2), bd0 + ((j * kChunkBox) >> 4) + kk * 2,
                            idesc_qk, (t != 0) || (kk != 0));
                }
              }
              if (!ok) break;
              umma_commit(smem_u32(&s_full[sb]));
            }
            if (!ok) break;
            // Both QK issuers release the query tile (count 2) once their
            // MMAs of this piece have finished reading it.
            umma_commit(smem_u32(&q_free));
          } else {
            for (int i = 0; i < nc; ++i, ++g) {
              const int s = g % NS;
              const bool first = i == 0;
              if (!mbar_wait(smem_u32(&p_full[s]), (g / NS) & 1, &abort_sh, P.status) ||
                  (first && pc > 0 &&
                   !mbar_wait(smem_u32(&o_free), (pc - 1) & 1, &abort_sh, P.status))) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint64_t ad0 = dpv0 + static_cast<uint64_t>((s * kSlotBytes) >> 4);
              // P^T of this page sits in its slot's RoPE box.
              const uint64_t bd0 =
                  dslot0 + static_cast<uint64_t>((s * kSlotBytes + kRopeBox * kChunkBox) >> 4);
#pragma unroll
              for (int m = 2 * half; m < 2 * half + 2; ++m) {
#pragma unroll
                for (int kk = 0; kk < kChunk / 16; ++kk) {
                  umma_bf16(tmem + kTmemO + 64 * m, ad0 + ((2 * m * kChunkBox + kk * 2048) >> 4),
                            bd0 + kk * 2, idesc_pv, !(first && kk == 0));
                }
                umma_commit(smem_u32(&slot_free[s][m]));  // latent boxes 2m, 2m+1
              }
              umma_commit(smem_u32(&slot_free[s][free_group(kRopeBox)]));  // P^T read
              umma_commit(smem_u32(&p_free[s]));
            }
            if (!ok) break;
            umma_commit(smem_u32(&o_full));
          }
          if (!ok) break;
          ++pc;
        }
      }
      // Drain this issuer's MMAs before TMEM is released.
      const uint32_t db = smem_u32(&drain_bar[warp == 8 ? 3 : warp - 1]);
      umma_commit(db);
      mbar_wait_drain(db, 0, P.status);
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ softmax + epilogue
    const int wq = warp - 4;                    // TMEM lane quarter
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    // Softmax ownership (M = 64 accumulator, 16x64b loads): this thread holds
    // row `srow_c` of the tile, keys of parity `par`; par 0 writes row results.
    const int rig = (lane >> 2) + 8 * (lane & 1);
    const int par = (lane >> 1) & 1;
    const int srow_c = 16 * wq + rig;
    const bool owner = par == 0;
    int g = 0, pc = 0;
    bool fail = false;
    // The next piece (and its sequence length) is found before the epilogue
    // of the current one waits for the last PV, so those dependent global
    // loads are off the path from the epilogue to the next piece's first
    // softmax.
    PieceStream ps(P, gi, NG, R * sets, sets);
    int task, b, pb, pe, L;
    bool have = ps.next(P, task, b, pb, pe, L);
    while (!fail && have) {
      {
        const int k = task / sets, tile = (task % sets) * tpg + ti;
        const int r = tile * kTileRows + srow_c;  // row within the sequence's T*H rows
        const bool row_ok = r < TH;
        // The epilogue's bookkeeping is loaded now, so that its memory round
        // trip is not on the path from the piece's last PV to the next
        // piece's first softmax.
        const int nsplit = P.seq_nsplit[b];
        const int split = k - P.seq_first[b];
        const int slot = P.seq_slot[b];
        const int n_row = row_ok ? L - P.T + r / P.H + 1 : 0;
        float m_used = -INFINITY, l = 0.0f;     // l: this thread's half of the row sum
        const ChunkRange cr(L, pb, pe);
        const int nc = cr.nchunks;
        for (int i = 0; i < nc; ++i, ++g) {
          const int sb = g % kSBufs;
          bool need = false;
          bool bad = !mbar_wait(smem_u32(&s_full[sb]), (g / kSBufs) & 1, &abort_sh, P.status);
          bad = __any_sync(0xffffffffu, bad);  // tcgen05.ld below is warp-collective
          uint32_t v[kChunk / 2];
          if (!bad) {
            tc_fence_after();
            uint32_t v2[kChunk / 2];
            tmem_ld_16x64b_x32(tmem + lane_off + 128 * sb, v);
            tmem_ld_16x64b_x32(tmem + lane_off + 128 * sb + 64, v2);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < kChunk / 2; ++j)
              v[j] = __float_as_uint(__uint_as_float(v[j]) + __uint_as_float(v2[j]));
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&s_free[sb]));
          if (!bad) {
            const int kb = cr.key0(i) + par;    // key of v[0]; v[j] is key kb + 2 j
            // Max over raw scores (scale > 0), masking only on a sequence's
            // last page; then p = 2^(s * scale * log2 e - m) with one FFMA.
            if (kb + 2 * (kChunk / 2 - 1) >= n_row) {
#pragma unroll
              for (int j = 0; j < kChunk / 2; ++j)
                if (kb + 2 * j >= n_row) v[j] = __float_as_uint(-INFINITY);
            }
            // Tree reduction with three-input maxima: 16 instructions, four
            // deep (two-input: 31, six deep).
            float a3[11];
#pragma unroll
            for (int t3 = 0; t3 < 10; ++t3)
              a3[t3] = fmax3(__uint_as_float(v[3 * t3]), __uint_as_float(v[3 * t3 + 1]),
                             __uint_as_float(v[3 * t3 + 2]));
            a3[10] = fmaxf(__uint_as_float(v[30]), __uint_as_float(v[31]));
            const float b0 = fmax3(a3[0], a3[1], a3[2]), b1 = fmax3(a3[3], a3[4], a3[5]),
                        b2 = fmax3(a3[6], a3[7], a3[8]), b3 = fmaxf(a3[9], a3[10]);
            float vmax = fmaxf(fmax3(b0, b1, b2), b3);
            vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, 2));
            const float pmax = vmax * P.scale_log2;
            float alpha = 1.0f;
            if (pmax > m_used + kRescaleThreshold) {
              alpha = (m_used == -INFINITY) ? 0.0f : ex2_approx(m_used - pmax);
              m_used = pmax;
              need = i > 0;
            }
            float p[kChunk / 2];
            float sum = 0.0f;
            if (m_used == -INFINITY) {
#pragma unroll
              for (int j = 0; j < kChunk / 2; ++j) p[j] = 0.0f;
            } else {
              const float neg_m = -m_used;
              float sm[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
              for (int j = 0; j < kChunk / 2; ++j) {
                p[j] = ex2_approx(fmaf(__uint_as_float(v[j]), P.scale_log2, neg_m));
                sm[j & 3] += p[j];
              }
              sum = (sm[0] + sm[1]) + (sm[2] + sm[3]);
            }
            l = l * alpha + sum;
            if (owner) alpha_sh[srow_c] = alpha;
            // Pair up neighbouring keys: the even-key thread writes keys 0..31
            // of the chunk, the odd-key thread keys 32..63.  The values cross
            // to the partner already rounded to bf16, two per shuffle (8
            // shuffles instead of 16: the shuffles queue behind the tensor
            // core's shared-memory reads), and byte permutes form the pairs.
            uint32_t packed[16];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              // Sent: p[2k], p[2k+1] (odd thread) or p[16+2k], p[16+2k+1]
              // (even thread); kept: the other half.
              const uint32_t first = pack_bf16x2(p[2 * k], p[2 * k + 1]);
              const uint32_t second = pack_bf16x2(p[16 + 2 * k], p[16 + 2 * k + 1]);
              const uint32_t send2 = par ? first : second;
              const uint32_t own2 = par ? second : first;
              const uint32_t recv2 = __shfl_xor_sync(0xffffffffu, send2, 2);
              // Even thread: (own key, partner key); odd thread: (partner,
              // own).  Low halves give pair 2k, high halves pair 2k + 1.
              const uint32_t lo_a = par ? recv2 : own2, lo_b = par ? own2 : recv2;
              packed[2 * k] = __byte_perm(lo_a, lo_b, 0x5410);
              packed[2 * k + 1] = __byte_perm(lo_a, lo_b, 0x7632);
            }
            // P^T goes into the page's RoPE box: QK^T, its only reader, is
            // complete (S is), and the box is not refilled before PV is done.
            // A quarter-warp's stores cover rows r and r + 8, whose swizzled
            // chunk positions coincide; the thread of row r + 8 writes its
            // four chunks in the order 2, 3, 0, 1, so each quarter-warp
            // store hits eight distinct positions (no bank conflict; measured
            // 1.5 % of the attention time).
            if (!bad) {
              const uint32_t rowaddr =
                  sSlot0 + (g % NS) * kSlotBytes + kRopeBox * kChunkBox + srow_c * 128;
              const bool hi8 = (srow_c >> 3) & 1;
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const int qq = hi8 ? (q ^ 2) : q;
                st_shared_v4(rowaddr + (((4 * par + qq) ^ (srow_c & 7)) << 4),
                             hi8 ? packed[4 * (q ^ 2)] : packed[4 * q],
                             hi8 ? packed[4 * (q ^ 2) + 1] : packed[4 * q + 1],
                             hi8 ? packed[4 * (q ^ 2) + 2] : packed[4 * q + 2],
                             hi8 ? packed[4 * (q ^ 2) + 3] : packed[4 * q + 3]);
              }
              fence_proxy_async_smem();
            }
          }
          // One barrier per chunk: a timeout anywhere or a rescale request.
          if (bar_any(1, 128, bad || need)) {
            // Some row's running max moved: rescale its O^T column (all 4
            // quarters) once the previous chunk's PV has landed.
            bool f = *static_cast<volatile int*>(&abort_sh) != 0;
            if (!f && g >= 1 &&
                !mbar_wait(smem_u32(&p_free[(g - 1) % NS]), ((g - 1) / NS) & 1, &abort_sh,
                           P.status))
              f = true;
            if (bar_any(1, 128, f)) { fail = true; break; }
            tc_fence_after();
#pragma unroll 1
            for (int m = 0; m < 4; ++m) {
#pragma unroll 1
              for (int h2 = 0; h2 < 2; ++h2) {
                uint32_t vv[32];
                const uint32_t ta = tmem + lane_off + kTmemO + 64 * m + 32 * h2;
                tmem_ld_x32(ta, vv);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j)
                  vv[j] = __float_as_uint(__uint_as_float(vv[j]) * alpha_sh[32 * h2 + j]);
                tmem_st_x32(ta, vv);
              }
            }
            tmem_wait_st();
            tc_fence_before();
            named_bar_sync(1, 128);  // alpha_sh is rewritten by the next chunk
          }
          // The barrier above ordered all four warps' P^T writes (and any
          // rescale) before this point: one arrival releases the PV issuers.
          if (threadIdx.x == 128) mbar_arrive(smem_u32(&p_full[g % NS]));
        }
        if (fail) break;
        const int cur_b = b;
        have = ps.next(P, task, b, pb, pe, L);

        // ---------------- epilogue for this piece
        bool bad = !mbar_wait(smem_u32(&o_full), pc & 1, &abort_sh, P.status);
        l += __shfl_xor_sync(0xffffffffu, l, 2);  // even + odd halves of the row sum
        if (owner) inv_l_sh[srow_c] = (row_ok && l > 0.0f) ? 1.0f / l : 0.0f;
        if (bar_any(1, 128, bad)) { fail = true; break; }
        tc_fence_after();
        const size_t row_base = static_cast<size_t>(cur_b) * TH + tile * kTileRows;
        const size_t part_base =
            nsplit > 1 ? (static_cast<size_t>(slot + split) * TH + tile * kTileRows) : 0;
        const int rows_here = min(kTileRows, TH - tile * kTileRows);
        // Row halves outer, latent blocks inner: each thread keeps the 32
        // reciprocals of its half in registers, so the stores (one row each,
        // coalesced over the warp's 32 latent columns) do not wait on
        // shared-memory loads.
#pragma unroll 1
        for (int h2 = 0; h2 < 2 && 32 * h2 < rows_here; ++h2) {  // skip empty row halves
          float il[32];
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            const float4 x = *reinterpret_cast<const float4*>(&inv_l_sh[32 * h2 + j]);
            il[j] = x.x;
            il[j + 1] = x.y;
            il[j + 2] = x.z;
            il[j + 3] = x.w;
          }
          const int nrow = min(32, rows_here - 32 * h2);
#pragma unroll 1
          for (int m = 0; m < 4; ++m) {
            const int lat = 128 * m + 32 * wq + lane;
            uint32_t v[32];
            tmem_ld_x32(tmem + lane_off + kTmemO + 64 * m + 32 * h2, v);
            tmem_wait_ld();
            // bf16 either way: o_lat of an unsplit sequence, or the partial
            // output of a split one (the merge rounds to bf16 again; bf16
            // partials halve the bytes of the split rows' round trip).
            __nv_bfloat16* dst = (nsplit > 1 ? P.opart : P.olat) +
                                 ((nsplit > 1 ? part_base : row_base) + 32 * h2) * kLora + lat;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j < nrow) dst[j * kLora] = __float2bfloat16_rn(__uint_as_float(v[j]) * il[j]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&o_free));
        named_bar_sync(1, 128);
        if (owner && row_ok) {
          // Natural-log LSE of this key range; the combine step adds the
          // first-order correction for the bf16 rounding of the query.
          const float lse2 = (l > 0.0f) ? m_used + __log2f(l) : -INFINITY;
          if (nsplit > 1)
            P.lpart[part_base + srow_c] = lse2 * kLn2;
          else
            P.lse[row_base + srow_c] = lse2 * kLn2;
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
// Page slots that fit next to the query tile.
int decode_num_slots(int T, int H) {
  const int q_bytes = kBoxes * decode_q_box_rows(T, H) * 128;
  int ns = (kDynSmemMax - 1024 - q_bytes) / kSlotBytes;
  return ns > kMaxSlots ? kMaxSlots : ns;
}
int decode_smem_bytes(int T, int H) {
  return 1024 + kBoxes * decode_q_box_rows(T, H) * 128 + decode_num_slots(T, H) * kSlotBytes;
}
// How the attention step spreads over the SMs.  One CTA per SM and per
// 64-row tile of a sequence's query rows.  When the tiles divide the SM
// count, a CTA group holds all of them and there is one work range per group.
// When they do not and the groups that fit would leave 3 % or more of the SMs
// idle (16 tiles on 152 SMs: 9 groups, 8 SMs idle), a group holds
// tpg = gcd(tiles, SMs) tiles instead, every SM gets a CTA, and the number of
// ranges is the smallest that deals each group the same number of
// (range, tile set) tasks.
struct DecodeShape {
  int tiles, tpg, sets, groups, ranges;
};
static int gcd_int(int a, int b) {
  while (b) {
    const int t = a % b;
    a = b;
    b = t;
  }
  return a;
}
static DecodeShape decode_shape(int T, int H, int sm_count) {
  DecodeShape d;
  d.tiles = decode_tiles(T, H);
  const int sms = sm_count > 0 ? sm_count : 1;
  const int idle = d.tiles <= sms ? sms % d.tiles : 0;
  d.tpg = (100 * idle >= 3 * sms) ? gcd_int(d.tiles, sms) : d.tiles;
  d.sets = d.tiles / d.tpg;
  d.groups = sms / d.tpg > 0 ? sms / d.tpg : 1;
  d.ranges = d.groups / gcd_int(d.groups, d.sets);
  return d;
}

// Default number of work ranges for the planner (see decode_shape).
cudaError_t decode_default_ranges(int T, int H, int sm_count, int* ranges) {
  const DecodeShape shape = decode_shape(T, H, sm_count);
  cudaError_t e = cudaFuncSetAttribute(
      shape.sets > 1 ? decode_kernel<true> : decode_kernel<false>,
      cudaFuncAttributeMaxDynamicSharedMemorySize, decode_smem_bytes(T, H));
  if (e != cudaSuccess) return e;
  *ranges = shape.ranges;
  return cudaSuccess;
}

cudaError_t launch_decode(const CUtensorMap& tm_q, const CUtensorMap& tm_c, int sm_count,
                          const int32_t* block_table, const int32_t* seq_len_eff,
                          const PlanHeader* header, void* ws, const int32_t* seq_first,
                          const int32_t* seq_nsplit, const int32_t* seq_slot,
                          __nv_bfloat16* olat, float* lse,
                          int32_t* status, int B, int T, int H, int max_pages,
                          int num_pages, float scale, cudaStream_t st) {
  const int smem = decode_smem_bytes(T, H);
  const DecodeShape shape = decode_shape(T, H, sm_count);
  auto kern = shape.sets > 1 ? decode_kernel<true> : decode_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
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
  P.tpg = shape.tpg;
  P.sets = shape.sets;
  P.pf_near = shape.tiles == 1 ? 1 : 0;
  P.q_box_rows = decode_q_box_rows(T, H);
  P.num_slots = decode_num_slots(T, H);
  P.scale = scale;
  P.scale_log2 = scale * 1.4426950408889634f;

  e = launch_pdl(kern, dim3(shape.groups * shape.tpg), dim3(kDecThreads), smem, st,
                 tm_q, tm_c, P);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace mla
