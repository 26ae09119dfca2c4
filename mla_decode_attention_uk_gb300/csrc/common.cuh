// common.cuh -- constants and workspace layout shared by the host API and the
// kernels of the MLA decode library.
#pragma once
#include <cstddef>
#include <cstdint>
#include <utility>

#include <cuda_runtime.h>

namespace mla {

// Launch with programmatic stream serialisation.  The kernel must call
// griddep_wait() before reading or writing global memory.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}


// DeepSeek MLA dimensions (the only ones supported).
constexpr int kNope = 128;             // q_nope width
constexpr int kRope = 64;              // q_pe / k_pe width
constexpr int kLora = 512;             // latent (kv_lora) width = latent value width
constexpr int kDqk = kLora + kRope;    // 576: latent cache row, absorbed query row
constexpr int kDq = kNope + kRope;     // 192: query row as given
constexpr int kVHead = 128;            // output width per head
constexpr int kPage = 64;              // tokens per cache page
constexpr int kMaxQLen = 8;            // new query tokens per sequence (speculative drafts)

// Decode tiling.
constexpr int kTileRows = 64;          // query rows (t, h) per decode CTA
constexpr int kBoxCols = 64;           // 64 bf16 = 128 B: one 128B-swizzle row
constexpr int kBoxes = kDqk / kBoxCols;        // 9 column boxes per 576-wide row
constexpr int kLatBoxes = kLora / kBoxCols;    // 8 of them hold latent columns
constexpr int kBoxBytes = 64 * 128;            // 64 rows x 128 B

// The residual of the absorbed query, q_lo = q_lat - bf16(q_lat), feeds only
// the first-order LSE correction scale * (q_lo . o_lat).  It is stored as FP8
// E4M3 of q_lo * 2^kQloShift (|q_lo| <= 2^-9 |q_lat|, so the scaled values of
// |q_lat| up to about 200 stay below E4M3's largest finite 448): half the bytes
// of bf16, at a cost of about 1e-4 in the LSE (the tolerance is 1e-3).
constexpr int kQloShift = 10;
constexpr float kQloScale = 1024.0f;          // 2^kQloShift
constexpr float kQloInvScale = 1.0f / 1024.0f;

// Cost of starting a piece of work (loading Q, writing the result), in pages.
constexpr int kPieceCost = 2;

// Device status word values (same numbering as mla_decode_status).
constexpr int MLA_STATUS_OK = 0;
constexpr int MLA_STATUS_BOUNDS = 5;
constexpr int MLA_STATUS_TIMEOUT = 6;

// Bounded waits give up after this long (ns).
constexpr unsigned long long kWaitTimeoutNs = 2000000000ull;

// Plan written by the planner kernel into the workspace.
//   ranges: num_ranges + 1 entries of (b, page) where range k starts;
//           entry num_ranges is (B, 0).
//   per sequence: first range touching it, number of ranges touching it
//           (= its split count) and the base of its partial-result slots
//           (-1 when unsplit).
struct PlanHeader {
  int32_t num_ranges;
  int32_t per;          // cost units per range
  int32_t total_cost;
  int32_t num_slots;    // partial slots in use
};

// Workspace layout.  Everything that depends only on (B, T, H) comes first at
// fixed offsets; the regions sized by the number of work ranges R come last,
// so kernels can locate them from the R the planner recorded in the header.
struct WsLayout {
  size_t status;      // int32 status word (always offset 0)
  size_t header;      // PlanHeader
  size_t seq_first;   // int32 [B]
  size_t seq_nsplit;  // int32 [B]
  size_t seq_slot;    // int32 [B]
  size_t seq_len_eff; // int32 [B]  lengths clamped to [T, max_pages*64]
  size_t prefix;      // int32 [B+1] exclusive prefix of per-sequence cost
  size_t qlat;        // bf16 [B*T*H, 576]  absorbed query, bf16 part
  size_t qlo;         // E4M3 [B*T*H, 512]  absorbed query residual (q_lat - bf16 part) * 2^10
  size_t olat;        // bf16 [B*T*H, 512]  latent attention output
  size_t range_b;     // int32 [R+1]                     (R-dependent from here on)
  size_t range_p;     // int32 [R+1]
  size_t lpart;       // fp32 [slots, T*H]       split partial LSE (natural log)
  size_t opart;       // bf16 [slots, T*H, 512]  split partial outputs (normalised)
  size_t total;
  int32_t num_ranges;
  int32_t max_slots;
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline WsLayout make_layout(int B, int T, int H, int R) {
  WsLayout L{};
  const size_t rows = static_cast<size_t>(B) * T * H;
  const int slots = 2 * R;  // each range has at most two pieces in split sequences
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes, 256); return at; };
  L.status = take(sizeof(int32_t));
  L.header = take(sizeof(PlanHeader));
  L.seq_first = take(sizeof(int32_t) * B);
  L.seq_nsplit = take(sizeof(int32_t) * B);
  L.seq_slot = take(sizeof(int32_t) * B);
  L.seq_len_eff = take(sizeof(int32_t) * B);
  L.prefix = take(sizeof(int32_t) * (B + 1));
  L.qlat = take(rows * kDqk * 2);
  L.qlo = take(rows * kLora);
  L.olat = take(rows * kLora * 2);
  L.range_b = take(sizeof(int32_t) * (R + 1));
  L.range_p = take(sizeof(int32_t) * (R + 1));
  L.lpart = take(static_cast<size_t>(slots) * T * H * 4);
  L.opart = take(static_cast<size_t>(slots) * T * H * kLora * 2);
  L.total = o;
  L.num_ranges = R;
  L.max_slots = slots;
  return L;
}

}  // namespace mla
