/*
 * mla_decode.h -- C ABI of the GB300 (sm_103a) MLA decode library
 *                 (libmla_decode.so).
 *
 * What it computes
 * ----------------
 * Multi-head Latent Attention decode in the weight-absorbed form without
 * materialised absorbed weights.  Source: vLLM PR #14770 "[Attention] MLA get
 * rid of materialization", PR description.  Instead of precomputing W_Q_UK and
 * W_UV_O, the decode step runs as sequential bf16 matmuls:
 *
 *   1. q-absorb bmm: q_lat[b,t,h] = [ q_nope[b,t,h] . W_UK[h] (512) || q_pe (64) ]
 *   2. latent attention: every head attends MQA-style to the shared latent
 *      cache row c_j = [c_kv (512) || k_pe (64)].  Query t of a T-token block
 *      sees keys [0, L_b - T + t]:
 *        s_j = scale * (q_lat . c_j),   lse = ln sum_j exp(s_j),
 *        o_lat = sum_j exp(s_j - lse) * c_j[0:512]
 *   3. UV bmm: out[b,t,h] = o_lat . W_UV[h] (128)
 *
 * The latent cache is paged with 64-token blocks and stored in BF16
 * ("DeepSeek publica FlashMLA como codigo abierto", feature list: BF16, paged
 * KV cache with block size 64, optimised for variable-length sequences).
 * Split-KV over key ranges and the log-sum-exp merge of the partial results
 * follow the FlashAttention line of work that the same page names as
 * FlashMLA's inspiration.
 *
 * Fixed model dimensions (DeepSeek MLA): qk_nope = 128, qk_rope = 64,
 * kv_lora = 512, v_head = 128, page_size = 64.  Other values are rejected with
 * MLA_DECODE_UNSUPPORTED.
 *
 * Conventions for every entry point
 * ---------------------------------
 * - Pointers are DEVICE pointers owned by the caller (for example PyTorch
 *   tensors), contiguous, 16-byte aligned.  The library keeps no pointer after
 *   a call returns and allocates no device memory: all scratch lives in the
 *   caller's workspace (size from mla_decode_workspace_size).
 * - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   All work is enqueued on it; calls do not synchronise the host, except
 *   mla_decode_check.
 * - Return value: an mla_decode_status.  Codes 1..3 are detected on the host
 *   before anything is enqueued (nothing runs); the whole-run calls check
 *   every argument of all their steps first.  Code 4 reports a failed CUDA
 *   call (tensor-map encoding, launch); for a whole-run call the steps before
 *   the failing one may already be enqueued.  Codes 5..6 are detected by the
 *   kernels, written to the workspace status word and reported by
 *   mla_decode_check; the offending unit of work is skipped or computed on a
 *   substitute page, never trapped.
 * - Thread safety: concurrent calls are safe when each uses its own
 *   workspace.  A plan written into a workspace stays valid for every run with
 *   the same dims and seq_lens contents (one plan serves all layers of a
 *   decode step).
 */
#ifndef MLA_DECODE_H
#define MLA_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int32_t batch;             /* B >= 1: sequences in the decode batch            */
  int32_t q_len;             /* T in 1..8: new query tokens per sequence; query t
                                sees keys [0, seq_len - T + t] (causal block)     */
  int32_t num_heads;         /* H, multiple of 16, 16 <= H <= 128                 */
  int32_t qk_nope;           /* must be 128                                       */
  int32_t qk_rope;           /* must be 64                                        */
  int32_t kv_lora;           /* must be 512                                       */
  int32_t v_head;            /* must be 128                                       */
  int32_t page_size;         /* must be 64                                        */
  int32_t num_pages;         /* pages in the cache pool (>= 1)                    */
  int32_t max_pages_per_seq; /* row length of block_table (>= 1)                  */
} mla_decode_dims;

typedef enum {
  MLA_DECODE_OK = 0,
  MLA_DECODE_INVALID_ARG = 1,       /* null / misaligned pointer, bad dims         */
  MLA_DECODE_UNSUPPORTED = 2,       /* q_len or model dims outside the fixed set   */
  MLA_DECODE_WORKSPACE_TOO_SMALL = 3,
  MLA_DECODE_CUDA_ERROR = 4,        /* a CUDA runtime/driver call failed            */
  MLA_DECODE_DEVICE_BOUNDS = 5,     /* block_table entry outside [0, num_pages) or
                                       seq_len outside [q_len, max_pages_per_seq*64] */
  MLA_DECODE_TIMEOUT = 6            /* a bounded device-side wait gave up           */
} mla_decode_status;

/* Bytes of device workspace needed for `dims` on the current device, with the
 * default number of work ranges (one per resident decode CTA group; when the
 * groups that hold all 64-row tiles of a sequence would leave 3 % or more of
 * the SMs idle, groups hold fewer tiles and the count is the smallest that
 * gives every group the same number of (range, tile set) tasks).
 * The workspace holds the split-KV plan, the absorbed query (step 1 above),
 * the latent output and the partial results of key ranges that the log-sum-exp
 * merge combines ("DeepSeek publica FlashMLA como codigo abierto": FlashMLA's
 * FlashAttention 2/3 lineage; vLLM PR #14770, PR description, for the
 * intermediates of the sequential matmuls).  The pages give no interface; the
 * caller-owned workspace is this library's packaging.
 * Needs a CUDA device (queries its SM count); returns CUDA_ERROR without one.
 * INVALID_ARG for a null `dims` or `bytes`; UNSUPPORTED for dims outside the
 * fixed set.  No device memory is touched. */
int mla_decode_workspace_size(const mla_decode_dims* dims, size_t* bytes);

/* Same, for a plan built with `num_ranges` work ranges (0 = default).  More
 * ranges means more key splits per sequence; used to exercise the split and
 * combine paths.  1 <= num_ranges <= 65536. */
int mla_decode_workspace_size_ex(const mla_decode_dims* dims, int32_t num_ranges,
                                 size_t* bytes);

/* Step a1, the planner.  Reads seq_lens (device int32 [B]) on the device and
 * writes into the workspace: the partition of all (sequence, page) work into
 * equal-cost contiguous ranges, each sequence's split count and its slots for
 * partial results.  Also clears the workspace status word.  No host sync.
 * Source: "DeepSeek publica FlashMLA como codigo abierto", feature list
 * (FlashMLA is built for serving batches whose sequences differ in length);
 * balancing the key ranges of such a batch over the SMs is this planner's
 * reading of that.  Errors: INVALID_ARG (null seq_lens or workspace, workspace not
 * 16-byte aligned), UNSUPPORTED (dims), WORKSPACE_TOO_SMALL, CUDA_ERROR
 * (launch); seq_lens outside [q_len, max_pages_per_seq * 64] are clamped on
 * the device and reported as DEVICE_BOUNDS by mla_decode_check. */
int mla_decode_plan(const mla_decode_dims* dims, const int32_t* seq_lens,
                    void* workspace, size_t workspace_bytes, void* stream);

/* mla_decode_plan with an explicit number of work ranges (0 = default). */
int mla_decode_plan_ex(const mla_decode_dims* dims, const int32_t* seq_lens,
                       int32_t num_ranges, void* workspace, size_t workspace_bytes,
                       void* stream);

/* Steps a2..a5 for one layer, after mla_decode_plan on the same workspace:
 *   q           bf16 [B, T, H, 192]   = [q_nope 128 || q_pe 64], RoPE applied
 *   kv_cache    bf16 [num_pages, 64, 576] = [c_kv 512 || k_pe 64] per token;
 *               rows past a sequence's length in its last page must be finite
 *   block_table int32 [B, max_pages_per_seq]: logical page -> physical page;
 *               entries past ceil(L_b/64) are never read
 *   seq_lens    int32 [B]: tokens in each sequence INCLUDING its T new tokens
 *   w_uk        bf16 [H, 128, 512];  w_uv bf16 [H, 512, 128]
 *   softmax_scale: multiplies q_lat . c_j (e.g. 1/sqrt(192)); must be finite
 *               and > 0, else INVALID_ARG (the attention step takes its
 *               running maximum over unscaled scores)
 *   out         bf16 [B, T, H, 128] (written)
 *   lse         fp32 [B, T, H] (written): natural-log log-sum-exp of the
 *               scaled scores of each query row
 * Enqueues four kernels: absorb, attend, combine, up-project.  For 128 tokens
 * (B*T) or more in more (128-token, head) tiles than the GPU has SMs, the
 * combine kernel merges split sequences only and the up-projection applies
 * the first-order LSE correction of the other rows (it stages their o_lat
 * and q_lo anyway); the result equals that of the four step calls below up
 * to the summation order of that correction (lse within a few ulp; out
 * bitwise). */
int mla_decode_run(const mla_decode_dims* dims, const void* q, const void* kv_cache,
                   const int32_t* block_table, const int32_t* seq_lens, const void* w_uk,
                   const void* w_uv, float softmax_scale, void* out, float* lse,
                   void* workspace, size_t workspace_bytes, void* stream);

/* The four steps of mla_decode_run as separate calls, in this order, on one
 * workspace after mla_decode_plan (for profiling one step at a time; for
 * large batches mla_decode_run moves part of the combine into its
 * up-projection, see above).
 *   absorb:     q, w_uk            -> q_lat (bf16 part, and the residual q_lo
 *                                     as E4M3 of q_lo * 2^10, workspace)
 *   attend:     q_lat, cache, ...  -> o_lat + lse (from the bf16 part of q_lat)
 *                                     for unsplit sequences, partials (o as
 *                                     bf16, lse as fp32) for split ones
 *   combine:    partials           -> o_lat + lse for split sequences; then
 *                                     every row's lse += scale * (q_lo . o_lat),
 *                                     the first-order correction for the bf16
 *                                     rounding of q_lat (lse is final only
 *                                     after this step)
 *   up_project: o_lat, w_uv        -> out
 * attend and combine take the softmax scale and reject one that is not
 * finite and > 0 with INVALID_ARG, as mla_decode_run does.                 */
int mla_decode_absorb(const mla_decode_dims* dims, const void* q, const void* w_uk,
                      void* workspace, size_t workspace_bytes, void* stream);
int mla_decode_attend(const mla_decode_dims* dims, const void* kv_cache,
                      const int32_t* block_table, const int32_t* seq_lens,
                      float softmax_scale, float* lse, void* workspace,
                      size_t workspace_bytes, void* stream);
int mla_decode_combine(const mla_decode_dims* dims, float softmax_scale, float* lse,
                       void* workspace, size_t workspace_bytes, void* stream);
int mla_decode_up_project(const mla_decode_dims* dims, const void* w_uv, void* out,
                          void* workspace, size_t workspace_bytes, void* stream);

/* The same steps with FP8 weights.  vLLM PR #14770 "[Attention] MLA get rid
 * of materialization" (PR description) notes that the absorbed form has no
 * FP8 bmm, so FP8 weights are decompressed to bf16 and the bmm runs in bf16;
 * here the bmm kernels decompress each weight tile as they load it.
 *   w_uk_fp8    uint8 [H, 128, 512]  FP8 E4M3 (4-bit exponent, bias 7, 3-bit
 *               mantissa, no infinities; S.1111.111 is NaN)
 *   w_uk_scale  fp32  [H, 1, 4]      one scale per 128 x 128 block (k, m)
 *   w_uv_fp8    uint8 [H, 512, 128]  FP8 E4M3
 *   w_uv_scale  fp32  [H, 4, 1]
 * The weight used is W = bf16(fp32(w8) * scale): the fp32 product rounded to
 * the nearest bf16 (ties to even).  Pointers as for the bf16 calls; the FP8
 * arrays need 16-byte alignment, the scales 4-byte alignment. */
int mla_decode_run_fp8w(const mla_decode_dims* dims, const void* q, const void* kv_cache,
                        const int32_t* block_table, const int32_t* seq_lens,
                        const uint8_t* w_uk_fp8, const float* w_uk_scale,
                        const uint8_t* w_uv_fp8, const float* w_uv_scale, float softmax_scale,
                        void* out, float* lse, void* workspace, size_t workspace_bytes,
                        void* stream);
int mla_decode_absorb_fp8w(const mla_decode_dims* dims, const void* q, const uint8_t* w_uk_fp8,
                           const float* w_uk_scale, void* workspace, size_t workspace_bytes,
                           void* stream);
int mla_decode_up_project_fp8w(const mla_decode_dims* dims, const uint8_t* w_uv_fp8,
                               const float* w_uv_scale, void* out, void* workspace,
                               size_t workspace_bytes, void* stream);

/* Waits for `stream`, then returns the first device-side status recorded in
 * the workspace since the last plan (OK, DEVICE_BOUNDS or TIMEOUT), or
 * CUDA_ERROR if the stream reports an error.  INVALID_ARG for a null
 * workspace.  The pages have no counterpart: the kernels never trap on a bad
 * block-table entry, a bad sequence length or a wait that gave up; they record
 * it in the workspace and this call reads it back. */
int mla_decode_check(const void* workspace, void* stream);

/* Static English text for a status code. */
const char* mla_decode_status_string(int status);

/* Introspection for tests and profiling: byte offsets inside a workspace
 * planned with `num_ranges` (0 = default) of the intermediate buffers
 *   offsets[0] q_lat  bf16 [B*T*H, 576]   (absorbed query, bf16 part)
 *   offsets[1] q_lo   uint8 [B*T*H, 512]  (residual q_lat - bf16 part, times
 *                                          2^10, as FP8 E4M3 codes)
 *   offsets[2] o_lat  bf16 [B*T*H, 512]   (latent attention output)
 *   offsets[3] plan header (int32 num_ranges, per, total_cost, num_slots)
 * n must be >= 4.  Not needed for normal use. */
int mla_decode_workspace_offsets(const mla_decode_dims* dims, int32_t num_ranges,
                                 int64_t* offsets, int32_t n);

/* Plan + run without a caller-provided workspace, for callers that cannot
 * allocate device memory: for example a custom operator inside a serving
 * engine whose memory pool owns the device and passes an operator only its
 * inputs and outputs, or code running under a stream capture whose mode
 * forbids new allocations.  The pages describing the method have no
 * counterpart to this call; it is a packaging choice of this library.
 *
 * Arguments are those of mla_decode_run minus the workspace, checked the same
 * way (INVALID_ARG, UNSUPPORTED) before anything is enqueued.  Scratch comes
 * from a fixed 32 MiB array in statically allocated device memory, which every
 * GPU that loads the library holds until the process exits; the call makes no
 * allocation of any kind.  If mla_decode_workspace_size(dims) exceeds 32 MiB
 * it returns MLA_DECODE_WORKSPACE_TOO_SMALL and enqueues nothing.  On a
 * 152-SM GB300 that admits up to 32 query rows per sequence (T * H <= 32, e.g.
 * 16 heads with one or two query tokens), up to roughly 130-460 sequences.
 * The first call on each device looks up that device's copy of the array
 * (cudaGetSymbolAddress) in the device's current context; make that first
 * call before any stream capture.  A later call in a different context of the
 * device (after cudaDeviceReset, for example) looks the address up again, so
 * make the first call after a reset before any capture too.  All calls on a device share the one array, which keeps the last
 * call's contents: calls whose work overlaps on the GPU (other streams, other
 * host threads) race and must be serialised by the caller.  Device-side
 * bounds errors are recorded in the shared array but cannot be queried
 * through this entry point; use mla_decode_run with a workspace and
 * mla_decode_check when that matters. */
int mla_decode_run_static_scratch(const mla_decode_dims* dims, const void* q,
                                  const void* kv_cache, const int32_t* block_table,
                                  const int32_t* seq_lens, const void* w_uk,
                                  const void* w_uv, float softmax_scale, void* out,
                                  float* lse, void* stream);

/* Number of kernels one whole run enqueues (launch accounting; the plan is
 * not counted): *kernels = 4 (absorb, attention, combine, up-projection), or
 * 3 when the run (mla_decode_run, or mla_decode_run_fp8w: fp8_weights
 * nonzero; the count is the same) takes the fused combine + up-projection of
 * small batches: fewer than 128 tokens (batch x q_len) whose 16-token tiles
 * of all heads fit in one wave on the device's SMs.  The count depends on the
 * current device's SM count.
 * Returns MLA_DECODE_INVALID_ARG for bad dims or a null `kernels`, before any
 * device query; MLA_DECODE_CUDA_ERROR if the device cannot be queried. */
int mla_decode_kernels_per_run(const mla_decode_dims* d, int32_t fp8_weights, int32_t* kernels);

/* Self-test of failure detection (no counterpart in the method): enqueues one
 * small kernel that waits, through the library's bounded device-side wait, on
 * a barrier that nothing ever completes.  The wait gives up after its limit
 * (about 2 s), writes MLA_DECODE_TIMEOUT into *status (a device int32 that
 * must hold 0 beforehand) and the kernel exits, leaving the context usable.
 * Returns INVALID_ARG for a null or misaligned pointer, CUDA_ERROR if the
 * launch fails, else OK (the status is written asynchronously). */
int mla_decode_selftest_wait_timeout(int32_t* status, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MLA_DECODE_H */
