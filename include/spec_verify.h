/*
 * spec_verify.h - C ABI of the GB300 speculative-decoding verify library.
 *
 * The library implements two steps of MTP/EAGLE-style speculative decoding as
 * described in inclusionAI/AReno PR #550, "feat(engine): MTP training loss
 * and speculative decoding for bailing_v3", section "What does this PR do?"
 * (Phase 2), and table "Per-step optimizations":
 *
 *   spec_verify  - the batched verify sampler: sampler-equivalent target
 *                  distribution (temperature, top-k, top-p), logprobs, exact
 *                  chain rejection sampling against the draft distributions,
 *                  residual or bonus draw by Gumbel-max over a Philox stream,
 *                  per-position acceptance mass alpha = sum_v min(p, q).
 *   spec_commit  - the commit of each row's accepted verify state from the
 *                  stacked (layer-major) verify-state buffer into the
 *                  recurrent/conv cache.
 *
 * Conventions shared by every entry point:
 *   - All array pointers are DEVICE pointers to dense row-major arrays owned
 *     by the caller.  The library allocates no device memory and keeps no
 *     device state between calls.
 *   - `cuda_stream` is a cudaStream_t (NULL = legacy default stream).  Work is
 *     enqueued asynchronously on it; no call synchronises with the host.
 *   - A negative return value is a host-detectable error (bad argument or a
 *     failed launch); nothing has been enqueued when an argument check fails.
 *   - Problems that depend on device data (NaN logits, out-of-range tokens or
 *     indices) never trap: they set bits in the per-row `flags` output.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SPEC_ABI_VERSION 5

/* Largest vocabulary and draft length accepted by spec_verify. */
#define SPEC_MAX_V 524288
#define SPEC_MAX_K 16

/* Logit element types. */
typedef enum { SPEC_F32 = 0, SPEC_BF16 = 1 } spec_dtype_t;

/* Per-row sampling parameters (16 bytes, device array [B]).
 *   temperature: 0 selects greedy decoding; otherwise a positive normal
 *                float.  Any other value sets SPEC_F_BAD_PARAM and the row
 *                is decoded greedily.
 *   top_k:       keep the top_k entries of the total order (larger logit
 *                first, ties by smaller index); <= 0 or >= V disables it.
 *   top_p:       keep the shortest prefix (of what top-k kept, renormalised)
 *                whose mass reaches top_p; 1 disables it; a value outside
 *                (0, 1] sets SPEC_F_BAD_PARAM (greedy).
 *   reserved:    ignored.                                                    */
typedef struct {
  float temperature;
  int32_t top_k;
  float top_p;
  uint32_t reserved;
} spec_params_t;

/* Status codes. */
enum {
  SPEC_OK = 0,
  SPEC_E_NULL = -1,      /* a required pointer is NULL                        */
  SPEC_E_DIM = -2,       /* a size is out of range                            */
  SPEC_E_DTYPE = -3,     /* unknown logits dtype                              */
  SPEC_E_ALIGN = -4,     /* a pointer is not aligned to its element size      */
  SPEC_E_WORKSPACE = -5, /* workspace missing or smaller than required        */
  SPEC_E_CUDA = -6,      /* a CUDA runtime call or kernel launch failed       */
  SPEC_E_ARCH = -7       /* the current device is not an sm_103 GPU           */
};

/* Per-row flag bits written by the device (OR-ed; never a trap). */
enum {
  SPEC_F_MARGIN_ACCEPT = 1,   /* an accept test had |u*q - p| < 1e-6            */
  SPEC_F_MARGIN_DRAW = 2,     /* the best two race scores were within the margin */
  SPEC_F_MARGIN_TOPP = 4,     /* a top-p boundary mass was within 1e-6 of top_p */
  SPEC_F_NAN = 8,             /* NaN/+inf logit, or a position with every logit -inf:
                                 the row is invalid (tokens -1, accept_len 0)   */
  SPEC_F_BAD_TOKEN = 16,      /* a draft token outside [0, V): that draft is rejected */
  SPEC_F_BAD_PARAM = 32,      /* invalid temperature/top_p: row decoded greedily */
  SPEC_F_RESIDUAL_EMPTY = 64, /* max(p - q, 0) was all zero: drew from p instead */
  SPEC_F_BAD_IDX = 128,       /* spec_commit: accept_len or cache slot out of range */
  SPEC_F_TIMEOUT = 256        /* a bounded wait inside the kernel gave up before the
                                 row's inputs were reduced: the row is invalid
                                 (tokens -1, accept_len 0); see the workspace notes */
};

/* Bytes of workspace spec_verify needs for a batch of B rows with k drafts.
 * The workspace must be zero-filled before its first use (for example with
 * cudaMemsetAsync).  Each call numbers itself from a count of the CTAs that
 * entered earlier calls (so every call on one workspace launches the same
 * grid: one workspace belongs to one device), counts in one of two sets of
 * counters in the 256-byte header by the parity of its number, and zeroes
 * the other set for the call after it.  The settles return the per-row
 * tickets and per-(row, position) tile counters to zero as they finish.
 * Every record behind them carries the tag of the call that wrote it (its
 * number + 1, never 0), so stale or foreign contents are never read as this
 * call's.  One workspace serves any number of later calls of the same B, k
 * and V on one stream (re-zero it once every 2^32 - 1 calls, when the tag
 * comes round again, and before a call of another shape, whose counters lie
 * elsewhere); two calls that may run concurrently need two workspaces.
 * Words of the 256-byte header for diagnosis and testing:
 *   bytes 20..23  must stay 0.  They exist to test the waits that give up:
 *                 bit 0 makes the finalize of row 0 wait for records that
 *                 never arrive (the row comes back with SPEC_F_TIMEOUT after
 *                 the wait's bound, a few hundred milliseconds); bit 1 makes
 *                 one CTA reach the first grid barrier of the top-p passes
 *                 1.5 s late, so that the others' wait gives up after about
 *                 a second and every top-p row comes back with
 *                 SPEC_F_TIMEOUT.
 *   bytes 24..27  the counter set (0 or 1) of the last call.
 *   bytes 52..55 (set 0) and 84..87 (set 1)  after a call: bits of the waits
 *                 that gave up in it (1 a tile's wait for its unit's state,
 *                 2 a tile's copy, 4 a settle or finalize wait for records,
 *                 8 the row-order wait of batches above 256 rows, 16 a grid
 *                 barrier of the top-p passes); 0 when every wait ended
 *                 normally.
 *   bytes 236..239  the tag of the last call.                              */
size_t spec_verify_workspace_size(int B, int k, int V);

/* spec_verify - one verify step for B rows of k drafts over a V-entry vocabulary.
 *
 * Source: inclusionAI/AReno PR #550, "What does this PR do?" Phase 2 (one
 * forward verifies k+1 tokens per row; sampler-equivalent target
 * distribution; exact chain rejection sampling; logprobs unchanged) and
 * table "Per-step optimizations" (Gumbel-max draws, one-pass logprobs, no
 * host syncs); table "On-policy accept probability" (alpha = sum min(p, q)).
 *
 * Inputs (device):
 *   logits        [B, k+1, V] of logits_dtype; position j holds the target
 *                 logits that score draft x_j (j < k) or the bonus token (j = k).
 *   draft_probs   [B, k, V] float32 draft distributions q_j, used exactly as
 *                 given.  May be NULL when k == 0.
 *   draft_tokens  [B, k] int32 draft tokens x_j.  May be NULL when k == 0.
 *   params        [B] spec_params_t.
 *   seed          key of the Philox4x32-10 stream.  The accept uniform of
 *                 draft j in row r comes from counter (0, j, R, 0); the race
 *                 uniform of vocabulary entry v at position j from counter
 *                 (v >> 2, j, R, 1), word v & 3; the race uniform of the
 *                 256-entry block b at position j from counter
 *                 (b >> 2, j, R, 2), word b & 3; U = ((w >> 9) + 1/2) * 2^-23.
 *                 R = row_base + r.
 *   row_base      the stream row of this call's row 0.  A batch split into
 *                 blocks of rows (one block per GPU, or per call) draws
 *                 exactly what the whole batch draws in one call when every
 *                 block passes the index of its first row here.
 * Outputs (device), all written for every row:
 *   tokens        [B, k+1] int32: x_0..x_{a-1}, then the drawn token, then -1.
 *   accept_len    [B] int32: a + 1 (accepted drafts plus the drawn token);
 *                 0 for an invalid row.
 *   logprobs      [B, k+1] float32: ln p_j(token) of each emitted token under
 *                 the filtered, temperature-scaled target (under greedy
 *                 decoding the raw log-softmax); 0 after the drawn token.
 *   alpha         [B, k] float32: sum_v min(p_j(v), q_j(v)) for every j.
 *                 May be NULL when k == 0.
 *   flags         [B] uint32: SPEC_F_* bits.  A row with SPEC_F_NAN or
 *                 SPEC_F_TIMEOUT is invalid: tokens -1, accept_len 0,
 *                 logprobs and alpha 0.
 * workspace / workspace_bytes: device scratch of at least
 *   spec_verify_workspace_size(B, k, V) bytes, zero-filled before first use.
 * Errors: SPEC_E_NULL, SPEC_E_DIM (B < 0, k outside [0, SPEC_MAX_K], V outside
 *   [1, SPEC_MAX_V]), SPEC_E_DTYPE, SPEC_E_ALIGN (a pointer not aligned to
 *   its element size), SPEC_E_WORKSPACE, SPEC_E_ARCH, SPEC_E_CUDA.
 * B == 0 returns SPEC_OK without enqueuing work.                             */
int spec_verify(const void* logits, int logits_dtype, const float* draft_probs,
                const int32_t* draft_tokens, const spec_params_t* params, uint64_t seed,
                uint32_t row_base, int B, int k, int V, int32_t* tokens, int32_t* accept_len,
                float* logprobs, float* alpha, uint32_t* flags, void* workspace,
                size_t workspace_bytes, void* cuda_stream);

/* spec_commit - gather each row's accepted verify state into its cache slot.
 *
 * Source: inclusionAI/AReno PR #550, "What does this PR do?" Phase 2 (the
 * recurrent and conv caches of the linear-attention layers are stacked across
 * layers; one verify-state buffer is shared by all graph buckets) and table
 * "Per-step optimizations" ("KDA caches stacked across layers, commit in 4
 * kernels"); "How was it tested?" (state after full and partial commits
 * matches sequential decode).
 *
 * For every layer l and row r with 1 <= accept_len[r] <= S:
 *   cache_rec[l, slot_r]  = verify_rec[l, r, accept_len[r] - 1]
 *   cache_conv[l, slot_r] = verify_conv[l, r, accept_len[r] - 1]
 * where slot_r = cache_slot[r] (or r when cache_slot is NULL).
 *   verify_rec   [L, B, S, H, Dk, Dv] float32   (NULL: no recurrent state)
 *   verify_conv  [L, B, S, W, C] 16-bit (bf16 bits)   (NULL: no conv state)
 *   accept_len   [B] int32, as written by spec_verify; 0 skips the row.
 *   cache_slot   [B] int32 or NULL.
 *   cache_rec    [L, slots, H, Dk, Dv] float32;  cache_conv [L, slots, W, C].
 *   flags        [B] uint32 or NULL: SPEC_F_BAD_IDX is OR-ed in for a row
 *                whose accept_len is outside [0, S] or whose slot is outside
 *                [0, slots); such a row is skipped.  Two rows naming the same
 *                slot race (which one lands is unspecified).
 * Errors: SPEC_E_NULL, SPEC_E_DIM, SPEC_E_ALIGN, SPEC_E_ARCH, SPEC_E_CUDA.  */
int spec_commit(const float* verify_rec, const uint16_t* verify_conv,
                const int32_t* accept_len, const int32_t* cache_slot, float* cache_rec,
                uint16_t* cache_conv, int L, int B, int S, int H, int Dk, int Dv, int W,
                int C, int slots, uint32_t* flags, void* cuda_stream);

/* spec_commit_swap - the zero-copy commit: a fully accepted row trades slot
 * numbers instead of copying its state.
 *
 * Source: InfiniTensor/InfiniLM PR #588, "feat: add mtp draft models for
 * speculative decoding", section 2 item 5 (the verify forward reads the
 * row's committed state slot and writes a scratch state slot; on full
 * accept the two slot numbers are swapped in O(1); on partial accept the
 * accepted position's state is brought into the committed slot -- there by
 * replay, here by a gather from the stacked verify buffer).
 *
 * Layout: of the S = k + 1 states of row r, the first S - 1 are stacked in
 *   verify_rec [L, B, S-1, H, Dk, Dv] float32 / verify_conv [L, B, S-1, W, C]
 *   16-bit, and the last one (after every fed token) is already in cache
 *   slot scratch_slot[r] of cache_rec [L, slots, H, Dk, Dv] / cache_conv
 *   [L, slots, W, C], where the verify forward wrote it.
 *   slot_of_row [B] int32 (in/out): the row's committed slot.
 *   scratch_slot [B] int32 (in/out): the row's scratch slot.
 * For each row r with a = accept_len[r]:
 *   a == S      : slot_of_row[r] and scratch_slot[r] trade values (nothing is copied);
 *   1 <= a < S  : cache[l, slot_of_row[r]] = verify[l, r, a - 1] for every layer l;
 *   a == 0      : nothing.
 * A row with a outside [0, S], a slot outside [0, slots), or equal committed
 * and scratch slots gets SPEC_F_BAD_IDX in flags (if given) and is left
 * alone.  Rows naming the same slot race.  verify_rec / verify_conv may be
 * NULL for a state kind the model does not have, as in spec_commit.
 * Errors: SPEC_E_NULL, SPEC_E_DIM, SPEC_E_ALIGN, SPEC_E_ARCH, SPEC_E_CUDA.  */
int spec_commit_swap(const float* verify_rec, const uint16_t* verify_conv, const int32_t* accept_len,
                     int32_t* slot_of_row, int32_t* scratch_slot, float* cache_rec,
                     uint16_t* cache_conv, int L, int B, int S, int H, int Dk, int Dv, int W, int C,
                     int slots, uint32_t* flags, void* cuda_stream);

/* spec_verify_noalloc - spec_verify for callers that cannot allocate device
 * memory.  The paper has no counterpart: this entry point exists for plugin
 * or custom-op hosts that pass a kernel only its inputs and outputs, for
 * engines whose allocator has reserved all of HBM, and for loops that cannot
 * take the synchronisation of cudaMalloc/cudaFree.
 *
 * Arguments and outputs are those of spec_verify without the workspace: the
 * scratch comes from an array of SPEC_NOALLOC_MAX_WORKSPACE bytes inside the
 * library (a file-scope device array, held on every GPU that loads the
 * library until the process exits).  The call allocates nothing.
 *   - Limit: spec_verify_workspace_size(B, k, V) must not exceed
 *     SPEC_NOALLOC_MAX_WORKSPACE (8 MiB; the workspace takes about 10.5 KB
 *     per (row, position) unit plus 126 bytes per unit per 1024 vocabulary
 *     entries, so at V = 151936 about 282 units fit, e.g. 94 rows at k = 2);
 *     a larger batch returns SPEC_E_WORKSPACE and enqueues nothing.
 *   - Arguments are checked exactly as spec_verify checks them, before
 *     anything is enqueued: a refused call enqueues nothing.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current and keeps it; make
 *     that first call before any stream capture begins.  The kept address
 *     belongs to the device's context at that time: after cudaDeviceReset on
 *     that device it is stale, so do not call this entry point again in the
 *     same process after a device reset.
 *   - Every call clears the part of the array it uses (cudaMemsetAsync on
 *     cuda_stream) before the kernel, because the array keeps the previous
 *     call's contents.
 *   - All calls share the one array: two calls that can overlap on the GPU
 *     (for example on two streams) race and corrupt each other's results;
 *     order them on one stream or use spec_verify with separate workspaces.
 * Errors: those of spec_verify, and SPEC_E_WORKSPACE for a batch beyond the
 * limit.                                                                    */
#define SPEC_NOALLOC_MAX_WORKSPACE (8u << 20)
int spec_verify_noalloc(const void* logits, int logits_dtype, const float* draft_probs,
                        const int32_t* draft_tokens, const spec_params_t* params, uint64_t seed,
                        uint32_t row_base, int B, int k, int V, int32_t* tokens,
                        int32_t* accept_len, float* logprobs, float* alpha, uint32_t* flags,
                        void* cuda_stream);

/* Diagnostic: out[i] = Philox4x32-10(ctr[i], key = (seed mod 2^32, seed >> 32))
 * for i < n, computed by the same device function spec_verify uses.  ctr and
 * out are device arrays of n uint4 (16-byte aligned).  Lets a test compare
 * the device stream with an independent host implementation.                */
int spec_philox4x32_10(const uint32_t* ctr, uint64_t seed, uint32_t* out, int64_t n,
                       void* cuda_stream);

/* Human-readable text for a status code (static storage). */
const char* spec_status_string(int code);

/* spec_verify_commit - spec_verify and spec_commit in one launch.
 *
 * Source: inclusionAI/AReno PR #550, "What does this PR do?" Phase 2 (the
 * verify step decides each row's accept length; the accepted position's
 * recurrent and conv states are then copied into the row's cache slot) and
 * table "Per-step optimizations" (fewer, larger kernels per decode step).
 *
 * Exactly the results of spec_verify(...) followed on the same stream by
 * spec_commit(verify_rec, verify_conv, accept_len, cache_slot, cache_rec,
 * cache_conv, L, B, k + 1, H, Dk, Dv, W, C, slots, flags, stream): the
 * verify outputs, the cache contents and SPEC_F_BAD_IDX in flags.  In the
 * one cooperative launch a row's state is copied as soon as the row is
 * finalized, while other rows are still being verified.
 *   Arguments 1-17: as spec_verify (the workspace is required).
 *   verify_rec, verify_conv, cache_slot, cache_rec, cache_conv, L, H, Dk, Dv,
 *   W, C, slots: as spec_commit, with S = k + 1 states per row; L == 0
 *   verifies only.
 * Errors: those of spec_commit and of spec_verify; every argument is checked
 * before the device is queried, and a refused call enqueues nothing. */
int spec_verify_commit(const void* logits, int logits_dtype, const float* draft_probs,
                       const int32_t* draft_tokens, const spec_params_t* params, uint64_t seed,
                       uint32_t row_base, int B, int k, int V, int32_t* tokens, int32_t* accept_len,
                       float* logprobs, float* alpha, uint32_t* flags, void* workspace,
                       size_t workspace_bytes, const float* verify_rec, const uint16_t* verify_conv,
                       const int32_t* cache_slot, float* cache_rec, uint16_t* cache_conv, int L, int H,
                       int Dk, int Dv, int W, int C, int slots, void* cuda_stream);

/* spec_draft_workspace_size - bytes of device workspace spec_draft_sample
 * needs for B rows over V entries (0 when B < 0 or V < 1); zero-filled
 * before first use, left reusable by every call, as spec_verify's. */
size_t spec_draft_workspace_size(int B, int V);

/* spec_draft_sample - one draft step: sample x_j ~ q_j for B rows and write
 * q_j, the distribution the verify later reads as draft_probs.
 *
 * Source: inclusionAI/AReno PR #550, "What does this PR do?" Phase 2 (the
 * MTP layer drafts EAGLE-style, one position at a time, with the sampler
 * settings of the target); areal-project/AReaL PR #1659 (EAGLE top-k draft
 * tokens passed through to the verify).
 *
 * q_j is the sampler-equivalent distribution of the draft logits: the
 * temperature, top-k, top-p filter and renormalisation of spec_verify's p,
 * with the same total order, parameter rules and invalid-input rules.  x_j
 * is drawn from q_j by spec_verify's two-level exponential race, on Philox
 * streams of their own: the race uniform of entry v from counter
 * (v >> 2, pos, R, 3), word v & 3, and of block b from counter
 * (b >> 2, pos, R, 4), word b & 3, R = row_base + r.  So draft draws and the
 * verify's accept and draw uniforms are independent, and a draft step is
 * reproducible from (seed, row, pos).
 * Inputs (device):
 *   logits        [B, V] of logits_dtype: the draft logits at position pos.
 *   params        [B] spec_params_t (the draft sampler's settings).
 *   seed, row_base: as spec_verify; pos: the draft position (counter word 1).
 * Outputs (device):
 *   q             [B, V] float32: q_j (0 outside the kept set; one-hot at the
 *                 argmax under greedy decoding; all 0 for an invalid row).
 *                 May be NULL: the tokens alone (no second kernel).
 *   tokens        [B] int32: x_j (-1 for an invalid row).
 *   logprobs      [B] float32: ln q_j(x_j) as spec_verify reports a drawn
 *                 token's logprob (the raw log-softmax under greedy decoding).
 *   flags         [B] uint32: SPEC_F_* (NAN, BAD_PARAM, MARGIN_TOPP,
 *                 MARGIN_DRAW, TIMEOUT).
 * workspace / workspace_bytes: at least spec_draft_workspace_size(B, V).
 * Errors: SPEC_E_NULL, SPEC_E_DIM, SPEC_E_DTYPE, SPEC_E_ALIGN,
 *   SPEC_E_WORKSPACE, SPEC_E_ARCH, SPEC_E_CUDA; every argument is checked
 *   before anything is enqueued.  B == 0 returns SPEC_OK. */
int spec_draft_sample(const void* logits, int logits_dtype, const spec_params_t* params, uint64_t seed,
                      uint32_t row_base, uint32_t pos, int B, int V, float* q, int32_t* tokens,
                      float* logprobs, uint32_t* flags, void* workspace, size_t workspace_bytes,
                      void* cuda_stream);

/* SPEC_ABI_VERSION of the loaded library. */
int spec_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
