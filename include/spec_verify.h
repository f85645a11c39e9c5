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

#define SPEC_ABI_VERSION 1

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
  SPEC_F_BAD_IDX = 128        /* spec_commit: accept_len or cache slot out of range */
};

/* Bytes of workspace spec_verify needs for a batch of B rows with k drafts.
 * The workspace must be zero-filled before its first use (for example with
 * cudaMemsetAsync).  Every completed spec_verify call returns the words that
 * must start at zero (the counters at the start of the 256-byte header and
 * one ticket per row) to zero and advances an epoch word in the header;
 * every record behind them carries the epoch of the call that wrote it, so
 * stale or foreign contents are never read as this call's.  One workspace
 * serves any number of later calls on one stream; two calls that may run
 * concurrently need two workspaces.                                         */
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
 *                 draft j in row r comes from counter (0, j, r, 0); the race
 *                 uniform of vocabulary entry v at position j from counter
 *                 (v >> 2, j, r, 1), word v & 3; U = ((w >> 9) + 1/2) * 2^-23.
 * Outputs (device), all written for every row:
 *   tokens        [B, k+1] int32: x_0..x_{a-1}, then the drawn token, then -1.
 *   accept_len    [B] int32: a + 1 (accepted drafts plus the drawn token);
 *                 0 for an invalid row.
 *   logprobs      [B, k+1] float32: ln p_j(token) of each emitted token under
 *                 the filtered, temperature-scaled target (under greedy
 *                 decoding the raw log-softmax); 0 after the drawn token.
 *   alpha         [B, k] float32: sum_v min(p_j(v), q_j(v)) for every j.
 *                 May be NULL when k == 0.
 *   flags         [B] uint32: SPEC_F_* bits.
 * workspace / workspace_bytes: device scratch of at least
 *   spec_verify_workspace_size(B, k, V) bytes, zero-filled before first use.
 * Errors: SPEC_E_NULL, SPEC_E_DIM (B < 0, k outside [0, SPEC_MAX_K], V outside
 *   [1, SPEC_MAX_V]), SPEC_E_DTYPE, SPEC_E_ALIGN (a pointer not aligned to
 *   its element size), SPEC_E_WORKSPACE, SPEC_E_ARCH, SPEC_E_CUDA.
 * B == 0 returns SPEC_OK without enqueuing work.                             */
int spec_verify(const void* logits, int logits_dtype, const float* draft_probs,
                const int32_t* draft_tokens, const spec_params_t* params, uint64_t seed,
                int B, int k, int V, int32_t* tokens, int32_t* accept_len, float* logprobs,
                float* alpha, uint32_t* flags, void* workspace, size_t workspace_bytes,
                void* cuda_stream);

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
 *     SPEC_NOALLOC_MAX_WORKSPACE (8 MiB; the workspace takes about 170 bytes
 *     per (row, position) unit per 1024 vocabulary entries, so at V = 151936
 *     about 325 units fit, e.g. 108 rows at k = 2); a larger batch returns
 *     SPEC_E_WORKSPACE and enqueues nothing.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture begins.
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
                        int B, int k, int V, int32_t* tokens, int32_t* accept_len, float* logprobs,
                        float* alpha, uint32_t* flags, void* cuda_stream);

/* Diagnostic: out[i] = Philox4x32-10(ctr[i], key = (seed mod 2^32, seed >> 32))
 * for i < n, computed by the same device function spec_verify uses.  ctr and
 * out are device arrays of n uint4 (16-byte aligned).  Lets a test compare
 * the device stream with an independent host implementation.                */
int spec_philox4x32_10(const uint32_t* ctr, uint64_t seed, uint32_t* out, int64_t n,
                       void* cuda_stream);

/* Human-readable text for a status code (static storage). */
const char* spec_status_string(int code);

/* SPEC_ABI_VERSION of the loaded library. */
int spec_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
