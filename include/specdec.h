/*
 * specdec.h — C ABI of the GB300 speculative-decoding verify/accept library
 * (libspecdec.so, sm_103a).
 *
 * Device operations, all asynchronous on the caller's CUDA stream, with no
 * host synchronisation and no device-to-host copy inside:
 *
 *   spec_verify             the batched verify/accept step of speculative
 *                           decoding on dense [B, n_max+1, V] logits;
 *   spec_verify_packed      the same step on packed ragged rows (cumulative
 *                           row offsets), with optional per-request position
 *                           offsets of the random counter;
 *   spec_verify_early_exit  spec_verify's results without reading the rows
 *                           after a request's first rejection;
 *   spec_verify_no_alloc    spec_verify on a library-owned workspace;
 *   mtp_shift_insert        the MTP bookkeeping step that shifts the
 *                           input-token buffer and inserts the newly accepted
 *                           target token.
 *
 * specdec_shard.h declares the same verify step on a vocabulary split into
 * shards (tensor-parallel ranks), in three calls per shard.
 *
 * Sources, by page title and section:
 *   "Accelerating Sonar through speculation" (Perplexity Research, 2025):
 *     §Speculative decoding — the target scores the drafted prefix, the
 *       longest acceptable prefix is kept, the target adds one token, so at
 *       most n+1 tokens leave one step (stages Acceptance, Target generation);
 *     §Target-draft — acceptance compares the full draft and target
 *       distributions; the accepted count drives the next sequence length;
 *     §MTP, §Single-token MTP scheduling — shift the input tokens left by one
 *       relative to the target hidden states and insert the next target token
 *       on the GPU, avoiding a GPU-to-CPU sync.
 *   "Fast Inference from Transformers via Speculative Decoding" (cited by the
 *     page above): accept with probability min(1, p/q), resample from
 *     norm(max(0, p - q)) on rejection, one bonus token from p otherwise.
 *   Salmon et al., "Parallel random numbers: as easy as 1, 2, 3" (SC'11):
 *     Philox4x32-10.
 *
 * Conventions
 *   - Every buffer is caller-owned device memory unless stated otherwise.  The
 *     library allocates nothing.
 *   - Argument errors are detected on the host and returned before anything is
 *     enqueued.  Launch failures return SPECDEC_ERR_CUDA.  Bad values found in
 *     device arrays never trap: they are clamped as described below and set a
 *     bit of the sticky device error word (read with specdec_get_error).
 *   - `stream` is a cudaStream_t passed as a plain pointer (NULL = the legacy
 *     default stream).
 *   - All calls are safe to capture into a CUDA graph (no allocation, no sync,
 *     no host-visible result).
 */
#ifndef SPECDEC_H_
#define SPECDEC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SPECDEC_OK = 0,
  SPECDEC_ERR_INVALID_ARG = 1, /* null pointer, size <= 0, bad dtype, ... */
  SPECDEC_ERR_UNSUPPORTED = 2, /* shape beyond the library's limits        */
  SPECDEC_ERR_WORKSPACE = 3,   /* workspace missing or too small           */
  SPECDEC_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed     */
  SPECDEC_ERR_DEVICE_DATA = 5, /* specdec_get_error: device data flagged   */
  SPECDEC_ERR_TIMEOUT = 6      /* specdec_get_error: a device wait ran out */
} specdec_status_t;

typedef enum { SPECDEC_F32 = 0, SPECDEC_BF16 = 1 } specdec_dtype_t;

/* Bits of the sticky device error word. */
#define SPECDEC_DEV_ERR_TOKEN 1u       /* a scored draft token was outside [0, V) */
#define SPECDEC_DEV_ERR_DRAFT_LEN 2u   /* draft_len[b] outside [0, n_max]; clamped */
#define SPECDEC_DEV_ERR_TEMPERATURE 4u /* T < 0, NaN, 0 < T < 1e-6, or T > 0 with
                                          draft_logits == NULL for a request
                                          with drafts; treated as T = 0 */
#define SPECDEC_DEV_ERR_TIMEOUT 8u     /* a device wait ran out (~2 s): the call's
                                          outputs are incomplete; the workspace is
                                          re-armed by the call itself */
#define SPECDEC_DEV_ERR_SEGMENT 16u    /* mtp_shift_insert: a segment outside [0, R)
                                          or a_b outside [0, n_b]; left unchanged */

/* Largest supported sizes. */
#define SPECDEC_MAX_VOCAB 262144 /* 2^18 */
#define SPECDEC_MAX_DRAFT 64
#define SPECDEC_MAX_BATCH 65536
#define SPECDEC_EARLY_EXIT_MAX_DRAFT 31 /* spec_verify_early_exit: n_max bound */

/*
 * Workspace for spec_verify, in bytes, for a batch of B requests with up to
 * n_max drafts over a vocabulary of V.  It holds per-request arrival counters,
 * per-row results, the race queue, the call's plan and the sticky error word
 * (its first 4 bytes).  It must be zero-filled once before its first use
 * (specdec_workspace_init or cudaMemset); every spec_verify call leaves it in
 * that state again, including a call whose device waits ran out
 * (SPECDEC_DEV_ERR_TIMEOUT: the last block to finish clears what the call left
 * behind), so it can be reused call after call.  One workspace serves one
 * in-flight call at a time.
 */
size_t specdec_verify_workspace_bytes(int32_t B, int32_t n_max, int32_t V);

/* Zero-fills `workspace` (bytes long) on `stream`. */
specdec_status_t specdec_workspace_init(void* workspace, size_t bytes, void* stream);

/*
 * spec_verify — batched verify/accept.
 *
 * Inputs (device):
 *   target_logits  [B, n_max+1, V] of dtype, row-major, row stride V elements.
 *                  Row j of request b holds the target's logits for the
 *                  position after draft j-1 (row 0: after the context).
 *   draft_logits   [B, n_max, V] of dtype, or NULL when every request is
 *                  greedy or has no drafts (n_b = 0: the token is sampled
 *                  from the target row alone).  Row j holds the draft's
 *                  logits that drew draft j.
 *   draft_tokens   int32 [B, n_max]: x_{b,j}.
 *   draft_len      int32 [B]: n_b in [0, n_max]; rows j > n_b (and draft rows
 *                  j >= n_b) are never read.
 *   temperature    float [B]: T_b >= 0; T_b == 0 selects greedy verification
 *                  (accept while x_j is the target's argmax, emit the argmax;
 *                  draft logits are not read for that request).  T_b > 0
 *                  applies logits * (1/T_b) to target and draft alike.
 *   seed           64-bit Philox key.  The random numbers of request b, row j
 *                  are Philox4x32-10(key = seed, counter = (v >> 2, j, b, k))
 *                  word v & 3, mapped to U = ((w >> 9) + 1/2) 2^-23; k = 0 is
 *                  the acceptance draw (v = 0), k = 1 the race draw of vocab
 *                  entry v.  b is the request's index in this call.
 * Rule (T_b > 0, s = 1/T_b): row j < n_b accepts iff u_j < p_j(x_j)/q_j(x_j)
 *   with p_j = softmax(s t_j), q_j = softmax(s d_j).  At the first rejected
 *   row a the emitted token is argmax_v r_v / E_v over r = max(0, p_a - q_a),
 *   E_v = -ln U_v (the exponential race, i.e. a draw from norm(r)); if every
 *   draft is accepted, a = n_b and the race runs on r = p_{n_b}.
 * Outputs (device):
 *   accepted_len   int32 [B]: a_b in [0, n_b], the number of accepted drafts.
 *   out_tokens     int32 [B, n_max+1]: x_{b,0..a-1}, then the target token,
 *                  then -1.  a_b + 1 tokens are valid.
 *   row_lse        optional float [B, n_max+1, 2], NULL allowed: for each
 *                  scored row of a T > 0 request, ln sum exp(s t_j) in [..,0]
 *                  and ln sum exp(s d_j) in [..,1] (draft rows j < n_b).
 *                  Entries of rows that are not scored are left unchanged.
 *   workspace      >= specdec_verify_workspace_bytes(B, n_max, V) bytes,
 *                  zero-filled before first use, 16-byte aligned.
 * Device-data errors: a draft token outside [0, V) rejects its row (greedy:
 * counts as a mismatch); draft_len is clamped into [0, n_max]; an invalid
 * temperature makes the request greedy.  Each sets an error bit.
 * Returns SPECDEC_OK once the work is enqueued.
 */
specdec_status_t spec_verify(const void* target_logits, const void* draft_logits,
                             specdec_dtype_t dtype, int32_t B, int32_t n_max, int32_t V,
                             const int32_t* draft_tokens, const int32_t* draft_len,
                             const float* temperature, uint64_t seed,
                             int32_t* accepted_len, int32_t* out_tokens, float* row_lse,
                             void* workspace, size_t workspace_bytes, void* stream);

/*
 * spec_verify_early_exit — spec_verify that does not read the rows a request
 * no longer needs: once row k of request b is rejected, its target and draft
 * rows after k are not streamed (those already in flight finish, unused).
 * The outputs are identical to spec_verify's (same rule, same random draws);
 * only the bytes read differ.  Rows are scheduled row-major across requests
 * (row j of every request before row j+1), so early rows are decided before
 * later ones are claimed.  The pages have no counterpart: the method only
 * ever needs the rows up to a request's first rejection, and this call
 * reads no more than that once the rejection is known.
 * A short batch (B (2 n_max + 1) V elt below 300 MB) claims every row before
 * the first decision can land, so skipping saves nothing there while the
 * row-by-row decisions cost time: such a batch is verified in spec_verify's
 * request order, every row read (same outputs).
 * Same arguments as spec_verify without row_lse (skipped rows have no
 * log-sum-exp), n_max <= SPECDEC_EARLY_EXIT_MAX_DRAFT (else
 * SPECDEC_ERR_UNSUPPORTED).  The logits bytes it reads (streamed rows plus
 * the race's re-reads) add up in the workspace until specdec_get_bytes_read
 * returns and clears them.
 */
specdec_status_t spec_verify_early_exit(const void* target_logits, const void* draft_logits,
                                        specdec_dtype_t dtype, int32_t B, int32_t n_max, int32_t V,
                                        const int32_t* draft_tokens, const int32_t* draft_len,
                                        const float* temperature, uint64_t seed,
                                        int32_t* accepted_len, int32_t* out_tokens,
                                        void* workspace, size_t workspace_bytes, void* stream);

/* Logits bytes read by spec_verify_early_exit calls on this workspace since
 * the last read; clears the count.  Synchronises the device (for tests and
 * profiling).  SPECDEC_OK, SPECDEC_ERR_INVALID_ARG or SPECDEC_ERR_CUDA. */
specdec_status_t specdec_get_bytes_read(void* workspace, uint64_t* bytes);

/*
 * spec_verify_packed — spec_verify on packed ragged rows: no padding in the
 * logits, the draft tokens or the outputs.  The pages have no API; the
 * layout is the usual cumulative-offset one of variable-length batches.
 * Random draws may follow each request's absolute position.
 *
 * Request b owns target rows cu_rows[b] .. cu_rows[b+1]-1; its draft length
 * is n_b = cu_rows[b+1] - cu_rows[b] - 1 (clamped to [0, n_max], which sets
 * SPECDEC_DEV_ERR_DRAFT_LEN), and its n_b draft rows and draft tokens start
 * at row cu_rows[b] - b of the draft tensors.
 *   target_logits  [total_rows, V] dtype, device.
 *   draft_logits   [total_rows - B, V] dtype, device; NULL when every request
 *                  is greedy (T == 0) or has no drafts.
 *   cu_rows        [B + 1] int32, device, non-decreasing, cu_rows[B] <=
 *                  total_rows.  A request whose segment is empty or reaches
 *                  outside the tensors is not read: accepted_len[b] = -1,
 *                  its outputs are left as they were, and
 *                  SPECDEC_DEV_ERR_DRAFT_LEN is set.
 *   total_rows     rows of target_logits (host int, >= B).
 *   draft_tokens   [total_rows - B] int32, device, laid out like the draft rows.
 *   temperature    [B] float, device, as in spec_verify.
 *   pos_offset     [B] int32, device, or NULL: request b draws with the row
 *                  word pos_offset[b] + j of the random counter (instead of
 *                  j), so its numbers can follow absolute positions.
 *   n_max          an upper bound of every n_b (host int, <= SPECDEC_MAX_DRAFT);
 *                  it sizes the workspace.
 * Outputs: accepted_len [B]; out_tokens [total_rows] laid out like the target
 * rows (request b's n_b + 1 slots: a accepted drafts, the sampled token,
 * then -1); row_lse [total_rows, 2] or NULL, laid out like the target rows.
 * Workspace: specdec_verify_workspace_bytes(B, n_max, V) bytes, prepared as
 * for spec_verify (the two calls may share one).  Same errors as spec_verify,
 * plus SPECDEC_ERR_INVALID_ARG when cu_rows is NULL or total_rows < B.
 */
specdec_status_t spec_verify_packed(const void* target_logits, const void* draft_logits,
                                    specdec_dtype_t dtype, int32_t B, int32_t n_max, int32_t V,
                                    const int32_t* cu_rows, int32_t total_rows,
                                    const int32_t* draft_tokens, const float* temperature,
                                    const int32_t* pos_offset, uint64_t seed,
                                    int32_t* accepted_len, int32_t* out_tokens, float* row_lse,
                                    void* workspace, size_t workspace_bytes, void* stream);

/*
 * mtp_shift_insert — MTP bookkeeping after verification.
 *
 * The token buffer is the flattened [R] list of the target's input tokens;
 * request b owns segment [s_b, s_b + n_b] (n_b + 1 slots), s_b = seg_start[b]
 * or b * (R / B) when seg_start is NULL.  Within each segment:
 *   out[s+i] = in[s+i+1] for i < n_b, out[s+n_b] = in[s+n_b],
 *   then out[s + a_b] = next token of request b,
 * where a_b = accepted_len[b] and the next token is next_token[b] when
 * next_token_stride == 0, else next_token[b * next_token_stride + a_b] (pass
 * spec_verify's out_tokens with stride n_max + 1).  Slots outside every
 * segment are not written.  tokens_in may equal tokens_out (in place).
 * Hidden states [R, H] of hidden_elem_bytes each stay where they are: row r
 * keeps hidden_in[r]; when hidden_out is non-NULL and differs from hidden_in
 * it receives a bitwise copy (both 16-byte aligned when R*H*elem is a multiple
 * of 16).  Reads accepted_len and next_token on the device: no host sync.
 * Device-data errors (a segment outside [0, R), a_b outside [0, n_b]) leave
 * the segment unchanged and set SPECDEC_DEV_ERR_SEGMENT in *error_word when
 * error_word is non-NULL (device memory; a spec_verify workspace may be passed,
 * its first word is its error word, so specdec_get_error reports both steps).
 */
specdec_status_t mtp_shift_insert(const int32_t* tokens_in, int32_t* tokens_out,
                                  const void* hidden_in, void* hidden_out, int32_t R, int32_t H,
                                  int32_t hidden_elem_bytes, const int32_t* seg_start,
                                  const int32_t* draft_len, const int32_t* accepted_len,
                                  const int32_t* next_token, int32_t next_token_stride,
                                  int32_t B, uint32_t* error_word, void* stream);

/*
 * Reads (and clears) the sticky device error word of a spec_verify workspace.
 * Synchronises the device: for tests and debugging, not for the hot path.
 * *error_bits receives the SPECDEC_DEV_ERR_* bits; returns
 * SPECDEC_ERR_TIMEOUT when SPECDEC_DEV_ERR_TIMEOUT is set (a call's device
 * waits ran out and its outputs are incomplete), else SPECDEC_ERR_DEVICE_DATA
 * when any other bit is set, SPECDEC_OK otherwise.
 */
specdec_status_t specdec_get_error(void* workspace, uint32_t* error_bits);

/*
 * spec_verify_no_alloc — spec_verify for callers that cannot allocate device
 * memory.  The pages this library follows have no counterpart: it exists for
 * code that must not call cudaMalloc at verification time (inside a custom
 * allocator or memory-pool callback, in runtimes that forbid allocation after
 * start-up because it synchronises the device, or in C hosts that only own the
 * tensors they pass in).
 *
 * Same arguments and results as spec_verify, without the workspace: the
 * library keeps a fixed device array of SPECDEC_NO_ALLOC_WORKSPACE_BYTES (8 MiB)
 * on every GPU that loads it, for the life of the process, and uses it as the
 * workspace.  A batch whose workspace would exceed that size
 * (specdec_verify_workspace_bytes(B, n_max, V) > SPECDEC_NO_ALLOC_WORKSPACE_BYTES)
 * is rejected with SPECDEC_ERR_WORKSPACE before anything is enqueued.
 *   - The first call on a device looks up the array's device address (with
 *     that device current); make that first call before any stream capture.
 *   - Every call clears the part of the array it uses on `stream` (a memset,
 *     no allocation) and then runs spec_verify there.
 *   - All calls on a device share the one array: calls that overlap on the
 *     GPU (different streams, not ordered) race and give wrong results;
 *     order them.
 *   - The device error word lives in the shared array and is cleared by the
 *     next call; it cannot be read through this entry point.
 * Returns what spec_verify returns, or SPECDEC_ERR_WORKSPACE for a batch that
 * does not fit.
 */
#define SPECDEC_NO_ALLOC_WORKSPACE_BYTES (8u << 20)
specdec_status_t spec_verify_no_alloc(const void* target_logits, const void* draft_logits,
                                      specdec_dtype_t dtype, int32_t B, int32_t n_max, int32_t V,
                                      const int32_t* draft_tokens, const int32_t* draft_len,
                                      const float* temperature, uint64_t seed, int32_t* accepted_len,
                                      int32_t* out_tokens, float* row_lse, void* stream);

/* Human-readable name of a status code (static string). */
const char* specdec_status_string(specdec_status_t status);

/* How spec_verify cuts a vocabulary row of V elements of `dtype` for a batch
 * of B requests with up to n_max drafts: the number of streamed chunks per row
 * and the elements per chunk (the last chunk holds the remainder).  Chunks are
 * 28 KB when the batch could stream 300 MB or more (B (2 n_max + 1) V
 * element bytes), else 24 KB.  For tests and profiling.  Returns SPECDEC_OK
 * or SPECDEC_ERR_INVALID_ARG. */
specdec_status_t specdec_verify_launch_shape(int32_t B, int32_t n_max, int32_t V, specdec_dtype_t dtype,
                                             int32_t* chunks_per_row, int32_t* chunk_elems);

#ifdef __cplusplus
}
#endif

#endif /* SPECDEC_H_ */
