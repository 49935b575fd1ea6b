/*
 * specdec_shard.h — vocabulary-sharded form of spec_verify (libspecdec.so,
 * sm_103a), for logits split over tensor-parallel ranks.
 *
 * Sources, by page title and section:
 *   "Accelerating Sonar through speculation" (Perplexity Research, 2025),
 *     §Draft-target scheduling — the target runs sharded over the ranks of a
 *       tensor-parallel group; the verify step then sees each row's logits
 *       split by vocabulary range across the ranks;
 *   "Fast Inference from Transformers via Speculative Decoding": the
 *     acceptance rule and residual / bonus sampling, exactly as spec_verify.
 *
 * The normalisers of a row (max and sum of exponentials of logit / T) combine
 * over shards by the usual log-sum-exp merge, and the exponential race that
 * picks a token from a distribution takes the entry with the largest
 * r_v / E_v, so it splits into a maximum per shard and a maximum over
 * shards.  The random numbers are keyed by the global vocabulary index, so a
 * sharded step gives the tokens the unsharded step gives on the same seed.
 *
 * Conventions are those of specdec.h (caller-owned device buffers, host
 * argument errors returned before anything is enqueued, device-data errors
 * as bits of an error word).
 */
#ifndef SPECDEC_SHARD_H_
#define SPECDEC_SHARD_H_

#include "specdec.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Vocabulary-sharded verify (tensor-parallel logits).  Each rank holds the
 * logits of one contiguous vocabulary range [v0, v0 + Vs) of every row:
 * target_shard [B, n_max+1, Vs], draft_shard [B, n_max, Vs] (dtype, device,
 * dense as in spec_verify; draft_shard NULL when every request is greedy or has
 * no drafts).
 * The step takes three calls per rank with two exchanges of small records
 * between ranks, which the caller performs (an all-gather on several GPUs;
 * on one GPU every shard simply writes its slice of the gathered buffer):
 *
 *   1. spec_verify_shard_stats: this shard's part of the row statistics of
 *      every row the step reads, into stats_out (float4 records,
 *      specdec_shard_stats_records(B, n_max) of them, 16 bytes each).
 *   -- gather: stats_all = the S shards' records, shard s at offset
 *      s * specdec_shard_stats_records(B, n_max), shards in vocabulary order.
 *   2. spec_verify_shard_race: combines stats_all into the row normalisers,
 *      runs the acceptance test (identical on every rank), writes
 *      accepted_len [B], and races over this shard's part of the row it
 *      samples from; race_out gets specdec_shard_race_records(B) records of
 *      16 bytes (a few per request; the count depends on B alone).
 *   -- gather: race_all = the S shards' race_out, shard s at offset
 *      s * specdec_shard_race_records(B) records.
 *   3. spec_verify_shard_finish: picks the winner over the shards and writes
 *      out_tokens [B, n_max+1] as spec_verify does.
 *
 * Arguments (every buffer caller-owned device memory on the calling GPU):
 *   V              the whole vocabulary; v0, Vs this shard's range.  The S
 *                  shards of one step must cover [0, V) in order (not
 *                  checked: other ranges give other tokens, never a read
 *                  outside the given buffers).
 *   draft_tokens   int32 [B, n_max], global vocabulary indices; draft_len
 *                  int32 [B]; temperature float [B]; seed: as spec_verify,
 *                  the same on every rank.
 *   stats_out      specdec_shard_stats_records(B, n_max) × 16 bytes, written
 *                  by call 1 (only the records of rows the step reads).
 *   stats_all      S × that, read by call 2.
 *   accepted_len   int32 [B], written by call 2, read by call 3.
 *   race_out       specdec_shard_race_records(B) × 16 bytes, written by
 *                  call 2; race_all S × that, read by call 3.
 *   out_tokens     int32 [B, n_max+1], written by call 3.
 *   error_word     optional uint32, device; bits are OR-ed in (never
 *                  cleared), as spec_verify's workspace error word.
 *   stream         cudaStream_t (NULL: the legacy default stream).  Each
 *                  call needs the previous call's outputs, and the gathered
 *                  buffers, complete when it starts: issue them in order on
 *                  one stream, or order the exchange between them.
 *
 * Same rule, random numbers (keyed by the global vocabulary index) and
 * outputs as spec_verify, which reads all the shards at once; device-data
 * errors set bits of *error_word when it is not NULL.  Every call is
 * asynchronous on `stream`; host argument errors return
 * SPECDEC_ERR_INVALID_ARG (v0 < 0, Vs <= 0, v0 + Vs > V, S <= 0, a NULL
 * buffer) or SPECDEC_ERR_UNSUPPORTED (limits), with nothing enqueued.
 */
size_t specdec_shard_stats_records(int32_t B, int32_t n_max);
size_t specdec_shard_race_records(int32_t B);
specdec_status_t spec_verify_shard_stats(const void* target_shard, const void* draft_shard,
                                         specdec_dtype_t dtype, int32_t B, int32_t n_max, int32_t V, int32_t v0,
                                         int32_t Vs, const int32_t* draft_tokens, const int32_t* draft_len,
                                         const float* temperature, void* stats_out, void* stream);
specdec_status_t spec_verify_shard_race(const void* target_shard, const void* draft_shard,
                                        specdec_dtype_t dtype, int32_t B, int32_t n_max, int32_t V, int32_t v0,
                                        int32_t Vs, const int32_t* draft_tokens, const int32_t* draft_len,
                                        const float* temperature, uint64_t seed, const void* stats_all, int32_t S,
                                        int32_t* accepted_len, void* race_out, uint32_t* error_word, void* stream);
specdec_status_t spec_verify_shard_finish(const void* race_all, int32_t S, int32_t B, int32_t n_max,
                                          const int32_t* draft_tokens, const int32_t* accepted_len,
                                          int32_t* out_tokens, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SPECDEC_SHARD_H_ */
