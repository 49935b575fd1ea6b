// Vocabulary-sharded verify entries (include/specdec_shard.h): argument
// checks, launch shapes and the kernels of shard_kernels.cuh.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "shard_kernels.cuh"
#include "specdec_shard.h"

using namespace specdec;

// ------------------------------------------------------------- vocabulary shards
namespace {
specdec_status_t shard_check(specdec_dtype_t dtype, int32_t B, int32_t n_max, int32_t V, int32_t v0, int32_t Vs) {
  if (dtype != SPECDEC_F32 && dtype != SPECDEC_BF16) return SPECDEC_ERR_INVALID_ARG;
  if (B < 0 || n_max < 0 || V <= 0 || v0 < 0 || Vs <= 0 || v0 > V - Vs) return SPECDEC_ERR_INVALID_ARG;
  if (V > SPECDEC_MAX_VOCAB || n_max > SPECDEC_MAX_DRAFT || B > SPECDEC_MAX_BATCH) return SPECDEC_ERR_UNSUPPORTED;
  return SPECDEC_OK;
}
}  // namespace

extern "C" size_t specdec_shard_stats_records(int32_t B, int32_t n_max) {
  if (B <= 0 || n_max < 0 || n_max > SPECDEC_MAX_DRAFT) return 0;
  return static_cast<size_t>(B) * (n_max + 1) * 2;
}

extern "C" size_t specdec_shard_race_records(int32_t B) {
  if (B <= 0 || B > SPECDEC_MAX_BATCH) return 0;
  return static_cast<size_t>(B) * shard_race_blocks(B);
}

extern "C" specdec_status_t spec_verify_shard_stats(const void* target_shard, const void* draft_shard,
                                                    specdec_dtype_t dtype, int32_t B, int32_t n_max, int32_t V,
                                                    int32_t v0, int32_t Vs, const int32_t* draft_tokens,
                                                    const int32_t* draft_len, const float* temperature,
                                                    void* stats_out, void* stream) {
  const specdec_status_t chk = shard_check(dtype, B, n_max, V, v0, Vs);
  if (chk != SPECDEC_OK) return chk;
  if (B == 0) return SPECDEC_OK;
  if (target_shard == nullptr || draft_len == nullptr || temperature == nullptr || stats_out == nullptr ||
      (n_max > 0 && draft_tokens == nullptr))
    return SPECDEC_ERR_INVALID_ARG;
  ShardArgs a;
  memset(&a, 0, sizeof a);
  a.target = target_shard;
  a.draft = n_max > 0 ? draft_shard : nullptr;
  a.B = B;
  a.n_max = n_max;
  a.V = V;
  a.v0 = v0;
  a.Vs = Vs;
  a.draft_tokens = draft_tokens;
  a.draft_len = draft_len;
  a.temperature = temperature;
  a.stats = static_cast<float4*>(stats_out);
  const unsigned grid = static_cast<unsigned>(B) * static_cast<unsigned>(2 * n_max + 1);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype == SPECDEC_F32)
    shard_stats_kernel<float><<<grid, kShardThreads, 0, st>>>(a);
  else
    shard_stats_kernel<uint16_t><<<grid, kShardThreads, 0, st>>>(a);
  return cudaGetLastError() == cudaSuccess ? SPECDEC_OK : SPECDEC_ERR_CUDA;
}

extern "C" specdec_status_t spec_verify_shard_race(const void* target_shard, const void* draft_shard,
                                                   specdec_dtype_t dtype, int32_t B, int32_t n_max, int32_t V,
                                                   int32_t v0, int32_t Vs, const int32_t* draft_tokens,
                                                   const int32_t* draft_len, const float* temperature,
                                                   uint64_t seed, const void* stats_all, int32_t S,
                                                   int32_t* accepted_len, void* race_out, uint32_t* error_word,
                                                   void* stream) {
  const specdec_status_t chk = shard_check(dtype, B, n_max, V, v0, Vs);
  if (chk != SPECDEC_OK) return chk;
  if (S <= 0) return SPECDEC_ERR_INVALID_ARG;
  if (B == 0) return SPECDEC_OK;
  if (target_shard == nullptr || draft_len == nullptr || temperature == nullptr || stats_all == nullptr ||
      accepted_len == nullptr || race_out == nullptr || (n_max > 0 && draft_tokens == nullptr))
    return SPECDEC_ERR_INVALID_ARG;
  ShardArgs a;
  memset(&a, 0, sizeof a);
  a.target = target_shard;
  a.draft = n_max > 0 ? draft_shard : nullptr;
  a.B = B;
  a.n_max = n_max;
  a.V = V;
  a.v0 = v0;
  a.Vs = Vs;
  a.draft_tokens = draft_tokens;
  a.draft_len = draft_len;
  a.temperature = temperature;
  a.seed_lo = static_cast<uint32_t>(seed & 0xFFFFFFFFull);
  a.seed_hi = static_cast<uint32_t>(seed >> 32);
  a.stats_all = static_cast<const float4*>(stats_all);
  a.S = S;
  a.accepted_len = accepted_len;
  a.race = static_cast<ulonglong2*>(race_out);
  a.err = error_word;
  a.R = shard_race_blocks(B);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const unsigned grid = static_cast<unsigned>(B) * static_cast<unsigned>(a.R);
  if (dtype == SPECDEC_F32)
    shard_race_kernel<float><<<grid, kShardThreads, 0, st>>>(a);
  else
    shard_race_kernel<uint16_t><<<grid, kShardThreads, 0, st>>>(a);
  return cudaGetLastError() == cudaSuccess ? SPECDEC_OK : SPECDEC_ERR_CUDA;
}

extern "C" specdec_status_t spec_verify_shard_finish(const void* race_all, int32_t S, int32_t B, int32_t n_max,
                                                     const int32_t* draft_tokens, const int32_t* accepted_len,
                                                     int32_t* out_tokens, void* stream) {
  if (S <= 0 || B < 0 || n_max < 0) return SPECDEC_ERR_INVALID_ARG;
  if (n_max > SPECDEC_MAX_DRAFT || B > SPECDEC_MAX_BATCH) return SPECDEC_ERR_UNSUPPORTED;
  if (B == 0) return SPECDEC_OK;
  if (race_all == nullptr || accepted_len == nullptr || out_tokens == nullptr || (n_max > 0 && draft_tokens == nullptr))
    return SPECDEC_ERR_INVALID_ARG;
  ShardArgs a;
  memset(&a, 0, sizeof a);
  a.B = B;
  a.n_max = n_max;
  a.S = S;
  a.draft_tokens = draft_tokens;
  a.accepted_len = const_cast<int32_t*>(accepted_len);
  a.race_all = static_cast<const ulonglong2*>(race_all);
  a.R = shard_race_blocks(B);
  a.out_tokens = out_tokens;
  shard_finish_kernel<<<(B + kShardFinishWarps - 1) / kShardFinishWarps, 32 * kShardFinishWarps, 0,
                        static_cast<cudaStream_t>(stream)>>>(a);
  return cudaGetLastError() == cudaSuccess ? SPECDEC_OK : SPECDEC_ERR_CUDA;
}

