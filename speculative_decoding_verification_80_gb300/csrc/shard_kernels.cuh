// shard_kernels.cuh — verify/accept on a vocabulary split into shards, the
// way tensor-parallel ranks hold the logits: each rank owns a contiguous
// range [v0, v0 + Vs) of every row.  Three steps per rank, with an exchange
// of small per-row records between ranks after the first two:
//
//   1. shard_stats_kernel: per valid row and tensor, the shard's part of the
//      row statistics — (K, S) with K = c max x (log2 units, c = log2(e)/T)
//      and S = sum 2^(c x - K) for sampled requests, (max, first index) for
//      greedy ones — plus the logit at the row's draft token when the token
//      falls in the shard.
//   2. shard_race_kernel: from every shard's records, the row normalisers
//      P = K + log2 S combined over shards (identical on every rank), the
//      acceptance test u_j < p_j(x_j)/q_j(x_j) and the first rejection a;
//      then the exponential race over this shard's part of row a, on r =
//      max(0, p - q) (or p for the bonus row) and also on p (the fallback
//      used when every residual weight in every shard vanished).  Random
//      numbers use the global vocabulary index, so the draws are the ones the
//      unsharded step uses.
//   3. shard_finish_kernel: the largest race key over the shards gives the
//      emitted token; outputs as in spec_verify.
//
// Sources: "Accelerating Sonar through speculation" §Speculative decoding
// and §Target-draft; the min(1, p/q) rule of "Fast Inference from
// Transformers via Speculative Decoding"; Philox4x32-10 from Salmon et al.
// (SC'11).  The pages name tensor-parallel serving; the split of the step
// into per-shard records is this library's.
#pragma once
#include <math.h>
#include <stdint.h>

#include "philox.cuh"
#include "specdec.h"

namespace specdec {

constexpr int kShardThreads = 256;

struct ShardArgs {
  const void* target;  // [B, n_max+1, Vs]
  const void* draft;   // [B, n_max, Vs] or null
  int B, n_max, V, v0, Vs;
  const int32_t* draft_tokens;  // [B, n_max]
  const int32_t* draft_len;     // [B]
  const float* temperature;     // [B]
  uint32_t seed_lo, seed_hi;
  float4* stats;                // step 1 output: [B * (n_max+1) * 2]
  const float4* stats_all;      // step 2 input: [S][B * (n_max+1) * 2]
  int S;
  int32_t* accepted_len;        // step 2 output [B]
  ulonglong2* race;             // step 2 output [B]: (best on r, best on p)
  const ulonglong2* race_all;   // step 3 input [S][B]
  int32_t* out_tokens;          // step 3 output [B, n_max+1]
  uint32_t* err;                // device error word (or null)
};

struct ShardReq {
  int L;
  float c;
  bool greedy;
};
__device__ __forceinline__ ShardReq shard_req(const ShardArgs& A, int b, bool* bad_len, bool* bad_t) {
  ShardReq r;
  const int Lr = A.draft_len[b];
  r.L = min(max(Lr, 0), A.n_max);
  const float T = A.temperature[b];
  r.greedy = !(T > 0.f) || T < 1e-6f || (A.draft == nullptr && r.L > 0);
  r.c = (1.0f / T) * 1.4426950408889634f;
  if (bad_len) *bad_len = Lr != r.L;
  if (bad_t) *bad_t = r.greedy && T != 0.f;
  return r;
}

template <typename Elt>
__device__ __forceinline__ float shard_at(const void* base, size_t i) {
  if constexpr (sizeof(Elt) == 4) {
    return static_cast<const float*>(base)[i];
  } else {
    return __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(base)[i]) << 16);
  }
}

__device__ __forceinline__ float shard_block_max(float v, float* red) {
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[w] = v;
  __syncthreads();
  float r = red[0];
  for (int k = 1; k < kShardThreads / 32; ++k) r = fmaxf(r, red[k]);
  return r;
}
__device__ __forceinline__ float shard_block_sum(float v, float* red) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[w] = v;
  __syncthreads();
  float r = 0.f;
  for (int k = 0; k < kShardThreads / 32; ++k) r += red[k];
  return r;
}
__device__ __forceinline__ int shard_block_min_i(int v, int* red) {
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[w] = v;
  __syncthreads();
  int r = red[0];
  for (int k = 1; k < kShardThreads / 32; ++k) r = min(r, red[k]);
  return r;
}
__device__ __forceinline__ unsigned long long shard_block_max_u64(unsigned long long v, unsigned long long* red) {
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long u = __shfl_xor_sync(0xFFFFFFFFu, v, o);
    v = u > v ? u : v;
  }
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[w] = v;
  __syncthreads();
  unsigned long long r = red[0];
  for (int k = 1; k < kShardThreads / 32; ++k) r = red[k] > r ? red[k] : r;
  return r;
}

// Step 1: one block per (request, row-tensor) unit, request-major.
template <typename Elt>
__global__ void __launch_bounds__(kShardThreads) shard_stats_kernel(const ShardArgs A) {
  __shared__ unsigned long long red[kShardThreads / 32];
  const int rows = A.n_max + 1;
  const int per_req = 2 * A.n_max + 1;
  const int b = blockIdx.x / per_req;
  const int r = blockIdx.x % per_req;
  const ShardReq q = shard_req(A, b, nullptr, nullptr);
  const int tensor = r < rows ? 0 : 1;
  const int j = tensor == 0 ? r : r - rows;
  if (tensor == 0 ? j > q.L : (q.greedy || j >= q.L)) return;  // rows the step never reads
  const void* base = tensor == 0 ? A.target : A.draft;
  const size_t row = tensor == 0 ? static_cast<size_t>(b) * rows + j : static_cast<size_t>(b) * A.n_max + j;
  const size_t off = row * A.Vs;
  float4 rec;
  if (q.greedy) {
    float m = -INFINITY;
    int idx = 0x7FFFFFFF;
    for (int v = threadIdx.x; v < A.Vs; v += kShardThreads) {
      const float x = shard_at<Elt>(base, off + v);
      if (x > m) {  // strictly: the first index keeps a tie
        m = x;
        idx = v;
      }
    }
    const float M = shard_block_max(m, reinterpret_cast<float*>(red));
    const int first = shard_block_min_i(m == M ? idx : 0x7FFFFFFF, reinterpret_cast<int*>(red));
    rec = make_float4(M, __int_as_float(first == 0x7FFFFFFF ? -1 : A.v0 + first), 0.f, 0.f);
  } else {
    float m = -INFINITY;
    for (int v = threadIdx.x; v < A.Vs; v += kShardThreads) m = fmaxf(m, shard_at<Elt>(base, off + v));
    const float M = shard_block_max(m, reinterpret_cast<float*>(red));
    const float K = M * q.c;
    float s = 0.f;
    if (M > -INFINITY)
      for (int v = threadIdx.x; v < A.Vs; v += kShardThreads) s += exp2f(fmaf(shard_at<Elt>(base, off + v), q.c, -K));
    const float Ssum = shard_block_sum(s, reinterpret_cast<float*>(red));
    // the logit at the row's draft token, if this shard holds it
    float xl = 0.f, has = 0.f;
    if (j < q.L) {
      const int x = A.draft_tokens[static_cast<size_t>(b) * A.n_max + j];
      if (x >= A.v0 && x < A.v0 + A.Vs) {
        xl = shard_at<Elt>(base, off + (x - A.v0));
        has = 1.f;
      }
    }
    rec = make_float4(K, Ssum, xl, has);
  }
  if (threadIdx.x == 0) A.stats[(static_cast<size_t>(b) * rows + j) * 2 + tensor] = rec;
}

__device__ __forceinline__ unsigned long long shard_pack(float key, int idx) {
  return (static_cast<unsigned long long>(__float_as_uint(key)) << 32) |
         static_cast<unsigned long long>(0xFFFFFFFFu - static_cast<uint32_t>(idx));
}

// Step 2: one block per request.
template <typename Elt>
__global__ void __launch_bounds__(kShardThreads) shard_race_kernel(const ShardArgs A) {
  __shared__ unsigned long long red[kShardThreads / 32];
  __shared__ float sP[2 * (SPECDEC_MAX_DRAFT + 1)];
  __shared__ int s_a;
  __shared__ int s_gidx;
  const int b = blockIdx.x;
  const int rows = A.n_max + 1;
  bool bad_len = false, bad_t = false;
  const ShardReq q = shard_req(A, b, &bad_len, &bad_t);
  const size_t shard_stride = static_cast<size_t>(A.B) * rows * 2;
  if (threadIdx.x == 0) {
    // Combine the shards' records row by row and find the first rejection.
    uint32_t errbits = (bad_len ? SPECDEC_DEV_ERR_DRAFT_LEN : 0u) | (bad_t ? SPECDEC_DEV_ERR_TEMPERATURE : 0u);
    int a = q.L, gidx = -1;
    for (int j = 0; j <= q.L; ++j) {
      const size_t rec = (static_cast<size_t>(b) * rows + j) * 2;
      if (q.greedy) {
        float M = -INFINITY;
        int idx = -1;
        for (int s = 0; s < A.S; ++s) {  // shards in vocabulary order: a tie keeps the lower index
          const float4 st = A.stats_all[s * shard_stride + rec];
          const int si = __float_as_int(st.y);
          if (si >= 0 && st.x > M) {
            M = st.x;
            idx = si;
          }
        }
        if (j == q.L) {
          gidx = idx;
          break;
        }
        const int x = A.draft_tokens[static_cast<size_t>(b) * A.n_max + j];
        if (!(x >= 0 && x < A.V)) errbits |= SPECDEC_DEV_ERR_TOKEN;
        if (x != idx) {
          a = j;
          gidx = idx;
          break;
        }
      } else {
        float P[2] = {0.f, 0.f}, xl[2] = {0.f, 0.f};
        for (int t = 0; t < 2; ++t) {
          if (t == 1 && j >= q.L) break;
          float K = -INFINITY;
          for (int s = 0; s < A.S; ++s) K = fmaxf(K, A.stats_all[s * shard_stride + rec + t].x);
          float Ssum = 0.f;
          for (int s = 0; s < A.S; ++s) {
            const float4 st = A.stats_all[s * shard_stride + rec + t];
            if (st.y > 0.f) Ssum += st.y * exp2f(st.x - K);
            if (st.w != 0.f) xl[t] = st.z;
          }
          P[t] = K + log2f(Ssum);
        }
        sP[2 * j] = P[0];
        sP[2 * j + 1] = P[1];
        if (j == q.L) break;
        const int x = A.draft_tokens[static_cast<size_t>(b) * A.n_max + j];
        bool accept = false;
        if (x >= 0 && x < A.V) {
          const float l2ratio = fmaf(xl[0], q.c, -P[0]) - fmaf(xl[1], q.c, -P[1]);
          const Philox4 r = philox4x32_10(0u, static_cast<uint32_t>(j), static_cast<uint32_t>(b), 0u, A.seed_lo,
                                          A.seed_hi);
          accept = uniform_from_word(r.w[0]) < exp2f(l2ratio);
        } else {
          errbits |= SPECDEC_DEV_ERR_TOKEN;
        }
        if (!accept) {
          a = j;
          break;
        }
      }
    }
    if (errbits && A.err != nullptr) atomicOr(A.err, errbits);
    s_a = a;
    s_gidx = gidx;
    A.accepted_len[b] = a;
  }
  __syncthreads();
  const int a = s_a;
  if (q.greedy) {
    // every rank knows the token; key +inf makes it win the combine
    if (threadIdx.x == 0) {
      const unsigned long long pk = shard_pack(INFINITY, s_gidx < 0 ? 0 : s_gidx);
      A.race[b] = make_ulonglong2(pk, pk);
    }
    return;
  }
  // The race over this shard's part of row a.
  const bool residual = a < q.L;
  const float Pt = sP[2 * a], Pd = sP[2 * a + 1];
  const size_t toff = (static_cast<size_t>(b) * rows + a) * A.Vs;
  const size_t doff = (static_cast<size_t>(b) * A.n_max + a) * A.Vs;
  unsigned long long best_r = 0ull, best_p = 0ull;
  for (int vl = threadIdx.x; vl < A.Vs; vl += kShardThreads) {
    const int v = A.v0 + vl;
    const float p = exp2f(fmaf(shard_at<Elt>(A.target, toff + vl), q.c, -Pt));
    const float qd = residual ? exp2f(fmaf(shard_at<Elt>(A.draft, doff + vl), q.c, -Pd)) : 0.f;
    const float rr = residual ? p - qd : p;
    const Philox4 rnd = philox4x32_10(static_cast<uint32_t>(v) >> 2, static_cast<uint32_t>(a),
                                      static_cast<uint32_t>(b), 1u, A.seed_lo, A.seed_hi);
    const float e = -logf(uniform_from_word(rnd.w[v & 3]));
    if (rr > 0.f) {
      const unsigned long long k = shard_pack(rr / e, v);
      best_r = k > best_r ? k : best_r;
    }
    if (residual && p > 0.f) {
      const unsigned long long k = shard_pack(p / e, v);
      best_p = k > best_p ? k : best_p;
    }
  }
  best_r = shard_block_max_u64(best_r, red);
  best_p = shard_block_max_u64(best_p, red);
  if (threadIdx.x == 0) A.race[b] = make_ulonglong2(best_r, residual ? best_p : best_r);
}

// Step 3: one thread per request.
__global__ void shard_finish_kernel(const ShardArgs A) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= A.B) return;
  const int rows = A.n_max + 1;
  unsigned long long br = 0ull, bp = 0ull;
  for (int s = 0; s < A.S; ++s) {
    const ulonglong2 r = A.race_all[static_cast<size_t>(s) * A.B + b];
    br = r.x > br ? r.x : br;
    bp = r.y > bp ? r.y : bp;
  }
  const unsigned long long best = br != 0ull ? br : bp;  // all residual weights vanished: race on p
  const int y = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(best & 0xFFFFFFFFull));
  const int a = A.accepted_len[b];
  int32_t* out = A.out_tokens + static_cast<size_t>(b) * rows;
  for (int k = 0; k < rows; ++k)
    out[k] = k < a ? A.draft_tokens[static_cast<size_t>(b) * A.n_max + k] : (k == a ? y : -1);
}

}  // namespace specdec
