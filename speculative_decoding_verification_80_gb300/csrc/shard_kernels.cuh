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
//   2. shard_race_kernel (R blocks per request): warp 0 of each block merges
//      every shard's records into the row normalisers P = K + log2 S
//      (identical on every rank) and runs the acceptance tests
//      u_j < p_j(x_j)/q_j(x_j), one lane per row, for the first rejection a;
//      then the block races over its slice of this shard's part of row a,
//      on r = max(0, p - q) (or p for the bonus row), and on p where no
//      residual weight was positive (the fallback used when every residual
//      weight in every shard vanished).  Random numbers use the global
//      vocabulary index, so the draws are the ones the unsharded step uses.
//   3. shard_finish_kernel: the largest race key over the shards' race
//      blocks gives the emitted token; outputs as in spec_verify.
//
// Rows are read with 16-byte vector loads (a scalar head up to the first
// 16-byte boundary, a scalar tail), four loads in flight per thread.
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
constexpr int kShardUnroll = 4;        // 16-byte loads in flight per thread

// Race blocks per request: about 512 blocks in all (one wave at three
// blocks per SM), 1 to 16 per request.  It depends on B alone, so every
// shard lays out its race records alike.
__host__ __device__ constexpr int shard_race_blocks(int B) {
  return B <= 32 ? 16 : (B >= 512 ? 1 : (512 + B - 1) / B);
}

struct ShardArgs {
  const void* target;  // [B, n_max+1, Vs]
  const void* draft;   // [B, n_max, Vs] or null
  int B, n_max, V, v0, Vs;
  int R;                        // race blocks per request: shard_race_blocks(B)
  const int32_t* draft_tokens;  // [B, n_max]
  const int32_t* draft_len;     // [B]
  const float* temperature;     // [B]
  uint32_t seed_lo, seed_hi;
  float4* stats;                // step 1 output: [B * (n_max+1) * 2]
  const float4* stats_all;      // step 2 input: [S][B * (n_max+1) * 2]
  int S;
  int32_t* accepted_len;        // step 2 output [B]
  ulonglong2* race;             // step 2 output [B][R]: (best on r, best on p) per race block
  const ulonglong2* race_all;   // step 3 input [S][B][R]
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
  // without draft logits only a request with no drafts can sample
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

// 16 bytes of logits as floats (bf16: element 0 in the low half of a word).
template <typename Elt>
__device__ __forceinline__ void shard_unpack(const uint4& u, float* x) {
  if constexpr (sizeof(Elt) == 4) {
    x[0] = __uint_as_float(u.x);
    x[1] = __uint_as_float(u.y);
    x[2] = __uint_as_float(u.z);
    x[3] = __uint_as_float(u.w);
  } else {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      x[2 * k] = __uint_as_float(w[k] << 16);
      x[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
  }
}

// Compile-time element count handed to the row visitors.
template <int C>
struct ShardCnt {
  static constexpr int value = C;
};

// Elements of a row that start at p before its first 16-byte boundary.
template <typename Elt>
__device__ __forceinline__ int shard_head(const void* p) {
  constexpr int E = 16 / sizeof(Elt);
  const int mis = static_cast<int>((reinterpret_cast<uintptr_t>(p) & 15u) / sizeof(Elt));
  return mis == 0 ? 0 : E - mis;
}

// Visits elements [0, n) of one row (tp) or of two rows side by side (tp
// and dp, dp may be null) over the block's threads; each thread sees its
// elements in increasing index order.  f(i0, xt, xd, cnt) gets cnt
// consecutive values from local index i0: cnt = 1 in the scalar head and
// tail, 16 / sizeof(Elt) in the middle, which is read in 16-byte words when
// both rows reach a 16-byte boundary at the same element (otherwise every
// element is read as a scalar).
template <typename Elt, typename F>
__device__ __forceinline__ void shard_walk(const void* tp, const void* dp, int n, F&& f) {
  constexpr int E = 16 / sizeof(Elt);
  const int ht = shard_head<Elt>(tp);
  const bool vec = dp == nullptr || shard_head<Elt>(dp) == ht;
  const int head = vec ? min(ht, n) : n;
  for (int i = threadIdx.x; i < head; i += kShardThreads) {
    const float xt = shard_at<Elt>(tp, i);
    const float xd = dp != nullptr ? shard_at<Elt>(dp, i) : 0.f;
    f(i, &xt, &xd, ShardCnt<1>{});
  }
  const int nv = (n - head) / E;
  const uint4* pt = reinterpret_cast<const uint4*>(static_cast<const Elt*>(tp) + head);
  const uint4* pd = dp != nullptr ? reinterpret_cast<const uint4*>(static_cast<const Elt*>(dp) + head) : nullptr;
  for (int k0 = threadIdx.x; k0 < nv; k0 += kShardThreads * kShardUnroll) {
    uint4 ut[kShardUnroll], ud[kShardUnroll];
#pragma unroll
    for (int q = 0; q < kShardUnroll; ++q) {
      const int k = k0 + q * kShardThreads;
      ut[q] = k < nv ? __ldg(pt + k) : make_uint4(0u, 0u, 0u, 0u);
      ud[q] = (pd != nullptr && k < nv) ? __ldg(pd + k) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int q = 0; q < kShardUnroll; ++q) {
      const int k = k0 + q * kShardThreads;
      if (k < nv) {
        float xt[E], xd[E];
        shard_unpack<Elt>(ut[q], xt);
        shard_unpack<Elt>(ud[q], xd);
        f(head + k * E, xt, xd, ShardCnt<E>{});
      }
    }
  }
  for (int i = head + nv * E + threadIdx.x; i < n; i += kShardThreads) {
    const float xt = shard_at<Elt>(tp, i);
    const float xd = dp != nullptr ? shard_at<Elt>(dp, i) : 0.f;
    f(i, &xt, &xd, ShardCnt<1>{});
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

// A race key: the positive float key's bits above the complemented index, so
// the larger key wins and an exact tie goes to the lower index.
__device__ __forceinline__ unsigned long long shard_pack(float key, int idx) {
  return (static_cast<unsigned long long>(__float_as_uint(key)) << 32) |
         static_cast<unsigned long long>(0xFFFFFFFFu - static_cast<uint32_t>(idx));
}

// Word k (0..3) of a Philox output, without indexing a local array.
__device__ __forceinline__ uint32_t shard_word(const Philox4& r, uint32_t k) {
  const uint32_t lo = (k & 1u) ? r.w[1] : r.w[0];
  const uint32_t hi = (k & 1u) ? r.w[3] : r.w[2];
  return (k & 2u) ? hi : lo;
}

// Normaliser P = K + log2 S of record t (0 target, 1 draft) of one row,
// merged over the S shards, and the logit at the row's draft token.
__device__ __forceinline__ float shard_merge(const ShardArgs& A, size_t rec, size_t stride, int t, float* xl) {
  float K = -INFINITY;
  for (int s = 0; s < A.S; ++s) K = fmaxf(K, A.stats_all[s * stride + rec + t].x);
  float Ssum = 0.f;
  for (int s = 0; s < A.S; ++s) {
    const float4 st = A.stats_all[s * stride + rec + t];
    if (st.y > 0.f) Ssum += st.y * exp2f(st.x - K);
    if (xl != nullptr && st.w != 0.f) *xl = st.z;
  }
  return K + log2f(Ssum);
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
  const size_t row = tensor == 0 ? static_cast<size_t>(b) * rows + j : static_cast<size_t>(b) * A.n_max + j;
  const void* rp = static_cast<const Elt*>(tensor == 0 ? A.target : A.draft) + row * A.Vs;
  float4 rec;
  if (q.greedy) {
    float m = -INFINITY;
    int idx = 0x7FFFFFFF;
    shard_walk<Elt>(rp, nullptr, A.Vs, [&](int i0, const float* x, const float*, auto cnt) {
      constexpr int C = decltype(cnt)::value;
#pragma unroll
      for (int e = 0; e < C; ++e)
        if (x[e] > m) {  // strictly: the first index keeps a tie
          m = x[e];
          idx = i0 + e;
        }
    });
    const float M = shard_block_max(m, reinterpret_cast<float*>(red));
    const int first = shard_block_min_i(m == M ? idx : 0x7FFFFFFF, reinterpret_cast<int*>(red));
    // a shard with no entry above -inf reports its first index at -inf
    rec = make_float4(M, __int_as_float(A.v0 + (first == 0x7FFFFFFF ? 0 : first)), 0.f, 0.f);
  } else {
    // one pass: per thread the running maximum m and S = sum 2^(c x - c m),
    // rescaled whenever a 16-byte word raises m
    const float c = q.c;
    float m = -INFINITY, s = 0.f;
    shard_walk<Elt>(rp, nullptr, A.Vs, [&](int, const float* x, const float*, auto cnt) {
      constexpr int C = decltype(cnt)::value;
      float vm = x[0];
#pragma unroll
      for (int e = 1; e < C; ++e) vm = fmaxf(vm, x[e]);
      if (vm > m) {
        s *= exp2f((m - vm) * c);
        m = vm;
      }
      if (m > -INFINITY) {
        const float mc = m * c;
#pragma unroll
        for (int e = 0; e < C; ++e) s += exp2f(fmaf(x[e], c, -mc));
      }
    });
    const float M = shard_block_max(m, reinterpret_cast<float*>(red));
    const float mine = m > -INFINITY ? s * exp2f((m - M) * c) : 0.f;
    const float Ssum = shard_block_sum(mine, reinterpret_cast<float*>(red));
    // the logit at the row's draft token, if this shard holds it
    float xl = 0.f, has = 0.f;
    if (j < q.L) {
      const int x = A.draft_tokens[static_cast<size_t>(b) * A.n_max + j];
      if (x >= A.v0 && x < A.v0 + A.Vs) {
        xl = shard_at<Elt>(rp, static_cast<size_t>(x - A.v0));
        has = 1.f;
      }
    }
    rec = make_float4(M * c, Ssum, xl, has);
  }
  if (threadIdx.x == 0) A.stats[(static_cast<size_t>(b) * rows + j) * 2 + tensor] = rec;
}

// Step 2, acceptance: called by one whole warp for request b; in round k,
// lane l tests row 32 k + l, and the lowest failing lane is the first
// rejection.  Returns a; *tok gets the greedy token (greedy requests),
// *errbits the request's device-data error bits.
__device__ __forceinline__ int shard_accept_warp(const ShardArgs& A, int b, const ShardReq& q, bool bad_len,
                                                 bool bad_t, int* tok, uint32_t* errbits) {
  const int lane = static_cast<int>(threadIdx.x & 31);
  const int rows = A.n_max + 1;
  const size_t stride = static_cast<size_t>(A.B) * rows * 2;
  int a = q.L;
  bool bad_tok = false;
  *tok = -1;
  for (int base = 0; base <= q.L; base += 32) {
    const int j = base + lane;
    bool fail = false, bad = false;
    int idx = -1;
    if (j <= q.L) {
      const size_t rec = (static_cast<size_t>(b) * rows + j) * 2;
      const int x = j < q.L ? A.draft_tokens[static_cast<size_t>(b) * A.n_max + j] : 0;
      const bool valid = x >= 0 && x < A.V;
      if (q.greedy) {
        float M = -INFINITY;
        for (int s = 0; s < A.S; ++s) {  // shards in vocabulary order: a tie keeps the lower index
          const float4 st = A.stats_all[s * stride + rec];
          if (idx < 0 || st.x > M) {
            M = st.x;
            idx = __float_as_int(st.y);
          }
        }
        if (j < q.L) {
          bad = !valid;
          fail = x != idx;
        }
      } else if (j < q.L) {
        float xt = 0.f, xd = 0.f;
        const float Pt = shard_merge(A, rec, stride, 0, &xt);
        const float Pd = shard_merge(A, rec, stride, 1, &xd);
        bool accept = false;
        if (valid) {
          const float l2ratio = fmaf(xt, q.c, -Pt) - fmaf(xd, q.c, -Pd);
          const Philox4 r = philox4x32_10(0u, static_cast<uint32_t>(j), static_cast<uint32_t>(b), 0u, A.seed_lo,
                                          A.seed_hi);
          accept = uniform_from_word(r.w[0]) < exp2f(l2ratio);
        }
        bad = !valid;
        fail = !accept;
      }
    }
    const unsigned fm = __ballot_sync(0xFFFFFFFFu, fail);
    const unsigned bm = __ballot_sync(0xFFFFFFFFu, bad);
    if (fm != 0u) {
      const int k = __ffs(fm) - 1;
      a = base + k;
      bad_tok = (bm >> k) & 1u;  // only the rejected row's token was tested and found invalid
      if (q.greedy) *tok = __shfl_sync(0xFFFFFFFFu, idx, k);
      break;
    }
    if (q.greedy && q.L < base + 32) *tok = __shfl_sync(0xFFFFFFFFu, idx, q.L - base);
  }
  *errbits = (bad_len ? SPECDEC_DEV_ERR_DRAFT_LEN : 0u) | (bad_t ? SPECDEC_DEV_ERR_TEMPERATURE : 0u) |
             (bad_tok ? SPECDEC_DEV_ERR_TOKEN : 0u);
  return a;
}

// Step 2: R blocks per request (shard_race_blocks(B)).  Warp 0 of every block
// runs the acceptance tests (the same decisions in every block and on every
// rank); block 0 of the request writes accepted_len and the error bits.
// Then each block races over its slice of this shard's part of row a and
// writes its own record race[b][r]: greedy requests the token under key
// +inf, sampled ones the packed best keys of the race on r and on p.
//
// The key of entry v is r_v / E_v with E_v = -ln U_v, and
// 1 - U <= -ln U <= (1 - U) / U, so r U / (1 - U) <= key <= r / (1 - U).
// The block first takes the largest lower bound over one entry per thread
// as a threshold (shrunk by 2^-18 so fp32 rounding keeps it below that
// entry's computed key); an entry whose upper bound does not exceed the
// thread's threshold cannot win and skips the logarithm and the division.
// The race on p (the fallback for a residual that vanished everywhere) runs
// only in blocks whose residual race found no positive weight: if any block
// of any shard found one, its result is never used.
template <typename Elt>
__global__ void __launch_bounds__(kShardThreads) shard_race_kernel(const ShardArgs A) {
  __shared__ unsigned long long red[kShardThreads / 32];
  __shared__ int s_a, s_tok;
  __shared__ float s_P[2];
  const int b = blockIdx.x / A.R;
  const int part = blockIdx.x % A.R;
  bool bad_len = false, bad_t = false;
  const ShardReq q = shard_req(A, b, &bad_len, &bad_t);
  const int rows = A.n_max + 1;
  const size_t stride = static_cast<size_t>(A.B) * rows * 2;
  if (threadIdx.x < 32) {
    int tok;
    uint32_t errbits;
    const int a = shard_accept_warp(A, b, q, bad_len, bad_t, &tok, &errbits);
    if (threadIdx.x == 0) {
      if (part == 0) {
        A.accepted_len[b] = a;
        if (errbits && A.err != nullptr) atomicOr(A.err, errbits);
      }
      s_a = a;
      s_tok = tok;
      if (!q.greedy) {
        const size_t rec = (static_cast<size_t>(b) * rows + a) * 2;
        s_P[0] = shard_merge(A, rec, stride, 0, nullptr);
        s_P[1] = a < q.L ? shard_merge(A, rec, stride, 1, nullptr) : 0.f;
      }
    }
  }
  __syncthreads();
  ulonglong2* slot = A.race + static_cast<size_t>(b) * A.R + part;
  if (q.greedy) {
    if (threadIdx.x == 0) {
      const unsigned long long pk = shard_pack(INFINITY, s_tok < 0 ? 0 : s_tok);
      *slot = make_ulonglong2(pk, pk);
    }
    return;
  }
  const int a = s_a;
  const bool residual = a < q.L;
  const float Pt = s_P[0], Pd = s_P[1];
  const int per = ((A.Vs + A.R - 1) / A.R + 7) & ~7;  // a multiple of 8 keeps every slice's alignment
  const int e0 = part * per;
  const int n = min(per, A.Vs - e0);
  if (n <= 0) {
    if (threadIdx.x == 0) *slot = make_ulonglong2(0ull, 0ull);
    return;
  }
  const void* tp = static_cast<const Elt*>(A.target) + (static_cast<size_t>(b) * rows + a) * A.Vs + e0;
  const void* dp =
      residual ? static_cast<const Elt*>(A.draft) + (static_cast<size_t>(b) * A.n_max + a) * A.Vs + e0 : nullptr;
  const uint32_t vbase = static_cast<uint32_t>(A.v0 + e0);
  const float c = q.c;
  const uint32_t row_word = static_cast<uint32_t>(a), req_word = static_cast<uint32_t>(b);

  // threshold seed from entry threadIdx.x of the slice
  float seed = 0.f;
  if (static_cast<int>(threadIdx.x) < n) {
    const int i = static_cast<int>(threadIdx.x);
    const uint32_t v = vbase + static_cast<uint32_t>(i);
    const uint32_t w = shard_word(philox4x32_10(v >> 2, row_word, req_word, 1u, A.seed_lo, A.seed_hi), v & 3u);
    const float p = exp2f(fmaf(shard_at<Elt>(tp, i), c, -Pt));
    const float rr = residual ? p - exp2f(fmaf(shard_at<Elt>(dp, i), c, -Pd)) : p;
    if (rr > 0.f)
      seed = rr * uniform_from_word(w) / one_minus_uniform_from_word(w) * (1.0f - 3.814697265625e-06f);
  }
  seed = shard_block_max(seed, reinterpret_cast<float*>(red));

  // one race over the slice: on r (residual rows), or on p
  auto race = [&](bool on_p, float thr) -> unsigned long long {
    unsigned long long best = 0ull;
    uint32_t grp = 0xFFFFFFFFu;
    Philox4 rnd;
    shard_walk<Elt>(tp, on_p ? nullptr : dp, n, [&](int i0, const float* xt, const float* xd, auto cnt) {
      constexpr int C = decltype(cnt)::value;
#pragma unroll
      for (int e = 0; e < C; ++e) {
        const uint32_t v = vbase + static_cast<uint32_t>(i0 + e);
        if ((v >> 2) != grp) {
          grp = v >> 2;
          rnd = philox4x32_10(grp, row_word, req_word, 1u, A.seed_lo, A.seed_hi);
        }
        const uint32_t w = shard_word(rnd, v & 3u);
        const float p = exp2f(fmaf(xt[e], c, -Pt));
        const float rr = (residual && !on_p) ? p - exp2f(fmaf(xd[e], c, -Pd)) : p;
        if (rr - thr * one_minus_uniform_from_word(w) > 0.f) {  // r / (1 - U) > thr
          const float key = rr / -logf(uniform_from_word(w));
          const unsigned long long k = shard_pack(key, static_cast<int>(v));
          if (k > best) {
            best = k;
            thr = fmaxf(thr, key);
          }
        }
      }
    });
    return shard_block_max_u64(best, red);
  };
  const unsigned long long best_r = race(false, seed);
  unsigned long long best_p = 0ull;
  if (residual && best_r == 0ull) best_p = race(true, 0.f);  // block-uniform
  if (threadIdx.x == 0) *slot = make_ulonglong2(best_r, best_p);
}

// Step 3: one warp per request; the best keys over every shard's race
// blocks, then the outputs.
constexpr int kShardFinishWarps = 4;
__global__ void __launch_bounds__(32 * kShardFinishWarps) shard_finish_kernel(const ShardArgs A) {
  const int lane = static_cast<int>(threadIdx.x & 31);
  const int b = blockIdx.x * kShardFinishWarps + static_cast<int>(threadIdx.x >> 5);
  if (b >= A.B) return;
  const int rows = A.n_max + 1;
  unsigned long long br = 0ull, bp = 0ull;
  for (int k = lane; k < A.S * A.R; k += 32) {
    const int s = k / A.R, part = k % A.R;
    const ulonglong2 r = A.race_all[(static_cast<size_t>(s) * A.B + b) * A.R + part];
    br = r.x > br ? r.x : br;
    bp = r.y > bp ? r.y : bp;
  }
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long ur = __shfl_xor_sync(0xFFFFFFFFu, br, o);
    const unsigned long long up = __shfl_xor_sync(0xFFFFFFFFu, bp, o);
    br = ur > br ? ur : br;
    bp = up > bp ? up : bp;
  }
  const unsigned long long best = br != 0ull ? br : bp;  // all residual weights vanished: race on p
  const int y = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(best & 0xFFFFFFFFull));
  const int a = A.accepted_len[b];
  int32_t* out = A.out_tokens + static_cast<size_t>(b) * rows;
  for (int k = lane; k < rows; k += 32)
    out[k] = k < a ? A.draft_tokens[static_cast<size_t>(b) * A.n_max + k] : (k == a ? y : -1);
}

}  // namespace specdec
