// verify_persistent.cuh — persistent, warp-specialised verify/accept kernel
// for sm_103a (one CTA per SM).
//
// Work is a stream of row-tensor units (request b, target row j or draft row
// j) in request-major order, claimed from a device counter.  Per CTA:
//   * a producer warp claims a unit and streams it in chunks of up to
//     kStageBytes through a ring of kStages shared-memory stages with 1-D bulk
//     copies (TMA engine); each stage has a "full" mbarrier (bytes landed) and
//     an "empty" mbarrier (consumer done);
//   * kGroups consumer groups of kGroupWarps warps take the stages in turn
//     (group g owns stages g, g+kGroups, ...) and reduce each chunk to a
//     partial: (K = max(x)*c, S = sum 2^(x c - K)) for sampled requests,
//     (max, first index of max) for greedy ones, with c = log2(e)/T;
//   * one thread of the group publishes the partial and bumps the row's
//     counter; the chunk that completes a row combines the partials into the
//     row's log-sum-exp, runs the acceptance test u_j < p_j(x_j)/q_j(x_j), and
//     bumps the request's counter; the row that completes a request finds the
//     first rejection a (or a = n_b) and either writes the greedy result or
//     queues the exponential race over row a as chunk jobs;
//   * producers serve queued race jobs before new units: the race re-reads
//     row a (target, plus draft when a < n_b) right after it was streamed, so
//     the bytes come from L2, and it runs exactly once per request.
// No CTA ever waits for another CTA's progress except the producer's bounded
// poll for queued race jobs once no unit is left; every wait is bounded.
//
// Sources: "Accelerating Sonar through speculation" §Speculative decoding
// (stages Acceptance and Target generation) and §Target-draft; the
// min(1, p/q) rule of "Fast Inference from Transformers via Speculative
// Decoding"; Philox4x32-10 from Salmon et al. (SC'11).
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "philox.cuh"
#include "ptx.cuh"
#include "specdec.h"

namespace specdec {

constexpr int kGroups = 4;
constexpr int kGroupWarps = 4;
constexpr int kGroupThreads = kGroupWarps * 32;
constexpr int kThreads = 32 + kGroups * kGroupThreads;  // producer warp + consumers
constexpr int kStages = 8;                              // a multiple of kGroups
constexpr int kStageBytes = 24 * 1024;
constexpr long long kWaitBudgetCycles = 4000000000LL;  // ~2 s of SM clock
constexpr long long kIdlePollLimit = 20000000LL;       // producer polls (~x 256 ns sleep)
static_assert(kStages % kGroups == 0, "each group owns whole stages");

enum : uint32_t { kItemStream = 1u, kItemRace = 2u, kItemExit = 3u };
// race job encoding in the queue: valid | chunk << 24 | round << 23 | b
constexpr uint32_t kJobValid = 0x80000000u;

struct ItemDesc {  // one per stage, written by the producer
  uint32_t kind;
  int b, j;      // request, row (race: row a)
  int tensor;    // stream: 0 target, 1 draft
  int e0, n;     // first vocab index and element count of the chunk
  int chunk;     // chunk index within the row-tensor (stream) or the race
  int greedy;
  float c;       // log2(e) / T
  float Pt, Pd;  // race: log2 normalisers of row a
  int residual;  // race: r = max(0, p - q) (else r = p)
  int round;     // race: 0, or 1 for the fallback on p
  int expect;    // stream: chunks that complete the row (both tensors)
  int pad[2];
};
static_assert(sizeof(ItemDesc) == 64, "descriptor layout");

struct PArgs {
  const void* target;
  const void* draft;
  const int32_t* draft_tokens;
  const int32_t* draft_len;
  const float* temperature;
  int32_t* accepted_len;
  int32_t* out_tokens;
  float* row_lse;
  uint32_t seed_lo, seed_hi;
  int B, n_max, V;
  int nch;        // stream chunks per row-tensor
  int ch;         // elements per stream chunk
  int nrc;        // race chunks per row
  int chr;        // elements per race chunk
  uint32_t n_units;  // B * (2 n_max + 1)
  // workspace
  uint32_t* err;
  uint32_t* ctr;  // [0] unit head, [1] race head, [2] race tail, [3] requests done, [4] CTAs exited
  uint32_t* race_q;                 // [2 * B * nrc]
  uint32_t* req_cnt;                // [B]
  unsigned long long* race_best;    // [B]
  uint32_t* race_cnt;               // [B]
  int32_t* race_row;                // [B]
  float2* race_P;                   // [B]
  uint32_t* row_cnt;                // [B * rows]
  float2* row_P;                    // [B * rows]
  int32_t* row_arg;                 // [B * rows]
  uint32_t* row_acc;                // [B * rows]
  float2* part;                     // [B * rows * 2 * nch]
};

// ------------------------------------------------------------- element types
__device__ __forceinline__ float fast_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <typename Elt>
struct EltOps;

template <>
struct EltOps<float> {
  static constexpr int kVec = 4;
  using MaxAcc = float;
  __device__ static __forceinline__ MaxAcc max_init() { return -INFINITY; }
  __device__ static __forceinline__ void max_vec(const uint4& w, MaxAcc& m) {
    m = fmaxf(fmaxf(m, __uint_as_float(w.x)), __uint_as_float(w.y));
    m = fmaxf(fmaxf(m, __uint_as_float(w.z)), __uint_as_float(w.w));
  }
  __device__ static __forceinline__ float max_value(MaxAcc m) { return m; }
  __device__ static __forceinline__ void sum_vec(const uint4& w, float2 cc, float2 nk, float2& acc) {
    const float2 a = __ffma2_rn(make_float2(__uint_as_float(w.x), __uint_as_float(w.y)), cc, nk);
    const float2 b = __ffma2_rn(make_float2(__uint_as_float(w.z), __uint_as_float(w.w)), cc, nk);
    acc = __fadd2_rn(acc, make_float2(fast_ex2(a.x), fast_ex2(a.y)));
    acc = __fadd2_rn(acc, make_float2(fast_ex2(b.x), fast_ex2(b.y)));
  }
  __device__ static __forceinline__ void unpack(const uint4& w, float (&f)[4]) {
    f[0] = __uint_as_float(w.x);
    f[1] = __uint_as_float(w.y);
    f[2] = __uint_as_float(w.z);
    f[3] = __uint_as_float(w.w);
  }
  __device__ static __forceinline__ float at(const float* p, size_t i) { return p[i]; }
};

// bf16 as raw 16-bit patterns: widening to fp32 is a shift; the max runs on
// packed pairs (exact).
template <>
struct EltOps<uint16_t> {
  static constexpr int kVec = 8;
  using MaxAcc = __nv_bfloat162;
  __device__ static __forceinline__ MaxAcc max_init() {
    return __halves2bfloat162(__ushort_as_bfloat16(0xFF80u), __ushort_as_bfloat16(0xFF80u));
  }
  __device__ static __forceinline__ __nv_bfloat162 as_bf2(uint32_t u) {
    return *reinterpret_cast<const __nv_bfloat162*>(&u);
  }
  __device__ static __forceinline__ void max_vec(const uint4& w, MaxAcc& m) {
    m = __hmax2(m, __hmax2(__hmax2(as_bf2(w.x), as_bf2(w.y)), __hmax2(as_bf2(w.z), as_bf2(w.w))));
  }
  __device__ static __forceinline__ float max_value(MaxAcc m) {
    return fmaxf(__bfloat162float(m.x), __bfloat162float(m.y));
  }
  __device__ static __forceinline__ float2 pair(uint32_t u) {
    return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
  }
  __device__ static __forceinline__ void sum_vec(const uint4& w, float2 cc, float2 nk, float2& acc) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 a = __ffma2_rn(pair(u[k]), cc, nk);
      acc = __fadd2_rn(acc, make_float2(fast_ex2(a.x), fast_ex2(a.y)));
    }
  }
  __device__ static __forceinline__ void unpack(const uint4& w, float (&f)[8]) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      f[2 * k] = __uint_as_float(u[k] << 16);
      f[2 * k + 1] = __uint_as_float(u[k] & 0xFFFF0000u);
    }
  }
  __device__ static __forceinline__ float at(const uint16_t* p, size_t i) {
    return __uint_as_float(static_cast<uint32_t>(p[i]) << 16);
  }
};

// ------------------------------------------------------------- group reductions
// Named barrier 1 + g synchronises the kGroupThreads threads of group g.
__device__ __forceinline__ void group_sync(int g) {
  asm volatile("bar.sync %0, %1;" ::"r"(g + 1), "r"(kGroupThreads) : "memory");
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}
__device__ __forceinline__ int warp_min_i(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}
__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long w = __shfl_xor_sync(0xFFFFFFFFu, v, o);
    v = w > v ? w : v;
  }
  return v;
}

// scratch: kGroupWarps 8-byte slots owned by the group.
__device__ __forceinline__ float group_max(float v, int g, unsigned long long* scratch) {
  v = warp_max(v);
  const int w = (threadIdx.x >> 5) & (kGroupWarps - 1);
  if ((threadIdx.x & 31) == 0) reinterpret_cast<float*>(scratch)[2 * w] = v;
  group_sync(g);
  float r = reinterpret_cast<float*>(scratch)[0];
#pragma unroll
  for (int k = 1; k < kGroupWarps; ++k) r = fmaxf(r, reinterpret_cast<float*>(scratch)[2 * k]);
  group_sync(g);
  return r;
}
__device__ __forceinline__ float group_sum(float v, int g, unsigned long long* scratch) {
  v = warp_sum(v);
  const int w = (threadIdx.x >> 5) & (kGroupWarps - 1);
  if ((threadIdx.x & 31) == 0) reinterpret_cast<float*>(scratch)[2 * w] = v;
  group_sync(g);
  float r = reinterpret_cast<float*>(scratch)[0];
#pragma unroll
  for (int k = 1; k < kGroupWarps; ++k) r += reinterpret_cast<float*>(scratch)[2 * k];
  group_sync(g);
  return r;
}
__device__ __forceinline__ int group_min_i(int v, int g, unsigned long long* scratch) {
  v = warp_min_i(v);
  const int w = (threadIdx.x >> 5) & (kGroupWarps - 1);
  if ((threadIdx.x & 31) == 0) reinterpret_cast<int*>(scratch)[2 * w] = v;
  group_sync(g);
  int r = reinterpret_cast<int*>(scratch)[0];
#pragma unroll
  for (int k = 1; k < kGroupWarps; ++k) r = min(r, reinterpret_cast<int*>(scratch)[2 * k]);
  group_sync(g);
  return r;
}
__device__ __forceinline__ unsigned long long group_max_u64(unsigned long long v, int g,
                                                            unsigned long long* scratch) {
  v = warp_max_u64(v);
  const int w = (threadIdx.x >> 5) & (kGroupWarps - 1);
  if ((threadIdx.x & 31) == 0) scratch[w] = v;
  group_sync(g);
  unsigned long long r = scratch[0];
#pragma unroll
  for (int k = 1; k < kGroupWarps; ++k) r = scratch[k] > r ? scratch[k] : r;
  group_sync(g);
  return r;
}

__device__ __forceinline__ unsigned long long pack_key(uint32_t key_bits, int idx) {
  return (static_cast<unsigned long long>(key_bits) << 32) |
         static_cast<unsigned long long>(0xFFFFFFFFu - static_cast<uint32_t>(idx));
}
__device__ __forceinline__ int unpack_index(unsigned long long packed) {
  return static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(packed & 0xFFFFFFFFull));
}

// Request parameters as every part of the kernel derives them.
struct ReqInfo {
  int L_raw, L;
  float T, c;
  bool greedy;
};
__device__ __forceinline__ ReqInfo req_info(const PArgs& A, int b) {
  ReqInfo r;
  r.L_raw = A.draft_len[b];
  r.L = min(max(r.L_raw, 0), A.n_max);
  r.T = A.temperature[b];
  r.greedy = !(r.T > 0.f) || r.T < 1e-6f || A.draft == nullptr;
  const float s = 1.0f / r.T;
  r.c = s * 1.4426950408889634f;  // log2(e) / T
  return r;
}


// ------------------------------------------------------------- bookkeeping
// Everything below runs on one thread.  Partial results are published with a
// fence before the counter that announces them; whoever observes the final
// count fences again before reading them (the last-arriver pattern).

__device__ __forceinline__ void enqueue_race(const PArgs& A, int b, int round) {
  const uint32_t base = atomicAdd(&A.ctr[2], static_cast<uint32_t>(A.nrc));
  for (int k = 0; k < A.nrc; ++k)
    ptx::st_release_u32(&A.race_q[base + k], kJobValid | (static_cast<uint32_t>(k) << 24) |
                                                 (static_cast<uint32_t>(round) << 23) |
                                                 static_cast<uint32_t>(b));
}

__device__ __forceinline__ void write_outputs(const PArgs& A, int b, int a, int y) {
  const int rows = A.n_max + 1;
  A.accepted_len[b] = a;
  int32_t* out = A.out_tokens + static_cast<size_t>(b) * rows;
  for (int k = 0; k < rows; ++k)
    out[k] = k < a ? A.draft_tokens[static_cast<size_t>(b) * A.n_max + k] : (k == a ? y : -1);
}

// The last row of request b is in: find the first rejection.
__device__ void request_finalize(const PArgs& A, int b) {
  __threadfence();
  const ReqInfo q = req_info(A, b);
  const int rows = A.n_max + 1;
  uint32_t errbits = 0;
  if (q.L_raw != q.L) errbits |= SPECDEC_DEV_ERR_DRAFT_LEN;
  if (q.greedy && q.T != 0.f) errbits |= SPECDEC_DEV_ERR_TEMPERATURE;
  int a = q.L;
  for (int jj = 0; jj < q.L; ++jj) {
    const size_t r = static_cast<size_t>(b) * rows + jj;
    const int x = A.draft_tokens[static_cast<size_t>(b) * A.n_max + jj];
    const bool valid = x >= 0 && x < A.V;
    if (!valid) errbits |= SPECDEC_DEV_ERR_TOKEN;
    const bool ok = q.greedy ? (valid && x == __ldcg(&A.row_arg[r])) : (__ldcg(&A.row_acc[r]) != 0u);
    if (!ok) {
      a = jj;
      break;
    }
  }
  if (errbits) atomicOr(A.err, errbits);
  A.req_cnt[b] = 0u;
  if (q.greedy) {
    write_outputs(A, b, a, __ldcg(&A.row_arg[static_cast<size_t>(b) * rows + a]));
    __threadfence();
    atomicAdd(&A.ctr[3], 1u);
    return;
  }
  A.race_row[b] = a;
  A.race_P[b] = __ldcg(&A.row_P[static_cast<size_t>(b) * rows + a]);
  __threadfence();
  enqueue_race(A, b, 0);
}

// The last chunk of row (b, j) is in: combine the partials.
template <typename Elt>
__device__ void row_combine(const PArgs& A, int b, int j) {
  __threadfence();
  const ReqInfo q = req_info(A, b);
  const int rows = A.n_max + 1;
  const size_t row = static_cast<size_t>(b) * rows + j;
  const float2* pt = A.part + (row * 2 + 0) * A.nch;
  if (q.greedy) {
    float bv = -INFINITY;
    int bi = 0;
    for (int k = 0; k < A.nch; ++k) {  // chunks in vocab order: ties keep the earlier one
      const float2 p = __ldcg(&pt[k]);
      if (k == 0 || p.x > bv) {
        bv = p.x;
        bi = __float_as_int(p.y);
      }
    }
    A.row_arg[row] = bi;
  } else {
    float Pt, Pd = 0.f;
    {
      float K = -INFINITY, S = 0.f;
      for (int k = 0; k < A.nch; ++k) K = fmaxf(K, __ldcg(&pt[k]).x);
      for (int k = 0; k < A.nch; ++k) {
        const float2 p = __ldcg(&pt[k]);
        if (p.y > 0.f) S += p.y * exp2f(p.x - K);
      }
      Pt = K + log2f(S);
    }
    const bool has_draft = j < q.L;
    if (has_draft) {
      const float2* pd = A.part + (row * 2 + 1) * A.nch;
      float K = -INFINITY, S = 0.f;
      for (int k = 0; k < A.nch; ++k) K = fmaxf(K, __ldcg(&pd[k]).x);
      for (int k = 0; k < A.nch; ++k) {
        const float2 p = __ldcg(&pd[k]);
        if (p.y > 0.f) S += p.y * exp2f(p.x - K);
      }
      Pd = K + log2f(S);
    }
    A.row_P[row] = make_float2(Pt, Pd);
    if (A.row_lse != nullptr) {
      A.row_lse[row * 2 + 0] = Pt * 0.69314718055994531f;
      if (has_draft) A.row_lse[row * 2 + 1] = Pd * 0.69314718055994531f;
    }
    if (has_draft) {
      uint32_t accept = 0;
      const int x = A.draft_tokens[static_cast<size_t>(b) * A.n_max + j];
      if (x >= 0 && x < A.V) {
        const size_t row_d = static_cast<size_t>(b) * A.n_max + j;
        const float tx = EltOps<Elt>::at(static_cast<const Elt*>(A.target), row * A.V + x);
        const float dx = EltOps<Elt>::at(static_cast<const Elt*>(A.draft), row_d * A.V + x);
        const float l2ratio = fmaf(tx, q.c, -Pt) - fmaf(dx, q.c, -Pd);  // log2 p(x) - log2 q(x)
        const Philox4 r = philox4x32_10(0u, static_cast<uint32_t>(j), static_cast<uint32_t>(b), 0u,
                                        A.seed_lo, A.seed_hi);
        accept = uniform_from_word(r.w[0]) < exp2f(l2ratio) ? 1u : 0u;
      }
      A.row_acc[row] = accept;
    }
  }
  A.row_cnt[row] = 0u;
  __threadfence();
  if (atomicAdd(&A.req_cnt[b], 1u) == static_cast<uint32_t>(q.L)) request_finalize(A, b);
}

// The last race chunk of request b is in.
__device__ void race_finalize(const PArgs& A, int b, int round) {
  __threadfence();
  const unsigned long long best = ptx::ld_relaxed_u64(&A.race_best[b]);
  const int a = __ldcg(&A.race_row[b]);
  const ReqInfo q = req_info(A, b);
  A.race_cnt[b] = 0u;
  if (best == 0ull && a < q.L && round == 0) {
    // Every residual weight vanished in fp32: race on p instead.
    __threadfence();
    enqueue_race(A, b, 1);
    return;
  }
  A.race_best[b] = 0ull;
  write_outputs(A, b, a, unpack_index(best));
  __threadfence();
  atomicAdd(&A.ctr[3], 1u);
}


// ------------------------------------------------------------- producer
// One thread (lane 0 of warp 0).
template <typename Elt, bool kDirect>
__device__ void producer(const PArgs& A, unsigned char* stages, ItemDesc* desc, uint64_t* full,
                         uint64_t* empty) {
  int stage = 0;
  uint32_t phase = 0;
  const int rows = A.n_max + 1;
  const uint32_t per_req = static_cast<uint32_t>(2 * A.n_max + 1);
  const uint64_t pol_first = ptx::policy_evict_first();
  uint32_t next = atomicAdd(&A.ctr[0], 1u);
  long long idle = 0;
  bool ok = true;

  auto acquire = [&]() -> bool {
    if (ptx::mbar_wait_bounded(ptx::smem_addr(&empty[stage]), phase ^ 1u, kWaitBudgetCycles)) return true;
    atomicOr(A.err, SPECDEC_DEV_ERR_TIMEOUT);
    return false;
  };
  auto advance = [&]() {
    if (++stage == kStages) {
      stage = 0;
      phase ^= 1u;
    }
  };

  while (ok) {
    // 1. queued race jobs first (their rows are still in L2)
    const uint32_t rh = ptx::ld_relaxed_u32(&A.ctr[1]);
    if (rh < ptx::ld_relaxed_u32(&A.ctr[2])) {
      const uint32_t job = ptx::ld_acquire_u32(&A.race_q[rh]);
      if (job & kJobValid) {
        if (atomicCAS(&A.ctr[1], rh, rh + 1u) == rh) {
          ptx::st_relaxed_u32(&A.race_q[rh], 0u);
          idle = 0;
          const int b = static_cast<int>(job & 0x7FFFFFu);
          const int round = static_cast<int>((job >> 23) & 1u);
          const int k = static_cast<int>((job >> 24) & 0x7Fu);
          const ReqInfo q = req_info(A, b);
          const int a = __ldcg(&A.race_row[b]);
          const float2 P = __ldcg(&A.race_P[b]);
          const bool residual = a < q.L && round == 0;
          if (!acquire()) {
            ok = false;
            break;
          }
          ItemDesc& d = desc[stage];
          d.kind = kItemRace;
          d.b = b;
          d.j = a;
          d.e0 = k * A.chr;
          d.n = min(A.chr, A.V - d.e0);
          d.chunk = k;
          d.c = q.c;
          d.Pt = P.x;
          d.Pd = P.y;
          d.residual = residual;
          d.round = round;
          const uint32_t bar = ptx::smem_addr(&full[stage]);
          if (kDirect) {
            ptx::mbar_arrive(bar);
          } else {
            const uint32_t bytes = static_cast<uint32_t>(d.n) * sizeof(Elt);
            unsigned char* buf = stages + static_cast<size_t>(stage) * kStageBytes;
            const Elt* gt = static_cast<const Elt*>(A.target) + (static_cast<size_t>(b) * rows + a) * A.V + d.e0;
            ptx::mbar_arrive_expect_tx(bar, residual ? 2 * bytes : bytes);
            ptx::bulk_g2s(ptx::smem_addr(buf), gt, bytes, bar, pol_first);
            if (residual) {
              const Elt* gd = static_cast<const Elt*>(A.draft) + (static_cast<size_t>(b) * A.n_max + a) * A.V + d.e0;
              ptx::bulk_g2s(ptx::smem_addr(buf + kStageBytes / 2), gd, bytes, bar, pol_first);
            }
          }
          advance();
        }
        continue;
      }
    }
    // 2. the next row-tensor unit
    if (next < A.n_units) {
      const uint32_t u = next;
      next = atomicAdd(&A.ctr[0], 1u);  // claim ahead: its latency overlaps this unit
      idle = 0;
      const int b = static_cast<int>(u / per_req);
      const int r = static_cast<int>(u % per_req);
      const ReqInfo q = req_info(A, b);
      const int tensor = r < rows ? 0 : 1;
      const int j = tensor == 0 ? r : r - rows;
      const bool valid = tensor == 0 ? (j <= q.L) : (!q.greedy && j < q.L);
      if (!valid) continue;  // ragged: rows beyond n_b are never read
      const int expect = A.nch * ((!q.greedy && j < q.L) ? 2 : 1);
      const size_t row = tensor == 0 ? static_cast<size_t>(b) * rows + j : static_cast<size_t>(b) * A.n_max + j;
      const Elt* src = static_cast<const Elt*>(tensor == 0 ? A.target : A.draft) + row * A.V;
      for (int k = 0; k < A.nch; ++k) {
        if (!acquire()) {
          ok = false;
          break;
        }
        ItemDesc& d = desc[stage];
        d.kind = kItemStream;
        d.b = b;
        d.j = j;
        d.tensor = tensor;
        d.e0 = k * A.ch;
        d.n = min(A.ch, A.V - d.e0);
        d.chunk = k;
        d.greedy = q.greedy;
        d.c = q.c;
        d.expect = expect;
        const uint32_t bar = ptx::smem_addr(&full[stage]);
        if (kDirect) {
          ptx::mbar_arrive(bar);
        } else {
          const uint32_t bytes = static_cast<uint32_t>(d.n) * sizeof(Elt);
          ptx::mbar_arrive_expect_tx(bar, bytes);
          ptx::bulk_g2s_nohint(ptx::smem_addr(stages + static_cast<size_t>(stage) * kStageBytes),
                               src + d.e0, bytes, bar);
        }
        advance();
      }
      continue;
    }
    // 3. nothing to claim: wait for the last race jobs, or leave.
    if (ptx::ld_relaxed_u32(&A.ctr[3]) >= static_cast<uint32_t>(A.B)) break;
    ptx::nanosleep(256);
    if (++idle > kIdlePollLimit) {
      atomicOr(A.err, SPECDEC_DEV_ERR_TIMEOUT);
      break;
    }
  }
  // One exit marker per consumer group: the next kGroups stages.
  for (int g = 0; g < kGroups; ++g) {
    if (!acquire()) break;
    desc[stage].kind = kItemExit;
    ptx::mbar_arrive(ptx::smem_addr(&full[stage]));
    advance();
  }
}


// ------------------------------------------------------------- consumers
template <typename Elt, bool kDirect>
__device__ void consumer(const PArgs& A, int g, unsigned char* stages, const ItemDesc* desc,
                         uint64_t* full, uint64_t* empty, unsigned long long* scratch) {
  using Ops = EltOps<Elt>;
  constexpr int VEC = Ops::kVec;
  const int gt = static_cast<int>(threadIdx.x) - 32 - g * kGroupThreads;
  const int rows = A.n_max + 1;
  int stage = g;
  uint32_t phase = 0;
  while (true) {
    if (!ptx::mbar_wait_bounded(ptx::smem_addr(&full[stage]), phase, kWaitBudgetCycles)) {
      if (gt == 0) atomicOr(A.err, SPECDEC_DEV_ERR_TIMEOUT);
      break;
    }
    const ItemDesc d = desc[stage];
    if (d.kind == kItemExit) break;
    const unsigned char* buf = stages + static_cast<size_t>(stage) * kStageBytes;
    const uint4* vbuf = reinterpret_cast<const uint4*>(buf);
    const int nvec = kDirect ? 0 : d.n / VEC;

    if (d.kind == kItemStream) {
      const size_t grow = d.tensor == 0 ? static_cast<size_t>(d.b) * rows + d.j
                                        : static_cast<size_t>(d.b) * A.n_max + d.j;
      const Elt* gsrc = static_cast<const Elt*>(d.tensor == 0 ? A.target : A.draft) + grow * A.V + d.e0;
      // chunk maximum
      typename Ops::MaxAcc macc = Ops::max_init();
      for (int vi = gt; vi < nvec; vi += kGroupThreads) Ops::max_vec(vbuf[vi], macc);
      float m = Ops::max_value(macc);
      if (kDirect)
        for (int e = gt; e < d.n; e += kGroupThreads) m = fmaxf(m, Ops::at(gsrc, e));
      const float M = group_max(m, g, scratch + g * kGroupWarps);
      float2 res;
      if (d.greedy) {
        int first = 0x7FFFFFFF;
        for (int vi = gt; vi < nvec && first == 0x7FFFFFFF; vi += kGroupThreads) {
          float f[VEC];
          Ops::unpack(vbuf[vi], f);
#pragma unroll
          for (int i = VEC - 1; i >= 0; --i)
            if (f[i] == M) first = vi * VEC + i;
        }
        if (kDirect)
          for (int e = gt; e < d.n && first == 0x7FFFFFFF; e += kGroupThreads)
            if (Ops::at(gsrc, e) == M) first = e;
        first = group_min_i(first, g, scratch + g * kGroupWarps);
        res = make_float2(M, __int_as_float(d.e0 + first));
      } else {
        const float K = M * d.c;
        float2 acc = make_float2(0.f, 0.f);
        const float2 cc = make_float2(d.c, d.c), nk = make_float2(-K, -K);
        for (int vi = gt; vi < nvec; vi += kGroupThreads) Ops::sum_vec(vbuf[vi], cc, nk, acc);
        if (kDirect)
          for (int e = gt; e < d.n; e += kGroupThreads) acc.x += fast_ex2(fmaf(Ops::at(gsrc, e), d.c, -K));
        const float S = group_sum(acc.x + acc.y, g, scratch + g * kGroupWarps);
        res = make_float2(K, S);
      }
      if (gt == 0) {
        ptx::mbar_arrive(ptx::smem_addr(&empty[stage]));  // the group is done with the stage
        const size_t row = static_cast<size_t>(d.b) * rows + d.j;
        A.part[(row * 2 + d.tensor) * A.nch + d.chunk] = res;
        __threadfence();
        if (atomicAdd(&A.row_cnt[row], 1u) == static_cast<uint32_t>(d.expect - 1))
          row_combine<Elt>(A, d.b, d.j);
      }
    } else {
      // ------------------------------------------------ race over one chunk of row a
      const Elt* gt_src = static_cast<const Elt*>(A.target) + (static_cast<size_t>(d.b) * rows + d.j) * A.V + d.e0;
      const Elt* gd_src = static_cast<const Elt*>(A.draft) + (static_cast<size_t>(d.b) * A.n_max + d.j) * A.V + d.e0;
      const uint4* vd = reinterpret_cast<const uint4*>(buf + kStageBytes / 2);
      float R = 0.f, Eb = 1.f;
      int idx = -1;
      for (int vi = gt; vi < nvec; vi += kGroupThreads) {
        float ft[VEC], fd[VEC];
        Ops::unpack(vbuf[vi], ft);
        if (d.residual) Ops::unpack(vd[vi], fd);
        const int v = d.e0 + vi * VEC;
#pragma unroll
        for (int q4 = 0; q4 < VEC / 4; ++q4) {
          const Philox4 rnd = philox4x32_10(static_cast<uint32_t>(v + 4 * q4) >> 2, static_cast<uint32_t>(d.j),
                                            static_cast<uint32_t>(d.b), 1u, A.seed_lo, A.seed_hi);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int e = 4 * q4 + i;
            float r = fast_ex2(fmaf(ft[e], d.c, -d.Pt));
            if (d.residual) r -= fast_ex2(fmaf(fd[e], d.c, -d.Pd));
            if (r > 0.f) {
              const float U = uniform_from_word(rnd.w[i]);
              // -ln U >= 1 - U: r / (1 - U) bounds the key r / E from above,
              // so only a possible winner pays for the logarithm.
              if (r * Eb > R * (1.0f - U)) {
                const float E = -logf(U);
                if (r * Eb > R * E) {
                  R = r;
                  Eb = E;
                  idx = v + e;
                }
              }
            }
          }
        }
      }
      if (kDirect) {
        for (int e = gt; e < d.n; e += kGroupThreads) {
          const int v = d.e0 + e;
          float r = fast_ex2(fmaf(Ops::at(gt_src, e), d.c, -d.Pt));
          if (d.residual) r -= fast_ex2(fmaf(Ops::at(gd_src, e), d.c, -d.Pd));
          if (r > 0.f) {
            const Philox4 rnd = philox4x32_10(static_cast<uint32_t>(v) >> 2, static_cast<uint32_t>(d.j),
                                              static_cast<uint32_t>(d.b), 1u, A.seed_lo, A.seed_hi);
            const float E = -logf(uniform_from_word(rnd.w[v & 3]));
            if (r * Eb > R * E) {
              R = r;
              Eb = E;
              idx = v;
            }
          }
        }
      }
      const unsigned long long mine = idx >= 0 ? pack_key(__float_as_uint(R / Eb), idx) : 0ull;
      const unsigned long long best = group_max_u64(mine, g, scratch + g * kGroupWarps);
      if (gt == 0) {
        ptx::mbar_arrive(ptx::smem_addr(&empty[stage]));
        if (best != 0ull) atomicMax(&A.race_best[d.b], best);
        __threadfence();
        if (atomicAdd(&A.race_cnt[d.b], 1u) == static_cast<uint32_t>(A.nrc - 1)) race_finalize(A, d.b, d.round);
      }
    }
    stage += kGroups;
    if (stage >= kStages) {
      stage -= kStages;
      phase ^= 1u;
    }
  }
}

// ------------------------------------------------------------- the kernel
template <typename Elt, bool kDirect>
__global__ void __launch_bounds__(kThreads, 1) verify_persistent_kernel(const PArgs A) {
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char* stages = smem;
  ItemDesc* desc = reinterpret_cast<ItemDesc*>(smem + kStages * kStageBytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(desc + kStages);
  uint64_t* empty = full + kStages;
  unsigned long long* scratch = reinterpret_cast<unsigned long long*>(empty + kStages);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(ptx::smem_addr(&full[s]), 1);
      ptx::mbar_init(ptx::smem_addr(&empty[s]), 1);
    }
    ptx::fence_mbarrier_init();
  }
  __syncthreads();
  const int warp = static_cast<int>(threadIdx.x >> 5);
  if (warp == 0) {
    if ((threadIdx.x & 31) == 0) producer<Elt, kDirect>(A, stages, desc, full, empty);
  } else {
    consumer<Elt, kDirect>(A, (warp - 1) / kGroupWarps, stages, desc, full, empty, scratch);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // The last CTA out re-arms the queue counters for the next call.
    __threadfence();
    if (atomicAdd(&A.ctr[4], 1u) == gridDim.x - 1) {
      for (int k = 0; k < 5; ++k) A.ctr[k] = 0u;
      __threadfence();
    }
  }
}

constexpr size_t kPersistentSmemBytes =
    static_cast<size_t>(kStages) * kStageBytes + kStages * sizeof(ItemDesc) + 2 * kStages * sizeof(uint64_t) +
    kGroups * kGroupWarps * sizeof(unsigned long long);

}  // namespace specdec
