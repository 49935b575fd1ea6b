// verify_persistent.cuh — persistent, warp-specialised verify/accept kernel
// for sm_103a (one CTA per SM).
//
// Work is a stream of segments (kSegChunks chunks) of row-tensor units
// (request b, target row j or draft row j), in request-major order, claimed
// from a device counter, so requests finish in order.  Per CTA:
//   * each consumer group owns a ring of kStagesPerGroup shared-memory stages
//     and a producer warp that streams the group's current segment into it,
//     kStageBytes at a time, with 1-D bulk copies (TMA engine); each stage has
//     a "full" mbarrier (bytes landed) and an "empty" mbarrier (every warp of
//     the group is done with it);
//   * a consumer group reduces its segment with running per-thread state —
//     (max, sum 2^(x c - K)) for sampled requests, (max, first index of the
//     max) for greedy ones, c = log2(e)/T — and publishes one partial per
//     segment;
//   * the segment that completes a row combines the row's partials into its
//     log-sum-exp and runs the acceptance test u_j < p_j(x_j)/q_j(x_j); the row
//     that completes a request finds the first rejection a (or a = n_b) and
//     either writes the greedy result or queues the exponential race over row
//     a as chunk jobs; this bookkeeping runs on one warp, lanes in parallel;
//   * a producer with no segment left serves queued race jobs: each re-reads
//     a piece of row a (target, plus draft when a < n_b), and the race runs
//     exactly once per request.
// No CTA waits for another CTA's progress except a producer's bounded poll for
// queued race jobs once no segment is left; every wait is bounded.  Race jobs
// are claimed by fetch-and-add (no compare-and-swap retries).
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
constexpr int kProducerWarps = kGroups;                 // one producer warp per group
constexpr int kThreads = 32 * kProducerWarps + kGroups * kGroupThreads;
constexpr int kStagesPerGroup = 2;
constexpr int kStages = kGroups * kStagesPerGroup;
constexpr int kStageBytes = 28 * 1024;  // shared-memory capacity of a stage
constexpr int kSegChunks = 3;                          // chunks per published partial
constexpr long long kWaitBudgetCycles = 4000000000LL;  // ~2 s of SM clock

// Device counters, each on its own 128-byte line (u32 indices).
constexpr int kCtrUnit = 0, kCtrRaceHead = 32, kCtrRaceTail = 64, kCtrDone = 96, kCtrExit = 128;
constexpr int kCtrReadBytes = 160;  // early exit: u64 logits bytes read, summed over calls until read
constexpr int kCtrWords = 192;

enum : uint32_t { kItemStream = 1u, kItemRace = 2u, kItemExit = 3u };
enum : int { kFirst = 1, kLast = 2, kGreedy = 4 };
// race job word: valid | chunk << 23 | round << 22 | b
constexpr uint32_t kJobValid = 0x80000000u;

struct ItemDesc {  // one per stage, written by the producer
  uint32_t kind;
  int b, j;      // request, row within the request (race: row a)
  int tensor;    // stream: 0 target, 1 draft
  int e0, n;     // first vocab index and element count of the chunk
  int seg;       // stream: segment index within the row-tensor; race: chunk index
  int flags;     // stream: kFirst | kLast | kGreedy
  int x;         // stream: draft token of the row (-1 if none or greedy)
  int trow;      // stream: row of the streamed tensor; race: target row of a
  float c;       // log2(e) / T
  float Pt, Pd;  // race: log2 normalisers of row a
  int residual;  // race: r = max(0, p - q) (else r = p)
  int round;     // race: 0, or 1 for the fallback on p
  int expect;    // stream: segments that complete the row (both tensors); race: jobs of the race
  int drow;      // race: draft row of a
  uint32_t rword;  // race: row word of the race's random counter (position offset + a)
  int pad[2];
};
static_assert(sizeof(ItemDesc) == 80, "descriptor layout");

struct PArgs {
  const void* target;
  const void* draft;
  const int32_t* draft_tokens;
  const int32_t* draft_len;   // dense layout: [B]
  const int32_t* cu_rows;     // packed layout: [B + 1] first target row of each request (else null)
  const int32_t* pos_offset;  // [B] position offset of each request's random counter (or null)
  int total_rows;             // packed layout: rows of the target tensor
  const float* temperature;
  int32_t* accepted_len;
  int32_t* out_tokens;
  float* row_lse;
  uint32_t seed_lo, seed_hi;
  int B, n_max, V;
  int nch;        // stream chunks per row-tensor
  int ch;         // elements per stream chunk
  int nseg;       // segments per row-tensor
  int nrc;        // race chunks per row
  int chr;        // elements per race chunk
  uint32_t n_units;   // B * (2 n_max + 1) row-tensor units
  uint32_t n_claims;  // n_units * nseg segments, claimed one at a time
  // workspace
  uint32_t* err;
  uint32_t* ctr;                    // [kCtrWords]
  uint32_t* race_q;                 // [2 * B * nrc]
  uint32_t* req_cnt;                // [B]
  unsigned long long* race_best;    // [B]
  uint32_t* race_cnt;               // [B]
  float4* race_desc;                // [B] (Pt, Pd, c, a | residual << 16)
  int4* race_rows;                  // [B] (first target row, first draft row, position offset, n_b)
  uint32_t* row_cnt;                // [B * rows]
  float2* row_P;                    // [B * rows]
  int32_t* row_arg;                 // [B * rows]
  uint32_t* row_acc;                // [B * rows]
  float2* part;                     // [B * rows * 2 * nseg]
  float2* row_x;                    // [B * rows] target / draft logit at the row's draft token
  // early exit only (zero between calls)
  uint32_t* rej_hi;                 // [B] max over rejected rows k of (n_max + 1 - k); 0: none yet
  uint32_t* row_done;               // [B] bit j: row j combined
  uint32_t* req_fin;                // [B] the request's outputs are claimed
};

// ------------------------------------------------------------- element types
__device__ __forceinline__ float fast_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float fast_rcp(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
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

// Request parameters as every part of the kernel derives them.  t0 and d0
// are the request's first row in the target and draft logits (and in the
// draft tokens and outputs): dense [B, n_max+1, V] / [B, n_max, V], or packed
// with target rows at cu_rows[b] + j and draft rows at cu_rows[b] - b + j.
// A packed segment that is empty or reaches outside the tensors is skipped
// (`skip`): nothing of it is read.
struct ReqInfo {
  int L_raw, L;
  int t0, d0;
  uint32_t o;  // position offset of the random counter's row word
  bool skip;
  float T, c;
  bool greedy;
};
__device__ __forceinline__ ReqInfo req_info(const PArgs& A, int b) {
  ReqInfo r;
  if (A.cu_rows != nullptr) {
    const int r0 = A.cu_rows[b], r1 = A.cu_rows[b + 1];
    r.t0 = r0;
    r.d0 = r0 - b;
    r.L_raw = r1 - r0 - 1;
    r.skip = r1 - r0 < 1 || r0 < 0 || r1 > A.total_rows || r.d0 < 0;
  } else {
    r.t0 = b * (A.n_max + 1);
    r.d0 = b * A.n_max;
    r.L_raw = A.draft_len[b];
    r.skip = false;
  }
  r.o = A.pos_offset != nullptr ? static_cast<uint32_t>(A.pos_offset[b]) : 0u;
  r.L = min(max(r.L_raw, 0), A.n_max);
  // packed: the draft rows d0 .. d0 + L - 1 must lie below total_rows - B
  if (A.cu_rows != nullptr && r.d0 + r.L > A.total_rows - A.B) r.skip = true;
  r.T = A.temperature[b];
  // without draft logits only a request with no drafts can sample
  r.greedy = !(r.T > 0.f) || r.T < 1e-6f || (A.draft == nullptr && r.L > 0);
  const float s = 1.0f / r.T;
  r.c = s * 1.4426950408889634f;  // log2(e) / T
  return r;
}


// ------------------------------------------------------------- bookkeeping
// Called by all 32 lanes of one warp together.  Partial results are published
// with a fence before the counter that announces them; whoever observes the
// final count fences again before reading them (the last-arriver pattern).

__device__ __forceinline__ int lane_id() { return static_cast<int>(threadIdx.x & 31); }

// Race jobs of a race: a residual race reads half a stage of target and
// half of draft per job; a race on p (the bonus row, or the fallback) reads
// a whole stage of target.
__device__ __forceinline__ int race_job_elems(const PArgs& A, bool residual) { return residual ? A.chr : 2 * A.chr; }
__device__ __forceinline__ int race_jobs(const PArgs& A, bool residual) {
  const int js = race_job_elems(A, residual);
  return (A.V + js - 1) / js;
}
static __device__ void enqueue_race_w(const PArgs& A, int b, int round, int njobs) {
  uint32_t base = 0;
  if (lane_id() == 0) base = atomicAdd(&A.ctr[kCtrRaceTail], static_cast<uint32_t>(njobs));
  base = __shfl_sync(0xFFFFFFFFu, base, 0);
  for (int k = lane_id(); k < njobs; k += 32)
    ptx::st_release_u32(&A.race_q[base + k], kJobValid | (static_cast<uint32_t>(k) << 23) |
                                                 (static_cast<uint32_t>(round) << 22) |
                                                 static_cast<uint32_t>(b));
}

// out_tokens of request b: a accepted drafts, then y, then -1 up to the
// request's last slot (n_max + 1 slots dense, n_b + 1 packed).
static __device__ void write_outputs_w(const PArgs& A, int b, int a, int y, int t0, int d0, int L) {
  const int slots = A.cu_rows != nullptr ? L + 1 : A.n_max + 1;
  if (lane_id() == 0) A.accepted_len[b] = a;
  int32_t* out = A.out_tokens + static_cast<size_t>(t0);
  for (int k = lane_id(); k < slots; k += 32)
    out[k] = k < a ? A.draft_tokens[static_cast<size_t>(d0) + k] : (k == a ? y : -1);
}

static __device__ void request_finish_w(const PArgs& A, int b, const ReqInfo& q, int a, bool bad_token);

// The last row of request b is in: find the first rejection.
static __device__ void request_finalize_w(const PArgs& A, int b, const ReqInfo& q) {
  __syncwarp();  // lane 0's acquire (the count that elected this warp) covers the whole warp
  const int rows = A.n_max + 1;
  const int lane = lane_id();
  int a = q.L;
  bool bad_token = false;
  for (int base = 0; base < q.L; base += 32) {
    const int jj = base + lane;
    bool fail = false, bad = false;
    if (jj < q.L) {
      const size_t r = static_cast<size_t>(b) * rows + jj;
      const int x = A.draft_tokens[static_cast<size_t>(q.d0) + jj];
      const bool valid = x >= 0 && x < A.V;
      bad = !valid;
      fail = q.greedy ? !(valid && x == __ldcg(&A.row_arg[r])) : (__ldcg(&A.row_acc[r]) == 0u);
    }
    const uint32_t fm = __ballot_sync(0xFFFFFFFFu, fail);
    if (fm) {
      a = base + __ffs(fm) - 1;
      // an invalid token always fails its row, so only row a can carry one
      bad_token = __shfl_sync(0xFFFFFFFFu, bad, __ffs(fm) - 1);
      break;
    }
  }
  if (lane == 0) A.req_cnt[b] = 0u;
  request_finish_w(A, b, q, a, bad_token);
}

// Request b's first rejection is row a (a = n_b: every draft accepted):
// write the greedy result, or queue the race over row a.
static __device__ void request_finish_w(const PArgs& A, int b, const ReqInfo& q, int a, bool bad_token) {
  const int rows = A.n_max + 1;
  const int lane = lane_id();
  if (lane == 0) {
    uint32_t errbits = bad_token ? SPECDEC_DEV_ERR_TOKEN : 0u;
    if (q.L_raw != q.L) errbits |= SPECDEC_DEV_ERR_DRAFT_LEN;
    if (q.greedy && q.T != 0.f) errbits |= SPECDEC_DEV_ERR_TEMPERATURE;
    if (errbits) atomicOr(A.err, errbits);
  }
  if (q.greedy) {
    write_outputs_w(A, b, a, __ldcg(&A.row_arg[static_cast<size_t>(b) * rows + a]), q.t0, q.d0, q.L);
    __syncwarp();
    if (lane == 0) atomicAdd(&A.ctr[kCtrDone], 1u);
    return;
  }
  if (lane == 0) {
    const float2 P = __ldcg(&A.row_P[static_cast<size_t>(b) * rows + a]);
    const uint32_t tag = static_cast<uint32_t>(a) | ((a < q.L ? 1u : 0u) << 16);
    A.race_desc[b] = make_float4(P.x, P.y, q.c, __uint_as_float(tag));
    A.race_rows[b] = make_int4(q.t0, q.d0, static_cast<int>(q.o), q.L);
    __threadfence();
  }
  __syncwarp();
  enqueue_race_w(A, b, 0, race_jobs(A, a < q.L));
}

// Early exit: row j of request b is combined.  Record a rejection (so later
// rows are not claimed), mark the row done, and finish the request once its
// rows 0..k decide it: rows 0..k-1 accepted and row k rejected, or every
// draft accepted and the bonus row done.  One warp, lanes in parallel (lane k
// looks at row k; n_max < 32).
static __device__ void row_decide_w(const PArgs& A, int b, int j, const ReqInfo& q) {
  const int rows = A.n_max + 1;
  const int lane = lane_id();
  const size_t r0 = static_cast<size_t>(b) * rows;
  auto accepted = [&](int k) -> bool {
    const int x = A.draft_tokens[static_cast<size_t>(q.d0) + k];
    if (!(x >= 0 && x < A.V)) return false;
    return q.greedy ? x == __ldcg(&A.row_arg[r0 + k]) : __ldcg(&A.row_acc[r0 + k]) != 0u;
  };
  uint32_t done = 0;
  if (lane == 0) {
    if (j < q.L && !accepted(j)) atomicMax(&A.rej_hi[b], static_cast<uint32_t>(rows - j));
    done = ptx::atom_or_acq_rel(&A.row_done[b], 1u << j) | (1u << j);  // publishes the row's results
  }
  done = __shfl_sync(0xFFFFFFFFu, done, 0);
  __syncwarp();  // lane 0's acquire covers the rows the other lanes read
  const bool ok = lane < q.L && ((done >> lane) & 1u) && accepted(lane);
  const uint32_t okm = __ballot_sync(0xFFFFFFFFu, ok);
  const int k = __ffs(~okm) - 1;  // first row that is not a done, accepted draft row
  if (k > q.L || !((done >> k) & 1u)) return;  // undecided: row k is still streaming
  uint32_t won = 0;
  if (lane == 0) won = atomicExch(&A.req_fin[b], 1u) == 0u ? 1u : 0u;
  if (!__shfl_sync(0xFFFFFFFFu, won, 0)) return;  // another row finished it
  bool bad = false;
  if (k < q.L) {
    const int x = A.draft_tokens[static_cast<size_t>(q.d0) + k];
    bad = !(x >= 0 && x < A.V);
  }
  request_finish_w(A, b, q, k, bad);
}

// The last segment of row (b, j) is in: combine the partials.
template <typename Elt, bool kEarly>
__device__ void row_combine_w(const PArgs& A, int b, int j, const ReqInfo& q) {
  __syncwarp();  // lane 0's acquire (the count that elected this warp) covers the whole warp
  const int rows = A.n_max + 1;
  const int lane = lane_id();
  const size_t row = static_cast<size_t>(b) * rows + j;
  const float2* pt = A.part + (row * 2 + 0) * A.nseg;
  uint32_t count = 0;
  if (q.greedy) {
    float v = -INFINITY;
    int i = 0x7FFFFFFF;
    if (lane < A.nseg) {  // one partial per lane: the host keeps nseg <= 32
      const float2 p = __ldcg(&pt[lane]);
      v = p.x;
      i = __float_as_int(p.y);
    }
    const float best = warp_max(v);
    const int idx = warp_min_i(v == best ? i : 0x7FFFFFFF);  // lowest index among equal maxima
    if (lane == 0) A.row_arg[row] = idx;
  } else {
    // one partial per lane: the host keeps nseg <= 32
    const bool has_draft = j < q.L;
    const float2 none = make_float2(-INFINITY, 0.f);
    const float2 ptk = lane < A.nseg ? __ldcg(&pt[lane]) : none;
    const float2 pdk = (has_draft && lane < A.nseg) ? __ldcg(&A.part[(row * 2 + 1) * A.nseg + lane]) : none;
    const float Kt = warp_max(ptk.x);
    const float Kd = warp_max(pdk.x);
    const float St = warp_sum(ptk.y > 0.f ? ptk.y * exp2f(ptk.x - Kt) : 0.f);
    const float Sd = warp_sum(pdk.y > 0.f ? pdk.y * exp2f(pdk.x - Kd) : 0.f);
    if (lane == 0) {
      const float Pt = Kt + log2f(St);
      const float Pd = has_draft ? Kd + log2f(Sd) : 0.f;
      A.row_P[row] = make_float2(Pt, Pd);
      if (A.row_lse != nullptr) {
        const size_t orow = static_cast<size_t>(q.t0) + j;  // laid out like the target rows
        A.row_lse[orow * 2 + 0] = Pt * 0.69314718055994531f;
        if (has_draft) A.row_lse[orow * 2 + 1] = Pd * 0.69314718055994531f;
      }
      if (has_draft) {
        uint32_t accept = 0;
        const int x = A.draft_tokens[static_cast<size_t>(q.d0) + j];
        if (x >= 0 && x < A.V) {
          const float2 lx = __ldcg(&A.row_x[row]);  // saved by the streaming pass
          const float tx = lx.x, dx = lx.y;
          const float l2ratio = fmaf(tx, q.c, -Pt) - fmaf(dx, q.c, -Pd);  // log2 p(x) - log2 q(x)
          const Philox4 r = philox4x32_10(0u, q.o + static_cast<uint32_t>(j), static_cast<uint32_t>(b), 0u,
                                          A.seed_lo, A.seed_hi);
          accept = uniform_from_word(r.w[0]) < exp2f(l2ratio) ? 1u : 0u;
        }
        A.row_acc[row] = accept;
      }
    }
  }
  if constexpr (kEarly) {
    row_decide_w(A, b, j, q);
    return;
  }
  if (lane == 0) {
    A.row_cnt[row] = 0u;
    count = ptx::atom_add_acq_rel(&A.req_cnt[b], 1u);  // publishes the row's results
  }
  count = __shfl_sync(0xFFFFFFFFu, count, 0);
  if (count == static_cast<uint32_t>(q.L)) request_finalize_w(A, b, q);
}

// The last race chunk of request b is in.
static __device__ void race_finalize_w(const PArgs& A, int b, int round) {
  __syncwarp();  // lane 0's acquire (the count that elected this warp) covers the whole warp
  unsigned long long best = 0;
  float4 rd = make_float4(0.f, 0.f, 0.f, 0.f);
  if (lane_id() == 0) {
    best = ptx::ld_relaxed_u64(&A.race_best[b]);
    rd = __ldcg(&A.race_desc[b]);
    A.race_cnt[b] = 0u;
  }
  best = __shfl_sync(0xFFFFFFFFu, best, 0);
  const uint32_t tag = __shfl_sync(0xFFFFFFFFu, __float_as_uint(rd.w), 0);
  const int a = static_cast<int>(tag & 0xFFFFu);
  const bool residual = (tag >> 16) != 0u;
  if (best == 0ull && residual && round == 0) {
    // Every residual weight vanished in fp32: race on p instead.
    if (lane_id() == 0) __threadfence();
    __syncwarp();
    enqueue_race_w(A, b, 1, race_jobs(A, false));
    return;
  }
  if (lane_id() == 0) A.race_best[b] = 0ull;
  const int4 rr = __ldcg(&A.race_rows[b]);  // (first target row, first draft row, offset, n_b)
  write_outputs_w(A, b, a, unpack_index(best), rr.x, rr.y, rr.w);
  __syncwarp();
  if (lane_id() == 0) atomicAdd(&A.ctr[kCtrDone], 1u);
}


// ------------------------------------------------------------- producers
// Lane 0 of producer warp g feeds consumer group g's ring: a queued race job
// if there is one, else the next chunk of the group's unit, claiming a new
// unit when the current one is done.  Each group has its own producer, so a
// producer blocked on a global load delays only its own group.
template <typename Elt, bool kDirect, bool kEarly>
__device__ void producer(const PArgs& A, int g, unsigned char* stages, ItemDesc* desc, uint64_t* full,
                         uint64_t* empty) {
  const int rows = A.n_max + 1;
  const uint32_t per_req = static_cast<uint32_t>(2 * A.n_max + 1);
  const uint64_t pol_first = ptx::policy_evict_first();
  int s = 0;
  uint32_t phase = 0;
  bool active = false;
  int ub = 0, uj = 0, utensor = 0, ugreedy = 0, uexpect = 0, uk = 0, uk_end = 0, ux = -1, urow = 0;
  float uc = 0.f;
  const Elt* usrc = nullptr;
  // Each group's first segment is its own index; later ones come from the
  // counter.
  const uint32_t n_static = gridDim.x * kGroups;
  uint32_t next = blockIdx.x * kGroups + g;
  // A claimed race-queue slot not served yet.  Claims are fetch-and-add, so
  // a producer may claim a slot whose job is not queued yet: it serves the
  // job when it appears.  Such a slot is never left behind: a job in it keeps
  // its request unfinished, and the producer stays until every request is.
  uint32_t pend = 0xFFFFFFFFu;
  uint32_t rh = 0, rt = 0;
  bool last_was_race = false;  // the most recent item issued was a race job
  long long last_progress = clock64();
  bool failed = false;

  while (true) {
    const int stage = g * kStagesPerGroup + s;
    if (!ptx::mbar_wait_bounded(ptx::smem_addr(&empty[stage]), phase ^ 1u, kWaitBudgetCycles)) {
      failed = true;
      break;
    }
    ItemDesc& d = desc[stage];
    const uint32_t bar = ptx::smem_addr(&full[stage]);
    unsigned char* buf = stages + static_cast<size_t>(stage) * kStageBytes;
    bool fed = false;
    // 1. between segments: a queued race job.  Stream first: a producer takes
    //    race jobs only once no segment is left for it, so the queue never
    //    delays a segment (and the request it belongs to); the races fill
    //    the groups as streaming drains.  The queue counters are read only
    //    here, so the chunks of a segment go out back to back.  When fewer
    //    jobs are queued than there are groups, a group runs one race job at
    //    a time (while the item issued just before is a race job still being
    //    consumed, jobs are left to idle groups); otherwise a second job is
    //    prefetched behind the first.
    if (!active && next >= A.n_claims) {
      rh = ptx::ld_relaxed_u32(&A.ctr[kCtrRaceHead]);
      rt = ptx::ld_relaxed_u32(&A.ctr[kCtrRaceTail]);
      bool may_race = true;
      if (last_was_race && static_cast<int>(rt - rh) < static_cast<int>(gridDim.x) * kGroups) {
        const int prev = g * kStagesPerGroup + (s == 0 ? kStagesPerGroup - 1 : s - 1);
        may_race = ptx::mbar_test_wait(ptx::smem_addr(&empty[prev]), s == 0 ? (phase ^ 1u) : phase);
      }
      if (may_race && pend == 0xFFFFFFFFu && rh < rt) pend = atomicAdd(&A.ctr[kCtrRaceHead], 1u);
    }
    if (!active && pend != 0xFFFFFFFFu && pend < rt) {
      const uint32_t job = ptx::ld_acquire_u32(&A.race_q[pend]);
      if (job & kJobValid) {
        ptx::st_relaxed_u32(&A.race_q[pend], 0u);
        pend = 0xFFFFFFFFu;
        const int b = static_cast<int>(job & 0x3FFFFFu);
        const int round = static_cast<int>((job >> 22) & 1u);
        const int k = static_cast<int>((job >> 23) & 0xFFu);
        const float4 rd = __ldcg(&A.race_desc[b]);
        const int4 rr = __ldcg(&A.race_rows[b]);  // (first target row, first draft row, offset, n_b)
        const uint32_t tag = __float_as_uint(rd.w);
        const int a = static_cast<int>(tag & 0xFFFFu);
        const bool residual = (tag >> 16) != 0u && round == 0;
        d.kind = kItemRace;
        last_was_race = true;
        d.b = b;
        d.j = a;
        d.trow = rr.x + a;
        d.drow = rr.y + a;
        d.rword = static_cast<uint32_t>(rr.z) + static_cast<uint32_t>(a);
        const int js = race_job_elems(A, residual);
        d.e0 = k * js;
        d.n = min(js, A.V - d.e0);
        d.expect = (A.V + js - 1) / js;  // jobs of this race
        d.seg = k;
        d.c = rd.z;
        d.Pt = rd.x;
        d.Pd = rd.y;
        d.residual = residual;
        d.round = round;
        if (kDirect) {
          ptx::mbar_arrive(bar);
        } else {
          const uint32_t bytes = static_cast<uint32_t>(d.n) * sizeof(Elt);
          const Elt* gt = static_cast<const Elt*>(A.target) + static_cast<size_t>(d.trow) * A.V + d.e0;
          ptx::mbar_arrive_expect_tx(bar, residual ? 2 * bytes : bytes);
          if (kEarly)
            atomicAdd(reinterpret_cast<unsigned long long*>(A.ctr + kCtrReadBytes),
                      static_cast<unsigned long long>(residual ? 2 * bytes : bytes));
          ptx::bulk_g2s(ptx::smem_addr(buf), gt, bytes, bar, pol_first);
          if (residual) {
            const Elt* gd = static_cast<const Elt*>(A.draft) + static_cast<size_t>(d.drow) * A.V + d.e0;
            ptx::bulk_g2s(ptx::smem_addr(buf + kStageBytes / 2), gd, bytes, bar, pol_first);
          }
        }
        fed = true;
      }
    }
    // 2. the next chunk of the group's segment, claiming a new one if needed
    if (!fed && !active) {
      while (next < A.n_claims) {
        const uint32_t u = next / static_cast<uint32_t>(A.nseg);  // unit
        const int seg = static_cast<int>(next % static_cast<uint32_t>(A.nseg));
        int b, r;
        if (kEarly) {
          // Row-major: target and draft row j of every request, then row j+1,
          // so a request's early rows are decided before its later ones are
          // claimed.
          const uint32_t two_b = 2u * static_cast<uint32_t>(A.B);
          const uint32_t rem = u % two_b;
          b = static_cast<int>(rem >> 1);
          r = static_cast<int>(u / two_b) + ((rem & 1u) ? rows : 0);
        } else {
          b = static_cast<int>(u / per_req);
          r = static_cast<int>(u % per_req);
        }
        const ReqInfo q = req_info(A, b);
        const int tensor = r < rows ? 0 : 1;
        const int j = tensor == 0 ? r : r - rows;
        bool valid = !q.skip && (tensor == 0 ? (j <= q.L) : (!q.greedy && j < q.L));
        if (valid && kEarly) {  // rows after a known rejection are not needed
          const uint32_t rh = ptx::ld_relaxed_u32(&A.rej_hi[b]);
          if (rh != 0u && j > rows - static_cast<int>(rh)) valid = false;
        }
        if (q.skip && r == 0 && seg == 0) {
          // A packed segment that cannot be read: finished here, unverified.
          A.accepted_len[b] = -1;
          atomicOr(A.err, SPECDEC_DEV_ERR_DRAFT_LEN);
          atomicAdd(&A.ctr[kCtrDone], 1u);
        }
        if (!valid) {  // ragged: rows beyond n_b are never read
          next = n_static + atomicAdd(&A.ctr[kCtrUnit], 1u);
          continue;
        }
        const size_t row = static_cast<size_t>(tensor == 0 ? q.t0 : q.d0) + j;
        active = true;
        ub = b;
        uj = j;
        utensor = tensor;
        ugreedy = q.greedy;
        uc = q.c;
        uexpect = A.nseg * ((!q.greedy && j < q.L) ? 2 : 1);
        ux = (!q.greedy && j < q.L) ? A.draft_tokens[static_cast<size_t>(q.d0) + j] : -1;
        urow = static_cast<int>(row);
        uk = seg * kSegChunks;
        uk_end = min(A.nch, uk + kSegChunks);
        usrc = static_cast<const Elt*>(tensor == 0 ? A.target : A.draft) + row * A.V;
        if (kEarly) {
          const int e_end = min(A.V, uk_end * A.ch);
          atomicAdd(reinterpret_cast<unsigned long long*>(A.ctr + kCtrReadBytes),
                    static_cast<unsigned long long>(e_end - uk * A.ch) * sizeof(Elt));
        }
        break;
      }
    }
    if (!fed && active) {
      d.kind = kItemStream;
      last_was_race = false;
      d.b = ub;
      d.j = uj;
      d.tensor = utensor;
      d.e0 = uk * A.ch;
      d.n = min(A.ch, A.V - d.e0);
      d.seg = uk / kSegChunks;
      d.flags = ((uk % kSegChunks) == 0 ? kFirst : 0) | (uk + 1 == uk_end ? kLast : 0) | (ugreedy ? kGreedy : 0);
      d.x = ux;
      d.trow = urow;
      d.c = uc;
      d.expect = uexpect;
      if (kDirect) {
        ptx::mbar_arrive(bar);
      } else {
        const uint32_t bytes = static_cast<uint32_t>(d.n) * sizeof(Elt);
        ptx::mbar_arrive_expect_tx(bar, bytes);
        ptx::bulk_g2s_nohint(ptx::smem_addr(buf), usrc + d.e0, bytes, bar);
      }
      if (++uk == uk_end) {
        // The next segment is claimed one chunk ahead: the atomic's latency
        // hides behind the wait for the next free stage, and no claimed
        // segment waits behind a whole segment of this group near the end.
        active = false;
        next = n_static + atomicAdd(&A.ctr[kCtrUnit], 1u);
      }
      fed = true;
    }
    if (fed) {
      last_progress = clock64();
      if (++s == kStagesPerGroup) {
        s = 0;
        phase ^= 1u;
      }
      continue;
    }
    // nothing to feed: finished, or waiting for race jobs
    if (next >= A.n_claims && ptx::ld_relaxed_u32(&A.ctr[kCtrDone]) >= static_cast<uint32_t>(A.B))
      break;  // every request is finished: no job can still appear in `pend`
    if (clock64() - last_progress > kWaitBudgetCycles) {
      failed = true;
      break;
    }
    ptx::nanosleep(64);
  }
  if (failed) atomicOr(A.err, SPECDEC_DEV_ERR_TIMEOUT);
  // The exit marker goes into the group's next stage.
  const int stage = g * kStagesPerGroup + s;
  if (ptx::mbar_wait_bounded(ptx::smem_addr(&empty[stage]), phase ^ 1u, kWaitBudgetCycles)) {
    desc[stage].kind = kItemExit;
    ptx::mbar_arrive(ptx::smem_addr(&full[stage]));
  } else {
    atomicOr(A.err, SPECDEC_DEV_ERR_TIMEOUT);
  }
}

// ------------------------------------------------------------- consumers
// A group of kGroupWarps warps working through its own ring of stages.
template <typename Elt, bool kDirect, bool kEarly>
__device__ void consumer(const PArgs& A, int g, unsigned char* stages, const ItemDesc* desc,
                         uint64_t* full, uint64_t* empty, unsigned long long* scratch) {
  using Ops = EltOps<Elt>;
  constexpr int VEC = Ops::kVec;
  const int gt = static_cast<int>(threadIdx.x) - 32 * kProducerWarps - g * kGroupThreads;
  const int wig = gt >> 5;  // warp within the group
  const int rows = A.n_max + 1;
  unsigned long long* my_scratch = scratch + g * kGroupWarps;
  int s = 0;
  uint32_t phase = 0;
  // running state of the segment being reduced
  float run_m = -INFINITY, run_s = 0.f;  // sampled: max and sum 2^(x c - run_m c)
  float run_gm = -INFINITY;              // greedy: max and its first index
  int run_gi = 0x7FFFFFFF;

  while (true) {
    const int stage = g * kStagesPerGroup + s;
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
      const Elt* gsrc = static_cast<const Elt*>(d.tensor == 0 ? A.target : A.draft) +
                        static_cast<size_t>(d.trow) * A.V + d.e0;
      if (d.flags & kFirst) {
        run_m = -INFINITY;
        run_s = 0.f;
        run_gm = -INFINITY;
        run_gi = 0x7FFFFFFF;
      }
      // this thread's maximum over its part of the chunk
      typename Ops::MaxAcc macc = Ops::max_init();
      for (int vi = gt; vi < nvec; vi += kGroupThreads) Ops::max_vec(vbuf[vi], macc);
      float cm = Ops::max_value(macc);
      if (kDirect)
        for (int e = gt; e < d.n; e += kGroupThreads) cm = fmaxf(cm, Ops::at(gsrc, e));
      const bool greedy = (d.flags & kGreedy) != 0;
      if (greedy) {
        if (cm > run_gm) {  // strictly larger: an earlier chunk keeps ties
          int first = 0x7FFFFFFF;
          for (int vi = gt; vi < nvec && first == 0x7FFFFFFF; vi += kGroupThreads) {
            float f[VEC];
            Ops::unpack(vbuf[vi], f);
#pragma unroll
            for (int i = VEC - 1; i >= 0; --i)
              if (f[i] == cm) first = vi * VEC + i;
          }
          if (kDirect)
            for (int e = gt; e < d.n && first == 0x7FFFFFFF; e += kGroupThreads)
              if (Ops::at(gsrc, e) == cm) first = e;
          run_gm = cm;
          run_gi = d.e0 + first;
        }
      } else {
        if (cm > run_m) {
          if (run_s > 0.f) run_s *= exp2f(run_m * d.c - cm * d.c);
          run_m = cm;
        }
        if (run_m > -INFINITY) {
          const float K = run_m * d.c;
          float2 acc = make_float2(0.f, 0.f);
          const float2 cc = make_float2(d.c, d.c), nk = make_float2(-K, -K);
          for (int vi = gt; vi < nvec; vi += kGroupThreads) Ops::sum_vec(vbuf[vi], cc, nk, acc);
          if (kDirect)
            for (int e = gt; e < d.n; e += kGroupThreads) acc.x += fast_ex2(fmaf(Ops::at(gsrc, e), d.c, -K));
          run_s += acc.x + acc.y;
        }
      }
      // The logit at the row's draft token, for the acceptance test.  Written
      // by the thread that publishes the segment, before it does.
      if (gt == 0 && d.x >= d.e0 && d.x < d.e0 + d.n) {
        const float vx = kDirect ? Ops::at(gsrc, d.x - d.e0) : Ops::at(reinterpret_cast<const Elt*>(buf), d.x - d.e0);
        reinterpret_cast<float*>(&A.row_x[static_cast<size_t>(d.b) * rows + d.j])[d.tensor] = vx;
      }
      // this warp is done with the stage
      __syncwarp();
      if ((gt & 31) == 0) ptx::mbar_arrive(ptx::smem_addr(&empty[stage]));
      if (d.flags & kLast) {
        float2 res;
        if (greedy) {
          const float M = group_max(run_gm, g, my_scratch);
          const int idx = group_min_i(run_gm == M ? run_gi : 0x7FFFFFFF, g, my_scratch);
          res = make_float2(M, __int_as_float(idx));
        } else {
          const float M = group_max(run_m, g, my_scratch);
          const float K = M * d.c;
          const float mine = run_s > 0.f ? run_s * exp2f(run_m * d.c - K) : 0.f;
          res = make_float2(K, group_sum(mine, g, my_scratch));
        }
        if (wig == 0) {
          uint32_t count = 0;
          const size_t row = static_cast<size_t>(d.b) * rows + d.j;
          if (gt == 0) {
            A.part[(row * 2 + d.tensor) * A.nseg + d.seg] = res;
            count = ptx::atom_add_acq_rel(&A.row_cnt[row], 1u);  // publishes the partial
          }
          count = __shfl_sync(0xFFFFFFFFu, count, 0);
          if (count == static_cast<uint32_t>(d.expect - 1)) row_combine_w<Elt, kEarly>(A, d.b, d.j, req_info(A, d.b));
        }
      }
    } else {
      // ------------------------------------------------ race over one chunk of row a
      const Elt* gt_src = static_cast<const Elt*>(A.target) + static_cast<size_t>(d.trow) * A.V + d.e0;
      const Elt* gd_src = static_cast<const Elt*>(A.draft) + static_cast<size_t>(d.drow) * A.V + d.e0;
      const uint4* vd = reinterpret_cast<const uint4*>(buf + kStageBytes / 2);
      // Race keys r / E.  `thr` is the best key any lane of this warp has
      // found so far; since -ln U > 1 - U, an entry with r <= thr (1 - U)
      // cannot beat it.  Per 16-byte vector all weights and draws are formed
      // first (independent work the scheduler can overlap), the bound is a
      // predicate, and only a vector holding a possible winner branches into
      // the accurate logarithm.  The key's division is the fast one (within
      // 2 ulp): keys closer than that are a near tie, which the method does
      // not order anyway beyond the lowest index.
      float best = 0.f, thr = 0.f;
      int idx = -1;
      // The loop runs the same number of times on every lane of a warp (lanes
      // past the end skip the work), so the warp-wide maxima below are uniform.
      const int lane = gt & 31;
      int it = 0;
      for (int vb = gt - lane; vb < nvec; vb += kGroupThreads, ++it) {
        const int vi = vb + lane;
        const bool live = vi < nvec;
        const int v = d.e0 + vi * VEC;
        // weights r and 1 - U as pairs (packed fp32 arithmetic)
        float2 r[VEC / 2], y[VEC / 2];
        if (live) {
          float ft[VEC];
          Ops::unpack(vbuf[vi], ft);
          const float2 cc = make_float2(d.c, d.c);
          const float2 npt = make_float2(-d.Pt, -d.Pt);
#pragma unroll
          for (int k = 0; k < VEC / 2; ++k) {
            const float2 a = __ffma2_rn(make_float2(ft[2 * k], ft[2 * k + 1]), cc, npt);
            r[k] = make_float2(fast_ex2(a.x), fast_ex2(a.y));
          }
          if (d.residual) {
            float fd[VEC];
            Ops::unpack(vd[vi], fd);
            const float2 npd = make_float2(-d.Pd, -d.Pd);
            const float2 m1 = make_float2(-1.f, -1.f);
#pragma unroll
            for (int k = 0; k < VEC / 2; ++k) {
              const float2 a = __ffma2_rn(make_float2(fd[2 * k], fd[2 * k + 1]), cc, npd);
              r[k] = __ffma2_rn(make_float2(fast_ex2(a.x), fast_ex2(a.y)), m1, r[k]);  // p - q
            }
          }
          // 1 - U = (2 - 2^-24) - f, f the float in [1, 2) holding the word's top 23 bits (exact)
          const float2 m1 = make_float2(-1.f, -1.f);
          const float2 two = make_float2(1.99999994039535522461f, 1.99999994039535522461f);
#pragma unroll
          for (int q4 = 0; q4 < VEC / 4; ++q4) {
            const Philox4 rnd = philox4x32_10(static_cast<uint32_t>(v + 4 * q4) >> 2, d.rword,
                                              static_cast<uint32_t>(d.b), 1u, A.seed_lo, A.seed_hi);
#pragma unroll
            for (int i = 0; i < 2; ++i)
              y[2 * q4 + i] = __ffma2_rn(make_float2(__uint_as_float(0x3F800000u | (rnd.w[2 * i] >> 9)),
                                                     __uint_as_float(0x3F800000u | (rnd.w[2 * i + 1] >> 9))),
                                         m1, two);
          }
        } else {
#pragma unroll
          for (int k = 0; k < VEC / 2; ++k) {
            r[k] = make_float2(0.f, 0.f);
            y[k] = make_float2(1.f, 1.f);
          }
        }
        if (it == 0) {
          // Seed the threshold with a lower bound of real keys: ln(1/U) <=
          // 1/U - 1 gives r / -ln U >= r U / (1 - U).  The factor 1 - 2^-18
          // covers the rounding of this product and of the exact key, so the
          // entry that gives the bound still passes the test below.
          float lb = 0.f;
#pragma unroll
          for (int k = 0; k < VEC / 2; ++k) {
            if (r[k].x > 0.f) lb = fmaxf(lb, r[k].x * ((1.0f - y[k].x) * fast_rcp(y[k].x)));
            if (r[k].y > 0.f) lb = fmaxf(lb, r[k].y * ((1.0f - y[k].y) * fast_rcp(y[k].y)));
          }
          thr = warp_max(lb) * 0.99999618530273438f;
        }
        // An entry can beat the threshold only if r - thr (1 - U) > 0 (this
        // also rejects r <= 0, as thr >= 0 and 1 - U > 0).
        float2 dd[VEC / 2];
        const float2 nthr = make_float2(-thr, -thr);
        float dmax = -INFINITY;
#pragma unroll
        for (int k = 0; k < VEC / 2; ++k) {
          dd[k] = __ffma2_rn(y[k], nthr, r[k]);
          dmax = fmaxf(dmax, fmaxf(dd[k].x, dd[k].y));
        }
        if (dmax > 0.f) {
#pragma unroll
          for (int k = 0; k < VEC / 2; ++k) {
            if (dd[k].x > 0.f) {
              const float key = __fdividef(r[k].x, -logf(1.0f - y[k].x));
              if (key > best) {  // strictly: the lower index keeps a tie
                best = key;
                idx = v + 2 * k;
              }
            }
            if (dd[k].y > 0.f) {
              const float key = __fdividef(r[k].y, -logf(1.0f - y[k].y));
              if (key > best) {
                best = key;
                idx = v + 2 * k + 1;
              }
            }
          }
        }
        if (it == 2) thr = fmaxf(thr, warp_max(best));
      }
      if (kDirect) {
        for (int e = gt; e < d.n; e += kGroupThreads) {
          const int v = d.e0 + e;
          float r = fast_ex2(fmaf(Ops::at(gt_src, e), d.c, -d.Pt));
          if (d.residual) r -= fast_ex2(fmaf(Ops::at(gd_src, e), d.c, -d.Pd));
          if (r > 0.f) {
            const Philox4 rnd = philox4x32_10(static_cast<uint32_t>(v) >> 2, d.rword,
                                              static_cast<uint32_t>(d.b), 1u, A.seed_lo, A.seed_hi);
            const float key = r / -logf(uniform_from_word(rnd.w[v & 3]));
            if (key > best) {
              best = key;
              idx = v;
            }
          }
        }
      }
      __syncwarp();
      if ((gt & 31) == 0) ptx::mbar_arrive(ptx::smem_addr(&empty[stage]));
      const unsigned long long mine = idx >= 0 ? pack_key(__float_as_uint(best), idx) : 0ull;
      const unsigned long long group_best = group_max_u64(mine, g, my_scratch);
      if (wig == 0) {
        uint32_t count = 0;
        if (gt == 0) {
          if (group_best != 0ull) atomicMax(&A.race_best[d.b], group_best);
          count = ptx::atom_add_acq_rel(&A.race_cnt[d.b], 1u);  // publishes the maximum
        }
        count = __shfl_sync(0xFFFFFFFFu, count, 0);
        if (count == static_cast<uint32_t>(d.expect - 1)) race_finalize_w(A, d.b, d.round);
      }
    }
    if (++s == kStagesPerGroup) {
      s = 0;
      phase ^= 1u;
    }
  }
}

// ------------------------------------------------------------- the kernel
template <typename Elt, bool kDirect, bool kEarly>
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
      ptx::mbar_init(ptx::smem_addr(&empty[s]), kGroupWarps);
    }
    ptx::fence_mbarrier_init();
  }
  __syncthreads();
  const int warp = static_cast<int>(threadIdx.x >> 5);
  if (warp < kProducerWarps) {
    if ((threadIdx.x & 31) == 0) producer<Elt, kDirect, kEarly>(A, warp, stages, desc, full, empty);
  } else {
    consumer<Elt, kDirect, kEarly>(A, (warp - kProducerWarps) / kGroupWarps, stages, desc, full, empty, scratch);
  }
  __syncthreads();
  // every group is done: the reduction scratch holds the last-CTA flag
  volatile int& last_cta = *reinterpret_cast<volatile int*>(scratch);
  if (threadIdx.x == 0) {
    // The last CTA out re-arms the queue counters for the next call.
    __threadfence();
    last_cta = atomicAdd(&A.ctr[kCtrExit], 1u) == gridDim.x - 1;
    if (last_cta) {
      A.ctr[kCtrUnit] = 0u;
      A.ctr[kCtrRaceHead] = 0u;
      A.ctr[kCtrRaceTail] = 0u;
      A.ctr[kCtrDone] = 0u;
      A.ctr[kCtrExit] = 0u;
      __threadfence();
    }
  }
  if (kEarly) {
    // Early exit leaves per-request state and the counters of rows that were
    // only partly streamed; every other CTA has finished, so the last one
    // clears them for the next call.
    __syncthreads();
    if (last_cta) {
      __threadfence();
      for (int i = threadIdx.x; i < A.B; i += blockDim.x) {
        A.rej_hi[i] = 0u;
        A.row_done[i] = 0u;
        A.req_fin[i] = 0u;
      }
      const int nrow = A.B * (A.n_max + 1);
      for (int i = threadIdx.x; i < nrow; i += blockDim.x) A.row_cnt[i] = 0u;
      __threadfence();
    }
  }
}

constexpr size_t kPersistentSmemBytes =
    static_cast<size_t>(kStages) * kStageBytes + kStages * sizeof(ItemDesc) + 2 * kStages * sizeof(uint64_t) +
    kGroups * kGroupWarps * sizeof(unsigned long long);

}  // namespace specdec
