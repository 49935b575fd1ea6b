// verify_persistent.cuh — persistent, warp-specialised verify/accept kernel
// for sm_103a (one CTA per SM).
//
// A plan kernel first lists the row-tensor units to stream (request b,
// target row j <= n_b or draft row j < n_b), in request-major order (row-major
// for early exit), with each request's parameters.  Segments (kSegChunks
// chunks) of those units are claimed one at a time from a device counter, so
// requests finish roughly in order.  Per CTA:
//   * each consumer group owns a ring of kStagesPerGroup shared-memory stages
//     and a producer warp that streams the group's current segment into it,
//     kStageBytes at a time, with 1-D bulk copies (TMA engine); each stage has
//     a "full" mbarrier (bytes landed) and an "empty" mbarrier (every warp of
//     the group is done with it); the producer claims its next segment and
//     loads that segment's unit record while the current one goes out;
//   * a consumer group reduces its segment with running per-thread state —
//     (max, sum 2^(x c - K)) for sampled requests, (max, first index of the
//     max) for greedy ones, c = log2(e)/T — and posts one partial per segment
//     to the CTA's mailbox in shared memory, then moves on at once;
//   * a publishing warp takes the mailbox entries (one lane per slot, their
//     global atomics in flight together) and publishes them; an entry that
//     completes a request (or, for early exit, a row, or a race) becomes a
//     task for the combining warp, which combines the request's rows
//     (log-sum-exp, acceptance test u_j < p_j(x_j)/q_j(x_j), one lane per
//     row), finds the first rejection a and either writes the greedy result
//     or queues the exponential race over row a as chunk jobs, and finishes
//     races;
//   * a dispatching warp takes tickets on the race queue and stages the jobs
//     it draws in the CTA's inbox; producers take a job from the inbox
//     between two segments (at most one while segments remain), so races
//     overlap the streaming and re-read row a soon after it was streamed,
//     mostly from L2.  A race first keeps only entries whose key can reach
//     a threshold; the rare race that finds none there runs again without.
// Every segment and every race job is claimed from a device counter, so a CTA
// that starts late (its SM busy with other work) finds the work taken and
// leaves: no CTA waits for another CTA to start.  Every wait is bounded.
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
constexpr int kBookWarp = kProducerWarps + kGroups * kGroupWarps;  // publishes the groups' results
constexpr int kCombineWarp = kBookWarp + 1;                        // combines requests, finishes races
constexpr int kDispatchWarp = kCombineWarp + 1;                    // stages race jobs for the CTA
constexpr int kThreads = 32 * (kDispatchWarp + 1);
constexpr int kStagesPerGroup = 2;
constexpr int kStages = kGroups * kStagesPerGroup;
constexpr int kStageBytes = 28 * 1024;  // shared-memory capacity of a stage
constexpr int kSegChunks = 3;                          // chunks per published partial
constexpr int kBoxDepth = 8;                           // mailbox slots per consumer group
constexpr int kBoxSlots = kGroups * kBoxDepth;         // one bookkeeping lane per slot
constexpr int kInbox = 8;                              // race jobs staged per CTA (one per dispatch lane)
constexpr int kSpecTickets = 4;                        // race-queue tickets a CTA holds ahead of the tail
constexpr int kMaxCtas = 256;                          // grid bound; with kInbox it bounds the queue's claim slack
constexpr int kTasks = 16;                             // publisher -> combiner task ring
#ifndef SPECDEC_WAIT_BUDGET_CYCLES
#define SPECDEC_WAIT_BUDGET_CYCLES 4000000000LL  // ~2 s of SM clock
#endif
constexpr long long kWaitBudgetCycles = SPECDEC_WAIT_BUDGET_CYCLES;  // every device wait gives up after this
static_assert(kBoxSlots == 32, "one publishing lane per mailbox slot");

// Device counters, each on its own 128-byte line (u32 indices).
constexpr int kCtrUnit = 0, kCtrRaceHead = 32, kCtrRaceTail = 64, kCtrDone = 96, kCtrExit = 128;
constexpr int kCtrReadBytes = 160;  // early exit: u64 logits bytes read, summed over calls until read
constexpr int kCtrFault = 176;      // a wait of this call ran out: the last CTA clears the call's state
constexpr int kCtrNever = 177;      // never written (the failure-path test waits on it)
constexpr int kCtrWords = 192;

enum : uint32_t { kItemStream = 1u, kItemRace = 2u, kItemExit = 3u };
enum : int { kFirst = 1, kLast = 2, kGreedy = 4 };
// race job word: valid | chunk << 24 | round << 22 | b
constexpr uint32_t kJobValid = 0x80000000u;
// Races run in rounds: round 0 keeps only entries whose key can reach kTau
// (of the race's total weight R: 1 for a race on p, the residual mass for a
// residual race); if no key reached it, round 1 runs the same race with no
// threshold; round 2 races on p when every residual weight vanished in fp32.
// The winning key of an exponential race of total weight R is 1 / Exp(R)
// distributed, so round 0 misses it with probability exp(-R / tau): e^-16
// for a race on p (R = 1, tau = 1/16); exp(-64 R) for a residual race, which
// happens with probability R itself, so at most tau / e of the rows need the
// second round whatever the distributions.
constexpr float kTauBonus = 0.0625f, kTauResidual = 0.015625f;
__host__ __device__ __forceinline__ float race_tau(bool residual, int round) {
  return round != 0 ? 0.f : (residual ? kTauResidual : kTauBonus);
}

struct ItemDesc {  // one per stage, written by the producer
  uint32_t kind;
  int b, j;      // request, row within the request (race: the job tag, a | residual << 16)
  int tensor;    // stream: 0 target, 1 draft
  int e0, n;     // first vocab index and element count of the chunk
  int seg;       // stream: segment index within the row-tensor; race: chunk index
  int flags;     // stream: kFirst | kLast | kGreedy
  int spare;     // unused: keeps the descriptor at 80 bytes
  int trow;      // stream: row of the streamed tensor; race: target row of a
  float c;       // log2(e) / T
  float Pt, Pd;  // race: log2 normalisers of row a
  int residual;  // race: r = max(0, p - q) (else r = p)
  int round;     // race: 0 (threshold kTau), 1 (no threshold), 2 (on p, no threshold)
  int expect;    // stream: segments that complete the row (both tensors); race: jobs of the race
  int drow;      // race: draft row of a
  uint32_t rword;  // race: row word of the race's random counter (position offset + a)
  int post_j;    // stream: the mailbox entry's j (the row)
  int post_ts;   // stream: the mailbox entry's ts (tensor | seg << 1)
};
static_assert(sizeof(ItemDesc) == 80, "descriptor layout");

// Mailbox entry: a consumer group's result for the bookkeeping warp.
enum : uint32_t { kBoxStream = 1u, kBoxRace = 2u, kBoxExit = 3u };
struct BoxEntry {
  uint32_t kind;   // kBoxStream, kBoxRace or kBoxExit
  int b;
  int j;           // stream: row; race: round
  int ts;          // stream: tensor | seg << 1; exit: entries the group posted before it
  int expect;      // segments that complete the row, or jobs that complete the race
  int pad;
  unsigned long long res;  // stream: partial (float2 bits); race: packed best key
};
static_assert(sizeof(BoxEntry) == 32, "mailbox entry layout");

// A race job staged in the CTA's inbox.
struct RaceJob {
  int b, tag, k, round;  // tag: a | residual << 16 (race_tag)
  int trow, drow, residual, expect;
  uint32_t rword;
  float c, Pt, Pd;
};
static_assert(sizeof(RaceJob) == 48, "inbox entry layout");

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
  // The plan (written by verify_plan_kernel just before the verify kernel):
  // request b's parameters, and one record per row-tensor that must be
  // streamed ("unit"), in streaming order — request-major, or row-major for
  // early exit — so that claims index only rows that exist.  Claim c is
  // segment c % nseg of unit c / nseg.
  int4* rinfo;        // [B] (t0, L | flags, c bits, position offset)
  int4* units;        // [B (2 n_max + 1)] (row, b | j << 16 | tensor << 23 | greedy << 24, c bits, expect)
  uint32_t* n_units;  // [1] units in the plan
  uint32_t race_q_cap;  // race queue slots: every job a call can queue plus kMaxCtas * kInbox
  int count_bytes;      // add the logits bytes read to the workspace counter (early-exit calls)
  // workspace
  uint32_t* err;
  uint32_t* ctr;                    // [kCtrWords]
  unsigned long long* race_q;       // [race_q_cap] job words: (a | residual << 16) << 32 | job
  uint32_t* req_cnt;                // [B]
  unsigned long long* race_best;    // [B] best packed key of the request's race so far
  uint32_t* race_cnt;               // [B]
  unsigned long long* race_desc;    // [B] (Pd, Pt) of row a as a result slot: zero until written
  uint32_t* row_cnt;                // [B * rows]
  float2* row_P;                    // [B * rows]
  int32_t* row_arg;                 // [B * rows]
  unsigned long long* part;         // [B * rows * 2 * nseg] segment partials (slot encoding)
  // early exit only (zero between calls)
  uint32_t* rej_hi;                 // [B] max over rejected rows k of (n_max + 1 - k); 0: none yet
  unsigned long long* row_done;     // [B] bit j: row j combined; bit 32 + j: draft j accepted
  uint32_t* req_fin;                // [B] the request's outputs are claimed
};

// Shared memory of one CTA (the stages come first, 1024-byte aligned).
struct Shared {
  unsigned char* stages;        // [kStages][kStageBytes]
  ItemDesc* desc;               // [kStages]
  uint64_t* full;               // [kStages]
  uint64_t* empty;              // [kStages]
  unsigned long long* scratch;  // [kGroups * kGroupWarps] group reductions
  BoxEntry* box;                // [kBoxSlots]
  uint64_t* box_full;           // [kBoxSlots]
  uint64_t* box_empty;          // [kBoxSlots]
  RaceJob* inbox;               // [kInbox]
  uint32_t* islot;              // [kInbox] inbox slot states: 0 free, 1 holds a job, 2 being taken
  unsigned long long* task;     // [kTasks] (kind << 32 | b): a request to combine or a race to finish
  uint32_t* flag;               // [4] task tail (publisher), task head (combiner), publisher done, last CTA out
};
constexpr size_t kSmemStages = static_cast<size_t>(kStages) * kStageBytes;
constexpr size_t kSmemDesc = kSmemStages;
constexpr size_t kSmemFull = kSmemDesc + kStages * sizeof(ItemDesc);
constexpr size_t kSmemEmpty = kSmemFull + kStages * sizeof(uint64_t);
constexpr size_t kSmemScratch = kSmemEmpty + kStages * sizeof(uint64_t);
constexpr size_t kSmemBox = kSmemScratch + kGroups * kGroupWarps * sizeof(unsigned long long);
constexpr size_t kSmemBoxFull = kSmemBox + kBoxSlots * sizeof(BoxEntry);
constexpr size_t kSmemBoxEmpty = kSmemBoxFull + kBoxSlots * sizeof(uint64_t);
constexpr size_t kSmemInbox = kSmemBoxEmpty + kBoxSlots * sizeof(uint64_t);
constexpr size_t kSmemIslot = kSmemInbox + kInbox * sizeof(RaceJob);
constexpr size_t kSmemTask = kSmemIslot + kInbox * sizeof(uint32_t);
constexpr size_t kSmemFlag = kSmemTask + kTasks * sizeof(unsigned long long);
constexpr size_t kPersistentSmemBytes = kSmemFlag + 4 * sizeof(uint32_t);
static_assert(kPersistentSmemBytes <= 227 * 1024, "fits the 227 KB a CTA may use");

__device__ __forceinline__ Shared shared_layout(unsigned char* smem) {
  Shared S;
  S.stages = smem;
  S.desc = reinterpret_cast<ItemDesc*>(smem + kSmemDesc);
  S.full = reinterpret_cast<uint64_t*>(smem + kSmemFull);
  S.empty = reinterpret_cast<uint64_t*>(smem + kSmemEmpty);
  S.scratch = reinterpret_cast<unsigned long long*>(smem + kSmemScratch);
  S.box = reinterpret_cast<BoxEntry*>(smem + kSmemBox);
  S.box_full = reinterpret_cast<uint64_t*>(smem + kSmemBoxFull);
  S.box_empty = reinterpret_cast<uint64_t*>(smem + kSmemBoxEmpty);
  S.inbox = reinterpret_cast<RaceJob*>(smem + kSmemInbox);
  S.islot = reinterpret_cast<uint32_t*>(smem + kSmemIslot);
  S.task = reinterpret_cast<unsigned long long*>(smem + kSmemTask);
  S.flag = reinterpret_cast<uint32_t*>(smem + kSmemFlag);
  return S;
}

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

// Segment partials are published in result slots without ordering: the
// writer stores the complemented value and then counts it with a relaxed
// atomic, so a publish is one round trip.  Zero means empty: every value
// stored has a high word other than 0xFFFFFFFF (a sum, which arithmetic never
// makes that NaN, or an index), so its complement is never zero.  The reader,
// once the count is complete, polls any slot still empty (a store not yet
// visible) and zeroes each slot it takes, so the slots are empty again for
// the next call.
__device__ __forceinline__ unsigned long long slot_encode(uint32_t hi, uint32_t lo) {
  if (hi == 0xFFFFFFFFu) hi = 0x7FFFFFFFu;  // a NaN stays a NaN
  return ~((static_cast<unsigned long long>(hi) << 32) | lo);
}

// Request parameters as every part of the kernel derives them.  t0 and d0
// are the request's first row in the target and draft logits (and in the
// draft tokens and outputs): dense [B, n_max+1, V] / [B, n_max, V], or packed
// with target rows at cu_rows[b] + j and draft rows at cu_rows[b] - b + j.
// A packed segment that is empty or reaches outside the tensors is skipped
// (`skip`): nothing of it is read.
struct ReqInfo {
  int L;
  int t0, d0;
  uint32_t o;    // position offset of the random counter's row word
  bool skip;
  float c;
  bool greedy;
  uint32_t err;  // device-data error bits the request raises (draft_len clamped, temperature)
};
// Request b's parameters from its inputs (read by the plan kernel).
__device__ __forceinline__ ReqInfo req_info(const PArgs& A, int b) {
  ReqInfo r;
  int L_raw;
  if (A.cu_rows != nullptr) {
    const int r0 = A.cu_rows[b], r1 = A.cu_rows[b + 1];
    r.t0 = r0;
    r.d0 = r0 - b;
    L_raw = r1 - r0 - 1;
    r.skip = r1 - r0 < 1 || r0 < 0 || r1 > A.total_rows || r.d0 < 0;
  } else {
    r.t0 = b * (A.n_max + 1);
    r.d0 = b * A.n_max;
    L_raw = A.draft_len[b];
    r.skip = false;
  }
  r.o = A.pos_offset != nullptr ? static_cast<uint32_t>(A.pos_offset[b]) : 0u;
  r.L = min(max(L_raw, 0), A.n_max);
  // packed: the draft rows d0 .. d0 + L - 1 must lie below total_rows - B
  if (A.cu_rows != nullptr && r.d0 + r.L > A.total_rows - A.B) r.skip = true;
  const float T = A.temperature[b];
  // without draft logits only a request with no drafts can sample
  r.greedy = !(T > 0.f) || T < 1e-6f || (A.draft == nullptr && r.L > 0);
  const float s = 1.0f / T;
  r.c = s * 1.4426950408889634f;  // log2(e) / T
  r.err = (L_raw != r.L ? SPECDEC_DEV_ERR_DRAFT_LEN : 0u) | (r.greedy && T != 0.f ? SPECDEC_DEV_ERR_TEMPERATURE : 0u);
  return r;
}

// rinfo flags (word y): L in bits 0..7, then these.
enum : int { kRiGreedy = 1 << 8, kRiSkip = 1 << 9, kRiErrShift = 12 };
__device__ __forceinline__ int4 pack_rinfo(const ReqInfo& q) {
  const int flags = q.L | (q.greedy ? kRiGreedy : 0) | (q.skip ? kRiSkip : 0) | static_cast<int>(q.err << kRiErrShift);
  return make_int4(q.t0, flags, __float_as_int(q.c), static_cast<int>(q.o));
}

// Plan entries e = (request b, row j), request-major, or row-major for early
// exit (row j of every request, then row j + 1).
__device__ __forceinline__ void entry_decode(const PArgs& A, uint32_t e, bool early, int& b, int& j) {
  if (early) {
    b = static_cast<int>(e % static_cast<uint32_t>(A.B));
    j = static_cast<int>(e / static_cast<uint32_t>(A.B));
  } else {
    b = static_cast<int>(e / static_cast<uint32_t>(A.n_max + 1));
    j = static_cast<int>(e % static_cast<uint32_t>(A.n_max + 1));
  }
}
// Units of entry (b, j): target row j <= n_b, then draft row j < n_b of a
// sampled request; none for a request that cannot be read.
__device__ __forceinline__ int entry_units(const ReqInfo& q, int j) {
  if (q.skip) return 0;
  return (j <= q.L ? 1 : 0) + ((!q.greedy && j < q.L) ? 1 : 0);
}
__device__ __forceinline__ ReqInfo unpack_rinfo(int4 ri, int b) {
  ReqInfo r;
  r.t0 = ri.x;
  r.d0 = ri.x - b;  // dense: b (n_max + 1) - b = b n_max; packed: cu_rows[b] - b
  r.L = ri.y & 0xFF;
  r.greedy = (ri.y & kRiGreedy) != 0;
  r.skip = (ri.y & kRiSkip) != 0;
  r.err = static_cast<uint32_t>(ri.y) >> kRiErrShift;
  r.c = __int_as_float(ri.z);
  r.o = static_cast<uint32_t>(ri.w);
  return r;
}
// Request b's parameters as the plan recorded them (read-only while the
// verify kernel runs, so the loads may be cached in L1).
__device__ __forceinline__ ReqInfo req_plan(const PArgs& A, int b) { return unpack_rinfo(__ldg(&A.rinfo[b]), b); }

// One CTA of kPlanThreads builds the plan: request parameters, then the
// units of every entry in order.  A packed request that cannot be read is
// finished here, unverified (accepted_len -1, error bit), and counts as done.
constexpr int kPlanThreads = 1024;

// Units of request b in request-major order: target rows 0 .. n_b, and draft
// rows 0 .. n_b - 1 of a sampled request.
__device__ __forceinline__ uint32_t request_units(const ReqInfo& q) {
  return q.skip ? 0u : static_cast<uint32_t>(q.L + 1 + (q.greedy ? 0 : q.L));
}
__device__ __forceinline__ void plan_request(const PArgs& A, int b, const ReqInfo& q, uint32_t& skipped) {
  A.rinfo[b] = pack_rinfo(q);
  if (q.skip) {
    A.accepted_len[b] = -1;
    atomicOr(A.err, SPECDEC_DEV_ERR_DRAFT_LEN);
    ++skipped;
  }
}
// Unit record: (row of its tensor, b | j << 16 | draft << 23 | greedy << 24,
// c bits, segments that complete the request (or, early exit, the row)).
__device__ __forceinline__ int4 unit_record(const PArgs& A, int b, int j, bool draft, const ReqInfo& q, bool early) {
  const int row = (draft ? q.d0 : q.t0) + j;
  const int expect = early ? A.nseg * ((!q.greedy && j < q.L) ? 2 : 1) : A.nseg * static_cast<int>(request_units(q));
  return make_int4(row, b | (j << 16) | ((draft ? 1 : 0) << 23) | ((q.greedy ? 1 : 0) << 24), __float_as_int(q.c),
                   expect);
}

// Request-major plan in one pass: every thread takes a contiguous range of
// requests, whose unit counts are known from their parameters alone (one
// read of the inputs), and the counts are scanned across the CTA with warp
// shuffles.
__device__ void plan_request_major(const PArgs& A) {
  constexpr int kWarps = kPlanThreads / 32;
  static_assert(kWarps == 32, "one warp scans the warp totals");
  __shared__ uint32_t wsum[kWarps];
  const int tid = static_cast<int>(threadIdx.x), lane = tid & 31, warp = tid >> 5;
  const int per = (A.B + kPlanThreads - 1) / kPlanThreads;
  const int b0 = min(A.B, tid * per), b1 = min(A.B, b0 + per);
  uint32_t local = 0, skipped = 0;
  ReqInfo q0;  // the range's first request, kept for the second pass
  q0.L = 0;
  q0.t0 = q0.d0 = 0;
  q0.o = 0u;
  q0.skip = true;
  q0.c = 0.f;
  q0.greedy = true;
  q0.err = 0u;
  for (int b = b0; b < b1; ++b) {
    const ReqInfo q = req_info(A, b);
    if (b == b0) q0 = q;
    plan_request(A, b, q, skipped);
    local += request_units(q);
  }
  if (skipped) atomicAdd(&A.ctr[kCtrDone], skipped);
  uint32_t incl = local;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += v;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const uint32_t w = wsum[lane];
    uint32_t wi = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, wi, off);
      if (lane >= off) wi += v;
    }
    wsum[lane] = wi - w;  // exclusive: units before warp `lane`
  }
  __syncthreads();
  uint32_t u = wsum[warp] + incl - local;  // first unit of this thread's range
  if (per == 1 && A.B > 256) {
    // One request (or none) per thread: the warp writes its lanes' records
    // together, lane l taking unit U = first + 32 k + l of the warp's range,
    // so a store instruction covers 512 contiguous bytes (one thread writing
    // its own records throttled the SM's load/store unit on large batches;
    // on small ones the shuffles' latency costs more).  The owner of U is
    // the last lane whose range starts at or before U: a binary search over
    // the lanes' starts, which never decrease, by shuffles.
    const uint32_t wfirst = __shfl_sync(0xFFFFFFFFu, u, 0);
    const uint32_t wend = __shfl_sync(0xFFFFFFFFu, u + local, 31);
    for (uint32_t U0 = wfirst; U0 < wend; U0 += 32) {  // warp-uniform
      const uint32_t U = U0 + static_cast<uint32_t>(lane);
      int o = 0;
#pragma unroll
      for (int step = 16; step > 0; step >>= 1) {
        const uint32_t s = __shfl_sync(0xFFFFFFFFu, u, o + step);
        if (s <= U) o += step;
      }
      ReqInfo q;
      q.skip = false;
      q.t0 = __shfl_sync(0xFFFFFFFFu, q0.t0, o);
      q.L = __shfl_sync(0xFFFFFFFFu, q0.L, o);
      q.greedy = __shfl_sync(0xFFFFFFFFu, q0.greedy ? 1 : 0, o) != 0;
      q.c = __shfl_sync(0xFFFFFFFFu, q0.c, o);
      const uint32_t k = U - __shfl_sync(0xFFFFFFFFu, u, o);  // unit within the request
      const int b = warp * 32 + o;
      q.d0 = q.t0 - b;
      if (U < wend) {
        int j = static_cast<int>(k);
        bool draft = false;
        if (!q.greedy && j < 2 * q.L) {  // target row j / 2, then draft row j / 2
          draft = (j & 1) != 0;
          j >>= 1;
        } else if (!q.greedy) {
          j = q.L;  // the bonus row
        }
        A.units[U] = unit_record(A, b, j, draft, q, false);
      }
    }
    u += local;
  } else {
    for (int b = b0; b < b1; ++b) {
      const ReqInfo q = b == b0 ? q0 : req_info(A, b);
      if (q.skip) continue;
      for (int j = 0; j <= q.L; ++j) {
        A.units[u++] = unit_record(A, b, j, false, q, false);
        if (!q.greedy && j < q.L) A.units[u++] = unit_record(A, b, j, true, q, false);
      }
    }
  }
  if (tid == kPlanThreads - 1) *A.n_units = u;  // the last range ends at the total
}

// Row-major plan (early exit): entries (b, j) = row j of every request, then
// row j + 1; per-thread ranges of entries, their unit counts scanned across
// the CTA.
__device__ void plan_row_major(const PArgs& A) {
  __shared__ uint32_t sums[kPlanThreads];
  const int tid = static_cast<int>(threadIdx.x);
  uint32_t skipped = 0;
  for (int b = tid; b < A.B; b += kPlanThreads) plan_request(A, b, req_info(A, b), skipped);
  if (skipped) atomicAdd(&A.ctr[kCtrDone], skipped);
  __syncthreads();  // this CTA's global writes are visible to its threads after the barrier
  const uint32_t E = static_cast<uint32_t>(A.B) * static_cast<uint32_t>(A.n_max + 1);
  const uint32_t per = (E + kPlanThreads - 1) / kPlanThreads;
  const uint32_t e0 = min(E, static_cast<uint32_t>(tid) * per), e1 = min(E, e0 + per);
  uint32_t local = 0;
  for (uint32_t e = e0; e < e1; ++e) {
    int b, j;
    entry_decode(A, e, true, b, j);
    local += entry_units(unpack_rinfo(__ldcg(&A.rinfo[b]), b), j);
  }
  sums[tid] = local;
  __syncthreads();
  // inclusive scan of the per-thread sums (Hillis-Steele over shared memory)
  for (int off = 1; off < kPlanThreads; off <<= 1) {
    const uint32_t v = tid >= off ? sums[tid - off] : 0u;
    __syncthreads();
    sums[tid] += v;
    __syncthreads();
  }
  uint32_t u = sums[tid] - local;  // first unit of this thread's range
  for (uint32_t e = e0; e < e1; ++e) {
    int b, j;
    entry_decode(A, e, true, b, j);
    const ReqInfo q = unpack_rinfo(__ldcg(&A.rinfo[b]), b);
    if (entry_units(q, j) == 0) continue;
    A.units[u++] = unit_record(A, b, j, false, q, true);
    if (!q.greedy && j < q.L) A.units[u++] = unit_record(A, b, j, true, q, true);
  }
  if (tid == kPlanThreads - 1) *A.n_units = sums[tid];
}

template <bool kEarly>
__global__ void __launch_bounds__(kPlanThreads) verify_plan_kernel(const PArgs A) {
  // The verify kernel may launch now: it waits for this grid to complete
  // before it reads anything written here.
  ptx::launch_dependents();
  if (kEarly)
    plan_row_major(A);
  else
    plan_request_major(A);
}

// A wait of this call ran out: flag it (sticky error bit) and have the last
// CTA out clear the state the call leaves behind, so the workspace stays
// usable.
__device__ __forceinline__ void raise_timeout(const PArgs& A) {
  atomicOr(A.err, SPECDEC_DEV_ERR_TIMEOUT);
  atomicExch(&A.ctr[kCtrFault], 1u);
}

// Takes a result slot whose count is complete: `v` is a first load of it.
// Polls while it is still empty (bounded, and not once the call has
// faulted), zeroes it and returns the value (0 if it stayed empty: the
// timeout is raised).
__device__ __forceinline__ unsigned long long slot_take(const PArgs& A, unsigned long long* p, unsigned long long v) {
  if (v == 0ull) {
    const long long t0 = clock64();
    do {
      ptx::nanosleep(32);
      v = ptx::ld_relaxed_u64(p);
    } while (v == 0ull && clock64() - t0 <= kWaitBudgetCycles && ptx::ld_relaxed_u32(&A.ctr[kCtrFault]) == 0u);
    if (v == 0ull) {
      raise_timeout(A);
      return 0ull;
    }
  }
  ptx::st_relaxed_u64(p, 0ull);
  return ~v;
}

// ------------------------------------------------------------- bookkeeping
// Run by one lane for one item; the lanes of the bookkeeping warp run their
// items side by side, so their L2 round trips overlap.  Results are published
// with an acquire-release count: whoever observes the final count has
// acquired everything published before it (the last-arriver pattern).

__device__ __forceinline__ int lane_id() { return static_cast<int>(threadIdx.x & 31); }

// Race jobs of a race: a residual race reads half a stage of target and
// half of draft per job; a race on p (the bonus row, or the fallback) reads
// a whole stage of target.
__device__ __forceinline__ int race_job_elems(const PArgs& A, bool residual) { return residual ? A.chr : 2 * A.chr; }
__device__ __forceinline__ int race_jobs(const PArgs& A, bool residual) {
  const int js = race_job_elems(A, residual);
  return (A.V + js - 1) / js;
}
// Queue the race of request b.  A job word carries the row a and whether the
// race is residual (`tag` = a | residual << 16); the log2 normalisers of row
// a travel in race_desc[b], a result slot the dispatcher polls until it is
// written, so neither side waits on a fence.  The queue holds every job a
// call can queue, so the bound never cuts; were it to, the race would never
// finish and the call would end on its timeout.
__device__ __forceinline__ uint32_t race_tag(int a, bool residual) {
  return static_cast<uint32_t>(a) | ((residual ? 1u : 0u) << 16);
}
static __device__ void enqueue_race_l(const PArgs& A, int b, int round, int njobs, uint32_t tag) {
  const uint32_t base = atomicAdd(&A.ctr[kCtrRaceTail], static_cast<uint32_t>(njobs));
  const unsigned long long hi = static_cast<unsigned long long>(tag) << 32;
  for (int k = 0; k < njobs; ++k)
    if (base + k < A.race_q_cap)
      ptx::st_relaxed_u64(&A.race_q[base + k], hi | kJobValid | (static_cast<uint32_t>(k) << 24) |
                                                   (static_cast<uint32_t>(round) << 22) | static_cast<uint32_t>(b));
}
// Row a's normalisers for the dispatcher (see enqueue_race_l).
__device__ __forceinline__ void store_race_desc(const PArgs& A, int b, float Pt, float Pd) {
  ptx::st_relaxed_u64(&A.race_desc[b], slot_encode(__float_as_uint(Pd), __float_as_uint(Pt)));
}

// out_tokens of request b: a accepted drafts, then y (left for the race to
// write when with_y is false), then -1 up to the request's last slot
// (n_max + 1 slots dense, n_b + 1 packed); and accepted_len.
static __device__ void write_outputs_l(const PArgs& A, int b, int a, int y, bool with_y, int t0, int d0, int L) {
  const int slots = A.cu_rows != nullptr ? L + 1 : A.n_max + 1;
  A.accepted_len[b] = a;
  int32_t* out = A.out_tokens + static_cast<size_t>(t0);
  for (int k = 0; k < slots; ++k) {
    if (k < a)
      out[k] = A.draft_tokens[static_cast<size_t>(d0) + k];
    else if (k > a)
      out[k] = -1;
    else if (with_y)
      out[k] = y;
  }
}

// Request b's first rejection is row a (a = n_b: every draft accepted), with
// row a's log2 normalisers (Pt, Pd) or, greedy, its argmax: write the greedy
// result, or write all but the sampled token and queue the race over row a.
static __device__ void request_finish_l(const PArgs& A, int b, const ReqInfo& q, int a, bool bad_token, float Pt,
                                        float Pd, int arg) {
  const uint32_t errbits = (bad_token ? SPECDEC_DEV_ERR_TOKEN : 0u) | q.err;
  if (errbits) atomicOr(A.err, errbits);
  write_outputs_l(A, b, a, arg, q.greedy, q.t0, q.d0, q.L);
  if (q.greedy) {
    atomicAdd(&A.ctr[kCtrDone], 1u);
    return;
  }
  store_race_desc(A, b, Pt, Pd);
  enqueue_race_l(A, b, 0, race_jobs(A, a < q.L), race_tag(a, a < q.L));
}

// The same outputs, all lanes of a warp: slot k by lane k mod 32.  Lane l
// < nx holds xl, the draft token of row l (just combined), so those slots
// need no load.
static __device__ void write_outputs_w(const PArgs& A, int b, int a, int y, bool with_y, int t0, int d0, int L,
                                       int xl, int nx) {
  const int slots = A.cu_rows != nullptr ? L + 1 : A.n_max + 1;
  if (lane_id() == 0) A.accepted_len[b] = a;
  int32_t* out = A.out_tokens + static_cast<size_t>(t0);
  for (int k = lane_id(); k < slots; k += 32) {
    if (k < a)
      out[k] = k < nx ? xl : A.draft_tokens[static_cast<size_t>(d0) + k];
    else if (k > a)
      out[k] = -1;
    else if (with_y)
      out[k] = y;
  }
}

// Folds a segment partial (K_s = c max, S_s = sum 2^(x c - K_s)) into the
// running (K, S) of a row: the larger K is kept and the other sum rescaled.
__device__ __forceinline__ void merge_partial(float& K, float& S, unsigned long long v) {
  const float k = __uint_as_float(static_cast<uint32_t>(v)), s = __uint_as_float(static_cast<uint32_t>(v >> 32));
  if (!(s > 0.f)) return;
  if (k > K) {
    S = S * exp2f(K - k) + s;  // S = 0 while K = -inf
    K = k;
  } else {
    S += s * exp2f(k - K);
  }
}

struct RowStats {
  float Pt, Pd;
  int arg;
  int x;  // draft token j (-1: the row has none)
  bool acc, bad;
};

// Statistics of row j of request b from its published results, by one lane
// (early exit decides row by row): the log2 normalisers Pt (target) and Pd
// (draft, rows j < n_b) and the acceptance test of draft j, or, greedy, the
// target argmax and whether draft j equals it.  The draft token and the
// segment partials are independent loads, issued together (one round trip for
// nseg <= 4), then the logits at the token; the partials merge into
// K = max_s K_s, S = sum_s S_s 2^(K_s - K).  Every slot read is left empty.
template <typename Elt>
static __device__ RowStats row_stats_l(const PArgs& A, int b, int j, const ReqInfo& q) {
  constexpr int kBatch = 4;  // per tensor: bf16 rows of up to 172K entries take one batch
  const int rows = A.n_max + 1;
  const size_t row = static_cast<size_t>(b) * rows + j;
  const bool has_draft = j < q.L;
  const bool sampled_x = !q.greedy && has_draft;  // the acceptance test reads the logits at x
  unsigned long long* pt = A.part + (row * 2 + 0) * A.nseg;
  unsigned long long* pd = A.part + (row * 2 + 1) * A.nseg;
  RowStats st;
  st.Pt = 0.f;
  st.Pd = 0.f;
  st.arg = 0;
  st.x = has_draft ? __ldg(&A.draft_tokens[static_cast<size_t>(q.d0) + j]) : -1;
  const bool x_ok = st.x >= 0 && st.x < A.V;
  st.bad = has_draft && !x_ok;
  if (q.greedy) {
    float best = -INFINITY;
    int idx = 0x7FFFFFFF;
    for (int s0 = 0; s0 < A.nseg; s0 += kBatch) {
      unsigned long long p[kBatch];
#pragma unroll
      for (int i = 0; i < kBatch; ++i) p[i] = s0 + i < A.nseg ? ptx::ld_relaxed_u64(&pt[s0 + i]) : 0ull;
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        if (s0 + i >= A.nseg) continue;
        const unsigned long long v = slot_take(A, &pt[s0 + i], p[i]);
        const float m = __uint_as_float(static_cast<uint32_t>(v));
        const int k = static_cast<int>(v >> 32);
        if (m > best || (m == best && k < idx)) {  // lowest index among equal maxima
          best = m;
          idx = k;
        }
      }
    }
    st.arg = idx;
    st.acc = has_draft && x_ok && st.x == idx;
    return st;
  }
  float Kt = -INFINITY, St = 0.f, Kd = -INFINITY, Sd = 0.f;
  for (int s0 = 0; s0 < A.nseg; s0 += kBatch) {
    unsigned long long p[kBatch], r[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      p[i] = s0 + i < A.nseg ? ptx::ld_relaxed_u64(&pt[s0 + i]) : 0ull;
      r[i] = (has_draft && s0 + i < A.nseg) ? ptx::ld_relaxed_u64(&pd[s0 + i]) : 0ull;
    }
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      if (s0 + i >= A.nseg) continue;
      merge_partial(Kt, St, slot_take(A, &pt[s0 + i], p[i]));
      if (has_draft) merge_partial(Kd, Sd, slot_take(A, &pd[s0 + i], r[i]));
    }
  }
  st.Pt = Kt + log2f(St);
  st.Pd = has_draft ? Kd + log2f(Sd) : 0.f;
  if (A.row_lse != nullptr) {
    const size_t orow = static_cast<size_t>(q.t0) + j;  // laid out like the target rows
    A.row_lse[orow * 2 + 0] = st.Pt * 0.69314718055994531f;
    if (has_draft) A.row_lse[orow * 2 + 1] = st.Pd * 0.69314718055994531f;
  }
  st.acc = false;
  if (sampled_x && x_ok) {
    const float tx = EltOps<Elt>::at(static_cast<const Elt*>(A.target) + static_cast<size_t>(q.t0 + j) * A.V, st.x);
    const float dx = EltOps<Elt>::at(static_cast<const Elt*>(A.draft) + static_cast<size_t>(q.d0 + j) * A.V, st.x);
    const float l2ratio = fmaf(tx, q.c, -st.Pt) - fmaf(dx, q.c, -st.Pd);  // log2 p(x) - log2 q(x)
    const Philox4 u = philox4x32_10(0u, q.o + static_cast<uint32_t>(j), static_cast<uint32_t>(b), 0u,
                                    A.seed_lo, A.seed_hi);
    st.acc = uniform_from_word(u.w[0]) < exp2f(l2ratio);
  }
  return st;
}

// Row statistics again, P lanes per row (P a power of two >= nseg, so each
// lane takes at most one segment of each tensor): the lanes of a row merge
// their partials with a butterfly of shuffles.  The merge is symmetric
// (K = max(K1, K2), S = S1 2^(K1 - K) + S2 2^(K2 - K)), so every lane of the
// row ends with the same bits.  Lane `sub` = 0 of the row also loads the
// draft token and the logits at it and runs the acceptance test; its
// RowStats are the row's.  Lanes of rows past n_b (live false) take part in
// the shuffles only.
__device__ __forceinline__ void merge_sym(float& K, float& S, float K2, float S2) {
  const float Km = fmaxf(K, K2);
  const float a = S > 0.f ? S * exp2f(K - Km) : 0.f;
  const float c = S2 > 0.f ? S2 * exp2f(K2 - Km) : 0.f;
  S = a + c;
  K = Km;
}
template <typename Elt>
static __device__ RowStats row_stats_w(const PArgs& A, int b, int j, int sub, int P, bool live, const ReqInfo& q) {
  const int rows = A.n_max + 1;
  const size_t row = static_cast<size_t>(b) * rows + j;
  const bool lead = sub == 0;
  const bool has_draft = live && j < q.L;
  const bool mine = live && sub < A.nseg;  // this lane's segment exists
  unsigned long long* pt = A.part + (row * 2 + 0) * A.nseg + sub;
  unsigned long long* pd = A.part + (row * 2 + 1) * A.nseg + sub;
  const bool sampled_x = lead && !q.greedy && has_draft;
  unsigned long long vt = 0ull, vd = 0ull;
  if (mine) vt = ptx::ld_relaxed_u64(pt);
  if (mine && has_draft && !q.greedy) vd = ptx::ld_relaxed_u64(pd);
  RowStats st;
  st.Pt = 0.f;
  st.Pd = 0.f;
  st.arg = 0;
  st.x = (lead && has_draft) ? __ldg(&A.draft_tokens[static_cast<size_t>(q.d0) + j]) : -1;
  const bool x_ok = st.x >= 0 && st.x < A.V;
  st.bad = has_draft && !x_ok;
  st.acc = false;
  if (q.greedy) {
    float best = -INFINITY;
    int idx = 0x7FFFFFFF;
    if (mine) {
      const unsigned long long v = slot_take(A, pt, vt);
      best = __uint_as_float(static_cast<uint32_t>(v));
      idx = static_cast<int>(v >> 32);
    }
    for (int o = 1; o < P; o <<= 1) {
      const float ob = __shfl_xor_sync(0xFFFFFFFFu, best, o);
      const int oi = __shfl_xor_sync(0xFFFFFFFFu, idx, o);
      if (ob > best || (ob == best && oi < idx)) {  // lowest index among equal maxima
        best = ob;
        idx = oi;
      }
    }
    st.arg = idx;
    st.acc = has_draft && x_ok && st.x == idx;
    return st;
  }
  float Kt = -INFINITY, St = 0.f, Kd = -INFINITY, Sd = 0.f;
  if (mine) {
    const unsigned long long v = slot_take(A, pt, vt);
    Kt = __uint_as_float(static_cast<uint32_t>(v));
    St = __uint_as_float(static_cast<uint32_t>(v >> 32));
    if (has_draft) {
      const unsigned long long w = slot_take(A, pd, vd);
      Kd = __uint_as_float(static_cast<uint32_t>(w));
      Sd = __uint_as_float(static_cast<uint32_t>(w >> 32));
    }
  }
  for (int o = 1; o < P; o <<= 1) {
    const float k1 = __shfl_xor_sync(0xFFFFFFFFu, Kt, o), s1 = __shfl_xor_sync(0xFFFFFFFFu, St, o);
    const float k2 = __shfl_xor_sync(0xFFFFFFFFu, Kd, o), s2 = __shfl_xor_sync(0xFFFFFFFFu, Sd, o);
    merge_sym(Kt, St, k1, s1);
    merge_sym(Kd, Sd, k2, s2);
  }
  st.Pt = Kt + log2f(St);
  st.Pd = has_draft ? Kd + log2f(Sd) : 0.f;
  if (lead && live && A.row_lse != nullptr) {
    const size_t orow = static_cast<size_t>(q.t0) + j;  // laid out like the target rows
    A.row_lse[orow * 2 + 0] = st.Pt * 0.69314718055994531f;
    if (has_draft) A.row_lse[orow * 2 + 1] = st.Pd * 0.69314718055994531f;
  }
  if (sampled_x && x_ok) {
    const float tx = EltOps<Elt>::at(static_cast<const Elt*>(A.target) + static_cast<size_t>(q.t0 + j) * A.V, st.x);
    const float dx = EltOps<Elt>::at(static_cast<const Elt*>(A.draft) + static_cast<size_t>(q.d0 + j) * A.V, st.x);
    const float l2ratio = fmaf(tx, q.c, -st.Pt) - fmaf(dx, q.c, -st.Pd);  // log2 p(x) - log2 q(x)
    const Philox4 u = philox4x32_10(0u, q.o + static_cast<uint32_t>(j), static_cast<uint32_t>(b), 0u,
                                    A.seed_lo, A.seed_hi);
    st.acc = uniform_from_word(u.w[0]) < exp2f(l2ratio);
  }
  return st;
}

// Every segment of request b is in (all lanes): rows are combined P lanes
// each, 32 / P rows a round (every row is read, so its slots are left empty);
// the lowest failing draft row is a (else a = n_b).  A greedy request is then
// finished; a sampled one gets every output but the sampled token, and its
// race is queued.
template <typename Elt>
static __device__ void request_combine_w(const PArgs& A, int b, const ReqInfo& q) {
  __syncwarp();
  const int lane = lane_id();
  int P = 1;
  while (P < A.nseg) P <<= 1;
  const int R = 32 / P, sub = lane & (P - 1);
  int a = q.L, x0 = -1, arg = 0;
  bool found = false, decided = false, bad = false;
  float Pt = 0.f, Pd = 0.f;
  for (int base = 0; base <= q.L; base += R) {  // warp-uniform
    const int j = base + lane / P;
    const RowStats st = row_stats_w<Elt>(A, b, j, sub, P, j <= q.L, q);
    if (base == 0) x0 = st.x;
    const uint32_t fm = __ballot_sync(0xFFFFFFFFu, sub == 0 && j < q.L && !st.acc);
    int src = -1;
    if (!decided && fm) {
      src = __ffs(fm) - 1;
      a = base + src / P;
      found = true;
    } else if (!decided && q.L < base + R) {
      src = (q.L - base) * P;  // every draft accepted: the bonus row
    }
    if (src >= 0) {
      decided = true;
      Pt = __shfl_sync(0xFFFFFFFFu, st.Pt, src);
      Pd = __shfl_sync(0xFFFFFFFFu, st.Pd, src);
      arg = __shfl_sync(0xFFFFFFFFu, st.arg, src);
      bad = __shfl_sync(0xFFFFFFFFu, found ? st.bad : false, src);  // only row a < n_b can hold a bad token
    }
  }
  // lane k takes the draft token of row k from the lead lane of that row
  const int xl = __shfl_sync(0xFFFFFFFFu, x0, (lane * P) & 31);
  if (lane == 0) {
    A.req_cnt[b] = 0u;
    const uint32_t errbits = (bad ? SPECDEC_DEV_ERR_TOKEN : 0u) | q.err;
    if (errbits) atomicOr(A.err, errbits);
  }
  if (lane == 0 && !q.greedy) {  // the race first: it is on the critical path, the outputs are not
    store_race_desc(A, b, Pt, Pd);
    enqueue_race_l(A, b, 0, race_jobs(A, a < q.L), race_tag(a, a < q.L));
  }
  write_outputs_w(A, b, a, arg, q.greedy, q.t0, q.d0, q.L, xl, R);
  __syncwarp();
  if (lane == 0 && q.greedy) atomicAdd(&A.ctr[kCtrDone], 1u);
  __syncwarp();
}

// The last race job of request b is in (all lanes): the best key is the
// winner, unless the round calls for another.  `tag` is the race's job tag.
static __device__ void race_finalize_w(const PArgs& A, int b, int round, uint32_t tag) {
  __syncwarp();
  const int lane = lane_id();
  unsigned long long best = 0ull;
  if (lane == 0) {
    A.race_cnt[b] = 0u;
    best = ptx::ld_relaxed_u64(&A.race_best[b]);
    A.race_best[b] = 0ull;
  }
  best = __shfl_sync(0xFFFFFFFFu, best, 0);
  const int a = static_cast<int>(tag & 0xFFFFu);
  const bool residual = (tag >> 16) != 0u;
  // Round 0 found no key at or above its threshold (with a margin for fp32
  // rounding of the keys): the winner may have been filtered out, so run the
  // race again without a threshold.  Round 1 with no positive residual weight
  // at all (every residual weight vanished in fp32): race on p.
  int again = -1;
  if (round == 0 && !(__uint_as_float(static_cast<uint32_t>(best >> 32)) >= race_tau(residual, 0) * 1.0000153f))
    again = 1;
  else if (round == 1 && best == 0ull && residual)
    again = 2;
  if (again >= 0) {
    if (lane == 0) {
      __threadfence();  // the cleared maximum is visible before the next round's jobs
      enqueue_race_l(A, b, again, race_jobs(A, residual && again == 1), tag);
    }
    __syncwarp();
    return;
  }
  if (lane == 0) {
    const int t0 = req_plan(A, b).t0;
    A.out_tokens[static_cast<size_t>(t0) + a] = unpack_index(best);  // the rest was written at the decision
    ptx::st_relaxed_u64(&A.race_desc[b], 0ull);  // every job has read it: empty for the next call
    atomicAdd(&A.ctr[kCtrDone], 1u);
  }
  __syncwarp();
}

// Early exit: the last segment of row (b, j) is in.  Combine it, record a
// rejection (so later rows are not claimed), mark the row done, and finish
// the request once its rows 0..k decide it: rows 0..k-1 accepted and row k
// rejected, or every draft accepted and the bonus row done (n_max < 32: one
// mask word).  One lane.
template <typename Elt>
static __device__ void row_decide_l(const PArgs& A, int b, int j, const ReqInfo& q) {
  const int rows = A.n_max + 1;
  const size_t r0 = static_cast<size_t>(b) * rows;
  const RowStats st = row_stats_l<Elt>(A, b, j, q);
  A.row_cnt[r0 + j] = 0u;  // complete and read: nothing to clear at the end
  A.row_P[r0 + j] = make_float2(st.Pt, st.Pd);
  A.row_arg[r0 + j] = st.arg;
  if (j < q.L && !st.acc) atomicMax(&A.rej_hi[b], static_cast<uint32_t>(rows - j));
  // publishes the row; the word returned holds every row's done and accepted bits
  const unsigned long long mine = (1ull << j) | ((j < q.L && st.acc) ? (1ull << (32 + j)) : 0ull);
  const unsigned long long w = ptx::atom_or_acq_rel_u64(&A.row_done[b], mine) | mine;
  const uint32_t done = static_cast<uint32_t>(w);
  const uint32_t accm = done & static_cast<uint32_t>(w >> 32) & ((1u << q.L) - 1u);  // done, accepted drafts
  const int k = __ffs(~accm) - 1;  // first row that is not a done, accepted draft row
  if (k > q.L || !((done >> k) & 1u)) return;  // undecided: row k is still streaming
  if (atomicExch(&A.req_fin[b], 1u) != 0u) return;  // another row finished it
  float2 P = make_float2(st.Pt, st.Pd);
  int arg = st.arg;
  if (k != j) {  // another row decided it: its statistics were published with its bit
    P = __ldcg(&A.row_P[r0 + k]);
    arg = __ldcg(&A.row_arg[r0 + k]);
  }
  bool bad = false;
  if (k < q.L) {
    const int x = A.draft_tokens[static_cast<size_t>(q.d0) + k];
    bad = !(x >= 0 && x < A.V);
  }
  request_finish_l(A, b, q, k, bad, P.x, P.y, arg);
}

// ------------------------------------------------------------- CTA-local queues
// Consumer group g posts `e` to its next mailbox slot (thread 0 of the group).
__device__ __forceinline__ bool box_post(const Shared& S, int g, uint32_t& box_n, const BoxEntry& e) {
  const int slot = g * kBoxDepth + static_cast<int>(box_n % kBoxDepth);
  const uint32_t par = (box_n / kBoxDepth) & 1u;
  if (!ptx::mbar_wait_bounded(ptx::smem_addr(&S.box_empty[slot]), par ^ 1u, kWaitBudgetCycles)) return false;
  S.box[slot] = e;
  ptx::mbar_arrive(ptx::smem_addr(&S.box_full[slot]));  // release: the entry is visible to the waiter
  ++box_n;
  return true;
}

// A producer takes a race job staged in the CTA's inbox, if there is one.
// Slot states: 0 free, 1 holds a job, 2 being copied out by a producer.  The
// states are scanned with two plain vector loads; only a slot seen holding a
// job is claimed (compare-and-swap) and, after an acquire fence, copied.
__device__ __forceinline__ bool inbox_take(const Shared& S, RaceJob& job) {
  static_assert(kInbox == 8, "two 16-byte loads scan the slot states");
  const uint4 s0 = ptx::ld_volatile_shared_v4(&S.islot[0]);
  const uint4 s1 = ptx::ld_volatile_shared_v4(&S.islot[4]);
  const uint32_t st[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
  for (int l = 0; l < kInbox; ++l) {
    if (st[l] != 1u) continue;
    if (atomicCAS(&S.islot[l], 1u, 2u) != 1u) continue;
    __threadfence_block();  // acquire: the job written before the slot was marked
    job = S.inbox[l];
    __threadfence_block();  // the job is copied out before the slot is handed back
    ptx::st_release_cta_shared_u32(&S.islot[l], 0u);
    return true;
  }
  return false;
}

// ------------------------------------------------------------- producers
// Lane 0 of producer warp g feeds consumer group g's ring: between two
// segments a race job staged in the CTA's inbox (one at most while segments
// remain), else the next chunk of the group's segment, claiming a new one
// from the counter when the current one is done.  Each group has its own
// producer, so a producer blocked on a global load delays only its own group.
template <typename Elt, bool kDirect, bool kEarly>
__device__ void producer(const PArgs& A, int g, const Shared& S) {
  const int rows = A.n_max + 1;
  const uint64_t pol_first = ptx::policy_evict_first();
  const uint64_t pol_last = ptx::policy_evict_last();
  const uint32_t nseg = static_cast<uint32_t>(A.nseg);
  const uint32_t total = nseg * __ldg(A.n_units);  // segments in the plan
  constexpr uint32_t kNone = 0xFFFFFFFFu;
  // The next segment is claimed and its unit record loaded ahead, while the
  // current segment's chunks go out: claim after one chunk, load after the
  // next, so neither round trip delays the segment that follows.
  uint32_t pf = atomicAdd(&A.ctr[kCtrUnit], 1u);
  int4 pf_rec = make_int4(0, 0, 0, 0);
  bool pf_have = false;
  int s = 0;
  uint32_t phase = 0;
  bool active = false;
  int ub = 0, uj = 0, utensor = 0, ugreedy = 0, uexpect = 0, uk = 0, uk_end = 0, urow = 0;
  float uc = 0.f;
  const Elt* usrc = nullptr;
  bool last_was_race = false;  // the most recent item issued was a race job
  long long last_progress = clock64();
  bool failed = false;

  while (true) {
    const int stage = g * kStagesPerGroup + s;
    if (!ptx::mbar_wait_bounded(ptx::smem_addr(&S.empty[stage]), phase ^ 1u, kWaitBudgetCycles)) {
      failed = true;
      break;
    }
    ItemDesc& d = S.desc[stage];
    const uint32_t bar = ptx::smem_addr(&S.full[stage]);
    unsigned char* buf = S.stages + static_cast<size_t>(stage) * kStageBytes;
    bool fed = false;
    // 1. between segments: a race job staged in the inbox; while segments
    //    remain, never two in a row, so the claimed segment is not starved.
    RaceJob job;
    const bool seg_left = !(pf != kNone && pf >= total);
    if (!active && !(last_was_race && seg_left) && inbox_take(S, job)) {
      d.kind = kItemRace;
      last_was_race = true;
      d.b = job.b;
      d.j = job.tag;
      d.trow = job.trow;
      d.drow = job.drow;
      d.rword = job.rword;
      const int js = race_job_elems(A, job.residual != 0);
      d.e0 = job.k * js;
      d.n = min(js, A.V - d.e0);
      d.expect = job.expect;
      d.seg = job.k;
      d.c = job.c;
      d.Pt = job.Pt;
      d.Pd = job.Pd;
      d.residual = job.residual;
      d.round = job.round;
      if (kDirect) {
        ptx::mbar_arrive(bar);
      } else {
        const uint32_t bytes = static_cast<uint32_t>(d.n) * sizeof(Elt);
        const Elt* gt = static_cast<const Elt*>(A.target) + static_cast<size_t>(d.trow) * A.V + d.e0;
        ptx::mbar_arrive_expect_tx(bar, job.residual ? 2 * bytes : bytes);
        if (kEarly || A.count_bytes)
          atomicAdd(reinterpret_cast<unsigned long long*>(A.ctr + kCtrReadBytes),
                    static_cast<unsigned long long>(job.residual ? 2 * bytes : bytes));
        ptx::bulk_g2s(ptx::smem_addr(buf), gt, bytes, bar, pol_first);
        if (job.residual) {
          const Elt* gd = static_cast<const Elt*>(A.draft) + static_cast<size_t>(d.drow) * A.V + d.e0;
          ptx::bulk_g2s(ptx::smem_addr(buf + kStageBytes / 2), gd, bytes, bar, pol_first);
        }
      }
      fed = true;
    }
    // 2. the next chunk of the group's segment, claiming a new one if needed
    if (!fed && !active) {
      while (true) {
        if (pf == kNone) pf = atomicAdd(&A.ctr[kCtrUnit], 1u);
        if (pf >= total) break;  // no segment left
        if (!pf_have) pf_rec = __ldg(&A.units[pf / nseg]);
        const int seg = static_cast<int>(pf % nseg);
        pf = kNone;
        pf_have = false;
        const int b = pf_rec.y & 0xFFFF, j = (pf_rec.y >> 16) & 0x7F;
        if (kEarly) {  // rows after a known rejection are not needed
          const uint32_t rh = ptx::ld_relaxed_u32(&A.rej_hi[b]);
          if (rh != 0u && j > rows - static_cast<int>(rh)) continue;
        }
        active = true;
        ub = b;
        uj = j;
        utensor = (pf_rec.y >> 23) & 1;
        ugreedy = (pf_rec.y >> 24) & 1;
        uc = __int_as_float(pf_rec.z);
        uexpect = pf_rec.w;
        urow = pf_rec.x;
        uk = seg * kSegChunks;
        uk_end = min(A.nch, uk + kSegChunks);
        usrc = static_cast<const Elt*>(utensor == 0 ? A.target : A.draft) + static_cast<size_t>(urow) * A.V;
        if (kEarly || A.count_bytes) {
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
      d.post_j = uj;
      d.post_ts = utensor | ((uk / kSegChunks) << 1);
      d.trow = urow;
      d.c = uc;
      d.expect = uexpect;
      if (kDirect) {
        ptx::mbar_arrive(bar);
      } else {
        const uint32_t bytes = static_cast<uint32_t>(d.n) * sizeof(Elt);
        ptx::mbar_arrive_expect_tx(bar, bytes);
        // The race re-reads row a, the first rejected row: row 0 most often
        // (about a third of the re-read bytes on ragged batches), row 1
        // next.  Row 0 is kept in L2 in preference, row 1 at the default
        // priority, later rows are let go first.
        if (uj == 0)
          ptx::bulk_g2s(ptx::smem_addr(buf), usrc + d.e0, bytes, bar, pol_last);
        else if (uj == 1)
          ptx::bulk_g2s_nohint(ptx::smem_addr(buf), usrc + d.e0, bytes, bar);
        else
          ptx::bulk_g2s(ptx::smem_addr(buf), usrc + d.e0, bytes, bar, pol_first);
      }
      if (++uk == uk_end) active = false;
      // advance the prefetch of the next segment by one step
      if (pf == kNone)
        pf = atomicAdd(&A.ctr[kCtrUnit], 1u);
      else if (!pf_have && pf < total) {
        pf_rec = __ldg(&A.units[pf / nseg]);
        pf_have = true;
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
    last_was_race = false;
    if (!seg_left && ptx::ld_relaxed_u32(&A.ctr[kCtrDone]) >= static_cast<uint32_t>(A.B))
      break;  // every request is finished: no race job is left anywhere
    if (clock64() - last_progress > kWaitBudgetCycles) {
      failed = true;
      break;
    }
    ptx::nanosleep(64);
  }
  if (failed) raise_timeout(A);
  // The exit marker goes into the group's next stage.
  const int stage = g * kStagesPerGroup + s;
  if (ptx::mbar_wait_bounded(ptx::smem_addr(&S.empty[stage]), phase ^ 1u, kWaitBudgetCycles)) {
    S.desc[stage].kind = kItemExit;
    ptx::mbar_arrive(ptx::smem_addr(&S.full[stage]));
  } else {
    raise_timeout(A);
  }
}

// One thread's part of a race over a staged chunk (the vectors of the chunk,
// and of the draft chunk for a residual race): the best key r / -ln U and its
// index, packed as (key bits << 32 | index).
template <typename Elt>
__device__ __forceinline__ unsigned long long race_vectors(const uint4* vbuf, const uint4* vd, int nvec, int gt, int e0,
                                                        float c, float Pt, float Pd, int residual, int round, int b,
                                                        uint32_t rword, uint32_t seed_lo, uint32_t seed_hi) {
  using Ops = EltOps<Elt>;
  constexpr int VEC = Ops::kVec;
  // Race keys r / E.  `thr` is a key the winner reaches: the round's
  // threshold (less a margin for fp32 rounding) or the best key any lane
  // of this warp has found so far; since -ln U > 1 - U, an entry with
  // r <= thr (1 - U) cannot beat it, and since 1 - U >= 2^-24, a vector
  // whose weights are all <= thr 2^-24 needs no random numbers at all.
  // Per 16-byte vector all weights and draws are formed first
  // (independent work the scheduler can overlap), the bound is a
  // predicate, and only a vector holding a possible winner branches into
  // the accurate logarithm.  The key's division is the fast one (within
  // 2 ulp): keys closer than that are a near tie, which the method does
  // not order anyway beyond the lowest index.
  float best = 0.f, thr = race_tau(residual != 0, round) * 0.99998474f;
  int idx = -1;
  // The loop runs the same number of times on every lane of a warp (lanes
  // past the end skip the work), so the warp-wide maxima below are uniform.
  const int lane = gt & 31;
  int it = 0;
  for (int vb = gt - lane; vb < nvec; vb += kGroupThreads, ++it) {
    const int vi = vb + lane;
    const bool live = vi < nvec;
    const int v = e0 + vi * VEC;
    // weights r and 1 - U as pairs (packed fp32 arithmetic)
    float2 r[VEC / 2], y[VEC / 2];
    if (live) {
      float ft[VEC];
      Ops::unpack(vbuf[vi], ft);
      const float2 cc = make_float2(c, c);
      const float2 npt = make_float2(-Pt, -Pt);
#pragma unroll
      for (int k = 0; k < VEC / 2; ++k) {
        const float2 a = __ffma2_rn(make_float2(ft[2 * k], ft[2 * k + 1]), cc, npt);
        r[k] = make_float2(fast_ex2(a.x), fast_ex2(a.y));
      }
      if (residual) {
        float fd[VEC];
        Ops::unpack(vd[vi], fd);
        const float2 npd = make_float2(-Pd, -Pd);
        const float2 m1 = make_float2(-1.f, -1.f);
#pragma unroll
        for (int k = 0; k < VEC / 2; ++k) {
          const float2 a = __ffma2_rn(make_float2(fd[2 * k], fd[2 * k + 1]), cc, npd);
          r[k] = __ffma2_rn(make_float2(fast_ex2(a.x), fast_ex2(a.y)), m1, r[k]);  // p - q
        }
      }
      float rmax = 0.f;
#pragma unroll
      for (int k = 0; k < VEC / 2; ++k) rmax = fmaxf(rmax, fmaxf(r[k].x, r[k].y));
      if (rmax > thr * 5.9604645e-8f) {
        // 1 - U exactly: the float in [1, 2) holding the complemented top
        // 23 bits, minus 1 - 2^-24 (one_minus_uniform_from_word, paired)
        const float2 off = make_float2(-0.99999994039535522461f, -0.99999994039535522461f);
#pragma unroll
        for (int q4 = 0; q4 < VEC / 4; ++q4) {
          const Philox4 rnd = philox4x32_10(static_cast<uint32_t>(v + 4 * q4) >> 2, rword,
                                            static_cast<uint32_t>(b), 1u, seed_lo, seed_hi);
#pragma unroll
          for (int i = 0; i < 2; ++i)
            y[2 * q4 + i] = __fadd2_rn(make_float2(__uint_as_float(one_minus_uniform_bits(rnd.w[2 * i])),
                                                   __uint_as_float(one_minus_uniform_bits(rnd.w[2 * i + 1]))),
                                       off);
        }
      } else {
        // no entry can pass: any 1 - U in (0, 1] keeps r - thr (1 - U) <= 0
#pragma unroll
        for (int k = 0; k < VEC / 2; ++k) y[k] = make_float2(1.f, 1.f);
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
      thr = fmaxf(thr, warp_max(lb) * 0.99999618530273438f);
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
  return idx >= 0 ? (static_cast<unsigned long long>(__float_as_uint(best)) << 32) | static_cast<uint32_t>(idx) : 0ull;
}

// The fields of a stage's descriptor that its mailbox entry needs, read
// afresh from shared memory (volatile, so not merged with the copy taken when
// the stage was entered).
__device__ __forceinline__ void post_fields(const ItemDesc& dsc, uint32_t& b, uint32_t& j, uint32_t& ts,
                                            uint32_t& expect) {
  b = ptx::ld_volatile_shared_u32(reinterpret_cast<const uint32_t*>(&dsc.b));
  j = ptx::ld_volatile_shared_u32(reinterpret_cast<const uint32_t*>(&dsc.post_j));
  ts = ptx::ld_volatile_shared_u32(reinterpret_cast<const uint32_t*>(&dsc.post_ts));
  expect = ptx::ld_volatile_shared_u32(reinterpret_cast<const uint32_t*>(&dsc.expect));
}

// ------------------------------------------------------------- consumers
// A group of kGroupWarps warps working through its own ring of stages.
template <typename Elt, bool kDirect, bool kEarly>
__device__ void consumer(const PArgs& A, int g, const Shared& S) {
  using Ops = EltOps<Elt>;
  constexpr int VEC = Ops::kVec;
  const int gt = static_cast<int>(threadIdx.x) - 32 * kProducerWarps - g * kGroupThreads;
  unsigned long long* my_scratch = S.scratch + g * kGroupWarps;
  int s = 0;
  uint32_t phase = 0;
  // running state of the segment being reduced
  float run_m = -INFINITY, run_s = 0.f;  // sampled: max and sum 2^(x c - run_m c)
  float run_gm = -INFINITY;              // greedy: max and its first index
  int run_gi = 0x7FFFFFFF;
  // thread 0 of the group: the mailbox entries posted so far
  uint32_t box_n = 0;
  bool box_ok = true;

  while (true) {
    const int stage = g * kStagesPerGroup + s;
    if (!ptx::mbar_wait_bounded(ptx::smem_addr(&S.full[stage]), phase, kWaitBudgetCycles)) {
      if (gt == 0) raise_timeout(A);
      break;
    }
    const ItemDesc d = S.desc[stage];
    if (d.kind == kItemExit) break;
    const unsigned char* buf = S.stages + static_cast<size_t>(stage) * kStageBytes;
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
      const bool greedy = (d.flags & kGreedy) != 0;
      // this thread's maximum over its part of the chunk
      auto chunk_max = [&]() {
        typename Ops::MaxAcc macc = Ops::max_init();
        for (int vi = gt; vi < nvec; vi += kGroupThreads) Ops::max_vec(vbuf[vi], macc);
        float m = Ops::max_value(macc);
        if (kDirect)
          for (int e = gt; e < d.n; e += kGroupThreads) m = fmaxf(m, Ops::at(gsrc, e));
        return m;
      };
      // A sampled row's sum needs a reference K only to keep 2^(x c - K)
      // from overflowing, not the exact maximum.  The thread takes the
      // largest element of its first vector in the segment (it adds 1 to the
      // sum, so the sum cannot underflow) and keeps it; there is no max pass.
      // A chunk whose sum comes out huge (an element far above the
      // reference) or not finite is summed again against its own maximum.
      float cm = -INFINITY;
      if (greedy) {
        cm = chunk_max();
      } else if (!(run_m > -INFINITY)) {
        if (kDirect) {
          if (gt < d.n) cm = Ops::at(gsrc, gt);
        } else if (gt < nvec) {
          typename Ops::MaxAcc macc = Ops::max_init();
          Ops::max_vec(vbuf[gt], macc);
          cm = Ops::max_value(macc);
        }
        if (!(cm > -INFINITY)) cm = chunk_max();  // that vector holds no finite value
      }
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
        auto chunk_sum = [&]() {
          const float K = run_m * d.c;
          // two accumulators: two independent chains of adds
          float2 acc = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
          const float2 cc = make_float2(d.c, d.c), nk = make_float2(-K, -K);
          int vi = gt;
          for (; vi + kGroupThreads < nvec; vi += 2 * kGroupThreads) {
            Ops::sum_vec(vbuf[vi], cc, nk, acc);
            Ops::sum_vec(vbuf[vi + kGroupThreads], cc, nk, acc1);
          }
          if (vi < nvec) Ops::sum_vec(vbuf[vi], cc, nk, acc);
          if (kDirect)
            for (int e = gt; e < d.n; e += kGroupThreads) acc.x += fast_ex2(fmaf(Ops::at(gsrc, e), d.c, -K));
          return (acc.x + acc.y) + (acc1.x + acc1.y);
        };
        if (run_m > -INFINITY) {
          float s = chunk_sum();
          if (!(s < 1.2676506e30f)) {  // 2^100
            cm = chunk_max();
            if (cm > run_m) {
              if (run_s > 0.f) run_s *= exp2f(run_m * d.c - cm * d.c);
              run_m = cm;
            }
            s = chunk_sum();
          }
          run_s += s;
        }
      }
      // The mailbox entry's fields are read now, while the stage is held, so
      // none of them stays in a register through the loops above.
      uint32_t pb = 0, pj = 0, pts = 0, pex = 0;
      if (gt == 0 && (d.flags & kLast)) post_fields(S.desc[stage], pb, pj, pts, pex);
      // this warp is done with the stage
      __syncwarp();
      if ((gt & 31) == 0) ptx::mbar_arrive(ptx::smem_addr(&S.empty[stage]));
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
        if (gt == 0 && box_ok) {
          BoxEntry e;
          e.kind = kBoxStream;
          e.b = static_cast<int>(pb);
          e.j = static_cast<int>(pj);
          e.ts = static_cast<int>(pts);
          e.expect = static_cast<int>(pex);
          e.pad = 0;
          e.res = (static_cast<unsigned long long>(__float_as_uint(res.y)) << 32) | __float_as_uint(res.x);
          box_ok = box_post(S, g, box_n, e);
        }
      }
    } else {
      // ------------------------------------------------ race over one chunk of row a
      const Elt* gt_src = static_cast<const Elt*>(A.target) + static_cast<size_t>(d.trow) * A.V + d.e0;
      const Elt* gd_src = static_cast<const Elt*>(A.draft) + static_cast<size_t>(d.drow) * A.V + d.e0;
      const uint4* vd = reinterpret_cast<const uint4*>(buf + kStageBytes / 2);
      const unsigned long long rv =
          kDirect ? 0ull
                  : race_vectors<Elt>(vbuf, vd, nvec, gt, d.e0, d.c, d.Pt, d.Pd, d.residual, d.round, d.b, d.rword,
                                      A.seed_lo, A.seed_hi);
      float best = rv != 0ull ? __uint_as_float(static_cast<uint32_t>(rv >> 32)) : 0.f;
      int idx = rv != 0ull ? static_cast<int>(static_cast<uint32_t>(rv)) : -1;
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
      if ((gt & 31) == 0) ptx::mbar_arrive(ptx::smem_addr(&S.empty[stage]));
      const unsigned long long mine = idx >= 0 ? pack_key(__float_as_uint(best), idx) : 0ull;
      const unsigned long long group_best = group_max_u64(mine, g, my_scratch);
      if (gt == 0 && box_ok) {
        BoxEntry e;
        e.kind = kBoxRace;
        e.b = d.b;
        e.j = d.round;
        e.ts = d.j;  // the race's job tag
        e.expect = d.expect;
        e.pad = 0;
        e.res = group_best;
        box_ok = box_post(S, g, box_n, e);
      }
    }
    if (++s == kStagesPerGroup) {
      s = 0;
      phase ^= 1u;
    }
  }
  // Tell the bookkeeping warp how many entries this group posted.
  if (gt == 0) {
    BoxEntry e;
    e.kind = kBoxExit;
    e.b = 0;
    e.j = 0;
    e.ts = static_cast<int>(box_n);
    e.expect = 0;
    e.pad = 0;
    e.res = 0ull;
    if (!box_ok || !box_post(S, g, box_n, e)) raise_timeout(A);
  }
}

// ------------------------------------------------------------- bookkeeping warps
// Tasks the publishing warp hands to the combining warp: (kind << 32 | arg).
enum : uint32_t { kTaskRequest = 1u, kTaskRow = 2u, kTaskRace = 4u };  // kTaskRace + round
// A race task's argument: b (< 2^16), a (<= SPECDEC_MAX_DRAFT < 2^7) and the
// residual bit of its tag.
__device__ __forceinline__ uint32_t race_task_arg(int b, uint32_t tag) {
  static_assert(SPECDEC_MAX_BATCH <= (1 << 16) && SPECDEC_MAX_DRAFT < (1 << 7), "race task argument fields");
  return static_cast<uint32_t>(b) | ((tag & 0x7Fu) << 16) | ((tag >> 16) << 23);
}

// Publishing warp.  Lane l serves mailbox slot l (group l / kBoxDepth).  Each
// round every lane whose slot holds an entry publishes it (the lanes' L2
// atomics overlap); an entry that completes a request, a row (early exit) or
// a race becomes a task for the combining warp, so a publish never waits
// behind a combine.
template <bool kEarly>
__device__ void bookkeeper(const PArgs& A, const Shared& S) {
  const int lane = lane_id();
  const int rows = A.n_max + 1;
  uint32_t par = 0;                  // phase parity of this lane's slot
  uint32_t seen[kGroups] = {0, 0, 0, 0};
  int want[kGroups] = {-1, -1, -1, -1};  // entries a group posted before its exit entry
  uint32_t ttail = 0;                // task ring tail, warp-uniform
  long long last_progress = clock64();
  bool failed = false;
#ifdef SPECDEC_TEST_WAIT_RUNS_OUT
  // Failure-path test builds only: CTA 0's publishing warp first waits for a
  // word that nothing writes, so the wait runs out; the consumers' posts then
  // fail, the requests they carried never finish, and every other wait of the
  // call runs out in turn.  The call reports SPECDEC_DEV_ERR_TIMEOUT and the
  // last CTA re-arms the workspace.
  if (blockIdx.x == 0) {
    const long long t0 = clock64();
    while (ptx::ld_relaxed_u32(&A.ctr[kCtrNever]) == 0u && clock64() - t0 <= kWaitBudgetCycles) ptx::nanosleep(256);
    if (lane == 0) raise_timeout(A);
    last_progress = clock64();
  }
#endif
  while (!failed) {
    const bool ready = ptx::mbar_test_wait(ptx::smem_addr(&S.box_full[lane]), par);
    const uint32_t rm = __ballot_sync(0xFFFFFFFFu, ready);
    uint32_t kind = 0;
    int ts = 0;
    unsigned long long task = 0ull;
    if (ready) {
      const BoxEntry e = S.box[lane];
      par ^= 1u;
      ptx::mbar_arrive(ptx::smem_addr(&S.box_empty[lane]));  // copied out: the slot is free again
      kind = e.kind;
      ts = e.ts;
      if (kind == kBoxStream) {
        const int tensor = ts & 1, seg = ts >> 1;
        const size_t row = static_cast<size_t>(e.b) * rows + e.j;
        ptx::st_relaxed_u64(&A.part[(row * 2 + tensor) * A.nseg + seg],
                            slot_encode(static_cast<uint32_t>(e.res >> 32), static_cast<uint32_t>(e.res)));
        // counts the partial: per row for early exit, else per request
        const uint32_t cnt = atomicAdd(kEarly ? &A.row_cnt[row] : &A.req_cnt[e.b], 1u);
        if (cnt == static_cast<uint32_t>(e.expect - 1))
          task = kEarly ? (static_cast<unsigned long long>(kTaskRow) << 32) | (static_cast<uint32_t>(e.j) << 20) |
                              static_cast<uint32_t>(e.b)
                        : (static_cast<unsigned long long>(kTaskRequest) << 32) | static_cast<uint32_t>(e.b);
      } else if (kind == kBoxRace) {
        // the maximum is ordered before the count by its release
        if (e.res != 0ull) atomicMax(&A.race_best[e.b], e.res);
        const uint32_t cnt = ptx::atom_add_acq_rel(&A.race_cnt[e.b], 1u);
        if (cnt == static_cast<uint32_t>(e.expect - 1))
          task = (static_cast<unsigned long long>(kTaskRace + static_cast<uint32_t>(e.j)) << 32) |
                 race_task_arg(e.b, static_cast<uint32_t>(e.ts));
      }
    }
    // Hand the tasks over in ring order, as room frees up.
    for (uint32_t pending = __ballot_sync(0xFFFFFFFFu, task != 0ull); pending;) {
      uint32_t room = 0;
      if (lane == 0) {
        const long long t0 = clock64();
        while ((room = kTasks - (ttail - ptx::ld_volatile_shared_u32(&S.flag[1]))) == 0u) {
          if (clock64() - t0 > kWaitBudgetCycles) break;
          ptx::nanosleep(32);
        }
      }
      room = __shfl_sync(0xFFFFFFFFu, room, 0);
      if (room == 0u) {
        failed = true;
        break;
      }
      const uint32_t rank = __popc(pending & ((1u << lane) - 1u));
      const bool put = ((pending >> lane) & 1u) && rank < room;
      if (put) S.task[(ttail + rank) % kTasks] = task;
      const uint32_t pm = __ballot_sync(0xFFFFFFFFu, put);
      pending &= ~pm;
      ttail += __popc(pm);
      __syncwarp();
      if (lane == 0) ptx::st_release_cta_shared_u32(&S.flag[0], ttail);
    }
#pragma unroll
    for (int g = 0; g < kGroups; ++g) {
      const bool mine = ready && lane / kBoxDepth == g;
      seen[g] += __popc(__ballot_sync(0xFFFFFFFFu, mine && kind != kBoxExit));
      const uint32_t xm = __ballot_sync(0xFFFFFFFFu, mine && kind == kBoxExit);
      if (xm) want[g] = __shfl_sync(0xFFFFFFFFu, ts, __ffs(xm) - 1);
    }
    bool all_out = true;
#pragma unroll
    for (int g = 0; g < kGroups; ++g) all_out = all_out && want[g] >= 0 && seen[g] == static_cast<uint32_t>(want[g]);
    if (all_out) break;
    if (rm) {
      last_progress = clock64();
    } else {
      if (clock64() - last_progress > kWaitBudgetCycles) failed = true;
      ptx::nanosleep(32);
    }
  }
  if (lane == 0) {
    if (failed) raise_timeout(A);
    ptx::st_release_cta_shared_u32(&S.flag[2], 1u);  // no more tasks
  }
}

// Combining warp: runs the tasks the publishing warp hands over, in order.
template <typename Elt, bool kEarly>
__device__ void combiner(const PArgs& A, const Shared& S) {
  const int lane = lane_id();
  uint32_t head = 0;
  long long last_progress = clock64();
  while (true) {
    uint32_t tail = 0, fin = 0;
    if (lane == 0) {
      fin = ptx::ld_acquire_cta_shared_u32(&S.flag[2]);
      tail = ptx::ld_acquire_cta_shared_u32(&S.flag[0]);  // read after `fin`: final once fin is set
    }
    tail = __shfl_sync(0xFFFFFFFFu, tail, 0);
    fin = __shfl_sync(0xFFFFFFFFu, fin, 0);
    if (head == tail) {
      if (fin) break;
      if (clock64() - last_progress > kWaitBudgetCycles) {
        if (lane == 0) raise_timeout(A);
        break;
      }
      ptx::nanosleep(32);
      continue;
    }
    while (head != tail) {
      if (kEarly) {
        // Row tasks at the head of the ring run side by side, one per lane
        // (kTasks <= 32): their round trips overlap.
        static_assert(kTasks <= 32, "one lane per pending task");
        const uint32_t avail = tail - head;
        unsigned long long tl = 0ull;
        if (static_cast<uint32_t>(lane) < avail) tl = S.task[(head + lane) % kTasks];
        const uint32_t rm =
            __ballot_sync(0xFFFFFFFFu, static_cast<uint32_t>(lane) < avail && static_cast<uint32_t>(tl >> 32) == kTaskRow);
        const int nrow = __ffs(~rm) - 1;  // row tasks before the first other one
        if (nrow > 0) {
          head += static_cast<uint32_t>(nrow);
          __syncwarp();
          if (lane == 0) ptx::st_release_cta_shared_u32(&S.flag[1], head);  // the slots are free again
          if (lane < nrow) {
            const uint32_t arg = static_cast<uint32_t>(tl);
            const int b = static_cast<int>(arg & 0xFFFFFu);
            row_decide_l<Elt>(A, b, static_cast<int>(arg >> 20), req_plan(A, b));
          }
          __syncwarp();
          continue;
        }
      }
      const unsigned long long t = S.task[head % kTasks];
      ++head;
      __syncwarp();
      if (lane == 0) ptx::st_release_cta_shared_u32(&S.flag[1], head);  // the slot is free again
      const uint32_t kind = static_cast<uint32_t>(t >> 32);
      const uint32_t arg = static_cast<uint32_t>(t);
      if (kind == kTaskRequest) {
        const int b = static_cast<int>(arg);
        if (!kEarly) request_combine_w<Elt>(A, b, req_plan(A, b));
      } else if (kind == kTaskRow) {
        if (kEarly && lane == 0) {
          const int b = static_cast<int>(arg & 0xFFFFFu);
          row_decide_l<Elt>(A, b, static_cast<int>(arg >> 20), req_plan(A, b));
        }
        __syncwarp();
      } else {
        race_finalize_w(A, static_cast<int>(arg & 0xFFFFu), static_cast<int>(kind - kTaskRace),
                        race_tag(static_cast<int>((arg >> 16) & 0x7Fu), (arg >> 23) != 0u));
      }
    }
    last_progress = clock64();
  }
}

// ------------------------------------------------------------- dispatch warp
// Lane l < kInbox owns inbox slot l.  A lane without a claim takes a ticket
// on the race queue (fetch-and-add on its head) while unclaimed jobs are
// visible, and up to kSpecTickets lanes hold one ahead of the tail; the job
// under a ticket may still be on its way, so the lane checks it every round
// and, once it and its row's normalisers are there and the slot is free,
// stages it for the CTA's producers.  Tickets past the last job are never
// filled and are dropped when every request is finished.  At most
// gridDim.x * kInbox tickets are open at once, which the queue's slack covers.
__device__ void dispatcher(const PArgs& A, const Shared& S) {
  constexpr uint32_t kNone = 0xFFFFFFFFu;
  const int lane = lane_id();
  const bool own = lane < kInbox;
  uint32_t ticket = kNone;
  long long last_progress = clock64();
  while (true) {
    uint32_t h = 0, t = 0, done = 0;
    unsigned long long job = 0ull;
    if (lane == 0) {
      h = ptx::ld_relaxed_u32(&A.ctr[kCtrRaceHead]);
      t = ptx::ld_relaxed_u32(&A.ctr[kCtrRaceTail]);
      done = ptx::ld_relaxed_u32(&A.ctr[kCtrDone]);
    }
    if (ticket != kNone && ticket < A.race_q_cap) job = ptx::ld_relaxed_u64(&A.race_q[ticket]);
    done = __shfl_sync(0xFFFFFFFFu, done, 0);
    if (done >= static_cast<uint32_t>(A.B)) break;  // every request is finished: no job is left
    h = __shfl_sync(0xFFFFFFFFu, h, 0);
    t = __shfl_sync(0xFFFFFFFFu, t, 0);
    bool prog = false;
    const uint32_t jw = static_cast<uint32_t>(job);
    unsigned long long desc = 0ull;
    if (own && (jw & kJobValid) && ptx::ld_acquire_cta_shared_u32(&S.islot[lane]) == 0u)
      desc = ptx::ld_relaxed_u64(&A.race_desc[jw & 0x3FFFFFu]);  // zero until the decision's store lands
    if (desc != 0ull) {
      RaceJob r;
      r.b = static_cast<int>(jw & 0x3FFFFFu);
      r.round = static_cast<int>((jw >> 22) & 3u);
      r.k = static_cast<int>((jw >> 24) & 0x7Fu);
      const uint32_t tag = static_cast<uint32_t>(job >> 32);
      const int a = static_cast<int>(tag & 0xFFFFu);
      const ReqInfo q = req_plan(A, r.b);
      r.tag = static_cast<int>(tag);
      r.residual = ((tag >> 16) != 0u && r.round < 2) ? 1 : 0;
      r.trow = q.t0 + a;
      r.drow = q.d0 + a;
      r.rword = q.o + static_cast<uint32_t>(a);
      r.expect = race_jobs(A, r.residual != 0);
      r.c = q.c;
      desc = ~desc;
      r.Pt = __uint_as_float(static_cast<uint32_t>(desc));
      r.Pd = __uint_as_float(static_cast<uint32_t>(desc >> 32));
      S.inbox[lane] = r;
      ptx::st_release_cta_shared_u32(&S.islot[lane], 1u);
      ptx::st_relaxed_u64(&A.race_q[ticket], 0ull);  // the queue is zero again for the next call
      ticket = kNone;
      prog = true;
    }
    // New tickets: as many lanes as there are unclaimed jobs in sight, and
    // up to kSpecTickets held ahead of the queue's tail, so that a job queued
    // after a quiet spell is seen with one load rather than three round trips
    // (see the tail, take a ticket, load the job).
    const int held = __popc(__ballot_sync(0xFFFFFFFFu, own && ticket != kNone));
    const bool wants = own && ticket == kNone;
    const uint32_t wm = __ballot_sync(0xFFFFFFFFu, wants);
    const int avail = max(static_cast<int>(t - h), 0) + max(kSpecTickets - held, 0);
    if (wants && __popc(wm & ((1u << lane) - 1u)) < avail) {
      ticket = atomicAdd(&A.ctr[kCtrRaceHead], 1u);
      prog = true;
    }
    if (__any_sync(0xFFFFFFFFu, prog)) {
      last_progress = clock64();
    } else {
      if (clock64() - last_progress > kWaitBudgetCycles) {
        if (lane == 0) raise_timeout(A);
        break;
      }
      ptx::nanosleep(64);
    }
  }
}

// ------------------------------------------------------------- the kernel
template <typename Elt, bool kDirect, bool kEarly>
__global__ void __launch_bounds__(kThreads, 1) verify_persistent_kernel(const PArgs A) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const Shared S = shared_layout(smem);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(ptx::smem_addr(&S.full[s]), 1);
      ptx::mbar_init(ptx::smem_addr(&S.empty[s]), kGroupWarps);
    }
    for (int s = 0; s < kBoxSlots; ++s) {
      ptx::mbar_init(ptx::smem_addr(&S.box_full[s]), 1);
      ptx::mbar_init(ptx::smem_addr(&S.box_empty[s]), 1);
    }
    for (int l = 0; l < kInbox; ++l) S.islot[l] = 0u;
    S.flag[0] = S.flag[1] = S.flag[2] = S.flag[3] = 0u;
    ptx::fence_mbarrier_init();
  }
  // Launched right behind the plan kernel: nothing global is read before the
  // plan (and the previous call) is complete.
  ptx::grid_dependency_wait();
  __syncthreads();
  const int warp = static_cast<int>(threadIdx.x >> 5);
  if (warp < kProducerWarps) {
    if ((threadIdx.x & 31) == 0) producer<Elt, kDirect, kEarly>(A, warp, S);
  } else if (warp < kBookWarp) {
    consumer<Elt, kDirect, kEarly>(A, (warp - kProducerWarps) / kGroupWarps, S);
  } else if (warp == kBookWarp) {
    bookkeeper<kEarly>(A, S);
  } else if (warp == kCombineWarp) {
    combiner<Elt, kEarly>(A, S);
  } else {
    dispatcher(A, S);
  }
  __syncthreads();
  volatile uint32_t& last_cta = S.flag[3];
  if (threadIdx.x == 0) {
    __threadfence();
    last_cta = atomicAdd(&A.ctr[kCtrExit], 1u) == gridDim.x - 1 ? 1u : 0u;
  }
  __syncthreads();
  if (!last_cta) return;
  // The last CTA out re-arms the workspace for the next call: every other CTA
  // has finished.  Early exit leaves the state of rows that were only partly
  // streamed; a call whose waits ran out may leave anything mid-flight.
  __threadfence();
  const bool fault = ptx::ld_relaxed_u32(&A.ctr[kCtrFault]) != 0u;
  const size_t nrow = static_cast<size_t>(A.B) * (A.n_max + 1);
  if (kEarly || fault) {
    for (int i = threadIdx.x; i < A.B; i += blockDim.x) {
      A.rej_hi[i] = 0u;
      A.row_done[i] = 0ull;
      A.req_fin[i] = 0u;
    }
    // rows that were only partly streamed (decided rows reset their count)
    // leave published slots behind
    for (size_t i = threadIdx.x; i < nrow; i += blockDim.x) {
      if (__ldcg(&A.row_cnt[i]) == 0u) continue;
      A.row_cnt[i] = 0u;
      for (int s = 0; s < 2 * A.nseg; ++s) A.part[i * 2 * A.nseg + s] = 0ull;
    }
  }
  if (fault) {
    for (int i = threadIdx.x; i < A.B; i += blockDim.x) {
      A.req_cnt[i] = 0u;
      A.race_cnt[i] = 0u;
      A.race_best[i] = 0ull;
      A.race_desc[i] = 0ull;
    }
    for (uint32_t i = threadIdx.x; i < A.race_q_cap; i += blockDim.x) A.race_q[i] = 0ull;
    for (size_t i = threadIdx.x; i < nrow * 2 * A.nseg; i += blockDim.x) A.part[i] = 0ull;

  }
  __syncthreads();
  if (threadIdx.x == 0) {
    A.ctr[kCtrUnit] = 0u;
    A.ctr[kCtrRaceHead] = 0u;
    A.ctr[kCtrRaceTail] = 0u;
    A.ctr[kCtrDone] = 0u;
    A.ctr[kCtrExit] = 0u;
    A.ctr[kCtrFault] = 0u;
  }
  __threadfence();
}

}  // namespace specdec
