// verify_kernel.cuh — the fused verify/accept kernel for sm_103a.
//
// One thread-block cluster of C CTAs scores one (request b, row j).  CTA r of
// the cluster owns vocabulary slice [r*S, min(V, (r+1)*S)).  Per CTA:
//   1. the slice of target row j (and of draft row j when the request samples
//      and j < n_b) is staged in shared memory with 1-D bulk copies (TMA
//      engine) in up to kChunks pieces, each tracked by its own mbarrier;
//   2. max and sum of exp(s*(x - max)) over the slice -> (m, S) per tensor;
//      the cluster combines the C partial pairs over distributed shared
//      memory into the row's log-sum-exp;
//   3. the acceptance test u_j < p_j(x_j) / q_j(x_j) (rows j < n_b);
//   4. only when the row is rejected, or is the bonus row j = n_b, the
//      exponential race argmax_v r_v / E_v runs over the slice still in
//      shared memory (r = max(0, p - q) or r = p), and the cluster combines
//      the C slice winners;
//   greedy requests (T = 0) replace 2-4 by an argmax of the target slice.
// CTA rank 0 publishes the row's result and bumps the request's arrival
// counter; whichever row of the request arrives last (device atomic, no
// waiting) scans the rows in order, picks the first rejection, writes
// accepted_len and out_tokens and re-arms the counter.
//
// Sources: "Accelerating Sonar through speculation" §Speculative decoding
// (stages Acceptance, Target generation), §Target-draft; the min(1, p/q) rule
// of "Fast Inference from Transformers via Speculative Decoding"; Philox from
// Salmon et al. (SC'11).
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "philox.cuh"
#include "ptx.cuh"
#include "specdec.h"

namespace specdec {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kChunks = 4;
constexpr int kScratchBytes = 1024;
// Roughly two seconds of SM clock: any wait on a bulk copy gives up after it.
constexpr long long kWaitBudgetCycles = 4000000000LL;

struct VerifyArgs {
  const void* target;
  const void* draft;
  const int32_t* draft_tokens;
  const int32_t* draft_len;
  const float* temperature;
  int32_t* accepted_len;
  int32_t* out_tokens;
  float* row_lse;
  uint32_t* err;                   // sticky error word
  uint32_t* arrivals;              // [B] rows of the request finished so far
  unsigned long long* row_winner;  // [B, n_max+1] packed (key, ~index)
  uint32_t* row_accept;            // [B, n_max+1] acceptance flag of row j
  uint32_t* row_state;             // [B, n_max+1] published verdict: 0 unknown, 1 accepted, 2 rejected
  uint32_t seed_lo, seed_hi;
  int B, n_max, V;
  int C;      // CTAs per row (cluster size)
  int S;      // slice length in elements
  int bulk;   // 1: rows are 16-byte aligned, stage with bulk copies
  int slice_stride_bytes;  // bytes reserved per staged slice in shared memory
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
  static constexpr int kVec = 4;  // elements per 16-byte vector
  using MaxAcc = float;
  __device__ static __forceinline__ MaxAcc max_init() { return -INFINITY; }
  __device__ static __forceinline__ void max_vec(const uint4& w, MaxAcc& m) {
    m = fmaxf(fmaxf(m, __uint_as_float(w.x)), __uint_as_float(w.y));
    m = fmaxf(fmaxf(m, __uint_as_float(w.z)), __uint_as_float(w.w));
  }
  __device__ static __forceinline__ float max_value(MaxAcc m) { return m; }
  // acc += 2^(x c - K) for the four elements, two lanes of f32x2 at a time
  __device__ static __forceinline__ void sum_vec(const uint4& w, float2 cc, float2 nk, float2& acc) {
    float2 a = __ffma2_rn(make_float2(__uint_as_float(w.x), __uint_as_float(w.y)), cc, nk);
    float2 b = __ffma2_rn(make_float2(__uint_as_float(w.z), __uint_as_float(w.w)), cc, nk);
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

// bf16 is handled as raw 16-bit patterns: widening to fp32 is a shift, and
// the max runs on packed pairs (exact).
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

// ------------------------------------------------------------- reductions
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
__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    unsigned long long w = __shfl_xor_sync(0xFFFFFFFFu, v, o);
    v = w > v ? w : v;
  }
  return v;
}
__device__ __forceinline__ int warp_min_i(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

// Two block-wide reductions at once; `red` holds 2*kWarps floats.
template <bool kMax>
__device__ __forceinline__ float2 block_reduce2(float a, float b, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  a = kMax ? warp_max(a) : warp_sum(a);
  b = kMax ? warp_max(b) : warp_sum(b);
  __syncthreads();  // `red` may still be read from a previous reduction
  if (lane == 0) {
    red[warp] = a;
    red[kWarps + warp] = b;
  }
  __syncthreads();
  float ra = red[0], rb = red[kWarps];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) {
    ra = kMax ? fmaxf(ra, red[w]) : ra + red[w];
    rb = kMax ? fmaxf(rb, red[kWarps + w]) : rb + red[kWarps + w];
  }
  return make_float2(ra, rb);
}

__device__ __forceinline__ unsigned long long block_max_u64(unsigned long long v,
                                                            unsigned long long* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_max_u64(v);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  unsigned long long r = red[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) r = red[w] > r ? red[w] : r;
  return r;
}

__device__ __forceinline__ int block_min_i(int v, int* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_min_i(v);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  int r = red[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) r = min(r, red[w]);
  return r;
}

// Order-preserving map of a float onto uint32 (larger float -> larger uint).
__device__ __forceinline__ uint32_t orderable(float f) {
  const uint32_t u = __float_as_uint(f + 0.0f);  // -0 -> +0: equal values, equal keys
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ unsigned long long pack_key(uint32_t key_bits, int idx) {
  return (static_cast<unsigned long long>(key_bits) << 32) |
         static_cast<unsigned long long>(0xFFFFFFFFu - static_cast<uint32_t>(idx));
}
__device__ __forceinline__ int unpack_index(unsigned long long packed) {
  return static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(packed & 0xFFFFFFFFull));
}

// E = -ln U, accurate to about one ulp relative even for U close to 1 (where
// the winning keys come from).
__device__ __forceinline__ float exp_variate(uint32_t word) {
  return -logf(uniform_from_word(word));
}

// ------------------------------------------------------------- the kernel
template <typename Elt>
__global__ void __launch_bounds__(kThreads) verify_kernel(const VerifyArgs A) {
  using Ops = EltOps<Elt>;
  constexpr int VEC = Ops::kVec;
  extern __shared__ __align__(1024) unsigned char smem[];
  uint64_t* mbar = reinterpret_cast<uint64_t*>(smem);                               // [kChunks]
  float* red_f = reinterpret_cast<float*>(smem + 64);                               // [2*kWarps]
  unsigned long long* red_u = reinterpret_cast<unsigned long long*>(smem + 128);    // [kWarps]
  int* red_i = reinterpret_cast<int*>(smem + 192);                                  // [kWarps]
  // cluster-visible slots (read by peers over distributed shared memory)
  float4* slot_lse = reinterpret_cast<float4*>(smem + 256);  // (K_t, S_t, K_d, S_d) of this slice
  uint32_t* slot_veto = reinterpret_cast<uint32_t*>(smem + 272);                     // rank 0 only
  unsigned long long* slot_win = reinterpret_cast<unsigned long long*>(smem + 280);
  unsigned long long* slot_alt = reinterpret_cast<unsigned long long*>(smem + 288);
  float* bcast = reinterpret_cast<float*>(smem + 320);                               // [8]
  Elt* st = reinterpret_cast<Elt*>(smem + kScratchBytes);
  Elt* sd = reinterpret_cast<Elt*>(smem + kScratchBytes + A.slice_stride_bytes);

  const int tid = threadIdx.x;
  const uint32_t rank = ptx::cluster_ctarank();
  const int rows = A.n_max + 1;
  // Row-major order over (row j, request b): every request's row 0 comes
  // before any row 1, so when row j is scored the verdicts of its request's
  // earlier rows are usually published already.
  const long long unit = static_cast<long long>(blockIdx.x) / A.C;
  const int j = static_cast<int>(unit / A.B);
  const int b = static_cast<int>(unit % A.B);

  const int L_raw = A.draft_len[b];
  const int L = min(max(L_raw, 0), A.n_max);
  if (j > L) return;  // every CTA of this cluster sees the same (b, j)

  const float T = A.temperature[b];
  const bool greedy = !(T > 0.f) || T < 1e-6f || A.draft == nullptr;
  const bool need_draft = !greedy && j < L;

  const int v0 = static_cast<int>(rank) * A.S;
  const int v1 = min(A.V, v0 + A.S);
  const int n_el = max(0, v1 - v0);
  const size_t row_t = static_cast<size_t>(b) * rows + j;
  const size_t row_d = static_cast<size_t>(b) * A.n_max + j;
  const Elt* gt = static_cast<const Elt*>(A.target) + row_t * A.V + v0;
  const Elt* gd = need_draft ? static_cast<const Elt*>(A.draft) + row_d * A.V + v0 : nullptr;

  // ------------------------------------------------ 1. stage the slices
  int chunk_elems = n_el;
  int nchunks = 1;
  bool timed_out = false;
  if (A.bulk) {
    chunk_elems = ((n_el + kChunks - 1) / kChunks + VEC - 1) / VEC * VEC;
    nchunks = chunk_elems > 0 ? (n_el + chunk_elems - 1) / chunk_elems : 0;
    if (tid == 0) {
      for (int k = 0; k < nchunks; ++k) ptx::mbar_init(ptx::smem_addr(&mbar[k]), 1);
      ptx::fence_mbarrier_init();
      const uint64_t pol = ptx::policy_evict_first();
      for (int k = 0; k < nchunks; ++k) {
        const int e0 = k * chunk_elems;
        const int e1 = min(n_el, e0 + chunk_elems);
        const uint32_t cb = static_cast<uint32_t>(e1 - e0) * sizeof(Elt);
        const uint32_t bar = ptx::smem_addr(&mbar[k]);
        ptx::mbar_arrive_expect_tx(bar, need_draft ? 2 * cb : cb);
        ptx::bulk_g2s(ptx::smem_addr(st + e0), gt + e0, cb, bar, pol);
        if (need_draft) ptx::bulk_g2s(ptx::smem_addr(sd + e0), gd + e0, cb, bar, pol);
      }
    }
    __syncthreads();  // the barriers are initialised before anyone waits on them
  } else {
    for (int e = tid; e < n_el; e += kThreads) {
      st[e] = gt[e];
      if (need_draft) sd[e] = gd[e];
    }
    __syncthreads();
  }
  const int nvec = n_el / VEC;  // whole 16-byte vectors; the rest is the tail
  const uint4* vt = reinterpret_cast<const uint4*>(st);
  const uint4* vd = reinterpret_cast<const uint4*>(sd);

  // ------------------------------------------------ 2a. slice maxima
  typename Ops::MaxAcc mta = Ops::max_init(), mda = Ops::max_init();
  for (int k = 0; k < nchunks; ++k) {
    if (A.bulk && !ptx::mbar_wait_bounded(ptx::smem_addr(&mbar[k]), 0, kWaitBudgetCycles))
      timed_out = true;
    const int e0 = k * chunk_elems;
    const int e1 = min(n_el, e0 + chunk_elems);
    const int vend = min(e1 / VEC, nvec);
    for (int vi = e0 / VEC + tid; vi < vend; vi += kThreads) {
      Ops::max_vec(vt[vi], mta);
      if (need_draft) Ops::max_vec(vd[vi], mda);
    }
  }
  float mt = Ops::max_value(mta), md = Ops::max_value(mda);
  for (int e = nvec * VEC + tid; e < n_el; e += kThreads) {
    mt = fmaxf(mt, Ops::at(st, e));
    if (need_draft) md = fmaxf(md, Ops::at(sd, e));
  }
  const float2 mm = block_reduce2<true>(mt, md, red_f);
  const float Mt_cta = mm.x, Md_cta = mm.y;

  unsigned long long row_packed = 0;
  uint32_t accept = 0;
  float lse_t = NAN, lse_d = NAN;

  if (greedy) {
    // ---------------------------------------------- greedy: slice argmax
    int first = 0x7FFFFFFF;
    for (int vi = tid; vi < nvec && first == 0x7FFFFFFF; vi += kThreads) {
      float f[VEC];
      Ops::unpack(vt[vi], f);
#pragma unroll
      for (int i = VEC - 1; i >= 0; --i)
        if (f[i] == Mt_cta) first = vi * VEC + i;
    }
    for (int e = nvec * VEC + tid; e < n_el; e += kThreads)
      if (Ops::at(st, e) == Mt_cta) first = min(first, e);
    first = block_min_i(first, red_i);
    if (tid == 0)
      *slot_win = (n_el > 0 && first != 0x7FFFFFFF) ? pack_key(orderable(Mt_cta), v0 + first) : 0ull;
    ptx::cluster_sync();
    if (tid == 0 && rank == 0) {
      unsigned long long best = 0;
      for (int r = 0; r < A.C; ++r) {
        unsigned long long w = ptx::ld_cluster_u64(ptx::map_to_rank(ptx::smem_addr(slot_win), r));
        best = w > best ? w : best;
      }
      row_packed = best;
    }
  } else {
    // ---------------------------------------------- 2b. sums and the row LSE
    // In log2 units: K = max(x) * c and S = sum 2^(x c - K), c = log2(e) / T,
    // so that ln sum exp(x / T) = ln 2 * (K + log2 S).
    const float s = 1.0f / T;
    const float c = s * 1.4426950408889634f;
    const float Kt_cta = Mt_cta * c, Kd_cta = Md_cta * c;
    float2 at2 = make_float2(0.f, 0.f), ad2 = make_float2(0.f, 0.f);
    if (n_el > 0) {
      const float2 cc = make_float2(c, c);
      const float2 nkt = make_float2(-Kt_cta, -Kt_cta), nkd = make_float2(-Kd_cta, -Kd_cta);
      for (int vi = tid; vi < nvec; vi += kThreads) {
        Ops::sum_vec(vt[vi], cc, nkt, at2);
        if (need_draft) Ops::sum_vec(vd[vi], cc, nkd, ad2);
      }
      for (int e = nvec * VEC + tid; e < n_el; e += kThreads) {
        at2.x += fast_ex2(fmaf(Ops::at(st, e), c, -Kt_cta));
        if (need_draft) ad2.x += fast_ex2(fmaf(Ops::at(sd, e), c, -Kd_cta));
      }
    }
    const float2 ss = block_reduce2<false>(at2.x + at2.y, ad2.x + ad2.y, red_f);
    if (tid == 0) {
      *slot_lse = make_float4(Kt_cta, ss.x, Kd_cta, ss.y);
      if (rank == 0) {
        // Veto the race when an earlier row of this request is already
        // published as rejected: this row cannot be the first rejection.
        uint32_t veto = 0;
        for (int jj = 0; jj < j && !veto; ++jj)
          veto = ptx::ld_relaxed_u32(&A.row_state[static_cast<size_t>(b) * rows + jj]) == 2u;
        *slot_veto = veto;
      }
    }
    ptx::cluster_sync();
    if (tid == 0) {
      // Fixed combine order over ranks: every CTA obtains identical values.
      float Kt = -INFINITY, Kd = -INFINITY;
      for (int r = 0; r < A.C; ++r) {
        const uint32_t a = ptx::map_to_rank(ptx::smem_addr(slot_lse), r);
        Kt = fmaxf(Kt, ptx::ld_cluster_f32(a));
        Kd = fmaxf(Kd, ptx::ld_cluster_f32(a + 8));
      }
      float St = 0.f, Sd = 0.f;
      for (int r = 0; r < A.C; ++r) {
        const uint32_t a = ptx::map_to_rank(ptx::smem_addr(slot_lse), r);
        const float kt = ptx::ld_cluster_f32(a), st_ = ptx::ld_cluster_f32(a + 4);
        const float kd = ptx::ld_cluster_f32(a + 8), sd_ = ptx::ld_cluster_f32(a + 12);
        if (st_ > 0.f) St += st_ * exp2f(kt - Kt);
        if (sd_ > 0.f) Sd += sd_ * exp2f(kd - Kd);
      }
      bcast[0] = Kt;
      bcast[1] = St;
      bcast[2] = Kd;
      bcast[3] = Sd;
      bcast[4] = __uint_as_float(ptx::ld_cluster_u32(ptx::map_to_rank(ptx::smem_addr(slot_veto), 0)));
    }
    __syncthreads();
    const float Kt = bcast[0], l2St = log2f(bcast[1]);
    const float Kd = bcast[2], l2Sd = need_draft ? log2f(bcast[3]) : 0.f;
    const bool veto = __float_as_uint(bcast[4]) != 0u;
    const float Pt = Kt + l2St, Pd = Kd + l2Sd;  // p_v = 2^(t_v c - Pt), q_v = 2^(d_v c - Pd)
    lse_t = Pt * 0.69314718055994531f;
    if (need_draft) lse_d = Pd * 0.69314718055994531f;

    // ---------------------------------------------- 3. acceptance test
    bool race = (j == L);
    if (j < L) {
      const int x = A.draft_tokens[static_cast<size_t>(b) * A.n_max + j];
      if (x >= 0 && x < A.V) {
        const float tx = Ops::at(static_cast<const Elt*>(A.target), row_t * A.V + x);
        const float dx = Ops::at(static_cast<const Elt*>(A.draft), row_d * A.V + x);
        // log2 p(x) - log2 q(x)
        const float l2ratio = (fmaf(tx, c, -Kt) - l2St) - (fmaf(dx, c, -Kd) - l2Sd);
        const float ratio = exp2f(l2ratio);
        const Philox4 r = philox4x32_10(0u, static_cast<uint32_t>(j), static_cast<uint32_t>(b), 0u,
                                        A.seed_lo, A.seed_hi);
        accept = (uniform_from_word(r.w[0]) < ratio) ? 1u : 0u;
      }
      race = !accept;
      if (rank == 0 && tid == 0)
        ptx::st_relaxed_u32(&A.row_state[row_t], accept ? 1u : 2u);  // publish early
    }
    if (veto) race = false;

    // ---------------------------------------------- 4. exponential race
    if (race) {
      for (int pass = 0; pass < 2; ++pass) {
        // pass 0: r = max(0, p - q) (rejected row) or r = p (bonus row);
        // pass 1 (only if every residual weight vanished): r = p.
        const bool residual = need_draft && pass == 0;
        float R = 0.f, Eb = 1.f;
        int idx = -1;
        for (int vi = tid; vi < nvec; vi += kThreads) {
          float ft[VEC], fd[VEC];
          Ops::unpack(vt[vi], ft);
          if (residual) Ops::unpack(vd[vi], fd);
          const int v = v0 + vi * VEC;
#pragma unroll
          for (int g = 0; g < VEC / 4; ++g) {
            const Philox4 rnd =
                philox4x32_10(static_cast<uint32_t>(v + 4 * g) >> 2, static_cast<uint32_t>(j),
                              static_cast<uint32_t>(b), 1u, A.seed_lo, A.seed_hi);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int e = 4 * g + i;
              float r = fast_ex2(fmaf(ft[e], c, -Pt));
              if (residual) r -= fast_ex2(fmaf(fd[e], c, -Pd));
              if (r > 0.f) {
                const float U = uniform_from_word(rnd.w[i]);
                // -ln U >= 1 - U, so r / (1 - U) bounds the key r / E from
                // above: only a possible winner pays for the logarithm.
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
        for (int e = nvec * VEC + tid; e < n_el; e += kThreads) {
          const int v = v0 + e;
          float r = fast_ex2(fmaf(Ops::at(st, e), c, -Pt));
          if (residual) r -= fast_ex2(fmaf(Ops::at(sd, e), c, -Pd));
          if (r > 0.f) {
            const Philox4 rnd = philox4x32_10(static_cast<uint32_t>(v) >> 2, static_cast<uint32_t>(j),
                                              static_cast<uint32_t>(b), 1u, A.seed_lo, A.seed_hi);
            const float E = exp_variate(rnd.w[v & 3]);
            if (r * Eb > R * E || (r * Eb == R * E && idx > v)) {
              R = r;
              Eb = E;
              idx = v;
            }
          }
        }
        unsigned long long mine = idx >= 0 ? pack_key(__float_as_uint(R / Eb), idx) : 0ull;
        mine = block_max_u64(mine, red_u);
        unsigned long long* slot = pass == 0 ? slot_win : slot_alt;
        if (tid == 0) *slot = mine;
        ptx::cluster_sync();
        if (tid == 0) {
          unsigned long long best = 0;
          for (int r = 0; r < A.C; ++r) {
            unsigned long long w = ptx::ld_cluster_u64(ptx::map_to_rank(ptx::smem_addr(slot), r));
            best = w > best ? w : best;
          }
          reinterpret_cast<unsigned long long*>(bcast)[3] = best;
        }
        __syncthreads();
        row_packed = reinterpret_cast<unsigned long long*>(bcast)[3];
        __syncthreads();
        if (row_packed != 0ull || !need_draft) break;
      }
    }
  }

  // Peers may still read this CTA's cluster-visible slots: wait for all of
  // them before anyone leaves.
  ptx::cluster_sync();

  if (timed_out) {
    // Give copies still in flight a second bounded chance to land before the
    // shared memory is released.
    for (int k = 0; k < nchunks; ++k)
      (void)ptx::mbar_wait_bounded(ptx::smem_addr(&mbar[k]), 0, kWaitBudgetCycles);
    if (tid == 0) atomicOr(A.err, SPECDEC_DEV_ERR_TIMEOUT);
  }
  if (rank != 0 || tid != 0) return;

  // ------------------------------------------------ publish the row
  A.row_winner[row_t] = row_packed;
  A.row_accept[row_t] = accept;
  if (A.row_lse != nullptr && !greedy) {
    A.row_lse[row_t * 2 + 0] = lse_t;
    if (need_draft) A.row_lse[row_t * 2 + 1] = lse_d;
  }
  __threadfence();
  const uint32_t arrived = atomicAdd(&A.arrivals[b], 1u);
  if (arrived != static_cast<uint32_t>(L)) return;

  // ------------------------------------------------ 5. finalise the request
  __threadfence();
  uint32_t errbits = 0;
  if (L_raw != L) errbits |= SPECDEC_DEV_ERR_DRAFT_LEN;
  if (greedy && T != 0.f) errbits |= SPECDEC_DEV_ERR_TEMPERATURE;
  int a = L, y = 0;
  for (int jj = 0; jj <= L; ++jj) {
    const size_t r = static_cast<size_t>(b) * rows + jj;
    const int win = unpack_index(__ldcg(&A.row_winner[r]));
    if (jj == L) {
      a = L;
      y = win;
      break;
    }
    const int x = A.draft_tokens[static_cast<size_t>(b) * A.n_max + jj];
    const bool valid = x >= 0 && x < A.V;
    if (!valid) errbits |= SPECDEC_DEV_ERR_TOKEN;
    const bool ok = greedy ? (valid && x == win) : (__ldcg(&A.row_accept[r]) != 0u);
    if (!ok) {
      a = jj;
      y = win;
      break;
    }
  }
  A.accepted_len[b] = a;
  int32_t* out = A.out_tokens + static_cast<size_t>(b) * rows;
  for (int k = 0; k < rows; ++k)
    out[k] = k < a ? A.draft_tokens[static_cast<size_t>(b) * A.n_max + k] : (k == a ? y : -1);
  for (int k = 0; k <= L; ++k) A.row_state[static_cast<size_t>(b) * rows + k] = 0u;
  A.arrivals[b] = 0u;
  if (errbits) atomicOr(A.err, errbits);
}

}  // namespace specdec
