// mtp_kernel.cuh — the MTP shift/insert kernel.
//
// "Accelerating Sonar through speculation", §MTP: the draft's input tokens
// are shifted left by one relative to the target's output hidden states;
// §Single-token MTP scheduling: after the shift a GPU kernel inserts the next
// target token at its position, so the CPU never waits for the accepted
// length.  One warp per request segment; blocks past the segment blocks copy
// the hidden states when a distinct output buffer is given.  A segment that
// lies outside the buffer, or whose accepted length is outside [0, n_b], is
// left unchanged and flagged in the error word.
#pragma once
#include <stdint.h>

#include "specdec.h"

namespace specdec {

constexpr int kMtpThreads = 256;
constexpr int kMtpWarps = kMtpThreads / 32;

struct MtpArgs {
  const int32_t* tokens_in;
  int32_t* tokens_out;
  const int32_t* seg_start;
  const int32_t* draft_len;
  const int32_t* accepted_len;
  const int32_t* next_token;
  int next_token_stride;
  int R, B;
  int seg_blocks;          // blocks [0, seg_blocks) handle token segments
  const uint4* hidden_in;  // bitwise copy of n16 16-byte words (may be null)
  uint4* hidden_out;
  const unsigned char* hidden_in_bytes;  // byte tail (or everything when unaligned)
  unsigned char* hidden_out_bytes;
  long long n16;
  long long tail_begin, tail_end;  // byte range copied bytewise
  uint32_t* err;                   // device error word, or null
};

__global__ void __launch_bounds__(kMtpThreads) mtp_shift_insert_kernel(const MtpArgs A) {
  if (static_cast<int>(blockIdx.x) < A.seg_blocks) {
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.x * kMtpWarps + (threadIdx.x >> 5);
    if (b >= A.B) return;
    const int s = A.seg_start ? A.seg_start[b] : b * (A.R / A.B);
    const int n = A.draft_len[b];
    const int a = A.accepted_len[b];
    if (s < 0 || n < 0 || static_cast<long long>(s) + n >= A.R || a < 0 || a > n) {
      if (lane == 0 && A.err != nullptr) atomicOr(A.err, SPECDEC_DEV_ERR_SEGMENT);
      return;
    }
    const int32_t tok = A.next_token_stride == 0
                            ? A.next_token[b]
                            : A.next_token[static_cast<size_t>(b) * A.next_token_stride + a];
    // Walk the segment in 32-slot pieces: each piece reads its sources (up
    // to one slot past its end) before writing, and later pieces only read
    // slots that no earlier piece wrote, so in-place use is safe.
    for (int base = 0; base <= n; base += 32) {
      const int i = base + lane;
      int32_t val = 0;
      if (i <= n) {
        val = (i < n) ? A.tokens_in[s + i + 1] : A.tokens_in[s + n];
        if (i == a) val = tok;
      }
      __syncwarp();
      if (i <= n) A.tokens_out[s + i] = val;
      __syncwarp();
    }
    return;
  }
  // Hidden-state carry copy: grid-stride over 16-byte words, four loads in
  // flight per thread before the four stores, then the tail.
  const long long nthreads = static_cast<long long>(gridDim.x - A.seg_blocks) * kMtpThreads;
  const long long t = static_cast<long long>(blockIdx.x - A.seg_blocks) * kMtpThreads + threadIdx.x;
  long long k = t;
  for (; k + 3 * nthreads < A.n16; k += 4 * nthreads) {
    const uint4 v0 = __ldcs(A.hidden_in + k);
    const uint4 v1 = __ldcs(A.hidden_in + k + nthreads);
    const uint4 v2 = __ldcs(A.hidden_in + k + 2 * nthreads);
    const uint4 v3 = __ldcs(A.hidden_in + k + 3 * nthreads);
    __stcs(A.hidden_out + k, v0);
    __stcs(A.hidden_out + k + nthreads, v1);
    __stcs(A.hidden_out + k + 2 * nthreads, v2);
    __stcs(A.hidden_out + k + 3 * nthreads, v3);
  }
  for (; k < A.n16; k += nthreads) A.hidden_out[k] = A.hidden_in[k];
  for (long long k = A.tail_begin + t; k < A.tail_end; k += nthreads)
    A.hidden_out_bytes[k] = A.hidden_in_bytes[k];
}

}  // namespace specdec
