// api.cu — the C ABI of libspecdec.so: argument checks, workspace layout,
// launch shapes and kernel launches.  The declarations, with the meaning of
// every argument, are in include/specdec.h.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "mtp_kernel.cuh"
#include "specdec.h"
#include "verify_persistent.cuh"

namespace specdec {
namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Chunking of a vocabulary row for elements of `elt` bytes.
struct Chunking {
  int ch, nch, nseg, chr, nrc;
};
// Bytes per stream chunk.  Larger chunks keep more bytes in flight per
// consumer group and win on long launches; short launches balance better
// with 24 KB chunks (measured on GB300 over batches of 148 MB to 2.8 GB).
constexpr int kSmallChunkBytes = 24 * 1024;
int chunk_bytes_for(int B, int n_max, int V, int elt) {
  const double upper = static_cast<double>(B) * (2 * n_max + 1) * V * elt;  // bytes if every row is read
  return upper >= 300e6 ? kStageBytes : kSmallChunkBytes;
}
Chunking chunking(int V, int elt, int chunk_bytes) {
  Chunking c;
  c.ch = chunk_bytes / elt;
  c.nch = (V + c.ch - 1) / c.ch;
  c.nseg = (c.nch + kSegChunks - 1) / kSegChunks;
  // Race job: half a chunk of target and half of draft (a race on p: a whole
  // chunk of target).  Short bf16 launches (24 KB chunks) take quarter-chunk
  // jobs instead: their races run mostly after the stream, on idle groups,
  // where shorter jobs finish a race sooner (measured on GB300: configs of
  // 148 and 199 MB 6 % and 5 % faster; eighth-chunk jobs and quarter-chunk
  // jobs on the long launches were slower).
  c.chr = (elt == 2 && chunk_bytes == kSmallChunkBytes) ? c.ch / 4 : c.ch / 2;
  c.nrc = (V + c.chr - 1) / c.chr;
  return c;
}

struct WsLayout {
  size_t race_q_cap;  // slots of the race queue
  size_t err, ctr, race_q, req_cnt, race_best, race_cnt, race_desc, rej_hi, row_done, req_fin,
      row_cnt, row_P, row_arg, part, rinfo, n_units, units, total;
};

// Every section is 256-byte aligned.  Sections that must start at zero
// (counters, queue, race maxima and descriptors, result slots) are re-zeroed
// by the kernel as it finishes.
WsLayout ws_layout(int B, int n_max, int V) {
  // the most chunks and race jobs any launch uses: fp32 with 24 KB chunks
  // (race jobs of 3 072 entries, as many as bf16's quarter-chunk jobs)
  const Chunking c = chunking(V, 4, kSmallChunkBytes);
  const size_t rows = static_cast<size_t>(B) * (n_max + 1);
  WsLayout w;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += align_up(bytes, kAlign);
    return at;
  };
  w.err = take(4);
  w.ctr = take(kCtrWords * 4);
  // every job a call can queue (at most 3 nrc per request: the thresholded
  // round, its rerun and the race on p, at most nrc jobs each) plus the
  // tickets the CTAs may hold past the last job
  w.race_q_cap = 3 * static_cast<size_t>(B) * c.nrc + static_cast<size_t>(kMaxCtas) * kInbox;
  w.race_q = take(w.race_q_cap * 8);
  w.req_cnt = take(4 * static_cast<size_t>(B));
  w.race_best = take(8 * static_cast<size_t>(B));
  w.race_cnt = take(4 * static_cast<size_t>(B));
  w.race_desc = take(8 * static_cast<size_t>(B));
  w.rej_hi = take(4 * static_cast<size_t>(B));
  w.row_done = take(8 * static_cast<size_t>(B));
  w.req_fin = take(4 * static_cast<size_t>(B));
  w.row_cnt = take(4 * rows);
  w.row_P = take(8 * rows);
  w.row_arg = take(4 * rows);
  w.part = take(8 * rows * 2 * c.nseg);
  // the plan, rewritten by every call: request parameters, the unit count
  // and a record per row-tensor to stream (at most B (2 n_max + 1))
  w.rinfo = take(16 * static_cast<size_t>(B));
  w.n_units = take(4);
  w.units = take(16 * static_cast<size_t>(B) * (2 * n_max + 1));
  w.total = off;
  return w;
}

template <typename Elt, bool kDirect, bool kEarly>
cudaError_t launch_persistent(const PArgs& args, cudaStream_t st) {
  verify_plan_kernel<kEarly><<<1, kPlanThreads, 0, st>>>(args);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  static int sms[64] = {0};
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (sms[dev] == 0) {
    e = cudaFuncSetAttribute(verify_persistent_kernel<Elt, kDirect, kEarly>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kPersistentSmemBytes));
    if (e != cudaSuccess) return e;
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    sms[dev] = n < kMaxCtas ? n : kMaxCtas;
  }
  // Programmatic dependent launch: the verify grid is scheduled while the
  // plan kernel runs and waits for it on the device (griddepcontrol.wait).
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(sms[dev]));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kPersistentSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, verify_persistent_kernel<Elt, kDirect, kEarly>, args);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace specdec

using namespace specdec;

extern "C" size_t specdec_verify_workspace_bytes(int32_t B, int32_t n_max, int32_t V) {
  if (B <= 0 || n_max < 0 || n_max > SPECDEC_MAX_DRAFT || V <= 0 || V > SPECDEC_MAX_VOCAB) return 0;
  if (B > SPECDEC_MAX_BATCH) return 0;
  return ws_layout(B, n_max, V).total;
}

extern "C" specdec_status_t specdec_workspace_init(void* workspace, size_t bytes, void* stream) {
  if (workspace == nullptr || bytes == 0) return SPECDEC_ERR_INVALID_ARG;
  return cudaMemsetAsync(workspace, 0, bytes, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? SPECDEC_OK
             : SPECDEC_ERR_CUDA;
}

extern "C" specdec_status_t specdec_verify_launch_shape(int32_t B, int32_t n_max, int32_t V,
                                                        specdec_dtype_t dtype, int32_t* chunks_per_row,
                                                        int32_t* chunk_elems) {
  if (B <= 0 || n_max < 0 || n_max > SPECDEC_MAX_DRAFT || V <= 0 || V > SPECDEC_MAX_VOCAB ||
      (dtype != SPECDEC_F32 && dtype != SPECDEC_BF16))
    return SPECDEC_ERR_INVALID_ARG;
  const int elt = dtype == SPECDEC_F32 ? 4 : 2;
  const Chunking c = chunking(V, elt, chunk_bytes_for(B, n_max, V, elt));
  if (chunks_per_row) *chunks_per_row = c.nch;
  if (chunk_elems) *chunk_elems = c.ch;
  return SPECDEC_OK;
}

namespace specdec {
namespace {

// One verify call, dense or packed (cu_rows != nullptr).
struct VerifyCall {
  const void* target;
  const void* draft;
  specdec_dtype_t dtype;
  int32_t B, n_max, V;
  const int32_t* draft_tokens;
  const int32_t* draft_len;   // dense
  const int32_t* cu_rows;     // packed
  int32_t total_rows;         // packed
  const int32_t* pos_offset;  // packed, optional
  int early_exit;
  const float* temperature;
  uint64_t seed;
  int32_t* accepted_len;
  int32_t* out_tokens;
  float* row_lse;
  void* workspace;
  size_t workspace_bytes;
  void* stream;
};

specdec_status_t verify_launch(const VerifyCall& c) {
  const int32_t B = c.B, n_max = c.n_max, V = c.V;
  const WsLayout wl = ws_layout(B, n_max, V);
  if (c.workspace == nullptr || !aligned16(c.workspace)) return SPECDEC_ERR_WORKSPACE;
  if (c.workspace_bytes < wl.total) return SPECDEC_ERR_WORKSPACE;
  const int elt = c.dtype == SPECDEC_F32 ? 4 : 2;
  const int chunk_bytes = chunk_bytes_for(B, n_max, V, elt);
  const Chunking ck = chunking(V, elt, chunk_bytes);
  // Early exit on a short batch: every row is claimed before the first
  // decision lands, so it runs in request order, counting the bytes it reads.
  const bool early = c.early_exit && chunk_bytes != kSmallChunkBytes;
  if (ck.nseg > 32 || ck.nrc >= 256) return SPECDEC_ERR_UNSUPPORTED;  // fixed by the vocabulary cap

  unsigned char* ws = static_cast<unsigned char*>(c.workspace);
  PArgs a;
  memset(&a, 0, sizeof a);
  a.target = c.target;
  a.draft = n_max > 0 ? c.draft : nullptr;
  a.draft_tokens = c.draft_tokens;
  a.draft_len = c.draft_len;
  a.cu_rows = c.cu_rows;
  a.total_rows = c.total_rows;
  a.pos_offset = c.pos_offset;
  a.temperature = c.temperature;
  a.accepted_len = c.accepted_len;
  a.out_tokens = c.out_tokens;
  a.row_lse = c.row_lse;
  a.seed_lo = static_cast<uint32_t>(c.seed & 0xFFFFFFFFull);
  a.seed_hi = static_cast<uint32_t>(c.seed >> 32);
  a.B = B;
  a.n_max = n_max;
  a.V = V;
  a.nch = ck.nch;
  a.nseg = ck.nseg;
  a.ch = ck.ch;
  a.nrc = ck.nrc;
  a.chr = ck.chr;
  a.race_q_cap = static_cast<uint32_t>(wl.race_q_cap);
  a.count_bytes = c.early_exit ? 1 : 0;
  a.err = reinterpret_cast<uint32_t*>(ws + wl.err);
  a.ctr = reinterpret_cast<uint32_t*>(ws + wl.ctr);
  a.race_q = reinterpret_cast<unsigned long long*>(ws + wl.race_q);
  a.req_cnt = reinterpret_cast<uint32_t*>(ws + wl.req_cnt);
  a.race_best = reinterpret_cast<unsigned long long*>(ws + wl.race_best);
  a.race_cnt = reinterpret_cast<uint32_t*>(ws + wl.race_cnt);
  a.race_desc = reinterpret_cast<unsigned long long*>(ws + wl.race_desc);
  a.row_cnt = reinterpret_cast<uint32_t*>(ws + wl.row_cnt);
  a.row_P = reinterpret_cast<float2*>(ws + wl.row_P);
  a.row_arg = reinterpret_cast<int32_t*>(ws + wl.row_arg);
  a.part = reinterpret_cast<unsigned long long*>(ws + wl.part);
  a.rinfo = reinterpret_cast<int4*>(ws + wl.rinfo);
  a.n_units = reinterpret_cast<uint32_t*>(ws + wl.n_units);
  a.units = reinterpret_cast<int4*>(ws + wl.units);
  a.rej_hi = reinterpret_cast<uint32_t*>(ws + wl.rej_hi);
  a.row_done = reinterpret_cast<unsigned long long*>(ws + wl.row_done);
  a.req_fin = reinterpret_cast<uint32_t*>(ws + wl.req_fin);
  // Bulk copies need 16-byte aligned rows and chunks.
  const bool bulk = (static_cast<long long>(V) * elt) % 16 == 0 && aligned16(c.target) &&
                    (a.draft == nullptr || aligned16(a.draft));

  cudaStream_t st = static_cast<cudaStream_t>(c.stream);
  cudaError_t e;
  if (early) {
    if (c.dtype == SPECDEC_F32)
      e = bulk ? launch_persistent<float, false, true>(a, st) : launch_persistent<float, true, true>(a, st);
    else
      e = bulk ? launch_persistent<uint16_t, false, true>(a, st) : launch_persistent<uint16_t, true, true>(a, st);
  } else {
    if (c.dtype == SPECDEC_F32)
      e = bulk ? launch_persistent<float, false, false>(a, st) : launch_persistent<float, true, false>(a, st);
    else
      e = bulk ? launch_persistent<uint16_t, false, false>(a, st) : launch_persistent<uint16_t, true, false>(a, st);
  }
  return e == cudaSuccess ? SPECDEC_OK : SPECDEC_ERR_CUDA;
}

}  // namespace
}  // namespace specdec

namespace {
// Host-side checks of spec_verify's arguments (shared with
// spec_verify_no_alloc, which must reject a bad call before it enqueues its
// workspace clear).
specdec_status_t check_verify_args(const void* target_logits, specdec_dtype_t dtype, int32_t B, int32_t n_max,
                                   int32_t V, const int32_t* draft_tokens, const int32_t* draft_len,
                                   const float* temperature, const int32_t* accepted_len, const int32_t* out_tokens) {
  if (dtype != SPECDEC_F32 && dtype != SPECDEC_BF16) return SPECDEC_ERR_INVALID_ARG;
  if (B < 0 || n_max < 0 || V <= 0) return SPECDEC_ERR_INVALID_ARG;
  if (V > SPECDEC_MAX_VOCAB || n_max > SPECDEC_MAX_DRAFT) return SPECDEC_ERR_UNSUPPORTED;
  if (B == 0) return SPECDEC_OK;
  if (target_logits == nullptr || draft_len == nullptr || temperature == nullptr ||
      accepted_len == nullptr || out_tokens == nullptr)
    return SPECDEC_ERR_INVALID_ARG;
  if (n_max > 0 && draft_tokens == nullptr) return SPECDEC_ERR_INVALID_ARG;
  if (B > SPECDEC_MAX_BATCH) return SPECDEC_ERR_UNSUPPORTED;
  return SPECDEC_OK;
}
}  // namespace

extern "C" specdec_status_t spec_verify(const void* target_logits, const void* draft_logits,
                                        specdec_dtype_t dtype, int32_t B, int32_t n_max, int32_t V,
                                        const int32_t* draft_tokens, const int32_t* draft_len,
                                        const float* temperature, uint64_t seed,
                                        int32_t* accepted_len, int32_t* out_tokens, float* row_lse,
                                        void* workspace, size_t workspace_bytes, void* stream) {
  const specdec_status_t chk = check_verify_args(target_logits, dtype, B, n_max, V, draft_tokens, draft_len,
                                                 temperature, accepted_len, out_tokens);
  if (chk != SPECDEC_OK || B == 0) return chk;
  VerifyCall c;
  memset(&c, 0, sizeof c);
  c.target = target_logits;
  c.draft = draft_logits;
  c.dtype = dtype;
  c.B = B;
  c.n_max = n_max;
  c.V = V;
  c.draft_tokens = draft_tokens;
  c.draft_len = draft_len;
  c.temperature = temperature;
  c.seed = seed;
  c.accepted_len = accepted_len;
  c.out_tokens = out_tokens;
  c.row_lse = row_lse;
  c.workspace = workspace;
  c.workspace_bytes = workspace_bytes;
  c.stream = stream;
  return verify_launch(c);
}

extern "C" specdec_status_t spec_verify_early_exit(const void* target_logits, const void* draft_logits,
                                                   specdec_dtype_t dtype, int32_t B, int32_t n_max, int32_t V,
                                                   const int32_t* draft_tokens, const int32_t* draft_len,
                                                   const float* temperature, uint64_t seed,
                                                   int32_t* accepted_len, int32_t* out_tokens,
                                                   void* workspace, size_t workspace_bytes, void* stream) {
  if (dtype != SPECDEC_F32 && dtype != SPECDEC_BF16) return SPECDEC_ERR_INVALID_ARG;
  if (B < 0 || n_max < 0 || V <= 0) return SPECDEC_ERR_INVALID_ARG;
  if (V > SPECDEC_MAX_VOCAB || n_max > SPECDEC_EARLY_EXIT_MAX_DRAFT) return SPECDEC_ERR_UNSUPPORTED;
  if (B == 0) return SPECDEC_OK;
  if (target_logits == nullptr || draft_len == nullptr || temperature == nullptr ||
      accepted_len == nullptr || out_tokens == nullptr)
    return SPECDEC_ERR_INVALID_ARG;
  if (n_max > 0 && draft_tokens == nullptr) return SPECDEC_ERR_INVALID_ARG;
  if (B > SPECDEC_MAX_BATCH) return SPECDEC_ERR_UNSUPPORTED;
  VerifyCall c;
  memset(&c, 0, sizeof c);
  c.target = target_logits;
  c.draft = draft_logits;
  c.dtype = dtype;
  c.B = B;
  c.n_max = n_max;
  c.V = V;
  c.draft_tokens = draft_tokens;
  c.draft_len = draft_len;
  c.early_exit = 1;
  c.temperature = temperature;
  c.seed = seed;
  c.accepted_len = accepted_len;
  c.out_tokens = out_tokens;
  c.workspace = workspace;
  c.workspace_bytes = workspace_bytes;
  c.stream = stream;
  return verify_launch(c);
}

extern "C" specdec_status_t spec_verify_packed(const void* target_logits, const void* draft_logits,
                                               specdec_dtype_t dtype, int32_t B, int32_t n_max, int32_t V,
                                               const int32_t* cu_rows, int32_t total_rows,
                                               const int32_t* draft_tokens, const float* temperature,
                                               const int32_t* pos_offset, uint64_t seed,
                                               int32_t* accepted_len, int32_t* out_tokens, float* row_lse,
                                               void* workspace, size_t workspace_bytes, void* stream) {
  if (dtype != SPECDEC_F32 && dtype != SPECDEC_BF16) return SPECDEC_ERR_INVALID_ARG;
  if (B < 0 || n_max < 0 || V <= 0 || total_rows < B) return SPECDEC_ERR_INVALID_ARG;
  if (V > SPECDEC_MAX_VOCAB || n_max > SPECDEC_MAX_DRAFT) return SPECDEC_ERR_UNSUPPORTED;
  if (B == 0) return SPECDEC_OK;
  if (target_logits == nullptr || cu_rows == nullptr || temperature == nullptr ||
      accepted_len == nullptr || out_tokens == nullptr)
    return SPECDEC_ERR_INVALID_ARG;
  if (total_rows > B && draft_tokens == nullptr) return SPECDEC_ERR_INVALID_ARG;
  if (B > SPECDEC_MAX_BATCH) return SPECDEC_ERR_UNSUPPORTED;
  VerifyCall c;
  memset(&c, 0, sizeof c);
  c.target = target_logits;
  c.draft = total_rows > B ? draft_logits : nullptr;
  c.dtype = dtype;
  c.B = B;
  c.n_max = n_max;
  c.V = V;
  c.draft_tokens = draft_tokens;
  c.cu_rows = cu_rows;
  c.total_rows = total_rows;
  c.pos_offset = pos_offset;
  c.temperature = temperature;
  c.seed = seed;
  c.accepted_len = accepted_len;
  c.out_tokens = out_tokens;
  c.row_lse = row_lse;
  c.workspace = workspace;
  c.workspace_bytes = workspace_bytes;
  c.stream = stream;
  return verify_launch(c);
}

extern "C" specdec_status_t mtp_shift_insert(const int32_t* tokens_in, int32_t* tokens_out,
                                             const void* hidden_in, void* hidden_out, int32_t R,
                                             int32_t H, int32_t hidden_elem_bytes,
                                             const int32_t* seg_start, const int32_t* draft_len,
                                             const int32_t* accepted_len, const int32_t* next_token,
                                             int32_t next_token_stride, int32_t B, uint32_t* error_word,
                                             void* stream) {
  if (R < 0 || B < 0 || next_token_stride < 0) return SPECDEC_ERR_INVALID_ARG;
  if (B == 0 || R == 0) return SPECDEC_OK;
  if (tokens_in == nullptr || tokens_out == nullptr || draft_len == nullptr ||
      accepted_len == nullptr || next_token == nullptr)
    return SPECDEC_ERR_INVALID_ARG;
  if (seg_start == nullptr && R % B != 0) return SPECDEC_ERR_INVALID_ARG;
  const bool copy = hidden_out != nullptr && hidden_in != nullptr && hidden_out != hidden_in;
  if (hidden_out != nullptr && hidden_in == nullptr) return SPECDEC_ERR_INVALID_ARG;
  if (copy && (H <= 0 || hidden_elem_bytes <= 0)) return SPECDEC_ERR_INVALID_ARG;

  MtpArgs a;
  memset(&a, 0, sizeof a);
  a.tokens_in = tokens_in;
  a.tokens_out = tokens_out;
  a.seg_start = seg_start;
  a.draft_len = draft_len;
  a.accepted_len = accepted_len;
  a.next_token = next_token;
  a.next_token_stride = next_token_stride;
  a.R = R;
  a.B = B;
  a.seg_blocks = (B + kMtpWarps - 1) / kMtpWarps;
  a.err = error_word;
  int copy_blocks = 0;
  if (copy) {
    const long long bytes = static_cast<long long>(R) * H * hidden_elem_bytes;
    const bool al = aligned16(hidden_in) && aligned16(hidden_out);
    a.hidden_in = static_cast<const uint4*>(hidden_in);
    a.hidden_out = static_cast<uint4*>(hidden_out);
    a.hidden_in_bytes = static_cast<const unsigned char*>(hidden_in);
    a.hidden_out_bytes = static_cast<unsigned char*>(hidden_out);
    a.n16 = al ? bytes / 16 : 0;
    a.tail_begin = a.n16 * 16;
    a.tail_end = bytes;
    // Enough blocks to keep every SM streaming; each thread moves several
    // 16-byte words.
    long long work = a.n16 + (a.tail_end - a.tail_begin);
    long long blocks = (work + kMtpThreads * 4 - 1) / (kMtpThreads * 4);
    copy_blocks = static_cast<int>(blocks > 152 * 8 ? 152 * 8 : (blocks < 1 ? 1 : blocks));
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  mtp_shift_insert_kernel<<<a.seg_blocks + copy_blocks, kMtpThreads, 0, st>>>(a);
  return cudaGetLastError() == cudaSuccess ? SPECDEC_OK : SPECDEC_ERR_CUDA;
}

extern "C" specdec_status_t specdec_get_error(void* workspace, uint32_t* error_bits) {
  if (workspace == nullptr || error_bits == nullptr) return SPECDEC_ERR_INVALID_ARG;
  uint32_t v = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return SPECDEC_ERR_CUDA;
  if (cudaMemcpy(&v, workspace, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess)
    return SPECDEC_ERR_CUDA;
  const uint32_t zero = 0;
  if (cudaMemcpy(workspace, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
    return SPECDEC_ERR_CUDA;
  *error_bits = v;
  if (v & SPECDEC_DEV_ERR_TIMEOUT) return SPECDEC_ERR_TIMEOUT;
  return v ? SPECDEC_ERR_DEVICE_DATA : SPECDEC_OK;
}

extern "C" specdec_status_t specdec_get_bytes_read(void* workspace, uint64_t* bytes) {
  if (workspace == nullptr || bytes == nullptr) return SPECDEC_ERR_INVALID_ARG;
  uint64_t v = 0;
  // the counter line does not depend on the batch shape
  unsigned char* ctr = static_cast<unsigned char*>(workspace) + ws_layout(1, 0, 1).ctr + 4 * kCtrReadBytes;
  if (cudaDeviceSynchronize() != cudaSuccess) return SPECDEC_ERR_CUDA;
  if (cudaMemcpy(&v, ctr, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return SPECDEC_ERR_CUDA;
  const uint64_t zero = 0;
  if (cudaMemcpy(ctr, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) return SPECDEC_ERR_CUDA;
  *bytes = v;
  return SPECDEC_OK;
}

extern "C" const char* specdec_status_string(specdec_status_t s) {
  switch (s) {
    case SPECDEC_OK: return "SPECDEC_OK";
    case SPECDEC_ERR_INVALID_ARG: return "SPECDEC_ERR_INVALID_ARG";
    case SPECDEC_ERR_UNSUPPORTED: return "SPECDEC_ERR_UNSUPPORTED";
    case SPECDEC_ERR_WORKSPACE: return "SPECDEC_ERR_WORKSPACE";
    case SPECDEC_ERR_CUDA: return "SPECDEC_ERR_CUDA";
    case SPECDEC_ERR_DEVICE_DATA: return "SPECDEC_ERR_DEVICE_DATA";
    case SPECDEC_ERR_TIMEOUT: return "SPECDEC_ERR_TIMEOUT";
  }
  return "SPECDEC_UNKNOWN_STATUS";
}

// ---------------------------------------------------------------------------
// spec_verify_no_alloc: spec_verify with a workspace the library owns.
//
// Some callers cannot allocate device memory at the point where they verify:
// code running inside a custom allocator or a memory-pool callback, runtimes
// that forbid cudaMalloc after start-up (it synchronises the device and can
// fragment a carefully planned pool), and C hosts that only hand over the
// tensors they already own.  For them the workspace lives in a fixed
// file-scope device array, loaded with the library on every GPU that loads it
// and held until the process exits.
namespace specdec {
namespace {

static __device__ __align__(256) unsigned char g_no_alloc_workspace[SPECDEC_NO_ALLOC_WORKSPACE_BYTES];

// Device address of the array, looked up once per device with that device
// current.  In host code the array's name is only a host-side stand-in.
void* no_alloc_workspace_address(specdec_status_t* status) {
  static void* addr[64] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    *status = SPECDEC_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_no_alloc_workspace) != cudaSuccess || p == nullptr) {
      *status = SPECDEC_ERR_CUDA;
      return nullptr;
    }
    addr[dev] = p;
  }
  *status = SPECDEC_OK;
  return addr[dev];
}

}  // namespace
}  // namespace specdec

extern "C" specdec_status_t spec_verify_no_alloc(const void* target_logits, const void* draft_logits,
                                                 specdec_dtype_t dtype, int32_t B, int32_t n_max, int32_t V,
                                                 const int32_t* draft_tokens, const int32_t* draft_len,
                                                 const float* temperature, uint64_t seed,
                                                 int32_t* accepted_len, int32_t* out_tokens,
                                                 float* row_lse, void* stream) {
  // Every host-side check runs before the workspace clear is enqueued.
  const specdec_status_t chk = check_verify_args(target_logits, dtype, B, n_max, V, draft_tokens, draft_len,
                                                 temperature, accepted_len, out_tokens);
  if (chk != SPECDEC_OK || B == 0) return chk;
  const size_t need = ws_layout(B, n_max, V).total;
  if (need > SPECDEC_NO_ALLOC_WORKSPACE_BYTES) return SPECDEC_ERR_WORKSPACE;  // batch too large
  specdec_status_t st = SPECDEC_OK;
  void* ws = no_alloc_workspace_address(&st);
  if (st != SPECDEC_OK) return st;
  // The array keeps whatever the previous call left: clear the part this
  // call uses (counters, queue and partials must start at zero).
  if (cudaMemsetAsync(ws, 0, need, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return SPECDEC_ERR_CUDA;
  return spec_verify(target_logits, draft_logits, dtype, B, n_max, V, draft_tokens, draft_len,
                     temperature, seed, accepted_len, out_tokens, row_lse, ws, need, stream);
}
