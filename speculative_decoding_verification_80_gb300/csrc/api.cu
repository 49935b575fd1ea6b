// api.cu — the C ABI of libspecdec.so: argument checks, workspace layout,
// launch shapes and kernel launches.  The declarations, with the meaning of
// every argument, are in include/specdec.h.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "mtp_kernel.cuh"
#include "specdec.h"
#include "verify_kernel.cuh"

namespace specdec {
namespace {

constexpr size_t kAlign = 256;
constexpr int kMaxCluster = 16;
constexpr int kMaxSmemPerCta = 227 * 1024;
// Target bytes of one staged slice per tensor: small enough that several
// CTAs share an SM (their copies and arithmetic overlap), large enough that
// the per-row reductions are amortised.
constexpr int kSliceTargetBytes = 32 * 1024;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct WsLayout {
  size_t err, arrivals, winner, accept, state, total;
};

WsLayout ws_layout(int B, int n_max) {
  WsLayout w;
  const size_t rows = static_cast<size_t>(B) * (n_max + 1);
  w.err = 0;
  w.arrivals = kAlign;
  w.winner = w.arrivals + align_up(4 * static_cast<size_t>(B), kAlign);
  w.accept = w.winner + align_up(8 * rows, kAlign);
  w.state = w.accept + align_up(4 * rows, kAlign);
  w.total = w.state + align_up(4 * rows, kAlign);
  return w;
}

struct Shape {
  int C, S, smem, stride;
};

// CTAs per row and slice length for V elements of `elt` bytes.
bool launch_shape(int V, int elt, Shape* out) {
  const int vec = 16 / elt;
  int C = static_cast<int>((static_cast<long long>(V) * elt + kSliceTargetBytes - 1) / kSliceTargetBytes);
  C = C < 1 ? 1 : (C > 8 ? 8 : C);
  for (;; ++C) {
    if (C > kMaxCluster) return false;
    int S = (V + C - 1) / C;
    S = (S + vec - 1) / vec * vec;
    const int stride = static_cast<int>(align_up(static_cast<size_t>(S) * elt, 128));
    const int smem = kScratchBytes + 2 * stride;
    if (smem <= kMaxSmemPerCta) {
      out->C = (V + S - 1) / S;  // no CTA without elements
      out->S = S;
      out->stride = stride;
      out->smem = smem;
      return true;
    }
  }
}

template <typename Elt>
cudaError_t prepare_kernel() {
  // Per device: allow the largest dynamic shared memory and clusters of 16.
  static bool done[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(verify_kernel<Elt>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kMaxSmemPerCta);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(verify_kernel<Elt>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64) done[dev] = true;
  return cudaSuccess;
}

template <typename Elt>
cudaError_t launch_verify(const VerifyArgs& args, const Shape& sh, long long units, cudaStream_t st) {
  cudaError_t e = prepare_kernel<Elt>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3(static_cast<unsigned>(units * sh.C), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(sh.smem);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(sh.C);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, verify_kernel<Elt>, args);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace specdec

using namespace specdec;

extern "C" size_t specdec_verify_workspace_bytes(int32_t B, int32_t n_max, int32_t V) {
  (void)V;
  if (B <= 0 || n_max < 0 || n_max > SPECDEC_MAX_DRAFT) return 0;
  return ws_layout(B, n_max).total;
}

extern "C" specdec_status_t specdec_workspace_init(void* workspace, size_t bytes, void* stream) {
  if (workspace == nullptr || bytes == 0) return SPECDEC_ERR_INVALID_ARG;
  return cudaMemsetAsync(workspace, 0, bytes, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? SPECDEC_OK
             : SPECDEC_ERR_CUDA;
}

extern "C" specdec_status_t specdec_verify_launch_shape(int32_t V, specdec_dtype_t dtype,
                                                        int32_t* ctas_per_row, int32_t* slice_elems) {
  if (V <= 0 || V > SPECDEC_MAX_VOCAB || (dtype != SPECDEC_F32 && dtype != SPECDEC_BF16))
    return SPECDEC_ERR_INVALID_ARG;
  Shape sh;
  if (!launch_shape(V, dtype == SPECDEC_F32 ? 4 : 2, &sh)) return SPECDEC_ERR_UNSUPPORTED;
  if (ctas_per_row) *ctas_per_row = sh.C;
  if (slice_elems) *slice_elems = sh.S;
  return SPECDEC_OK;
}

extern "C" specdec_status_t spec_verify(const void* target_logits, const void* draft_logits,
                                        specdec_dtype_t dtype, int32_t B, int32_t n_max, int32_t V,
                                        const int32_t* draft_tokens, const int32_t* draft_len,
                                        const float* temperature, uint64_t seed,
                                        int32_t* accepted_len, int32_t* out_tokens, float* row_lse,
                                        void* workspace, size_t workspace_bytes, void* stream) {
  if (dtype != SPECDEC_F32 && dtype != SPECDEC_BF16) return SPECDEC_ERR_INVALID_ARG;
  if (B < 0 || n_max < 0 || V <= 0) return SPECDEC_ERR_INVALID_ARG;
  if (V > SPECDEC_MAX_VOCAB || n_max > SPECDEC_MAX_DRAFT) return SPECDEC_ERR_UNSUPPORTED;
  if (B == 0) return SPECDEC_OK;
  if (target_logits == nullptr || draft_len == nullptr || temperature == nullptr ||
      accepted_len == nullptr || out_tokens == nullptr)
    return SPECDEC_ERR_INVALID_ARG;
  if (n_max > 0 && draft_tokens == nullptr) return SPECDEC_ERR_INVALID_ARG;
  if (workspace == nullptr || !aligned16(workspace)) return SPECDEC_ERR_WORKSPACE;
  const WsLayout wl = ws_layout(B, n_max);
  if (workspace_bytes < wl.total) return SPECDEC_ERR_WORKSPACE;
  const long long units = static_cast<long long>(B) * (n_max + 1);
  const int elt = dtype == SPECDEC_F32 ? 4 : 2;
  Shape sh;
  if (!launch_shape(V, elt, &sh)) return SPECDEC_ERR_UNSUPPORTED;
  if (units * sh.C > 0x7FFFFFFFLL) return SPECDEC_ERR_UNSUPPORTED;

  unsigned char* ws = static_cast<unsigned char*>(workspace);
  VerifyArgs a;
  memset(&a, 0, sizeof a);
  a.target = target_logits;
  a.draft = n_max > 0 ? draft_logits : nullptr;
  a.draft_tokens = draft_tokens;
  a.draft_len = draft_len;
  a.temperature = temperature;
  a.accepted_len = accepted_len;
  a.out_tokens = out_tokens;
  a.row_lse = row_lse;
  a.err = reinterpret_cast<uint32_t*>(ws + wl.err);
  a.arrivals = reinterpret_cast<uint32_t*>(ws + wl.arrivals);
  a.row_winner = reinterpret_cast<unsigned long long*>(ws + wl.winner);
  a.row_accept = reinterpret_cast<uint32_t*>(ws + wl.accept);
  a.row_state = reinterpret_cast<uint32_t*>(ws + wl.state);
  a.seed_lo = static_cast<uint32_t>(seed & 0xFFFFFFFFull);
  a.seed_hi = static_cast<uint32_t>(seed >> 32);
  a.B = B;
  a.n_max = n_max;
  a.V = V;
  a.C = sh.C;
  a.S = sh.S;
  a.slice_stride_bytes = sh.stride;
  // Bulk copies need 16-byte aligned rows and slices.
  a.bulk = (static_cast<long long>(V) * elt) % 16 == 0 && aligned16(target_logits) &&
           (a.draft == nullptr || aligned16(a.draft));

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = dtype == SPECDEC_F32 ? launch_verify<float>(a, sh, units, st)
                                       : launch_verify<uint16_t>(a, sh, units, st);
  return e == cudaSuccess ? SPECDEC_OK : SPECDEC_ERR_CUDA;
}

extern "C" specdec_status_t mtp_shift_insert(const int32_t* tokens_in, int32_t* tokens_out,
                                             const void* hidden_in, void* hidden_out, int32_t R,
                                             int32_t H, int32_t hidden_elem_bytes,
                                             const int32_t* seg_start, const int32_t* draft_len,
                                             const int32_t* accepted_len, const int32_t* next_token,
                                             int32_t next_token_stride, int32_t B, void* stream) {
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
  return v ? SPECDEC_ERR_DEVICE_DATA : SPECDEC_OK;
}

extern "C" const char* specdec_status_string(specdec_status_t s) {
  switch (s) {
    case SPECDEC_OK: return "SPECDEC_OK";
    case SPECDEC_ERR_INVALID_ARG: return "SPECDEC_ERR_INVALID_ARG";
    case SPECDEC_ERR_UNSUPPORTED: return "SPECDEC_ERR_UNSUPPORTED";
    case SPECDEC_ERR_WORKSPACE: return "SPECDEC_ERR_WORKSPACE";
    case SPECDEC_ERR_CUDA: return "SPECDEC_ERR_CUDA";
    case SPECDEC_ERR_DEVICE_DATA: return "SPECDEC_ERR_DEVICE_DATA";
  }
  return "SPECDEC_UNKNOWN_STATUS";
}
