// lion_noalloc.cu -- the recurrent form of the operator for callers that
// cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: code running inside a host framework
// that owns every byte of device memory through its own allocator, or a
// latency-critical loop where an allocation (and the implicit device-wide
// synchronisation cudaMalloc/cudaFree may bring) is not allowed.  The
// regular entry points either take a caller workspace or allocate one on
// the stream; this one takes neither.  Its scratch -- the per-token forward
// normaliser c^F_i that the backward sweep of the recurrent form reads back
// -- lives in a fixed array of this library, `g_noalloc_cF`, sized for
// LION_NOALLOC_MAX_HEAD_TOKENS = 2^20 head-tokens (B * H * L), i.e. 4 MiB.
// Every GPU that loads the library holds that array until the process exits.
//
// Host code may not use the array's name as a device address (on the host it
// is only a stand-in).  The device address is looked up once per device with
// cudaGetSymbolAddress, with that device current, by the first call made on
// that device; make that first call before any stream capture.  The address
// is kept for the life of the process: a cudaDeviceReset after the first
// call is not supported.
//
// All calls share the one array and it keeps the previous call's contents.
// The recurrent kernel writes every c^F_i before it reads it, so nothing
// needs clearing.  Calls whose executions overlap on the GPU (different
// streams, no ordering between them) race on the array: order them.
#include <atomic>

#include "../../include/lion.h"
#include "lion_common.cuh"
#include "lion_internal.h"

namespace {

constexpr size_t kMaxHeadTokens = LION_NOALLOC_MAX_HEAD_TOKENS;

static __device__ __align__(256) float g_noalloc_cF[kMaxHeadTokens];

// Device address of the array, per device, resolved once.  Concurrent first
// calls from several host threads may both resolve it; they store the same
// value, and the atomic makes that well defined.
constexpr int kMaxDevices = 64;
std::atomic<float*> g_noalloc_ptr[kMaxDevices];

// Device address of the scratch array on the current device (set-up on the
// first call per device).
float* noalloc_scratch() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  float* ptr = g_noalloc_ptr[dev].load(std::memory_order_acquire);
  if (!ptr) {
    if (cudaGetSymbolAddress((void**)&ptr, g_noalloc_cF) != cudaSuccess || !ptr) {
      cudaGetLastError();
      return nullptr;
    }
    g_noalloc_ptr[dev].store(ptr, std::memory_order_release);
  }
  return ptr;
}

}  // namespace

extern "C" lion_status lion_attn_fwd_rnn_noalloc(const void* q, const void* k, const void* v,
                                                 const float* log_lambda, int B, int H, int L, int d,
                                                 int mask_kind, int dtype, float* out,
                                                 cudaStream_t stream) {
  // the checks of every other forward entry point (no workspace: the form's
  // scratch is the fixed array)
  lion_args a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.log_lambda = log_lambda;
  a.out = out;
  a.B = B;
  a.H = H;
  a.L = L;
  a.d = d;
  a.mask_kind = mask_kind;
  a.form = LION_FORM_RNN;
  a.chunk = 1;
  a.dtype = dtype;
  a.phi = LION_PHI_DEFAULT;
  a.workspace = nullptr;
  a.workspace_bytes = 0;
  a.stream = stream;
  a.out_bf16 = 0;
  // the scratch holds one float per head-token
  if (B >= 1 && H >= 1 && L >= 1 &&
      (unsigned long long)B * (unsigned long long)H * (unsigned long long)L > kMaxHeadTokens)
    return LION_ERR_UNSUPPORTED;
  const lion_status st = lion::validate_args(&a);
  if (st != LION_OK) return st;
  float* scratch = noalloc_scratch();
  if (!scratch) return LION_ERR_CUDA;
  lion::Problem p;
  p.q = q;
  p.k = k;
  p.v = v;
  p.log_lambda = log_lambda;
  p.out = out;
  p.B = B;
  p.H = H;
  p.L = L;
  p.d = d;
  p.mask_kind = mask_kind;
  p.phi = lion::resolve_phi(mask_kind, LION_PHI_DEFAULT);
  p.dtype = dtype;
  p.chunk = 1;
  // c^F alone in the fixed array: every column CTA computes its features
  const size_t cf_bytes = sizeof(float) * (size_t)B * H * L;
  return lion::launch_rnn_simt(p, scratch, cf_bytes, stream) == cudaSuccess ? LION_OK : LION_ERR_CUDA;
}
