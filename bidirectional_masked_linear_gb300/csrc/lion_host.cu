// lion_host.cu -- lion_attn_fwd_host: the forward operator on inputs and
// output in host memory.  The batch is cut into slices; slice s is copied in
// on one stream, computed on the caller's stream and copied out on a third,
// with two device buffer sets, so that the copies of neighbouring slices
// overlap the compute and each other (the link carries the inputs in and the
// output out at the same time).  Every copy is one cudaMemcpyAsync of a
// contiguous slice.  Four slices is the default: at ViT-B (64 x 12 x 197,
// d = 64) on one GB300 a call took 0.470 / 0.455 / 0.445 / 0.455 / 0.483 ms
// with 2 / 3 / 4 / 5 / 8 slices (the first and last at half size), against
// 0.322 ms for the copies in and out alone when run at the same time.  Equal
// slices gave 0.473 ms at 4.  Finer slices lose because the kernel's time per
// slice hardly shrinks with the heads in it.
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "../../include/lion.h"
#include "host_plan.h"
#include "lion_common.cuh"
#include "lion_internal.h"

namespace {

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Host memory: page-locked (registered or allocated by CUDA) or pageable.
bool host_memory(const void* p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeHost || at.type == cudaMemoryTypeUnregistered;
}

lion_status validate_host(const lion_host_args* a) {
  if (!a || !a->q || !a->k || !a->v || !a->out) return LION_ERR_INVALID_ARG;
  if (a->B < 1 || a->H < 1 || a->L < 1) return LION_ERR_INVALID_ARG;
  if (a->d != 16 && a->d != 32 && a->d != 64 && a->d != 128) return LION_ERR_INVALID_ARG;
  if (a->mask_kind < LION_MASK_LIT || a->mask_kind > LION_MASK_S) return LION_ERR_INVALID_ARG;
  if (a->form < LION_FORM_FULL || a->form > LION_FORM_CHUNK) return LION_ERR_INVALID_ARG;
  if (a->dtype != LION_DTYPE_BF16 && a->dtype != LION_DTYPE_FP32) return LION_ERR_INVALID_ARG;
  if (a->phi < LION_PHI_DEFAULT || a->phi > LION_PHI_IDENTITY) return LION_ERR_INVALID_ARG;
  if (a->form == LION_FORM_CHUNK && a->chunk < 1) return LION_ERR_INVALID_ARG;
  if (a->slices < 0) return LION_ERR_INVALID_ARG;
  if (a->mask_kind != LION_MASK_LIT && !a->log_lambda) return LION_ERR_INVALID_ARG;
  if ((long long)a->B * a->H > 0x7fffffffLL || (long long)a->L * a->d > 0x7fffffffLL) return LION_ERR_INVALID_ARG;
  if (!host_memory(a->q) || !host_memory(a->k) || !host_memory(a->v) || !host_memory(a->out))
    return LION_ERR_INVALID_ARG;
  if (a->mask_kind != LION_MASK_LIT && !host_memory(a->log_lambda)) return LION_ERR_INVALID_ARG;
  if (a->form == LION_FORM_FULL && a->L > LION_FULL_MAX_L) return LION_ERR_UNSUPPORTED;
  return LION_OK;
}

// The two copy streams and the call's events, created once per device and
// reused by every call on it.  A call holds the device's lock while it
// enqueues its work, so calls from several host threads take turns; a reused
// event is recorded again only after the earlier call's waits on it were
// enqueued, which is all that stream ordering needs.
struct CopyEngine {
  std::mutex m;
  bool ready = false;
  cudaStream_t copy_in = nullptr, copy_out = nullptr;
  cudaEvent_t ev[9] = {};   // start, in[2], comp[2], freed[2], done_in, done_out
};
constexpr int kMaxDevices = 64;
CopyEngine g_engines[kMaxDevices];

// Creates the device's streams and events on first use (lock held).
cudaError_t engine_ready(CopyEngine& ce) {
  if (ce.ready) return cudaSuccess;
  cudaError_t e = cudaStreamCreateWithFlags(&ce.copy_in, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&ce.copy_out, cudaStreamNonBlocking);
  for (int i = 0; i < 9 && e == cudaSuccess; ++i) e = cudaEventCreateWithFlags(&ce.ev[i], cudaEventDisableTiming);
  if (e != cudaSuccess) {
    for (cudaEvent_t& ev : ce.ev)
      if (ev) cudaEventDestroy(ev), ev = nullptr;
    if (ce.copy_in) cudaStreamDestroy(ce.copy_in), ce.copy_in = nullptr;
    if (ce.copy_out) cudaStreamDestroy(ce.copy_out), ce.copy_out = nullptr;
    return e;
  }
  ce.ready = true;
  return cudaSuccess;
}

}  // namespace

extern "C" {

lion_status lion_attn_fwd_host(const lion_host_args* a) {
  lion_status st = validate_host(a);
  if (st != LION_OK) return st;
  const int B = a->B, H = a->H, L = a->L, d = a->d;
  // Slice sizes: the first slice's copy in and the last slice's copy out
  // overlap nothing, so with three or more slices those two get half the
  // batch rows of the others.
  const int S = a->slices > 0 ? (a->slices < B ? a->slices : B) : (B < 4 ? B : 4);
  int bounds[lion::kMaxSlices + 1];
  const int nslices = lion::slice_bounds(B, S < lion::kMaxSlices ? S : lion::kMaxSlices, bounds);
  int Bs = 0;
  for (int sl = 0; sl < nslices; ++sl) Bs = bounds[sl + 1] - bounds[sl] > Bs ? bounds[sl + 1] - bounds[sl] : Bs;
  const size_t esz = a->dtype == LION_DTYPE_BF16 ? 2 : 4;
  const size_t head_tokens = (size_t)H * L;                 // per batch row
  const size_t in_bytes = head_tokens * d * esz;            // q, k or v of one batch row
  const size_t out_bytes = head_tokens * d * sizeof(float);
  const bool sel = a->mask_kind == LION_MASK_S, fixed = a->mask_kind == LION_MASK_D;
  const size_t ll_bytes = sel ? head_tokens * sizeof(float) : 0;   // LION-S, per batch row
  const size_t ws_bytes = lion_attn_workspace_bytes(Bs, H, L, d, a->form, a->chunk);
  // two buffer sets: q, k, v, log-lambda and out for one slice; then the
  // LION-D decays (whole) and the kernels' workspace (one, compute is serial)
  const size_t set_bytes = 3 * align256(in_bytes * Bs) + align256(ll_bytes * Bs) + align256(out_bytes * Bs);
  const size_t total = 2 * set_bytes + align256(fixed ? sizeof(float) * H : 0) + align256(ws_bytes);
  cudaStream_t s = a->stream;
  uint8_t* base = nullptr;
  cudaError_t e = cudaMallocAsync(reinterpret_cast<void**>(&base), total, s);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return e == cudaErrorMemoryAllocation ? LION_ERR_NO_MEMORY : LION_ERR_CUDA;
  }
  struct Set {
    uint8_t *q, *k, *v;
    float *ll, *out;
  } set[2];
  for (int i = 0; i < 2; ++i) {
    uint8_t* w = base + i * set_bytes;
    set[i].q = w;
    w += align256(in_bytes * Bs);
    set[i].k = w;
    w += align256(in_bytes * Bs);
    set[i].v = w;
    w += align256(in_bytes * Bs);
    set[i].ll = reinterpret_cast<float*>(w);
    w += align256(ll_bytes * Bs);
    set[i].out = reinterpret_cast<float*>(w);
  }
  float* ll_fixed = reinterpret_cast<float*>(base + 2 * set_bytes);
  void* ws = base + 2 * set_bytes + align256(fixed ? sizeof(float) * H : 0);

  lion_status result = LION_OK;
  auto fail = [&](cudaError_t err) {
    if (result == LION_OK) result = err == cudaErrorMemoryAllocation ? LION_ERR_NO_MEMORY : LION_ERR_CUDA;
  };
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaFreeAsync(base, s);
    return LION_ERR_CUDA;
  }
  CopyEngine& ce = g_engines[dev];
  std::lock_guard<std::mutex> lock(ce.m);
  if ((e = engine_ready(ce)) != cudaSuccess) {
    cudaFreeAsync(base, s);
    return e == cudaErrorMemoryAllocation ? LION_ERR_NO_MEMORY : LION_ERR_CUDA;
  }
  cudaStream_t copy_in = ce.copy_in, copy_out = ce.copy_out;
  cudaEvent_t start = ce.ev[0], in[2] = {ce.ev[1], ce.ev[2]}, comp[2] = {ce.ev[3], ce.ev[4]},
              freed[2] = {ce.ev[5], ce.ev[6]};
  {
    // the copies start after the caller's earlier work on its stream
    if ((e = cudaEventRecord(start, s)) != cudaSuccess || (e = cudaStreamWaitEvent(copy_in, start, 0)) != cudaSuccess)
      fail(e);
    if (result == LION_OK && fixed)
      if ((e = cudaMemcpyAsync(ll_fixed, a->log_lambda, sizeof(float) * H, cudaMemcpyHostToDevice, copy_in)) !=
          cudaSuccess)
        fail(e);
  }
  for (int sl = 0; sl < nslices && result == LION_OK; ++sl) {
    const int b0 = bounds[sl], nb = bounds[sl + 1] - bounds[sl], i = sl & 1;
    // copy in, once the slice two back has left this buffer set
    if (sl >= 2 && (e = cudaStreamWaitEvent(copy_in, freed[i], 0)) != cudaSuccess) {
      fail(e);
      break;
    }
    const uint8_t* hq = static_cast<const uint8_t*>(a->q) + (size_t)b0 * in_bytes;
    const uint8_t* hk = static_cast<const uint8_t*>(a->k) + (size_t)b0 * in_bytes;
    const uint8_t* hv = static_cast<const uint8_t*>(a->v) + (size_t)b0 * in_bytes;
    if ((e = cudaMemcpyAsync(set[i].q, hq, in_bytes * nb, cudaMemcpyHostToDevice, copy_in)) != cudaSuccess ||
        (e = cudaMemcpyAsync(set[i].k, hk, in_bytes * nb, cudaMemcpyHostToDevice, copy_in)) != cudaSuccess ||
        (e = cudaMemcpyAsync(set[i].v, hv, in_bytes * nb, cudaMemcpyHostToDevice, copy_in)) != cudaSuccess) {
      fail(e);
      break;
    }
    if (sel && (e = cudaMemcpyAsync(set[i].ll, a->log_lambda + (size_t)b0 * head_tokens, ll_bytes * nb,
                                    cudaMemcpyHostToDevice, copy_in)) != cudaSuccess) {
      fail(e);
      break;
    }
    if ((e = cudaEventRecord(in[i], copy_in)) != cudaSuccess || (e = cudaStreamWaitEvent(s, in[i], 0)) != cudaSuccess) {
      fail(e);
      break;
    }
    // compute on the caller's stream
    lion_args g;
    memset(&g, 0, sizeof(g));
    g.q = set[i].q;
    g.k = set[i].k;
    g.v = set[i].v;
    g.log_lambda = sel ? set[i].ll : fixed ? ll_fixed : nullptr;
    g.out = set[i].out;
    g.B = nb;
    g.H = H;
    g.L = L;
    g.d = d;
    g.mask_kind = a->mask_kind;
    g.form = a->form;
    g.chunk = a->chunk;
    g.dtype = a->dtype;
    g.phi = a->phi;
    g.workspace = ws_bytes ? ws : nullptr;
    g.workspace_bytes = ws_bytes;
    g.stream = s;
    const lion_status fs = lion::forward_checked(&g);
    if (fs != LION_OK) {
      result = fs;
      break;
    }
    // copy out
    if ((e = cudaEventRecord(comp[i], s)) != cudaSuccess || (e = cudaStreamWaitEvent(copy_out, comp[i], 0)) != cudaSuccess ||
        (e = cudaMemcpyAsync(a->out + (size_t)b0 * head_tokens * d, set[i].out, out_bytes * nb,
                             cudaMemcpyDeviceToHost, copy_out)) != cudaSuccess ||
        (e = cudaEventRecord(freed[i], copy_out)) != cudaSuccess) {
      fail(e);
      break;
    }
  }
  // the caller's stream resumes after the last copies; the buffers are freed
  // in its order after them
  {
    cudaEvent_t done_in = ce.ev[7], done_out = ce.ev[8];
    if (cudaEventRecord(done_in, copy_in) != cudaSuccess || cudaEventRecord(done_out, copy_out) != cudaSuccess ||
        cudaStreamWaitEvent(s, done_in, 0) != cudaSuccess || cudaStreamWaitEvent(s, done_out, 0) != cudaSuccess) {
      cudaGetLastError();
      cudaStreamSynchronize(copy_in);
      cudaStreamSynchronize(copy_out);
      fail(cudaErrorUnknown);
    }
  }
  cudaFreeAsync(base, s);
  if (result == LION_OK && cudaGetLastError() != cudaSuccess) result = LION_ERR_CUDA;
  return result;
}

}  // extern "C"
