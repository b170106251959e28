// lion_api.cu -- the C ABI declared in include/lion.h: argument checks,
// workspace handling and the choice of kernel for each form.
#include <stdint.h>
#include <string.h>

#include "../../include/lion.h"
#include "lion_common.cuh"
#include "lion_internal.h"


namespace {

using lion::Problem;

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// A pointer the GPU can dereference: device or managed memory, or host memory
// registered/allocated with a device mapping.  Host-only memory would make a
// kernel fault, so it is refused here instead.
bool device_accessible(const void* p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();  // clear the sticky-free error of the query
    return false;
  }
  if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) return true;
  return at.type == cudaMemoryTypeHost && at.devicePointer != nullptr;
}

bool valid_d(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }


// Workspace bytes for (form, path).
size_t simt_workspace_bytes(int B, int H, int L, int d, int form, int chunk) {
  if (form == LION_FORM_FULL && (d == 64 || d == 128)) return lion::full_tiled_workspace_bytes(B, H, L, d);
  if (form == LION_FORM_RNN) return lion::rnn_workspace_bytes(B, H, L, d);
  if (form == LION_FORM_CHUNK && chunk >= 1 && chunk <= lion::kChunkTileMax)
    return lion::chunk_tile_workspace_bytes(B, H, L, d);
  if (form == LION_FORM_CHUNK) return sizeof(float) * (size_t)B * H * L;
  return 0;
}

lion_status validate(const lion_args* a) {
  if (!a) return LION_ERR_INVALID_ARG;
  if (!a->q || !a->k || !a->v || !a->out) return LION_ERR_INVALID_ARG;
  if (a->B < 1 || a->H < 1 || a->L < 1 || !valid_d(a->d)) return LION_ERR_INVALID_ARG;
  if (a->mask_kind < LION_MASK_LIT || a->mask_kind > LION_MASK_S) return LION_ERR_INVALID_ARG;
  if (a->form < LION_FORM_FULL || a->form > LION_FORM_CHUNK) return LION_ERR_INVALID_ARG;
  if (a->dtype != LION_DTYPE_BF16 && a->dtype != LION_DTYPE_FP32) return LION_ERR_INVALID_ARG;
  if (a->phi < LION_PHI_DEFAULT || a->phi > LION_PHI_IDENTITY) return LION_ERR_INVALID_ARG;
  if (a->form == LION_FORM_CHUNK && a->chunk < 1) return LION_ERR_INVALID_ARG;
  if (a->out_bf16 != 0 && a->out_bf16 != 1) return LION_ERR_INVALID_ARG;
  if (a->mask_kind != LION_MASK_LIT && !a->log_lambda) return LION_ERR_INVALID_ARG;
  // 32-bit launch and index limits: B*H heads on one grid axis, L*d per head.
  if ((long long)a->B * a->H > 0x7fffffffLL || (long long)a->L * a->d > 0x7fffffffLL)
    return LION_ERR_INVALID_ARG;
  if (!aligned(a->q, 16) || !aligned(a->k, 16) || !aligned(a->v, 16) || !aligned(a->out, 16))
    return LION_ERR_INVALID_ARG;
  if (a->log_lambda && !aligned(a->log_lambda, 4)) return LION_ERR_INVALID_ARG;
  if (a->workspace && !aligned(a->workspace, 256)) return LION_ERR_INVALID_ARG;
  if (!device_accessible(a->q) || !device_accessible(a->k) || !device_accessible(a->v) ||
      !device_accessible(a->out))
    return LION_ERR_INVALID_ARG;
  if (a->mask_kind != LION_MASK_LIT && !device_accessible(a->log_lambda)) return LION_ERR_INVALID_ARG;
  if (a->workspace && !device_accessible(a->workspace)) return LION_ERR_INVALID_ARG;
  if (a->form == LION_FORM_FULL && a->L > LION_FULL_MAX_L) return LION_ERR_UNSUPPORTED;
  return LION_OK;
}

}  // namespace

// Shared by every entry point that takes a lion_args (also the
// allocation-free recurrent form in lion_noalloc.cu).
lion_status lion::validate_args(const lion_args* a) { return validate(a); }

namespace {

lion_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return LION_OK;
  if (e == cudaErrorMemoryAllocation) return LION_ERR_NO_MEMORY;
  return LION_ERR_CUDA;
}

}  // namespace

extern "C" {

int lion_abi_version(void) { return 2; }

const char* lion_status_string(lion_status s) {
  switch (s) {
    case LION_OK: return "ok";
    case LION_ERR_INVALID_ARG: return "invalid argument";
    case LION_ERR_UNSUPPORTED: return "unsupported problem";
    case LION_ERR_CUDA: return "CUDA error";
    case LION_ERR_NO_MEMORY: return "out of device memory";
    case LION_ERR_TIMEOUT: return "device-side wait timed out";
    case LION_ERR_RANGE: return "a value exceeded the fp16 range of the tensor-core path";
  }
  return "unknown status";
}

size_t lion_attn_workspace_bytes(int B, int H, int L, int d, int form, int chunk) {
  if (B < 1 || H < 1 || L < 1 || !valid_d(d)) return 0;
  size_t need = simt_workspace_bytes(B, H, L, d, form, chunk);
  if (form == LION_FORM_CHUNK && d == 64 && chunk == 64) {
    const size_t tc = lion::chunk_tc_workspace_bytes(B, H, L);
    if (tc > need) need = tc;
  }
  if (form == LION_FORM_CHUNK && d == 64 && chunk == 128 && L > 256) {
    const size_t tc = lion::chunk128_long_workspace_bytes(B, H, L);
    if (tc > need) need = tc;
  }
  return need;
}

size_t lion_attn_bwd_workspace_bytes(int B, int H, int L, int d) {
  if (B < 1 || H < 1 || L < 1 || !valid_d(d)) return 0;
  return lion::bwd_workspace_bytes(B, H, L, d);
}

}  // extern "C"

namespace {

// Argument checks shared by the two gradient entry points (everything but
// the length limit and the workspace size).
lion_status validate_bwd(const lion_bwd_args* a) {
  if (!a) return LION_ERR_INVALID_ARG;
  if (!a->q || !a->k || !a->v || !a->dy || !a->dq || !a->dk || !a->dv) return LION_ERR_INVALID_ARG;
  if (a->B < 1 || a->H < 1 || a->L < 1 || !valid_d(a->d)) return LION_ERR_INVALID_ARG;
  if (a->mask_kind < LION_MASK_LIT || a->mask_kind > LION_MASK_S) return LION_ERR_INVALID_ARG;
  if (a->dtype != LION_DTYPE_BF16 && a->dtype != LION_DTYPE_FP32) return LION_ERR_INVALID_ARG;
  if (a->phi < LION_PHI_DEFAULT || a->phi > LION_PHI_IDENTITY) return LION_ERR_INVALID_ARG;
  if (a->mask_kind != LION_MASK_LIT && (!a->log_lambda || !a->dlog_lambda)) return LION_ERR_INVALID_ARG;
  if ((long long)a->B * a->H > 0x7fffffffLL || (long long)a->L * a->d > 0x7fffffffLL) return LION_ERR_INVALID_ARG;
  const void* ptrs[] = {a->q, a->k, a->v, a->dy, a->dq, a->dk, a->dv};
  for (const void* q : ptrs)
    if (!aligned(q, 16) || !device_accessible(q)) return LION_ERR_INVALID_ARG;
  if (a->mask_kind != LION_MASK_LIT &&
      (!aligned(a->log_lambda, 4) || !aligned(a->dlog_lambda, 4) || !device_accessible(a->log_lambda) ||
       !device_accessible(a->dlog_lambda)))
    return LION_ERR_INVALID_ARG;
  if (a->workspace && (!aligned(a->workspace, 256) || !device_accessible(a->workspace))) return LION_ERR_INVALID_ARG;
  return LION_OK;
}

// The gradients through the form `chunkwise` selects, on checked arguments.
lion_status run_bwd(const lion_bwd_args* a, bool chunkwise) {
  const size_t need = chunkwise ? lion::bwd_chunk_workspace_bytes(a->B, a->H, a->L, a->d)
                                : lion::bwd_workspace_bytes(a->B, a->H, a->L, a->d);
  if (a->workspace && a->workspace_bytes < need) return LION_ERR_INVALID_ARG;
  Problem p;
  p.q = a->q;
  p.k = a->k;
  p.v = a->v;
  p.log_lambda = a->log_lambda;
  p.out = nullptr;
  p.B = a->B;
  p.H = a->H;
  p.L = a->L;
  p.d = a->d;
  p.mask_kind = a->mask_kind;
  p.phi = lion::resolve_phi(a->mask_kind, a->phi);
  p.dtype = a->dtype;
  p.chunk = 0;
  cudaStream_t s = a->stream;
  void* ws = a->workspace;
  bool owned = false;
  if (!ws) {
    cudaError_t e = cudaMallocAsync(&ws, need, s);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return e == cudaErrorMemoryAllocation ? LION_ERR_NO_MEMORY : LION_ERR_CUDA;
    }
    owned = true;
  }
  cudaError_t e = chunkwise ? lion::launch_bwd_chunk(p, a->dy, a->dq, a->dk, a->dv, a->dlog_lambda, ws, s)
                            : lion::launch_bwd(p, a->dy, a->dq, a->dk, a->dv, a->dlog_lambda, ws, s);
  if (owned) {
    cudaError_t f = cudaFreeAsync(ws, s);
    if (e == cudaSuccess) e = f;
  }
  return from_cuda(e);
}

}  // namespace

extern "C" {

lion_status lion_attn_bwd(const lion_bwd_args* a) {
  const lion_status st = validate_bwd(a);
  if (st != LION_OK) return st;
  if (a->L > LION_FULL_MAX_L) return LION_ERR_UNSUPPORTED;
  return run_bwd(a, false);
}

lion_status lion_attn_bwd_chunk(const lion_bwd_args* a) {
  const lion_status st = validate_bwd(a);
  if (st != LION_OK) return st;
  // one CTA per (head, chunk) on one grid axis
  const long long chunks = ((long long)a->L + lion::bwd_chunk_length(a->d) - 1) / lion::bwd_chunk_length(a->d);
  if ((long long)a->B * a->H * chunks > 0x7fffffffLL || (long long)a->B * a->H * 1024 > 0x7fffffffLL)
    return LION_ERR_UNSUPPORTED;
  return run_bwd(a, true);
}

size_t lion_attn_bwd_chunk_workspace_bytes(int B, int H, int L, int d) {
  if (B < 1 || H < 1 || L < 1 || !valid_d(d)) return 0;
  return lion::bwd_chunk_workspace_bytes(B, H, L, d);
}

lion_status lion_attn_fwd_ex(const lion_args* a) {
  lion_status st = validate(a);
  if (st != LION_OK) return st;
  return lion::forward_checked(a);
}

}  // extern "C"

// The forward on arguments that already passed validate(): the kernel choice,
// the workspace and the launches (also the per-slice step of the host-buffer
// entry point, whose buffers the library allocated itself).
lion_status lion::forward_checked(const lion_args* a) {
  Problem p;
  p.q = a->q;
  p.k = a->k;
  p.v = a->v;
  p.log_lambda = a->log_lambda;
  p.out = a->out;
  p.B = a->B;
  p.H = a->H;
  p.L = a->L;
  p.d = a->d;
  p.mask_kind = a->mask_kind;
  p.phi = lion::resolve_phi(a->mask_kind, a->phi);
  p.dtype = a->dtype;
  p.chunk = a->chunk;
  cudaStream_t s = a->stream;

  const bool use_tc128 = a->form == LION_FORM_CHUNK && lion::chunk128_tc_supported(p);
  const bool use_tc128l = a->form == LION_FORM_CHUNK && lion::chunk128_long_supported(p);
  const bool use_tc = !use_tc128 && !use_tc128l && a->form == LION_FORM_CHUNK && lion::chunk_tc_supported(p);
  if (a->form == LION_FORM_CHUNK && !use_tc && !use_tc128 && !use_tc128l && a->chunk > lion::kSimtMaxChunk)
    return LION_ERR_UNSUPPORTED;
  int* dstatus = nullptr;
  if (use_tc || use_tc128 || use_tc128l) {
    dstatus = lion::device_status_ptr();
    if (!dstatus) return LION_ERR_CUDA;
  }
  const size_t need = use_tc128   ? 0
                      : use_tc128l ? lion::chunk128_long_workspace_bytes(a->B, a->H, a->L)
                      : use_tc     ? lion::chunk_tc_workspace_bytes(a->B, a->H, a->L)
                                   : simt_workspace_bytes(a->B, a->H, a->L, a->d, a->form, a->chunk);
  void* ws = a->workspace;
  bool owned = false;
  if (need > 0 && ws && a->workspace_bytes < need) return LION_ERR_INVALID_ARG;
  if (need > 0 && !ws) {
    cudaError_t e = cudaMallocAsync(&ws, need, s);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return e == cudaErrorMemoryAllocation ? LION_ERR_NO_MEMORY : LION_ERR_CUDA;
    }
    owned = true;
  }
  // bfloat16 output: stored by the chunk-128 kernels themselves; the other
  // paths write fp32 into a stream-ordered temporary that is then rounded
  const size_t n_out = (size_t)a->B * a->H * a->L * a->d;
  float* tmp = nullptr;
  if (a->out_bf16 && (use_tc128 || use_tc128l)) {
    p.out_bf16 = 1;
  } else if (a->out_bf16) {
    cudaError_t e = cudaMallocAsync(reinterpret_cast<void**>(&tmp), sizeof(float) * n_out, s);
    if (e != cudaSuccess) {
      cudaGetLastError();
      if (owned) cudaFreeAsync(ws, s);
      return e == cudaErrorMemoryAllocation ? LION_ERR_NO_MEMORY : LION_ERR_CUDA;
    }
    p.out = tmp;
  }
  cudaError_t e = cudaSuccess;
  switch (a->form) {
    case LION_FORM_FULL:
      e = lion::full_tiled_supported(p) ? lion::launch_full_tiled(p, ws, s) : lion::launch_full_simt(p, s);
      break;
    case LION_FORM_RNN: e = lion::launch_rnn_simt(p, (float*)ws, need, s); break;
    case LION_FORM_CHUNK:
      e = use_tc128    ? lion::launch_chunk128_tc(p, dstatus, s)
          : use_tc128l ? lion::launch_chunk128_long(p, ws, dstatus, s)
          : use_tc     ? lion::launch_chunk_tc(p, ws, dstatus, s)
          : lion::chunk_tile_supported(p) ? lion::launch_chunk_tile(p, (float*)ws, s)
                                          : lion::launch_chunk_simt(p, (float*)ws, s);
      break;
  }
  if (tmp) {
    if (e == cudaSuccess) e = lion::launch_f32_to_bf16(tmp, a->out, n_out, s);
    cudaError_t f = cudaFreeAsync(tmp, s);
    if (e == cudaSuccess) e = f;
  }
  if (owned) {
    cudaError_t f = cudaFreeAsync(ws, s);
    if (e == cudaSuccess) e = f;
  }
  return from_cuda(e);
}

extern "C" {

lion_status lion_sync_status(cudaStream_t stream) {
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return LION_ERR_CUDA;
  int* flag = lion::device_status_ptr();
  if (!flag) return LION_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, flag, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return LION_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpy(flag, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return LION_ERR_CUDA;
    return v == lion::kStatusBadOrder ? LION_ERR_INVALID_ARG
           : v == lion::kStatusRange  ? LION_ERR_RANGE
                                      : LION_ERR_TIMEOUT;
  }
  return LION_OK;
}

lion_status lion_attn_fwd_causal(const lion_args* a) {
  lion_status st = validate(a);
  if (st != LION_OK) return st;
  if (a->form == LION_FORM_CHUNK && a->chunk > lion::kSimtMaxChunk) return LION_ERR_UNSUPPORTED;
  Problem p;
  p.q = a->q;
  p.k = a->k;
  p.v = a->v;
  p.log_lambda = a->log_lambda;
  p.out = a->out;
  p.B = a->B;
  p.H = a->H;
  p.L = a->L;
  p.d = a->d;
  p.mask_kind = a->mask_kind;
  p.phi = lion::resolve_phi(a->mask_kind, a->phi);
  p.dtype = a->dtype;
  p.chunk = a->chunk;
  p.causal = 1;
  cudaStream_t s = a->stream;
  const size_t need = simt_workspace_bytes(a->B, a->H, a->L, a->d, a->form, a->chunk);
  void* ws = a->workspace;
  bool owned = false;
  if (need > 0 && ws && a->workspace_bytes < need) return LION_ERR_INVALID_ARG;
  if (need > 0 && !ws) {
    cudaError_t e = cudaMallocAsync(&ws, need, s);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return e == cudaErrorMemoryAllocation ? LION_ERR_NO_MEMORY : LION_ERR_CUDA;
    }
    owned = true;
  }
  const size_t n_out = (size_t)a->B * a->H * a->L * a->d;
  float* tmp = nullptr;
  if (a->out_bf16) {   // fp32 into a temporary, then rounded to bfloat16
    cudaError_t e = cudaMallocAsync(reinterpret_cast<void**>(&tmp), sizeof(float) * n_out, s);
    if (e != cudaSuccess) {
      cudaGetLastError();
      if (owned) cudaFreeAsync(ws, s);
      return e == cudaErrorMemoryAllocation ? LION_ERR_NO_MEMORY : LION_ERR_CUDA;
    }
    p.out = tmp;
  }
  cudaError_t e = cudaSuccess;
  switch (a->form) {
    case LION_FORM_FULL:
      e = lion::full_tiled_supported(p) ? lion::launch_full_tiled(p, ws, s) : lion::launch_full_simt(p, s);
      break;
    case LION_FORM_RNN: e = lion::launch_rnn_simt(p, (float*)ws, need, s); break;
    case LION_FORM_CHUNK:
      e = lion::chunk_tile_supported(p) ? lion::launch_chunk_tile(p, (float*)ws, s)
                                        : lion::launch_chunk_simt(p, (float*)ws, s);
      break;
  }
  if (tmp) {
    if (e == cudaSuccess) e = lion::launch_f32_to_bf16(tmp, a->out, n_out, s);
    cudaError_t f = cudaFreeAsync(tmp, s);
    if (e == cudaSuccess) e = f;
  }
  if (owned) {
    cudaError_t f = cudaFreeAsync(ws, s);
    if (e == cudaSuccess) e = f;
  }
  return from_cuda(e);
}

size_t lion_attn_reordered_bwd_workspace_bytes(int B, int H, int L, int d) {
  if (B < 1 || H < 1 || L < 1 || (d != 64 && d != 128)) return 0;
  return lion::reorder_bwd_workspace_bytes(B, H, L, d);
}

lion_status lion_attn_bwd_reordered(const lion_reorder_bwd_args* a) {
  if (!a) return LION_ERR_INVALID_ARG;
  if (!a->q || !a->k || !a->v || !a->dy || !a->dq || !a->dk || !a->dv || !a->order) return LION_ERR_INVALID_ARG;
  if (a->B < 1 || a->H < 1 || a->L < 1 || !valid_d(a->d)) return LION_ERR_INVALID_ARG;
  if (a->mask_kind < LION_MASK_LIT || a->mask_kind > LION_MASK_S) return LION_ERR_INVALID_ARG;
  if (a->dtype != LION_DTYPE_BF16 && a->dtype != LION_DTYPE_FP32) return LION_ERR_INVALID_ARG;
  if (a->phi < LION_PHI_DEFAULT || a->phi > LION_PHI_IDENTITY) return LION_ERR_INVALID_ARG;
  if (a->mask_kind != LION_MASK_LIT && (!a->log_lambda || !a->dlog_lambda)) return LION_ERR_INVALID_ARG;
  if ((long long)a->B * a->H > 0x7fffffffLL || (long long)a->L * a->d > 0x7fffffffLL) return LION_ERR_INVALID_ARG;
  const void* ptrs[] = {a->q, a->k, a->v, a->dy, a->dq, a->dk, a->dv};
  for (const void* q : ptrs)
    if (!aligned(q, 16) || !device_accessible(q)) return LION_ERR_INVALID_ARG;
  if (!aligned(a->order, 4) || !device_accessible(a->order)) return LION_ERR_INVALID_ARG;
  if (a->mask_kind != LION_MASK_LIT &&
      (!aligned(a->log_lambda, 4) || !aligned(a->dlog_lambda, 4) || !device_accessible(a->log_lambda) ||
       !device_accessible(a->dlog_lambda)))
    return LION_ERR_INVALID_ARG;
  if (a->workspace && (!aligned(a->workspace, 256) || !device_accessible(a->workspace))) return LION_ERR_INVALID_ARG;
  if (a->L > LION_FULL_MAX_L || (a->d != 64 && a->d != 128)) return LION_ERR_UNSUPPORTED;
  const size_t need = lion::reorder_bwd_workspace_bytes(a->B, a->H, a->L, a->d);
  if (a->workspace && a->workspace_bytes < need) return LION_ERR_INVALID_ARG;
  int* dstatus = lion::device_status_ptr();
  if (!dstatus) return LION_ERR_CUDA;
  Problem p;
  p.q = a->q;
  p.k = a->k;
  p.v = a->v;
  p.log_lambda = a->log_lambda;
  p.out = nullptr;
  p.B = a->B;
  p.H = a->H;
  p.L = a->L;
  p.d = a->d;
  p.mask_kind = a->mask_kind;
  p.phi = lion::resolve_phi(a->mask_kind, a->phi);
  p.dtype = a->dtype;
  p.chunk = 0;
  cudaStream_t s = a->stream;
  void* ws = a->workspace;
  bool owned = false;
  if (!ws) {
    cudaError_t e = cudaMallocAsync(&ws, need, s);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return e == cudaErrorMemoryAllocation ? LION_ERR_NO_MEMORY : LION_ERR_CUDA;
    }
    owned = true;
  }
  cudaError_t e = lion::launch_reordered_bwd(p, a->order, a->dy, a->dq, a->dk, a->dv, a->dlog_lambda, ws, dstatus, s);
  if (owned) {
    cudaError_t f = cudaFreeAsync(ws, s);
    if (e == cudaSuccess) e = f;
  }
  return from_cuda(e);
}

size_t lion_attn_reordered_workspace_bytes(int B, int H, int L, int d) {
  if (B < 1 || H < 1 || L < 1 || (d != 64 && d != 128)) return 0;
  return lion::reorder_workspace_bytes(B, H, L, d);
}

lion_status lion_attn_fwd_reordered(const lion_reorder_args* a) {
  if (!a) return LION_ERR_INVALID_ARG;
  lion_args g;
  memset(&g, 0, sizeof(g));
  g.q = a->q;
  g.k = a->k;
  g.v = a->v;
  g.log_lambda = a->log_lambda;
  g.out = a->out;
  g.B = a->B;
  g.H = a->H;
  g.L = a->L;
  g.d = a->d;
  g.mask_kind = a->mask_kind;
  g.form = LION_FORM_FULL;
  g.dtype = a->dtype;
  g.phi = a->phi;
  g.workspace = a->workspace;
  g.workspace_bytes = a->workspace_bytes;
  g.stream = a->stream;
  lion_status st = validate(&g);
  if (st != LION_OK) return st;
  if (!a->order || !aligned(a->order, 4) || !device_accessible(a->order)) return LION_ERR_INVALID_ARG;
  if (a->d != 64 && a->d != 128) return LION_ERR_UNSUPPORTED;
  const size_t need = lion::reorder_workspace_bytes(a->B, a->H, a->L, a->d);
  if (a->workspace && a->workspace_bytes < need) return LION_ERR_INVALID_ARG;
  int* dstatus = lion::device_status_ptr();
  if (!dstatus) return LION_ERR_CUDA;
  Problem p;
  p.q = a->q;
  p.k = a->k;
  p.v = a->v;
  p.log_lambda = a->log_lambda;
  p.out = a->out;
  p.B = a->B;
  p.H = a->H;
  p.L = a->L;
  p.d = a->d;
  p.mask_kind = a->mask_kind;
  p.phi = lion::resolve_phi(a->mask_kind, a->phi);
  p.dtype = a->dtype;
  p.chunk = 0;
  cudaStream_t s = a->stream;
  void* ws = a->workspace;
  bool owned = false;
  if (!ws) {
    cudaError_t e = cudaMallocAsync(&ws, need, s);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return e == cudaErrorMemoryAllocation ? LION_ERR_NO_MEMORY : LION_ERR_CUDA;
    }
    owned = true;
  }
  cudaError_t e = lion::launch_reordered(p, a->order, ws, dstatus, s);
  if (owned) {
    cudaError_t f = cudaFreeAsync(ws, s);
    if (e == cudaSuccess) e = f;
  }
  return from_cuda(e);
}

lion_status lion_attn_fwd(const void* q, const void* k, const void* v, const float* log_lambda,
                          int B, int H, int L, int d, int mask_kind, int form, int chunk,
                          float* out, cudaStream_t stream) {
  lion_args a;
  memset(&a, 0, sizeof(a));
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
  a.form = form;
  a.chunk = chunk;
  a.dtype = LION_DTYPE_BF16;
  a.phi = LION_PHI_DEFAULT;
  a.stream = stream;
  return lion_attn_fwd_ex(&a);
}

lion_status lion_rnn_step(const void* q, const void* k, const void* v, const float* log_lambda,
                          float* S, float* z, float* y_part, float* c_part, int B, int H, int d,
                          int mask_kind, int dtype, cudaStream_t stream) {
  if (!q || !k || !v || !S || !z || !y_part || !c_part) return LION_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || !valid_d(d)) return LION_ERR_INVALID_ARG;
  if (mask_kind < LION_MASK_LIT || mask_kind > LION_MASK_S) return LION_ERR_INVALID_ARG;
  if (dtype != LION_DTYPE_BF16 && dtype != LION_DTYPE_FP32) return LION_ERR_INVALID_ARG;
  if (mask_kind != LION_MASK_LIT && !log_lambda) return LION_ERR_INVALID_ARG;
  if ((long long)B * H > 0x7fffffffLL) return LION_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, S, z, y_part, c_part};
  for (const void* ptr : ptrs)
    if (!aligned(ptr, 4) || !device_accessible(ptr)) return LION_ERR_INVALID_ARG;
  if (!aligned(S, 16)) return LION_ERR_INVALID_ARG;   // the state moves as float4 rows
  if (mask_kind != LION_MASK_LIT && !device_accessible(log_lambda)) return LION_ERR_INVALID_ARG;
  const int phi = lion::resolve_phi(mask_kind, LION_PHI_DEFAULT);
  return from_cuda(lion::launch_rnn_step(q, k, v, log_lambda, S, z, y_part, c_part, B, H, d,
                                         mask_kind, phi, dtype, stream));
}

}  // extern "C"
