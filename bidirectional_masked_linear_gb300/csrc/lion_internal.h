// lion_internal.h -- interface between the C ABI layer and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

namespace lion {

struct Problem {
  const void* q;
  const void* k;
  const void* v;
  const float* log_lambda;
  float* out;
  int B, H, L, d;
  int mask_kind;
  int phi;     // resolved (never PHI_DEFAULT)
  int dtype;   // DT_BF16 / DT_FP32
  int chunk;
};

// SIMT (CUDA-core) kernels: any d in {16,32,64,128}, both dtypes.
cudaError_t launch_full_simt(const Problem& p, cudaStream_t s);
cudaError_t launch_rnn_simt(const Problem& p, float* ws_c /*[B*H*L]*/, cudaStream_t s);
cudaError_t launch_chunk_simt(const Problem& p, float* ws_den /*[B*H*L]*/, cudaStream_t s);
cudaError_t launch_rnn_step(const void* q, const void* k, const void* v, const float* log_lambda,
                            float* S, float* z, float* y_part, float* c_part, int B, int H,
                            int d, int mask_kind, int phi, int dtype, cudaStream_t s);

// Tensor-core chunkwise kernel (tcgen05 + TMEM + TMA): bf16, d = 64,
// chunk = 64, any L.  Sequences longer than 256 tokens take three launches
// and a workspace of chunk_tc_workspace_bytes (0 for L <= 256).
bool chunk_tc_supported(const Problem& p);
size_t chunk_tc_workspace_bytes(int B, int H, int L);
int chunk_tc_launches(int B, int H, int L);
cudaError_t launch_chunk_tc(const Problem& p, void* ws, int* status, cudaStream_t s);

// Tensor-core chunkwise kernel with 128-token chunks: bf16, d = 64,
// chunk = 128, L <= 256 (one launch, no workspace).
bool chunk128_tc_supported(const Problem& p);
cudaError_t launch_chunk128_tc(const Problem& p, int* status, cudaStream_t s);

// Device-side status word that kernels set when a bounded wait gives up
// (address on the current device; nullptr if it cannot be resolved).
int* device_status_ptr();

// Largest chunk the SIMT chunk kernel takes (its chunk-local prefix lives in
// shared memory).
constexpr int kSimtMaxChunk = 1024;

}  // namespace lion
