// lion_internal.h -- interface between the C ABI layer and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

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

// Backward pre-pass and segment scan of the chunk-64 kernel, run for the
// 128-token-chunk main pass of sequences longer than 256 tokens.  Per head the
// sequence is cut into 256-token blocks and segments of `SEGB` blocks:
//   gloc[bh][b]  backward state entering block b from the right, from the
//                blocks after it within its segment (anchored at the first
//                token after the block);
//   gmid[bh][b]  the same at the block's token 128 (anchored there), also
//                taking in the block's own tokens 128..255;
// both fp16 [64 rows m][64 columns n] followed by fp32 z[64];
//   segsum[bh][s] (fp32): forward summary [64][80], backward summary
//                [64][80], then the sum of log(lambda) over the segment;
//   segin[bh][s]  (fp32): forward state entering segment s from the left
//                [64][80], backward state entering it from the right [64][80]
// (column 64 of a [64][80] state is z; 65..79 are zero).
constexpr int kLongStateCols = 80;
constexpr int kGlocBytes = 64 * 64 * 2 + 64 * 4;
constexpr int kSegSumFloats = 2 * 64 * kLongStateCols + 4;
constexpr int kSegInFloats = 2 * 64 * kLongStateCols;
struct LongStates {
  int NBL, SEGB, nseg;
  const uint8_t* gloc;
  const uint8_t* gmid;
  const float* segsum;
  const float* segin;
};
size_t long_states_workspace_bytes(int B, int H, int L);
cudaError_t launch_long_states(const Problem& p, void* ws, int* status, cudaStream_t s, LongStates* out);

// Tensor-core chunkwise kernel with 128-token chunks: bf16, d = 64,
// chunk = 128.  L <= 256: one launch, no workspace.
bool chunk128_tc_supported(const Problem& p);
cudaError_t launch_chunk128_tc(const Problem& p, int* status, cudaStream_t s);
// The same for L > 256: the chunk-64 pre-pass and segment scan above, then a
// 128-token-chunk main pass (three launches; workspace as returned).
bool chunk128_long_supported(const Problem& p);
size_t chunk128_long_workspace_bytes(int B, int H, int L);
cudaError_t launch_chunk128_long(const Problem& p, void* ws, int* status, cudaStream_t s);

// Device-side status word that kernels set when a bounded wait gives up
// (address on the current device; nullptr if it cannot be resolved).
int* device_status_ptr();

// Largest chunk the SIMT chunk kernel takes (its chunk-local prefix lives in
// shared memory).
constexpr int kSimtMaxChunk = 1024;

}  // namespace lion
