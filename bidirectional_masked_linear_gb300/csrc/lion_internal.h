// lion_internal.h -- interface between the C ABI layer and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/lion.h"

namespace lion {

// Argument checks of lion_attn_fwd_ex (null pointers, sizes, enums,
// alignment, device-accessible memory, the full form's length limit), done
// on the host before anything is launched.
lion_status validate_args(const lion_args* a);
// The forward on arguments that already passed validate_args.
lion_status forward_checked(const lion_args* a);

struct Problem {
  const void* q;
  const void* k;
  const void* v;
  const float* log_lambda;
  float* out;        // bfloat16 [B][H][L][d] when out_bf16 (chunk-128 kernels only)
  int B, H, L, d;
  int mask_kind;
  int phi;     // resolved (never PHI_DEFAULT)
  int dtype;   // DT_BF16 / DT_FP32
  int chunk;
  int causal = 0;   // 1: only j <= i (the forward half), SIMT kernels only
  int out_bf16 = 0; // 1: the chunk-128 tensor-core kernels store y as bfloat16
};

// SIMT (CUDA-core) kernels: any d in {16,32,64,128}, both dtypes.
cudaError_t launch_full_simt(const Problem& p, cudaStream_t s);
// The recurrent form.  The workspace holds c^F (B*H*L floats) and, when it
// is rnn_workspace_bytes long, the features of every token, computed once
// by a first launch, and room for the backward sweep's sums when the two
// sweeps run apart; with the c^F part alone each column CTA computes the
// features and runs both sweeps.
size_t rnn_workspace_bytes(int B, int H, int L, int d);
cudaError_t launch_rnn_simt(const Problem& p, float* ws, size_t ws_bytes, cudaStream_t s);
cudaError_t launch_chunk_simt(const Problem& p, float* ws_den /*[B*H*L]*/, cudaStream_t s);
// The chunk form on the CUDA cores with register-tiled block products, for
// chunks of at most kChunkTileMax tokens: a workspace of
// chunk_tile_workspace_bytes (the normalisers and the features of every
// token), two launches.
constexpr int kChunkTileMax = 64;
bool chunk_tile_supported(const Problem& p);
size_t chunk_tile_workspace_bytes(int B, int H, int L, int d);
cudaError_t launch_chunk_tile(const Problem& p, float* ws, cudaStream_t s);
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

// Segment plan and segment scan of the long-sequence tensor-core paths.  Per
// head the sequence is cut into 256-token blocks and segments of `SEGB`
// blocks (`nseg` of them, so that B*H*nseg fills the SMs).  A pre-pass
// writes per segment
//   segsum[bh][s] (fp32): forward summary [64 m][80] (sum over the segment of
//                 exp(P_last - P_j) phi(k_j) [v_j; 1]^T, anchored at its last
//                 token), backward summary [64][80] (exp(P_j - P_first) ...,
//                 anchored at its first token), then the sum of log(lambda)
//                 over the segment;
// and the chunk-64 path's scan chains them into
//   segin[bh][s]  (fp32): forward state entering segment s from the left
//                 [64][80], backward state entering it from the right [64][80]
// (column 64 of a [64][80] state is z; 65..79 are zero).  The chunk-128
// path's main pass chains them itself, with the same recurrences.
constexpr int kLongStateCols = 80;
constexpr int kSegSumFloats = 2 * 64 * kLongStateCols + 4;
constexpr int kSegInFloats = 2 * 64 * kLongStateCols;
struct LongPlan {
  int NBL, SEGB, nseg;
};
LongPlan long_plan(int B, int H, int L);

// Per-chunk backward states of the 128-token-chunk path: for chunk c of a
// head, the backward state entering it from the right, from the tokens after
// it within its segment, anchored at the first token after the chunk, stored
// transposed as 65 rows (row n < 64: column n of the state over the 64 key
// features m; row 64: z) of 64 fp16 values, the 16-byte pieces of row r in
// the order j ^ (r & 7) (the 128-byte swizzle of the operand tiles).
constexpr int kGstBytes = 65 * 128;

// Tensor-core chunkwise kernel with 128-token chunks: bf16, d = 64,
// chunk = 128.  L <= 256: one launch, no workspace.
bool chunk128_tc_supported(const Problem& p);
cudaError_t launch_chunk128_tc(const Problem& p, int* status, cudaStream_t s);
// The same for L > 256: a backward pre-pass over 128-token chunks (per-chunk
// states and segment summaries) and the main pass, which chains the
// segment summaries at its start (two launches; workspace as returned).
bool chunk128_long_supported(const Problem& p);
size_t chunk128_long_workspace_bytes(int B, int H, int L);
cudaError_t launch_chunk128_long(const Problem& p, void* ws, int* status, cudaStream_t s);
cudaError_t launch_chunk128_pre(const Problem& p, const LongPlan& plan, uint8_t* gst, float* segsum, int* status,
                                cudaStream_t s);

// Gradients through the full form (fp32, CUDA cores): dq, dk, dv [B][H][L][d],
// dll as the public entry point describes; workspace of bwd_workspace_bytes.
size_t bwd_workspace_bytes(int B, int H, int L, int d);
cudaError_t launch_bwd(const Problem& p, const float* dy, float* dq, float* dk, float* dv, float* dll, void* ws,
                       cudaStream_t s);

// dlog_lambda from the row and column terms of dLoss/dP ([B*H][L] each):
// LION-S the suffix sums (position 0: 0), LION-D the position-weighted sum
// per head (dsum, [B*H] doubles) and then over the batch; LIT nothing.
cudaError_t launch_dlog_lambda(int B, int H, int L, int mask_kind, const float* rowd, const float* cold, double* dsum,
                               float* dll, cudaStream_t s);

// Gradients through the chunkwise form (fp32, CUDA cores), any L: chunks of
// bwd_chunk_length(d) tokens, states scanned across chunks; outputs as
// launch_bwd; workspace of bwd_chunk_workspace_bytes; bwd_chunk_launches
// kernels a call.
int bwd_chunk_length(int d);
size_t bwd_chunk_workspace_bytes(int B, int H, int L, int d);
int bwd_chunk_launches(int mask_kind);
cudaError_t launch_bwd_chunk(const Problem& p, const float* dy, float* dq, float* dk, float* dv, float* dll, void* ws,
                             cudaStream_t s);

// Full form with the mask averaged over two traversal orders (order: device
// int32 [2][L]); fp32 on the CUDA cores, d in {64, 128}; workspace of
// reorder_workspace_bytes; reorder_launches kernels a call.
size_t reorder_workspace_bytes(int B, int H, int L, int d);
// The plain full form (d = 64 or 128) on the reordered form's register-tiled
// kernel with the tokens' own order: phi(q), phi(k) and LION-S's prefix in a
// workspace of full_tiled_workspace_bytes, full_tiled_launches kernels.
bool full_tiled_supported(const Problem& p);
size_t full_tiled_workspace_bytes(int B, int H, int L, int d);
int full_tiled_launches(int mask_kind);
cudaError_t launch_full_tiled(const Problem& p, void* ws, cudaStream_t s);
int reorder_launches(int mask_kind);
cudaError_t launch_reordered(const Problem& p, const int* order, void* ws, int* status, cudaStream_t s);
// Its gradients: dq, dk, dv [B][H][L][d], dll (LION-D [H], LION-S [B][H][L]).
size_t reorder_bwd_workspace_bytes(int B, int H, int L, int d);
int reorder_bwd_launches(int mask_kind);
cudaError_t launch_reordered_bwd(const Problem& p, const int* order, const float* dy, float* dq, float* dk, float* dv,
                                 float* dll, void* ws, int* status, cudaStream_t s);

// y (fp32, n values) rounded to nearest even bfloat16.
cudaError_t launch_f32_to_bf16(const float* src, void* dst, size_t n, cudaStream_t s);

// Device-side status word that kernels set when a bounded wait gives up
// (kStatusTimeout), a traversal order is not a permutation
// (kStatusBadOrder), or a tensor-core kernel met a value that its fp16
// operands cannot hold (kStatusRange); address on the current device,
// nullptr if it cannot be resolved.
constexpr int kStatusTimeout = 1;
constexpr int kStatusBadOrder = 2;
constexpr int kStatusRange = 3;   // a value past the fp16 range of a tensor-core operand
int* device_status_ptr();

// Bound, in SM clock cycles, on every mbarrier wait of the tensor-core
// kernels (a launch parameter; lion_debug_set_wait_cycles changes it).
long long wait_limit_cycles();

// Largest chunk the SIMT chunk kernel takes (its chunk-local prefix lives in
// shared memory).
constexpr int kSimtMaxChunk = 1024;

}  // namespace lion
