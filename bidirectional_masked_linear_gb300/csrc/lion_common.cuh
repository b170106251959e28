// lion_common.cuh -- device helpers shared by the LION kernels.
//
// Feature maps (rebuttal page "LION: A bidirectional framework ...", reply
// "4) Default non-linearity"): elu(x)+1 for LION-LIT / LION-D and SiLU
// followed by an L2 normalisation over the head dimension for LION-S.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace lion {

enum { MASK_LIT = 0, MASK_D = 1, MASK_S = 2 };
enum { PHI_DEFAULT = 0, PHI_ELU1 = 1, PHI_SILU_L2 = 2, PHI_IDENTITY = 3 };
enum { DT_BF16 = 0, DT_FP32 = 1 };

__host__ __device__ inline int resolve_phi(int mask_kind, int phi) {
  if (phi != PHI_DEFAULT) return phi;
  return mask_kind == MASK_S ? PHI_SILU_L2 : PHI_ELU1;
}

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

__device__ __forceinline__ float elu1(float x) { return x > 0.f ? x + 1.f : expf(x); }
__device__ __forceinline__ float silu(float x) { return x / (1.f + expf(-x)); }

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Apply phi in place to `rows` rows of `D` floats in shared memory (row
// stride `ld`).  Rows at or beyond `valid` are zeroed (padding tokens must
// contribute nothing: phi(0) = 1 for elu+1).  Whole block participates;
// one warp per row.
__device__ inline void phi_rows_inplace(float* tile, int rows, int valid, int D, int ld, int phi) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  for (int r = warp; r < rows; r += nw) {
    float* row = tile + r * ld;
    if (r >= valid) {
      for (int m = lane; m < D; m += 32) row[m] = 0.f;
      continue;
    }
    if (phi == PHI_ELU1) {
      for (int m = lane; m < D; m += 32) row[m] = elu1(row[m]);
    } else if (phi == PHI_SILU_L2) {
      float ss = 0.f;
      for (int m = lane; m < D; m += 32) {
        float u = silu(row[m]);
        row[m] = u;
        ss += u * u;
      }
      ss = warp_sum(ss);
      float inv = 1.f / fmaxf(sqrtf(ss), 1e-12f);
      for (int m = lane; m < D; m += 32) row[m] *= inv;
    }
    // identity: nothing
  }
}

// Mask exponent log(M_ij) for tokens i, j of one chunk/panel set whose
// inclusive prefix values (relative to any common origin) are Pi, Pj.
// M_ij = exp(P_max(i,j) - P_min(i,j)) with max/min taken over the INDEX.
__device__ __forceinline__ float mask_exponent(int i, int j, float Pi, float Pj) {
  return i >= j ? Pi - Pj : Pj - Pi;
}


// Launches kern as a programmatic dependent of the work before it on s: it
// may start before that work ends, and waits for it (griddepcontrol.wait)
// before it reads what that work wrote.
template <typename... Args>
cudaError_t launch_dependent(void (*kern)(Args...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

}  // namespace lion
