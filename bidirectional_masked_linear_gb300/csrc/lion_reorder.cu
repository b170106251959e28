// lion_reorder.cu -- the full form with the mask averaged over two traversal
// orders of the tokens: LION-S (v2) and the reordered-patch LION-D / LION-S
// (rebuttal page "LION: A bidirectional framework that trains like a
// Transformer and infers like an RNN", reply "P2: Comparison against vision
// SSMs", item 1, which averages the two masks of its Figure 7 b and c; results
// page "LION Part IV - Results", "Model Comparisons", the rows marked natural).
// The figure is not on the pages, so the two orders are inputs.
//
// Along an order, position t holds token order[t], and the mask between two
// tokens is LION's mask of the reordered sequence: the product of the decays
// of the tokens at the positions after the earlier of the two, up to and
// including the later one.  Written with a per-token coordinate C^p,
//   M^p_ab = exp(-|C^p_a - C^p_b| w),
// where LION-S takes C^p_a = the inclusive prefix of the reordered
// log-decays at a's position and w = 1 (the decays are <= 1), and LION-D
// takes C^p_a = a's position and w = -log(lambda_h); LIT has M = 1.  The
// operator is y_i = sum_j M_ij s_ij v_j / sum_j M_ij s_ij with
// M = (M^1 + M^2) / 2 inside the row-sum normaliser.
//
// Kernels, fp32 on the CUDA cores, d in {64, 128}: (1) per order, check that
// it is a permutation and write each token's position (an invalid order sets
// the library's status word to kStatusBadOrder; indices are clamped so that
// every access stays in bounds); (2) LION-S: per head and order, the prefix of
// the reordered log-decays (a block scan in double) scattered to the tokens;
// (3) phi(q), phi(k) into the workspace; (4) per block of 32 queries, the
// register-tiled full form over key tiles of 64 tokens (tile_simt.cuh).
#include "lion_common.cuh"
#include "lion_internal.h"
#include "tile_simt.cuh"

namespace lion {
namespace {

struct ReorderParams {
  const void* q;
  const void* k;
  const void* v;
  const float* log_lambda;
  const int* order;   // [2][L]
  float* out;
  int B, H, L, mask_kind;
  float* fq;          // [BH][L][D] phi(q)
  float* fk;          // [BH][L][D] phi(k)
  int* pos;           // [2][L]     position of each token in each order
  float* coord;       // LION-S [2][BH][L] prefixes; LION-D [2][L] positions
  int* status;
};

__device__ __forceinline__ int clamp_token(int a, int L) { return a < 0 ? 0 : a >= L ? L - 1 : a; }

// (1) one CTA per order; dynamic shared memory: L ints.
constexpr int kOrderThreads = 1024;
__global__ void __launch_bounds__(kOrderThreads) order_positions_kernel(ReorderParams p) {
  extern __shared__ int cnt[];
  const int L = p.L, o = blockIdx.x;
  const int* ord = p.order + (size_t)o * L;
  int* pos = p.pos + (size_t)o * L;
  for (int t = threadIdx.x; t < L; t += blockDim.x) {
    cnt[t] = 0;
    pos[t] = 0;
  }
  __syncthreads();
  int bad = 0;
  for (int t = threadIdx.x; t < L; t += blockDim.x) {
    const int a = ord[t];
    if (a < 0 || a >= L) {
      bad = 1;
      continue;
    }
    atomicAdd(&cnt[a], 1);
    pos[a] = t;   // a token listed twice makes the order invalid; the value stays in range
  }
  __syncthreads();
  for (int t = threadIdx.x; t < L; t += blockDim.x) bad |= cnt[t] != 1;
  if (__syncthreads_or(bad) && threadIdx.x == 0) atomicExch(p.status, kStatusBadOrder);
  if (p.mask_kind == MASK_D)
    for (int t = threadIdx.x; t < L; t += blockDim.x) p.coord[(size_t)o * L + t] = (float)pos[t];
}

// (2) LION-S: grid (B*H, 2), kScanThreads threads.
__global__ void __launch_bounds__(kScanThreads) order_prefix_kernel(ReorderParams p) {
  const int L = p.L, bh = blockIdx.x, o = blockIdx.y, t0 = threadIdx.x;
  const int* ord = p.order + (size_t)o * L;
  const float* ll = p.log_lambda + (size_t)bh * L;
  float* C = p.coord + ((size_t)o * gridDim.x + bh) * L;
  const int per = (L + kScanThreads - 1) / kScanThreads;
  const int lo = min(L, t0 * per), hi = min(L, lo + per);
  double run = 0.0, all;
  for (int t = lo; t < hi; ++t) run += (double)ll[clamp_token(ord[t], L)];
  double off = block_scan(run, &all) - run;
  for (int t = lo; t < hi; ++t) {
    const int a = clamp_token(ord[t], L);
    off += (double)ll[a];
    C[a] = (float)off;
  }
}

template <int D>
constexpr size_t reorder_smem() {
  return sizeof(float) * ((size_t)(kTR + 2 * kTC) * (D + 4) + kTR * kTAL + 2 * kTC);
}

// (4) 32 queries per CTA.
template <typename T, int D>
__global__ void __launch_bounds__(kTThreads) reorder_full_kernel(ReorderParams p) {
  constexpr int LD = D + 4, MF = D / 16, U = D / 64;
  extern __shared__ __align__(16) float smem[];
  float* sQ = smem;                  // [kTR][LD]   phi(q) of the block
  float* sK = sQ + kTR * LD;         // [kTC][LD]   phi(k) of the tile
  float* sV = sK + kTC * LD;         // [kTC][LD]   v of the tile
  float* sA = sV + kTC * LD;         // [kTR][kTAL] M (.) S
  float* sC = sA + kTR * kTAL;       // [2][kTC]    coordinates of the tile's keys
  const int L = p.L, BH = gridDim.x, bh = blockIdx.x, h = bh % p.H, i0 = blockIdx.y * kTR;
  const int nr = min(kTR, L - i0);
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const bool lit = p.mask_kind == MASK_LIT;
  const float w = p.mask_kind == MASK_D ? -p.log_lambda[h] : 1.f;
  const float* C0 = nullptr;
  const float* C1 = nullptr;
  if (p.mask_kind == MASK_S) {
    C0 = p.coord + (size_t)bh * L;
    C1 = p.coord + ((size_t)BH + bh) * L;
  } else if (p.mask_kind == MASK_D) {
    C0 = p.coord;
    C1 = p.coord + L;
  }
  const float* fkh = p.fk + (size_t)bh * L * D;
  const T* vh = head_of<T>(p.v, bh, L, D);
  stage_rows<D>(sQ, p.fq + (size_t)bh * L * D, i0, kTR, L);
  int ia[4];
  bool live[4];
  float c0[4], c1[4];
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    ia[a] = i0 + ty + 8 * a;
    live[a] = ia[a] < L;
    c0[a] = !lit && live[a] ? C0[ia[a]] : 0.f;
    c1[a] = !lit && live[a] ? C1[ia[a]] : 0.f;
  }
  float den[4], num[4][MF];
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    den[a] = 0.f;
#pragma unroll
    for (int f = 0; f < MF; ++f) num[a][f] = 0.f;
  }
  for (int j0 = 0; j0 < L; j0 += kTC) {
    stage_rows<D>(sK, fkh, j0, kTC, L);
    stage_rows<D>(sV, vh, j0, kTC, L);
    if (!lit) {
      stage_vec(sC, C0, j0, kTC, L);
      stage_vec(sC + kTC, C1, j0, kTC, L);
    }
    __syncthreads();
    const int nc = min(kTC, L - j0);
    float s[4][4];
    tile_scores<D>(sQ, sK, ty, tx, nr, nc, s);
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int jl = tx + 16 * b, j = j0 + jl;
        float m = 0.f;
        if (live[a] && j < L)
          m = lit ? 1.f
                  : 0.5f * (expf(-fabsf(c0[a] - sC[jl]) * w) + expf(-fabsf(c1[a] - sC[kTC + jl]) * w));
        const float x = m * s[a][b];
        den[a] += x;
        sA[(ty + 8 * a) * kTAL + jl] = x;
      }
    __syncthreads();
    tile_apply<D>(sA, sV, (nc + 3) & ~3, ty, tx, nr, num);
    __syncthreads();
  }
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const float dn = group_sum<16>(den[a]);
    if (!live[a]) continue;
    float* y = p.out + ((size_t)bh * L + ia[a]) * D;
#pragma unroll
    for (int u = 0; u < U; ++u)
      *reinterpret_cast<float4*>(y + 4 * tx + 64 * u) =
          make_float4(num[a][4 * u] / dn, num[a][4 * u + 1] / dn, num[a][4 * u + 2] / dn, num[a][4 * u + 3] / dn);
  }
}

template <typename Kern>
cudaError_t allow_smem(Kern kern, size_t bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <typename T, int D>
cudaError_t reorder_launch(const ReorderParams& p, int phi, cudaStream_t s) {
  const long BH = (long)p.B * p.H;
  order_positions_kernel<<<2, kOrderThreads, sizeof(int) * (size_t)p.L, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (p.mask_kind == MASK_S) {
    order_prefix_kernel<<<dim3((unsigned)BH, 2), kScanThreads, 0, s>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if ((e = launch_phi_rows<T, D>(p.q, p.k, p.fq, p.fk, BH * p.L, phi, s)) != cudaSuccess) return e;
  constexpr size_t smem = reorder_smem<D>();
  if ((e = allow_smem(reorder_full_kernel<T, D>, smem)) != cudaSuccess) return e;
  reorder_full_kernel<T, D><<<dim3((unsigned)BH, (p.L + kTR - 1) / kTR), kTThreads, smem, s>>>(p);
  return cudaGetLastError();
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

size_t reorder_workspace_bytes(int B, int H, int L, int d) {
  const size_t BH = (size_t)B * H, n = BH * L;
  return 2 * align256(sizeof(float) * n * d) + align256(sizeof(int) * 2 * (size_t)L) +
         align256(sizeof(float) * 2 * n);
}

int reorder_launches(int mask_kind) { return mask_kind == MASK_S ? 4 : 3; }

cudaError_t launch_reordered(const Problem& pr, const int* order, void* ws, int* status, cudaStream_t s) {
  ReorderParams p;
  p.q = pr.q;
  p.k = pr.k;
  p.v = pr.v;
  p.log_lambda = pr.log_lambda;
  p.order = order;
  p.out = pr.out;
  p.B = pr.B;
  p.H = pr.H;
  p.L = pr.L;
  p.mask_kind = pr.mask_kind;
  p.status = status;
  const size_t BH = (size_t)pr.B * pr.H, n = BH * pr.L;
  uint8_t* w = static_cast<uint8_t*>(ws);
  p.fq = reinterpret_cast<float*>(w);
  w += align256(sizeof(float) * n * pr.d);
  p.fk = reinterpret_cast<float*>(w);
  w += align256(sizeof(float) * n * pr.d);
  p.pos = reinterpret_cast<int*>(w);
  w += align256(sizeof(int) * 2 * (size_t)pr.L);
  p.coord = reinterpret_cast<float*>(w);
  const bool bf = pr.dtype == DT_BF16;
  switch (pr.d) {
    case 64: return bf ? reorder_launch<__nv_bfloat16, 64>(p, pr.phi, s) : reorder_launch<float, 64>(p, pr.phi, s);
    case 128: return bf ? reorder_launch<__nv_bfloat16, 128>(p, pr.phi, s) : reorder_launch<float, 128>(p, pr.phi, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace lion
