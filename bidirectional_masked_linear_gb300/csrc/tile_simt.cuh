// tile_simt.cuh -- CUDA-core building blocks shared by the full-form passes
// that run in fp32 with register tiling (the gradients, and the forward with
// the mask averaged over two traversal orders): lane-group sums, vector loads,
// a block scan in double, the feature-map pass, and the staging and tile
// products of a 128-thread CTA that holds 32 rows of one side and walks the
// other side in tiles of 64 tokens.
#pragma once

#include "lion_common.cuh"

namespace lion {
namespace {

template <typename T>
__device__ __forceinline__ const T* head_of(const void* base, int bh, int L, int D) {
  return reinterpret_cast<const T*>(base) + (size_t)bh * L * D;
}

// sum over W adjacent lanes (W a power of two, the group aligned to W)
template <int W = 8>
__device__ __forceinline__ float group_sum(float x) {
#pragma unroll
  for (int o = 1; o < W; o <<= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Four consecutive features as fp32 (16-byte aligned for fp32, 8 for bf16).
__device__ __forceinline__ float4 load4(const float* src) { return *reinterpret_cast<const float4*>(src); }
__device__ __forceinline__ float4 load4(const __nv_bfloat16* src) {
  const uint2 u = *reinterpret_cast<const uint2*>(src);
  const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  return make_float4(lo.x, lo.y, hi.x, hi.y);
}
__device__ __forceinline__ float elem(const float4& x, int e) {
  return e == 0 ? x.x : e == 1 ? x.y : e == 2 ? x.z : x.w;
}

// Inclusive scan of x over a block of kScanThreads threads in double (lane
// shuffles, then the warp totals); *total receives the block's sum.
constexpr int kScanThreads = 256;
__device__ __forceinline__ double block_scan(double x, double* total) {
  __shared__ double warp_tot[kScanThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  double off = 0.0, all = 0.0;
#pragma unroll
  for (int u = 0; u < kScanThreads / 32; ++u) {
    off += u < warp ? warp_tot[u] : 0.0;
    all += warp_tot[u];
  }
  *total = all;
  return x + off;
}

// dphi -> dx for this thread's NC features of one row, the row's W threads
// (adjacent lanes) together holding all of its features and cooperating on
// the SiLU + L2 norm.
template <int NC, int W = 8>
__device__ __forceinline__ void phi_backward(int phi, const float* x, const float* dphi, float* dx) {
  if (phi == PHI_ELU1) {
#pragma unroll
    for (int c = 0; c < NC; ++c) dx[c] = x[c] > 0.f ? dphi[c] : expf(x[c]) * dphi[c];
  } else if (phi == PHI_SILU_L2) {
    float u[NC], sg[NC], ss = 0.f;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      sg[c] = 1.f / (1.f + expf(-x[c]));
      u[c] = x[c] * sg[c];
      ss += u[c] * u[c];
    }
    const float nrm = sqrtf(group_sum<W>(ss));
    float dx_scale, dot = 0.f;
    if (nrm >= 1e-12f) {
#pragma unroll
      for (int c = 0; c < NC; ++c) dot += u[c] / nrm * dphi[c];
      dot = group_sum<W>(dot);
      dx_scale = 1.f / nrm;
    } else {
      dx_scale = 1e12f;
    }
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      const float f = nrm >= 1e-12f ? u[c] / nrm : 0.f;
      const float du = (dphi[c] - f * dot) * dx_scale;
      dx[c] = du * sg[c] * (1.f + x[c] * (1.f - sg[c]));
    }
  } else {
#pragma unroll
    for (int c = 0; c < NC; ++c) dx[c] = dphi[c];
  }
}

// phi(q) and phi(k) of `rows` rows each into fq and fk (fp32): D/4 adjacent
// lanes per row, four features a lane.
template <typename T, int D>
__global__ void __launch_bounds__(256) phi_rows_kernel(const void* q, const void* k, float* fq, float* fk, long rows,
                                                       int phi) {
  constexpr int W = D / 4;   // divides 32: a row's lanes never straddle a warp
  const long t = (long)blockIdx.x * blockDim.x + threadIdx.x;
  // lanes past the last row work on it without storing, so that every lane
  // takes part in its group's shuffles
  const bool ok = t / W < 2 * rows;
  const long r = ok ? t / W : 2 * rows - 1;
  const int c = (int)(t % W) * 4;
  const bool isq = r < rows;
  const long rr = isq ? r : r - rows;
  float4 x = load4(reinterpret_cast<const T*>(isq ? q : k) + (size_t)rr * D + c);
  if (phi == PHI_ELU1) {
    x = make_float4(elu1(x.x), elu1(x.y), elu1(x.z), elu1(x.w));
  } else if (phi == PHI_SILU_L2) {
    x = make_float4(silu(x.x), silu(x.y), silu(x.z), silu(x.w));
    const float ss = group_sum<W>(x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w);
    const float inv = 1.f / fmaxf(sqrtf(ss), 1e-12f);
    x = make_float4(x.x * inv, x.y * inv, x.z * inv, x.w * inv);
  }
  if (ok) *reinterpret_cast<float4*>((isq ? fq : fk) + (size_t)rr * D + c) = x;
}
template <typename T, int D>
cudaError_t launch_phi_rows(const void* q, const void* k, float* fq, float* fk, long rows, int phi, cudaStream_t s) {
  phi_rows_kernel<T, D><<<(unsigned)((2 * rows * (D / 4) + 255) / 256), 256, 0, s>>>(q, k, fq, fk, rows, phi);
  return cudaGetLastError();
}

// Tiles.  A CTA of 128 threads is an 8 x 16 grid (ty = 0..7, tx = 0..15).
// Each thread computes the 4 x 4 piece (rows ty + 8a, columns tx + 16b) of a
// 32 x 64 tile of scores with whole dot products over the features in its own
// registers, and accumulates outputs for its 4 rows and the d/16 features
// 4tx + 64u + e.  Operand rows sit in shared memory with a stride of d + 4
// floats and are read as float4 along the features: consecutive column
// threads read consecutive rows (4 banks apart: no conflicts) and the row
// threads of a quarter warp read one address (a broadcast).
constexpr int kTR = 32;            // rows of a block
constexpr int kTC = 64;            // tokens of a tile of the other side
constexpr int kTAL = kTC + 16;     // row stride of the staged score tiles (floats)
constexpr int kTThreads = 128;


// Rows [row0, row0 + nrows) of a [L][D] head array into dst (row stride
// D + 4 floats), zero past L.  Whole block.
template <int D, typename T>
__device__ __forceinline__ void stage_rows(float* dst, const T* src, int row0, int nrows, int L) {
  constexpr int V = D / 4, LD = D + 4;
  for (int idx = threadIdx.x; idx < nrows * V; idx += blockDim.x) {
    const int r = idx / V, c = (idx - r * V) * 4, i = row0 + r;
    const float4 x = i < L ? load4(src + (size_t)i * D + c) : make_float4(0.f, 0.f, 0.f, 0.f);
    *reinterpret_cast<float4*>(dst + r * LD + c) = x;
  }
}
__device__ __forceinline__ void stage_vec(float* dst, const float* src, int row0, int n, int L) {
  for (int t = threadIdx.x; t < n; t += blockDim.x) dst[t] = row0 + t < L ? src[row0 + t] : 0.f;
}

// acc[a][b] = sum_m X[ty + 8a][m] Y[tx + 16b][m] for a < NA, b < NB (the
// caller zeroes acc)
template <int D, int NA, int NB>
__device__ __forceinline__ void tile_scores_n(const float* X, const float* Y, int ty, int tx, float (&acc)[4][4]) {
  constexpr int LD = D + 4;
#pragma unroll 4
  for (int m = 0; m < D; m += 4) {
    float4 x[NA], y[NB];
#pragma unroll
    for (int a = 0; a < NA; ++a) x[a] = *reinterpret_cast<const float4*>(X + (ty + 8 * a) * LD + m);
#pragma unroll
    for (int b = 0; b < NB; ++b) y[b] = *reinterpret_cast<const float4*>(Y + (tx + 16 * b) * LD + m);
#pragma unroll
    for (int a = 0; a < NA; ++a)
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        float t = acc[a][b];
        t = fmaf(x[a].x, y[b].x, t);
        t = fmaf(x[a].y, y[b].y, t);
        t = fmaf(x[a].z, y[b].z, t);
        acc[a][b] = fmaf(x[a].w, y[b].w, t);
      }
  }
}

// Row (column) slices a thread needs when only the first nr rows of X (nc of
// Y) are real tokens: 1, 2 or all 4 (uniform over the CTA).
__device__ __forceinline__ int slices(int n, int step) { return n > 2 * step ? 4 : n > step ? 2 : 1; }

// acc[a][b] = sum_m X[ty + 8a][m] Y[tx + 16b][m]; entries whose row is past
// nr or whose column is past nc are left 0.
template <int D>
__device__ __forceinline__ void tile_scores(const float* X, const float* Y, int ty, int tx, int nr, int nc,
                                            float (&acc)[4][4]) {
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;
  const int na = slices(nr, 8), nb = slices(nc, 16);
  if (na == 4) {
    if (nb == 4) tile_scores_n<D, 4, 4>(X, Y, ty, tx, acc);
    else if (nb == 2) tile_scores_n<D, 4, 2>(X, Y, ty, tx, acc);
    else tile_scores_n<D, 4, 1>(X, Y, ty, tx, acc);
  } else if (na == 2) {
    if (nb == 4) tile_scores_n<D, 2, 4>(X, Y, ty, tx, acc);
    else if (nb == 2) tile_scores_n<D, 2, 2>(X, Y, ty, tx, acc);
    else tile_scores_n<D, 2, 1>(X, Y, ty, tx, acc);
  } else {
    if (nb == 4) tile_scores_n<D, 1, 4>(X, Y, ty, tx, acc);
    else if (nb == 2) tile_scores_n<D, 1, 2>(X, Y, ty, tx, acc);
    else tile_scores_n<D, 1, 1>(X, Y, ty, tx, acc);
  }
}

// out[a][4u + e] += sum_{t < n} S[ty + 8a][t] Z[t][4tx + 64u + e] for a < NA;
// n is a multiple of 4 and S is zero from the last real token to n.
template <int D, int NA>
__device__ __forceinline__ void tile_apply_n(const float* S, const float* Z, int n, int ty, int tx,
                                             float (&out)[4][D / 16]) {
  constexpr int LD = D + 4, U = D / 64;
#pragma unroll 2
  for (int t = 0; t < n; t += 4) {
    float4 s[NA];
#pragma unroll
    for (int a = 0; a < NA; ++a) s[a] = *reinterpret_cast<const float4*>(S + (ty + 8 * a) * kTAL + t);
#pragma unroll
    for (int e = 0; e < 4; ++e)
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const float4 z = *reinterpret_cast<const float4*>(Z + (t + e) * LD + 4 * tx + 64 * u);
#pragma unroll
        for (int a = 0; a < NA; ++a) {
          const float w = elem(s[a], e);
          out[a][4 * u + 0] = fmaf(w, z.x, out[a][4 * u + 0]);
          out[a][4 * u + 1] = fmaf(w, z.y, out[a][4 * u + 1]);
          out[a][4 * u + 2] = fmaf(w, z.z, out[a][4 * u + 2]);
          out[a][4 * u + 3] = fmaf(w, z.w, out[a][4 * u + 3]);
        }
      }
  }
}
// The same for the first nr rows of S (the rows past nr keep their values).
template <int D>
__device__ __forceinline__ void tile_apply(const float* S, const float* Z, int n, int ty, int tx, int nr,
                                           float (&out)[4][D / 16]) {
  const int na = slices(nr, 8);
  if (na == 4) tile_apply_n<D, 4>(S, Z, n, ty, tx, out);
  else if (na == 2) tile_apply_n<D, 2>(S, Z, n, ty, tx, out);
  else tile_apply_n<D, 1>(S, Z, n, ty, tx, out);
}

// out[a][4u + e] += sum_{t < n} S[t][4ty + a] Z[t][4tx + 64u + e] (S with
// row stride lds, its rows read as one float4 a thread: a broadcast)
template <int D>
__device__ __forceinline__ void tile_apply_t(const float* S, int lds, const float* Z, int n, int ty, int tx,
                                             float (&out)[4][D / 16]) {
  constexpr int LD = D + 4, U = D / 64;
#pragma unroll 4
  for (int t = 0; t < n; ++t) {
    const float4 s = *reinterpret_cast<const float4*>(S + t * lds + 4 * ty);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const float4 z = *reinterpret_cast<const float4*>(Z + t * LD + 4 * tx + 64 * u);
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const float w = elem(s, a);
        out[a][4 * u + 0] = fmaf(w, z.x, out[a][4 * u + 0]);
        out[a][4 * u + 1] = fmaf(w, z.y, out[a][4 * u + 1]);
        out[a][4 * u + 2] = fmaf(w, z.z, out[a][4 * u + 2]);
        out[a][4 * u + 3] = fmaf(w, z.w, out[a][4 * u + 3]);
      }
    }
  }
}

constexpr int kTSL = kTR + 4;   // row stride of the stored-tile slices (floats)
}  // namespace
}  // namespace lion
