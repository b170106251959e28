// lion_simt.cu -- CUDA-core kernels for the three forms of the LION operator.
//
// These are the general kernels: every head dimension d in {16,32,64,128},
// bfloat16 or float32 inputs, float32 arithmetic throughout.  They carry the
// FP32 path (whose tolerance the tensor-core path cannot meet) and every
// shape the tensor-core chunk kernel does not take.
//
// Forms (rebuttal page "LION: A bidirectional framework that trains like a
// Transformer and infers like an RNN"):
//   full_simt_kernel   Theorem 3.3 Eq 25, Y = SCALE(QK^T (.) M) V, with the
//                      mask value generated per (i, j) -- never stored.
//   (the recurrent form, Theorem 3.3 Eq 20-24, is in lion_rnn.cu)
//   chunk_simt_kernel  chunkwise form ("LION Part IV - Results", "LION
//                      Chunk"): a right-to-left sweep applies the backward
//                      chunk state, then a left-to-right sweep adds the
//                      intra-chunk masked attention and the forward state.
// With Problem::causal each computes the forward half alone, y_i =
// sum_{j<=i} M_ij s_ij v_j / sum_{j<=i} M_ij s_ij: the causal recurrence of the
// Linear Transformer with the decay (rebuttal page reply "1: Recurrence Form";
// the unidirectional LION-S of reply "Q5").
#include "lion_common.cuh"
#include "lion_internal.h"

namespace lion {
namespace {

template <typename T>
__device__ __forceinline__ const T* head_ptr(const void* base, int bh, int L, int D) {
  return reinterpret_cast<const T*>(base) + (size_t)bh * L * D;
}

// Inclusive prefix sum of a[0..n) in shared memory; whole block.
__device__ void block_inclusive_scan(float* a, int n, float* scratch /*[32]*/) {
  const int T = blockDim.x, t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int per = (n + T - 1) / T;
  const int lo = min(n, t * per), hi = min(n, lo + per);
  float run = 0.f;
  for (int i = lo; i < hi; ++i) { run += a[i]; a[i] = run; }
  float x = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    float y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    const int nw = T >> 5;
    float w = lane < nw ? scratch[lane] : 0.f;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      float y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    scratch[lane] = w;
  }
  __syncthreads();
  const float excl = x - run + (warp > 0 ? scratch[warp - 1] : 0.f);
  for (int i = lo; i < hi; ++i) a[i] += excl;
  __syncthreads();
}

template <typename T>
__device__ void load_rows(float* dst, int ld, const T* src, int row0, int rows, int L, int D) {
  for (int idx = threadIdx.x; idx < rows * D; idx += blockDim.x) {
    const int r = idx / D, m = idx - r * D, i = row0 + r;
    dst[r * ld + m] = i < L ? to_f32(src[(size_t)i * D + m]) : 0.f;
  }
}

// ------------------------------------------------------------------ FULL --
constexpr int kFullRows = 32;   // query rows per CTA
constexpr int kFullGroup = 8;   // threads per query row
constexpr int kFullTile = 32;   // key tokens per shared-memory tile

template <typename T, int D>
__global__ void __launch_bounds__(256) full_simt_kernel(Problem p) {
  constexpr int LDQ = D + 8;
  constexpr int NC = D / kFullGroup;
  extern __shared__ float smem[];
  float* sQ = smem;                          // [kFullRows][LDQ]
  float* sK = sQ + kFullRows * LDQ;          // [kFullTile][D]
  float* sV = sK + kFullTile * D;            // [kFullTile][D]
  float* sP = sV + kFullTile * D;            // [L] prefix of log lambda (LION-S)
  __shared__ float scratch[32];

  const int L = p.L, H = p.H, bh = blockIdx.x, h = bh % H;
  const int i0 = blockIdx.y * kFullRows;
  const T* q = head_ptr<T>(p.q, bh, L, D);
  const T* k = head_ptr<T>(p.k, bh, L, D);
  const T* v = head_ptr<T>(p.v, bh, L, D);
  float lh = 0.f;
  if (p.mask_kind == MASK_S) {
    for (int t = threadIdx.x; t < L; t += blockDim.x) sP[t] = p.log_lambda[(size_t)bh * L + t];
    __syncthreads();
    block_inclusive_scan(sP, L, scratch);
  } else if (p.mask_kind == MASK_D) {
    lh = p.log_lambda[h];
  }
  load_rows<T>(sQ, LDQ, q, i0, kFullRows, L, D);
  __syncthreads();
  phi_rows_inplace(sQ, kFullRows, min(kFullRows, L - i0), D, LDQ, p.phi);
  __syncthreads();

  const int r = threadIdx.x / kFullGroup, g = threadIdx.x % kFullGroup, i = i0 + r;
  const float Pi = (p.mask_kind == MASK_S && i < L) ? sP[i] : 0.f;
  float acc[NC];
#pragma unroll
  for (int c = 0; c < NC; ++c) acc[c] = 0.f;
  float den = 0.f;
  const int jend = p.causal ? min(L, i0 + kFullRows) : L;   // causal: keys up to the block's last row
  for (int j0 = 0; j0 < jend; j0 += kFullTile) {
    const int nj = min(kFullTile, L - j0);
    load_rows<T>(sK, D, k, j0, kFullTile, L, D);
    load_rows<T>(sV, D, v, j0, kFullTile, L, D);
    __syncthreads();
    phi_rows_inplace(sK, kFullTile, nj, D, D, p.phi);
    __syncthreads();
    for (int jj = 0; jj < nj; ++jj) {
      float s = 0.f;
#pragma unroll
      for (int c = 0; c < NC; ++c) s += sQ[r * LDQ + g + c * kFullGroup] * sK[jj * D + g + c * kFullGroup];
      s += __shfl_xor_sync(0xffffffffu, s, 1);
      s += __shfl_xor_sync(0xffffffffu, s, 2);
      s += __shfl_xor_sync(0xffffffffu, s, 4);
      const int j = j0 + jj;
      float w = (p.causal && j > i) ? 0.f : s;
      if (p.mask_kind == MASK_D) w *= expf(fabsf((float)(i - j)) * lh);
      else if (p.mask_kind == MASK_S) w *= expf(mask_exponent(i, j, Pi, sP[j]));
      den += w;
#pragma unroll
      for (int c = 0; c < NC; ++c) acc[c] += w * sV[jj * D + g + c * kFullGroup];
    }
    __syncthreads();
  }
  if (i < L) {
    float* out = p.out + ((size_t)bh * L + i) * D;
    const float inv = 1.f / den;
#pragma unroll
    for (int c = 0; c < NC; ++c) out[g + c * kFullGroup] = acc[c] * inv;
  }
}

// ----------------------------------------------------------------- CHUNK --
constexpr int kPanel = 32;      // tokens per shared-memory panel

template <typename T, int D>
__global__ void __launch_bounds__(256) chunk_simt_kernel(Problem p, float* den_all) {
  constexpr int W = D + 1;          // value columns + normaliser column
  constexpr int LDQ = D + 8;
  extern __shared__ float smem[];
  float* sQ = smem;                      // [kPanel][LDQ]  phi(q) of a query panel
  float* sK = sQ + kPanel * LDQ;         // [kPanel][D]    phi(k) of a key panel
  float* sV = sK + kPanel * D;           // [kPanel][D]
  float* sS = sV + kPanel * D;           // [kPanel][kPanel+1] masked scores
  float* sAcc = sS + kPanel * (kPanel + 1);  // [kPanel][W]
  float* sSt = sAcc + kPanel * W;        // [D][W] chunk state (F or G)
  float* sW = sSt + D * W;               // [kPanel] per-token state weights
  float* sPc = sW + kPanel;              // [chunk] chunk-local inclusive prefix
  __shared__ float scratch[32];

  const int L = p.L, H = p.H, C = p.chunk, bh = blockIdx.x, h = bh % H;
  const int N = (L + C - 1) / C;
  const T* q = head_ptr<T>(p.q, bh, L, D);
  const T* k = head_ptr<T>(p.k, bh, L, D);
  const T* v = head_ptr<T>(p.v, bh, L, D);
  float* out = p.out + (size_t)bh * L * D;
  float* den = den_all + (size_t)bh * L;
  const float* ll = p.mask_kind == MASK_S ? p.log_lambda + (size_t)bh * L : nullptr;
  const float lh = p.mask_kind == MASK_D ? p.log_lambda[h] : 0.f;
  auto ell = [&](int t) -> float { return p.mask_kind == MASK_S ? ll[t] : lh; };

  for (int sweep = p.causal ? 1 : 0; sweep < 2; ++sweep) {
    const bool fwd = sweep == 1;
    for (int x = threadIdx.x; x < D * W; x += blockDim.x) sSt[x] = 0.f;
    __syncthreads();
    for (int cc = 0; cc < N; ++cc) {
      const int c = fwd ? cc : N - 1 - cc;
      const int s = c * C, e = min(L, s + C) - 1, len = e - s + 1;
      // chunk-local inclusive prefix p_t = sum_{u=s}^{s+t} l_u
      if (p.mask_kind == MASK_S) {
        for (int t = threadIdx.x; t < len; t += blockDim.x) sPc[t] = ll[s + t];
        __syncthreads();
        block_inclusive_scan(sPc, len, scratch);
      } else {
        for (int t = threadIdx.x; t < len; t += blockDim.x) sPc[t] = (float)(t + 1) * lh;
        __syncthreads();
      }
      const float lnext = (e + 1 < L) ? ell(e + 1) : 0.f;   // l at s_{c+1}
      const bool has_state = fwd ? (c > 0) : (c < N - 1);

      // ---- rows of this chunk, one query panel at a time
      for (int qa = s; qa <= e; qa += kPanel) {
        const int nq = min(kPanel, e + 1 - qa);
        load_rows<T>(sQ, LDQ, q, qa, kPanel, e + 1, D);
        __syncthreads();
        phi_rows_inplace(sQ, kPanel, nq, D, LDQ, p.phi);
        __syncthreads();
        for (int idx = threadIdx.x; idx < kPanel * W; idx += blockDim.x) {
          const int r = idx / W, n = idx - r * W;
          float a = 0.f;
          if (has_state && r < nq) {
            const int i = qa + r;
            // forward: exp(P_i - P_{e_{c-1}}); backward: exp(P_{s_{c+1}} - P_i)
            const float sc = fwd ? expf(sPc[i - s]) : expf(sPc[len - 1] - sPc[i - s] + lnext);
            float dot = 0.f;
            for (int m = 0; m < D; ++m) dot += sQ[r * LDQ + m] * sSt[m * W + n];
            a = sc * dot;
          }
          sAcc[idx] = a;
        }
        __syncthreads();
        if (fwd) {
          // intra-chunk masked attention, both triangles, diagonal once
          for (int ka = s; ka <= e; ka += kPanel) {
            const int nk = min(kPanel, e + 1 - ka);
            load_rows<T>(sK, D, k, ka, kPanel, e + 1, D);
            load_rows<T>(sV, D, v, ka, kPanel, e + 1, D);
            __syncthreads();
            phi_rows_inplace(sK, kPanel, nk, D, D, p.phi);
            __syncthreads();
            for (int idx = threadIdx.x; idx < kPanel * kPanel; idx += blockDim.x) {
              const int r = idx / kPanel, jj = idx - r * kPanel;
              float w = 0.f;
              if (r < nq && jj < nk && (!p.causal || ka + jj <= qa + r)) {
                const int i = qa + r, j = ka + jj;
                float dot = 0.f;
                for (int m = 0; m < D; ++m) dot += sQ[r * LDQ + m] * sK[jj * D + m];
                w = dot * expf(mask_exponent(i, j, sPc[i - s], sPc[j - s]));
              }
              sS[r * (kPanel + 1) + jj] = w;
            }
            __syncthreads();
            for (int idx = threadIdx.x; idx < kPanel * W; idx += blockDim.x) {
              const int r = idx / W, n = idx - r * W;
              float a = 0.f;
              for (int jj = 0; jj < nk; ++jj)
                a += sS[r * (kPanel + 1) + jj] * (n < D ? sV[jj * D + n] : 1.f);
              sAcc[idx] += a;
            }
            __syncthreads();
          }
        }
        // write: backward sweep parks its partial sums, forward sweep finishes
        for (int idx = threadIdx.x; idx < nq * W; idx += blockDim.x) {
          const int r = idx / W, n = idx - r * W, i = qa + r;
          if (!fwd) {
            if (n < D) out[(size_t)i * D + n] = sAcc[idx];
            else den[i] = sAcc[idx];
          }
        }
        if (fwd) {
          __syncthreads();
          for (int idx = threadIdx.x; idx < nq * D; idx += blockDim.x) {
            const int r = idx / D, n = idx - r * D, i = qa + r;
            // (causal: no backward sweep parked anything)
            const float dn = sAcc[r * W + D] + (p.causal ? 0.f : den[i]);
            out[(size_t)i * D + n] = (sAcc[r * W + n] + (p.causal ? 0.f : out[(size_t)i * D + n])) / dn;
          }
        }
        __syncthreads();
      }

      // ---- carry the state across this chunk
      // forward:  F_{c+1} = exp(T_c) F_c + sum_j exp(P_{e_c} - P_j) phi(k_j)[v_j;1]^T
      // backward: G_{c-1} = exp(P_{s_{c+1}} - P_{s_c}) G_c + sum_j exp(P_j - P_{s_c}) phi(k_j)[v_j;1]^T
      const float decay = fwd ? expf(sPc[len - 1]) : expf(sPc[len - 1] - sPc[0] + lnext);
      for (int x = threadIdx.x; x < D * W; x += blockDim.x) sSt[x] *= decay;
      __syncthreads();
      for (int ka = s; ka <= e; ka += kPanel) {
        const int nk = min(kPanel, e + 1 - ka);
        load_rows<T>(sK, D, k, ka, kPanel, e + 1, D);
        load_rows<T>(sV, D, v, ka, kPanel, e + 1, D);
        for (int jj = threadIdx.x; jj < kPanel; jj += blockDim.x) {
          float w = 0.f;
          if (jj < nk) {
            const int t = ka + jj - s;
            w = fwd ? expf(sPc[len - 1] - sPc[t]) : expf(sPc[t] - sPc[0]);
          }
          sW[jj] = w;
        }
        __syncthreads();
        phi_rows_inplace(sK, kPanel, nk, D, D, p.phi);
        __syncthreads();
        for (int x = threadIdx.x; x < D * W; x += blockDim.x) {
          const int m = x / W, n = x - m * W;
          float a = 0.f;
          for (int jj = 0; jj < nk; ++jj)
            a += sW[jj] * sK[jj * D + m] * (n < D ? sV[jj * D + n] : 1.f);
          sSt[x] += a;
        }
        __syncthreads();
      }
    }
  }
}

// ------------------------------------------------------------ RNN step --
// One token of one direction for every head: a CTA per head, the state read
// and written as float4 rows (four value columns a thread, the head's rows
// split over the rest of the CTA), so that each row of S moves as whole
// coalesced segments; the column sums of phi(q) . S are reduced through
// shared memory.
constexpr int kStepThreads = 256;

template <int D>
struct StepCfg {
  static constexpr int CG = D / 4;                                   // float4 column groups
  static constexpr int RG = kStepThreads / CG < D ? kStepThreads / CG : D;   // row groups
  static constexpr int RPT = D / RG;                                 // rows per thread
};

template <typename T, int D>
__global__ void __launch_bounds__(kStepThreads) rnn_step_kernel(
    const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
    const float* __restrict__ log_lambda, float* __restrict__ S, float* __restrict__ z,
    float* __restrict__ y_part, float* __restrict__ c_part, int H, int mask_kind, int phi) {
  using C = StepCfg<D>;
  __shared__ float sQ[D], sK[D], sV[D];
  __shared__ __align__(16) float red[C::RG][D];
  const int bh = blockIdx.x, h = bh % H, t = threadIdx.x;
  for (int m = t; m < D; m += blockDim.x) {
    sQ[m] = to_f32(q[(size_t)bh * D + m]);
    sK[m] = to_f32(k[(size_t)bh * D + m]);
    sV[m] = to_f32(v[(size_t)bh * D + m]);
  }
  __syncthreads();
  if (t < 32) {
    phi_rows_inplace(sQ, 1, 1, D, D, phi);   // warp 0 only: one row each
    phi_rows_inplace(sK, 1, 1, D, D, phi);
  }
  __syncthreads();
  float l = 0.f;
  if (mask_kind == MASK_D) l = log_lambda[h];
  else if (mask_kind == MASK_S) l = log_lambda[bh];
  const float lam = expf(l);
  float* Sh = S + (size_t)bh * D * D;
  const int cg = t % C::CG, rg = t / C::CG, n0 = 4 * cg;
  if (rg < C::RG) {
    const float4 v4 = *reinterpret_cast<const float4*>(sV + n0);
    float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int a = 0; a < C::RPT; ++a) {
      const int m = rg + C::RG * a;
      float4* row = reinterpret_cast<float4*>(Sh + (size_t)m * D + n0);
      float4 s4 = *row;
      const float km = sK[m], qm = sQ[m];
      s4.x = fmaf(lam, s4.x, km * v4.x);
      s4.y = fmaf(lam, s4.y, km * v4.y);
      s4.z = fmaf(lam, s4.z, km * v4.z);
      s4.w = fmaf(lam, s4.w, km * v4.w);
      *row = s4;
      y.x = fmaf(qm, s4.x, y.x);
      y.y = fmaf(qm, s4.y, y.y);
      y.z = fmaf(qm, s4.z, y.z);
      y.w = fmaf(qm, s4.w, y.w);
    }
    *reinterpret_cast<float4*>(&red[rg][n0]) = y;
  }
  // z and its dot product: one thread a row
  float c = 0.f;
  if (t < D) {
    float* zh = z + (size_t)bh * D;
    const float z_new = lam * zh[t] + sK[t];
    zh[t] = z_new;
    c = sQ[t] * z_new;
  }
  __syncthreads();
  if (t < D) {
    float y = 0.f;
#pragma unroll 8
    for (int r = 0; r < C::RG; ++r) y += red[r][t];
    y_part[(size_t)bh * D + t] = y;
  }
  // c = phi(q) . z: the first D threads hold the terms (whole warps, at most four)
  __shared__ float cw[4];
  if (t < 32 * ((D + 31) / 32)) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    if ((t & 31) == 0) cw[t >> 5] = c;
  }
  __syncthreads();
  if (t == 0) {
    float cs = 0.f;
#pragma unroll
    for (int w = 0; w < (D + 31) / 32; ++w) cs += cw[w];
    c_part[bh] = cs;
  }
}

// ------------------------------------------------------------ launchers --
template <typename Kern>
cudaError_t allow_smem(Kern kern, size_t bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <typename T, int D>
cudaError_t full_launch(const Problem& p, cudaStream_t s) {
  size_t smem = sizeof(float) * ((size_t)kFullRows * (D + 8) + 2 * kFullTile * D +
                                 (p.mask_kind == MASK_S ? p.L : 0));
  auto kern = full_simt_kernel<T, D>;
  cudaError_t e = allow_smem(kern, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.B * p.H, (p.L + kFullRows - 1) / kFullRows);
  kern<<<grid, 256, smem, s>>>(p);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t chunk_launch(const Problem& p, float* ws, cudaStream_t s) {
  constexpr int W = D + 1;
  size_t smem = sizeof(float) * ((size_t)kPanel * (D + 8) + 2 * kPanel * D + kPanel * (kPanel + 1) +
                                 kPanel * W + (size_t)D * W + kPanel + p.chunk);
  auto kern = chunk_simt_kernel<T, D>;
  cudaError_t e = allow_smem(kern, smem);
  if (e != cudaSuccess) return e;
  kern<<<p.B * p.H, 256, smem, s>>>(p, ws);
  return cudaGetLastError();
}

template <template <typename, int> class F, typename... A>
cudaError_t dispatch(const Problem& p, A... args) {
  const bool bf = p.dtype == DT_BF16;
  switch (p.d) {
    case 16: return bf ? F<__nv_bfloat16, 16>::run(p, args...) : F<float, 16>::run(p, args...);
    case 32: return bf ? F<__nv_bfloat16, 32>::run(p, args...) : F<float, 32>::run(p, args...);
    case 64: return bf ? F<__nv_bfloat16, 64>::run(p, args...) : F<float, 64>::run(p, args...);
    case 128: return bf ? F<__nv_bfloat16, 128>::run(p, args...) : F<float, 128>::run(p, args...);
  }
  return cudaErrorInvalidValue;
}

template <typename T, int D> struct FullF {
  static cudaError_t run(const Problem& p, cudaStream_t s) { return full_launch<T, D>(p, s); }
};
template <typename T, int D> struct ChunkF {
  static cudaError_t run(const Problem& p, float* ws, cudaStream_t s) { return chunk_launch<T, D>(p, ws, s); }
};

template <typename T, int D>
cudaError_t step_launch(const void* q, const void* k, const void* v, const float* ll, float* S,
                        float* z, float* y, float* c, int B, int H, int mask_kind, int phi,
                        cudaStream_t s) {
  rnn_step_kernel<T, D><<<B * H, kStepThreads, 0, s>>>(
      (const T*)q, (const T*)k, (const T*)v, ll, S, z, y, c, H, mask_kind, phi);
  return cudaGetLastError();
}

}  // namespace

namespace {
// fp32 -> bfloat16, round to nearest even, four values a thread
__global__ void __launch_bounds__(256) f32_to_bf16_kernel(const float* src, __nv_bfloat16* dst, size_t n) {
  const size_t i = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (i + 4 <= n) {
    const float4 v = *reinterpret_cast<const float4*>(src + i);
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&lo);
    u.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(dst + i) = u;
  } else {
    for (size_t t = i; t < n; ++t) dst[t] = __float2bfloat16_rn(src[t]);
  }
}
}  // namespace

cudaError_t launch_f32_to_bf16(const float* src, void* dst, size_t n, cudaStream_t s) {
  const size_t threads = (n + 3) / 4;
  f32_to_bf16_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, s>>>(src, static_cast<__nv_bfloat16*>(dst), n);
  return cudaGetLastError();
}

cudaError_t launch_full_simt(const Problem& p, cudaStream_t s) { return dispatch<FullF>(p, s); }
cudaError_t launch_chunk_simt(const Problem& p, float* ws, cudaStream_t s) { return dispatch<ChunkF>(p, ws, s); }

cudaError_t launch_rnn_step(const void* q, const void* k, const void* v, const float* ll,
                            float* S, float* z, float* y, float* c, int B, int H, int d,
                            int mask_kind, int phi, int dtype, cudaStream_t s) {
  const bool bf = dtype == DT_BF16;
#define LION_STEP(D)                                                                   \
  return bf ? step_launch<__nv_bfloat16, D>(q, k, v, ll, S, z, y, c, B, H, mask_kind, phi, s) \
            : step_launch<float, D>(q, k, v, ll, S, z, y, c, B, H, mask_kind, phi, s)
  switch (d) {
    case 16: LION_STEP(16);
    case 32: LION_STEP(32);
    case 64: LION_STEP(64);
    case 128: LION_STEP(128);
  }
#undef LION_STEP
  return cudaErrorInvalidValue;
}

}  // namespace lion
