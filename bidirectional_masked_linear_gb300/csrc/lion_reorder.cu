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
//
// Gradients (lion_attn_bwd_reordered): the products are those of the
// full-form backward with the averaged mask; for the decays, with
// e_ij = s_ij dA_ij = dLoss/dM_ij, the coordinate gradient along order p is
//   dLoss/dC^p_a = -(1/2) sum_b sgn(pos_p(b) - pos_p(a)) M^p_ab (e_ab + e_ba)
// (LION-S), split into a row part R^p_a (the pairs with a as query, summed
// by the rows pass) and a column part K^p_a (a as key, the columns pass);
// dlog(lambda_u) is the suffix sum of these along each order from u's
// position, over both orders.  LION-D: dLoss/dlog(lambda_h) =
// sum_ij e_ij (1/2) sum_p |pos_p(i) - pos_p(j)| M^p_ij, over the batch too.
// Up to kRbwdStoreMaxL tokens the rows pass keeps s_ij and dA_ij and the
// columns pass reads them; longer sequences recompute the scores there.
#include <string.h>

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
  int B, H, L, mask_kind, phi;
  int causal;         // 1: keys j <= i only (the natural order's forward half)
  float* fq;          // [BH][L][D] phi(q)
  float* fk;          // [BH][L][D] phi(k)
  int* pos;           // [2][L]     position of each token in each order
  float* coord;       // LION-S [2][BH][L] prefixes; LION-D [2][L] positions
  int* status;
  // gradients
  const float* dy;    // [BH][L][D]
  float* dq;
  float* dk;
  float* dv;
  float* dll;         // LION-D [H]; LION-S [BH][L]
  float* g;           // [BH][L][D] dnum
  float* hd;          // [BH][L]    dden
  float* R;           // [2][BH][L] row terms per order (LION-S)
  float* K;           // [2][BH][L] column terms per order (LION-S)
  float* dterm;       // [BH][L]    LION-D: each row's share of dLoss/dlog(lambda)
  double* dsum;       // [BH]       LION-D: per head
  // stored-tile build (L <= kRbwdStoreMaxL): s_ij and dA_ij, [BH][L (i)][LP (j)]
  float* St;
  float* Dt;
  int LP;
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

// (2) LION-S: grid (B*H, orders), kScanThreads threads.  Without an order
// array (the plain full form) the order is the tokens' own.
__global__ void __launch_bounds__(kScanThreads) order_prefix_kernel(ReorderParams p) {
  const int L = p.L, bh = blockIdx.x, o = blockIdx.y, t0 = threadIdx.x;
  const int* ord = p.order ? p.order + (size_t)o * L : nullptr;
  const float* ll = p.log_lambda + (size_t)bh * L;
  float* C = p.coord + ((size_t)o * gridDim.x + bh) * L;
  const int per = (L + kScanThreads - 1) / kScanThreads;
  const int lo = min(L, t0 * per), hi = min(L, lo + per);
  double run = 0.0, all;
  for (int t = lo; t < hi; ++t) run += (double)ll[ord ? clamp_token(ord[t], L) : t];
  double off = block_scan(run, &all) - run;
  for (int t = lo; t < hi; ++t) {
    const int a = ord ? clamp_token(ord[t], L) : t;
    off += (double)ll[a];
    C[a] = (float)off;
  }
}

template <int D>
constexpr size_t reorder_smem() {
  return sizeof(float) * ((size_t)(kTR + 2 * kTC) * (D + 4) + kTR * kTAL + 2 * kTC);
}

// (4) 32 queries per CTA.  NORD = 2: the mask averaged over the two orders;
// NORD = 1: the plain full form, the tokens' own order (LION-D's coordinate
// is then the token index itself), with p.causal keeping the keys j <= i.
template <typename T, int D, int NORD>
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
  } else if (p.mask_kind == MASK_D && NORD == 2) {
    C0 = p.coord;
    C1 = p.coord + L;
  }
  const bool index_coord = NORD == 1 && p.mask_kind == MASK_D;
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
    c0[a] = index_coord ? (float)ia[a] : !lit && live[a] ? C0[ia[a]] : 0.f;
    c1[a] = NORD == 2 && !lit && live[a] ? C1[ia[a]] : 0.f;
  }
  float den[4], num[4][MF];
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    den[a] = 0.f;
#pragma unroll
    for (int f = 0; f < MF; ++f) num[a][f] = 0.f;
  }
  const int jend = p.causal ? min(L, i0 + kTR) : L;   // causal: keys up to the block's last row
  for (int j0 = 0; j0 < jend; j0 += kTC) {
    stage_rows<D>(sK, fkh, j0, kTC, L);
    stage_rows<D>(sV, vh, j0, kTC, L);
    if (!lit && !index_coord) {
      stage_vec(sC, C0, j0, kTC, L);
      if (NORD == 2) stage_vec(sC + kTC, C1, j0, kTC, L);
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
        if (live[a] && j < L && (!p.causal || j <= ia[a])) {
          if (lit) m = 1.f;
          else if (NORD == 1) m = expf(-fabsf(c0[a] - (index_coord ? (float)j : sC[jl])) * w);
          else m = 0.5f * (expf(-fabsf(c0[a] - sC[jl]) * w) + expf(-fabsf(c1[a] - sC[kTC + jl]) * w));
        }
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

// ------------------------------------------------------------ gradients --
__device__ __forceinline__ void stage_pos(float* dst, const int* pos, int j0, int n, int L) {
  for (int t = threadIdx.x; t < n; t += blockDim.x) dst[t] = j0 + t < L ? (float)pos[j0 + t] : 0.f;
}
__device__ __forceinline__ float sgnf(float x) { return x > 0.f ? 1.f : x < 0.f ? -1.f : 0.f; }

template <int D>
constexpr size_t rbwd_rows_smem() {
  return sizeof(float) * ((size_t)(2 * kTR + 2 * kTC) * (D + 4) + kTR * kTAL + 4 * kTC);
}
template <int D>
constexpr size_t rbwd_cols_smem() {
  return sizeof(float) * ((size_t)(2 * kTR + 2 * kTC) * (D + 4) + 2 * kTR * kTAL + 5 * kTC);
}

// Rows: 32 queries per CTA.  Pass A: den, num; then y, dnum, dden; pass B:
// dphi(q) and the decay terms of each row.
template <typename T, int D, bool STORE>
__global__ void __launch_bounds__(kTThreads) rbwd_rows_kernel(ReorderParams p) {
  constexpr int LD = D + 4, MF = D / 16, U = D / 64;
  extern __shared__ __align__(16) float smem[];
  float* sQ = smem;                  // [kTR][LD]   phi(q) of the block
  float* sG = sQ + kTR * LD;         // [kTR][LD]   dnum of the block
  float* sK = sG + kTR * LD;         // [kTC][LD]   phi(k) of the tile
  float* sV = sK + kTC * LD;         // [kTC][LD]   v of the tile
  float* sA = sV + kTC * LD;         // [kTR][kTAL] A, then M (.) dA
  float* sC = sA + kTR * kTAL;       // [2][kTC]    coordinates of the tile's keys
  float* sPs = sC + 2 * kTC;         // [2][kTC]    their positions
  const int L = p.L, BH = gridDim.x, bh = blockIdx.x, h = bh % p.H, i0 = blockIdx.y * kTR;
  const int nr = min(kTR, L - i0);
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const bool lit = p.mask_kind == MASK_LIT, ms = p.mask_kind == MASK_S;
  const float w = p.mask_kind == MASK_D ? -p.log_lambda[h] : 1.f;
  const float* C0 = ms ? p.coord + (size_t)bh * L : p.coord;
  const float* C1 = ms ? p.coord + ((size_t)BH + bh) * L : p.coord + L;
  const int* P0 = p.pos;
  const int* P1 = p.pos + L;
  const float* fkh = p.fk + (size_t)bh * L * D;
  const T* vh = head_of<T>(p.v, bh, L, D);
  float* St = STORE ? p.St + (size_t)bh * L * p.LP : nullptr;
  float* Dt = STORE ? p.Dt + (size_t)bh * L * p.LP : nullptr;
  stage_rows<D>(sQ, p.fq + (size_t)bh * L * D, i0, kTR, L);
  int ia[4];
  bool live[4];
  float c0[4], c1[4], q0[4], q1[4];
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    ia[a] = i0 + ty + 8 * a;
    live[a] = ia[a] < L;
    c0[a] = !lit && live[a] ? C0[ia[a]] : 0.f;
    c1[a] = !lit && live[a] ? C1[ia[a]] : 0.f;
    q0[a] = !lit && live[a] ? (float)P0[ia[a]] : 0.f;
    q1[a] = !lit && live[a] ? (float)P1[ia[a]] : 0.f;
  }
  auto stage_tile = [&](int j0) {
    stage_rows<D>(sK, fkh, j0, kTC, L);
    stage_rows<D>(sV, vh, j0, kTC, L);
    if (!lit) {
      stage_vec(sC, C0, j0, kTC, L);
      stage_vec(sC + kTC, C1, j0, kTC, L);
      stage_pos(sPs, P0, j0, kTC, L);
      stage_pos(sPs + kTC, P1, j0, kTC, L);
    }
  };
  // ---- pass A
  float den[4], num[4][MF];
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    den[a] = 0.f;
#pragma unroll
    for (int f = 0; f < MF; ++f) num[a][f] = 0.f;
  }
  for (int j0 = 0; j0 < L; j0 += kTC) {
    stage_tile(j0);
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
        if (STORE && live[a] && j < L) St[(size_t)ia[a] * p.LP + j] = s[a][b];
      }
    __syncthreads();
    tile_apply<D>(sA, sV, (nc + 3) & ~3, ty, tx, nr, num);
    __syncthreads();
  }
  // ---- y_i, dnum_i = dy_i / den_i, dden_i = -(dy_i . y_i) / den_i
  float hi[4];
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const float dn = group_sum<16>(den[a]);
    const float* dyr = p.dy + ((size_t)bh * L + (live[a] ? ia[a] : 0)) * D;
    float dyy = 0.f, gi[MF];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const float4 d4 = live[a] ? load4(dyr + 4 * tx + 64 * u) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float dd = elem(d4, e);
        dyy += dd * (num[a][4 * u + e] / dn);
        gi[4 * u + e] = live[a] ? dd / dn : 0.f;
      }
    }
    dyy = group_sum<16>(dyy);
    hi[a] = live[a] ? -dyy / dn : 0.f;
    float* gs = sG + (ty + 8 * a) * LD;
    float* gw = p.g + ((size_t)bh * L + (live[a] ? ia[a] : 0)) * D;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const float4 g4 = make_float4(gi[4 * u], gi[4 * u + 1], gi[4 * u + 2], gi[4 * u + 3]);
      *reinterpret_cast<float4*>(gs + 4 * tx + 64 * u) = g4;
      if (live[a]) *reinterpret_cast<float4*>(gw + 4 * tx + 64 * u) = g4;
    }
    if (live[a] && tx == 0) p.hd[(size_t)bh * L + ia[a]] = hi[a];
  }
  // ---- pass B
  float dfq[4][MF], r0[4], r1[4];
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    r0[a] = r1[a] = 0.f;
#pragma unroll
    for (int f = 0; f < MF; ++f) dfq[a][f] = 0.f;
  }
  for (int j0 = 0; j0 < L; j0 += kTC) {
    float s[4][4], gv[4][4];
    if (STORE) {   // s_ij as this thread wrote it in pass A
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const int j = j0 + tx + 16 * b;
          s[a][b] = live[a] && j < L ? St[(size_t)ia[a] * p.LP + j] : 0.f;
        }
    }
    stage_tile(j0);
    __syncthreads();
    const int nc = min(kTC, L - j0);
    if (!STORE) tile_scores<D>(sQ, sK, ty, tx, nr, nc, s);
    tile_scores<D>(sG, sV, ty, tx, nr, nc, gv);
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int jl = tx + 16 * b, j = j0 + jl;
        const bool ok = live[a] && j < L;
        float m0 = 0.f, m1 = 0.f;
        if (ok && !lit) {
          m0 = expf(-fabsf(c0[a] - sC[jl]) * w);
          m1 = expf(-fabsf(c1[a] - sC[kTC + jl]) * w);
        }
        const float m = !ok ? 0.f : lit ? 1.f : 0.5f * (m0 + m1);
        const float da = gv[a][b] + hi[a], e = s[a][b] * da;
        sA[(ty + 8 * a) * kTAL + jl] = m * da;
        if (STORE && ok) Dt[(size_t)ia[a] * p.LP + j] = da;
        if (ms) {
          r0[a] += sgnf(sPs[jl] - q0[a]) * m0 * e;
          r1[a] += sgnf(sPs[kTC + jl] - q1[a]) * m1 * e;
        } else if (!lit) {
          r0[a] += 0.5f * (fabsf(sPs[jl] - q0[a]) * m0 + fabsf(sPs[kTC + jl] - q1[a]) * m1) * e;
        }
      }
    __syncthreads();
    tile_apply<D>(sA, sK, (nc + 3) & ~3, ty, tx, nr, dfq);
    __syncthreads();
  }
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const float t0 = group_sum<16>(r0[a]), t1 = group_sum<16>(r1[a]);
    const T* qr = head_of<T>(p.q, bh, L, D) + (size_t)(live[a] ? ia[a] : L - 1) * D;
    float x[MF], dx[MF];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const float4 x4 = load4(qr + 4 * tx + 64 * u);
#pragma unroll
      for (int e = 0; e < 4; ++e) x[4 * u + e] = elem(x4, e);
    }
    phi_backward<MF, 16>(p.phi, x, dfq[a], dx);
    if (live[a]) {
      float* dq = p.dq + ((size_t)bh * L + ia[a]) * D;
#pragma unroll
      for (int u = 0; u < U; ++u)
        *reinterpret_cast<float4*>(dq + 4 * tx + 64 * u) =
            make_float4(dx[4 * u], dx[4 * u + 1], dx[4 * u + 2], dx[4 * u + 3]);
      if (tx == 0 && ms) {
        p.R[(size_t)bh * L + ia[a]] = t0;
        p.R[((size_t)BH + bh) * L + ia[a]] = t1;
      } else if (tx == 0 && !lit) {
        p.dterm[(size_t)bh * L + ia[a]] = t0;
      }
    }
  }
}

// Columns: 32 keys per CTA.  dphi(k_j) = sum_i M_ij dA_ij phi(q_i),
// dv_j = sum_i A_ij dnum_i, and the column part of each order's decay term.
template <typename T, int D>
__global__ void __launch_bounds__(kTThreads) rbwd_cols_kernel(ReorderParams p) {
  constexpr int LD = D + 4, MF = D / 16, U = D / 64;
  extern __shared__ __align__(16) float smem[];
  float* sK = smem;                  // [kTR][LD]   phi(k) of the block
  float* sVb = sK + kTR * LD;        // [kTR][LD]   v of the block
  float* sQ = sVb + kTR * LD;        // [kTC][LD]   phi(q) of the tile
  float* sG = sQ + kTC * LD;         // [kTC][LD]   dnum of the tile
  float* sA = sG + kTC * LD;         // [kTR][kTAL] A^T
  float* sD = sA + kTR * kTAL;       // [kTR][kTAL] (M (.) dA)^T
  float* sH = sD + kTR * kTAL;       // [kTC]       dden of the tile
  float* sC = sH + kTC;              // [2][kTC]    coordinates of the tile's queries
  float* sPs = sC + 2 * kTC;         // [2][kTC]    their positions
  const int L = p.L, BH = gridDim.x, bh = blockIdx.x, h = bh % p.H, j0b = blockIdx.y * kTR;
  const int nr = min(kTR, L - j0b);
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const bool lit = p.mask_kind == MASK_LIT, ms = p.mask_kind == MASK_S;
  const float w = p.mask_kind == MASK_D ? -p.log_lambda[h] : 1.f;
  const float* C0 = ms ? p.coord + (size_t)bh * L : p.coord;
  const float* C1 = ms ? p.coord + ((size_t)BH + bh) * L : p.coord + L;
  const int* P0 = p.pos;
  const int* P1 = p.pos + L;
  const float* fqh = p.fq + (size_t)bh * L * D;
  const float* gh = p.g + (size_t)bh * L * D;
  const float* hh = p.hd + (size_t)bh * L;
  stage_rows<D>(sK, p.fk + (size_t)bh * L * D, j0b, kTR, L);
  stage_rows<D>(sVb, head_of<T>(p.v, bh, L, D), j0b, kTR, L);
  int ja[4];
  bool live[4];
  float c0[4], c1[4], q0[4], q1[4];
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    ja[a] = j0b + ty + 8 * a;
    live[a] = ja[a] < L;
    c0[a] = !lit && live[a] ? C0[ja[a]] : 0.f;
    c1[a] = !lit && live[a] ? C1[ja[a]] : 0.f;
    q0[a] = !lit && live[a] ? (float)P0[ja[a]] : 0.f;
    q1[a] = !lit && live[a] ? (float)P1[ja[a]] : 0.f;
  }
  float dfk[4][MF], dvj[4][MF], k0[4], k1[4];
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    k0[a] = k1[a] = 0.f;
#pragma unroll
    for (int f = 0; f < MF; ++f) dfk[a][f] = dvj[a][f] = 0.f;
  }
  for (int i0 = 0; i0 < L; i0 += kTC) {
    stage_rows<D>(sQ, fqh, i0, kTC, L);
    stage_rows<D>(sG, gh, i0, kTC, L);
    stage_vec(sH, hh, i0, kTC, L);
    if (!lit) {
      stage_vec(sC, C0, i0, kTC, L);
      stage_vec(sC + kTC, C1, i0, kTC, L);
      stage_pos(sPs, P0, i0, kTC, L);
      stage_pos(sPs + kTC, P1, i0, kTC, L);
    }
    __syncthreads();
    const int nc = min(kTC, L - i0);
    float s[4][4], gv[4][4];
    tile_scores<D>(sK, sQ, ty, tx, nr, nc, s);
    tile_scores<D>(sVb, sG, ty, tx, nr, nc, gv);
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int il = tx + 16 * b, i = i0 + il;
        const bool ok = live[a] && i < L;
        float m0 = 0.f, m1 = 0.f;
        if (ok && !lit) {
          m0 = expf(-fabsf(c0[a] - sC[il]) * w);
          m1 = expf(-fabsf(c1[a] - sC[kTC + il]) * w);
        }
        const float m = !ok ? 0.f : lit ? 1.f : 0.5f * (m0 + m1);
        const float da = gv[a][b] + sH[il], e = s[a][b] * da;
        sA[(ty + 8 * a) * kTAL + il] = m * s[a][b];
        sD[(ty + 8 * a) * kTAL + il] = m * da;
        if (ms) {
          k0[a] += sgnf(sPs[il] - q0[a]) * m0 * e;
          k1[a] += sgnf(sPs[kTC + il] - q1[a]) * m1 * e;
        }
      }
    __syncthreads();
    const int n4 = (nc + 3) & ~3;
    tile_apply<D>(sD, sQ, n4, ty, tx, nr, dfk);
    tile_apply<D>(sA, sG, n4, ty, tx, nr, dvj);
    __syncthreads();
  }
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const float t0 = group_sum<16>(k0[a]), t1 = group_sum<16>(k1[a]);
    const T* kr = head_of<T>(p.k, bh, L, D) + (size_t)(live[a] ? ja[a] : L - 1) * D;
    float x[MF], dx[MF];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const float4 x4 = load4(kr + 4 * tx + 64 * u);
#pragma unroll
      for (int e = 0; e < 4; ++e) x[4 * u + e] = elem(x4, e);
    }
    phi_backward<MF, 16>(p.phi, x, dfk[a], dx);
    if (live[a]) {
      float* dk = p.dk + ((size_t)bh * L + ja[a]) * D;
      float* dv = p.dv + ((size_t)bh * L + ja[a]) * D;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        *reinterpret_cast<float4*>(dk + 4 * tx + 64 * u) =
            make_float4(dx[4 * u], dx[4 * u + 1], dx[4 * u + 2], dx[4 * u + 3]);
        *reinterpret_cast<float4*>(dv + 4 * tx + 64 * u) =
            make_float4(dvj[a][4 * u], dvj[a][4 * u + 1], dvj[a][4 * u + 2], dvj[a][4 * u + 3]);
      }
      if (tx == 0 && ms) {
        p.K[(size_t)bh * L + ja[a]] = t0;
        p.K[((size_t)BH + bh) * L + ja[a]] = t1;
      }
    }
  }
}

template <int D>
constexpr size_t rbwd_cols_stored_smem() {
  return sizeof(float) * ((size_t)2 * kTC * (D + 4) + 2 * kTC * kTSL + 4 * kTC + 2 * 4 * kTR);
}

// Columns from the stored s_ij and dA_ij: 32 keys per CTA.  Each tile is
// first turned into A = M (.) s and M (.) dA in place (thread: one key, 16 of
// the tile's queries, which also sums the key's column terms), then the two
// products run with each thread holding keys 4ty + a (tile_apply_t).
template <typename T, int D>
__global__ void __launch_bounds__(kTThreads) rbwd_cols_stored_kernel(ReorderParams p) {
  constexpr int LD = D + 4, MF = D / 16, U = D / 64, J4 = kTR / 4;
  extern __shared__ __align__(16) float smem[];
  float* sQ = smem;                  // [kTC][LD]   phi(q) of the tile
  float* sG = sQ + kTC * LD;         // [kTC][LD]   dnum of the tile
  float* sS = sG + kTC * LD;         // [kTC][kTSL] s, then A, over the tile's queries x the block's keys
  float* sE = sS + kTC * kTSL;       // [kTC][kTSL] dA, then M (.) dA
  float* sC = sE + kTC * kTSL;       // [2][kTC]    coordinates of the tile's queries
  float* sPs = sC + 2 * kTC;         // [2][kTC]    their positions
  float* sKp = sPs + 2 * kTC;        // [2][4][kTR] column terms per query group
  const int L = p.L, LP = p.LP, BH = gridDim.x, bh = blockIdx.x, h = bh % p.H, j0b = blockIdx.y * kTR;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int kj = threadIdx.x & 31, grp = threadIdx.x >> 5;   // conversion role: key, query group
  const bool lit = p.mask_kind == MASK_LIT, ms = p.mask_kind == MASK_S;
  const float w = p.mask_kind == MASK_D ? -p.log_lambda[h] : 1.f;
  const float* C0 = ms ? p.coord + (size_t)bh * L : p.coord;
  const float* C1 = ms ? p.coord + ((size_t)BH + bh) * L : p.coord + L;
  const int* P0 = p.pos;
  const int* P1 = p.pos + L;
  const float* fqh = p.fq + (size_t)bh * L * D;
  const float* gh = p.g + (size_t)bh * L * D;
  const float* St = p.St + (size_t)bh * L * LP;
  const float* Dt = p.Dt + (size_t)bh * L * LP;
  const int jk = j0b + kj;
  const bool klive = jk < L;
  const float kc0 = !lit && klive ? C0[jk] : 0.f, kc1 = !lit && klive ? C1[jk] : 0.f;
  const float kp0 = !lit && klive ? (float)P0[jk] : 0.f, kp1 = !lit && klive ? (float)P1[jk] : 0.f;
  float k0 = 0.f, k1 = 0.f;
  float dfk[4][MF], dvj[4][MF];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int f = 0; f < MF; ++f) dfk[a][f] = dvj[a][f] = 0.f;
  for (int i0 = 0; i0 < L; i0 += kTC) {
    stage_rows<D>(sQ, fqh, i0, kTC, L);
    stage_rows<D>(sG, gh, i0, kTC, L);
    if (!lit) {
      stage_vec(sC, C0, i0, kTC, L);
      stage_vec(sC + kTC, C1, i0, kTC, L);
      stage_pos(sPs, P0, i0, kTC, L);
      stage_pos(sPs + kTC, P1, i0, kTC, L);
    }
    for (int idx = threadIdx.x; idx < kTC * J4; idx += kTThreads) {
      const int r = idx / J4, c = (idx - r * J4) * 4, i = i0 + r, j = j0b + c;
      float4 a4 = make_float4(0.f, 0.f, 0.f, 0.f), d4 = a4;
      if (i < L && j < L) {
        a4 = load4(St + (size_t)i * LP + j);
        d4 = load4(Dt + (size_t)i * LP + j);
        if (j + 1 >= L) a4.y = d4.y = 0.f;
        if (j + 2 >= L) a4.z = d4.z = 0.f;
        if (j + 3 >= L) a4.w = d4.w = 0.f;
      }
      *reinterpret_cast<float4*>(sS + r * kTSL + c) = a4;
      *reinterpret_cast<float4*>(sE + r * kTSL + c) = d4;
    }
    __syncthreads();
    const int nc = min(kTC, L - i0);
#pragma unroll 4
    for (int t = 0; t < 16; ++t) {
      const int tq = 16 * grp + t;
      const bool ok = klive && tq < nc;
      const float sv = sS[tq * kTSL + kj], dav = sE[tq * kTSL + kj];
      float m0 = 0.f, m1 = 0.f;
      if (ok && !lit) {
        m0 = expf(-fabsf(sC[tq] - kc0) * w);
        m1 = expf(-fabsf(sC[kTC + tq] - kc1) * w);
      }
      const float m = !ok ? 0.f : lit ? 1.f : 0.5f * (m0 + m1);
      sS[tq * kTSL + kj] = m * sv;
      sE[tq * kTSL + kj] = m * dav;
      if (ms && ok) {
        const float e = sv * dav;
        k0 += sgnf(sPs[tq] - kp0) * m0 * e;
        k1 += sgnf(sPs[kTC + tq] - kp1) * m1 * e;
      }
    }
    __syncthreads();
    const int n4 = (nc + 3) & ~3;
    tile_apply_t<D>(sE, kTSL, sQ, n4, ty, tx, dfk);
    tile_apply_t<D>(sS, kTSL, sG, n4, ty, tx, dvj);
    __syncthreads();
  }
  if (ms) {   // the key's column terms over the four query groups, in a fixed order
    sKp[grp * kTR + kj] = k0;
    sKp[(4 + grp) * kTR + kj] = k1;
    __syncthreads();
    if (grp == 0 && klive) {
      p.K[(size_t)bh * L + jk] = sKp[kj] + sKp[kTR + kj] + sKp[2 * kTR + kj] + sKp[3 * kTR + kj];
      p.K[((size_t)BH + bh) * L + jk] =
          sKp[4 * kTR + kj] + sKp[5 * kTR + kj] + sKp[6 * kTR + kj] + sKp[7 * kTR + kj];
    }
  }
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int ja = j0b + 4 * ty + a;
    const bool live = ja < L;
    const T* kr = head_of<T>(p.k, bh, L, D) + (size_t)(live ? ja : L - 1) * D;
    float x[MF], dx[MF];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const float4 x4 = load4(kr + 4 * tx + 64 * u);
#pragma unroll
      for (int e = 0; e < 4; ++e) x[4 * u + e] = elem(x4, e);
    }
    phi_backward<MF, 16>(p.phi, x, dfk[a], dx);
    if (live) {
      float* dk = p.dk + ((size_t)bh * L + ja) * D;
      float* dv = p.dv + ((size_t)bh * L + ja) * D;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        *reinterpret_cast<float4*>(dk + 4 * tx + 64 * u) =
            make_float4(dx[4 * u], dx[4 * u + 1], dx[4 * u + 2], dx[4 * u + 3]);
        *reinterpret_cast<float4*>(dv + 4 * tx + 64 * u) =
            make_float4(dvj[a][4 * u], dvj[a][4 * u + 1], dvj[a][4 * u + 2], dvj[a][4 * u + 3]);
      }
    }
  }
}

// LION-S, one CTA per head: dlog(lambda_u) = sum over the orders of the
// suffix sum, from u's position, of -(1/2)(R + K) taken in that order.
__global__ void __launch_bounds__(kScanThreads) rbwd_dl_kernel(ReorderParams p, int BH) {
  const int L = p.L, bh = blockIdx.x, t0 = threadIdx.x;
  const int per = (L + kScanThreads - 1) / kScanThreads;
  const int lo = min(L, t0 * per), hi = min(L, lo + per);
  float* dl = p.dll + (size_t)bh * L;
  for (int o = 0; o < 2; ++o) {
    const int* ord = p.order + (size_t)o * L;
    const float* R = p.R + ((size_t)o * BH + bh) * L;
    const float* K = p.K + ((size_t)o * BH + bh) * L;
    auto val = [&](int t) {
      const int a = clamp_token(ord[t], L);
      return -0.5 * ((double)R[a] + (double)K[a]);
    };
    double run = 0.0, all;
    for (int t = lo; t < hi; ++t) run += val(t);
    const double incl = block_scan(run, &all);
    double right = all - incl;   // the positions after this thread's chunk
    for (int t = hi - 1; t >= lo; --t) {
      right += val(t);
      const int a = clamp_token(ord[t], L);
      dl[a] = o == 0 ? (float)right : dl[a] + (float)right;
    }
    __syncthreads();
  }
}

// LION-D: per head, the sum of the rows' shares; then over the batch.
__global__ void __launch_bounds__(kScanThreads) rbwd_dsum_kernel(ReorderParams p) {
  const int L = p.L, bh = blockIdx.x;
  double acc = 0.0, all;
  for (int i = threadIdx.x; i < L; i += blockDim.x) acc += (double)p.dterm[(size_t)bh * L + i];
  block_scan(acc, &all);
  if (threadIdx.x == 0) p.dsum[bh] = all;
}
__global__ void rbwd_heads_kernel(ReorderParams p) {
  const int h = blockIdx.x * blockDim.x + threadIdx.x;
  if (h >= p.H) return;
  double acc = 0.0;
  for (int b = 0; b < p.B; ++b) acc += p.dsum[(size_t)b * p.H + h];
  p.dll[h] = (float)acc;
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
  if ((e = allow_smem(reorder_full_kernel<T, D, 2>, smem)) != cudaSuccess) return e;
  reorder_full_kernel<T, D, 2><<<dim3((unsigned)BH, (p.L + kTR - 1) / kTR), kTThreads, smem, s>>>(p);
  return cudaGetLastError();
}

// The plain full form: features, LION-S's prefix, the tiled pass.
template <typename T, int D>
cudaError_t full_tiled_launch(const ReorderParams& p, cudaStream_t s) {
  const long BH = (long)p.B * p.H;
  cudaError_t e;
  if (p.mask_kind == MASK_S) {
    order_prefix_kernel<<<dim3((unsigned)BH, 1), kScanThreads, 0, s>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if ((e = launch_phi_rows<T, D>(p.q, p.k, p.fq, p.fk, BH * p.L, p.phi, s)) != cudaSuccess) return e;
  constexpr size_t smem = reorder_smem<D>();
  if ((e = allow_smem(reorder_full_kernel<T, D, 1>, smem)) != cudaSuccess) return e;
  reorder_full_kernel<T, D, 1><<<dim3((unsigned)BH, (p.L + kTR - 1) / kTR), kTThreads, smem, s>>>(p);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t rbwd_launch(const ReorderParams& p, cudaStream_t s) {
  const long BH = (long)p.B * p.H;
  order_positions_kernel<<<2, kOrderThreads, sizeof(int) * (size_t)p.L, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (p.mask_kind == MASK_S) {
    order_prefix_kernel<<<dim3((unsigned)BH, 2), kScanThreads, 0, s>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if ((e = launch_phi_rows<T, D>(p.q, p.k, p.fq, p.fk, BH * p.L, p.phi, s)) != cudaSuccess) return e;
  const dim3 grid((unsigned)BH, (p.L + kTR - 1) / kTR);
  constexpr size_t smem_r = rbwd_rows_smem<D>();
  if (p.St) {
    constexpr size_t smem_c = rbwd_cols_stored_smem<D>();
    if ((e = allow_smem(rbwd_rows_kernel<T, D, true>, smem_r)) != cudaSuccess) return e;
    if ((e = allow_smem(rbwd_cols_stored_kernel<T, D>, smem_c)) != cudaSuccess) return e;
    rbwd_rows_kernel<T, D, true><<<grid, kTThreads, smem_r, s>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    rbwd_cols_stored_kernel<T, D><<<grid, kTThreads, smem_c, s>>>(p);
  } else {
    constexpr size_t smem_c = rbwd_cols_smem<D>();
    if ((e = allow_smem(rbwd_rows_kernel<T, D, false>, smem_r)) != cudaSuccess) return e;
    if ((e = allow_smem(rbwd_cols_kernel<T, D>, smem_c)) != cudaSuccess) return e;
    rbwd_rows_kernel<T, D, false><<<grid, kTThreads, smem_r, s>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    rbwd_cols_kernel<T, D><<<grid, kTThreads, smem_c, s>>>(p);
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (p.mask_kind == MASK_S) {
    rbwd_dl_kernel<<<(unsigned)BH, kScanThreads, 0, s>>>(p, (int)BH);
    e = cudaGetLastError();
  } else if (p.mask_kind == MASK_D) {
    rbwd_dsum_kernel<<<(unsigned)BH, kScanThreads, 0, s>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    rbwd_heads_kernel<<<(p.H + 127) / 128, 128, 0, s>>>(p);
    e = cudaGetLastError();
  }
  return e;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

size_t reorder_workspace_bytes(int B, int H, int L, int d) {
  const size_t BH = (size_t)B * H, n = BH * L;
  return 2 * align256(sizeof(float) * n * d) + align256(sizeof(int) * 2 * (size_t)L) +
         align256(sizeof(float) * 2 * n);
}

int reorder_launches(int mask_kind) { return mask_kind == MASK_S ? 4 : 3; }

bool full_tiled_supported(const Problem& p) { return p.d == 64 || p.d == 128; }

size_t full_tiled_workspace_bytes(int B, int H, int L, int d) {
  const size_t n = (size_t)B * H * L;
  return 2 * align256(sizeof(float) * n * d) + align256(sizeof(float) * n);
}

int full_tiled_launches(int mask_kind) { return mask_kind == MASK_S ? 3 : 2; }

cudaError_t launch_full_tiled(const Problem& pr, void* ws, cudaStream_t s) {
  ReorderParams p;
  memset(&p, 0, sizeof(p));
  p.q = pr.q;
  p.k = pr.k;
  p.v = pr.v;
  p.log_lambda = pr.log_lambda;
  p.out = pr.out;
  p.B = pr.B;
  p.H = pr.H;
  p.L = pr.L;
  p.mask_kind = pr.mask_kind;
  p.phi = pr.phi;
  p.causal = pr.causal;
  const size_t n = (size_t)pr.B * pr.H * pr.L;
  uint8_t* w = static_cast<uint8_t*>(ws);
  p.fq = reinterpret_cast<float*>(w);
  w += align256(sizeof(float) * n * pr.d);
  p.fk = reinterpret_cast<float*>(w);
  w += align256(sizeof(float) * n * pr.d);
  p.coord = reinterpret_cast<float*>(w);
  const bool bf = pr.dtype == DT_BF16;
  switch (pr.d) {
    case 64: return bf ? full_tiled_launch<__nv_bfloat16, 64>(p, s) : full_tiled_launch<float, 64>(p, s);
    case 128: return bf ? full_tiled_launch<__nv_bfloat16, 128>(p, s) : full_tiled_launch<float, 128>(p, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_reordered(const Problem& pr, const int* order, void* ws, int* status, cudaStream_t s) {
  ReorderParams p;
  memset(&p, 0, sizeof(p));
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
  p.phi = pr.phi;
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

// Sequences up to this length keep s and dA in the workspace (8 L^2 bytes a
// head) instead of recomputing the scores in the columns pass.
constexpr int kRbwdStoreMaxL = 1024;

size_t reorder_bwd_workspace_bytes(int B, int H, int L, int d) {
  const size_t BH = (size_t)B * H, n = BH * L, LP = ((size_t)L + 3) & ~(size_t)3;
  return 3 * align256(sizeof(float) * n * d) + align256(sizeof(float) * n) + align256(sizeof(int) * 2 * (size_t)L) +
         3 * align256(sizeof(float) * 2 * n) + align256(sizeof(float) * n) + align256(sizeof(double) * BH) +
         (L <= kRbwdStoreMaxL ? 2 * align256(sizeof(float) * BH * L * LP) : 0);
}

int reorder_bwd_launches(int mask_kind) { return mask_kind == MASK_S ? 6 : mask_kind == MASK_D ? 6 : 4; }

cudaError_t launch_reordered_bwd(const Problem& pr, const int* order, const float* dy, float* dq, float* dk, float* dv,
                                 float* dll, void* ws, int* status, cudaStream_t s) {
  ReorderParams p;
  memset(&p, 0, sizeof(p));
  p.q = pr.q;
  p.k = pr.k;
  p.v = pr.v;
  p.log_lambda = pr.log_lambda;
  p.order = order;
  p.B = pr.B;
  p.H = pr.H;
  p.L = pr.L;
  p.mask_kind = pr.mask_kind;
  p.phi = pr.phi;
  p.status = status;
  p.dy = dy;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.dll = dll;
  const size_t BH = (size_t)pr.B * pr.H, n = BH * pr.L;
  uint8_t* w = static_cast<uint8_t*>(ws);
  p.fq = reinterpret_cast<float*>(w);
  w += align256(sizeof(float) * n * pr.d);
  p.fk = reinterpret_cast<float*>(w);
  w += align256(sizeof(float) * n * pr.d);
  p.g = reinterpret_cast<float*>(w);
  w += align256(sizeof(float) * n * pr.d);
  p.hd = reinterpret_cast<float*>(w);
  w += align256(sizeof(float) * n);
  p.pos = reinterpret_cast<int*>(w);
  w += align256(sizeof(int) * 2 * (size_t)pr.L);
  p.coord = reinterpret_cast<float*>(w);
  w += align256(sizeof(float) * 2 * n);
  p.R = reinterpret_cast<float*>(w);
  w += align256(sizeof(float) * 2 * n);
  p.K = reinterpret_cast<float*>(w);
  w += align256(sizeof(float) * 2 * n);
  p.dterm = reinterpret_cast<float*>(w);
  w += align256(sizeof(float) * n);
  p.dsum = reinterpret_cast<double*>(w);
  w += align256(sizeof(double) * BH);
  p.LP = (pr.L + 3) & ~3;
  p.St = p.Dt = nullptr;
  if (pr.L <= kRbwdStoreMaxL) {
    p.St = reinterpret_cast<float*>(w);
    w += align256(sizeof(float) * BH * pr.L * p.LP);
    p.Dt = reinterpret_cast<float*>(w);
  }
  const bool bf = pr.dtype == DT_BF16;
  switch (pr.d) {
    case 64: return bf ? rbwd_launch<__nv_bfloat16, 64>(p, s) : rbwd_launch<float, 64>(p, s);
    case 128: return bf ? rbwd_launch<__nv_bfloat16, 128>(p, s) : rbwd_launch<float, 128>(p, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace lion
