// lion_bwd.cu -- gradients of the LION operator through its full form, on
// the CUDA cores in fp32, for any d in {16, 32, 64, 128} and bfloat16 or
// float32 inputs.
//
// Full form (rebuttal page "LION: A bidirectional framework that trains like
// a Transformer and infers like an RNN", reply "Concern 1", Theorem 3.3
// Eq 25): per head, with A_ij = M_ij s_ij, s_ij = phi(q_i) . phi(k_j),
// num_i = sum_j A_ij v_j, den_i = sum_j A_ij and y_i = num_i / den_i.  Given
// dy = dLoss/dy, with dnum_i = dy_i / den_i and dden_i = -(dy_i . y_i) / den_i:
//   dA_ij     = dnum_i . v_j + dden_i
//   dv_j      = sum_i A_ij dnum_i
//   dphi(q_i) = sum_j M_ij dA_ij phi(k_j),   dphi(k_j) = sum_i M_ij dA_ij phi(q_i)
// and, M_ij being exp(P_max(i,j) - P_min(i,j)) with P the inclusive prefix of
// l = log(lambda), dLoss/dP_m = sum_{j<m} c_mj - sum_{i>m} c_im
// + sum_{i<m} c_im - sum_{j>m} c_mj with c_ij = A_ij dA_ij, so that
// dl_u = sum_{m >= u} dLoss/dP_m (l_0 never enters M: dl_0 = 0).  The
// feature maps' derivatives follow by the chain rule.
//
// Kernels: (1) phi(q), phi(k) into the workspace; (2) one pass per block of
// 32 query rows: y, dnum, dden (stored), then dphi(q), dq and the row terms
// of dLoss/dP; (3) one pass per block of 32 key rows: dphi(k), dk, dv and the
// column terms; (4) per head, dl (LION-S: suffix sums; LION-D: the sum over
// positions, sum_m m dLoss/dP_m) in double, and for LION-D the sum over the
// batch.  The mask value is generated per (i, j) as in the forward full form.
// Passes (2) and (3) come in two builds: for d = 16 and 32, 8 threads share a
// row and reduce each dot product by shuffles; for d = 64 and 128 a thread
// holds a 4 x 4 tile of scores and whole dot products (register tiling, with
// LION-S reading a per-head prefix of l that a small kernel writes first).
#include "lion_common.cuh"
#include "lion_internal.h"
#include "tile_simt.cuh"

namespace lion {
namespace {

constexpr int kRows = 32;    // rows of a block (queries in pass 2, keys in pass 3)
constexpr int kGroup = 8;    // threads per row
constexpr int kTile = 32;    // tokens per staged tile of the other side

// Inclusive prefix of l over the head into sP[0..L) (LION-S), whole block.
__device__ void prefix_log_lambda(const float* ll, int L, float* sP, float* scratch) {
  const int T = blockDim.x, t = threadIdx.x, lane = t & 31, warp = t >> 5;
  for (int i = t; i < L; i += T) sP[i] = ll[i];
  __syncthreads();
  const int per = (L + T - 1) / T;
  const int lo = min(L, t * per), hi = min(L, lo + per);
  float run = 0.f;
  for (int i = lo; i < hi; ++i) { run += sP[i]; sP[i] = run; }
  float x = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    float w = lane < (T >> 5) ? scratch[lane] : 0.f;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    scratch[lane] = w;
  }
  __syncthreads();
  const float excl = x - run + (warp > 0 ? scratch[warp - 1] : 0.f);
  for (int i = lo; i < hi; ++i) sP[i] += excl;
  __syncthreads();
}

// log M_ij for the head's decay kind.
__device__ __forceinline__ float log_mask(int mask_kind, int i, int j, float lh, const float* sP) {
  if (mask_kind == MASK_D) return fabsf((float)(i - j)) * lh;
  if (mask_kind == MASK_S) return i >= j ? sP[i] - sP[j] : sP[j] - sP[i];
  return 0.f;
}

struct BwdParams {
  const void* q;
  const void* k;
  const void* v;
  const float* log_lambda;
  const float* dy;
  float* dq;
  float* dk;
  float* dv;
  float* dll;
  int B, H, L;
  int mask_kind, phi;
  // workspace
  float* fq;     // [BH][L][D] phi(q)
  float* fk;     // [BH][L][D] phi(k)
  float* g;      // [BH][L][D] dnum
  float* hd;     // [BH][L]    dden
  float* rowd;   // [BH][L]    row terms of dLoss/dP
  float* cold;   // [BH][L]    column terms of dLoss/dP
  double* dsum;  // [BH]       LION-D: sum over positions of dl
  float* P;      // [BH][L]    LION-S: inclusive prefix of l (tiled passes)
  // stored-tile build (L <= kBwdStoreMaxL): A_ij and M_ij dA_ij, [BH][L (i)]
  // [LP (j)], and the rows pass's column terms per block of 32 rows
  float* At;
  float* Dt;
  float* colpart;  // [BH][nblk][L]
  int LP, nblk;
};

__device__ __forceinline__ void load_tile(float* dst, int ld, const float* src, int row0, int rows, int L, int D) {
  for (int idx = threadIdx.x; idx < rows * D; idx += blockDim.x) {
    const int r = idx / D, m = idx - r * D, i = row0 + r;
    dst[r * ld + m] = i < L ? src[(size_t)i * D + m] : 0.f;
  }
}
template <typename T>
__device__ __forceinline__ void load_tile_in(float* dst, int ld, const T* src, int row0, int rows, int L, int D) {
  for (int idx = threadIdx.x; idx < rows * D; idx += blockDim.x) {
    const int r = idx / D, m = idx - r * D, i = row0 + r;
    dst[r * ld + m] = i < L ? to_f32(src[(size_t)i * D + m]) : 0.f;
  }
}

// (2) rows: 32 queries per CTA, 8 threads per query.
template <typename T, int D>
__global__ void __launch_bounds__(256) bwd_rows_kernel(BwdParams p) {
  constexpr int LD = D + 8, NC = D / kGroup;
  extern __shared__ float smem[];
  float* sQ = smem;                   // [kRows][LD] phi(q)
  float* sK = sQ + kRows * LD;        // [kTile][D]  phi(k)
  float* sV = sK + kTile * D;         // [kTile][D]  v
  float* sP = sV + kTile * D;         // [L] prefix (LION-S)
  __shared__ float scratch[32];
  const int L = p.L, bh = blockIdx.x, h = bh % p.H, i0 = blockIdx.y * kRows;
  const float lh = p.mask_kind == MASK_D ? p.log_lambda[h] : 0.f;
  if (p.mask_kind == MASK_S) prefix_log_lambda(p.log_lambda + (size_t)bh * L, L, sP, scratch);
  load_tile(sQ, LD, p.fq + (size_t)bh * L * D, i0, kRows, L, D);
  __syncthreads();
  const int r = threadIdx.x / kGroup, g = threadIdx.x % kGroup, i0r = i0 + r;
  const bool live = i0r < L;
  // rows past L run on row L-1's mask values (in bounds) and store nothing;
  // every thread takes part in its group's shuffles
  const int i = live ? i0r : L - 1;
  const T* vh = head_of<T>(p.v, bh, L, D);
  // ---- pass A: y_i, then dnum_i and dden_i
  float acc[NC], den = 0.f;
#pragma unroll
  for (int c = 0; c < NC; ++c) acc[c] = 0.f;
  for (int j0 = 0; j0 < L; j0 += kTile) {
    const int nj = min(kTile, L - j0);
    load_tile(sK, D, p.fk + (size_t)bh * L * D, j0, kTile, L, D);
    load_tile_in<T>(sV, D, vh, j0, kTile, L, D);
    __syncthreads();
    for (int jj = 0; jj < nj; ++jj) {
      float s = 0.f;
#pragma unroll
      for (int c = 0; c < NC; ++c) s += sQ[r * LD + g + c * kGroup] * sK[jj * D + g + c * kGroup];
      s = group_sum(s);
      const float a = s * expf(log_mask(p.mask_kind, i, j0 + jj, lh, sP));
      den += a;
#pragma unroll
      for (int c = 0; c < NC; ++c) acc[c] += a * sV[jj * D + g + c * kGroup];
    }
    __syncthreads();
  }
  float gi[NC], hi = 0.f;
  {
    const float* dy = p.dy + ((size_t)bh * L + (live ? i : 0)) * D;
    float dyy = 0.f;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      const float d = live ? dy[g + c * kGroup] : 0.f;
      dyy += d * (acc[c] / den);
      gi[c] = live ? d / den : 0.f;
    }
    const float gs = group_sum(dyy);
    hi = live ? -gs / den : 0.f;
    if (live) {
      float* gw = p.g + ((size_t)bh * L + i) * D;
#pragma unroll
      for (int c = 0; c < NC; ++c) gw[g + c * kGroup] = gi[c];
      if (g == 0) p.hd[(size_t)bh * L + i] = hi;
    }
  }
  // ---- pass B: dphi(q_i) and the row terms of dLoss/dP
  float dfq[NC], rowl = 0.f, rowu = 0.f;
#pragma unroll
  for (int c = 0; c < NC; ++c) dfq[c] = 0.f;
  for (int j0 = 0; j0 < L; j0 += kTile) {
    const int nj = min(kTile, L - j0);
    load_tile(sK, D, p.fk + (size_t)bh * L * D, j0, kTile, L, D);
    load_tile_in<T>(sV, D, vh, j0, kTile, L, D);
    __syncthreads();
    for (int jj = 0; jj < nj; ++jj) {
      float s = 0.f, gv = 0.f;
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        s += sQ[r * LD + g + c * kGroup] * sK[jj * D + g + c * kGroup];
        gv += gi[c] * sV[jj * D + g + c * kGroup];
      }
      s = group_sum(s);
      gv = group_sum(gv);
      const int j = j0 + jj;
      const float m = expf(log_mask(p.mask_kind, i, j, lh, sP));
      const float da = gv + hi, ds = m * da, cij = m * s * da;
#pragma unroll
      for (int c = 0; c < NC; ++c) dfq[c] += ds * sK[jj * D + g + c * kGroup];
      if (j < i) rowl += cij;
      else if (j > i) rowu += cij;
    }
    __syncthreads();
  }
  {
    const T* qr = head_of<T>(p.q, bh, L, D) + (size_t)i * D;
    float x[NC], dx[NC];
#pragma unroll
    for (int c = 0; c < NC; ++c) x[c] = to_f32(qr[g + c * kGroup]);
    phi_backward<NC>(p.phi, x, dfq, dx);   // gi = 0 on dead rows: dfq = 0
    if (live) {
      float* dq = p.dq + ((size_t)bh * L + i) * D;
#pragma unroll
      for (int c = 0; c < NC; ++c) dq[g + c * kGroup] = dx[c];
      if (g == 0) p.rowd[(size_t)bh * L + i] = rowl - rowu;
    }
  }
}

// (3) columns: 32 keys per CTA, 8 threads per key.
template <typename T, int D>
__global__ void __launch_bounds__(256) bwd_cols_kernel(BwdParams p) {
  constexpr int LD = D + 8, NC = D / kGroup;
  extern __shared__ float smem[];
  float* sK = smem;                   // [kRows][LD] phi(k) of this block's keys
  float* sVc = sK + kRows * LD;       // [kRows][LD] v of this block's keys
  float* sQ = sVc + kRows * LD;       // [kTile][D]  phi(q)
  float* sG = sQ + kTile * D;         // [kTile][D]  dnum
  float* sH = sG + kTile * D;         // [kTile]     dden
  float* sP = sH + kTile;             // [L] prefix (LION-S)
  __shared__ float scratch[32];
  const int L = p.L, bh = blockIdx.x, h = bh % p.H, j0b = blockIdx.y * kRows;
  const float lh = p.mask_kind == MASK_D ? p.log_lambda[h] : 0.f;
  if (p.mask_kind == MASK_S) prefix_log_lambda(p.log_lambda + (size_t)bh * L, L, sP, scratch);
  load_tile(sK, LD, p.fk + (size_t)bh * L * D, j0b, kRows, L, D);
  load_tile_in<T>(sVc, LD, head_of<T>(p.v, bh, L, D), j0b, kRows, L, D);
  __syncthreads();
  const int r = threadIdx.x / kGroup, g = threadIdx.x % kGroup, j0r = j0b + r;
  const bool live = j0r < L;
  const int j = live ? j0r : L - 1;   // in-bounds mask values; stores only when live
  float dfk[NC], dvj[NC], coll = 0.f, colu = 0.f;
#pragma unroll
  for (int c = 0; c < NC; ++c) dfk[c] = dvj[c] = 0.f;
  for (int i0 = 0; i0 < L; i0 += kTile) {
    const int ni = min(kTile, L - i0);
    load_tile(sQ, D, p.fq + (size_t)bh * L * D, i0, kTile, L, D);
    load_tile(sG, D, p.g + (size_t)bh * L * D, i0, kTile, L, D);
    for (int t = threadIdx.x; t < kTile; t += blockDim.x) sH[t] = i0 + t < L ? p.hd[(size_t)bh * L + i0 + t] : 0.f;
    __syncthreads();
    for (int ii = 0; ii < ni; ++ii) {
      float s = 0.f, gv = 0.f;
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        s += sQ[ii * D + g + c * kGroup] * sK[r * LD + g + c * kGroup];
        gv += sG[ii * D + g + c * kGroup] * sVc[r * LD + g + c * kGroup];
      }
      s = group_sum(s);
      gv = group_sum(gv);
      const int i = i0 + ii;
      const float m = expf(log_mask(p.mask_kind, i, j, lh, sP));
      const float a = m * s, da = gv + sH[ii], ds = m * da, cij = a * da;
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        dfk[c] += ds * sQ[ii * D + g + c * kGroup];
        dvj[c] += a * sG[ii * D + g + c * kGroup];
      }
      if (i > j) coll += cij;
      else if (i < j) colu += cij;
    }
    __syncthreads();
  }
  {
    const T* kr = head_of<T>(p.k, bh, L, D) + (size_t)j * D;
    float x[NC], dx[NC];
#pragma unroll
    for (int c = 0; c < NC; ++c) x[c] = to_f32(kr[g + c * kGroup]);
    phi_backward<NC>(p.phi, x, dfk, dx);
    if (live) {
      float* dk = p.dk + ((size_t)bh * L + j) * D;
      float* dv = p.dv + ((size_t)bh * L + j) * D;
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        dk[g + c * kGroup] = dx[c];
        dv[g + c * kGroup] = dvj[c];
      }
      if (g == 0) p.cold[(size_t)bh * L + j] = colu - coll;
    }
  }
}

// ---------------------------------------------------------------------------
// Register-tiled passes (2) and (3) for d in {64, 128}, on the tile products
// of tile_simt.cuh.  The mask value is generated per (i, j) exactly as in the
// one-row-per-group passes.

// M_ij of query i and key j (Pi, Pj: the prefix at i and j for LION-S).
__device__ __forceinline__ float mask_value(int mask_kind, int i, int j, float Pi, float Pj, float lh) {
  if (mask_kind == MASK_D) return expf(fabsf((float)(i - j)) * lh);
  if (mask_kind == MASK_S) return expf(i >= j ? Pi - Pj : Pj - Pi);
  return 1.f;
}

// LION-S: the inclusive prefix of l per head into P (one CTA per head),
// accumulated in double and stored in fp32.
constexpr int kPrefixThreads = kScanThreads;
__global__ void __launch_bounds__(kPrefixThreads) bwd_prefix_kernel(BwdParams p) {
  const int L = p.L, bh = blockIdx.x, t = threadIdx.x;
  const float* ll = p.log_lambda + (size_t)bh * L;
  float* P = p.P + (size_t)bh * L;
  const int per = (L + kPrefixThreads - 1) / kPrefixThreads;
  const int lo = min(L, t * per), hi = min(L, lo + per);
  double run = 0.0, all;
  for (int m = lo; m < hi; ++m) run += (double)ll[m];
  double off = block_scan(run, &all) - run;
  for (int m = lo; m < hi; ++m) {
    off += (double)ll[m];
    P[m] = (float)off;
  }
}

template <int D>
constexpr size_t rows_tiled_smem(bool store) {
  return sizeof(float) * ((size_t)(2 * kTR + 2 * kTC) * (D + 4) + kTR * kTAL + kTC + (store ? 4 * kTC : 0));
}
template <int D>
constexpr size_t cols_tiled_smem() {
  return sizeof(float) * ((size_t)(2 * kTR + 2 * kTC) * (D + 4) + 2 * kTR * kTAL + 2 * kTC);
}

// (2) rows, tiled: 32 queries per CTA.  STORE: pass A writes A_ij and pass
// B reads it back instead of recomputing the scores, writes M_ij dA_ij, and
// sums the column terms of its 32 rows per key (the columns pass then needs
// no scores of its own).
template <typename T, int D, bool STORE>
__global__ void __launch_bounds__(kTThreads) bwd_rows_tiled(BwdParams p) {
  constexpr int LD = D + 4, MF = D / 16, U = D / 64;
  extern __shared__ __align__(16) float smem[];
  float* sQ = smem;                  // [kTR][LD]   phi(q) of the block
  float* sG = sQ + kTR * LD;         // [kTR][LD]   dnum of the block
  float* sK = sG + kTR * LD;         // [kTC][LD]   phi(k) of the tile
  float* sV = sK + kTC * LD;         // [kTC][LD]   v of the tile
  float* sA = sV + kTC * LD;         // [kTR][kTAL] A (pass A), M (.) dA (pass B)
  float* sPt = sA + kTR * kTAL;      // [kTC]       P of the tile (LION-S)
  float* sCol = sPt + kTC;           // [4][kTC]    column terms per warp (STORE)
  const int L = p.L, bh = blockIdx.x, h = bh % p.H, i0 = blockIdx.y * kTR, nr = min(kTR, L - i0);
  float* At = STORE ? p.At + (size_t)bh * L * p.LP : nullptr;
  float* Dt = STORE ? p.Dt + (size_t)bh * L * p.LP : nullptr;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const bool ms = p.mask_kind == MASK_S;
  const float lh = p.mask_kind == MASK_D ? p.log_lambda[h] : 0.f;
  const float* Ph = ms ? p.P + (size_t)bh * L : nullptr;
  const float* fkh = p.fk + (size_t)bh * L * D;
  const T* vh = head_of<T>(p.v, bh, L, D);
  stage_rows<D>(sQ, p.fq + (size_t)bh * L * D, i0, kTR, L);
  int ia[4];
  bool live[4];
  float Pi[4];
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    ia[a] = i0 + ty + 8 * a;
    live[a] = ia[a] < L;
    Pi[a] = ms && live[a] ? Ph[ia[a]] : 0.f;
  }
  // ---- pass A: den_i and num_i
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
    if (ms) stage_vec(sPt, Ph, j0, kTC, L);
    __syncthreads();
    const int nc = min(kTC, L - j0);
    float s[4][4];
    tile_scores<D>(sQ, sK, ty, tx, nr, nc, s);
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int jl = tx + 16 * b, j = j0 + jl;
        const float m = live[a] && j < L ? mask_value(p.mask_kind, ia[a], j, Pi[a], sPt[jl], lh) : 0.f;
        const float x = m * s[a][b];
        den[a] += x;
        sA[(ty + 8 * a) * kTAL + jl] = x;
        if (STORE && live[a] && j < L) At[(size_t)ia[a] * p.LP + j] = x;
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
        const float d = elem(d4, e);
        dyy += d * (num[a][4 * u + e] / dn);
        gi[4 * u + e] = live[a] ? d / dn : 0.f;
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
  // ---- pass B: dphi(q_i) and the row terms of dLoss/dP
  float dfq[4][MF], rowl[4], rowu[4];
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    rowl[a] = rowu[a] = 0.f;
#pragma unroll
    for (int f = 0; f < MF; ++f) dfq[a][f] = 0.f;
  }
  for (int j0 = 0; j0 < L; j0 += kTC) {
    float s[4][4], gv[4][4];
    if (STORE) {   // A_ij as this thread wrote it in pass A, in flight during the staging
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const int j = j0 + tx + 16 * b;
          s[a][b] = live[a] && j < L ? At[(size_t)ia[a] * p.LP + j] : 0.f;
        }
    }
    stage_rows<D>(sK, fkh, j0, kTC, L);
    stage_rows<D>(sV, vh, j0, kTC, L);
    if (ms) stage_vec(sPt, Ph, j0, kTC, L);
    __syncthreads();
    const int nc = min(kTC, L - j0);
    if (!STORE) tile_scores<D>(sQ, sK, ty, tx, nr, nc, s);
    tile_scores<D>(sG, sV, ty, tx, nr, nc, gv);
    float cs[4] = {0.f, 0.f, 0.f, 0.f};   // signed column terms of this thread's rows
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int jl = tx + 16 * b, j = j0 + jl;
        const float m = live[a] && j < L ? mask_value(p.mask_kind, ia[a], j, Pi[a], sPt[jl], lh) : 0.f;
        const float x = STORE ? s[a][b] : m * s[a][b];
        const float da = gv[a][b] + hi[a], c = x * da, ds = m * da;
        sA[(ty + 8 * a) * kTAL + jl] = ds;
        if (STORE) {
          cs[b] += j > ia[a] ? c : j < ia[a] ? -c : 0.f;
          if (live[a] && j < L) Dt[(size_t)ia[a] * p.LP + j] = ds;
        }
        if (j < ia[a]) rowl[a] += c;
        else if (j > ia[a]) rowu[a] += c;
      }
    if (STORE) {   // the two row threads of a column in a warp, then one slot per warp
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        cs[b] += __shfl_xor_sync(0xffffffffu, cs[b], 16);
        if ((ty & 1) == 0) sCol[(ty >> 1) * kTC + tx + 16 * b] = cs[b];
      }
    }
    __syncthreads();
    tile_apply<D>(sA, sK, (nc + 3) & ~3, ty, tx, nr, dfq);
    if (STORE && threadIdx.x < nc)
      p.colpart[((size_t)bh * p.nblk + blockIdx.y) * L + j0 + threadIdx.x] =
          sCol[threadIdx.x] + sCol[kTC + threadIdx.x] + sCol[2 * kTC + threadIdx.x] + sCol[3 * kTC + threadIdx.x];
    __syncthreads();
  }
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const float rl = group_sum<16>(rowl[a]), ru = group_sum<16>(rowu[a]);
    // dead rows run on row L-1's inputs with dfq = 0 and store nothing; every
    // thread takes part in its group's shuffles
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
      if (tx == 0) p.rowd[(size_t)bh * L + ia[a]] = rl - ru;
    }
  }
}

// (3) columns, tiled: 32 keys per CTA.
template <typename T, int D>
__global__ void __launch_bounds__(kTThreads) bwd_cols_tiled(BwdParams p) {
  constexpr int LD = D + 4, MF = D / 16, U = D / 64;
  extern __shared__ __align__(16) float smem[];
  float* sK = smem;                  // [kTR][LD]   phi(k) of the block
  float* sVb = sK + kTR * LD;        // [kTR][LD]   v of the block
  float* sQ = sVb + kTR * LD;        // [kTC][LD]   phi(q) of the tile
  float* sG = sQ + kTC * LD;         // [kTC][LD]   dnum of the tile
  float* sA = sG + kTC * LD;         // [kTR][kTAL] A^T
  float* sD = sA + kTR * kTAL;       // [kTR][kTAL] (M (.) dA)^T
  float* sHt = sD + kTR * kTAL;      // [kTC]       dden of the tile
  float* sPt = sHt + kTC;            // [kTC]       P of the tile (LION-S)
  const int L = p.L, bh = blockIdx.x, h = bh % p.H, j0b = blockIdx.y * kTR, nr = min(kTR, L - j0b);
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const bool ms = p.mask_kind == MASK_S;
  const float lh = p.mask_kind == MASK_D ? p.log_lambda[h] : 0.f;
  const float* Ph = ms ? p.P + (size_t)bh * L : nullptr;
  const float* fqh = p.fq + (size_t)bh * L * D;
  const float* gh = p.g + (size_t)bh * L * D;
  const float* hh = p.hd + (size_t)bh * L;
  stage_rows<D>(sK, p.fk + (size_t)bh * L * D, j0b, kTR, L);
  stage_rows<D>(sVb, head_of<T>(p.v, bh, L, D), j0b, kTR, L);
  int ja[4];
  bool live[4];
  float Pj[4];
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    ja[a] = j0b + ty + 8 * a;
    live[a] = ja[a] < L;
    Pj[a] = ms && live[a] ? Ph[ja[a]] : 0.f;
  }
  float dfk[4][MF], dvj[4][MF], coll[4], colu[4];
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    coll[a] = colu[a] = 0.f;
#pragma unroll
    for (int f = 0; f < MF; ++f) dfk[a][f] = dvj[a][f] = 0.f;
  }
  for (int i0 = 0; i0 < L; i0 += kTC) {
    stage_rows<D>(sQ, fqh, i0, kTC, L);
    stage_rows<D>(sG, gh, i0, kTC, L);
    stage_vec(sHt, hh, i0, kTC, L);
    if (ms) stage_vec(sPt, Ph, i0, kTC, L);
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
        const float m = live[a] && i < L ? mask_value(p.mask_kind, i, ja[a], sPt[il], Pj[a], lh) : 0.f;
        const float x = m * s[a][b], da = gv[a][b] + sHt[il], c = x * da;
        sA[(ty + 8 * a) * kTAL + il] = x;
        sD[(ty + 8 * a) * kTAL + il] = m * da;
        if (i > ja[a]) coll[a] += c;
        else if (i < ja[a]) colu[a] += c;
      }
    __syncthreads();
    const int n4 = (nc + 3) & ~3;
    tile_apply<D>(sD, sQ, n4, ty, tx, nr, dfk);
    tile_apply<D>(sA, sG, n4, ty, tx, nr, dvj);
    __syncthreads();
  }
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const float cl = group_sum<16>(coll[a]), cu = group_sum<16>(colu[a]);
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
      if (tx == 0) p.cold[(size_t)bh * L + ja[a]] = cu - cl;
    }
  }
}

template <int D>
constexpr size_t cols_stored_smem() {
  return sizeof(float) * ((size_t)2 * kTC * (D + 4) + 2 * kTC * kTSL);
}

// (3) columns from the stored A_ij and M_ij dA_ij: 32 keys per CTA, thread
// (ty, tx) holding keys 4ty + a; dphi(k_j) = sum_i M_ij dA_ij phi(q_i) and
// dv_j = sum_i A_ij dnum_i; the column terms are the sums of the rows pass's
// per-block partials.
template <typename T, int D>
__global__ void __launch_bounds__(kTThreads) bwd_cols_stored(BwdParams p) {
  constexpr int LD = D + 4, MF = D / 16, U = D / 64, J4 = kTR / 4;
  extern __shared__ __align__(16) float smem[];
  float* sQ = smem;                  // [kTC][LD]   phi(q) of the tile
  float* sG = sQ + kTC * LD;         // [kTC][LD]   dnum of the tile
  float* sA = sG + kTC * LD;         // [kTC][kTSL] A over the tile's queries x the block's keys
  float* sD = sA + kTC * kTSL;       // [kTC][kTSL] M (.) dA, the same
  const int L = p.L, LP = p.LP, bh = blockIdx.x, j0b = blockIdx.y * kTR;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const float* fqh = p.fq + (size_t)bh * L * D;
  const float* gh = p.g + (size_t)bh * L * D;
  const float* At = p.At + (size_t)bh * L * LP;
  const float* Dt = p.Dt + (size_t)bh * L * LP;
  float dfk[4][MF], dvj[4][MF];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int f = 0; f < MF; ++f) dfk[a][f] = dvj[a][f] = 0.f;
  for (int i0 = 0; i0 < L; i0 += kTC) {
    stage_rows<D>(sQ, fqh, i0, kTC, L);
    stage_rows<D>(sG, gh, i0, kTC, L);
    // the block's 32 columns of A and M (.) dA over the tile's rows; entries
    // past L (rows, and the row padding up to LP that is never written) read as 0
    for (int idx = threadIdx.x; idx < kTC * J4; idx += kTThreads) {
      const int r = idx / J4, c = (idx - r * J4) * 4, i = i0 + r, j = j0b + c;
      float4 a4 = make_float4(0.f, 0.f, 0.f, 0.f), d4 = a4;
      if (i < L && j < L) {
        a4 = load4(At + (size_t)i * LP + j);
        d4 = load4(Dt + (size_t)i * LP + j);
        if (j + 1 >= L) a4.y = d4.y = 0.f;
        if (j + 2 >= L) a4.z = d4.z = 0.f;
        if (j + 3 >= L) a4.w = d4.w = 0.f;
      }
      *reinterpret_cast<float4*>(sA + r * kTSL + c) = a4;
      *reinterpret_cast<float4*>(sD + r * kTSL + c) = d4;
    }
    __syncthreads();
    const int n4 = (min(kTC, L - i0) + 3) & ~3;
    tile_apply_t<D>(sD, kTSL, sQ, n4, ty, tx, dfk);
    tile_apply_t<D>(sA, kTSL, sG, n4, ty, tx, dvj);
    __syncthreads();
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
      if (tx == 0) {
        float cs = 0.f;
        for (int blk = 0; blk < p.nblk; ++blk) cs += p.colpart[((size_t)bh * p.nblk + blk) * L + ja];
        p.cold[(size_t)bh * L + ja] = cs;
      }
    }
  }
}

// (4) dl of one head (one CTA): dLoss/dP_m = rowd_m + cold_m; LION-S writes
// the suffix sums (position 0: 0), LION-D the total sum_m m dLoss/dP_m.
constexpr int kDlThreads = kScanThreads;
__global__ void __launch_bounds__(kDlThreads) bwd_dl_kernel(BwdParams p) {
  __shared__ double part[kDlThreads];
  const int L = p.L, bh = blockIdx.x, t = threadIdx.x;
  const float* rd = p.rowd + (size_t)bh * L;
  const float* cd = p.cold + (size_t)bh * L;
  const int per = (L + kDlThreads - 1) / kDlThreads;
  const int lo = min(L, t * per), hi = min(L, lo + per);
  if (p.mask_kind == MASK_D) {
    double acc = 0.0;
    for (int m = lo; m < hi; ++m) acc += (double)m * ((double)rd[m] + (double)cd[m]);
    part[t] = acc;
    __syncthreads();
    for (int o = kDlThreads / 2; o > 0; o >>= 1) {
      if (t < o) part[t] += part[t + o];
      __syncthreads();
    }
    if (t == 0) p.dsum[bh] = part[0];
    return;
  }
  // suffix sums: this thread's chunk total, then the totals of the chunks to its right
  double run = 0.0, all;
  for (int m = lo; m < hi; ++m) run += (double)rd[m] + (double)cd[m];
  double right = block_scan(run, &all);
  right = all - right;
  float* out = p.dll + (size_t)bh * L;
  for (int m = hi - 1; m >= lo; --m) {
    right += (double)rd[m] + (double)cd[m];
    out[m] = m == 0 ? 0.f : (float)right;
  }
}

// LION-D: dlog_lambda[h] = sum over the batch of the per-head totals.
__global__ void bwd_dl_heads_kernel(BwdParams p) {
  const int h = blockIdx.x * blockDim.x + threadIdx.x;
  if (h >= p.H) return;
  double acc = 0.0;
  for (int b = 0; b < p.B; ++b) acc += p.dsum[(size_t)b * p.H + h];
  p.dll[h] = (float)acc;
}

template <typename Kern>
cudaError_t allow(Kern kern, size_t bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <typename T, int D>
cudaError_t bwd_launch(const BwdParams& p, cudaStream_t s) {
  cudaError_t e = launch_phi_rows<T, D>(p.q, p.k, p.fq, p.fk, (long)p.B * p.H * p.L, p.phi, s);
  if (e != cudaSuccess) return e;
  if constexpr (D >= 64) {
    if (p.mask_kind == MASK_S) {
      bwd_prefix_kernel<<<p.B * p.H, kPrefixThreads, 0, s>>>(p);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    const dim3 grid(p.B * p.H, (p.L + kTR - 1) / kTR);
    if (p.At) {
      constexpr size_t smem_r = rows_tiled_smem<D>(true), smem_c = cols_stored_smem<D>();
      if ((e = allow(bwd_rows_tiled<T, D, true>, smem_r)) != cudaSuccess) return e;
      if ((e = allow(bwd_cols_stored<T, D>, smem_c)) != cudaSuccess) return e;
      bwd_rows_tiled<T, D, true><<<grid, kTThreads, smem_r, s>>>(p);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
      bwd_cols_stored<T, D><<<grid, kTThreads, smem_c, s>>>(p);
    } else {
      constexpr size_t smem_r = rows_tiled_smem<D>(false), smem_c = cols_tiled_smem<D>();
      if ((e = allow(bwd_rows_tiled<T, D, false>, smem_r)) != cudaSuccess) return e;
      if ((e = allow(bwd_cols_tiled<T, D>, smem_c)) != cudaSuccess) return e;
      bwd_rows_tiled<T, D, false><<<grid, kTThreads, smem_r, s>>>(p);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
      bwd_cols_tiled<T, D><<<grid, kTThreads, smem_c, s>>>(p);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  } else {
    const size_t sp = p.mask_kind == MASK_S ? (size_t)p.L : 0;
    const size_t smem_r = sizeof(float) * ((size_t)kRows * (D + 8) + 2 * kTile * D + sp);
    const size_t smem_c = sizeof(float) * (2 * (size_t)kRows * (D + 8) + 2 * kTile * D + kTile + sp);
    if ((e = allow(bwd_rows_kernel<T, D>, smem_r)) != cudaSuccess) return e;
    if ((e = allow(bwd_cols_kernel<T, D>, smem_c)) != cudaSuccess) return e;
    const dim3 grid(p.B * p.H, (p.L + kRows - 1) / kRows);
    bwd_rows_kernel<T, D><<<grid, 256, smem_r, s>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    bwd_cols_kernel<T, D><<<grid, 256, smem_c, s>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (p.mask_kind != MASK_LIT) {
    bwd_dl_kernel<<<p.B * p.H, kDlThreads, 0, s>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (p.mask_kind == MASK_D) {
      bwd_dl_heads_kernel<<<(p.H + 127) / 128, 128, 0, s>>>(p);
      e = cudaGetLastError();
    }
  }
  return e;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Sequences up to this length keep A and M (.) dA in the workspace (8 L^2
// bytes a head) instead of recomputing the scores in two more passes.
constexpr int kBwdStoreMaxL = 1024;
bool bwd_stores(int L, int d) { return d >= 64 && L <= kBwdStoreMaxL; }
size_t stored_bytes(size_t BH, int L) {
  const size_t LP = ((size_t)L + 3) & ~(size_t)3, nblk = ((size_t)L + kTR - 1) / kTR;
  return 2 * align256(sizeof(float) * BH * L * LP) + align256(sizeof(float) * BH * nblk * L);
}

}  // namespace

cudaError_t launch_dlog_lambda(int B, int H, int L, int mask_kind, const float* rowd, const float* cold, double* dsum,
                               float* dll, cudaStream_t s) {
  if (mask_kind == MASK_LIT) return cudaSuccess;
  BwdParams p = {};
  p.B = B;
  p.H = H;
  p.L = L;
  p.mask_kind = mask_kind;
  p.rowd = const_cast<float*>(rowd);
  p.cold = const_cast<float*>(cold);
  p.dsum = dsum;
  p.dll = dll;
  bwd_dl_kernel<<<B * H, kDlThreads, 0, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || mask_kind != MASK_D) return e;
  bwd_dl_heads_kernel<<<(H + 127) / 128, 128, 0, s>>>(p);
  return cudaGetLastError();
}

size_t bwd_workspace_bytes(int B, int H, int L, int d) {
  const size_t BH = (size_t)B * H, n = BH * L;
  return 3 * align256(sizeof(float) * n * d) + 4 * align256(sizeof(float) * n) + align256(sizeof(double) * BH) +
         (bwd_stores(L, d) ? stored_bytes(BH, L) : 0);
}

cudaError_t launch_bwd(const Problem& pr, const float* dy, float* dq, float* dk, float* dv, float* dll, void* ws,
                       cudaStream_t s) {
  BwdParams p;
  p.q = pr.q;
  p.k = pr.k;
  p.v = pr.v;
  p.log_lambda = pr.log_lambda;
  p.dy = dy;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.dll = dll;
  p.B = pr.B;
  p.H = pr.H;
  p.L = pr.L;
  p.mask_kind = pr.mask_kind;
  p.phi = pr.phi;
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
  p.rowd = reinterpret_cast<float*>(w);
  w += align256(sizeof(float) * n);
  p.cold = reinterpret_cast<float*>(w);
  w += align256(sizeof(float) * n);
  p.dsum = reinterpret_cast<double*>(w);
  w += align256(sizeof(double) * BH);
  p.P = reinterpret_cast<float*>(w);
  w += align256(sizeof(float) * n);
  p.LP = (pr.L + 3) & ~3;
  p.nblk = (pr.L + kTR - 1) / kTR;
  p.At = p.Dt = p.colpart = nullptr;
  if (bwd_stores(pr.L, pr.d)) {
    p.At = reinterpret_cast<float*>(w);
    w += align256(sizeof(float) * BH * pr.L * p.LP);
    p.Dt = reinterpret_cast<float*>(w);
    w += align256(sizeof(float) * BH * pr.L * p.LP);
    p.colpart = reinterpret_cast<float*>(w);
  }
  const bool bf = pr.dtype == DT_BF16;
  switch (pr.d) {
    case 16: return bf ? bwd_launch<__nv_bfloat16, 16>(p, s) : bwd_launch<float, 16>(p, s);
    case 32: return bf ? bwd_launch<__nv_bfloat16, 32>(p, s) : bwd_launch<float, 32>(p, s);
    case 64: return bf ? bwd_launch<__nv_bfloat16, 64>(p, s) : bwd_launch<float, 64>(p, s);
    case 128: return bf ? bwd_launch<__nv_bfloat16, 128>(p, s) : bwd_launch<float, 128>(p, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace lion
