// lion_bwd_chunk.cu -- gradients of the LION operator through its chunkwise
// form, for any sequence length, on the CUDA cores in fp32 (d in {16, 32,
// 64, 128}, bfloat16 or float32 inputs).
//
// The gradients are those of the full form (rebuttal page "LION: A
// bidirectional framework that trains like a Transformer and infers like an
// RNN", reply "Concern 1", Theorem 3.3 Eq 25; the forms agree).  Per head,
// with A_ij = M_ij s_ij, num_i = sum_j A_ij [v_j; 1] (its last entry den_i),
// y_i = num_i / den_i and, given dy_i,
//   G_i = [dy_i / den_i ; -(dy_i . y_i) / den_i]          (d + 1 values)
//   dA_ij = G_i . [v_j; 1]
// every gradient is a product of the same masked structure the forward
// scans ("LION Part IV - Results", "LION Chunk"; the recurrences of
// Theorem 3.3 Eq 20-24), once with the states of phi(k) [v; 1]^T and once
// with the states of phi(q) G^T:
//   dphi(q_i) = sum_j M_ij phi(k_j) [v_j; 1]^T G_i
//   dphi(k_j) = sum_i M_ij phi(q_i) G_i^T [v_j; 1]
//   dv_j      = sum_i M_ij (phi(q_i) . phi(k_j)) G_i[0:d]
//   dLoss/dP_m = sum_{j<m} c_mj - sum_{j>m} c_mj + sum_{i<m} c_im - sum_{i>m} c_im,
//                c_ij = A_ij dA_ij,
// with P the inclusive prefix of l = log(lambda), and dl_u = sum_{m>=u}
// dLoss/dP_m (l_0 never enters M).  The row terms of dLoss/dP are phi(q_m)
// against the strict forward / backward phi(k)-states applied to G_m, the
// column terms phi(k_m) against the strict phi(q)G-states applied to
// [v_m; 1].
//
// Chunks of CB tokens (64; 32 at d = 128).  512 threads a CTA.  For chunk c starting at s with
// local inclusive prefix p_t = sum_{u=s}^{t} l_u and total T = p_e:
//   forward summary  U^F_c = sum_{j in c} exp(T - p_j) x_j w_j^T
//   backward summary U^B_c = sum_{j in c} exp(p_j) x_j w_j^T
//   scans            F_{c+1} = exp(T_c) F_c + U^F_c   (F_0 = 0)
//                    B_{c-1} = exp(T_c) B_c + U^B_c   (B_{N-1} = 0)
// so that for a token i of chunk c the tokens left of the chunk contribute
// exp(p_i) F_c and the tokens right of it exp(T - p_i) B_c; inside the chunk
// M_ij = exp(-|p_i - p_j|).  Every decay is <= 1.  States are stored
// transposed, [n][m] (n the [v; 1] or G index, m the feature), in
// (d + 4) x (d + 4) fp32 blocks with zero padding.
//
// Launches: (1) phi(k)[v;1]^T chunk summaries; (2) their scans; (3) per chunk
// the forward recomputed (y, den), G, dphi(q) and dq, the row terms, and the
// phi(q)G^T summaries written over the consumed states; (4) their scans;
// (5) per chunk dphi(k), dk, dv and the column terms; (6) dl from the row
// and column terms (suffix sums for LION-S, the position-weighted sum and
// the batch sum for LION-D), shared with the full-form gradients.
#include "lion_common.cuh"
#include "lion_internal.h"
#include "tile_simt.cuh"

namespace lion {
namespace {

constexpr int kThreads = 512;   // 32 x 16 thread grid for the block products

template <int D>
struct Cfg {
  static constexpr int CB = D >= 128 ? 32 : 64;   // tokens per chunk
  static constexpr int LDT = D + 4;                // row stride of d-wide (and [v;1]) rows
  static constexpr int LDC = CB + 4;               // row stride of chunk-wide rows
  static constexpr int SR = D + 4;                 // state rows (n), padded
  static constexpr int SZ = SR * LDT;              // floats of one stored state
};

struct BcParams {
  const void* q;
  const void* k;
  const void* v;
  const float* log_lambda;
  const float* dy;
  float* dq;
  float* dk;
  float* dv;
  int B, H, L, N;       // N chunks per head
  int mask_kind, phi;
  float* st;            // [BH][N][2][SZ] states (summaries, then scanned)
  float* T;             // [BH][N] chunk totals of l
  float* G;             // [BH][L][LDT] G_i
  float* rowd;          // [BH][L] row terms of dLoss/dP
  float* cold;          // [BH][L] column terms
};

// ---------------------------------------------------------------- products
// Out[a][b] = sum_{k<K} X[a*ldx + k] Y[b*ldy + k] for a < MA, b < NB (the
// "dot" form: the contraction index is contiguous in both operands).  Thread
// (ti, tj) = (t / 16, t % 16) holds a = a0 + ti + 32 alpha (alpha < 2),
// b = b0 + tj + 16 beta (beta < 4) of each 64 x 64 block and reads float4
// along k; K % 4 == 0, ld % 4 == 0.  epi(a, b, value) receives every valid
// output exactly once.
template <typename Epi>
__device__ __forceinline__ void mm_dot(const float* X, int ldx, const float* Y, int ldy, int MA, int NB, int K,
                                       Epi epi) {
  const int ti = threadIdx.x >> 4, tj = threadIdx.x & 15;
  for (int a0 = 0; a0 < MA; a0 += 64) {
    for (int b0 = 0; b0 < NB; b0 += 64) {
      if (a0 + ti >= MA || b0 + tj >= NB) continue;
      float acc[2][4];
#pragma unroll
      for (int x = 0; x < 2; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) acc[x][y] = 0.f;
      const float* xr[2];
      const float* yr[4];
#pragma unroll
      for (int u = 0; u < 2; ++u) xr[u] = X + (size_t)min(a0 + ti + 32 * u, MA - 1) * ldx;
#pragma unroll
      for (int u = 0; u < 4; ++u) yr[u] = Y + (size_t)min(b0 + tj + 16 * u, NB - 1) * ldy;
      for (int k = 0; k < K; k += 4) {
        float4 xv[2], yv[4];
#pragma unroll
        for (int u = 0; u < 2; ++u) xv[u] = *reinterpret_cast<const float4*>(xr[u] + k);
#pragma unroll
        for (int u = 0; u < 4; ++u) yv[u] = *reinterpret_cast<const float4*>(yr[u] + k);
#pragma unroll
        for (int x = 0; x < 2; ++x)
#pragma unroll
          for (int y = 0; y < 4; ++y) {
            acc[x][y] = fmaf(xv[x].x, yv[y].x, acc[x][y]);
            acc[x][y] = fmaf(xv[x].y, yv[y].y, acc[x][y]);
            acc[x][y] = fmaf(xv[x].z, yv[y].z, acc[x][y]);
            acc[x][y] = fmaf(xv[x].w, yv[y].w, acc[x][y]);
          }
      }
#pragma unroll
      for (int x = 0; x < 2; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) {
          const int a = a0 + ti + 32 * x, b = b0 + tj + 16 * y;
          if (a < MA && b < NB) epi(a, b, acc[x][y]);
        }
    }
  }
}

// Out[a][b] = sum_{k<K} w_k X[k*ldx + a] Y[k*ldy + b] (the "outer" form: the
// contraction index is the row of both operands; w == nullptr means 1).
// Thread (ta, tb) holds the contiguous a = a0 + 2 ta + alpha (alpha < 2),
// b = b0 + 4 tb + beta (beta < 4); MA is even and NB a multiple of 4.
template <typename Epi>
__device__ __forceinline__ void mm_outer(const float* X, int ldx, const float* Y, int ldy, const float* w, int MA,
                                         int NB, int K, Epi epi) {
  const int ta = threadIdx.x >> 4, tb = threadIdx.x & 15;
  for (int a0 = 0; a0 < MA; a0 += 64) {
    for (int b0 = 0; b0 < NB; b0 += 64) {
      const int a = a0 + 2 * ta, b = b0 + 4 * tb;
      if (a >= MA || b >= NB) continue;
      float acc[2][4];
#pragma unroll
      for (int x = 0; x < 2; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) acc[x][y] = 0.f;
#pragma unroll 4
      for (int k = 0; k < K; ++k) {
        float2 xv = *reinterpret_cast<const float2*>(X + (size_t)k * ldx + a);
        const float4 yv = *reinterpret_cast<const float4*>(Y + (size_t)k * ldy + b);
        if (w) {
          const float wk = w[k];
          xv = make_float2(xv.x * wk, xv.y * wk);
        }
        const float xs[2] = {xv.x, xv.y}, ys[4] = {yv.x, yv.y, yv.z, yv.w};
#pragma unroll
        for (int x = 0; x < 2; ++x)
#pragma unroll
          for (int y = 0; y < 4; ++y) acc[x][y] = fmaf(xs[x], ys[y], acc[x][y]);
      }
#pragma unroll
      for (int x = 0; x < 2; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) epi(a + x, b + y, acc[x][y]);
    }
  }
}

// ------------------------------------------------------------ chunk setup
// Local inclusive prefix p[t] of l over the chunk's tokens s..s+len-1 (zero
// beyond len), and the chunk total into *T.  Whole block; CB <= 64.
__device__ __forceinline__ void chunk_prefix(const BcParams& p, int bh, int s, int len, float* sp) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const float lh = p.mask_kind == MASK_D ? __ldg(p.log_lambda + bh % p.H) : 0.f;
    float a = 0.f, b = 0.f;
    if (p.mask_kind != MASK_LIT) {
      const int t0 = 2 * lane, t1 = 2 * lane + 1;
      if (p.mask_kind == MASK_S) {
        const float* ll = p.log_lambda + (size_t)bh * p.L + s;
        a = t0 < len ? __ldg(ll + t0) : 0.f;
        b = t1 < len ? __ldg(ll + t1) : 0.f;
      } else {
        a = t0 < len ? lh : 0.f;
        b = t1 < len ? lh : 0.f;
      }
    }
    b += a;
    float x = b;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    const float excl = x - b;
    sp[2 * lane] = a + excl;
    sp[2 * lane + 1] = x;
  }
}

// rows [0, CB) of a token-major tile: the chunk's tokens (converted to fp32)
// and zeros beyond len; row stride LDT, columns D..LDT-1 zero.
template <typename T, int D>
__device__ __forceinline__ void load_tokens(float* dst, const T* src, int s, int len) {
  using C = Cfg<D>;
  for (int idx = threadIdx.x; idx < C::CB * (D / 4); idx += kThreads) {
    const int r = idx / (D / 4), c4 = (idx - r * (D / 4)) * 4;
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (r < len) x = load4(src + (size_t)(s + r) * D + c4);
    *reinterpret_cast<float4*>(dst + r * C::LDT + c4) = x;
  }
  for (int r = threadIdx.x; r < C::CB; r += kThreads)
    *reinterpret_cast<float4*>(dst + r * C::LDT + D) = make_float4(0.f, 0.f, 0.f, 0.f);
}

// [v; 1] rows: v as loaded, 1 in column D for tokens of the chunk.
template <int D>
__device__ __forceinline__ void set_ones(float* vb, int len) {
  using C = Cfg<D>;
  for (int r = threadIdx.x; r < C::CB; r += kThreads) vb[r * C::LDT + D] = r < len ? 1.f : 0.f;
}

template <int D>
__device__ __forceinline__ void load_state(float* dst, const float* src) {
  using C = Cfg<D>;
  for (int x = threadIdx.x * 4; x < C::SZ; x += kThreads * 4)
    *reinterpret_cast<float4*>(dst + x) = *reinterpret_cast<const float4*>(src + x);
}

// Stores the two summaries of one chunk: rows n < D from the block product,
// row D from the column sums of the weighted features (wz_t = 1 for the
// phi(k) states, h_t = G_t[D] for the phi(q) states), padding zero.
//   dst[dir][n][m] = sum_t w^dir_t Xn[t][n] Ym[t][m],  w^0 = exp(T - p_t), w^1 = exp(p_t)
template <int D>
__device__ void write_summaries(float* dst, const float* Xn, const float* Ym, const float* w0, const float* w1,
                                int len) {
  using C = Cfg<D>;
  for (int dir = 0; dir < 2; ++dir) {
    float* out = dst + (size_t)dir * C::SZ;
    const float* w = dir == 0 ? w0 : w1;
    mm_outer(Xn, C::LDT, Ym, C::LDT, w, D, D, C::CB,
             [&](int n, int m, float val) { out[n * C::LDT + m] = val; });
    // row D: four lanes per feature m, tokens strided by four
    for (int m0 = 0; m0 < C::LDT; m0 += kThreads / 4) {
      const int m = m0 + (int)(threadIdx.x >> 2), sub = threadIdx.x & 3;
      float z = 0.f;
      if (m < D)
        for (int t = sub; t < len; t += 4) z = fmaf(w[t] * Xn[t * C::LDT + D], Ym[t * C::LDT + m], z);
      z = group_sum<4>(z);
      if (m < C::LDT && sub == 0) {
        out[D * C::LDT + m] = z;
        for (int n = D + 1; n < C::SR; ++n) out[n * C::LDT + m] = 0.f;
      }
    }
    for (int x = threadIdx.x; x < D; x += kThreads)
      *reinterpret_cast<float4*>(out + x * C::LDT + D) = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// (1) phi(k)[v;1]^T summaries of every chunk, and the chunk totals.
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) bwc_summary_kernel(BcParams p) {
  using C = Cfg<D>;
  extern __shared__ float4 smem4[];
  float* sm = reinterpret_cast<float*>(smem4);
  float* Kf = sm;                       // [CB][LDT]
  float* Vb = Kf + C::CB * C::LDT;      // [CB][LDT]
  float* sp = Vb + C::CB * C::LDT;      // [64] prefix
  float* w0 = sp + 64;                  // [CB] exp(T - p_t)
  float* w1 = w0 + C::CB;               // [CB] exp(p_t)
  const int c = (int)(blockIdx.x % (unsigned)p.N), bh = (int)(blockIdx.x / (unsigned)p.N), L = p.L;
  const int s = c * C::CB, len = min(C::CB, L - s);
  chunk_prefix(p, bh, s, len, sp);
  load_tokens<T, D>(Kf, reinterpret_cast<const T*>(p.k) + (size_t)bh * L * D, s, len);
  load_tokens<T, D>(Vb, reinterpret_cast<const T*>(p.v) + (size_t)bh * L * D, s, len);
  __syncthreads();
  set_ones<D>(Vb, len);
  phi_rows_inplace(Kf, C::CB, len, D, C::LDT, p.phi);
  const float Tc = sp[len - 1];
  for (int t = threadIdx.x; t < C::CB; t += kThreads) {
    w0[t] = t < len ? expf(Tc - sp[t]) : 0.f;
    w1[t] = t < len ? expf(sp[t]) : 0.f;
  }
  if (threadIdx.x == 0) p.T[(size_t)bh * p.N + c] = Tc;
  __syncthreads();
  write_summaries<D>(p.st + ((size_t)bh * p.N + c) * 2 * C::SZ, Vb, Kf, w0, w1, len);
}

// (2), (4) the scans: F_c (dir 0, from the left) and B_c (dir 1, from the
// right) replace the summaries in place.  One thread per state element,
// with the loads of U chunks in flight at once (16 for long sequences, 4 for
// short ones, where more registers would only cost resident CTAs).
template <int D, int U>
__global__ void __launch_bounds__(kThreads) bwc_scan_kernel(BcParams p) {
  using C = Cfg<D>;
  constexpr int NB = (C::SZ + kThreads - 1) / kThreads;   // blocks per state
  const int blk = (int)(blockIdx.x % NB), bh = (int)(blockIdx.x / NB), dir = blockIdx.y;
  const int x = blk * kThreads + threadIdx.x;
  if (x >= C::SZ) return;
  const int N = p.N;
  float* base = p.st + (size_t)bh * N * 2 * C::SZ + (size_t)dir * C::SZ + x;
  const float* Tt = p.T + (size_t)bh * N;
  float run = 0.f;
  for (int n0 = 0; n0 < N; n0 += U) {
    float u[U], e[U];
#pragma unroll
    for (int r = 0; r < U; ++r) {
      const int n = n0 + r, c = dir == 0 ? n : N - 1 - n;
      u[r] = n < N ? base[(size_t)c * 2 * C::SZ] : 0.f;
      e[r] = n < N ? __expf(Tt[c]) : 0.f;
    }
#pragma unroll
    for (int r = 0; r < U; ++r) {
      const int n = n0 + r, c = dir == 0 ? n : N - 1 - n;
      if (n < N) {
        base[(size_t)c * 2 * C::SZ] = run;
        run = fmaf(run, e[r], u[r]);
      }
    }
  }
}

template <int D>
constexpr size_t rows_smem_floats() {
  using C = Cfg<D>;
  return 5 * (size_t)C::CB * C::LDT + (size_t)C::SR * C::LDC + 2 * (size_t)C::CB * C::LDC + C::SZ + 64 + 6 * C::CB;
}

// (3) per chunk: num and den recomputed, G, dphi(q) -> dq, the row terms,
// and the phi(q) G^T summaries over the consumed phi(k) states.
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) bwc_rows_kernel(BcParams p) {
  using C = Cfg<D>;
  constexpr int CB = C::CB, LDT = C::LDT, LDC = C::LDC;
  extern __shared__ float4 smem4[];
  float* sm = reinterpret_cast<float*>(smem4);
  float* Qf = sm;                  // [CB][LDT] phi(q)
  float* Kf = Qf + CB * LDT;       // [CB][LDT] phi(k)
  float* Vb = Kf + CB * LDT;       // [CB][LDT] [v; 1]
  float* Gb = Vb + CB * LDT;       // [CB][LDT] num, then G
  float* Dq = Gb + CB * LDT;       // [CB][LDT] dphi(q)
  float* Gt = Dq + CB * LDT;       // [SR][LDC] G transposed
  float* At = Gt + C::SR * LDC;    // [CB][LDC] A transposed: At[j][i] = A_ij
  float* Dt = At + CB * LDC;       // [CB][LDC] (M (.) dA) transposed
  float* St = Dt + CB * LDC;       // [SR][LDT] one state
  float* sp = St + C::SZ;          // [64]
  float* wl = sp + 64;             // [CB] exp(p_i)
  float* wr = wl + CB;             // [CB] exp(T - p_i)
  float* den = wr + CB;            // [CB]
  float* rowt = den + CB;          // [CB]
  float* dyy = rowt + CB;          // [CB] dy_i . y_i
  const int c = (int)(blockIdx.x % (unsigned)p.N), bh = (int)(blockIdx.x / (unsigned)p.N), L = p.L;
  const int s = c * CB, len = min(CB, L - s);
  const size_t tok0 = (size_t)bh * L + s;
  float* stc = p.st + ((size_t)bh * p.N + c) * 2 * C::SZ;

  chunk_prefix(p, bh, s, len, sp);
  load_tokens<T, D>(Qf, reinterpret_cast<const T*>(p.q) + (size_t)bh * L * D, s, len);
  load_tokens<T, D>(Kf, reinterpret_cast<const T*>(p.k) + (size_t)bh * L * D, s, len);
  load_tokens<T, D>(Vb, reinterpret_cast<const T*>(p.v) + (size_t)bh * L * D, s, len);
  __syncthreads();
  set_ones<D>(Vb, len);
  phi_rows_inplace(Qf, CB, len, D, LDT, p.phi);
  phi_rows_inplace(Kf, CB, len, D, LDT, p.phi);
  const float Tc = sp[len - 1];
  for (int t = threadIdx.x; t < CB; t += kThreads) {
    wl[t] = t < len ? expf(sp[t]) : 0.f;
    wr[t] = t < len ? expf(Tc - sp[t]) : 0.f;
    rowt[t] = 0.f;
  }
  __syncthreads();

  // A_ij = M_ij s_ij inside the chunk (transposed store), zero outside it
  mm_dot(Qf, LDT, Kf, LDT, CB, CB, D, [&](int i, int j, float sv) {
    At[j * LDC + i] = (i < len && j < len) ? sv * expf(-fabsf(sp[i] - sp[j])) : 0.f;
  });
  __syncthreads();
  // num[i][n] (n < D) = sum_j A_ij v_j, then the states' parts
  mm_outer(At, LDC, Vb, LDT, nullptr, CB, D, CB, [&](int i, int n, float val) { Gb[i * LDT + n] = val; });
  // the chunk's dy rows, staged in the dphi(q) buffer (not yet in use)
  const float* dyh = p.dy + tok0 * D;
  for (int x = threadIdx.x; x < CB * (D / 4); x += kThreads) {
    const int i = x / (D / 4), c4 = (x - i * (D / 4)) * 4;
    *reinterpret_cast<float4*>(Dq + i * LDT + c4) =
        i < len ? *reinterpret_cast<const float4*>(dyh + (size_t)i * D + c4) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  // four lanes per row below (CB <= 64 rows for 256 threads)
  const int r4 = (int)(threadIdx.x >> 2), s4 = threadIdx.x & 3;
  {
    float a = 0.f;
    if (r4 < CB)
      for (int j = s4; j < len; j += 4) a += At[j * LDC + r4];
    a = group_sum<4>(a);
    if (r4 < CB && s4 == 0) den[r4] = a;
  }
  for (int dir = 0; dir < 2; ++dir) {
    __syncthreads();
    load_state<D>(St, stc + (size_t)dir * C::SZ);
    __syncthreads();
    const float* w = dir == 0 ? wl : wr;
    mm_dot(Qf, LDT, St, LDT, CB, D, D, [&](int i, int n, float val) { Gb[i * LDT + n] += w[i] * val; });
    float a = 0.f;
    if (r4 < CB)
      for (int m = s4; m < D; m += 4) a = fmaf(Qf[r4 * LDT + m], St[D * LDT + m], a);
    a = group_sum<4>(a);
    if (r4 < CB && s4 == 0) den[r4] += w[r4] * a;
  }
  __syncthreads();
  // G_i = [dy_i / den_i ; -(dy_i . y_i) / den_i]; rows past the chunk 0
  {
    float a = 0.f;
    if (r4 < len)
      for (int n = s4; n < D; n += 4) a = fmaf(Dq[r4 * LDT + n], Gb[r4 * LDT + n], a);
    a = group_sum<4>(a);
    if (r4 < CB && s4 == 0) dyy[r4] = r4 < len ? a / den[r4] : 0.f;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < CB * LDT; idx += kThreads) {
    const int i = idx / LDT, n = idx - i * LDT;
    float g = 0.f;
    if (i < len) {
      const float inv = 1.f / den[i];
      g = n < D ? Dq[i * LDT + n] * inv : n == D ? -dyy[i] * inv : 0.f;
    }
    Gb[idx] = g;
    Gt[n * LDC + i] = g;
    if (i < len) p.G[(tok0 + i) * LDT + n] = g;
  }
  __syncthreads();

  // dA_ij = G_i . [v_j; 1]: the masked copy for dphi(q), and the row terms
  // sum_{j<i} c_ij - sum_{j>i} c_ij, c_ij = A_ij dA_ij
  {
    float part[2] = {0.f, 0.f};
    const int ti = threadIdx.x >> 4;
    mm_dot(Gb, LDT, Vb, LDT, CB, CB, LDT, [&](int i, int j, float da) {
      const float a = At[j * LDC + i];
      Dt[j * LDC + i] = (i < len && j < len) ? da * expf(-fabsf(sp[i] - sp[j])) : 0.f;
      const float cij = a * da;
      part[(i - ti) >> 5] += j < i ? cij : j > i ? -cij : 0.f;
    });
    // the 16 lanes with the same ti hold rows ti + 32 alpha
#pragma unroll
    for (int x = 0; x < 2; ++x) part[x] = group_sum<16>(part[x]);
    if ((threadIdx.x & 15) == 0)
#pragma unroll
      for (int x = 0; x < 2; ++x)
        if (ti + 32 * x < CB) rowt[ti + 32 * x] += part[x];
  }
  __syncthreads();
  // dphi(q_i) = sum_j M_ij dA_ij phi(k_j), then the states' parts; the row
  // terms' state parts are phi(q_i) . (its forward part) - phi(q_i) . (backward)
  mm_outer(Dt, LDC, Kf, LDT, nullptr, CB, D, CB, [&](int i, int m, float val) { Dq[i * LDT + m] = val; });
  for (int dir = 0; dir < 2; ++dir) {
    __syncthreads();
    load_state<D>(St, stc + (size_t)dir * C::SZ);
    __syncthreads();
    const float* w = dir == 0 ? wl : wr;
    const float sgn = dir == 0 ? 1.f : -1.f;
    float part[2] = {0.f, 0.f};
    const int ta = threadIdx.x >> 4;
    mm_outer(Gt, LDC, St, LDT, nullptr, CB, D, C::SR, [&](int i, int m, float val) {
      const float x = w[i] * val;
      Dq[i * LDT + m] += x;
      part[i & 1] += Qf[i * LDT + m] * x;
    });
    // lanes with the same ta share rows 2 ta, 2 ta + 1 (per 64-column block a
    // lane adds once per block, so the sums below cover every column)
#pragma unroll
    for (int x = 0; x < 2; ++x) part[x] = group_sum<16>(part[x]);
    if ((threadIdx.x & 15) == 0)
#pragma unroll
      for (int x = 0; x < 2; ++x)
        if (2 * ta + x < CB) rowt[2 * ta + x] += sgn * part[x];
  }
  __syncthreads();
  // the phi(q) G^T summaries over this chunk's (consumed) states
  write_summaries<D>(stc, Gb, Qf, wr, wl, len);
  // dq = J_phi(q)^T dphi(q), row by row (W lanes a row, D / W features each)
  {
    constexpr int W = D / 4 < 16 ? D / 4 : 16, NC = D / W;
    const T* qh = reinterpret_cast<const T*>(p.q) + tok0 * D;
    for (int r0 = 0; r0 < CB; r0 += kThreads / W) {
      const int i = r0 + (int)threadIdx.x / W, c0 = ((int)threadIdx.x % W) * NC;
      const bool ok = i < len;
      float x[NC], g[NC], dx[NC];
#pragma unroll
      for (int e = 0; e < NC; ++e) {
        x[e] = ok ? to_f32(qh[(size_t)i * D + c0 + e]) : 0.f;
        g[e] = ok ? Dq[i * LDT + c0 + e] : 0.f;
      }
      phi_backward<NC, W>(p.phi, x, g, dx);
      if (ok)
#pragma unroll
        for (int e = 0; e < NC; ++e) p.dq[(tok0 + i) * D + c0 + e] = dx[e];
    }
  }
  for (int i = threadIdx.x; i < len; i += kThreads) p.rowd[tok0 + i] = rowt[i];
}

template <int D>
constexpr size_t cols_smem_floats() {
  using C = Cfg<D>;
  return 6 * (size_t)C::CB * C::LDT + (size_t)C::SR * C::LDC + 2 * (size_t)C::CB * C::LDC + C::SZ + 64 +
         (3 + kThreads / 32) * C::CB;
}

// (5) per chunk: dphi(k) -> dk, dv and the column terms.
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) bwc_cols_kernel(BcParams p) {
  using C = Cfg<D>;
  constexpr int CB = C::CB, LDT = C::LDT, LDC = C::LDC;
  extern __shared__ float4 smem4[];
  float* sm = reinterpret_cast<float*>(smem4);
  float* Qf = sm;                  // [CB][LDT] phi(q)
  float* Kf = Qf + CB * LDT;       // [CB][LDT] phi(k)
  float* Vb = Kf + CB * LDT;       // [CB][LDT] [v; 1]
  float* Gb = Vb + CB * LDT;       // [CB][LDT] G
  float* Dk = Gb + CB * LDT;       // [CB][LDT] dphi(k)
  float* Dv = Dk + CB * LDT;       // [CB][LDT] dv
  float* Vt = Dv + CB * LDT;       // [SR][LDC] [v; 1] transposed
  float* Am = Vt + C::SR * LDC;    // [CB][LDC] A_ij (row i)
  float* Dm = Am + CB * LDC;       // [CB][LDC] M_ij dA_ij (row i)
  float* St = Dm + CB * LDC;       // [SR][LDT] one state
  float* sp = St + C::SZ;          // [64]
  float* wl = sp + 64;             // [CB]
  float* wr = wl + CB;             // [CB]
  float* colt = wr + CB;           // [CB]
  float* cpart = colt + CB;        // [warps][CB] per-warp column sums
  const int c = (int)(blockIdx.x % (unsigned)p.N), bh = (int)(blockIdx.x / (unsigned)p.N), L = p.L;
  const int s = c * CB, len = min(CB, L - s);
  const size_t tok0 = (size_t)bh * L + s;
  const float* stc = p.st + ((size_t)bh * p.N + c) * 2 * C::SZ;

  chunk_prefix(p, bh, s, len, sp);
  load_tokens<T, D>(Qf, reinterpret_cast<const T*>(p.q) + (size_t)bh * L * D, s, len);
  load_tokens<T, D>(Kf, reinterpret_cast<const T*>(p.k) + (size_t)bh * L * D, s, len);
  load_tokens<T, D>(Vb, reinterpret_cast<const T*>(p.v) + (size_t)bh * L * D, s, len);
  for (int idx = threadIdx.x * 4; idx < CB * LDT; idx += kThreads * 4) {
    const int i = idx / LDT;
    float4 g = make_float4(0.f, 0.f, 0.f, 0.f);
    if (i < len) g = *reinterpret_cast<const float4*>(p.G + tok0 * LDT + idx);
    *reinterpret_cast<float4*>(Gb + idx) = g;
  }
  __syncthreads();
  set_ones<D>(Vb, len);
  phi_rows_inplace(Qf, CB, len, D, LDT, p.phi);
  phi_rows_inplace(Kf, CB, len, D, LDT, p.phi);
  const float Tc = sp[len - 1];
  for (int t = threadIdx.x; t < CB; t += kThreads) {
    wl[t] = t < len ? expf(sp[t]) : 0.f;
    wr[t] = t < len ? expf(Tc - sp[t]) : 0.f;
    colt[t] = 0.f;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < CB * LDT; idx += kThreads) {
    const int j = idx / LDT, n = idx - j * LDT;
    Vt[n * LDC + j] = Vb[idx];
  }
  mm_dot(Qf, LDT, Kf, LDT, CB, CB, D, [&](int i, int j, float sv) {
    Am[i * LDC + j] = (i < len && j < len) ? sv * expf(-fabsf(sp[i] - sp[j])) : 0.f;
  });
  __syncthreads();
  // dA_ij: the masked copy, and the column terms sum_{i<j} c_ij - sum_{i>j} c_ij
  {
    float part[4] = {0.f, 0.f, 0.f, 0.f};
    const int tj = threadIdx.x & 15;
    mm_dot(Gb, LDT, Vb, LDT, CB, CB, LDT, [&](int i, int j, float da) {
      Dm[i * LDC + j] = (i < len && j < len) ? da * expf(-fabsf(sp[i] - sp[j])) : 0.f;
      const float cij = Am[i * LDC + j] * da;
      part[(j - tj) >> 4] += i < j ? cij : i > j ? -cij : 0.f;
    });
    // lanes tj and tj + 16 of a warp share columns; the warps' sums are
    // added in warp order (deterministic)
#pragma unroll
    for (int x = 0; x < 4; ++x) part[x] += __shfl_xor_sync(0xffffffffu, part[x], 16);
    if ((threadIdx.x & 31) < 16)
#pragma unroll
      for (int x = 0; x < 4; ++x)
        if (tj + 16 * x < CB) cpart[(threadIdx.x >> 5) * CB + tj + 16 * x] = part[x];
  }
  __syncthreads();
  for (int j = threadIdx.x; j < CB; j += kThreads) {
    float a = 0.f;
#pragma unroll
    for (int wv = 0; wv < kThreads / 32; ++wv) a += cpart[wv * CB + j];
    colt[j] = a;
  }
  // dphi(k_j) = sum_i M_ij dA_ij phi(q_i);  dv_j = sum_i A_ij G_i[0:D]
  mm_outer(Dm, LDC, Qf, LDT, nullptr, CB, D, CB, [&](int j, int m, float val) { Dk[j * LDT + m] = val; });
  mm_outer(Am, LDC, Gb, LDT, nullptr, CB, D, CB, [&](int j, int n, float val) { Dv[j * LDT + n] = val; });
  for (int dir = 0; dir < 2; ++dir) {
    __syncthreads();
    load_state<D>(St, stc + (size_t)dir * C::SZ);
    __syncthreads();
    const float* w = dir == 0 ? wl : wr;
    const float sgn = dir == 0 ? 1.f : -1.f;
    float part[2] = {0.f, 0.f};
    const int ta = threadIdx.x >> 4;
    mm_outer(Vt, LDC, St, LDT, nullptr, CB, D, C::SR, [&](int j, int m, float val) {
      const float x = w[j] * val;
      Dk[j * LDT + m] += x;
      part[j & 1] += Kf[j * LDT + m] * x;
    });
#pragma unroll
    for (int x = 0; x < 2; ++x) part[x] = group_sum<16>(part[x]);
    if ((threadIdx.x & 15) == 0)
#pragma unroll
      for (int x = 0; x < 2; ++x)
        if (2 * ta + x < CB) colt[2 * ta + x] += sgn * part[x];
    __syncthreads();
    mm_dot(Kf, LDT, St, LDT, CB, D, D, [&](int j, int n, float val) { Dv[j * LDT + n] += w[j] * val; });
  }
  __syncthreads();
  {
    constexpr int W = D / 4 < 16 ? D / 4 : 16, NC = D / W;
    const T* kh = reinterpret_cast<const T*>(p.k) + tok0 * D;
    for (int r0 = 0; r0 < CB; r0 += kThreads / W) {
      const int j = r0 + (int)threadIdx.x / W, c0 = ((int)threadIdx.x % W) * NC;
      const bool ok = j < len;
      float x[NC], g[NC], dx[NC];
#pragma unroll
      for (int e = 0; e < NC; ++e) {
        x[e] = ok ? to_f32(kh[(size_t)j * D + c0 + e]) : 0.f;
        g[e] = ok ? Dk[j * LDT + c0 + e] : 0.f;
      }
      phi_backward<NC, W>(p.phi, x, g, dx);
      if (ok)
#pragma unroll
        for (int e = 0; e < NC; ++e) {
          p.dk[(tok0 + j) * D + c0 + e] = dx[e];
          p.dv[(tok0 + j) * D + c0 + e] = Dv[j * LDT + c0 + e];
        }
    }
  }
  for (int j = threadIdx.x; j < len; j += kThreads) p.cold[tok0 + j] = colt[j];
}

template <typename Kern>
cudaError_t allow_smem(Kern kern, size_t bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <typename T, int D>
cudaError_t bwc_launch(const BcParams& p, cudaStream_t s) {
  using C = Cfg<D>;
  const int BH = p.B * p.H;
  // one CTA per (head, chunk) and per (head, 256 state elements), on the x axis
  const dim3 gchunks((unsigned)((size_t)p.N * BH)), gscan((unsigned)((size_t)BH * ((C::SZ + kThreads - 1) / kThreads)), 2);
  const size_t sm1 = sizeof(float) * (2 * (size_t)C::CB * C::LDT + 64 + 2 * C::CB);
  const size_t sm3 = sizeof(float) * rows_smem_floats<D>();
  const size_t sm5 = sizeof(float) * cols_smem_floats<D>();
  cudaError_t e;
  if ((e = allow_smem(bwc_summary_kernel<T, D>, sm1)) != cudaSuccess) return e;
  if ((e = allow_smem(bwc_rows_kernel<T, D>, sm3)) != cudaSuccess) return e;
  if ((e = allow_smem(bwc_cols_kernel<T, D>, sm5)) != cudaSuccess) return e;
  auto scan = p.N >= 32 ? bwc_scan_kernel<D, 16> : bwc_scan_kernel<D, 4>;
  bwc_summary_kernel<T, D><<<gchunks, kThreads, sm1, s>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  scan<<<gscan, kThreads, 0, s>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  bwc_rows_kernel<T, D><<<gchunks, kThreads, sm3, s>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  scan<<<gscan, kThreads, 0, s>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  bwc_cols_kernel<T, D><<<gchunks, kThreads, sm5, s>>>(p);
  return cudaGetLastError();
}

size_t al256(size_t x) { return (x + 255) & ~(size_t)255; }

int chunk_of(int d) { return d >= 128 ? 32 : 64; }
int ldt_of(int d) { return d + 4; }
size_t state_floats(int d) { return (size_t)(d + 4) * (d + 4); }

}  // namespace

int bwd_chunk_length(int d) { return chunk_of(d); }

size_t bwd_chunk_workspace_bytes(int B, int H, int L, int d) {
  const size_t BH = (size_t)B * H, N = (size_t)(L + chunk_of(d) - 1) / chunk_of(d);
  return al256(sizeof(float) * BH * N * 2 * state_floats(d)) + al256(sizeof(float) * BH * N) +
         al256(sizeof(float) * BH * L * ldt_of(d)) + 2 * al256(sizeof(float) * BH * L) + al256(sizeof(double) * BH);
}

int bwd_chunk_launches(int mask_kind) { return 5 + (mask_kind != MASK_LIT) + (mask_kind == MASK_D); }

cudaError_t launch_bwd_chunk(const Problem& pr, const float* dy, float* dq, float* dk, float* dv, float* dll,
                             void* ws, cudaStream_t s) {
  BcParams p;
  p.q = pr.q;
  p.k = pr.k;
  p.v = pr.v;
  p.log_lambda = pr.log_lambda;
  p.dy = dy;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.B = pr.B;
  p.H = pr.H;
  p.L = pr.L;
  p.N = (pr.L + chunk_of(pr.d) - 1) / chunk_of(pr.d);
  p.mask_kind = pr.mask_kind;
  p.phi = pr.phi;
  const size_t BH = (size_t)pr.B * pr.H;
  uint8_t* w = static_cast<uint8_t*>(ws);
  p.st = reinterpret_cast<float*>(w);
  w += al256(sizeof(float) * BH * p.N * 2 * state_floats(pr.d));
  p.T = reinterpret_cast<float*>(w);
  w += al256(sizeof(float) * BH * p.N);
  p.G = reinterpret_cast<float*>(w);
  w += al256(sizeof(float) * BH * pr.L * ldt_of(pr.d));
  p.rowd = reinterpret_cast<float*>(w);
  w += al256(sizeof(float) * BH * pr.L);
  p.cold = reinterpret_cast<float*>(w);
  w += al256(sizeof(float) * BH * pr.L);
  double* dsum = reinterpret_cast<double*>(w);
  const bool bf = pr.dtype == DT_BF16;
  cudaError_t e = cudaErrorInvalidValue;
  switch (pr.d) {
    case 16: e = bf ? bwc_launch<__nv_bfloat16, 16>(p, s) : bwc_launch<float, 16>(p, s); break;
    case 32: e = bf ? bwc_launch<__nv_bfloat16, 32>(p, s) : bwc_launch<float, 32>(p, s); break;
    case 64: e = bf ? bwc_launch<__nv_bfloat16, 64>(p, s) : bwc_launch<float, 64>(p, s); break;
    case 128: e = bf ? bwc_launch<__nv_bfloat16, 128>(p, s) : bwc_launch<float, 128>(p, s); break;
  }
  if (e != cudaSuccess || pr.mask_kind == MASK_LIT) return e;
  return launch_dlog_lambda(pr.B, pr.H, pr.L, pr.mask_kind, p.rowd, p.cold, dsum, dll, s);
}

}  // namespace lion
