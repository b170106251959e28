// lion_chunk_tile.cu -- the chunkwise form of the LION operator on the CUDA
// cores for chunks of at most 64 tokens (fp32 arithmetic, d in {16, 32, 64,
// 128}, bfloat16 or float32 inputs): one CTA per head, the chunk's tiles and
// the d x (d + 1) state in shared memory, and every step a register-tiled
// block product.
//
// Chunkwise form ("LION Part IV - Results", "LION Chunk"; rebuttal page
// "LION: A bidirectional framework that trains like a Transformer and infers
// like an RNN", Theorem 3.3 Eq 20-24 taken a chunk at a time).  Per head,
// chunk c covers tokens [s_c, e_c]; p is the chunk-local inclusive prefix of
// l = log(lambda) and T_c = p at e_c:
//   right to left, the state G_c of the tokens after the chunk (anchored at
//   s_{c+1}):
//     num_i += b_i phi(q_i) [G_c],  b_i = exp(T_c - p_i + l_{s_{c+1}})
//     G_{c-1} = exp(T_c - l_{s_c} + l_{s_{c+1}}) G_c
//               + sum_{j in c} exp(p_j - l_{s_c}) phi(k_j) [v_j; 1]^T
//   left to right, the state F_c of the tokens before it (anchored at
//   e_{c-1}), and the chunk itself:
//     num_i += sum_{j in c} exp(-|p_i - p_j|) s_ij [v_j; 1] + a_i phi(q_i) [F_c],
//     a_i = exp(p_i),  F_{c+1} = exp(T_c) F_c + sum_{j in c} exp(T_c - p_j) phi(k_j) [v_j; 1]^T
//   y_i = num_i[0:d] / num_i[d].
// Every decay is at most 1.  The right-to-left sweep parks its part of num
// in `out` (the values) and the workspace (the normaliser); the
// left-to-right sweep adds its own and divides.  With Problem::causal only
// the left-to-right sweep runs, with j <= i inside the chunk.
//
// phi(q) and phi(k) of every token go to the workspace first (one launch,
// the same kernel as the full form's), so that the two sweeps read fp32
// features as float4 rows and compute no feature map.
//
// Products (256 threads as a 16 x 16 grid, 4 x 4 outputs a thread, float4
// operand reads from shared memory): "dot" when the contraction index is
// contiguous in both operands (scores, the state applied to the queries),
// "outer" when it is the row index of both (scores times values, the state
// update).  The normaliser column (the 1 of [v; 1], the z row of a state)
// is summed apart, so that each product covers exactly d columns.
#include "lion_common.cuh"
#include "lion_internal.h"
#include "tile_simt.cuh"

namespace lion {
namespace {

constexpr int kThr = 256;

template <int D, int CT>
struct TileCfg {
  static constexpr int LD = D + 4;       // row stride of d-wide rows (column d: the 1 of [v; 1])
  static constexpr int LDS = CT + 4;     // row stride of the transposed scores
  static constexpr int SR = D + 4;       // state rows: d value columns, z, padding
  static constexpr size_t floats = 4 * (size_t)CT * LD + (size_t)SR * LD + (size_t)CT * LDS + 3 * CT + 4;
};

// out[a][b] = sum_{k<K} X[a*ldx + k] Y[b*ldy + k] for a < MA, b < NB.  Thread
// (ti, tj) holds a = a0 + ti + 16 alpha (alpha < RA), b = b0 + tj + 16 beta
// (beta < RB) of each (16 RA) x (16 RB) block, so that a chunk of 16 or 32
// rows takes one or two rows a thread; K % 4 == 0.  epi(a, b, value) sees
// every output once.
template <int RA, int RB, typename Epi>
__device__ __forceinline__ void dot_tiles(const float* X, int ldx, const float* Y, int ldy, int MA, int NB, int K,
                                          Epi epi) {
  const int ti = threadIdx.x >> 4, tj = threadIdx.x & 15;
  for (int a0 = 0; a0 < MA; a0 += 16 * RA) {
    for (int b0 = 0; b0 < NB; b0 += 16 * RB) {
      if (a0 + ti >= MA || b0 + tj >= NB) continue;
      float acc[RA][RB];
#pragma unroll
      for (int x = 0; x < RA; ++x)
#pragma unroll
        for (int y = 0; y < RB; ++y) acc[x][y] = 0.f;
      const float* xr[RA];
      const float* yr[RB];
#pragma unroll
      for (int u = 0; u < RA; ++u) xr[u] = X + (size_t)min(a0 + ti + 16 * u, MA - 1) * ldx;
#pragma unroll
      for (int u = 0; u < RB; ++u) yr[u] = Y + (size_t)min(b0 + tj + 16 * u, NB - 1) * ldy;
      for (int k = 0; k < K; k += 4) {
        float4 xv[RA], yv[RB];
#pragma unroll
        for (int u = 0; u < RA; ++u) xv[u] = *reinterpret_cast<const float4*>(xr[u] + k);
#pragma unroll
        for (int u = 0; u < RB; ++u) yv[u] = *reinterpret_cast<const float4*>(yr[u] + k);
#pragma unroll
        for (int x = 0; x < RA; ++x)
#pragma unroll
          for (int y = 0; y < RB; ++y) {
            acc[x][y] = fmaf(xv[x].x, yv[y].x, acc[x][y]);
            acc[x][y] = fmaf(xv[x].y, yv[y].y, acc[x][y]);
            acc[x][y] = fmaf(xv[x].z, yv[y].z, acc[x][y]);
            acc[x][y] = fmaf(xv[x].w, yv[y].w, acc[x][y]);
          }
      }
#pragma unroll
      for (int x = 0; x < RA; ++x)
#pragma unroll
        for (int y = 0; y < RB; ++y) {
          const int a = a0 + ti + 16 * x, b = b0 + tj + 16 * y;
          if (a < MA && b < NB) epi(a, b, acc[x][y]);
        }
    }
  }
}

// out[a][b] = sum_{k<K} w_k X[k*ldx + a] Y[k*ldy + b] (w == nullptr: 1).
// Thread (ti, tj) holds the contiguous a = a0 + 4 ti + alpha, b = b0 + 4 tj
// + beta; MA and NB are multiples of 4.
template <typename Epi>
__device__ __forceinline__ void outer_tiles(const float* X, int ldx, const float* Y, int ldy, const float* w,
                                            int MA, int NB, int K, Epi epi) {
  const int ti = threadIdx.x >> 4, tj = threadIdx.x & 15;
  for (int a0 = 0; a0 < MA; a0 += 64) {
    for (int b0 = 0; b0 < NB; b0 += 64) {
      const int a = a0 + 4 * ti, b = b0 + 4 * tj;
      if (a >= MA || b >= NB) continue;
      float acc[4][4];
#pragma unroll
      for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) acc[x][y] = 0.f;
#pragma unroll 4
      for (int k = 0; k < K; ++k) {
        float4 xv = *reinterpret_cast<const float4*>(X + (size_t)k * ldx + a);
        const float4 yv = *reinterpret_cast<const float4*>(Y + (size_t)k * ldy + b);
        if (w) {
          const float wk = w[k];
          xv = make_float4(xv.x * wk, xv.y * wk, xv.z * wk, xv.w * wk);
        }
        const float xs[4] = {xv.x, xv.y, xv.z, xv.w}, ys[4] = {yv.x, yv.y, yv.z, yv.w};
#pragma unroll
        for (int x = 0; x < 4; ++x)
#pragma unroll
          for (int y = 0; y < 4; ++y) acc[x][y] = fmaf(xs[x], ys[y], acc[x][y]);
      }
#pragma unroll
      for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) epi(a + x, b + y, acc[x][y]);
    }
  }
}

// Rows [s, s + len) of a token-major [L][D] tensor into a [CT][LD] fp32 tile,
// four features a thread, zero beyond len.
template <typename T, int D, int CT>
__device__ __forceinline__ void load_tile(float* dst, const T* src, int s, int len) {
  constexpr int LD = TileCfg<D, CT>::LD, V = D / 4;
  for (int idx = threadIdx.x; idx < CT * V; idx += kThr) {
    const int r = idx / V, m = (idx - r * V) * 4;
    *reinterpret_cast<float4*>(dst + r * LD + m) =
        r < len ? load4(src + (size_t)(s + r) * D + m) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// Workspace (floats, each section padded to 64): the right-to-left sweep's
// normalisers [BH L], phi(q) [BH L d], phi(k) [BH L d].
__host__ __device__ constexpr size_t pad64(size_t n) { return (n + 63) & ~size_t(63); }
struct TileWs {
  size_t den, fq, fk, total;
  __host__ __device__ TileWs(size_t BHL, int d) {
    den = 0;
    fq = pad64(BHL);
    fk = fq + pad64(BHL * (size_t)d);
    total = fk + pad64(BHL * (size_t)d);
  }
};

template <typename T, int D, int CT>
__global__ void __launch_bounds__(kThr) chunk_tile_kernel(Problem p, float* ws) {
  using C = TileCfg<D, CT>;
  constexpr int LD = C::LD, LDS = C::LDS;
  constexpr int RC = CT / 16;                 // chunk rows (or columns) a thread in a dot product
  constexpr int RD = D >= 64 ? 4 : D / 16;    // feature columns a thread
  extern __shared__ float4 smem4[];
  float* sm = reinterpret_cast<float*>(smem4);
  float* sQ = sm;                     // [CT][LD] phi(q)
  float* sK = sQ + CT * LD;           // [CT][LD] phi(k)
  float* sV = sK + CT * LD;           // [CT][LD] [v; 1]
  float* sAcc = sV + CT * LD;         // [CT][LD] num (column D: den)
  float* sSt = sAcc + CT * LD;        // [SR][LD] state, row n = column n of [v; 1], columns = features
  float* sS = sSt + C::SR * LD;       // [CT][LDS] masked scores, transposed: sS[j][i]
  float* sP = sS + CT * LDS;          // [CT] chunk-local inclusive prefix
  float* sW = sP + CT;                // [CT] state weights of the chunk's keys
  float* sR = sW + CT;                // [CT] state factors of the chunk's queries
  float* sLn = sR + CT;               // [1] l at the token after the chunk

  const int L = p.L, H = p.H, Cr = p.chunk, bh = blockIdx.x;
  const int N = (L + Cr - 1) / Cr;
  const TileWs w((size_t)p.B * H * L, D);
  const float* fq = ws + w.fq + (size_t)bh * L * D;
  const float* fk = ws + w.fk + (size_t)bh * L * D;
  const T* v = reinterpret_cast<const T*>(p.v) + (size_t)bh * L * D;
  float* out = p.out + (size_t)bh * L * D;
  float* den = ws + w.den + (size_t)bh * L;
  const float* ll = p.mask_kind == MASK_S ? p.log_lambda + (size_t)bh * L : nullptr;
  const float lh = p.mask_kind == MASK_D ? __ldg(p.log_lambda + bh % H) : 0.f;
  auto ell = [&](int t) -> float { return ll ? __ldg(ll + t) : lh; };

  for (int sweep = p.causal ? 1 : 0; sweep < 2; ++sweep) {
    const bool fwd = sweep == 1;
    for (int x = threadIdx.x; x < C::SR * LD; x += kThr) sSt[x] = 0.f;
    for (int cc = 0; cc < N; ++cc) {
      const int c = fwd ? cc : N - 1 - cc;
      const int s = c * Cr, len = min(Cr, L - s);
      const bool has_state = fwd ? c > 0 : c < N - 1;
      const bool carry = fwd ? c < N - 1 : c > 0;
      // ---- tiles and prefix (the decays are requested first, so that their
      //      loads overlap the tiles')
      float la = 0.f, lb = 0.f, ln = 0.f;
      if (threadIdx.x < 32 && p.mask_kind != MASK_LIT) {
        // two tokens a lane (CT <= 64), and l after the chunk
        const int lane = threadIdx.x;
        if (2 * lane < len) la = ell(s + 2 * lane);
        if (2 * lane + 1 < len) lb = ell(s + 2 * lane + 1);
        if (lane == 0 && s + len < L) ln = ell(s + len);
      }
      load_tile<float, D, CT>(sQ, fq, s, len);
      load_tile<float, D, CT>(sK, fk, s, len);
      load_tile<T, D, CT>(sV, v, s, len);
      for (int r = threadIdx.x; r < CT; r += kThr) sV[r * LD + D] = r < len ? 1.f : 0.f;
      if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        const float a = la, b = lb;
        if (lane == 0) *sLn = ln;
        float x = a + b;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, x, o);
          if (lane >= o) x += y;
        }
        if (2 * lane < CT) sP[2 * lane] = x - b;
        if (2 * lane + 1 < CT) sP[2 * lane + 1] = x;
      }
      __syncthreads();
      {
        const float T_c = sP[len - 1], l0 = sP[0], lnext = *sLn;
        for (int t = threadIdx.x; t < CT; t += kThr) {
          const bool ok = t < len;
          // query factor of the state applied to this chunk, key weight in
          // the state it passes on
          sR[t] = !ok ? 0.f : fwd ? expf(sP[t]) : expf(T_c - sP[t] + lnext);
          sW[t] = !ok ? 0.f : fwd ? expf(T_c - sP[t]) : expf(sP[t] - l0);
        }
      }
      __syncthreads();
      // ---- num: the chunk's own keys (left-to-right sweep), then the state
      if (fwd) {
        dot_tiles<RC, RC>(sQ, LD, sK, LD, CT, CT, D, [&](int i, int j, float sv) {
          const bool in = i < len && j < len && (!p.causal || j <= i);
          sS[j * LDS + i] = in ? sv * expf(-fabsf(sP[i] - sP[j])) : 0.f;
        });
        __syncthreads();
        outer_tiles(sS, LDS, sV, LD, nullptr, CT, D, CT, [&](int i, int n, float val) { sAcc[i * LD + n] = val; });
        for (int i = threadIdx.x; i < CT; i += kThr) {
          float a = 0.f;
          for (int j = 0; j < len; ++j) a += sS[j * LDS + i];
          sAcc[i * LD + D] = a;
        }
      }
      if (has_state) {
        if (fwd) __syncthreads();
        dot_tiles<RC, RD>(sQ, LD, sSt, LD, CT, D, D, [&](int i, int n, float val) {
          sAcc[i * LD + n] = (fwd ? sAcc[i * LD + n] : 0.f) + sR[i] * val;
        });
        for (int i = threadIdx.x; i < CT; i += kThr) {
          float a = 0.f;
          for (int m = 0; m < D; m += 4) {
            const float4 qv = *reinterpret_cast<const float4*>(sQ + i * LD + m);
            const float4 zv = *reinterpret_cast<const float4*>(sSt + D * LD + m);
            a += qv.x * zv.x + qv.y * zv.y + qv.z * zv.z + qv.w * zv.w;
          }
          sAcc[i * LD + D] = (fwd ? sAcc[i * LD + D] : 0.f) + sR[i] * a;
        }
      } else if (!fwd) {
        for (int x = threadIdx.x; x < CT * LD; x += kThr) sAcc[x] = 0.f;
      }
      __syncthreads();
      // ---- out: park the right-to-left part, or add it and divide
      for (int idx = threadIdx.x; idx < len * D; idx += kThr) {
        const int i = idx / D, n = idx - i * D;
        const size_t o = (size_t)(s + i) * D + n;
        if (!fwd) {
          out[o] = sAcc[i * LD + n];
        } else {
          const float dn = sAcc[i * LD + D] + (p.causal ? 0.f : den[s + i]);
          out[o] = (sAcc[i * LD + n] + (p.causal ? 0.f : out[o])) / dn;
        }
      }
      if (!fwd)
        for (int i = threadIdx.x; i < len; i += kThr) den[s + i] = sAcc[i * LD + D];
      // ---- the state carried to the next chunk of the sweep
      if (carry) {
        const float decay = fwd ? expf(sP[len - 1]) : expf(sP[len - 1] - sP[0] + *sLn);
        outer_tiles(sV, LD, sK, LD, sW, D, D, CT,
                    [&](int n, int m, float val) { sSt[n * LD + m] = decay * sSt[n * LD + m] + val; });
        for (int m = threadIdx.x; m < D; m += kThr) {
          float a = 0.f;
          for (int j = 0; j < len; ++j) a += sW[j] * sK[j * LD + m];
          sSt[D * LD + m] = decay * sSt[D * LD + m] + a;
        }
      }
      __syncthreads();
    }
  }
}

template <typename T, int D, int CT>
cudaError_t tile_launch(const Problem& p, float* ws, cudaStream_t s) {
  const TileWs w((size_t)p.B * p.H * p.L, D);
  cudaError_t e = launch_phi_rows<T, D>(p.q, p.k, ws + w.fq, ws + w.fk, (long)p.B * p.H * p.L, p.phi, s);
  if (e != cudaSuccess) return e;
  const size_t bytes = sizeof(float) * TileCfg<D, CT>::floats;
  auto kern = chunk_tile_kernel<T, D, CT>;
  if (bytes > 48 * 1024) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
  }
  kern<<<p.B * p.H, kThr, bytes, s>>>(p, ws);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t tile_launch_ct(const Problem& p, float* ws, cudaStream_t s) {
  if (p.chunk <= 16) return tile_launch<T, D, 16>(p, ws, s);
  if (p.chunk <= 32) return tile_launch<T, D, 32>(p, ws, s);
  return tile_launch<T, D, 64>(p, ws, s);
}

}  // namespace

bool chunk_tile_supported(const Problem& p) { return p.chunk >= 1 && p.chunk <= kChunkTileMax; }

size_t chunk_tile_workspace_bytes(int B, int H, int L, int d) {
  return sizeof(float) * TileWs((size_t)B * H * L, d).total;
}

cudaError_t launch_chunk_tile(const Problem& p, float* ws, cudaStream_t s) {
  const bool bf = p.dtype == DT_BF16;
  switch (p.d) {
    case 16: return bf ? tile_launch_ct<__nv_bfloat16, 16>(p, ws, s) : tile_launch_ct<float, 16>(p, ws, s);
    case 32: return bf ? tile_launch_ct<__nv_bfloat16, 32>(p, ws, s) : tile_launch_ct<float, 32>(p, ws, s);
    case 64: return bf ? tile_launch_ct<__nv_bfloat16, 64>(p, ws, s) : tile_launch_ct<float, 64>(p, ws, s);
    case 128: return bf ? tile_launch_ct<__nv_bfloat16, 128>(p, ws, s) : tile_launch_ct<float, 128>(p, ws, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace lion
