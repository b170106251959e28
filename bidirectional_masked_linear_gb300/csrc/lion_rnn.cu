// lion_rnn.cu -- the recurrent form of the LION operator on the CUDA cores
// (fp32 arithmetic, d in {16, 32, 64, 128}, bfloat16 or float32 inputs).
//
// Theorem 3.3 Eq 20-24 (rebuttal page "LION: A bidirectional framework that
// trains like a Transformer and infers like an RNN"): per head
//   forward   S^F_i = lambda_i S^F_{i-1} + phi(k_i) v_i^T,   z^F_i likewise with v = 1
//   backward  S^B_i = lambda_{i+1} S^B_{i+1} + phi(k_i) v_i^T
//   y_i = (phi(q_i)^T S^F_i + phi(q_i)^T S^B_i - s_ii v_i)
//         / (phi(q_i)^T z^F_i + phi(q_i)^T z^B_i - s_ii),   s_ii = phi(q_i) . phi(k_i),
// keeping only y^F_i and c^F_i = phi(q_i)^T z^F_i between the two sweeps
// (reply "1: Recurrence Form": O(Ld + L) side storage).  With Problem::causal
// the forward sweep alone gives y_i = y^F_i / c^F_i.
//
// Columns of the state are independent recurrences: column n of S follows
// v_n, and z is the column of a constant 1.  So each CTA runs the whole
// sequence for 8 columns of one head plus z, and a head's d columns spread
// over d / 8 CTAs.  Every CTA of a head computes z, so each has the
// normaliser it divides by without waiting for another; they all store the
// same c^F_i (the same arithmetic on the same inputs).  Every CTA of a head
// also computes phi of the whole tile, so splitting a head finer (4 columns
// a CTA when the heads are few) made the feature map, not the recurrence,
// the larger share of each CTA's work and the form slower.
//
// Inside a CTA a warp holds four state columns, eight lanes a column and
// d / 8 rows of it per lane, in registers.  A token costs each lane its rows'
// multiply-adds for S and for the partial phi(q) . S; the partial sums of 32
// tokens are then reduced across the column's eight lanes in one transposing
// pass (28 shuffles for 32 tokens), which leaves four tokens' sums per lane.
// Token tiles of 32 are copied asynchronously (cp.async) one tile ahead;
// phi of the tile (and s_ii) is computed once per CTA into shared memory,
// eight lanes a row.
#include "lion_common.cuh"
#include "lion_internal.h"

namespace lion {
namespace {

constexpr int kSlots = 4;                                   // state columns per warp
constexpr int kG = 32 / kSlots;                             // lanes per column
constexpr int kTile = 32;                                   // tokens per staged tile
// NC columns of v per CTA: NC + 1 state columns with z, four a warp
template <int NC>
struct Cols {
  static constexpr int kWarps = (NC + 1 + kSlots - 1) / kSlots;
  static constexpr int kThr = 32 * kWarps;
};

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  const uint32_t s = (uint32_t)__cvta_generic_to_shared(dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async8(void* dst, const void* src) {
  const uint32_t s = (uint32_t)__cvta_generic_to_shared(dst);
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(s), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <typename T, int D, int NC>
struct Lay {
  static constexpr int kRawQ = kTile * D * (int)sizeof(T);      // bytes of a raw q (or k) tile
  static constexpr int kRawV = kTile * NC * (int)sizeof(T);     // the CTA's columns of v
  static constexpr int kRaw = 2 * kRawQ + ((kRawV + 15) & ~15); // one raw slot
  static constexpr int kF32 = (2 * kTile * D + kTile * NC + 3 * kTile) * 4;
  static constexpr int kBytes = 2 * kRaw + kF32;
};

// Issue the copies of tile [t0, t0 + nt) of q, k and the CTA's v columns into
// raw slot `dst` (one commit group).
template <typename T, int D, int NC>
__device__ __forceinline__ void issue_tile(uint8_t* dst, const T* q, const T* k, const T* v, int n0, int t0,
                                           int nt) {
  using Y = Lay<T, D, NC>;
  constexpr int kThr = Cols<NC>::kThr;
  constexpr int kRowChunks = D * (int)sizeof(T) / 16;       // 16-byte pieces of a q row
  constexpr int kVBytes = NC * (int)sizeof(T);              // the CTA's v columns in a row
  constexpr int kVPiece = kVBytes < 16 ? kVBytes : 16;      // 8 (four bf16 columns) or 16
  constexpr int kVChunks = kVBytes / kVPiece;
  for (int x = threadIdx.x; x < 2 * nt * kRowChunks; x += kThr) {
    const int which = x / (nt * kRowChunks), r = (x / kRowChunks) % nt, c = x % kRowChunks;
    const T* src = (which == 0 ? q : k) + (size_t)(t0 + r) * D + c * (16 / (int)sizeof(T));
    cp_async16(dst + which * Y::kRawQ + r * D * (int)sizeof(T) + 16 * c, src);
  }
  for (int x = threadIdx.x; x < nt * kVChunks; x += kThr) {
    const int r = x / kVChunks, c = x % kVChunks;
    uint8_t* to = dst + 2 * Y::kRawQ + r * kVBytes + kVPiece * c;
    const T* from = v + (size_t)(t0 + r) * D + n0 + c * (kVPiece / (int)sizeof(T));
    if constexpr (kVPiece == 16) cp_async16(to, from);
    else cp_async8(to, from);
  }
  cp_commit();
}

// phi of one raw row's PER features held by this lane; the row's other
// features sit in the 7 lanes next to it (xor 1, 2, 4).
// (The fast exponential and division err by a few ulp, far below what the
// fp32 recurrence itself accumulates.)
template <int PER>
__device__ __forceinline__ void phi_lane(float* x, int phi) {
  if (phi == PHI_ELU1) {
#pragma unroll
    for (int e = 0; e < PER; ++e) x[e] = x[e] > 0.f ? x[e] + 1.f : __expf(x[e]);
  } else if (phi == PHI_SILU_L2) {
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < PER; ++e) {
      x[e] = __fdividef(x[e], 1.f + __expf(-x[e]));
      ss = fmaf(x[e], x[e], ss);
    }
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float inv = 1.f / fmaxf(sqrtf(ss), 1e-12f);
#pragma unroll
    for (int e = 0; e < PER; ++e) x[e] *= inv;
  }
}

// phi(q) and phi(k) of the tile's rows, from the raw copies into fp32 rows,
// and s_ii = phi(q_i) . phi(k_i): eight lanes a row (D/8 features each), four
// rows a warp at a time.  Rows at or past nt come out zero.
template <typename T, int D, int NC>
__device__ __forceinline__ void phi_tile(float* sQ, float* sK, float* sSii, const T* rq, const T* rk, int nt,
                                         int phi) {
  constexpr int PER = D / 8;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 3, sub = lane & 7;
  for (int r0 = 4 * warp; r0 < kTile; r0 += 4 * Cols<NC>::kWarps) {
    const int r = r0 + g, c0 = r * D + sub * PER;
    const bool ok = r < nt;
    float xq[PER], xk[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) {
      xq[e] = ok ? to_f32(rq[c0 + e]) : 0.f;
      xk[e] = ok ? to_f32(rk[c0 + e]) : 0.f;
    }
    phi_lane<PER>(xq, phi);
    phi_lane<PER>(xk, phi);
    float sii = 0.f;
#pragma unroll
    for (int e = 0; e < PER; ++e) {
      if (!ok) xq[e] = xk[e] = 0.f;   // padding contributes nothing (phi(0) = 1 for elu+1)
      sQ[c0 + e] = xq[e];
      sK[c0 + e] = xk[e];
      sii = fmaf(xq[e], xk[e], sii);
    }
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) sii += __shfl_xor_sync(0xffffffffu, sii, o);
    if (sub == 0) sSii[r] = sii;
  }
}

template <typename T, int D, int NC>
__global__ void __launch_bounds__(Cols<NC>::kThr) rnn_cols_kernel(Problem p, float* cF_all) {
  using Y = Lay<T, D, NC>;
  constexpr int kCols = NC, kThr = Cols<NC>::kThr;
  constexpr int RPL = D / kG;                  // state rows per lane
  constexpr int VW = RPL < 4 ? RPL : 4;        // rows read per vector load
  constexpr int NB = D / kCols;                // CTAs per head
  extern __shared__ float4 smem4[];
  uint8_t* raw = reinterpret_cast<uint8_t*>(smem4);
  float* sQ = reinterpret_cast<float*>(raw + 2 * Y::kRaw);   // [kTile][D] phi(q)
  float* sK = sQ + kTile * D;                                 // [kTile][D] phi(k)
  float* sV = sK + kTile * D;                                 // [kTile][kCols]
  float* sLam = sV + kTile * kCols;                           // [kTile] decay of each step
  float* sSii = sLam + kTile;                                 // [kTile] s_ii
  float* sC = sSii + kTile;                                   // [kTile] this tile's z sums

  const int L = p.L, H = p.H;
  const int bh = (int)(blockIdx.x / NB), n0 = (int)(blockIdx.x % NB) * kCols;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int col = warp * kSlots + lane / kG;   // 0..kCols-1: v columns; kCols: z; above: idle
  const int sub = lane % kG;
  const T* q = reinterpret_cast<const T*>(p.q) + (size_t)bh * L * D;
  const T* k = reinterpret_cast<const T*>(p.k) + (size_t)bh * L * D;
  const T* v = reinterpret_cast<const T*>(p.v) + (size_t)bh * L * D;
  float* out = p.out + (size_t)bh * L * D;
  float* cF = cF_all + (size_t)bh * L;
  const float* ll = p.mask_kind == MASK_S ? p.log_lambda + (size_t)bh * L : nullptr;
  const float lh = p.mask_kind == MASK_D ? __ldg(p.log_lambda + bh % H) : 0.f;
  const int ntiles = (L + kTile - 1) / kTile;

  for (int sweep = 0; sweep < (p.causal ? 1 : 2); ++sweep) {
    const bool fwd = sweep == 0;
    float S[RPL];
#pragma unroll
    for (int r = 0; r < RPL; ++r) S[r] = 0.f;
    auto tile_t0 = [&](int i) { return (fwd ? i : ntiles - 1 - i) * kTile; };
    issue_tile<T, D, NC>(raw, q, k, v, n0, tile_t0(0), min(kTile, L - tile_t0(0)));
    for (int i = 0; i < ntiles; ++i) {
      const int t0 = tile_t0(i), nt = min(kTile, L - t0);
      uint8_t* slot = raw + (i & 1) * Y::kRaw;
      if (i + 1 < ntiles) {
        const int t1 = tile_t0(i + 1);
        issue_tile<T, D, NC>(raw + ((i + 1) & 1) * Y::kRaw, q, k, v, n0, t1, min(kTile, L - t1));
        cp_wait<1>();
      } else {
        cp_wait<0>();
      }
      __syncthreads();
      // ---- fp32 tile, phi, decays, s_ii
      const T* rq = reinterpret_cast<const T*>(slot);
      const T* rk = reinterpret_cast<const T*>(slot + Y::kRawQ);
      const T* rv = reinterpret_cast<const T*>(slot + 2 * Y::kRawQ);
      phi_tile<T, D, NC>(sQ, sK, sSii, rq, rk, nt, p.phi);
      for (int x = threadIdx.x; x < kTile * kCols; x += kThr) sV[x] = x / kCols < nt ? to_f32(rv[x]) : 0.f;
      if (threadIdx.x < kTile) {
        // forward: lambda_t; backward: lambda_{t+1} (none after the last token)
        const int t = t0 + (int)threadIdx.x + (fwd ? 0 : 1);
        float l = 0.f;
        bool have = t < L;
        if (have) l = ll ? __ldg(ll + t) : lh;
        sLam[threadIdx.x] = have ? expf(l) : 0.f;
      }
      __syncthreads();
      // ---- the recurrence over the tile, in sweep order u (token tt = u
      //      forward, kTile - 1 - u backward): part[u] = phi(q_tt) . (column of
      //      S after tt)
      float part[kTile];
#pragma unroll
      for (int u = 0; u < kTile; ++u) {
        const int tt = fwd ? u : kTile - 1 - u;
        float a = 0.f;
        if (tt < nt) {
          const float lam = sLam[tt];
          const float vn = col < kCols ? sV[tt * kCols + col] : (col == kCols ? 1.f : 0.f);
#pragma unroll
          for (int r4 = 0; r4 < RPL / VW; ++r4) {
            const int m = VW * sub + kG * VW * r4;
            float kv[VW], qv[VW];
            if constexpr (VW == 4) {
              const float4 k4 = *reinterpret_cast<const float4*>(sK + tt * D + m);
              const float4 q4 = *reinterpret_cast<const float4*>(sQ + tt * D + m);
              kv[0] = k4.x; kv[1] = k4.y; kv[2] = k4.z; kv[3] = k4.w;
              qv[0] = q4.x; qv[1] = q4.y; qv[2] = q4.z; qv[3] = q4.w;
            } else {
              const float2 k2 = *reinterpret_cast<const float2*>(sK + tt * D + m);
              const float2 q2 = *reinterpret_cast<const float2*>(sQ + tt * D + m);
              kv[0] = k2.x; kv[1] = k2.y;
              qv[0] = q2.x; qv[1] = q2.y;
            }
#pragma unroll
            for (int e = 0; e < VW; ++e) {
              float& sr = S[r4 * VW + e];
              sr = fmaf(lam, sr, kv[e] * vn);
              a = fmaf(qv[e], sr, a);
            }
          }
        }
        part[u] = a;
      }
      // ---- sums over the column's kG lanes, transposed: afterwards lane
      //      `sub` holds sweep positions 4 sub .. 4 sub + 3 in part[0..3]
#pragma unroll
      for (int sh = kG / 2, cnt = kTile; sh >= 1; sh >>= 1, cnt >>= 1) {
        const bool up = (lane & sh) != 0;
#pragma unroll
        for (int x = 0; x < cnt / 2; ++x) {
          const float send = up ? part[x] : part[x + cnt / 2];
          const float keep = up ? part[x + cnt / 2] : part[x];
          part[x] = keep + __shfl_xor_sync(0xffffffffu, send, sh);
        }
      }
      constexpr int kPer = kTile / kG;   // tokens per lane after the reduction
      auto token_of = [&](int e) { return fwd ? kPer * sub + e : kTile - 1 - (kPer * sub + e); };
      if (col == kCols) {
#pragma unroll
        for (int e = 0; e < kPer; ++e) {
          const int tt = token_of(e);
          if (tt < nt) {
            sC[tt] = part[e];
            if (fwd && !p.causal) cF[t0 + tt] = part[e];
          }
        }
      }
      __syncthreads();
      if (col < kCols) {
        const int n = n0 + col;
#pragma unroll
        for (int e = 0; e < kPer; ++e) {
          const int tt = token_of(e);
          if (tt >= nt) continue;
          const size_t o = (size_t)(t0 + tt) * D + n;
          if (p.causal) {
            out[o] = part[e] / sC[tt];
          } else if (fwd) {
            out[o] = part[e];
          } else {
            const float sii = sSii[tt], vn = sV[tt * kCols + col];
            out[o] = (out[o] + part[e] - sii * vn) / (cF[t0 + tt] + sC[tt] - sii);
          }
        }
      }
      __syncthreads();
    }
  }
}

template <typename T, int D, int NC>
cudaError_t rnn_launch_nc(const Problem& p, float* ws, cudaStream_t s) {
  using Y = Lay<T, D, NC>;
  auto kern = rnn_cols_kernel<T, D, NC>;
  if (Y::kBytes > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Y::kBytes);
    if (e != cudaSuccess) return e;
  }
  const size_t grid = (size_t)p.B * p.H * (D / NC);
  kern<<<(unsigned)grid, Cols<NC>::kThr, Y::kBytes, s>>>(p, ws);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t rnn_launch(const Problem& p, float* ws, cudaStream_t s) {
  return rnn_launch_nc<T, D, 8>(p, ws, s);
}

}  // namespace

cudaError_t launch_rnn_simt(const Problem& p, float* ws, cudaStream_t s) {
  const bool bf = p.dtype == DT_BF16;
  switch (p.d) {
    case 16: return bf ? rnn_launch<__nv_bfloat16, 16>(p, ws, s) : rnn_launch<float, 16>(p, ws, s);
    case 32: return bf ? rnn_launch<__nv_bfloat16, 32>(p, ws, s) : rnn_launch<float, 32>(p, ws, s);
    case 64: return bf ? rnn_launch<__nv_bfloat16, 64>(p, ws, s) : rnn_launch<float, 64>(p, ws, s);
    case 128: return bf ? rnn_launch<__nv_bfloat16, 128>(p, ws, s) : rnn_launch<float, 128>(p, ws, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace lion
