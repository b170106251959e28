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
// same c^F_i (the same arithmetic on the same inputs).
//
// Sweeps.  When the heads are few (under two column CTAs an SM), the sequence
// has 256 tokens or more and the workspace is whole, the two sweeps run at
// the same time in separate CTAs
// (gridDim.y = 2): the backward CTAs store their sums y^B_i and c^B_i
// beside y^F_i and c^F_i (the O(Ld + L) side storage of both directions),
// and a last launch combines them.  Otherwise each CTA runs the forward
// sweep, then the backward one, which combines as it goes.  Both ways the
// combination is one helper with every rounding explicit, so they give the
// same bits.
//
// Feature maps.  With a workspace of rnn_workspace_bytes, a first launch
// writes phi(q), phi(k) (fp32) and s_ii of every token once, and the column
// CTAs of a head copy them in; with only the c^F scratch (the allocation-
// free entry point) every column CTA computes phi of its tiles itself.  Both
// run the same code on the same eight-lane row split, so the two give the
// same bits.
//
// Inside a CTA each state column sits on G lanes (8 at d < 64; 16 at
// d >= 64, or 32 when the heads are few), d / G rows of it per lane, in
// registers, as pairs updated by the packed two-lane fp32 instructions.  A
// token costs each lane its rows' multiply-adds for S and for the partial
// phi(q) . S; the partial sums of a tile of tokens are then reduced across
// the column's G lanes in one transposing pass, which leaves tile / G
// tokens' sums per lane.  Tiles hold 16 tokens at G = 16 (a smaller shared-
// memory and register footprint: more CTAs resident when the heads are
// many) and 32 otherwise; they are copied asynchronously (cp.async) one
// tile ahead.
#include <algorithm>
#include <type_traits>

#include "c128_common.cuh"
#include "lion_common.cuh"
#include "lion_internal.h"

namespace lion {
namespace {

using c128::fma2;
using c128::mul2;

constexpr int kNC = 8;                                      // v columns per CTA
constexpr int kTileMany = 16;                               // tokens per tile at G = 16
// G lanes per state column, d / G rows a lane: 8 at d < 64; at d >= 64, 16
// (two columns a warp), or 32 (one) when the heads are too few to fill the
// GPU otherwise -- more warps a head and shorter dependent chains, against
// more warps' share of the column sums and of z.
template <int D, int G>
struct Split {
  static constexpr int kG = G;                                      // lanes per column
  static constexpr int kSlots = 32 / kG;                            // state columns per warp
  static constexpr int kWarps = (kNC + 1 + kSlots - 1) / kSlots;    // kNC + 1 state columns with z
  static constexpr int kThr = 32 * kWarps;
  static constexpr int kSlotCols = kSlots * kWarps;                 // every lane group's column: v, z, idle
};

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  const uint32_t s = (uint32_t)__cvta_generic_to_shared(dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  const uint32_t s = (uint32_t)__cvta_generic_to_shared(dst);
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(s), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Workspace sections (floats, each padded to 64): c^F [BH L], s_ii [BH L],
// phi(q) [BH L d], phi(k) [BH L d] (up to `features`), then for the split
// sweeps y^B [BH L d] and c^B [BH L].
__host__ __device__ constexpr size_t pad64(size_t n) { return (n + 63) & ~size_t(63); }
struct RnnWs {
  size_t cF, sii, fq, fk, yB, cB, features, total;   // float offsets and sizes
  __host__ __device__ RnnWs(size_t BHL, int d) {
    cF = 0;
    sii = pad64(BHL);
    fq = sii + pad64(BHL);
    fk = fq + pad64(BHL * (size_t)d);
    features = fk + pad64(BHL * (size_t)d);
    yB = features;
    cB = yB + pad64(BHL * (size_t)d);
    total = cB + pad64(BHL);
  }
};

// y_i from the two sweeps' sums, each of which counts the diagonal term:
// (y^F + y^B - s_ii v) / (c^F + c^B - s_ii), every rounding explicit.
__device__ __forceinline__ float combine_y(float yf, float yb, float sii, float vn, float cf, float cb) {
  return __fdiv_rn(__fmaf_rn(-sii, vn, __fadd_rn(yf, yb)), __fsub_rn(__fadd_rn(cf, cb), sii));
}

// phi of one row's PER features held by this lane; the row's other
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

// phi(q) and phi(k) of one row (eight lanes a row, PER = D / 8 features
// each, starting at feature c0 of the rows rq and rk) and s_ii = phi(q) .
// phi(k), which every lane of the row returns.  A row that is not `ok`
// comes out zero (phi(0) = 1 for elu + 1, so padding is zeroed after phi).
template <typename T, int PER>
__device__ __forceinline__ float phi_row(const T* rq, const T* rk, int c0, bool ok, int phi, float* xq,
                                         float* xk) {
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
    if (!ok) xq[e] = xk[e] = 0.f;
    sii = fmaf(xq[e], xk[e], sii);
  }
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) sii += __shfl_xor_sync(0xffffffffu, sii, o);
  return sii;
}

// ---------------------------------------------------------------- pre-pass
// phi(q), phi(k) and s_ii of every token, once: a warp takes four rows at a
// time, eight lanes a row.
template <typename T, int D>
__global__ void __launch_bounds__(256) rnn_phi_kernel(Problem p, float* ws) {
  constexpr int PER = D / 8;
  const size_t rows = (size_t)p.B * p.H * p.L;
  const RnnWs w(rows, D);
  const int lane = threadIdx.x & 31, g = lane >> 3, sub = lane & 7;
  const size_t warp0 = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const size_t nwarps = ((size_t)gridDim.x * blockDim.x) >> 5;
  const T* q = reinterpret_cast<const T*>(p.q);
  const T* k = reinterpret_cast<const T*>(p.k);
  for (size_t r0 = 4 * warp0; r0 < rows; r0 += 4 * nwarps) {
    const size_t r = r0 + g;
    const bool ok = r < rows;
    const size_t rr = ok ? r : rows - 1;
    float xq[PER], xk[PER];
    const float sii = phi_row<T, PER>(q + rr * D, k + rr * D, sub * PER, ok, p.phi, xq, xk);
    if (ok) {
      float* fq = ws + w.fq + r * D + sub * PER;
      float* fk = ws + w.fk + r * D + sub * PER;
#pragma unroll
      for (int e = 0; e < PER; e += 2) {
        *reinterpret_cast<float2*>(fq + e) = make_float2(xq[e], xq[e + 1]);
        *reinterpret_cast<float2*>(fk + e) = make_float2(xk[e], xk[e + 1]);
      }
      if (sub == 0) ws[w.sii + r] = sii;
    }
  }
}

// ------------------------------------------------------------ column CTAs
// Shared memory: two raw slots (the tile's q and k as loaded, or with PRE
// their fp32 features and s_ii, plus the CTA's v columns), then without PRE
// the fp32 features of the tile, then the v column table, decays, s_ii and
// the tile's z sums.
template <typename T, int D, int G, int kTile, bool PRE>
struct Lay {
  static constexpr int kQK = kTile * D * (PRE ? 4 : (int)sizeof(T));   // bytes of one q (or k) tile
  static constexpr int kVB = kTile * kNC * (int)sizeof(T);              // the CTA's columns of v
  static constexpr int kSiiB = PRE ? kTile * 4 : 0;
  static constexpr int kRaw = 2 * kQK + kVB + kSiiB;                    // one raw slot
  static constexpr int kF32 = ((PRE ? 0 : 2 * kTile * D) + kTile * Split<D, G>::kSlotCols + 3 * kTile) * 4;
  static constexpr int kBytes = 2 * kRaw + kF32;
  static_assert(kQK % 16 == 0 && kVB % 16 == 0 && kRaw % 16 == 0, "16-byte copies");
};

// Issue the copies of tile [t0, t0 + nt) into raw slot `dst` (one commit
// group): the q and k rows (or their features and s_ii) and the CTA's v
// columns.
template <typename T, int D, int G, int kTile, bool PRE>
__device__ __forceinline__ void issue_tile(uint8_t* dst, const void* q, const void* k, const float* sii,
                                           const T* v, int n0, int t0, int nt) {
  using Y = Lay<T, D, G, kTile, PRE>;
  using E = typename std::conditional<PRE, float, T>::type;
  constexpr int kThr = Split<D, G>::kThr;
  constexpr int kRowChunks = D * (int)sizeof(E) / 16;       // 16-byte pieces of a q row
  constexpr int kVChunks = kNC * (int)sizeof(T) / 16;
  const E* qe = reinterpret_cast<const E*>(q);
  const E* ke = reinterpret_cast<const E*>(k);
  for (int x = threadIdx.x; x < 2 * nt * kRowChunks; x += kThr) {
    const int which = x / (nt * kRowChunks), r = (x / kRowChunks) % nt, c = x % kRowChunks;
    const E* src = (which == 0 ? qe : ke) + (size_t)(t0 + r) * D + c * (16 / (int)sizeof(E));
    cp_async16(dst + which * Y::kQK + r * D * (int)sizeof(E) + 16 * c, src);
  }
  for (int x = threadIdx.x; x < nt * kVChunks; x += kThr) {
    const int r = x / kVChunks, c = x % kVChunks;
    cp_async16(dst + 2 * Y::kQK + r * kNC * (int)sizeof(T) + 16 * c,
               v + (size_t)(t0 + r) * D + n0 + c * (16 / (int)sizeof(T)));
  }
  if (PRE && (int)threadIdx.x < nt) cp_async4(dst + 2 * Y::kQK + Y::kVB + 4 * threadIdx.x, sii + t0 + threadIdx.x);
  cp_commit();
}

template <typename T, int D, int G, int kTile, bool PRE>
__global__ void __launch_bounds__(Split<D, G>::kThr) rnn_cols_kernel(Problem p, float* ws) {
  using Y = Lay<T, D, G, kTile, PRE>;
  constexpr int kG = G, kSlots = Split<D, G>::kSlots, kWarps = Split<D, G>::kWarps;
  constexpr int kThr = Split<D, G>::kThr, kSlotCols = Split<D, G>::kSlotCols;
  constexpr int PER = D / 8;
  constexpr int RPL = D / kG;                  // state rows per lane
  constexpr int VW = RPL < 4 ? RPL : 4;        // rows read per vector load
  constexpr int NB = D / kNC;                  // CTAs per head
  extern __shared__ float4 smem4[];
  uint8_t* raw = reinterpret_cast<uint8_t*>(smem4);
  float* sQc = reinterpret_cast<float*>(raw + 2 * Y::kRaw);   // without PRE: [kTile][D] phi(q)
  float* sKc = sQc + (PRE ? 0 : kTile * D);                   // without PRE: [kTile][D] phi(k)
  float* sV = sKc + (PRE ? 0 : kTile * D);                    // [kTile][kSlotCols] v columns, 1 (z), 0
  float* sLam = sV + kTile * kSlotCols;                       // [kTile] decay of each step
  float* sSiic = sLam + kTile;                                // without PRE: [kTile] s_ii
  float* sC = sSiic + kTile;                                  // [kTile] this tile's z sums

  const int L = p.L, H = p.H;
  const RnnWs w((size_t)p.B * H * L, D);
  const int bh = (int)(blockIdx.x / NB), n0 = (int)(blockIdx.x % NB) * kNC;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int col = warp * kSlots + lane / kG;   // 0..kNC-1: v columns; kNC: z; above: idle
  const int sub = lane % kG;
  const void* qsrc = PRE ? static_cast<const void*>(ws + w.fq + (size_t)bh * L * D)
                         : static_cast<const void*>(reinterpret_cast<const T*>(p.q) + (size_t)bh * L * D);
  const void* ksrc = PRE ? static_cast<const void*>(ws + w.fk + (size_t)bh * L * D)
                         : static_cast<const void*>(reinterpret_cast<const T*>(p.k) + (size_t)bh * L * D);
  const float* siisrc = PRE ? ws + w.sii + (size_t)bh * L : nullptr;
  const T* v = reinterpret_cast<const T*>(p.v) + (size_t)bh * L * D;
  float* out = p.out + (size_t)bh * L * D;
  float* cF = ws + w.cF + (size_t)bh * L;
  // split sweeps: this CTA's direction is blockIdx.y (0 forward, 1 backward)
  const bool split = gridDim.y == 2;
  float* yB = split ? ws + w.yB + (size_t)bh * L * D : nullptr;
  float* cB = split ? ws + w.cB + (size_t)bh * L : nullptr;
  const float* ll = p.mask_kind == MASK_S ? p.log_lambda + (size_t)bh * L : nullptr;
  const float lh = p.mask_kind == MASK_D ? __ldg(p.log_lambda + bh % H) : 0.f;
  const int ntiles = (L + kTile - 1) / kTile;

  // One sweep; the direction is a compile-time constant so that every token
  // of the unrolled tile loop addresses shared memory at a fixed offset.
  // Rows past L enter as phi = 0, v = 0 and decay 1: they leave S unchanged,
  // so the loop needs no bounds test.
  auto sweep = [&](auto dir) {
    constexpr bool fwd = decltype(dir)::value;
    float2 S[RPL / 2];
#pragma unroll
    for (int r = 0; r < RPL / 2; ++r) S[r] = make_float2(0.f, 0.f);
    auto tile_t0 = [&](int i) { return (fwd ? i : ntiles - 1 - i) * kTile; };
    issue_tile<T, D, G, kTile, PRE>(raw, qsrc, ksrc, siisrc, v, n0, tile_t0(0), min(kTile, L - tile_t0(0)));
    for (int i = 0; i < ntiles; ++i) {
      const int t0 = tile_t0(i), nt = min(kTile, L - t0);
      uint8_t* slot = raw + (i & 1) * Y::kRaw;
      // this tile landed and every thread is done with the previous one, so
      // the next tile may go into the slot the one before it used
      cp_wait<0>();
      __syncthreads();
      if (i + 1 < ntiles) {
        const int t1 = tile_t0(i + 1);
        issue_tile<T, D, G, kTile, PRE>(raw + ((i + 1) & 1) * Y::kRaw, qsrc, ksrc, siisrc, v, n0, t1,
                                        min(kTile, L - t1));
      }
      // ---- the tile's features and s_ii, the v column table, the decays
      const float* tQ;
      const float* tK;
      const float* tSii;
      if constexpr (PRE) {
        float* fq = reinterpret_cast<float*>(slot);
        float* fk = reinterpret_cast<float*>(slot + Y::kQK);
        tQ = fq;
        tK = fk;
        tSii = reinterpret_cast<const float*>(slot + 2 * Y::kQK + Y::kVB);
        // rows past L were not copied: zero features leave S unchanged
        for (int x = nt * D + (int)threadIdx.x; x < kTile * D; x += kThr) fq[x] = fk[x] = 0.f;
      } else {
        const T* rq = reinterpret_cast<const T*>(slot);
        const T* rk = reinterpret_cast<const T*>(slot + Y::kQK);
        const int g = lane >> 3, s8 = lane & 7;
        for (int r0 = 4 * warp; r0 < kTile; r0 += 4 * kWarps) {
          const int r = r0 + g, c0 = r * D + s8 * PER;
          float xq[PER], xk[PER];
          const float sii = phi_row<T, PER>(rq, rk, c0, r < nt, p.phi, xq, xk);
#pragma unroll
          for (int e = 0; e < PER; ++e) {
            sQc[c0 + e] = xq[e];
            sKc[c0 + e] = xk[e];
          }
          if (s8 == 0) sSiic[r] = sii;
        }
        tQ = sQc;
        tK = sKc;
        tSii = sSiic;
      }
      const T* rv = reinterpret_cast<const T*>(slot + 2 * Y::kQK);
      for (int x = threadIdx.x; x < kTile * kSlotCols; x += kThr) {
        const int r = x / kSlotCols, c = x - r * kSlotCols;
        sV[x] = r >= nt ? 0.f : c < kNC ? to_f32(rv[r * kNC + c]) : c == kNC ? 1.f : 0.f;
      }
      if (threadIdx.x < kTile) {
        // forward: lambda_t; backward: lambda_{t+1} (none after the last
        // token, where S is still zero); 1 on the rows past L
        const int t = t0 + (int)threadIdx.x + (fwd ? 0 : 1);
        sLam[threadIdx.x] = t < L ? expf(ll ? __ldg(ll + t) : lh) : 1.f;
      }
      __syncthreads();
      // ---- the recurrence over the tile, in sweep order u (token tt = u
      //      forward, kTile - 1 - u backward): part[u] = phi(q_tt) . (column of
      //      S after tt).  Rows go in pairs through the packed instructions;
      //      the even and odd rows' dot-product terms are summed apart.
      float part[kTile];
#pragma unroll
      for (int u = 0; u < kTile; ++u) {
        const int tt = fwd ? u : kTile - 1 - u;
        const float lam = sLam[tt];
        const float vn = sV[tt * kSlotCols + col];
        const float2 lam2 = make_float2(lam, lam), vn2 = make_float2(vn, vn);
        float2 a2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int r4 = 0; r4 < RPL / VW; ++r4) {
          const int m = VW * sub + kG * VW * r4;
          float2 kv[VW / 2], qv[VW / 2];
          if constexpr (VW == 4) {
            const float4 k4 = *reinterpret_cast<const float4*>(tK + tt * D + m);
            const float4 q4 = *reinterpret_cast<const float4*>(tQ + tt * D + m);
            kv[0] = make_float2(k4.x, k4.y);
            kv[1] = make_float2(k4.z, k4.w);
            qv[0] = make_float2(q4.x, q4.y);
            qv[1] = make_float2(q4.z, q4.w);
          } else {
            kv[0] = *reinterpret_cast<const float2*>(tK + tt * D + m);
            qv[0] = *reinterpret_cast<const float2*>(tQ + tt * D + m);
          }
#pragma unroll
          for (int e = 0; e < VW / 2; ++e) {
            float2& sr = S[r4 * (VW / 2) + e];
            sr = fma2(lam2, sr, mul2(kv[e], vn2));
            a2 = fma2(qv[e], sr, a2);
          }
        }
        part[u] = a2.x + a2.y;
      }
      // ---- sums over the column's kG lanes, transposed: afterwards lane
      //      `sub` holds sweep positions kPer sub .. kPer sub + kPer - 1 in
      //      part[0..kPer-1] (kPer = 32 / kG)
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
      if (col == kNC) {
#pragma unroll
        for (int e = 0; e < kPer; ++e) {
          const int tt = token_of(e);
          if (tt < nt) {
            sC[tt] = part[e];
            if (fwd && !p.causal) cF[t0 + tt] = part[e];
            if (!fwd && split) cB[t0 + tt] = part[e];
          }
        }
      }
      __syncthreads();
      if (col < kNC) {
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
          } else if (split) {
            yB[o] = part[e];
          } else {
            out[o] = combine_y(out[o], part[e], tSii[tt], sV[tt * kSlotCols + col], cF[t0 + tt], sC[tt]);
          }
        }
      }
    }
    __syncthreads();   // the next sweep's first tile reuses slot 0
  };
  if (!split || blockIdx.y == 0) sweep(std::integral_constant<bool, true>{});
  if (!p.causal && (!split || blockIdx.y == 1)) sweep(std::integral_constant<bool, false>{});
}

// The split sweeps' combination, four features of one token a thread.
template <typename T, int D>
__global__ void __launch_bounds__(256) rnn_combine_kernel(Problem p, const float* ws) {
  constexpr int Q = D / 4;
  const size_t rows = (size_t)p.B * p.H * p.L, n = rows * Q;
  const RnnWs w(rows, D);
  const T* v = reinterpret_cast<const T*>(p.v);
  for (size_t x = (size_t)blockIdx.x * blockDim.x + threadIdx.x; x < n; x += (size_t)gridDim.x * blockDim.x) {
    const size_t r = x / Q, o = r * D + 4 * (x - r * Q);
    const float4 yb = *reinterpret_cast<const float4*>(ws + w.yB + o);
    float4 y = *reinterpret_cast<const float4*>(p.out + o);
    const float sii = ws[w.sii + r], cf = ws[w.cF + r], cb = ws[w.cB + r];
    y.x = combine_y(y.x, yb.x, sii, to_f32(v[o]), cf, cb);
    y.y = combine_y(y.y, yb.y, sii, to_f32(v[o + 1]), cf, cb);
    y.z = combine_y(y.z, yb.z, sii, to_f32(v[o + 2]), cf, cb);
    y.w = combine_y(y.w, yb.w, sii, to_f32(v[o + 3]), cf, cb);
    *reinterpret_cast<float4*>(p.out + o) = y;
  }
}

template <typename T, int D, int G, int TT>
cudaError_t rnn_launch_g(const Problem& p, float* ws, bool pre, bool split, cudaStream_t s) {
  auto kern = pre ? rnn_cols_kernel<T, D, G, TT, true> : rnn_cols_kernel<T, D, G, TT, false>;
  const int bytes = pre ? Lay<T, D, G, TT, true>::kBytes : Lay<T, D, G, TT, false>::kBytes;
  if (bytes > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
  }
  const size_t grid = (size_t)p.B * p.H * (D / kNC);
  kern<<<dim3((unsigned)grid, split ? 2u : 1u), Split<D, G>::kThr, bytes, s>>>(p, ws);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || !split) return e;
  const size_t n = (size_t)p.B * p.H * p.L * (D / 4);
  const unsigned blocks = (unsigned)std::min<size_t>((n + 255) / 256, (size_t)c128::sm_count() * 8);
  rnn_combine_kernel<T, D><<<blocks, 256, 0, s>>>(p, ws);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t rnn_launch(const Problem& p, float* ws, size_t ws_floats, cudaStream_t s) {
  const size_t BHL = (size_t)p.B * p.H * p.L;
  const RnnWs w(BHL, D);
  const bool pre = ws_floats >= w.features;
  // the two sweeps at once when the column CTAs leave the SMs under two each
  // and the sequence is long enough for a sweep to outlast the extra launch
  const long long ctas = (long long)p.B * p.H * (D / kNC);
  const bool split = pre && ws_floats >= w.total && !p.causal && ctas < 2LL * c128::sm_count() && p.L >= 256;
  if (pre) {
    const size_t warps = (BHL + 3) / 4;
    const unsigned blocks = (unsigned)std::min<size_t>((warps + 7) / 8, (size_t)c128::sm_count() * 16);
    rnn_phi_kernel<T, D><<<blocks, 256, 0, s>>>(p, ws);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if constexpr (D >= 64) {
    // one column a warp when two a warp would leave fewer than two CTAs an SM
    if (ctas < 2LL * c128::sm_count()) return rnn_launch_g<T, D, 32, 32>(p, ws, pre, split, s);
    return rnn_launch_g<T, D, 16, kTileMany>(p, ws, pre, split, s);
  } else {
    return rnn_launch_g<T, D, 8, 32>(p, ws, pre, split, s);
  }
}

}  // namespace

size_t rnn_workspace_bytes(int B, int H, int L, int d) {
  return sizeof(float) * RnnWs((size_t)B * H * L, d).total;
}

cudaError_t launch_rnn_simt(const Problem& p, float* ws, size_t ws_bytes, cudaStream_t s) {
  const bool bf = p.dtype == DT_BF16;
  const size_t n = ws_bytes / sizeof(float);
  switch (p.d) {
    case 16: return bf ? rnn_launch<__nv_bfloat16, 16>(p, ws, n, s) : rnn_launch<float, 16>(p, ws, n, s);
    case 32: return bf ? rnn_launch<__nv_bfloat16, 32>(p, ws, n, s) : rnn_launch<float, 32>(p, ws, n, s);
    case 64: return bf ? rnn_launch<__nv_bfloat16, 64>(p, ws, n, s) : rnn_launch<float, 64>(p, ws, n, s);
    case 128: return bf ? rnn_launch<__nv_bfloat16, 128>(p, ws, n, s) : rnn_launch<float, 128>(p, ws, n, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace lion
