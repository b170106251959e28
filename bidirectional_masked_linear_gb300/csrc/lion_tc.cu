// lion_tc.cu -- chunkwise LION forward on the 5th-generation tensor cores
// (tcgen05 + TMEM + TMA), bfloat16 inputs, head dim 64, chunk 64.
//
// Chunkwise form ("LION Part IV - Results", "LION Chunk"; rebuttal page
// "LION: A bidirectional framework ...", reply "4: Practicality of Recurrent
// Inference" -- chunking).  Per head, chunk c covers tokens [s_c, e_c]; p is
// the chunk-local inclusive prefix of l = log(lambda):
//
//   intra     num_i += sum_{j in c} M_ij s_ij [v_j; 1],  M_ij = exp(p_max - p_min)
//   states    U^F_c = sum_j exp(p_e - p_j) phi(k_j) [v_j; 1]^T
//             U^B_c = sum_j exp(p_j - p_s) phi(k_j) [v_j; 1]^T
//   scans     F_{c+1} = exp(T_c) F_c + U^F_c,
//             G_{c-1} = exp(P_{s_{c+1}} - P_{s_c}) G_c + U^B_c
//   apply     num_i += a_i phi(q_i) [F_c z^F_c] + b_i phi(q_i) [G_c z^G_c]
//             a_i = exp(P_i - P_{e_{c-1}}),  b_i = exp(P_{s_{c+1}} - P_i)
//   y_i = num_i[0:d] / num_i[d]
//
// Normalisers ride on the tensor cores: products with V use B = [V_c | 1]
// (N = 80; a constant tile whose first column is 1 is the second atom), so
// U carries z as its column 64 and A V carries the intra-chunk row sum; the
// scanned z vectors of all chunks sit in one small operand tile.
//
// Precision: MMA operands are fp16 (11-bit significand) with fp32
// accumulation; phi(K), the decay-weighted phi(K), phi(Q), the chunk states,
// z, V and the masked scores are each rounded once to fp16.  (One bf16
// rounding of the unit-norm SiLU features costs ~5e-3 relative error; fp16
// stays within about half of the 2e-3 budget.)  Precondition of this path:
// |phi(q)|, |phi(k)|, |v| and the chunk states below the fp16 range (65504).
//
// Work split.  A persistent CTA (one per SM) walks heads bh = blockIdx.x,
// blockIdx.x + gridDim.x, ...  Per head:
//   A  per chunk: phi(K_c) -> fp16 in place, V_c -> fp16 in place, the
//      decay-weighted copies Kf_c, Kb_c; one M=128 MMA per chunk computes
//      U^F_c (TMEM lanes 0-63) and U^B_c (lanes 64-127):
//      A = [Kf_c ; Kb_c]^T (MN-major, two atoms), B = [V_c | 1] (MN-major).
//   B  scans over chunks (lanes 0-63 forward, 64-127 backward), writing the
//      states entering each chunk as fp16 operand tiles.
//   C  a two-deep pipeline over chunks: S = phi(Q_c) phi(K_c)^T,
//      O_F = phi(Q_c) F_c, O_G = phi(Q_c) G_c, Z = phi(Q_c) [z tiles]
//      (M=64 MMAs) run while the previous chunk's epilogue works; the decay
//      mask is applied to S on the CUDA cores (factorised as
//      exp(p_i - p_0) exp(p_0 - p_j) when the chunk's decay range allows);
//      O_I = A [V_c | 1]; the epilogue combines, normalises and stores fp32.
//      As chunk c of this head retires, TMA refills its K/V tiles with chunk
//      c of the next head; Q streams through a four-slot ring.
//
// Every mbarrier wait is bounded (one waiting thread, then a voting barrier);
// on timeout the CTA records an error in `status`, releases its TMEM and
// returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "lion_common.cuh"
#include "lion_internal.h"
#include "tc_ptx.cuh"

namespace lion {
namespace {

using namespace tc;

constexpr int kC = 64;           // chunk length handled here
constexpr int kD = 64;           // head dim
constexpr int kMaxChunks = 4;    // L <= 256
constexpr int kThreads = 512;
constexpr int kTile = kC * 128;  // bytes of one 64-row x 64-element 16-bit swizzled tile
constexpr int kQSlots = 4;
constexpr long long kWaitCycles = 2000000000LL;  // ~1 s at 2 GHz
constexpr float kMaxFactorRange = 80.f;          // exp(80) stays finite in fp32

// shared-memory map (bytes from a 1024-aligned base)
constexpr int OFF_K = 0;                               // phi(K) tiles, one per chunk
constexpr int OFF_V = OFF_K + kMaxChunks * kTile;      // V tiles
constexpr int OFF_ONES = OFF_V + kMaxChunks * kTile;   // column 0 = 1: the normaliser atom
constexpr int OFF_WORK = OFF_ONES + kTile;             // phase A: Kf/Kb tiles; B/C: states + z
constexpr int OFF_A = OFF_WORK + 2 * kMaxChunks * kTile;  // masked scores, 2 buffers
constexpr int OFF_Q = OFF_A + 2 * kTile;               // Q ring
constexpr int OFF_P = OFF_Q + kQSlots * kTile;         // float[256] chunk-local prefix
constexpr int OFF_E = OFF_P + 256 * 4;                 // float[2][2][64] mask factors per region
constexpr int OFF_MISC = OFF_E + 2 * 2 * kC * 4;       // float[8]: l at chunk starts
constexpr int OFF_BAR = OFF_MISC + 8 * 4;
constexpr int OFF_TSLOT = OFF_BAR + 16 * 8;
constexpr int kSmemBytes = OFF_TSLOT + 16 + 1024;      // + alignment slack
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

// work-region tiles in phases B/C: F_c (c = 1..3) at 0..2, G_c (c = 0..2) at
// 3..5, the z tile at 6 (column 2c: z^F_c, column 2c+1: z^G_c)
constexpr int W_Z = 6;

constexpr int BAR_KV = 0;    // + chunk
constexpr int BAR_Q = 4;     // + slot
constexpr int BAR_M1 = 8;    // + region: S, O_F, O_G, Z done
constexpr int BAR_M2 = 10;   // + region: O_I done
constexpr int BAR_A = 12;    // phase-A MMAs done

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSlot = 80;       // phase A/B: chunk-state slot (64 values + z + 15 zero)
constexpr uint32_t kRegion = 240;    // phase C: per in-flight chunk
constexpr uint32_t R_SI = 0, R_OF = 80, R_OG = 144, R_Z = 208;

struct TcParams {
  float* out;
  const float* log_lambda;
  int BH, H, L;
  int* status;
};

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ uint32_t pack_h2(float a, float b) { return h2u(__floats2half2_rn(a, b)); }
__device__ __forceinline__ float2 bf2_to_f2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
__device__ __forceinline__ uint4 pack8_h(const float* x) {
  return make_uint4(pack_h2(x[0], x[1]), pack_h2(x[2], x[3]), pack_h2(x[4], x[5]), pack_h2(x[6], x[7]));
}
__device__ __forceinline__ void unpack8_bf(uint4 v, float* x) {
  float2 a = bf2_to_f2(v.x), b = bf2_to_f2(v.y), c = bf2_to_f2(v.z), d = bf2_to_f2(v.w);
  x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y; x[4] = c.x; x[5] = c.y; x[6] = d.x; x[7] = d.y;
}
__device__ __forceinline__ void unpack8_h(uint4 v, float* x) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
    x[2 * e] = f.x;
    x[2 * e + 1] = f.y;
  }
}
__device__ __forceinline__ uint4* chunk16(uint8_t* tile, int r, int c8) {
  return reinterpret_cast<uint4*>(tile + sw128_offset(r, c8));
}
__device__ __forceinline__ __half* elem16(uint8_t* tile, int r, int col) {
  return reinterpret_cast<__half*>(tile + sw128_offset(r, col >> 3) + ((col & 7) << 1));
}

// phi on 8 features of one row; the row's 8 owners are lanes l..l+7 (xor 1,2,4).
template <int PHI>
__device__ __forceinline__ void phi8(float* x) {
  if (PHI == PHI_ELU1) {
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = x[e] > 0.f ? x[e] + 1.f : __expf(x[e]);
  } else if (PHI == PHI_SILU_L2) {
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      x[e] = __fdividef(x[e], 1.f + __expf(-x[e]));
      ss += x[e] * x[e];
    }
    ss += __shfl_xor_sync(0xffffffffu, ss, 1);
    ss += __shfl_xor_sync(0xffffffffu, ss, 2);
    ss += __shfl_xor_sync(0xffffffffu, ss, 4);
    const float inv = rsqrtf(fmaxf(ss, 1e-24f));
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] *= inv;
  }
}

__device__ __forceinline__ uint32_t lane_addr(uint32_t tbase, int warp, uint32_t col) {
  return tbase + ((uint32_t)(32 * (warp & 3)) << 16) + col;
}
__device__ __forceinline__ uint64_t kmaj(const uint8_t* tile, int k) {
  return desc_sw128(smem_u32(tile) + 32 * k, 16, 1024);
}
__device__ __forceinline__ uint64_t mnmaj(const uint8_t* tile, int k, uint32_t lbo) {
  return desc_sw128(smem_u32(tile) + 2048 * k, lbo, 1024);
}

template <int MASK, int PHI>
__global__ void __launch_bounds__(kThreads, 1)
    lion_chunk64_tc_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
                           const __grid_constant__ CUtensorMap mapV, TcParams prm) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sOnes = smem + OFF_ONES;
  uint8_t* sWork = smem + OFF_WORK;
  float* sP = reinterpret_cast<float*>(smem + OFF_P);
  float* sE = reinterpret_cast<float*>(smem + OFF_E);
  float* sMisc = reinterpret_cast<float*>(smem + OFF_MISC);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + OFF_TSLOT);
  auto Kt = [&](int c) { return smem + OFF_K + c * kTile; };
  auto Vt = [&](int c) { return smem + OFF_V + c * kTile; };
  auto Wt = [&](int i) { return sWork + i * kTile; };
  auto At = [&](int r) { return smem + OFF_A + r * kTile; };
  auto Qt = [&](int slot) { return smem + OFF_Q + slot * kTile; };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int L = prm.L, NC = (L + kC - 1) / kC;
  const int quarter = warp & 3, wg = warp >> 2;   // TMEM lane quarter, column group
  bool ok = true;                                 // uniform across the CTA

  // thread 0 waits on an mbarrier phase; the rest park in the voting barrier
  auto wait_all = [&](int b, uint32_t parity) {
    bool mine = true;
    if (tid == 0) mine = mbar_wait(&bars[b], parity, kWaitCycles);
    ok = __syncthreads_and(mine) && ok;
  };

  if (tid == 0) {
    prefetch_tmap(&mapQ);
    prefetch_tmap(&mapK);
    prefetch_tmap(&mapV);
    for (int b = 0; b < 13; ++b) mbar_init(&bars[b], 1);
    fence_mbar_init();
  }
  for (int x = tid; x < kC * 8; x += kThreads) {
    const int r = x >> 3, c8 = x & 7;
    *chunk16(sOnes, r, c8) = make_uint4(c8 == 0 ? pack_h2(1.f, 0.f) : 0u, 0u, 0u, 0u);
  }
  if (warp == 0) tmem_alloc(tslot, kTmemCols);
  fence_async_smem();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;

  auto issue_kv = [&](int bh_, int c) {
    mbar_arrive_expect_tx(&bars[BAR_KV + c], (uint32_t)(2 * kTile));
    tma_load_3d(Kt(c), &mapK, &bars[BAR_KV + c], 0, c * kC, bh_);
    tma_load_3d(Vt(c), &mapV, &bars[BAR_KV + c], 0, c * kC, bh_);
  };
  // the g-th Q chunk this CTA processes -> (head, chunk)
  auto issue_q = [&](int g) {
    const int itg = g / NC, c = g - itg * NC;
    const int bh_ = blockIdx.x + itg * gridDim.x;
    if (bh_ >= prm.BH) return;
    const int sl = g % kQSlots;
    mbar_arrive_expect_tx(&bars[BAR_Q + sl], (uint32_t)kTile);
    tma_load_3d(Qt(sl), &mapQ, &bars[BAR_Q + sl], 0, c * kC, bh_);
  };
  if (tid == 0) {
    for (int c = 0; c < NC; ++c) issue_kv(blockIdx.x, c);
    for (int g = 0; g < kQSlots; ++g) issue_q(g);
  }

  int gq = 0;   // chunks this CTA has taken through phase C
  int it = 0;
  for (int bh = blockIdx.x; bh < prm.BH && ok; bh += gridDim.x, ++it) {
    const int h = bh % prm.H;
    const float lh = MASK == MASK_D ? prm.log_lambda[h] : 0.f;
    // chunk-local inclusive prefixes (one warp per chunk, 2 tokens per lane)
    if (warp < NC) {
      const int c = warp, s = c * kC;
      float l0 = 0.f, l1 = 0.f;
      const int t0 = s + 2 * lane, t1 = t0 + 1;
      if (MASK == MASK_S) {
        const float* ll = prm.log_lambda + (size_t)bh * L;
        l0 = t0 < L ? ll[t0] : 0.f;
        l1 = t1 < L ? ll[t1] : 0.f;
      } else if (MASK == MASK_D) {
        l0 = t0 < L ? lh : 0.f;
        l1 = t1 < L ? lh : 0.f;
      }
      const float pair = l0 + l1;
      float x = pair;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      const float excl = x - pair;
      sP[s + 2 * lane] = excl + l0;
      sP[s + 2 * lane + 1] = excl + l0 + l1;
      if (lane == 0) sMisc[c] = l0;   // l at s_c
    }
    if (tid == 0) sMisc[NC] = 0.f;    // no token after the sequence
    __syncthreads();

    // ---------------- phase A: chunk states ------------------------------
    for (int c = 0; c < NC; ++c) {
      wait_all(BAR_KV + c, it & 1);
      if (!ok) break;
      const int len = min(kC, L - c * kC);
      const int r = tid >> 3, c8 = tid & 7;
      float x[8];
      unpack8_bf(*chunk16(Kt(c), r, c8), x);
      phi8<PHI>(x);      // every lane: phi8 shuffles within the row's 8 lanes
      if (r >= len) {    // padding tokens contribute nothing
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = 0.f;
      }
      const uint4 kh = pack8_h(x);
      *chunk16(Kt(c), r, c8) = kh;
      unpack8_h(kh, x);  // the decay weights multiply the fp16 phi(k) that S sees
      float wf = 1.f, wb = 1.f;
      if (MASK != MASK_LIT) {
        const float pj = sP[c * kC + r];
        wf = __expf(sP[c * kC + len - 1] - pj);
        wb = __expf(pj - sP[c * kC]);
      }
      float y[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) y[e] = wf * x[e];
      *chunk16(Wt(2 * c), r, c8) = pack8_h(y);
#pragma unroll
      for (int e = 0; e < 8; ++e) y[e] = wb * x[e];
      *chunk16(Wt(2 * c + 1), r, c8) = pack8_h(y);
      float v8[8];
      unpack8_bf(*chunk16(Vt(c), r, c8), v8);
      *chunk16(Vt(c), r, c8) = pack8_h(v8);
    }
    if (!ok) break;
    fence_async_smem();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      const uint32_t idA = idesc_f16(128, 80, true, true);
      for (int c = 0; c < NC; ++c) {
        const uint32_t lbo_v = (uint32_t)(sOnes - Vt(c));
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_bf16(tbase + kSlot * c, mnmaj(Wt(2 * c), k, kTile), mnmaj(Vt(c), k, lbo_v), idA, k > 0 ? 1u : 0u);
      }
      mma_commit(&bars[BAR_A]);
    }
    wait_all(BAR_A, it & 1);
    if (!ok) break;
    tc_fence_after();

    // ---------------- phase B: scans -> fp16 state operand tiles ----------
    {
      // zero the z tile's first 16 columns (stale phase-A data otherwise)
      if (tid < 2 * kC) *chunk16(Wt(W_Z), tid >> 1, tid & 1) = make_uint4(0u, 0u, 0u, 0u);
      __syncthreads();
      const bool fwd = quarter < 2;
      const int m = 32 * (quarter & 1) + lane;
      const int ncol = wg == 3 ? 2 : 1;   // column group 3 also carries the z column
      float stv[2][16];
#pragma unroll
      for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int e = 0; e < 16; ++e) stv[a][e] = 0.f;
      for (int cc = 0; cc < NC; ++cc) {
        const int c = fwd ? cc : NC - 1 - cc;
        const int len = min(kC, L - c * kC);
        const bool write = fwd ? c > 0 : c < NC - 1;
        uint8_t* dst = fwd ? Wt(c - 1) : Wt(3 + c);
        float u[2][16];
#pragma unroll
        for (int a = 0; a < 2; ++a)
          if (a < ncol) tmem_ld16(lane_addr(tbase, warp, kSlot * c + (a == 0 ? 16 * wg : 64)), u[a]);
        if (write) {   // state entering chunk c
          *chunk16(dst, m, 2 * wg) = pack8_h(stv[0]);
          *chunk16(dst, m, 2 * wg + 1) = pack8_h(stv[0] + 8);
          if (wg == 3) *elem16(Wt(W_Z), m, 2 * c + (fwd ? 0 : 1)) = __float2half_rn(stv[1][0]);
        }
        tmem_wait_ld();
        float decay = 1.f;
        if (MASK != MASK_LIT) {
          const float T = sP[c * kC + len - 1];
          decay = fwd ? __expf(T) : __expf(T - sMisc[c] + sMisc[c + 1]);
        }
#pragma unroll
        for (int a = 0; a < 2; ++a)
          if (a < ncol)
#pragma unroll
            for (int e = 0; e < 16; ++e) stv[a][e] = decay * stv[a][e] + u[a][e];
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---------------- phase C: two-deep pipeline over chunks ---------------
    const uint32_t idS = idesc_f16(64, 64, false, false);
    const uint32_t idO = idesc_f16(64, 64, false, true);
    const uint32_t idI = idesc_f16(64, 80, false, true);
    const uint32_t idZ = idesc_f16(64, 8, false, true);
    const int i_row = 16 * quarter + lane;     // M=64 accumulator row of this lane
    const bool row_thread = lane < 16;

    // phi(Q_c) -> fp16, mask factors of chunk c, then the first MMA group
    auto prep_and_mma1 = [&](int c, int g) {
      const int sl = g % kQSlots, rg = g & 1;
      wait_all(BAR_Q + sl, (g / kQSlots) & 1);
      if (!ok) return;
      const int len = min(kC, L - c * kC);
      {
        const int r = tid >> 3, c8 = tid & 7;
        float x[8];
        unpack8_bf(*chunk16(Qt(sl), r, c8), x);
        phi8<PHI>(x);
        if (r >= len) {
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] = 0.f;
        }
        *chunk16(Qt(sl), r, c8) = pack8_h(x);
      }
      if (MASK != MASK_LIT && tid < 2 * kC) {
        // E[t] = exp(p_t - p_0), Einv[t] = exp(p_0 - p_t)
        const int t = tid & 63;
        const float d = sP[c * kC + t] - sP[c * kC];
        sE[(rg * 2 + (tid >> 6)) * kC + t] = tid < 64 ? __expf(d) : __expf(-d);
      }
      fence_async_smem();
      __syncthreads();
      if (tid == 0) {
        tc_fence_after();
        const uint32_t base = tbase + kRegion * rg;
        const uint8_t* qt = Qt(sl);
#pragma unroll
        for (int k = 0; k < 4; ++k) mma_bf16(base + R_SI, kmaj(qt, k), kmaj(Kt(c), k), idS, k > 0 ? 1u : 0u);
        if (c > 0) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_bf16(base + R_OF, kmaj(qt, k), mnmaj(Wt(c - 1), k, kTile), idO, k > 0 ? 1u : 0u);
        }
        if (c < NC - 1) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_bf16(base + R_OG, kmaj(qt, k), mnmaj(Wt(3 + c), k, kTile), idO, k > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) mma_bf16(base + R_Z, kmaj(qt, k), mnmaj(Wt(W_Z), k, kTile), idZ, k > 0 ? 1u : 0u);
        mma_commit(&bars[BAR_M1 + rg]);
      }
    };

    // masked scores -> fp16 A tile, then O_I = A [V_c | 1]
    auto epi1_and_mma2 = [&](int c, int g) {
      const int rg = g & 1, sl = g % kQSlots;
      wait_all(BAR_M1 + rg, (g >> 1) & 1);
      if (!ok) return;
      tc_fence_after();
      if (tid == 0) issue_q(g + kQSlots);   // this Q slot's MMAs are done
      const int s = c * kC, len = min(kC, L - s);
      const uint32_t base = tbase + kRegion * rg;
      float w[16];
      tmem_ld16(lane_addr(base, warp, R_SI + 16 * wg), w);
      tmem_wait_ld();
      if (row_thread) {
        const int i = i_row;
        const float* E = sE + (rg * 2) * kC;
        const float* Einv = E + kC;
        const bool factor = (MASK == MASK_LIT) || (sP[s] - sP[s + len - 1] < kMaxFactorRange);
        const float Ei = MASK == MASK_LIT ? 1.f : E[i];
        const float Einvi = MASK == MASK_LIT ? 1.f : Einv[i];
        const float pi = sP[s + i];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int j = 16 * wg + e;
          float mval;
          if (MASK == MASK_LIT) {
            mval = 1.f;
          } else if (factor) {
            mval = j <= i ? Ei * Einv[j] : Einvi * E[j];
          } else {
            const float pj = sP[s + j];
            mval = __expf(j <= i ? pi - pj : pj - pi);
          }
          w[e] = (i < len && j < len) ? w[e] * mval : 0.f;
        }
        *chunk16(At(rg), i, 2 * wg) = pack8_h(w);
        *chunk16(At(rg), i, 2 * wg + 1) = pack8_h(w + 8);
      }
      fence_async_smem();
      tc_fence_before();
      __syncthreads();
      if (tid == 0) {
        tc_fence_after();
        const uint32_t lbo_v = (uint32_t)(sOnes - Vt(c));
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_bf16(base + R_SI, kmaj(At(rg), k), mnmaj(Vt(c), k, lbo_v), idI, k > 0 ? 1u : 0u);
        mma_commit(&bars[BAR_M2 + rg]);
      }
      (void)sl;
    };

    // combine, normalise, store; then hand chunk c's K/V tiles to the next head
    auto epi2 = [&](int c, int g) {
      const int rg = g & 1;
      wait_all(BAR_M2 + rg, (g >> 1) & 1);
      if (!ok) return;
      tc_fence_after();
      const int s = c * kC, len = min(kC, L - s);
      const bool hasF = c > 0, hasG = c < NC - 1;
      const uint32_t base = tbase + kRegion * rg;
      float oi[16], of[16], og[16], zz[16];
      tmem_ld16(lane_addr(base, warp, R_SI + 16 * wg), oi);
      const float dI = tmem_ld1(lane_addr(base, warp, R_SI + 64));
      if (hasF) tmem_ld16(lane_addr(base, warp, R_OF + 16 * wg), of);
      if (hasG) tmem_ld16(lane_addr(base, warp, R_OG + 16 * wg), og);
      const float dF = tmem_ld1(lane_addr(base, warp, R_Z + 2 * c));
      const float dG = tmem_ld1(lane_addr(base, warp, R_Z + 2 * c + 1));
      tmem_wait_ld();
      (void)zz;
      if (row_thread && i_row < len) {
        const int i = i_row;
        const float pi = sP[s + i];
        float a = 0.f, b = 0.f;
        if (hasF) a = MASK == MASK_LIT ? 1.f : __expf(pi);
        if (hasG) b = MASK == MASK_LIT ? 1.f : __expf(sP[s + len - 1] - pi + sMisc[c + 1]);
        float den = dI;
        if (hasF) den += a * dF;
        if (hasG) den += b * dG;
        const float inv = 1.f / den;
        float y[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float acc = oi[e];
          if (hasF) acc += a * of[e];
          if (hasG) acc += b * og[e];
          y[e] = acc * inv;
        }
        float* orow = prm.out + ((size_t)bh * L + s + i) * kD + 16 * wg;
#pragma unroll
        for (int e = 0; e < 16; e += 4)
          *reinterpret_cast<float4*>(orow + e) = make_float4(y[e], y[e + 1], y[e + 2], y[e + 3]);
      }
      tc_fence_before();
      __syncthreads();
      // K_c and V_c are no longer read: refill them with the next head's chunk c
      if (tid == 0 && bh + (int)gridDim.x < prm.BH) issue_kv(bh + gridDim.x, c);
    };

    prep_and_mma1(0, gq);
    if (NC > 1 && ok) prep_and_mma1(1, gq + 1);
    if (ok) epi1_and_mma2(0, gq);
    for (int c = 1; c < NC && ok; ++c) {
      epi1_and_mma2(c, gq + c);
      if (ok) epi2(c - 1, gq + c - 1);
      if (ok && c + 1 < NC) prep_and_mma1(c + 1, gq + c + 1);
    }
    if (ok) epi2(NC - 1, gq + NC - 1);
    gq += NC;
  }

  if (!ok && tid == 0) atomicExch(prm.status, 1);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
    tmem_relinquish();
  }
}

__device__ int g_lion_status;

// ------------------------------------------------------------- host side --
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// [BH][L][64] bf16 viewed as a 3-D tensor; box = 64 columns x 64 rows x 1.
bool make_map(CUtensorMap* m, const void* base, int L, int BH) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)L, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)L * kD * 2};
  cuuint32_t box[3] = {(cuuint32_t)kD, (cuuint32_t)kC, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int* device_status_ptr() {
  static int* cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (!cache[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_lion_status) != cudaSuccess) return nullptr;
    cache[dev] = static_cast<int*>(p);
  }
  return cache[dev];
}

bool chunk_tc_supported(const Problem& p) {
  return p.dtype == DT_BF16 && p.d == kD && p.chunk == kC && p.L <= kMaxChunks * kC;
}


cudaError_t launch_chunk_tc(const Problem& p, int* status, cudaStream_t s) {
  CUtensorMap mq, mk, mv;
  const int BH = p.B * p.H;
  if (!make_map(&mq, p.q, p.L, BH) || !make_map(&mk, p.k, p.L, BH) || !make_map(&mv, p.v, p.L, BH))
    return cudaErrorInvalidValue;
  TcParams prm;
  prm.out = p.out;
  prm.log_lambda = p.log_lambda;
  prm.BH = BH;
  prm.H = p.H;
  prm.L = p.L;
  prm.status = status;
  static int num_sms = 0;
  if (!num_sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (num_sms <= 0) num_sms = 1;
  }
  const int grid = BH < num_sms ? BH : num_sms;
  void (*kern)(const CUtensorMap, const CUtensorMap, const CUtensorMap, TcParams) = nullptr;
#define LION_TC_CASE(M, F) \
  if (p.mask_kind == M && p.phi == F) kern = lion_chunk64_tc_kernel<M, F>;
  LION_TC_CASE(MASK_LIT, PHI_ELU1)
  LION_TC_CASE(MASK_LIT, PHI_SILU_L2)
  LION_TC_CASE(MASK_LIT, PHI_IDENTITY)
  LION_TC_CASE(MASK_D, PHI_ELU1)
  LION_TC_CASE(MASK_D, PHI_SILU_L2)
  LION_TC_CASE(MASK_D, PHI_IDENTITY)
  LION_TC_CASE(MASK_S, PHI_ELU1)
  LION_TC_CASE(MASK_S, PHI_SILU_L2)
  LION_TC_CASE(MASK_S, PHI_IDENTITY)
#undef LION_TC_CASE
  if (!kern) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, kSmemBytes, s>>>(mq, mk, mv, prm);
  return cudaGetLastError();
}

}  // namespace lion
