// lion_tc.cu -- chunkwise LION forward on the 5th-generation tensor cores
// (tcgen05 + TMEM + TMA), bfloat16 inputs, head dim 64, chunk 64.
//
// Chunkwise form ("LION Part IV - Results", "LION Chunk"; rebuttal page
// "LION: A bidirectional framework ...", reply "4: Practicality of Recurrent
// Inference" -- chunking).  Per head, chunk c covers tokens [s_c, e_c]; p is
// the chunk-local inclusive prefix of l = log(lambda):
//
//   intra     num_i += sum_{j in c} M_ij s_ij v_j,  M_ij = exp(p_max - p_min)
//   states    U^F_c = sum_j exp(p_e - p_j) phi(k_j) [v_j; 1]^T
//             U^B_c = sum_j exp(p_j - p_s) phi(k_j) [v_j; 1]^T
//   scans     F_{c+1} = exp(T_c) F_c + U^F_c,
//             G_{c-1} = exp(P_{s_{c+1}} - P_{s_c}) G_c + U^B_c
//   apply     num_i += exp(p_i) phi(q_i) F_c + exp(P_{s_{c+1}} - P_i) phi(q_i) G_c
//   y_i = num_i / den_i   (the row-sum normaliser rides along as column d+1)
//
// One CTA owns one (batch, head) sequence of L <= 256 tokens (<= 4 chunks).
// Phases inside the CTA:
//   0  TMA loads Q, K, V (128-byte swizzled tiles, out-of-range rows zero);
//      chunk-local prefixes of l; phi applied in place (padding rows zeroed);
//      decay-weighted copies of phi(K) for the two state directions;
//      normaliser columns z^F_c, z^B_c (CUDA cores).
//   A  one M=128 MMA per chunk computes U^F_c (TMEM lanes 0-63) and U^B_c
//      (lanes 64-127) together: A = [Kf_c ; Kb_c]^T (MN-major, two atoms),
//      B = V_c (MN-major).
//   B  warps 0-1 scan the forward states, warps 2-3 the backward states, each
//      thread one state row, and write them as bf16 MMA operands.
//   C  per chunk: S = phi(Q_c) phi(K_c)^T, O_F = phi(Q_c) F_c,
//      O_G = phi(Q_c) G_c (M=64 MMAs); the mask is applied to S in
//      registers and written back as an exact hi+lo bf16 pair; O_intra =
//      (A_hi + A_lo) V_c; the epilogue combines, normalises, stores fp32.
//
// Every mbarrier wait is bounded; on timeout the CTA records an error in
// `status`, releases its TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>

#include "lion_common.cuh"
#include "lion_internal.h"
#include "tc_ptx.cuh"

namespace lion {
namespace {

using namespace tc;

constexpr int kC = 64;           // chunk length handled here
constexpr int kD = 64;           // head dim
constexpr int kMaxChunks = 4;    // L <= 256
constexpr int kThreads = 128;
constexpr int kTile = kC * 128;  // bytes of one 64-row x 64-bf16 swizzled tile
constexpr long long kWaitCycles = 2000000000LL;  // ~1 s at 2 GHz

// shared-memory map (bytes from a 1024-aligned base)
constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + kMaxChunks * kTile;
constexpr int OFF_V = OFF_K + kMaxChunks * kTile;
constexpr int OFF_KF = OFF_V + kMaxChunks * kTile;   // phase 0/A; then F tiles
constexpr int OFF_KB = OFF_KF + kMaxChunks * kTile;  // phase 0/A; then G tiles
constexpr int OFF_AHI = OFF_KB + kMaxChunks * kTile;
constexpr int OFF_ALO = OFF_AHI + kTile;
constexpr int OFF_P = OFF_ALO + kTile;               // float[256] chunk-local prefix
constexpr int OFF_ZFL = OFF_P + 256 * 4;             // float[4][64] chunk-local z (fwd)
constexpr int OFF_ZBL = OFF_ZFL + kMaxChunks * kD * 4;
constexpr int OFF_ZF = OFF_ZBL + kMaxChunks * kD * 4;  // float[4][64] scanned z (fwd)
constexpr int OFF_ZB = OFF_ZF + kMaxChunks * kD * 4;
constexpr int OFF_MISC = OFF_ZB + kMaxChunks * kD * 4;  // float[16]: l at chunk starts etc.
constexpr int OFF_BAR = OFF_MISC + 16 * 4;
constexpr int OFF_TSLOT = OFF_BAR + 8 * 8;
constexpr int kSmemBytes = OFF_TSLOT + 16 + 1024;   // + alignment slack

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t TM_U = 0;      // phase A: 4 x 64 columns
constexpr uint32_t TM_S = 256;    // phase C
constexpr uint32_t TM_OF = 320;
constexpr uint32_t TM_OG = 384;
constexpr uint32_t TM_OI = 448;

struct TcParams {
  float* out;
  const float* log_lambda;
  int H, L, mask_kind, phi;
  int* status;
};

__device__ __forceinline__ float bf2f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }
__device__ __forceinline__ uint16_t f2bf(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  return (uint32_t)f2bf(a) | ((uint32_t)f2bf(b) << 16);
}

// element (row r, column m) of a swizzled 64x64 bf16 tile
__device__ __forceinline__ uint16_t* tile_elem(uint8_t* tile, int r, int m) {
  return reinterpret_cast<uint16_t*>(tile + sw128_offset(r, m >> 3) + ((m & 7) << 1));
}

// write 64 fp32 values as one bf16 row of a swizzled tile
__device__ __forceinline__ void store_row_bf16(uint8_t* tile, int r, const float* x) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    uint4 v;
    v.x = pack2(x[8 * c + 0], x[8 * c + 1]);
    v.y = pack2(x[8 * c + 2], x[8 * c + 3]);
    v.z = pack2(x[8 * c + 4], x[8 * c + 5]);
    v.w = pack2(x[8 * c + 6], x[8 * c + 7]);
    *reinterpret_cast<uint4*>(tile + sw128_offset(r, c)) = v;
  }
}

__device__ __forceinline__ void load_row_f32(const uint8_t* tile, int r, float* x) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint4 v = *reinterpret_cast<const uint4*>(tile + sw128_offset(r, c));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      x[8 * c + 2 * e] = bf2f((uint16_t)(w[e] & 0xffffu));
      x[8 * c + 2 * e + 1] = bf2f((uint16_t)(w[e] >> 16));
    }
  }
}

__device__ __forceinline__ void phi_row(float* x, int phi) {
  if (phi == PHI_ELU1) {
#pragma unroll
    for (int m = 0; m < kD; ++m) x[m] = x[m] > 0.f ? x[m] + 1.f : __expf(x[m]);
  } else if (phi == PHI_SILU_L2) {
    float ss = 0.f;
#pragma unroll
    for (int m = 0; m < kD; ++m) {
      const float u = x[m] / (1.f + __expf(-x[m]));
      x[m] = u;
      ss += u * u;
    }
    const float inv = 1.f / fmaxf(sqrtf(ss), 1e-12f);
#pragma unroll
    for (int m = 0; m < kD; ++m) x[m] *= inv;
  }
}

// 16 TMEM columns of this thread's lane -> v
__device__ __forceinline__ void tmem_row16(uint32_t tbase, int warp, uint32_t col, float* v) {
  tmem_ld16(tbase + ((uint32_t)(32 * warp) << 16) + col, v);
}

__global__ void __launch_bounds__(kThreads, 1)
    lion_chunk64_tc_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
                           const __grid_constant__ CUtensorMap mapV, TcParams prm) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + OFF_Q;
  uint8_t* sK = smem + OFF_K;
  uint8_t* sV = smem + OFF_V;
  uint8_t* sKf = smem + OFF_KF;
  uint8_t* sKb = smem + OFF_KB;
  uint8_t* sF = sKf;   // reused after phase A
  uint8_t* sG = sKb;
  uint8_t* sAhi = smem + OFF_AHI;
  uint8_t* sAlo = smem + OFF_ALO;
  float* sP = reinterpret_cast<float*>(smem + OFF_P);
  float* sZFl = reinterpret_cast<float*>(smem + OFF_ZFL);
  float* sZBl = reinterpret_cast<float*>(smem + OFF_ZBL);
  float* sZF = reinterpret_cast<float*>(smem + OFF_ZF);
  float* sZB = reinterpret_cast<float*>(smem + OFF_ZB);
  float* sMisc = reinterpret_cast<float*>(smem + OFF_MISC);   // [c] = l at s_c
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);  // 0: TMA, 1: MMA
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + OFF_TSLOT);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bh = blockIdx.x, h = bh % prm.H, L = prm.L;
  const int NC = (L + kC - 1) / kC;
  const float lh = prm.mask_kind == MASK_D ? prm.log_lambda[h] : 0.f;
  bool ok = true;   // kept uniform across the CTA (every wait is followed by a voting barrier)

  if (tid == 0) {
    prefetch_tmap(&mapQ);
    prefetch_tmap(&mapK);
    prefetch_tmap(&mapV);
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tslot, kTmemCols);
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  uint32_t mma_phase = 0;

  // ---------------- phase 0: loads, prefixes, phi, weighted copies ------
  if (tid == 0) {
    mbar_arrive_expect_tx(&bars[0], (uint32_t)(3 * NC * kTile));
    for (int c = 0; c < NC; ++c) {
      tma_load_3d(sQ + c * kTile, &mapQ, &bars[0], 0, c * kC, bh);
      tma_load_3d(sK + c * kTile, &mapK, &bars[0], 0, c * kC, bh);
      tma_load_3d(sV + c * kTile, &mapV, &bars[0], 0, c * kC, bh);
    }
  }
  // chunk-local inclusive prefixes (one warp per chunk, 2 tokens per lane)
  if (warp < NC) {
    const int c = warp, s = c * kC;
    float l0 = 0.f, l1 = 0.f;
    const int t0 = s + 2 * lane, t1 = t0 + 1;
    if (prm.mask_kind == MASK_S) {
      const float* ll = prm.log_lambda + (size_t)bh * L;
      l0 = t0 < L ? ll[t0] : 0.f;
      l1 = t1 < L ? ll[t1] : 0.f;
    } else if (prm.mask_kind == MASK_D) {
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
  if (tid == 0) sMisc[NC] = 0.f;    // no token after the block
  ok = mbar_wait(&bars[0], 0, kWaitCycles);
  ok = __syncthreads_and(ok);

  if (ok) {
    // phi in place on Q and K (one thread per row) and the decay-weighted
    // phi(K) copies of the two state directions; padding rows become zero.
    for (int r = tid; r < NC * kC; r += kThreads) {
      const int c = r / kC, j = r - c * kC;
      const int len = min(kC, L - c * kC);
      float x[kD];
      load_row_f32(sQ + c * kTile, j, x);
      if (j < len) {
        phi_row(x, prm.phi);
      } else {
#pragma unroll
        for (int m = 0; m < kD; ++m) x[m] = 0.f;
      }
      store_row_bf16(sQ + c * kTile, j, x);
      load_row_f32(sK + c * kTile, j, x);
      if (j < len) {
        phi_row(x, prm.phi);
      } else {
#pragma unroll
        for (int m = 0; m < kD; ++m) x[m] = 0.f;
      }
      store_row_bf16(sK + c * kTile, j, x);
      // forward weight exp(p_e - p_j), backward weight exp(p_j - p_s)
      const float pj = sP[c * kC + j];
      const float wf = j < len ? __expf(sP[c * kC + len - 1] - pj) : 0.f;
      const float wb = j < len ? __expf(pj - sP[c * kC]) : 0.f;
      load_row_f32(sK + c * kTile, j, x);   // the rounded phi(k) the MMAs see
      float y[kD];
#pragma unroll
      for (int m = 0; m < kD; ++m) y[m] = wf * x[m];
      store_row_bf16(sKf + c * kTile, j, y);
#pragma unroll
      for (int m = 0; m < kD; ++m) y[m] = wb * x[m];
      store_row_bf16(sKb + c * kTile, j, y);
    }
    fence_async_smem();
    __syncthreads();

    // ---------------- phase A: chunk states on the tensor cores ---------
    if (tid == 0) {
      tc_fence_after();
      const uint32_t idA = idesc_bf16(128, 64, true, true);
      const uint32_t lbo = (uint32_t)(OFF_KB - OFF_KF);
      for (int c = 0; c < NC; ++c) {
        const uint32_t aKf = smem_u32(sKf + c * kTile), aV = smem_u32(sV + c * kTile);
#pragma unroll
        for (int k = 0; k < kC / 16; ++k)
          mma_bf16(tbase + TM_U + 64 * c, desc_sw128(aKf + 2048 * k, lbo, 1024),
                   desc_sw128(aV + 2048 * k, 8192, 1024), idA, k > 0 ? 1u : 0u);
      }
      mma_commit(&bars[1]);
    }
    // normaliser columns of the chunk states (CUDA cores, same bf16 values)
    {
      const int m = tid & 63;
      const bool fwd = tid < 64;
      uint8_t* src = fwd ? sKf : sKb;
      float* dst = fwd ? sZFl : sZBl;
      for (int c = 0; c < NC; ++c) {
        float acc = 0.f;
        for (int j = 0; j < kC; ++j) acc += bf2f(*tile_elem(src + c * kTile, j, m));
        dst[c * kD + m] = acc;
      }
    }
    ok = mbar_wait(&bars[1], mma_phase, kWaitCycles);
    mma_phase ^= 1;
    tc_fence_after();
    ok = __syncthreads_and(ok);   // z sums done before sKf/sKb are overwritten
  }

  if (ok) {
    // ---------------- phase B: scans over chunks -------------------------
    const bool fwd = warp < 2;
    const int m = tid & 63;
    float st[kD];
#pragma unroll
    for (int n = 0; n < kD; ++n) st[n] = 0.f;
    float z = 0.f;
    for (int cc = 0; cc < NC; ++cc) {
      const int c = fwd ? cc : NC - 1 - cc;
      const int len = min(kC, L - c * kC);
      if (fwd && c > 0) {
        store_row_bf16(sF + c * kTile, m, st);
        sZF[c * kD + m] = z;
      }
      if (!fwd && c < NC - 1) {
        store_row_bf16(sG + c * kTile, m, st);
        sZB[c * kD + m] = z;
      }
      // carry across chunk c: forward exp(T_c); backward exp(P_{s_{c+1}} - P_{s_c})
      const float T = sP[c * kC + len - 1];
      const float decay = fwd ? __expf(T) : __expf(T - sMisc[c] + sMisc[c + 1]);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        float u[16];
        tmem_row16(tbase, warp, TM_U + 64 * c + 16 * q4, u);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e) st[16 * q4 + e] = decay * st[16 * q4 + e] + u[e];
      }
      z = decay * z + (fwd ? sZFl : sZBl)[c * kD + m];
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }

  // ---------------- phase C: per-chunk outputs ----------------------------
  const int rrow = 16 * warp + lane;        // M=64 row held by this thread
  const bool row_thread = lane < 16;
  for (int c = 0; c < NC && ok; ++c) {
    const int s = c * kC, len = min(kC, L - s);
    const bool hasF = c > 0, hasG = c < NC - 1;
    if (tid == 0) {
      tc_fence_after();
      const uint32_t aQ = smem_u32(sQ + c * kTile), aK = smem_u32(sK + c * kTile);
      const uint32_t idS = idesc_bf16(64, 64, false, false);
      const uint32_t idO = idesc_bf16(64, 64, false, true);
#pragma unroll
      for (int k = 0; k < 4; ++k)
        mma_bf16(tbase + TM_S, desc_sw128(aQ + 32 * k, 16, 1024), desc_sw128(aK + 32 * k, 16, 1024), idS,
                 k > 0 ? 1u : 0u);
      if (hasF) {
        const uint32_t aF = smem_u32(sF + c * kTile);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_bf16(tbase + TM_OF, desc_sw128(aQ + 32 * k, 16, 1024), desc_sw128(aF + 2048 * k, 8192, 1024),
                   idO, k > 0 ? 1u : 0u);
      }
      if (hasG) {
        const uint32_t aG = smem_u32(sG + c * kTile);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_bf16(tbase + TM_OG, desc_sw128(aQ + 32 * k, 16, 1024), desc_sw128(aG + 2048 * k, 8192, 1024),
                   idO, k > 0 ? 1u : 0u);
      }
      mma_commit(&bars[1]);
    }
    ok = mbar_wait(&bars[1], mma_phase, kWaitCycles);
    mma_phase ^= 1;
    tc_fence_after();
    ok = __syncthreads_and(ok);
    if (!ok) break;

    // epilogue 1: mask S in registers, row sums, exact hi + lo bf16 split
    float den_intra = 0.f;
    {
      const int i = rrow;
      const float pi = row_thread ? sP[s + i] : 0.f;
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        float w[16];
        tmem_row16(tbase, warp, TM_S + 16 * q4, w);
        tmem_wait_ld();
        if (row_thread) {
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            float hv[8], lv[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const int j = 16 * q4 + 8 * half + e;
              float x = 0.f;
              if (i < len && j < len) {
                float ex;
                if (prm.mask_kind == MASK_LIT) ex = 0.f;
                else if (prm.mask_kind == MASK_D) ex = (float)(i >= j ? i - j : j - i) * lh;
                else ex = i >= j ? pi - sP[s + j] : sP[s + j] - pi;
                x = w[8 * half + e] * __expf(ex);
              }
              den_intra += x;
              const float xh = __bfloat162float(__float2bfloat16_rn(x));
              hv[e] = xh;
              lv[e] = x - xh;
            }
            const int c8 = 2 * q4 + half;
            *reinterpret_cast<uint4*>(sAhi + sw128_offset(i, c8)) =
                make_uint4(pack2(hv[0], hv[1]), pack2(hv[2], hv[3]), pack2(hv[4], hv[5]), pack2(hv[6], hv[7]));
            *reinterpret_cast<uint4*>(sAlo + sw128_offset(i, c8)) =
                make_uint4(pack2(lv[0], lv[1]), pack2(lv[2], lv[3]), pack2(lv[4], lv[5]), pack2(lv[6], lv[7]));
          }
        }
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      const uint32_t aH = smem_u32(sAhi), aL = smem_u32(sAlo), aV = smem_u32(sV + c * kTile);
      const uint32_t idO = idesc_bf16(64, 64, false, true);
#pragma unroll
      for (int k = 0; k < 4; ++k)
        mma_bf16(tbase + TM_OI, desc_sw128(aH + 32 * k, 16, 1024), desc_sw128(aV + 2048 * k, 8192, 1024), idO,
                 k > 0 ? 1u : 0u);
#pragma unroll
      for (int k = 0; k < 4; ++k)
        mma_bf16(tbase + TM_OI, desc_sw128(aL + 32 * k, 16, 1024), desc_sw128(aV + 2048 * k, 8192, 1024), idO,
                 1u);
      mma_commit(&bars[1]);
    }
    ok = mbar_wait(&bars[1], mma_phase, kWaitCycles);
    mma_phase ^= 1;
    tc_fence_after();
    ok = __syncthreads_and(ok);
    if (!ok) break;

    // epilogue 2: combine the three contributions, normalise, store
    {
      const int i = rrow;
      const bool live = row_thread && i < len;
      float a = 0.f, b = 0.f, den = den_intra;
      if (live) {
        const float pi = sP[s + i];
        float q[kD];
        load_row_f32(sQ + c * kTile, i, q);
        if (hasF) {
          a = __expf(pi);
          float dz = 0.f;
#pragma unroll
          for (int m = 0; m < kD; ++m) dz += q[m] * sZF[c * kD + m];
          den += a * dz;
        }
        if (hasG) {
          b = __expf(sP[s + len - 1] - pi + sMisc[c + 1]);
          float dz = 0.f;
#pragma unroll
          for (int m = 0; m < kD; ++m) dz += q[m] * sZB[c * kD + m];
          den += b * dz;
        }
      }
      const float inv = 1.f / den;
      float* orow = prm.out + ((size_t)bh * L + s + (live ? i : 0)) * kD;
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        float oi[16], of[16], og[16];
        tmem_row16(tbase, warp, TM_OI + 16 * q4, oi);
        if (hasF) tmem_row16(tbase, warp, TM_OF + 16 * q4, of);
        if (hasG) tmem_row16(tbase, warp, TM_OG + 16 * q4, og);
        tmem_wait_ld();
        if (live) {
          float y[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float acc = oi[e];
            if (hasF) acc += a * of[e];
            if (hasG) acc += b * og[e];
            y[e] = acc * inv;
          }
#pragma unroll
          for (int e = 0; e < 16; e += 4)
            *reinterpret_cast<float4*>(orow + 16 * q4 + e) = make_float4(y[e], y[e + 1], y[e + 2], y[e + 3]);
        }
      }
    }
    tc_fence_before();
    __syncthreads();
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

__device__ int g_lion_status;

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
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(lion_chunk64_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBytes);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  TcParams prm;
  prm.out = p.out;
  prm.log_lambda = p.log_lambda;
  prm.H = p.H;
  prm.L = p.L;
  prm.mask_kind = p.mask_kind;
  prm.phi = p.phi;
  prm.status = status;
  lion_chunk64_tc_kernel<<<BH, kThreads, kSmemBytes, s>>>(mq, mk, mv, prm);
  return cudaGetLastError();
}

}  // namespace lion
