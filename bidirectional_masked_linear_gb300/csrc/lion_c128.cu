// lion_c128.cu -- chunkwise LION forward with 128-token chunks on the
// 5th-generation tensor cores (tcgen05 + TMEM + TMA), bfloat16 inputs, head
// dim 64, sequences of one or two chunks (L <= 256: the ViT patch sequences).
//
// Chunkwise form ("LION Part IV - Results", "LION Chunk"; rebuttal page
// "LION: A bidirectional framework ...", reply "4: Practicality of Recurrent
// Inference").  P is the inclusive prefix of l = log(lambda) and
// M_ij = exp(P_max(i,j) - P_min(i,j)).  With chunk 0 = tokens [0, 128) and
// chunk 1 = [128, L):
//
//   intra   num_i += sum_{j in c(i)} M_ij s_ij [v_j; 1],  s_ij = phi(q_i).phi(k_j)
//   states  F_1 = sum_{j in c0} exp(P_127 - P_j) phi(k_j) [v_j; 1]^T   (forward)
//           G_0 = sum_{j in c1} exp(P_j - P_128) phi(k_j) [v_j; 1]^T   (backward)
//   apply   num_i += exp(P_128 - P_i) phi(q_i) G_0      (i in chunk 0)
//           num_i += exp(P_i - P_127) phi(q_i) F_1      (i in chunk 1)
//   y_i = num_i[0:64] / num_i[64]
//
// With two chunks the forward and backward scans are single steps (F_1 is the
// state of chunk 0, G_0 the state of chunk 1).
//
// Design.  One persistent CTA per SM walks heads; the head's Q and V tiles
// are double-buffered so the next head streams in while this one computes,
// and the warps are specialised:
//   warp 0      TMA loads (Q, V per head slot; K single-buffered, refilled as
//               soon as the score MMAs (LIT: and the state MMAs) have read it);
//   warp 1      tcgen05 MMA issue (one thread);
//   warps 2-9   "prep", one thread per token: decay prefix, phi(k) in place
//               (fp16), the decay-weighted phi(k) copy for the state MMA,
//               V -> fp16 in place, phi(q) in place, mask factors;
//   warps 10-17 "epi", one thread per TMEM lane (= row of a chunk): the decay
//               mask on S (P = S * M, fp16, written back into TMEM as the A
//               operand of P [V | 1]), the state tiles, the decay-scaled
//               phi(q) for the state product, and the normalised output.
// prep of head h+1 overlaps epi of head h.  MMAs per head:
//   S_c  = phi(Q_c) phi(K_c)^T                      M=128 N=128 K=64
//   U_c  = (w_c o phi(K_c))^T [V_c | 1]             M=64  N=80  K=128
//   O_c  = P_c [V_c | 1] + (sigma o phi(Q_c)) X_c   M=128 N=80  K=128 (+ N=64 K=64)
// where X_0 = G_0, X_1 = F_1.  The ones column of [V | 1] comes from a 2 KB
// constant tile addressed through the descriptor's leading byte offset; the
// normaliser contribution of the states, sigma_i phi(q_i).z, is a CUDA-core
// dot product in fp32.
//
// TMEM (512 columns): U_0/O_0 at [0, 80), U_1/O_1 at [80, 160), S_0 at
// [160, 288), S_1 at [288, 416); P_c overwrites the first 64 columns of S_c.
//
// Mask factors: within a chunk M_ij = alpha_i rho_j (j <= i) or rho_i alpha_j
// (j > i) with alpha_t = exp(p_t - p_ref), rho_t = 1 / alpha_t and p_ref the
// middle of the chunk's prefix range; chunks whose decay range exceeds
// 2 * 80 nats take exp(-|p_i - p_j|) per element instead.
//
// Precision: MMA operands are fp16 (11-bit significand) with fp32
// accumulation; phi(K), phi(Q), the weighted phi(K), V, P and the two
// states are each rounded once to fp16, and the decay-scaled phi(q) twice.
// Precondition: |phi(q)|, |phi(k)|, |v| and the states below 65504.
//
// Every mbarrier wait is bounded; on timeout the kernel records an error in
// `status`, waits (bounded) for its own copies and MMAs in flight, releases
// its TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "lion_common.cuh"
#include "lion_internal.h"
#include "tc_ptx.cuh"

namespace lion {
namespace {

using namespace tc;

constexpr int kC = 128;                 // chunk length
constexpr int kD = 64;                  // head dim
constexpr int kRows = 2 * kC;           // tokens per head at most
constexpr int kTile = kC * 128;         // 128 rows x 64 16-bit values, 128-byte swizzle
constexpr int kStTile = kD * 128;       // 64 x 64 16-bit state tile
constexpr int kPrepWarps = 8, kEpiWarps = 8;
constexpr int W_TMA = 0, W_MMA = 1, W_PREP = 2, W_EPI = W_PREP + kPrepWarps;
constexpr int kThreads = (W_EPI + kEpiWarps) * 32;   // 576
constexpr long long kWaitCycles = 2000000000LL;       // ~1 s at 2 GHz
constexpr uint32_t kSleepNs = 2000u;
constexpr float kMaxFactorRange = 80.f;               // exp(80) stays finite in fp32

// shared-memory map (bytes from a 1024-aligned base)
constexpr int OFF_Q = 0;                          // [slot][chunk] phi(Q) tiles
constexpr int OFF_V = OFF_Q + 4 * kTile;          // [slot][chunk] V tiles
constexpr int OFF_K = OFF_V + 4 * kTile;          // [chunk] phi(K) tiles
constexpr int OFF_KW = OFF_K + 2 * kTile;         // [chunk] decay-weighted phi(K)
constexpr int OFF_ST = OFF_KW + 2 * kTile;        // [chunk] state applied to that chunk
constexpr int OFF_ONES = OFF_ST + 2 * kStTile;    // 16 rows, column 0 = 1
constexpr int OFF_FAC = OFF_ONES + 2048;          // [slot] float alpha[256], rho[256], sig[256], p[256]
constexpr int OFF_INFO = OFF_FAC + 2 * 4 * kRows * 4;  // [slot] float[8] per-head scalars
constexpr int OFF_Z = OFF_INFO + 2 * 8 * 4;       // [chunk] float[64] z of the state applied
constexpr int OFF_RED = OFF_Z + 2 * kD * 4;       // [parity] float[16] prep scan scratch
constexpr int OFF_BAR = OFF_RED + 2 * 16 * 4;
constexpr int kNumBars = 16;
constexpr int OFF_TSLOT = OFF_BAR + kNumBars * 8;
constexpr int kSmemBytes = OFF_TSLOT + 16 + 1024;  // + alignment slack
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
static_assert(OFF_ONES % 1024 == 0 && OFF_ST % 1024 == 0, "swizzled tiles need 1024-byte alignment");

// per-head scalars (INFO): 0 T_0 (chunk-0 total), 1 l_128, 2/3 p_ref of
// chunk 0/1, 4/5 exact-mask flag of chunk 0/1
enum { I_T0 = 0, I_L128 = 1, I_REF0 = 2, I_REF1 = 3, I_EX0 = 4, I_EX1 = 5 };

// mbarriers
enum {
  B_QV0 = 0,      // + slot: Q, V tiles landed (TMA, tx bytes)
  B_K = 2,        // K tiles landed
  B_KVR = 3,      // prep: phi(K), weighted phi(K), V written (8 arrivals)
  B_QR = 4,       // prep: phi(Q) and factors written (8 arrivals)
  B_S = 5,        // MMA commit: S done
  B_KE = 6,       // MMA commit: K tiles free
  B_U = 7,        // MMA commit: states done
  B_KWE = 8,      // MMA commit: weighted phi(K) free
  B_PR = 9,       // epi: P, state tiles, scaled phi(Q) written (8 arrivals)
  B_O = 10,       // MMA commit: O done
  B_QVE0 = 11,    // + slot: MMA commit: Q, V tiles free
  B_ED = 13,      // epi: O read (8 arrivals)
  B_DRAIN = 14,   // MMA commit used when unwinding
};
__host__ __device__ constexpr uint32_t bar_count(int b) {
  return (b == B_KVR || b == B_QR) ? (uint32_t)kPrepWarps : (b == B_PR || b == B_ED) ? (uint32_t)kEpiWarps : 1u;
}

// TMEM columns
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t T_O = 0;       // + 80 c: U_c then O_c
constexpr uint32_t T_S = 160;     // + 128 c: S_c, P_c in its first 64 columns

struct C128Params {
  float* out;
  const float* log_lambda;
  int BH, H, L;
  int* status;
};

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ uint32_t pack_h2(float a, float b) { return h2u(__floats2half2_rn(a, b)); }
__device__ __forceinline__ uint4 pack8_h(const float* x) {
  return make_uint4(pack_h2(x[0], x[1]), pack_h2(x[2], x[3]), pack_h2(x[4], x[5]), pack_h2(x[6], x[7]));
}
__device__ __forceinline__ void unpack8_bf(uint4 v, float* x) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    x[2 * e] = __uint_as_float(w[e] << 16);
    x[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
  }
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
// bf16 -> fp16 for 8 values (exact for |v| in the fp16 normal range)
__device__ __forceinline__ uint4 bf8_to_h8(uint4 v) {
  float x[8];
  unpack8_bf(v, x);
  return pack8_h(x);
}

// phi over the 64 features of one row held by this thread.
template <int PHI>
__device__ __forceinline__ void phi_row(float* x) {
  if (PHI == PHI_ELU1) {
#pragma unroll
    for (int e = 0; e < kD; ++e) x[e] = x[e] > 0.f ? x[e] + 1.f : __expf(x[e]);
  } else if (PHI == PHI_SILU_L2) {
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < kD; ++e) {
      x[e] = __fdividef(x[e], 1.f + __expf(-x[e]));
      ss = fmaf(x[e], x[e], ss);
    }
    const float inv = rsqrtf(fmaxf(ss, 1e-24f));
#pragma unroll
    for (int e = 0; e < kD; ++e) x[e] *= inv;
  }
}

__device__ __forceinline__ uint64_t kmaj(const uint8_t* tile, int k) {
  return desc_sw128(smem_u32(tile) + 32 * k, 16, 1024);
}
// MN-major operand, K step k (16 rows of the tile); the second 64-wide atom
// along MN sits `lbo` bytes after the first.
__device__ __forceinline__ uint64_t mnmaj(uint32_t addr, int k, uint32_t lbo) {
  return desc_sw128(addr + 2048 * k, lbo, 1024);
}

template <int MASK>
__device__ __forceinline__ float ell_of(const C128Params& p, int bh, int t, float lh) {
  if (t >= p.L) return 0.f;
  if (MASK == MASK_S) return __ldg(p.log_lambda + (size_t)bh * p.L + t);
  if (MASK == MASK_D) return lh;
  return 0.f;
}

template <int MASK, int PHI>
__global__ void __launch_bounds__(kThreads, 1)
    lion_chunk128_tc_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
                            const __grid_constant__ CUtensorMap mapV, C128Params prm) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + OFF_TSLOT);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + OFF_TSLOT + 8);
  auto Qt = [&](int s, int c) { return smem + OFF_Q + (2 * s + c) * kTile; };
  auto Vt = [&](int s, int c) { return smem + OFF_V + (2 * s + c) * kTile; };
  auto Kt = [&](int c) { return smem + OFF_K + c * kTile; };
  auto KWt = [&](int c) { return smem + OFF_KW + c * kTile; };
  auto STt = [&](int c) { return smem + OFF_ST + c * kStTile; };
  auto fac = [&](int s) { return reinterpret_cast<float*>(smem + OFF_FAC) + s * 4 * kRows; };
  auto info = [&](int s) { return reinterpret_cast<float*>(smem + OFF_INFO) + s * 8; };
  float* sZ = reinterpret_cast<float*>(smem + OFF_Z);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int L = prm.L;
  const int nch = L > kC ? 2 : 1;
  const bool states = nch == 2;

  if (tid == 0) {
    prefetch_tmap(&mapQ);
    prefetch_tmap(&mapK);
    prefetch_tmap(&mapV);
    for (int b = 0; b < kNumBars; ++b) mbar_init(&bars[b], bar_count(b));
    *s_abort = 0;
    fence_mbar_init();
  }
  // the ones tile: 16 rows of the normaliser atom, 1 at column 0
  for (int x = tid; x < 16 * 8; x += kThreads) {
    const int r = x >> 3, c8 = x & 7;
    *reinterpret_cast<uint4*>(smem + OFF_ONES + sw128_offset(r, c8)) =
        make_uint4(c8 == 0 ? pack_h2(1.f, 0.f) : 0u, 0u, 0u, 0u);
  }
  if (warp == W_TMA) tmem_alloc(tslot, kTmemCols);
  fence_async_smem();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;

  // bounded wait; after any timeout every later wait returns false at once
  auto waitb = [&](int b, uint32_t parity) -> bool {
    if (*s_abort) return false;
    if (mbar_try_wait(&bars[b], parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait_sleep(&bars[b], parity, kSleepNs)) {
      if (*s_abort) return false;
      if (clock64() - t0 > kWaitCycles) {
        *s_abort = 1;
        return false;
      }
    }
    return true;
  };
  const int nheads = prm.BH > (int)blockIdx.x ? (prm.BH - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  auto head_of = [&](int n) { return (int)blockIdx.x + n * (int)gridDim.x; };

  if (warp == W_TMA) {
    // =========================== TMA producer ===================================
    if (lane == 0) {
      int issued_qv[2] = {0, 0}, issued_k = 0;
      for (int n = 0; n < nheads; ++n) {
        const int bh = head_of(n), s = n & 1;
        if (n >= 2 && !waitb(B_QVE0 + s, ((n >> 1) - 1) & 1)) break;
        mbar_arrive_expect_tx(&bars[B_QV0 + s], (uint32_t)(2 * nch * kTile));
        for (int c = 0; c < nch; ++c) {
          tma_load_3d(Qt(s, c), &mapQ, &bars[B_QV0 + s], 0, c * kC, bh);
          tma_load_3d(Vt(s, c), &mapV, &bars[B_QV0 + s], 0, c * kC, bh);
        }
        ++issued_qv[s];
        if (n >= 1 && !waitb(B_KE, (n - 1) & 1)) break;
        mbar_arrive_expect_tx(&bars[B_K], (uint32_t)(nch * kTile));
        for (int c = 0; c < nch; ++c) tma_load_3d(Kt(c), &mapK, &bars[B_K], 0, c * kC, bh);
        ++issued_k;
      }
      if (*s_abort) {
        // let the copies already issued land before the CTA lets go of its memory
        const long long lim = kWaitCycles / 4;
        for (int s = 0; s < 2; ++s)
          if (issued_qv[s]) mbar_wait(&bars[B_QV0 + s], (issued_qv[s] - 1) & 1, lim);
        if (issued_k) mbar_wait(&bars[B_K], (issued_k - 1) & 1, lim);
      }
    }
  } else if (warp == W_MMA) {
    // =========================== MMA issuer =====================================
    if (lane == 0) {
      const uint32_t idS = idesc_f16(128, 128, false, false);
      const uint32_t idU = idesc_f16(64, 80, true, true);
      const uint32_t idPV = idesc_f16(128, 80, false, true);
      const uint32_t idQX = idesc_f16(128, 64, false, true);
      const uint32_t ones = smem_u32(smem + OFF_ONES);
      bool issued = false;
      for (int n = 0; n < nheads; ++n) {
        const int s = n & 1;
        if (!waitb(B_KVR, n & 1) || !waitb(B_QR, n & 1)) break;
        if (n >= 1 && !waitb(B_O, (n - 1) & 1)) break;   // P of the previous head consumed
        tc_fence_after();
        for (int c = 0; c < nch; ++c)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_bf16(tbase + T_S + 128 * c, kmaj(Qt(s, c), k), kmaj(Kt(c), k), idS, k > 0 ? 1u : 0u);
        mma_commit(&bars[B_S]);
        // LIT's state MMA reads phi(K) itself: K stays until the states are done
        const bool k_after_u = states && MASK == MASK_LIT;
        if (!k_after_u) mma_commit(&bars[B_KE]);
        issued = true;
        if (n >= 1 && !waitb(B_ED, (n - 1) & 1)) break;   // O of the previous head read
        tc_fence_after();
        if (states) {
          for (int c = 0; c < 2; ++c) {
            const uint32_t a = smem_u32(MASK == MASK_LIT ? Kt(c) : KWt(c));
            const uint32_t v = smem_u32(Vt(s, c));
#pragma unroll
            for (int k = 0; k < 8; ++k)
              mma_bf16(tbase + T_O + 80 * c, mnmaj(a, k, 0), mnmaj(v, k, ones - (v + 2048 * k)), idU,
                       k > 0 ? 1u : 0u);
          }
          mma_commit(&bars[B_U]);
          mma_commit(&bars[B_KWE]);
          if (k_after_u) mma_commit(&bars[B_KE]);
        }
        if (!waitb(B_PR, n & 1)) break;
        tc_fence_after();
        for (int c = 0; c < nch; ++c) {
          const uint32_t v = smem_u32(Vt(s, c));
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma_tmem_a(tbase + T_O + 80 * c, tbase + T_S + 128 * c + 8 * k, mnmaj(v, k, ones - (v + 2048 * k)),
                       idPV, k > 0 ? 1u : 0u);
          if (states) {
            const uint32_t x = smem_u32(STt(c));
#pragma unroll
            for (int k = 0; k < 4; ++k) mma_bf16(tbase + T_O + 80 * c, kmaj(Qt(s, c), k), mnmaj(x, k, 0), idQX, 1u);
          }
        }
        mma_commit(&bars[B_O]);
        mma_commit(&bars[B_QVE0 + s]);
      }
      if (*s_abort && issued) {
        mma_commit(&bars[B_DRAIN]);
        mbar_wait(&bars[B_DRAIN], 0, kWaitCycles / 4);
      }
    }
  } else if (warp < W_EPI) {
    // =========================== prep: one thread per token ======================
    const int pw = warp - W_PREP;
    const int t = 32 * pw + lane;           // token within the head
    const int c = t >> 7, r = t & (kC - 1);
    float* red = reinterpret_cast<float*>(smem + OFF_RED);
    bool good = true;
    float ell_next = 0.f, lh_next = 0.f;
    if (nheads > 0) {
      const int bh0 = head_of(0);
      lh_next = MASK == MASK_D ? __ldg(prm.log_lambda + bh0 % prm.H) : 0.f;
      ell_next = ell_of<MASK>(prm, bh0, t, lh_next);
    }
    for (int n = 0; n < nheads; ++n) {
      const int bh = head_of(n), s = n & 1;
      const float ell = ell_next;
      // ---- chunk-local inclusive prefix of l over this thread's chunk
      float x = ell;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      float* rd = red + 16 * (n & 1);
      if (lane == 31) rd[pw] = x;
      if (t == 0) rd[8] = ell;          // l at the first token of chunk 0
      if (t == kC) rd[9] = ell;         // l at the first token of chunk 1
      good = bar_and(1, kPrepWarps * 32, good);
      if (!good) break;
      float pre = 0.f;
      for (int w = 4 * c; w < pw; ++w) pre += rd[w];
      const float p = x + pre;                                      // p_t
      const float T0 = rd[0] + rd[1] + rd[2] + rd[3];               // chunk-0 total
      const float T1 = rd[4] + rd[5] + rd[6] + rd[7];
      const float l128 = rd[9];
      const float pfirst = c == 0 ? rd[8] : rd[9], plast = c == 0 ? T0 : T1;
      const float pref = 0.5f * (pfirst + plast);
      const bool exact = (pfirst - plast) > 2.f * kMaxFactorRange;
      // weight of this token in its chunk's state, and the decay applied to
      // the state product of this token's query
      const float w = c == 0 ? __expf(T0 - p) : __expf(p - l128);
      const float sig = !states ? 0.f : c == 0 ? __expf(T0 + l128 - p) : __expf(p);

      // ---- K: phi(k) in place; the decay-weighted copy for the state MMA
      if (!waitb(B_K, n & 1)) good = false;
      if (good && t < L) {
        uint8_t* kt = Kt(c);
        float kv[kD];
#pragma unroll
        for (int j = 0; j < 8; ++j) unpack8_bf(*reinterpret_cast<const uint4*>(kt + sw128_offset(r, j)), kv + 8 * j);
        phi_row<PHI>(kv);
#pragma unroll
        for (int j = 0; j < 8; ++j) *reinterpret_cast<uint4*>(kt + sw128_offset(r, j)) = pack8_h(kv + 8 * j);
        if (states && MASK != MASK_LIT) {
          if (n >= 1 && !waitb(B_KWE, (n - 1) & 1)) good = false;
          if (good) {
            uint8_t* kw = KWt(c);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              float y8[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) y8[e] = w * kv[8 * j + e];
              *reinterpret_cast<uint4*>(kw + sw128_offset(r, j)) = pack8_h(y8);
            }
          }
        }
      } else if (good && states && MASK != MASK_LIT) {
        // padding token: a zero row in the weighted copy (phi(K) keeps the
        // zeros the copy engine filled in)
        if (n >= 1 && !waitb(B_KWE, (n - 1) & 1)) good = false;
        if (good) {
          uint8_t* kw = KWt(c);
#pragma unroll
          for (int j = 0; j < 8; ++j) *reinterpret_cast<uint4*>(kw + sw128_offset(r, j)) = make_uint4(0, 0, 0, 0);
        }
      }
      // ---- V -> fp16 in place
      if (!waitb(B_QV0 + s, (n >> 1) & 1)) good = false;
      if (good && t < L) {
        uint8_t* vt = Vt(s, c);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          uint4* a = reinterpret_cast<uint4*>(vt + sw128_offset(r, j));
          *a = bf8_to_h8(*a);
        }
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_KVR]);
      // ---- mask factors and phi(q)
      if (good) {
        float* f = fac(s);
        const float d = p - pref;
        f[t] = __expf(d);
        f[kRows + t] = __expf(-d);
        f[2 * kRows + t] = sig;
        f[3 * kRows + t] = p;
        if (t == 0) {
          float* in = info(s);
          in[I_T0] = T0;
          in[I_L128] = l128;
          in[I_REF0] = pref;
          in[I_EX0] = exact ? 1.f : 0.f;
        }
        if (t == kC) {
          float* in = info(s);
          in[I_REF1] = pref;
          in[I_EX1] = exact ? 1.f : 0.f;
        }
      }
      if (good && t < L) {
        uint8_t* qt = Qt(s, c);
        float qv[kD];
#pragma unroll
        for (int j = 0; j < 8; ++j) unpack8_bf(*reinterpret_cast<const uint4*>(qt + sw128_offset(r, j)), qv + 8 * j);
        phi_row<PHI>(qv);
#pragma unroll
        for (int j = 0; j < 8; ++j) *reinterpret_cast<uint4*>(qt + sw128_offset(r, j)) = pack8_h(qv + 8 * j);
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_QR]);
      // ---- the next head's decays, loaded while this head is in flight
      if (n + 1 < nheads) {
        const int bhn = head_of(n + 1);
        lh_next = MASK == MASK_D ? __ldg(prm.log_lambda + bhn % prm.H) : 0.f;
        ell_next = ell_of<MASK>(prm, bhn, t, lh_next);
      }
    }
  } else {
    // =========================== epi: one thread per row of a chunk ===============
    const int ew = warp - W_EPI;
    const int g = ew >> 2;                 // chunk of this warp's rows
    const int q = warp & 3;                // TMEM lane quarter
    const int i = 32 * q + lane;           // row within chunk g
    const int tok = kC * g + i;
    const bool row_ok = tok < L;
    const bool warp_ok = kC * g + 32 * q < L && g < nch;
    const uint32_t lane_off = (uint32_t)(32 * q) << 16;
    bool good = true;
    for (int n = 0; n < nheads; ++n) {
      const int bh = head_of(n), s = n & 1;
      const float* f = fac(s);
      const float* alpha = f + kC * g;
      const float* rho = f + kRows + kC * g;
      const float* pp = f + 3 * kRows + kC * g;
      float dstate = 0.f;
      // ---- P = S * M, fp16, into the first 64 columns of S
      if (!waitb(B_S, n & 1)) good = false;
      good = __all_sync(0xffffffffu, good);   // TMEM loads below are warp-collective
      tc_fence_after();
      if (good && warp_ok) {
        const bool exact = info(s)[I_EX0 + g] != 0.f;
        const float ai = alpha[i], ri = rho[i], pi = pp[i];
        const uint32_t sa = tbase + lane_off + T_S + 128 * g;
#pragma unroll 1
        for (int jj = 0; jj < 8; ++jj) {
          float sv[16];
          tmem_ld16(sa + 16 * jj, sv);
          tmem_wait_ld();
          const int j0 = 16 * jj;
          if (MASK != MASK_LIT) {
            if (exact) {
#pragma unroll
              for (int e = 0; e < 16; ++e) sv[e] *= __expf(-fabsf(pi - pp[j0 + e]));
            } else if (j0 + 15 < 32 * q) {         // whole block left of every row of the warp
#pragma unroll
              for (int e = 0; e < 16; ++e) sv[e] *= ai * rho[j0 + e];
            } else if (j0 > 32 * q + 31) {         // whole block right of every row
#pragma unroll
              for (int e = 0; e < 16; ++e) sv[e] *= ri * alpha[j0 + e];
            } else {
#pragma unroll
              for (int e = 0; e < 16; ++e) sv[e] *= (j0 + e <= i) ? ai * rho[j0 + e] : ri * alpha[j0 + e];
            }
          }
          uint32_t pk[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) pk[e] = pack_h2(sv[2 * e], sv[2 * e + 1]);
          tmem_st8(sa + 8 * jj, pk);
        }
      }
      // ---- state tiles (group g writes the state applied to chunk g) and the
      //      decay-scaled phi(q) for the state product
      if (states) {
        if (!waitb(B_U, n & 1)) good = false;
        good = __all_sync(0xffffffffu, good);
        tc_fence_after();
        if (good) {
          // U of the other chunk: M=64 rows 16q..16q+15 in lanes 32q..32q+15
          const uint32_t ua = tbase + lane_off + T_O + 80 * (1 - g);
          uint8_t* st = STt(g);
          const int m0 = 16 * q + (lane >> 2), m1 = m0 + 8;
          const int cc = 2 * (lane & 3);
#pragma unroll
          for (int jb = 0; jb < 4; ++jb) {
            float u[8];
            tmem_ld_16x256b_x2(ua + 16 * jb, u);
            tmem_wait_ld();
            // columns 16jb + cc, +1 (u[0..1] row m0, u[2..3] row m1) and 16jb + 8 + cc, +1 (u[4..7])
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const int col = 16 * jb + 8 * hh + cc;
              *reinterpret_cast<uint32_t*>(st + sw128_offset(m0, col >> 3) + 2 * (col & 7)) =
                  pack_h2(u[4 * hh], u[4 * hh + 1]);
              *reinterpret_cast<uint32_t*>(st + sw128_offset(m1, col >> 3) + 2 * (col & 7)) =
                  pack_h2(u[4 * hh + 2], u[4 * hh + 3]);
            }
          }
          float zz[4];
          tmem_ld_16x256b(ua + 64, zz);
          tmem_wait_ld();
          if ((lane & 3) == 0) {
            sZ[kD * g + m0] = zz[0];
            sZ[kD * g + m1] = zz[2];
          }
        }
        fence_async_smem();
        good = bar_and(2 + g, 128, good);
        if (good && row_ok) {
          const float sg = f[2 * kRows + tok];
          uint8_t* qt = Qt(s, g);
          const float* z = sZ + kD * g;
          float acc = 0.f;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            uint4* a = reinterpret_cast<uint4*>(qt + sw128_offset(i, j));
            float x8[8];
            unpack8_h(*a, x8);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              acc = fmaf(x8[e], z[8 * j + e], acc);
              x8[e] *= sg;
            }
            *a = pack8_h(x8);
          }
          dstate = sg * acc;
        }
      }
      tmem_wait_st();
      tc_fence_before();
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_PR]);
      // ---- y = O[0:64] / (O[64] + state normaliser)
      if (!waitb(B_O, n & 1)) good = false;
      good = __all_sync(0xffffffffu, good);
      tc_fence_after();
      if (good && warp_ok) {
        const uint32_t oa = tbase + lane_off + T_O + 80 * g;
        const float inv = 1.f / (tmem_ld1(oa + 64) + dstate);
        float4* dst = reinterpret_cast<float4*>(prm.out + ((size_t)bh * L + tok) * kD);
#pragma unroll 1
        for (int jb = 0; jb < 4; ++jb) {
          float o[16];
          tmem_ld16(oa + 16 * jb, o);
          tmem_wait_ld();
          if (row_ok) {
#pragma unroll
            for (int e = 0; e < 4; ++e)
              __stcs(dst + 4 * jb + e,
                     make_float4(o[4 * e] * inv, o[4 * e + 1] * inv, o[4 * e + 2] * inv, o[4 * e + 3] * inv));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_ED]);
      // leave together: the group's named barrier needs all four warps
      if (!bar_and(2 + g, 128, good)) break;
    }
  }

  __syncthreads();
  if (tid == 0 && *s_abort) atomicExch(prm.status, 1);
  if (warp == W_TMA) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
    tmem_relinquish();
  }
}

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

// [BH][L][64] bf16 viewed as a 3-D tensor; box = 64 columns x 128 rows x 1
// (rows past L read as zeros).
bool make_map128(CUtensorMap* m, const void* base, int L, int BH) {
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

int sm_count() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}

}  // namespace

bool chunk128_tc_supported(const Problem& p) {
  return p.dtype == DT_BF16 && p.d == kD && p.chunk == kC && p.L <= kRows;
}

cudaError_t launch_chunk128_tc(const Problem& p, int* status, cudaStream_t s) {
  CUtensorMap mq, mk, mv;
  const int BH = p.B * p.H;
  if (!make_map128(&mq, p.q, p.L, BH) || !make_map128(&mk, p.k, p.L, BH) || !make_map128(&mv, p.v, p.L, BH))
    return cudaErrorInvalidValue;
  C128Params prm;
  prm.out = p.out;
  prm.log_lambda = p.log_lambda;
  prm.BH = BH;
  prm.H = p.H;
  prm.L = p.L;
  prm.status = status;
  void (*kern)(const CUtensorMap, const CUtensorMap, const CUtensorMap, C128Params) = nullptr;
#define LION_C128_CASE(M, F) \
  if (p.mask_kind == M && p.phi == F) kern = lion_chunk128_tc_kernel<M, F>;
  LION_C128_CASE(MASK_LIT, PHI_ELU1)
  LION_C128_CASE(MASK_LIT, PHI_SILU_L2)
  LION_C128_CASE(MASK_LIT, PHI_IDENTITY)
  LION_C128_CASE(MASK_D, PHI_ELU1)
  LION_C128_CASE(MASK_D, PHI_SILU_L2)
  LION_C128_CASE(MASK_D, PHI_IDENTITY)
  LION_C128_CASE(MASK_S, PHI_ELU1)
  LION_C128_CASE(MASK_S, PHI_SILU_L2)
  LION_C128_CASE(MASK_S, PHI_IDENTITY)
#undef LION_C128_CASE
  if (!kern) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const int grid = BH < sm_count() ? BH : sm_count();
  kern<<<grid, kThreads, kSmemBytes, s>>>(mq, mk, mv, prm);
  return cudaGetLastError();
}

}  // namespace lion
