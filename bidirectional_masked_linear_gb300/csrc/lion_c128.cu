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
// Design.  One persistent CTA per SM walks heads.  Each head's Q and V tiles
// are double-buffered, so the next head streams in while this one computes.
// The warps are specialised:
//   warp 0      TMA loads, polling three streams (V, K, Q) so that none waits
//               behind another; K is single-buffered and refilled as soon as
//               the score MMAs (LIT: and the state MMAs) have read it;
//   warp 1      tcgen05 MMA issue (one thread);
//   warps 2-17  "prep", two threads per token (32 features each): decay
//               prefix, V -> fp16 in place, phi(k) in place, the
//               decay-weighted phi(k) copy for the state MMA, phi(q) in
//               place, mask factors;
//   warps 18-25 "epi", one thread per TMEM lane (= row of a chunk), one
//               group of four warps per chunk: the decay mask on S (P = S * M,
//               fp16, written back into TMEM as the A operand of P [V | 1]),
//               the state tile, the decay-scaled phi(q) for the state
//               product, and the normalised output, staged per warp in the
//               head's spent Q tile and written by TMA;
//               the TMA warp also pulls each head's K and Q into L2 when it
//               loads its V.
// prep of head h+1 overlaps epi of head h, and the two chunks run as two
// pipelines (one epi warp group each, per-chunk barriers).  MMAs per head,
// n_c = columns of chunk c rounded up to 16 (padding beyond is skipped):
//   S_c   = phi(Q_c) phi(K_c)^T                     M=128 N=n_c K=64
//   X_c^T = [V_c' | 1]^T (w_c' o phi(K_c'))          M=128 N=64  K=n_c'
//   O_c   = P_c [V_c | 1] + (sigma o phi(Q_c)) X_c  M=128 N=80  K=n_c (+ K=64)
// where c' = 1 - c is the chunk whose state chunk c applies (X_0 = G_0 from
// chunk 1's backward weights, X_1 = F_1 from chunk 0's forward weights).
// The state comes out transposed (TMEM lane = output column, lane 64 = the
// normaliser z), so the epi warps write it as a K-major operand tile of 80
// rows with whole-row 16-byte stores, and the state product's column 64 is
// the state part of the row sum.  The ones of [V | 1] come from a 2 KB
// constant tile addressed through the descriptor's leading byte offset.
//
// TMEM (512 columns): X_0^T at [0, 64), X_1^T then O_1 at [80, 160), S_0 at
// [160, 288), S_1 at [288, 416), O_0 at [416, 496) (LION-S; see below); P_c
// overwrites the first 64 columns of S_c.  For LION-S, O_0 has columns of its
// own so that P_0 [V_0 | 1] can start before X_0 has been read into its tile:
// group 0 hands P_0 to the MMA thread two 16-column blocks at a time, and each
// pair's K steps run while the group masks the next pair.  The state product
// follows the last pair, in the same accumulation order as a single hand-off.
// D and LIT hand each chunk over once, with O_0 over X_0 at [0, 80).
//
// Mask factors: within a chunk M_ij = alpha_i rho_j (j <= i) or rho_i alpha_j
// (j > i) with alpha_t = exp(p_t - p_ref), rho_t = 1 / alpha_t and p_ref the
// middle of the chunk's prefix range; chunks whose decay range exceeds
// 2 * 80 nats take exp(-|p_i - p_j|) per element instead.
//
// State decay folded into the row (SiLU + L2 features, LION-S and LION-D):
// y_i is num_i / den_i, so scaling all of row i's O by 1/sigma_i changes
// nothing.  The epi warps multiply row i's mask factors by 1/sigma_i, and the
// state product takes phi(q_i) as prep wrote it, with no pass over the Q
// tile.  Normalised features give |s_ij| <= 1, so P_ij / sigma_i stays below
// 2^15 (fp16 holds it) for sigma_i >= 2^-15; rows with a smaller sigma_i
// keep the in-place decay-scaled phi(q_i) and unscaled factors.  LIT needs
// neither (sigma = 1); elu+1 and identity features, whose scores have no
// fixed bound, keep the scaled phi(q) on every row.
//
// Precision: MMA operands are fp16 (11-bit significand) with fp32
// accumulation; phi(K), phi(Q), the weighted phi(K), V, P and the two
// states (with their z) are each rounded once to fp16, and the decay-scaled
// phi(q) (rows that do not fold) twice.
// Precondition: |phi(q)|, |phi(k)|, |v| and the states below 65504.  A v past
// that range (checked as prep converts it), or a non-finite row sum (an
// infinite feature or score reached the row), sets the CTA's range flag,
// which the kernel reports in `status` as kStatusRange at exit.
//
// Every mbarrier wait is bounded; on timeout the kernel records an error in
// `status`, waits (bounded) for its own copies and MMAs in flight, releases
// its TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "c128_common.cuh"
#include "lion_common.cuh"
#include "lion_internal.h"
#include "tc_ptx.cuh"

namespace lion {
namespace {

using namespace tc;
using namespace c128;

constexpr int kRows = 2 * kC;           // tokens per head at most
constexpr int kStRows = 80;             // state tile rows: 64 columns of X, z, 15 zero rows
constexpr int kStTile = kStRows * 128;  // K-major 16-bit state tile
constexpr int kPrepWarps = 16, kEpiWarps = 8;
constexpr int W_TMA = 0, W_MMA = 1, W_PREP = 2, W_EPI = W_PREP + kPrepWarps;
constexpr int kThreads = (W_EPI + kEpiWarps) * 32;   // 832
constexpr float kFoldMinSigma = 1.f / 32768.f;        // rows that fold 1/sigma into P
constexpr uint32_t kSleepNs = 2000u;
constexpr int KPB = 2;   // P blocks per hand-off (LION-S)
// LION-S hands P_0 over in pairs of blocks, with O_0 in columns of its own
// (its mask takes long enough for the earlier pairs' products to run under
// it); D and LIT, whose cheaper masks gained nothing from it (and whose
// builds then spilled), hand each chunk over once, with O_0 over X_0.
template <int MASK>
__host__ __device__ constexpr bool split_o() { return MASK == MASK_S; }

// shared-memory map (bytes from a 1024-aligned base)
constexpr int OFF_Q = 0;                          // [slot][chunk] phi(Q) tiles; output staging
constexpr int OFF_V = OFF_Q + 4 * kTile;          // [slot][chunk] V tiles
constexpr int OFF_K = OFF_V + 4 * kTile;          // [chunk] phi(K) tiles
constexpr int OFF_KW = OFF_K + 2 * kTile;         // [chunk] decay-weighted phi(K)
constexpr int OFF_ST = OFF_KW + 2 * kTile;        // [chunk] state applied to that chunk
constexpr int OFF_ONES = OFF_ST + 2 * kStTile;    // 16 rows, column 0 = 1
constexpr int OFF_FAC = OFF_ONES + 2048;          // [slot] float alpha[256], rho[256], sig[256], p[256]
constexpr int OFF_INFO = OFF_FAC + 2 * 4 * kRows * 4;  // [slot] float[8] per-head scalars
constexpr int OFF_RED = OFF_INFO + 2 * 8 * 4;     // [parity] float[32] prep scan scratch
constexpr int OFF_BAR = OFF_RED + 2 * 32 * 4;
constexpr int kNumBars = 28;
constexpr int OFF_TSLOT = OFF_BAR + kNumBars * 8;
constexpr int kSmemBytes = OFF_TSLOT + 16 + 1024;  // + alignment slack
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
static_assert(OFF_ONES % 1024 == 0 && OFF_ST % 1024 == 0, "swizzled tiles need 1024-byte alignment");

// per-head scalars (INFO): exact-mask flag of chunk 0/1
enum { I_EX0 = 0, I_EX1 = 1 };

// mbarriers ("+ c": one per chunk, "+ slot": one per Q/V slot)
enum {
  B_V0 = 0,       // + slot: V tiles landed (TMA, tx bytes)
  B_Q0 = 2,       // + slot: Q tiles landed
  B_K = 4,        // K tiles landed
  B_KVR = 5,      // prep: V, phi(K), weighted phi(K) written (16 arrivals)
  B_QR = 6,       // prep: phi(Q) and factors written (16 arrivals)
  B_S0 = 7,       // + c: MMA commit: S_c done
  B_KE = 9,       // MMA commit: K tiles free
  B_U0 = 10,      // + c: MMA commit: the state chunk c applies is done
  B_KWE = 12,     // MMA commit: weighted phi(K) free
  B_PR0 = 13,     // + c: epi group c: P_c, state tile, scaled phi(Q_c) written (4 arrivals)
  B_O0 = 15,      // + c: MMA commit: O_c done
  B_VE0 = 17,     // + slot: MMA commit: V tiles free
  B_QE0 = 19,     // + slot: Q tiles free: every epi warp's output store has read its staging
  B_ED0 = 21,     // + c: epi group c: O_c read (4 arrivals)
  B_DRAIN = 23,   // MMA commit used when unwinding
  B_PP0 = 24,     // + pair: epi group 0: P_0 for keys [32 pair, 32 pair + 32) written (4 arrivals)
};
__device__ __forceinline__ uint32_t bar_count(int b, int nch) {
  if (b == B_KVR || b == B_QR) return kPrepWarps;
  if (b == B_PR0 || b == B_PR0 + 1 || b == B_ED0 || b == B_ED0 + 1) return 4;
  if (b >= B_PP0 && b < B_PP0 + 4) return 4;
  if (b == B_QE0 || b == B_QE0 + 1) return 4 * nch;   // the warps of the groups with a chunk
  return 1;
}

// TMEM columns
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t T_O = 0;       // + 80 c: the transposed state chunk c applies (chunk 1: then O_1)
constexpr uint32_t T_S = 160;     // + 128 c: S_c, P_c in its first 64 columns
constexpr uint32_t T_O0 = 416;    // O_0, apart from its state so that P_0 [V_0 | 1] can start early
template <int MASK>
__device__ __forceinline__ uint32_t o_col(int c) { return c == 0 && split_o<MASK>() ? T_O0 : T_O + 80 * c; }

struct C128Params {
  const float* log_lambda;
  int BH, H, L;
  int out_bf16;   // 1: y stored as bfloat16 (one 64-column store per warp)
  int* status;
  long long wait_cycles;   // bound of every mbarrier wait, in clock cycles
};

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
                            const __grid_constant__ CUtensorMap mapV, const __grid_constant__ CUtensorMap mapO,
                            C128Params prm) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + OFF_TSLOT);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + OFF_TSLOT + 8);
  volatile int* s_range = reinterpret_cast<volatile int*>(smem + OFF_TSLOT + 12);
  auto Qt = [&](int s, int c) { return smem + OFF_Q + (2 * s + c) * kTile; };
  auto Vt = [&](int s, int c) { return smem + OFF_V + (2 * s + c) * kTile; };
  auto Kt = [&](int c) { return smem + OFF_K + c * kTile; };
  auto KWt = [&](int c) { return smem + OFF_KW + c * kTile; };
  auto STt = [&](int c) { return smem + OFF_ST + c * kStTile; };
  auto fac = [&](int s) { return reinterpret_cast<float*>(smem + OFF_FAC) + s * 4 * kRows; };
  auto info = [&](int s) { return reinterpret_cast<float*>(smem + OFF_INFO) + s * 8; };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int L = prm.L;
  const int nch = L > kC ? 2 : 1;
  const bool states = nch == 2;
  // 16-column steps holding tokens, per chunk (the rest is padding)
  const int nk0 = nch == 2 ? 8 : (L + 15) >> 4;
  const int nk1 = nch == 2 ? (L - kC + 15) >> 4 : 0;

  if (tid == 0) {
    prefetch_tmap(&mapQ);
    prefetch_tmap(&mapK);
    prefetch_tmap(&mapV);
    prefetch_tmap(&mapO);
    for (int b = 0; b < kNumBars; ++b) mbar_init(&bars[b], bar_count(b, nch));
    *s_abort = 0;
    *s_range = 0;
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
    return mbar_wait_or_abort(&bars[b], parity, prm.wait_cycles, kSleepNs, s_abort);
  };
  const int nheads = prm.BH > (int)blockIdx.x ? (prm.BH - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  auto head_of = [&](int n) { return (int)blockIdx.x + n * (int)gridDim.x; };

  if (warp == W_TMA) {
    // =========================== TMA producer ===================================
    // Three independent streams; each load goes out as soon as its buffer is
    // free: V(n) after O(n-2), K(n) after S(n-1) (LIT: U(n-1)), Q(n) after
    // head n-2's output left the Q tiles.
    if (lane == 0) {
      int nv = 0, nk = 0, nq = 0;
      long long idle0 = clock64();
      while ((nv < nheads || nk < nheads || nq < nheads) && !*s_abort) {
        bool progress = false;
        if (nv < nheads && (nv < 2 || mbar_try_wait(&bars[B_VE0 + (nv & 1)], ((nv >> 1) - 1) & 1))) {
          const int s = nv & 1, bh = head_of(nv);
          mbar_arrive_expect_tx(&bars[B_V0 + s], (uint32_t)(nch * kTile));
          for (int c = 0; c < nch; ++c) tma_load_3d(Vt(s, c), &mapV, &bars[B_V0 + s], 0, c * kC, bh);
          // K and Q of this head wait for buffers a while longer: start them towards L2
          for (int c = 0; c < nch; ++c) {
            tma_prefetch_3d(&mapK, 0, c * kC, bh);
            tma_prefetch_3d(&mapQ, 0, c * kC, bh);
          }
          ++nv;
          progress = true;
        }
        if (nk < nheads && (nk < 1 || mbar_try_wait(&bars[B_KE], (nk - 1) & 1))) {
          const int bh = head_of(nk);
          mbar_arrive_expect_tx(&bars[B_K], (uint32_t)(nch * kTile));
          for (int c = 0; c < nch; ++c) tma_load_3d(Kt(c), &mapK, &bars[B_K], 0, c * kC, bh);
          ++nk;
          progress = true;
        }
        if (nq < nheads && (nq < 2 || mbar_try_wait(&bars[B_QE0 + (nq & 1)], ((nq >> 1) - 1) & 1))) {
          const int s = nq & 1, bh = head_of(nq);
          mbar_arrive_expect_tx(&bars[B_Q0 + s], (uint32_t)(nch * kTile));
          for (int c = 0; c < nch; ++c) tma_load_3d(Qt(s, c), &mapQ, &bars[B_Q0 + s], 0, c * kC, bh);
          ++nq;
          progress = true;
        }
        if (progress) {
          idle0 = clock64();
        } else {
          __nanosleep(64);
          if (clock64() - idle0 > prm.wait_cycles) *s_abort = 1;
        }
      }
      if (*s_abort) {
        // let the copies already issued land before the CTA lets go of its memory
        const long long lim = prm.wait_cycles / 4;
        for (int s = 0; s < 2; ++s) {
          const int v_is = (nv - s + 1) / 2, q_is = (nq - s + 1) / 2;   // loads issued into slot s
          if (v_is) mbar_wait(&bars[B_V0 + s], (v_is - 1) & 1, lim);
          if (q_is) mbar_wait(&bars[B_Q0 + s], (q_is - 1) & 1, lim);
        }
        if (nk) mbar_wait(&bars[B_K], (nk - 1) & 1, lim);
      }
    }
  } else if (warp == W_MMA) {
    // =========================== MMA issuer =====================================
    if (lane == 0) {
      const uint32_t idUT = idesc_f16(128, 64, true, true);
      const uint32_t idPV = idesc_f16(128, 80, false, true);
      const uint32_t idQX = idesc_f16(128, 80, false, false);
      const uint32_t ones = smem_u32(smem + OFF_ONES);
      // LIT's state MMA reads phi(K) itself: K stays until the states are done
      const bool k_after_u = states && MASK == MASK_LIT;
      bool issued = false, ok = true;
      for (int n = 0; n < nheads && ok; ++n) {
        const int s = n & 1;
        if (!waitb(B_KVR, n & 1) || !waitb(B_QR, n & 1)) break;
        for (int c = 0; c < nch && ok; ++c) {
          if (n >= 1 && !waitb(B_O0 + c, (n - 1) & 1)) ok = false;   // P_c of the previous head consumed
          if (!ok) break;
          tc_fence_after();
          const int nk = c == 0 ? nk0 : nk1;
          const uint32_t idS = idesc_f16(128, 16 * nk, false, false);
          {
            uint64_t da = kmaj(Qt(s, c), 0), db = kmaj(Kt(c), 0);
#pragma unroll
            for (int k = 0; k < 4; ++k, da += kKmajStep, db += kKmajStep)
              mma_bf16(tbase + T_S + 128 * c, da, db, idS, k > 0 ? 1u : 0u);
          }
          mma_commit(&bars[B_S0 + c]);
          issued = true;
        }
        if (!ok) break;
        if (!k_after_u) mma_commit(&bars[B_KE]);
        if (states) {
          // the state group g applies comes from chunk 1 - g
          for (int g = 0; g < 2 && ok; ++g) {
            // X_1 shares its columns with O_1: wait until the previous head's O_1
            // is read.  X_0 has columns of its own, read (into the state tile)
            // before the previous head's O_0 was committed.
            if ((g == 1 || !split_o<MASK>()) && n >= 1 && !waitb(B_ED0 + g, (n - 1) & 1)) ok = false;
            if (!ok) break;
            tc_fence_after();
            const int c = 1 - g, nk = c == 0 ? nk0 : nk1;
            const uint32_t a = smem_u32(Vt(s, c));
            const uint32_t b = smem_u32(MASK == MASK_LIT ? Kt(c) : KWt(c));
            uint64_t da = mnmaj(a, 0, ones - a), db = mnmaj(b, 0, 0);
            for (int k = 0; k < nk; ++k, da += kMnmajOnesStep, db += kMnmajStep)
              mma_bf16(tbase + T_O + 80 * g, da, db, idUT, k > 0 ? 1u : 0u);
            mma_commit(&bars[B_U0 + g]);
          }
          if (!ok) break;
          mma_commit(&bars[B_KWE]);
          if (k_after_u) mma_commit(&bars[B_KE]);
        }
        // O_0 = P_0 [V_0 | 1] goes out a pair of 16-column blocks at a time, as
        // group 0 writes P_0, then its state product once the state tile is
        // written; then O_1, once group 1 has handed over P_1 and its state
        // tile.  (A pair arrival of head n also means that group 0 has read
        // O_0 of head n - 1: its warps arrive in that order.)
        if constexpr (split_o<MASK>()) {
          {
            const int np0 = (nk0 + KPB - 1) / KPB;
            auto o_state = [&](int c) {
              if (states) {
                uint64_t dq = kmaj(Qt(s, c), 0), dx = kmaj(STt(c), 0);
  #pragma unroll
                for (int k = 0; k < 4; ++k, dq += kKmajStep, dx += kKmajStep)
                  mma_bf16(tbase + o_col<MASK>(c), dq, dx, idQX, 1u);
              }
              mma_commit(&bars[B_O0 + c]);
            };
            const uint32_t v0 = smem_u32(Vt(s, 0));
            const uint64_t dv0 = mnmaj(v0, 0, ones - v0);
            for (int kp = 0; kp < np0 && ok; ++kp) {
              if (!waitb(B_PP0 + kp, n & 1)) { ok = false; break; }
              tc_fence_after();
              for (int k = KPB * kp; k < KPB * kp + KPB && k < nk0; ++k)
                mma_tmem_a(tbase + T_O0, tbase + T_S + 8 * k, dv0 + (uint64_t)k * kMnmajOnesStep, idPV,
                           k > 0 ? 1u : 0u);
            }
            if (ok && waitb(B_PR0, n & 1)) {
              tc_fence_after();
              o_state(0);
            } else {
              ok = false;
            }
            if (ok && nch == 2) {
              if (waitb(B_PR0 + 1, n & 1)) {
                tc_fence_after();
                const uint32_t v = smem_u32(Vt(s, 1));
                uint64_t dv = mnmaj(v, 0, ones - v);
                for (int k = 0; k < nk1; ++k, dv += kMnmajOnesStep)
                  mma_tmem_a(tbase + o_col<MASK>(1), tbase + T_S + 128 + 8 * k, dv, idPV, k > 0 ? 1u : 0u);
                o_state(1);
              } else {
                ok = false;
              }
            }
          }
        } else {
          for (int c = 0; c < nch && ok; ++c) {
            if (!states && n >= 1 && !waitb(B_ED0 + c, (n - 1) & 1)) ok = false;
            if (ok && !waitb(B_PR0 + c, n & 1)) ok = false;
            if (!ok) break;
            tc_fence_after();
            const int nk = c == 0 ? nk0 : nk1;
            const uint32_t v = smem_u32(Vt(s, c));
            uint64_t dv = mnmaj(v, 0, ones - v);
            for (int k = 0; k < nk; ++k, dv += kMnmajOnesStep)
              mma_tmem_a(tbase + T_O + 80 * c, tbase + T_S + 128 * c + 8 * k, dv, idPV, k > 0 ? 1u : 0u);
            if (states) {
              uint64_t dq = kmaj(Qt(s, c), 0), dx = kmaj(STt(c), 0);
#pragma unroll
              for (int k = 0; k < 4; ++k, dq += kKmajStep, dx += kKmajStep)
                mma_bf16(tbase + T_O + 80 * c, dq, dx, idQX, 1u);
            }
            mma_commit(&bars[B_O0 + c]);
          }
        }
        if (!ok) break;
        mma_commit(&bars[B_VE0 + s]);
      }
      if (*s_abort && issued) {
        mma_commit(&bars[B_DRAIN]);
        mbar_wait(&bars[B_DRAIN], 0, prm.wait_cycles / 4);
      }
    }
  } else if (warp < W_EPI) {
    // =========================== prep: two threads per token =====================
    const int pw = warp - W_PREP;            // 0..15; chunk c = pw / 8
    const int pt = 32 * pw + lane;
    const int t = pt >> 1, h = pt & 1;       // token within the head, half row
    const int c = t >> 7, r = t & (kC - 1);
    const uint32_t pair = 3u << (lane & 30);
    float* red = reinterpret_cast<float*>(smem + OFF_RED);
    bool good = true;
    float ell_next = 0.f;
    if (nheads > 0) {
      const int bh0 = head_of(0);
      const float lh = MASK == MASK_D ? __ldg(prm.log_lambda + bh0 % prm.H) : 0.f;
      ell_next = ell_of<MASK>(prm, bh0, t, lh);
    }
    for (int n = 0; n < nheads; ++n) {
      const int s = n & 1;
      const float ell = ell_next;
      // ---- chunk-local inclusive prefix of l (each token's value sits in
      //      both lanes of its pair, so steps of two lanes)
      float x = ell;
#pragma unroll
      for (int o = 2; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      float* rd = red + 32 * (n & 1);
      if (lane == 31) rd[pw] = x;
      if (pt == 0) rd[16] = ell;              // l at the first token of chunk 0
      if (pt == 2 * kC) rd[17] = ell;         // l at the first token of chunk 1
      good = bar_and(1, kPrepWarps * 32, good);
      if (!good) break;
      float pre = 0.f;
      for (int w = 8 * c; w < pw; ++w) pre += rd[w];
      const float p = x + pre;                                      // p_t
      float T0 = 0.f, T1 = 0.f;
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        T0 += rd[w];
        T1 += rd[8 + w];
      }
      const float l128 = rd[17];
      const float pfirst = c == 0 ? rd[16] : rd[17], plast = c == 0 ? T0 : T1;
      const float pref = 0.5f * (pfirst + plast);
      const bool exact = (pfirst - plast) > 2.f * kMaxFactorRange;
      const bool live = t < L;
      const int j0 = 4 * h;                   // first 16-byte chunk of this half row

      // ---- V -> fp16 in place
      if (!waitb(B_V0 + s, (n >> 1) & 1)) good = false;
      good = __all_sync(0xffffffffu, good);   // pairs must agree before phi's pair shuffle
      if (good && live) {
        uint8_t* vt = Vt(s, c);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint4* a = reinterpret_cast<uint4*>(vt + sw128_offset(r, j0 + j));
          *a = bf8_to_h8_chk(*a, s_range);
        }
      }
      // ---- K: phi(k) in place; the decay-weighted copy for the state MMA
      if (!waitb(B_K, n & 1)) good = false;
      good = __all_sync(0xffffffffu, good);
      const bool kw = states && MASK != MASK_LIT;
      if (good && live) {
        uint8_t* kt = Kt(c);
        float kv[32];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          unpack8_bf(*reinterpret_cast<const uint4*>(kt + sw128_offset(r, j0 + j)), kv + 8 * j);
        phi_part<PHI, 32, 2>(kv, pair);
#pragma unroll
        for (int j = 0; j < 4; ++j) *reinterpret_cast<uint4*>(kt + sw128_offset(r, j0 + j)) = pack8_h(kv + 8 * j);
        if (kw) {
          if (n >= 1 && !waitb(B_KWE, (n - 1) & 1)) good = false;
          if (good) {
            // weight of this token in its chunk's state
            const float w = c == 0 ? ex2((T0 - p) * kLog2e) : ex2((p - l128) * kLog2e);
            const float2 w2 = make_float2(w, w);
            uint8_t* kwt = KWt(c);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              float y8[8];
#pragma unroll
              for (int e = 0; e < 8; e += 2) {
                const float2 u = mul2(make_float2(kv[8 * j + e], kv[8 * j + e + 1]), w2);
                y8[e] = u.x;
                y8[e + 1] = u.y;
              }
              *reinterpret_cast<uint4*>(kwt + sw128_offset(r, j0 + j)) = pack8_h(y8);
            }
          }
        }
      } else if (good && kw) {
        // padding token: a zero row in the weighted copy (phi(K) keeps the
        // zeros the copy engine filled in)
        if (n >= 1 && !waitb(B_KWE, (n - 1) & 1)) good = false;
        if (good) {
          uint8_t* kwt = KWt(c);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            *reinterpret_cast<uint4*>(kwt + sw128_offset(r, j0 + j)) = make_uint4(0, 0, 0, 0);
        }
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_KVR]);
      // ---- mask factors and phi(q)
      if (good && h == 0) {
        float* f = fac(s);
        const float d = (p - pref) * kLog2e;
        f[t] = ex2(d);
        f[kRows + t] = ex2(-d);
        // decay applied to the state product of this token's query
        f[2 * kRows + t] = !states ? 0.f : c == 0 ? ex2((T0 + l128 - p) * kLog2e) : ex2(p * kLog2e);
        f[3 * kRows + t] = p;
        if (r == 0) info(s)[I_EX0 + c] = exact ? 1.f : 0.f;
      }
      if (!waitb(B_Q0 + s, (n >> 1) & 1)) good = false;
      good = __all_sync(0xffffffffu, good);
      if (good && live) {
        uint8_t* qt = Qt(s, c);
        float qv[32];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          unpack8_bf(*reinterpret_cast<const uint4*>(qt + sw128_offset(r, j0 + j)), qv + 8 * j);
        phi_part<PHI, 32, 2>(qv, pair);
#pragma unroll
        for (int j = 0; j < 4; ++j) *reinterpret_cast<uint4*>(qt + sw128_offset(r, j0 + j)) = pack8_h(qv + 8 * j);
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_QR]);
      // ---- the next head's decays, loaded while this head is in flight
      if (n + 1 < nheads) {
        const int bhn = head_of(n + 1);
        const float lh = MASK == MASK_D ? __ldg(prm.log_lambda + bhn % prm.H) : 0.f;
        ell_next = ell_of<MASK>(prm, bhn, t, lh);
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
    const bool warp_ok = kC * g + 32 * q < L;
    const int nk = g == 0 ? nk0 : nk1;
    const uint32_t lane_off = (uint32_t)(32 * q) << 16;
    bool good = true;
    for (int n = 0; n < nheads && g < nch; ++n) {
      const int bh = head_of(n), s = n & 1;
      const float* f = fac(s);
      const float* alpha = f + kC * g;
      const float* rho = f + kRows + kC * g;
      const float* pp = f + 3 * kRows + kC * g;
      // ---- P = S * M, fp16, into the first 64 columns of S
      if (!waitb(B_S0 + g, n & 1)) good = false;
      good = __all_sync(0xffffffffu, good);   // TMEM loads below are warp-collective
      tc_fence_after();
      // this row's state decay sigma_i folded into its mask factors (header);
      // factors large enough to overflow once scaled do not fold
      const bool exact = info(s)[I_EX0 + g] != 0.f;
      float ai = alpha[i], ri = rho[i], lrow = 0.f;
      const float pi = pp[i];
      const float sg = states && row_ok ? f[2 * kRows + tok] : 1.f;
      const bool fold = states && MASK != MASK_LIT && PHI == PHI_SILU_L2 && sg >= kFoldMinSigma &&
                        (exact || fmaxf(ai, ri) <= 1e33f);
      // group 0 hands P_0 over a pair of blocks at a time (warps without rows,
      // and all warps after an abort, arrive for every pair)
      const int npair = g == 0 && split_o<MASK>() ? (nk + KPB - 1) / KPB : 0;
      int handed = 0;
      if (good && warp_ok) {
        if (fold) {
          const float is = rcp(sg);
          ai *= is;
          ri *= is;
          lrow = -__log2f(sg);
        }
        const uint32_t sa = tbase + lane_off + T_S + 128 * g;
        float sb0[16], sb1[16];
        tmem_ld16(sa, sb0);
        tmem_wait_ld();
        reg_fence16(sb0);
#pragma unroll 1
        for (int jj = 0; jj < nk; jj += 2) {
          uint32_t pk[8];
          const bool has1 = jj + 1 < nk, has2 = jj + 2 < nk;
          if (has1) tmem_ld16(sa + 16 * (jj + 1), sb1);
          mask_block<MASK>(sb0, 16 * jj, i, 32 * q, exact, ai, ri, pi, alpha, rho, pp, lrow);
#pragma unroll
          for (int e = 0; e < 8; ++e) pk[e] = pack_h2(sb0[2 * e], sb0[2 * e + 1]);
          tmem_st8(sa + 8 * jj, pk);
          if (has1) {
            tmem_wait_ld();
            reg_fence16(sb1);
            if (has2) tmem_ld16(sa + 16 * (jj + 2), sb0);
            mask_block<MASK>(sb1, 16 * (jj + 1), i, 32 * q, exact, ai, ri, pi, alpha, rho, pp, lrow);
#pragma unroll
            for (int e = 0; e < 8; ++e) pk[e] = pack_h2(sb1[2 * e], sb1[2 * e + 1]);
            tmem_st8(sa + 8 * (jj + 1), pk);
            if (has2) {
              tmem_wait_ld();
              reg_fence16(sb0);
            }
          }
          if (split_o<MASK>() && g == 0 && ((jj + 2) % KPB == 0 || jj + 2 >= nk)) {
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_PP0 + handed]);
            ++handed;
          }
        }
      }
      for (; handed < npair; ++handed)
        if (lane == 0) mbar_arrive(&bars[B_PP0 + handed]);
      // ---- the state tile this chunk applies (K-major, rows = output
      //      columns, row 64 = z) and the decay-scaled phi(q)
      if (states) {
        if (!waitb(B_U0 + g, n & 1)) good = false;
        good = __all_sync(0xffffffffu, good);
        tc_fence_after();
        if (good && q < 3) {
          // transposed state: TMEM lane 32q + lane = tile row, 64 columns
          const uint32_t ua = tbase + lane_off + T_O + 80 * g;
          float u0[16], u1[16];
          tmem_ld16(ua, u0);
          tmem_ld16(ua + 16, u1);
          tmem_wait_ld();
          reg_fence16(u0);
          reg_fence16(u1);
          uint8_t* row = STt(g) + i * 128;
          const bool st_row = i < kStRows;
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            if (st_row) {
              *reinterpret_cast<uint4*>(row + ((j ^ (i & 7)) << 4)) = pack8_h(u0 + 8 * j);
              *reinterpret_cast<uint4*>(row + (((2 + j) ^ (i & 7)) << 4)) = pack8_h(u1 + 8 * j);
            }
          }
          tmem_ld16(ua + 32, u0);
          tmem_ld16(ua + 48, u1);
          tmem_wait_ld();
          reg_fence16(u0);
          reg_fence16(u1);
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            if (st_row) {
              *reinterpret_cast<uint4*>(row + (((4 + j) ^ (i & 7)) << 4)) = pack8_h(u0 + 8 * j);
              *reinterpret_cast<uint4*>(row + (((6 + j) ^ (i & 7)) << 4)) = pack8_h(u1 + 8 * j);
            }
          }
        }
        // sigma_i phi(q_i), in place: the A operand of the state product, for
        // the rows that do not fold (LIT: sigma = 1, nothing to do)
        const bool scale_row = MASK != MASK_LIT && row_ok && !fold;
        if (good && __any_sync(0xffffffffu, scale_row) && scale_row) {
          const float2 sg2 = make_float2(sg, sg);
          uint8_t* qt = Qt(s, g);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            uint4* a = reinterpret_cast<uint4*>(qt + sw128_offset(i, j));
            float x8[8];
            unpack8_h(*a, x8);
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
              const float2 y = mul2(make_float2(x8[e], x8[e + 1]), sg2);
              x8[e] = y.x;
              x8[e + 1] = y.y;
            }
            *a = pack8_h(x8);
          }
        }
      }
      tmem_wait_st();
      tc_fence_before();
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_PR0 + g]);
      // ---- y = O[0:64] / O[64].  Each warp stages its 32 rows, 32 columns at
      //      a time, with a 128-byte swizzle in its own 4 KB of this chunk's
      //      Q tile (spent once O is done) and writes them with a TMA store,
      //      which drops the rows past L.
      if (!waitb(B_O0 + g, n & 1)) good = false;
      good = __all_sync(0xffffffffu, good);
      tc_fence_after();
      if (good && warp_ok) {
        const uint32_t oa = tbase + lane_off + o_col<MASK>(g);
        uint8_t* stg = Qt(s, g) + 32 * q * 128;
        float ob0[16], ob1[16];
        tmem_ld16(oa + 64, ob1);            // column 64: the row sum
        tmem_ld16(oa, ob0);
        tmem_wait_ld();
        reg_fence16(ob0);
        reg_fence16(ob1);
        const float inv = 1.f / ob1[0];
        // a score past the fp16 range (unbounded features) leaves the row sum
        // non-finite: fp16 operands cannot make an fp32 sum overflow otherwise
        if (row_ok && !(fabsf(ob1[0]) <= 3.0e38f)) *s_range = 1;
        const float2 inv2 = make_float2(inv, inv);
        uint8_t* row = stg + lane * 128;
        if (prm.out_bf16) {
          // the row's 64 columns as bfloat16 fill one 128-byte staging row:
          // one store, the same values as the fp32 path, rounded
#pragma unroll 1
          for (int blk = 0; blk < 4; ++blk) {
            if (blk > 0) {
              tmem_ld16(oa + 16 * blk, ob0);
              tmem_wait_ld();
              reg_fence16(ob0);
            }
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              float y8[8];
#pragma unroll
              for (int t = 0; t < 4; ++t) {
                const float2 y = mul2(make_float2(ob0[8 * e + 2 * t], ob0[8 * e + 2 * t + 1]), inv2);
                y8[2 * t] = y.x;
                y8[2 * t + 1] = y.y;
              }
              *reinterpret_cast<uint4*>(row + (((2 * blk + e) ^ (lane & 7)) << 4)) = pack8_bf(y8);
            }
          }
          fence_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(&mapO, stg, 0, kC * g + 32 * q, bh);
            bulk_commit();
          }
        }
#pragma unroll 1
        for (int half = 0; half < 2 && !prm.out_bf16; ++half) {
          if (half == 1) {
            // the first store has to be done reading the staging
            if (lane == 0) bulk_wait_read();
            __syncwarp();
          }
          tmem_ld16(oa + 32 * half + 16, ob1);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 a = mul2(make_float2(ob0[4 * e], ob0[4 * e + 1]), inv2);
            const float2 b = mul2(make_float2(ob0[4 * e + 2], ob0[4 * e + 3]), inv2);
            *reinterpret_cast<float4*>(row + ((e ^ (lane & 7)) << 4)) = make_float4(a.x, a.y, b.x, b.y);
          }
          tmem_wait_ld();
          reg_fence16(ob1);
          if (half == 0) tmem_ld16(oa + 32, ob0);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 a = mul2(make_float2(ob1[4 * e], ob1[4 * e + 1]), inv2);
            const float2 b = mul2(make_float2(ob1[4 * e + 2], ob1[4 * e + 3]), inv2);
            *reinterpret_cast<float4*>(row + (((4 + e) ^ (lane & 7)) << 4)) = make_float4(a.x, a.y, b.x, b.y);
          }
          fence_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(&mapO, stg, 32 * half, kC * g + 32 * q, bh);
            bulk_commit();
          }
          if (half == 0) {
            tmem_wait_ld();
            reg_fence16(ob0);
          }
        }
      }
      // O_c is read: the next head's state MMA may use these TMEM columns
      // while the second store is still reading the staging
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars[B_ED0 + g]);
        bulk_wait_read();
        mbar_arrive(&bars[B_QE0 + s]);
      }
      // leave together (the group's warps vote)
      if (!bar_and(2 + g, 128, good)) break;
    }
    if (lane == 0) bulk_wait_all();
  }

  __syncthreads();
  if (tid == 0 && *s_abort) atomicExch(prm.status, kStatusTimeout);
  if (tid == 0 && !*s_abort && *s_range) atomicExch(prm.status, kStatusRange);
  if (warp == W_TMA) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
    tmem_relinquish();
  }
}

}  // namespace

bool chunk128_tc_supported(const Problem& p) {
  return p.dtype == DT_BF16 && p.d == kD && p.chunk == kC && p.L <= kRows;
}

cudaError_t launch_chunk128_tc(const Problem& p, int* status, cudaStream_t s) {
  CUtensorMap mq, mk, mv, mo;
  const int BH = p.B * p.H;
  if (!make_map128(&mq, p.q, p.L, BH) || !make_map128(&mk, p.k, p.L, BH) || !make_map128(&mv, p.v, p.L, BH) ||
      !(p.out_bf16 ? make_out_map_bf16(&mo, p.out, p.L, BH, 64) : make_out_map(&mo, p.out, p.L, BH)))
    return cudaErrorInvalidValue;
  C128Params prm;
  prm.log_lambda = p.log_lambda;
  prm.BH = BH;
  prm.H = p.H;
  prm.L = p.L;
  prm.out_bf16 = p.out_bf16;
  prm.status = status;
  prm.wait_cycles = wait_limit_cycles();
  void (*kern)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap, C128Params) = nullptr;
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
  kern<<<grid, kThreads, kSmemBytes, s>>>(mq, mk, mv, mo, prm);
  return cudaGetLastError();
}

}  // namespace lion
