// lion_c128L.cu -- main pass of the chunkwise LION forward with 128-token
// chunks for sequences longer than 256 tokens, on the 5th-generation tensor
// cores (tcgen05 + TMEM + TMA), bfloat16 inputs, head dim 64.
//
// Chunkwise form ("LION Part IV - Results", "LION Chunk"; rebuttal page
// "LION: A bidirectional framework ...", reply "4: Practicality of Recurrent
// Inference").  With P the inclusive prefix of l = log(lambda), chunk c =
// tokens [s_c, e_c] and p the chunk-local prefix, row i of chunk c is
//
//   y_i = (O_i + a_i T_i + b_i R_i)[0:64] / (O_i + a_i T_i + b_i R_i)[64]
//   O_i = sum_{j in c} M_ij s_ij [v_j; 1]               (intra-chunk)
//   T_i = phi(q_i) F_c,  a_i = exp(P_i - P_{e_{c-1}}) = exp(p_i)
//   R_i = phi(q_i) G_c,  b_i = exp(P_{s_{c+1}} - P_i)
//
// F_c is the forward state entering chunk c from the left (anchored at
// e_{c-1}) and G_c the backward state entering it from the right (anchored
// at s_{c+1}), both [phi(k) (x) [v; 1]] sums weighted by the decay.
//
// The sequence is cut into segments of 256-token blocks.  A pre-pass (run
// right to left over each segment, lion_c128P.cu) provides, per chunk, the
// backward state entering it from the right within its segment, and per
// segment its forward and backward summaries.  This pass chains the
// summaries of the other segments of its head into the states entering its
// segment from both sides (with several segments a head each CTA has one
// segment, so the chaining runs once, before the first chunk; with one
// segment a head both are zero), then walks the segment left to right, one
// chunk at a time:
//   F_c     carried in TMEM (fp32, transposed: lane = output column, lane 64
//           = z), starting from the segment's entering state, and advanced
//           after every chunk: F_{c+1} = exp(T_c) F_c + U_c with
//           U_c^T = [V_c | 1]^T (w_c o phi(K_c)), w_j = exp(p_e - p_j);
//   G_c     the pre-pass state at the chunk's right edge plus the segment's
//           entering backward state decayed to it, built by prep in place in
//           the chunk's copy of the pre-pass tile (which has the operand
//           tile's layout);
// both as K-major fp16 operand tiles of 80 rows (row 64 = z).  MMAs per chunk
// (n = columns with tokens, rounded up to 16):
//   S   = phi(Q) phi(K)^T            M=128 N=n  K=64
//   U^T = [V | 1]^T (w o phi(K))     M=128 N=64 K=n
//   T   = phi(Q) X_F,  R = phi(Q) X_G  M=128 N=80 K=64
//   O   = P [V | 1]                  M=128 N=80 K=n  (A operand P in TMEM)
// with the decay mask applied to S on the CUDA cores as in lion_c128.cu.
//
// Warps: 0 TMA (Q, K, V and the pre-pass state of a chunk into one of two
// slots), 1 MMA issue, 2-17 "prep" (the segment's entering states; then four
// threads per token: prefix, V -> fp16, phi(k) and its weighted copy,
// phi(q), factors, the X_G tile), 18-25 "epi" (two warps per TMEM lane
// quarter, each one column half: mask, carried state and the next chunk's
// X_F while the chunk's output product runs, then the output through TMA).
// Prep of chunk c+1 overlaps the epilogue of chunk c.
//
// TMEM (512 columns): S [0,128) (P in columns 0-31 and 64-95), O [128,208),
// T [208,288), R [288,368), F^T [368,432), U^T [432,496).
//
// Precision as lion_c128.cu: fp16 operands, fp32 accumulation, the states
// rounded once to fp16 per use.  Every mbarrier wait is bounded; on timeout
// the kernel records an error in `status`, waits (bounded) for its own copies
// and MMAs in flight, releases its TMEM and returns.
#include "c128_common.cuh"
#include "lion_common.cuh"
#include "lion_internal.h"
#include "tc_ptx.cuh"

namespace lion {
namespace {

using namespace tc;
using namespace c128;

constexpr int kStRows = 80;                 // state tile rows: 64 columns, z, 15 zero rows
constexpr int kStTile = kStRows * 128;
constexpr int kPrepWarps = 16, kEpiWarps = 8;
constexpr int W_TMA = 0, W_MMA = 1, W_PREP = 2, W_EPI = W_PREP + kPrepWarps;
constexpr int kThreads = (W_EPI + kEpiWarps) * 32;   // 832
constexpr uint32_t kSleepNs = 2000u;
constexpr int kGsegBytes = 64 * kLongStateCols * 4;  // one fp32 [64][80] state

// shared-memory map (bytes from a 1024-aligned base)
constexpr int kSlotG = kStTile;                       // pre-pass state of a chunk, then its X_G tile
constexpr int kSlotBytes = 3 * kTile + kSlotG;        // Q, K, V, pre-pass state
constexpr int OFF_SLOT = 0;                           // [2] slots
constexpr int OFF_KW = OFF_SLOT + 2 * kSlotBytes;     // weighted phi(K)
constexpr int OFF_XF = OFF_KW + kTile;                // X_F operand tile
constexpr int OFF_ONES = OFF_XF + kStTile;            // 16 rows, column 0 = 1
constexpr int OFF_STG = OFF_ONES + 2048;              // [8 epi warps] 4 KB output staging
constexpr int OFF_GSEG = OFF_STG + kEpiWarps * 4096;  // the segment's entering backward state (fp32 [64][80])
constexpr int OFF_FAC = OFF_GSEG + kGsegBytes;        // [slot] alpha, rho, a, b, p [128] each
constexpr int OFF_INFO = OFF_FAC + 2 * 5 * kC * 4;    // [slot] float[8] per-chunk scalars
constexpr int OFF_BAR = OFF_INFO + 2 * 8 * 4;
constexpr int kNumBars = 24;
constexpr int OFF_TSLOT = OFF_BAR + kNumBars * 8;
constexpr int kSmemBytes = OFF_TSLOT + 16 + 1024;     // + alignment slack
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
static_assert(kSlotBytes % 1024 == 0 && OFF_KW % 1024 == 0 && OFF_XF % 1024 == 0 && OFF_ONES % 1024 == 0 &&
                  OFF_STG % 1024 == 0 &&
                  (3 * kTile) % 1024 == 0,
              "swizzled tiles need 1024-byte alignment");
static_assert(kGstBytes <= kSlotG && kGstBytes % 16 == 0 && kGsegBytes % 16 == 0, "bulk copies");

// per-chunk scalars (INFO)
enum { I_EXACT = 0, I_T = 1, I_LNEXT = 2 };

// mbarriers
enum {
  B_LD0 = 0,     // + slot: Q, K, V, pre-pass state landed (TMA, tx bytes)
  B_KVR = 3,     // prep: V, phi(K), weighted phi(K) written (16 arrivals)
  B_QR = 4,      // prep: phi(Q), factors written (16 arrivals)
  B_S = 5,       // MMA commit: S done
  B_U = 6,       // MMA commit: U^T done
  B_PVD = 7,     // MMA commit: P [V | 1] done (S's columns free)
  B_O = 8,       // MMA commit: O, T, R done
  B_KE0 = 9,     // + slot: MMA commit: every MMA of the step read the slot (Q, K, V, X_G)
  B_KWE = 11,    // MMA commit: weighted phi(K) read
  B_XF = 12,     // epi: X_F written (8 arrivals)
  B_XG = 13,     // prep: X_G written (16 arrivals)
  B_CU = 14,     // epi: carried state advanced, U^T read (8 arrivals)
  B_PM = 15,     // epi: P written (8 arrivals)
  B_ED = 16,     // epi: O, T, R read (8 arrivals)
  B_DRAIN = 19,  // MMA commit used when unwinding
  B_TD = 21,     // MMA commit: T done (X_F read)
};
__device__ __forceinline__ uint32_t bar_count(int b) {
  if (b == B_KVR || b == B_QR || b == B_XG) return kPrepWarps;
  if (b == B_XF || b == B_CU || b == B_PM || b == B_ED) return kEpiWarps;
  return 1;
}

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t T_S = 0, T_O = 128, T_T = 208, T_R = 288, T_F = 368, T_U = 432;
// P (fp16, two per column) over S: keys 16j..16j+15 are packed into the
// first 8 of the 16 columns that held their scores, which the warp writing
// them has just read, so any split of the key blocks between the two epi
// warps of a lane quarter is safe.  The split is by parity of the block, so
// that each warp takes one of its quarter's two diagonal blocks.

struct LongParams {
  const float* log_lambda;
  int BH, H, L;
  int NBL, SEGB, nseg;
  const uint8_t* gst;       // [BH][chunks] pre-pass states (kGstBytes each)
  const float* segsum;
  int out_bf16;   // 1: y stored as bfloat16 (64-byte staging rows)
  int* status;
  long long wait_cycles;   // bound of every mbarrier wait, in clock cycles
};

// 1-D bulk copy global -> shared, completion counted on `bar` (bytes).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

template <int MASK>
__device__ __forceinline__ float ell_at(const LongParams& p, int bh, int t, float lh) {
  if (t >= p.L || t < 0) return 0.f;
  if (MASK == MASK_S) return __ldg(p.log_lambda + (size_t)bh * p.L + t);
  if (MASK == MASK_D) return lh;
  return 0.f;
}

// The per-CTA sequence of steps: work items (segments of heads) blockIdx.x,
// + gridDim.x, ...; the 128-token chunks of each item left to right.
struct Step {
  int item, c, c_lo, c_hi;   // chunk c of [c_lo, c_hi)
  int bh, seg;               // the item's head and segment
  __device__ void set_item(const LongParams& p, int it) {
    item = it;
    bh = it / p.nseg;
    seg = it - bh * p.nseg;
    const int nch = (p.L + kC - 1) / kC;
    c_lo = 2 * seg * p.SEGB;
    c_hi = min(nch, 2 * (seg + 1) * p.SEGB);
    c = c_lo;
  }
  __device__ bool valid(const LongParams& p) const { return item < p.BH * p.nseg; }
  __device__ void next(const LongParams& p) {
    if (++c == c_hi) {
      item += gridDim.x;
      if (valid(p)) set_item(p, item);
    }
  }
};

template <int MASK, int PHI>
__global__ void __launch_bounds__(kThreads, 1)
    lion_chunk128_long_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
                              const __grid_constant__ CUtensorMap mapV, const __grid_constant__ CUtensorMap mapO,
                              LongParams prm) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + OFF_TSLOT);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + OFF_TSLOT + 8);
  volatile int* s_range = reinterpret_cast<volatile int*>(smem + OFF_TSLOT + 12);
  auto Qt = [&](int s) { return smem + OFF_SLOT + s * kSlotBytes; };
  auto Kt = [&](int s) { return smem + OFF_SLOT + s * kSlotBytes + kTile; };
  auto Vt = [&](int s) { return smem + OFF_SLOT + s * kSlotBytes + 2 * kTile; };
  auto Gt = [&](int s) { return smem + OFF_SLOT + s * kSlotBytes + 3 * kTile; };
  uint8_t* KWt = smem + OFF_KW;
  uint8_t* XFt = smem + OFF_XF;
  const float* gseg = reinterpret_cast<const float*>(smem + OFF_GSEG);
  auto fac = [&](int s) { return reinterpret_cast<float*>(smem + OFF_FAC) + s * 5 * kC; };
  auto info = [&](int s) { return reinterpret_cast<float*>(smem + OFF_INFO) + s * 8; };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int L = prm.L;

  if (tid == 0) {
    prefetch_tmap(&mapQ);
    prefetch_tmap(&mapK);
    prefetch_tmap(&mapV);
    prefetch_tmap(&mapO);
    for (int b = 0; b < kNumBars; ++b) mbar_init(&bars[b], bar_count(b));
    *s_abort = 0;
    *s_range = 0;
    fence_mbar_init();
  }
  for (int x = tid; x < 16 * 8; x += kThreads) {
    const int r = x >> 3, c8 = x & 7;
    *reinterpret_cast<uint4*>(smem + OFF_ONES + sw128_offset(r, c8)) =
        make_uint4(c8 == 0 ? pack_h2(1.f, 0.f) : 0u, 0u, 0u, 0u);
  }
  // rows 65..79 of the state tiles (X_F, and X_G in each slot past the
  // 65 rows its copy brings) stay zero
  for (int x = tid; x < 3 * 15 * 8; x += kThreads) {
    const int w = x / (15 * 8);
    uint8_t* t = w == 0 ? XFt : Gt(w - 1);
    const int y = x % (15 * 8), r = 65 + y / 8, c8 = y % 8;
    *reinterpret_cast<uint4*>(t + sw128_offset(r, c8)) = make_uint4(0u, 0u, 0u, 0u);
  }
  if (warp == W_TMA) tmem_alloc(tslot, kTmemCols);
  fence_async_smem();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;

  auto waitb = [&](int b, uint32_t parity) -> bool {
    return mbar_wait_or_abort(&bars[b], parity, prm.wait_cycles, kSleepNs, s_abort);
  };
  auto nk_of = [&](int c) { return (min(kC, L - kC * c) + 15) >> 4; };
  // pre-pass state at the right edge of chunk c
  const int nch_all = (L + kC - 1) / kC;
  auto gsrc = [&](int bh, int c) { return prm.gst + ((size_t)bh * nch_all + c) * kGstBytes; };

  if (warp == W_TMA) {
    // =========================== TMA producer ===================================
    pdl_wait();   // the pre-pass tiles come from the grid before this one
    // Step n's Q, K, V and pre-pass state go into slot n & 1 once step n-2's
    // MMAs have read K and its output stores Q and V.
    if (lane == 0) {
      Step ld;
      ld.item = blockIdx.x;
      if (ld.valid(prm)) ld.set_item(prm, ld.item);
      int n = 0;   // steps issued
      int issued_ld[2] = {0, 0};
      long long idle0 = clock64();
      while (ld.valid(prm) && !*s_abort) {
        bool progress = false;
        const int s = n & 1;
        if (n < 2 || mbar_try_wait(&bars[B_KE0 + s], ((n >> 1) - 1) & 1)) {
          const int bh = ld.bh;
          mbar_arrive_expect_tx(&bars[B_LD0 + s], (uint32_t)(3 * kTile + kGstBytes));
          tma_load_3d(Vt(s), &mapV, &bars[B_LD0 + s], 0, kC * ld.c, bh);
          tma_load_3d(Kt(s), &mapK, &bars[B_LD0 + s], 0, kC * ld.c, bh);
          tma_load_3d(Qt(s), &mapQ, &bars[B_LD0 + s], 0, kC * ld.c, bh);
          bulk_load(Gt(s), gsrc(bh, ld.c), (uint32_t)kGstBytes, &bars[B_LD0 + s]);
          ++issued_ld[s];
          ++n;
          ld.next(prm);
          {
            // the step after next waits for this slot's successor: start its
            // tiles towards L2 now
            Step pf = ld;
            pf.next(prm);
            if (pf.valid(prm)) {
              const int bhp = pf.bh;
              tma_prefetch_3d(&mapV, 0, kC * pf.c, bhp);
              tma_prefetch_3d(&mapK, 0, kC * pf.c, bhp);
              tma_prefetch_3d(&mapQ, 0, kC * pf.c, bhp);
            }
          }
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
        const long long lim = prm.wait_cycles / 4;
        for (int s = 0; s < 2; ++s)
          if (issued_ld[s]) mbar_wait(&bars[B_LD0 + s], (issued_ld[s] - 1) & 1, lim);
      }
    }
  } else if (warp == W_MMA) {
    // =========================== MMA issuer =====================================
    if (lane == 0) {
      const uint32_t idUT = idesc_f16(128, 64, true, true);
      const uint32_t idPV = idesc_f16(128, 80, false, true);
      const uint32_t idX = idesc_f16(128, 80, false, false);
      const uint32_t ones = smem_u32(smem + OFF_ONES);
      bool issued = false;
      Step st;
      st.item = blockIdx.x;
      if (st.valid(prm)) st.set_item(prm, st.item);
      for (int n = 0; st.valid(prm); ++n, st.next(prm)) {
        const int s = n & 1, nk = nk_of(st.c);
        if (!waitb(B_KVR, n & 1) || !waitb(B_QR, n & 1)) break;
        if (n >= 1 && !waitb(B_PVD, (n - 1) & 1)) break;   // S's columns: P of the previous chunk read
        tc_fence_after();
        const uint32_t idS = idesc_f16(128, 16 * nk, false, false);
#pragma unroll
        {
          uint64_t da = kmaj(Qt(s), 0), db = kmaj(Kt(s), 0);
#pragma unroll
          for (int k = 0; k < 4; ++k, da += kKmajStep, db += kKmajStep)
            mma_bf16(tbase + T_S, da, db, idS, k > 0 ? 1u : 0u);
        }
        mma_commit(&bars[B_S]);
        issued = true;
        if (n >= 1 && !waitb(B_CU, (n - 1) & 1)) break;    // U^T of the previous chunk read
        tc_fence_after();
        {
          const uint32_t a = smem_u32(Vt(s));
          const uint32_t b = smem_u32(MASK == MASK_LIT ? Kt(s) : KWt);
          uint64_t da = mnmaj(a, 0, ones - a), db = mnmaj(b, 0, 0);
          for (int k = 0; k < nk; ++k, da += kMnmajOnesStep, db += kMnmajStep)
            mma_bf16(tbase + T_U, da, db, idUT, k > 0 ? 1u : 0u);
        }
        mma_commit(&bars[B_U]);
        mma_commit(&bars[B_KWE]);
        if (n >= 1 && !waitb(B_ED, (n - 1) & 1)) break;    // O, T, R of the previous chunk read
        if (!waitb(B_XF, n & 1)) break;
        tc_fence_after();
#pragma unroll
        {
          uint64_t da = kmaj(Qt(s), 0), db = kmaj(XFt, 0);
#pragma unroll
          for (int k = 0; k < 4; ++k, da += kKmajStep, db += kKmajStep)
            mma_bf16(tbase + T_T, da, db, idX, k > 0 ? 1u : 0u);
        }
        mma_commit(&bars[B_TD]);
        if (!waitb(B_XG, n & 1)) break;
        tc_fence_after();
#pragma unroll
        {
          uint64_t da = kmaj(Qt(s), 0), db = kmaj(Gt(s), 0);
#pragma unroll
          for (int k = 0; k < 4; ++k, da += kKmajStep, db += kKmajStep)
            mma_bf16(tbase + T_R, da, db, idX, k > 0 ? 1u : 0u);
        }
        if (!waitb(B_PM, n & 1)) break;
        tc_fence_after();
        {
          const uint32_t v = smem_u32(Vt(s));
          uint64_t dv = mnmaj(v, 0, ones - v);
          for (int k = 0; k < nk; ++k, dv += kMnmajOnesStep)
            mma_tmem_a(tbase + T_O, tbase + T_S + 16 * k, dv, idPV, k > 0 ? 1u : 0u);
        }
        mma_commit(&bars[B_PVD]);
        mma_commit(&bars[B_O]);
        mma_commit(&bars[B_KE0 + s]);
      }
      if (*s_abort && issued) {
        mma_commit(&bars[B_DRAIN]);
        mbar_wait(&bars[B_DRAIN], 0, prm.wait_cycles / 4);
      }
    }
  } else if (warp < W_EPI) {
    // =========================== prep: four threads per token ====================
    pdl_wait();   // the segment summaries come from the grid before this one
    const int pw = warp - W_PREP;            // 0..15: tokens 8 pw .. 8 pw + 7
    const int pt = 32 * pw + lane;
    const int t = pt >> 2, qq = pt & 3;      // token within the chunk, quarter row
    const int j0 = 2 * qq;                   // first 16-byte chunk of this quarter row
    const uint32_t peers = 0xfu << (lane & 28);
    bool good = true;
    Step st;
    st.item = blockIdx.x;
    if (st.valid(prm)) st.set_item(prm, st.item);
    // l of the chunk's tokens 4 lane .. 4 lane + 3 (every warp takes the whole
    // chunk's prefix by itself)
    float ell_next[4] = {0.f, 0.f, 0.f, 0.f}, lnext_next = 0.f;
    auto load_ell = [&](const Step& x, float* e, float* en) {
      const int bh = x.bh;
      const float lh = MASK == MASK_D ? __ldg(prm.log_lambda + bh % prm.H) : 0.f;
#pragma unroll
      for (int r = 0; r < 4; ++r) e[r] = ell_at<MASK>(prm, bh, kC * x.c + 4 * lane + r, lh);
      *en = ell_at<MASK>(prm, bh, kC * x.c + kC, lh);   // first token after the chunk
    };
    if (st.valid(prm)) load_ell(st, ell_next, &lnext_next);
    float cum = 0.f, tseg = 0.f, lafter = 0.f;
    for (int n = 0; st.valid(prm); ++n) {
      const int s = n & 1, tok = kC * st.c + t;
      float ell[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) ell[r] = ell_next[r];
      const float lnext = lnext_next;
      const bool first = st.c == st.c_lo;
      if (first) {
        // a new segment: bookkeeping for its backward entering state
        const int bh = st.bh, seg = st.seg;
        tseg = prm.nseg > 1 ? __ldg(prm.segsum + (size_t)st.item * kSegSumFloats + 2 * 64 * kLongStateCols) : 0.f;
        const float lh = MASK == MASK_D ? __ldg(prm.log_lambda + bh % prm.H) : 0.f;
        lafter = ell_at<MASK>(prm, bh, 256 * min(prm.NBL, (seg + 1) * prm.SEGB), lh);
        cum = 0.f;
        if (prm.nseg > 1) {
          // The segment's entering states, chained from the summaries the
          // pre-pass wrote (with several segments a head each CTA has one
          // item, so this runs once, before any chunk):
          // * forward, into the carried TMEM state: F = exp(T_s) F + U_s for
          //   s = 0 .. seg - 1 (this warp: TMEM lanes of its quarter, 16 of
          //   the 64 columns m);
          // * backward, into shared memory: G = d_s G + U_s from the last
          //   segment down to seg + 1, d_s the decay across segment s shifted
          //   by one token.
          {
            const int lq = warp & 3, ln = 32 * lq + lane;   // TMEM lane = state column n
            const int m0 = 16 * ((warp - W_PREP) >> 2);
            float v[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] = 0.f;
            if (ln < kLongStateCols) {
#pragma unroll 1
              for (int sg = 0; sg < seg; ++sg) {
                const float* ss = prm.segsum + ((size_t)bh * prm.nseg + sg) * kSegSumFloats;
                const float dsg = __expf(__ldg(ss + 2 * 64 * kLongStateCols));
#pragma unroll
                for (int e = 0; e < 16; ++e) v[e] = dsg * v[e] + __ldg(ss + (m0 + e) * kLongStateCols + ln);
              }
            }
            tmem_st16(tbase + ((uint32_t)(32 * lq) << 16) + T_F + m0, v);
            tmem_wait_st();
          }
          const int segtok = prm.SEGB * 256;
          float* gw = reinterpret_cast<float*>(smem + OFF_GSEG);
          float g[10];
#pragma unroll
          for (int r = 0; r < 10; ++r) g[r] = 0.f;
#pragma unroll 1
          for (int sg = prm.nseg - 1; sg > seg; --sg) {
            // every load of a segment in flight at once
            const float* ss = prm.segsum + ((size_t)bh * prm.nseg + sg) * kSegSumFloats;
            float u[10];
#pragma unroll
            for (int r = 0; r < 10; ++r) u[r] = __ldg(ss + 64 * kLongStateCols + pt + 512 * r);
            const float ts = __ldg(ss + 2 * 64 * kLongStateCols);
            const float lfirst = ell_at<MASK>(prm, bh, sg * segtok, lh);
            const float lnx = ell_at<MASK>(prm, bh, (sg + 1) * segtok, lh);
            const float dsg = __expf(ts - lfirst + lnx);
#pragma unroll
            for (int r = 0; r < 10; ++r) g[r] = dsg * g[r] + u[r];
          }
#pragma unroll
          for (int r = 0; r < 10; ++r) gw[pt + 512 * r] = g[r];
          tc_fence_before();
          // every prep thread's share written, and the epilogue may read the
          // carried state
          bar_and(3, (kPrepWarps + kEpiWarps) * 32, true);
        }
      }
      // ---- chunk-local inclusive prefix
      float p, T, pfirst;
      chunk_prefix_warp(ell, t, &p, &T, &pfirst);
      {
        // the next step's decays, loaded a whole step ahead of their use
        Step nx = st;
        nx.next(prm);
        if (nx.valid(prm)) load_ell(nx, ell_next, &lnext_next);
      }
      const float pref = 0.5f * (pfirst + T);
      const bool exact = (pfirst - T) > 2.f * kMaxFactorRange;
      const bool live = tok < L;

      if (!waitb(B_LD0 + s, (n >> 1) & 1)) good = false;
      good = __all_sync(0xffffffffu, good);
      // ---- V -> fp16 in place
      if (good && live) {
        uint8_t* vt = Vt(s);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          uint4* a = reinterpret_cast<uint4*>(vt + sw128_offset(t, j0 + j));
          *a = bf8_to_h8_chk(*a, s_range);
        }
      }
      // ---- phi(k) in place and its weighted copy w_j phi(k_j), w_j = exp(p_e - p_j)
      if (good && live) {
        uint8_t* kt = Kt(s);
        float kv[16];
#pragma unroll
        for (int j = 0; j < 2; ++j)
          unpack8_bf(*reinterpret_cast<const uint4*>(kt + sw128_offset(t, j0 + j)), kv + 8 * j);
        phi_part<PHI, 16, 4>(kv, peers);
#pragma unroll
        for (int j = 0; j < 2; ++j) *reinterpret_cast<uint4*>(kt + sw128_offset(t, j0 + j)) = pack8_h(kv + 8 * j);
        if (MASK != MASK_LIT) {
          if (n >= 1 && !waitb(B_KWE, (n - 1) & 1)) good = false;
          if (good) {
            const float w = ex2((T - p) * kLog2e);
            const float2 w2 = make_float2(w, w);
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              float y8[8];
#pragma unroll
              for (int e = 0; e < 8; e += 2) {
                const float2 u = mul2(make_float2(kv[8 * j + e], kv[8 * j + e + 1]), w2);
                y8[e] = u.x;
                y8[e + 1] = u.y;
              }
              *reinterpret_cast<uint4*>(KWt + sw128_offset(t, j0 + j)) = pack8_h(y8);
            }
          }
        }
      } else if (good && MASK != MASK_LIT) {
        if (n >= 1 && !waitb(B_KWE, (n - 1) & 1)) good = false;
        if (good) {
#pragma unroll
          for (int j = 0; j < 2; ++j)
            *reinterpret_cast<uint4*>(KWt + sw128_offset(t, j0 + j)) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      // Arrivals on KVR and QR wait for the previous chunk's state MMA (issued
      // after the MMA thread's own waits on them) and on XG for its output
      // product, so that no barrier the MMA thread polls runs two phases ahead
      // of its wait.  LION-S and -D already waited above for the weighted copy.
      if (MASK == MASK_LIT && n >= 1 && !waitb(B_KWE, (n - 1) & 1)) good = false;
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_KVR]);
      // ---- factors and phi(q)
      if (good && qq == 0) {
        float* f = fac(s);
        const float d = (p - pref) * kLog2e;
        f[t] = ex2(d);
        f[kC + t] = ex2(-d);
        f[2 * kC + t] = ex2(p * kLog2e);                       // a_i
        f[3 * kC + t] = ex2((T + lnext - p) * kLog2e);         // b_i
        f[4 * kC + t] = p;
        if (t == 0) {
          float* in = info(s);
          in[I_EXACT] = exact ? 1.f : 0.f;
          in[I_T] = T;
          in[I_LNEXT] = lnext;
        }
      }
      if (good && live) {
        uint8_t* qt = Qt(s);
        float qv[16];
#pragma unroll
        for (int j = 0; j < 2; ++j)
          unpack8_bf(*reinterpret_cast<const uint4*>(qt + sw128_offset(t, j0 + j)), qv + 8 * j);
        phi_part<PHI, 16, 4>(qv, peers);
#pragma unroll
        for (int j = 0; j < 2; ++j) *reinterpret_cast<uint4*>(qt + sw128_offset(t, j0 + j)) = pack8_h(qv + 8 * j);
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_QR]);
      // ---- X_G = pre-pass state + decay * the segment's backward entering
      //      state, in place in the slot's pre-pass tile (row i = state column
      //      i, 64 = z; this thread: row t, state rows m = 16 qq .. 16 qq + 15)
      // (one segment a head: no entering state, X_G is the tile as loaded)
      if (prm.nseg > 1 && good && t < 65) {
        // exp(P at the first token after the segment - P at the first token after the chunk)
        const float fdec = __expf(tseg - (cum + T) - lnext + lafter);
        uint8_t* grow = Gt(s) + t * 128;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int off = ((j0 + j) ^ (t & 7)) << 4;
          float y8[8];
          unpack8_h(*reinterpret_cast<const uint4*>(grow + off), y8);
#pragma unroll
          for (int e = 0; e < 8; ++e) y8[e] = fmaf(fdec, gseg[(8 * (j0 + j) + e) * kLongStateCols + t], y8[e]);
          *reinterpret_cast<uint4*>(grow + off) = pack8_h(y8);
        }
      }
      cum += T;
      if (n >= 1 && !waitb(B_O, (n - 1) & 1)) good = false;
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_XG]);
      st.next(prm);
    }
  } else {
    // =========================== epi: two warps per TMEM lane quarter =============
    const int ew = warp - W_EPI;
    const int q = warp & 3;                  // TMEM lane quarter: rows 32q..32q+31
    const int hc = ew >> 2;                  // column half
    const int i = 32 * q + lane;             // row (and state-tile row)
    const uint32_t lane_off = (uint32_t)(32 * q) << 16;
    const bool st_row = i < kStRows;         // lanes holding a state-tile row
    bool good = true;
    // X_F = the carried state, transposed, K-major fp16 (rows = output columns)
    auto write_xf = [&]() {
      if (q < 3) {
        float u0[16], u1[16];
        const uint32_t fa = tbase + lane_off + T_F + 32 * hc;
        tmem_ld16(fa, u0);
        tmem_ld16(fa + 16, u1);
        tmem_wait_ld();
        reg_fence16(u0);
        reg_fence16(u1);
        if (st_row) {
          uint8_t* row = XFt + i * 128;
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            *reinterpret_cast<uint4*>(row + (((4 * hc + j) ^ (i & 7)) << 4)) = pack8_h(u0 + 8 * j);
            *reinterpret_cast<uint4*>(row + (((4 * hc + 2 + j) ^ (i & 7)) << 4)) = pack8_h(u1 + 8 * j);
          }
        }
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_XF]);
    };
    Step st;
    st.item = blockIdx.x;
    if (st.valid(prm)) st.set_item(prm, st.item);
    // with several segments a head the prep warps chain the entering forward
    // state into the carried TMEM state before any chunk: wait for it
    if (prm.nseg > 1 && st.valid(prm)) {
      bar_and(3, (kPrepWarps + kEpiWarps) * 32, true);
      tc_fence_after();
    }
    for (int n = 0; st.valid(prm) && good; ++n) {
      const int s = n & 1, c = st.c, nk = nk_of(c), bh = st.bh;
      const bool first = c == st.c_lo, last = c + 1 == st.c_hi, warp_ok = kC * c + 32 * q < L;
      const float* f = fac(s);
      const float* alpha = f;
      const float* rho = f + kC;
      const float* pp = f + 4 * kC;
      if (first) {
        // a new segment: its forward entering state into the carried TMEM
        // state, then X_F once the previous chunk's T has read the tile
        // (with several segments a head the state was chained before the loop)
        if (prm.nseg == 1 && q < 3) {
          float v[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] = 0.f;
          tmem_st16(tbase + lane_off + T_F + 32 * hc, v);
          tmem_st16(tbase + lane_off + T_F + 32 * hc + 16, v);
          tmem_wait_st();
        }
        if (n >= 1 && !waitb(B_TD, (n - 1) & 1)) good = false;
        good = __all_sync(0xffffffffu, good);
        if (!good) break;
        write_xf();
      }
      // ---- P = S * M, fp16, over S (this warp's key blocks: those of parity hc)
      if (!waitb(B_S, n & 1)) good = false;
      good = __all_sync(0xffffffffu, good);
      tc_fence_after();
      if (good && warp_ok && hc < nk) {
        const bool exact = info(s)[I_EXACT] != 0.f;
        const float ai = alpha[i], ri = rho[i], pi = pp[i];
        const uint32_t sa = tbase + lane_off + T_S;
        float sb0[16], sb1[16];
#pragma unroll 1
        for (int jj = hc; jj < nk; jj += 4) {
          uint32_t pk[8];
          const bool has1 = jj + 2 < nk;
          tmem_ld16(sa + 16 * jj, sb0);
          if (has1) tmem_ld16(sa + 16 * (jj + 2), sb1);
          tmem_wait_ld();
          reg_fence16(sb0);
          reg_fence16(sb1);
          mask_block<MASK>(sb0, 16 * jj, i, 32 * q, exact, ai, ri, pi, alpha, rho, pp);
#pragma unroll
          for (int e = 0; e < 8; ++e) pk[e] = pack_h2(sb0[2 * e], sb0[2 * e + 1]);
          tmem_st8(sa + 16 * jj, pk);
          if (has1) {
            mask_block<MASK>(sb1, 16 * (jj + 2), i, 32 * q, exact, ai, ri, pi, alpha, rho, pp);
#pragma unroll
            for (int e = 0; e < 8; ++e) pk[e] = pack_h2(sb1[2 * e], sb1[2 * e + 1]);
            tmem_st8(sa + 16 * (jj + 2), pk);
          }
        }
      }
      // this step's scalars, read before P is handed over (the output product
      // needs P): once that product is done the slot, and with it these
      // factors, may be refilled for step n + 2.  Read here rather than before
      // the mask, they hold no registers through it.
      const float dec = MASK == MASK_LIT ? 1.f : __expf(info(s)[I_T]);
      const float a_out = f[2 * kC + i], b_out = f[3 * kC + i];
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_PM]);
      // ---- advance the carried state: F <- exp(T_c) F + U^T (the U commit
      //      also means prep's per-chunk scalars of this step are written),
      //      then the next chunk's X_F once this chunk's T has read the tile;
      //      the output product runs meanwhile
      if (!waitb(B_U, n & 1)) good = false;
      good = __all_sync(0xffffffffu, good);
      tc_fence_after();
      if (good && q < 3) {
#pragma unroll 1
        for (int h2 = 0; h2 < 2; ++h2) {
          float fv[16], uv[16];
          const uint32_t off = lane_off + 32 * hc + 16 * h2;
          tmem_ld16(tbase + off + T_F, fv);
          tmem_ld16(tbase + off + T_U, uv);
          tmem_wait_ld();
          reg_fence16(fv);
          reg_fence16(uv);
#pragma unroll
          for (int e = 0; e < 16; ++e) fv[e] = fmaf(dec, fv[e], uv[e]);
          tmem_st16(tbase + off + T_F, fv);
        }
        tmem_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_CU]);
      if (!last) {
        if (!waitb(B_TD, n & 1)) good = false;
        good = __all_sync(0xffffffffu, good);
        if (good) {
          tc_fence_after();
          write_xf();
        }
      }
      // ---- y = (O + a T + b R)[0:64] / (O + a T + b R)[64], this warp's 32
      //      columns, staged (128-byte swizzle) in its own 4 KB once its
      //      previous store has read them, written by TMA
      if (!waitb(B_O, n & 1)) good = false;
      good = __all_sync(0xffffffffu, good);
      tc_fence_after();
      if (lane == 0) bulk_wait_read();
      __syncwarp();
      if (good && warp_ok) {
        const float2 a2 = make_float2(a_out, a_out), b2 = make_float2(b_out, b_out);
        const uint32_t base = tbase + lane_off;
        uint8_t* stg = smem + OFF_STG + ew * 4096;
        uint8_t* row = stg + lane * 128;
        float2 inv2 = make_float2(0.f, 0.f);
        {
          // column 64, the row sums
          float z[3];
          z[0] = tmem_ld1(base + T_O + 64);
          z[1] = tmem_ld1(base + T_T + 64);
          z[2] = tmem_ld1(base + T_R + 64);
          tmem_wait_ld();
          asm volatile("" : "+f"(z[0]), "+f"(z[1]), "+f"(z[2]));
          const float den = z[0] + a_out * z[1] + b_out * z[2];
          const float inv = 1.f / den;
          // a score past the fp16 range (unbounded features) leaves the row sum
          // non-finite: fp16 operands cannot make an fp32 sum overflow otherwise
          if (!(fabsf(den) <= 3.0e38f)) *s_range = 1;
          inv2 = make_float2(inv, inv);
        }
#pragma unroll 1
        for (int h4 = 0; h4 < 4; ++h4) {
          const int col = 32 * hc + 8 * h4;
          float o[8], tt[8], rr[8];
          tmem_ld8(base + T_O + col, o);
          tmem_ld8(base + T_T + col, tt);
          tmem_ld8(base + T_R + col, rr);
          tmem_wait_ld();
          reg_fence8(o);
          reg_fence8(tt);
          reg_fence8(rr);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float2 x = make_float2(o[2 * e], o[2 * e + 1]);
            x = fma2(a2, make_float2(tt[2 * e], tt[2 * e + 1]), x);
            x = fma2(b2, make_float2(rr[2 * e], rr[2 * e + 1]), x);
            x = mul2(x, inv2);
            o[2 * e] = x.x;
            o[2 * e + 1] = x.y;
          }
          if (prm.out_bf16) {
            // bfloat16: 64-byte staging rows, no swizzle
            *reinterpret_cast<uint4*>(stg + lane * 64 + (h4 << 4)) = pack8_bf(o);
          } else {
#pragma unroll
            for (int e = 0; e < 2; ++e)
              *reinterpret_cast<float4*>(row + (((2 * h4 + e) ^ (lane & 7)) << 4)) =
                  make_float4(o[4 * e], o[4 * e + 1], o[4 * e + 2], o[4 * e + 3]);
          }
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_3d(&mapO, stg, 32 * hc, kC * c + 32 * q, bh);
          bulk_commit();
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_ED]);
      st.next(prm);
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

bool chunk128_long_supported(const Problem& p) {
  return p.dtype == DT_BF16 && p.d == kD && p.chunk == kC && p.L > 2 * kC;
}

namespace {
size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
struct LongWs {
  size_t gst, segsum;
};
LongWs long_ws(int B, int H, int L, const LongPlan& plan) {
  const size_t BH = (size_t)B * H, nch = (size_t)(L + kC - 1) / kC;
  return {align256(BH * nch * kGstBytes), align256(BH * plan.nseg * kSegSumFloats * 4)};
}
}  // namespace

size_t chunk128_long_workspace_bytes(int B, int H, int L) {
  if (L <= 2 * kC) return 0;
  const LongWs w = long_ws(B, H, L, long_plan(B, H, L));
  return w.gst + w.segsum;
}

cudaError_t launch_chunk128_long(const Problem& p, void* ws, int* status, cudaStream_t s) {
  if (!ws) return cudaErrorInvalidValue;
  const LongPlan plan = long_plan(p.B, p.H, p.L);
  const LongWs w = long_ws(p.B, p.H, p.L, plan);
  uint8_t* gst = static_cast<uint8_t*>(ws);
  float* segsum = reinterpret_cast<float*>(gst + w.gst);
  const int BH = p.B * p.H;
  // The main pass chains the segments' entering states itself from the
  // pre-pass summaries, which needs one item a CTA when heads are cut into
  // segments (B * H * segments never exceeds the SMs then)
  if (plan.nseg > 1 && BH * plan.nseg > sm_count()) return cudaErrorInvalidValue;
  cudaError_t e = launch_chunk128_pre(p, plan, gst, segsum, status, s);
  if (e != cudaSuccess) return e;
  CUtensorMap mq, mk, mv, mo;
  if (!make_map128(&mq, p.q, p.L, BH) || !make_map128(&mk, p.k, p.L, BH) || !make_map128(&mv, p.v, p.L, BH) ||
      !(p.out_bf16 ? make_out_map_bf16(&mo, p.out, p.L, BH, 32) : make_out_map(&mo, p.out, p.L, BH)))
    return cudaErrorInvalidValue;
  LongParams prm;
  prm.out_bf16 = p.out_bf16;
  prm.log_lambda = p.log_lambda;
  prm.BH = BH;
  prm.H = p.H;
  prm.L = p.L;
  prm.NBL = plan.NBL;
  prm.SEGB = plan.SEGB;
  prm.nseg = plan.nseg;
  prm.gst = gst;
  prm.segsum = segsum;
  prm.status = status;
  prm.wait_cycles = wait_limit_cycles();
  void (*kern)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap, LongParams) = nullptr;
#define LION_C128L_CASE(M, F) \
  if (p.mask_kind == M && p.phi == F) kern = lion_chunk128_long_kernel<M, F>;
  LION_C128L_CASE(MASK_LIT, PHI_ELU1)
  LION_C128L_CASE(MASK_LIT, PHI_SILU_L2)
  LION_C128L_CASE(MASK_LIT, PHI_IDENTITY)
  LION_C128L_CASE(MASK_D, PHI_ELU1)
  LION_C128L_CASE(MASK_D, PHI_SILU_L2)
  LION_C128L_CASE(MASK_D, PHI_IDENTITY)
  LION_C128L_CASE(MASK_S, PHI_ELU1)
  LION_C128L_CASE(MASK_S, PHI_SILU_L2)
  LION_C128L_CASE(MASK_S, PHI_IDENTITY)
#undef LION_C128L_CASE
  if (!kern) return cudaErrorInvalidValue;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const int items = BH * plan.nseg;
  const int grid = items < sm_count() ? items : sm_count();
  // launched as a programmatic dependent of the pre-pass, so that its launch
  // and set-up overlap the pre-pass's end; the warps that read the pre-pass's
  // output wait for it (pdl_wait).  (The pre-pass signals nothing early: main
  // pass CTAs idling on the SMs the pre-pass leaves free cost more than they
  // saved at the LRA shape, 186.5 against 184.8 us.)
  e = launch_dependent(kern, dim3(grid), dim3(kThreads), kSmemBytes, s, mq, mk, mv, mo, prm);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace lion
