// lion_c128P.cu -- backward pre-pass of the chunkwise LION forward with
// 128-token chunks, for sequences longer than 256 tokens, on the
// 5th-generation tensor cores (tcgen05 + TMEM + TMA), bfloat16 inputs, head
// dim 64.
//
// Chunkwise form ("LION Part IV - Results", "LION Chunk"; rebuttal page
// "LION: A bidirectional framework ...", reply "4: Practicality of Recurrent
// Inference").  With P the inclusive prefix of l = log(lambda) and chunk c =
// tokens [s_c, e_c], the backward state entering chunk c from the right is
//
//   G_c = sum_{j > e_c} exp(P_j - P_{s_{c+1}}) phi(k_j) [v_j; 1]^T
//
// (anchored at the first token after the chunk), and it obeys
//
//   G_{c-1} = exp(P_{s_{c+1}} - P_{s_c}) G_c + U^B_c,
//   U^B_c   = sum_{j in c} exp(P_j - P_{s_c}) phi(k_j) [v_j; 1]^T,
//
// where P_{s_{c+1}} - P_{s_c} = T_c - l_{s_c} + l_{s_{c+1}} (T_c the sum of l
// over the chunk: the backward decay is shifted by one token).  Each CTA walks
// one segment of a head (the 256-token-block segments of the segment plan)
// from right to left, one chunk at a time, and writes
//   * G_c restricted to the segment (zero for the segment's last chunk) for
//     every chunk, as an fp16 tile transposed to rows n of [state column n
//     over m; z], the layout of the main pass's operand tile;
//   * the segment's backward summary (G after its first chunk) and forward
//     summary sum_j exp(P_last - P_j) phi(k_j) [v_j; 1]^T, with the sum of l
//     over the segment, which the main pass chains into each segment's
//     entering states.
// The carried G lives in TMEM (fp32, transposed: lane n = state column, lane
// 64 = z) and is advanced by the epilogue warps; U^B_c and the forward
// summary come from MMAs
//   U^B_c^T   = [V_c | 1]^T (w^B o phi(K_c))   M=128 N=64 K=n_c
//   F_acc^T  += [V_c | 1]^T (w^F o phi(K_c))   (accumulated over the segment)
// with w^B_j = exp(P_j - P_{s_c}) and w^F_j = exp(P_last - P_j), both <= 1.
// A weight below the fp16 range stands for a term that is negligible against
// the tokens near the anchor.  LION-LIT has no decay: phi(K) serves both.
//
// Warps: 0 TMA (K and V of a chunk into one of two slots), 1 MMA issue, 2-17
// "prep" (four threads per token: prefix of l, V -> fp16, phi(k) and its two
// weighted copies), 18-25 "epi" (two warps per TMEM lane quarter, each one
// half of the 64 state columns m: state tiles out, carry, summaries).  Prep of
// chunk c-1 overlaps the epilogue of chunk c.
//
// Every mbarrier wait is bounded; on timeout the kernel records an error in
// `status`, waits (bounded) for its own copies and MMAs in flight, releases
// its TMEM and returns.
#include "c128_common.cuh"
#include "lion_common.cuh"
#include "lion_internal.h"
#include "tc_ptx.cuh"

namespace lion {
namespace {

using namespace tc;
using namespace c128;

constexpr int kPrepWarps = 16, kEpiWarps = 8;
constexpr int W_TMA = 0, W_MMA = 1, W_PREP = 2, W_EPI = W_PREP + kPrepWarps;
constexpr int kThreads = (W_EPI + kEpiWarps) * 32;   // 832
constexpr uint32_t kSleepNs = 2000u;

// shared-memory map (bytes from a 1024-aligned base)
constexpr int kSlotBytes = 2 * kTile;                 // K, V
constexpr int OFF_SLOT = 0;                           // [2] slots
constexpr int OFF_KB = OFF_SLOT + 2 * kSlotBytes;     // w^B o phi(K)
constexpr int OFF_KF = OFF_KB + kTile;                // w^F o phi(K)
constexpr int OFF_ONES = OFF_KF + kTile;              // 16 rows, column 0 = 1
constexpr int OFF_INFO = OFF_ONES + 2048;             // [slot] float[8] per-chunk scalars
constexpr int OFF_BAR = OFF_INFO + 2 * 8 * 4;
constexpr int kNumBars = 12;
constexpr int OFF_TSLOT = OFF_BAR + kNumBars * 8;
constexpr int kSmemBytes = OFF_TSLOT + 16 + 1024;     // + alignment slack
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
static_assert(OFF_KB % 1024 == 0 && OFF_KF % 1024 == 0 && OFF_ONES % 1024 == 0, "swizzled tiles");

// per-chunk scalars (INFO)
enum { I_T = 0, I_DEC = 1 };

// mbarriers
enum {
  B_LD0 = 0,    // + slot: K and V landed (TMA, tx bytes)
  B_KVR = 2,    // prep: V, the weighted phi(K) copies and the chunk's scalars written (16 arrivals)
  B_U = 3,      // MMA commit: U^B and the forward summary of the chunk done
  B_KWE = 4,    // MMA commit: the weighted copies read
  B_KVE0 = 5,   // + slot: MMA commit: the slot's K and V read
  B_CU = 7,     // epi: U^B read and the carried state advanced (8 arrivals)
  B_DRAIN = 8,  // MMA commit used when unwinding
};
__device__ __forceinline__ uint32_t bar_count(int b) {
  if (b == B_KVR) return kPrepWarps;
  if (b == B_CU) return kEpiWarps;
  return 1;
}

// TMEM columns
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t T_G = 0;     // carried backward state, transposed
constexpr uint32_t T_U = 64;    // U^B of the chunk, transposed
constexpr uint32_t T_FA = 128;  // forward summary of the segment so far, transposed

struct PreParams {
  const float* log_lambda;
  int BH, H, L;
  int NBL, SEGB, nseg;
  uint8_t* gst;     // [BH][chunks] kGstBytes each
  float* segsum;    // [BH][nseg] kSegSumFloats each
  int* status;
  long long wait_cycles;   // bound of every mbarrier wait, in clock cycles
};

template <int MASK>
__device__ __forceinline__ float ell_at(const PreParams& p, int bh, int t, float lh) {
  if (t >= p.L || t < 0) return 0.f;
  if (MASK == MASK_S) return __ldg(p.log_lambda + (size_t)bh * p.L + t);
  if (MASK == MASK_D) return lh;
  return 0.f;
}

// The per-CTA sequence of steps: work items (segments of heads) blockIdx.x,
// + gridDim.x, ...; the 128-token chunks of each item right to left.
struct Step {
  int item, c, c_lo, c_hi;   // chunk c of [c_lo, c_hi)
  int bh, seg;               // the item's head and segment
  __device__ void set_item(const PreParams& p, int it) {
    item = it;
    bh = it / p.nseg;
    seg = it - bh * p.nseg;
    const int nch = (p.L + kC - 1) / kC;
    c_lo = 2 * seg * p.SEGB;
    c_hi = min(nch, 2 * (seg + 1) * p.SEGB);
    c = c_hi - 1;
  }
  __device__ bool valid(const PreParams& p) const { return item < p.BH * p.nseg; }
  __device__ void next(const PreParams& p) {
    if (c-- == c_lo) {
      item += gridDim.x;
      if (valid(p)) set_item(p, item);
    }
  }
};

template <int MASK, int PHI>
__global__ void __launch_bounds__(kThreads, 1)
    lion_chunk128_pre_kernel(const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapV,
                             PreParams prm) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + OFF_TSLOT);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + OFF_TSLOT + 8);
  volatile int* s_range = reinterpret_cast<volatile int*>(smem + OFF_TSLOT + 12);
  auto Kt = [&](int s) { return smem + OFF_SLOT + s * kSlotBytes; };
  auto Vt = [&](int s) { return smem + OFF_SLOT + s * kSlotBytes + kTile; };
  uint8_t* KBt = smem + OFF_KB;
  uint8_t* KFt = smem + OFF_KF;
  auto info = [&](int s) { return reinterpret_cast<float*>(smem + OFF_INFO) + s * 8; };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int L = prm.L;
  const int nch = (L + kC - 1) / kC;

  if (tid == 0) {
    prefetch_tmap(&mapK);
    prefetch_tmap(&mapV);
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
  if (warp == W_TMA) tmem_alloc(tslot, kTmemCols);
  fence_async_smem();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;

  auto waitb = [&](int b, uint32_t parity) -> bool {
    return mbar_wait_or_abort(&bars[b], parity, prm.wait_cycles, kSleepNs, s_abort);
  };
  auto nk_of = [&](int c) { return (min(kC, L - kC * c) + 15) >> 4; };

  if (warp == W_TMA) {
    // =========================== TMA producer ===================================
    // Step n's K and V go into slot n & 1 once step n-2's MMAs have read them.
    if (lane == 0) {
      Step ld;
      ld.item = blockIdx.x;
      if (ld.valid(prm)) ld.set_item(prm, ld.item);
      int n = 0;
      int issued[2] = {0, 0};
      long long idle0 = clock64();
      while (ld.valid(prm) && !*s_abort) {
        const int s = n & 1;
        if (n < 2 || mbar_try_wait(&bars[B_KVE0 + s], ((n >> 1) - 1) & 1)) {
          const int bh = ld.bh;
          mbar_arrive_expect_tx(&bars[B_LD0 + s], (uint32_t)(2 * kTile));
          tma_load_3d(Kt(s), &mapK, &bars[B_LD0 + s], 0, kC * ld.c, bh);
          tma_load_3d(Vt(s), &mapV, &bars[B_LD0 + s], 0, kC * ld.c, bh);
          ++issued[s];
          ++n;
          ld.next(prm);
          {
            // the step after next waits for this slot's successor: start its
            // tiles towards L2 now
            Step pf = ld;
            pf.next(prm);
            if (pf.valid(prm)) {
              tma_prefetch_3d(&mapK, 0, kC * pf.c, pf.bh);
              tma_prefetch_3d(&mapV, 0, kC * pf.c, pf.bh);
            }
          }
          idle0 = clock64();
        } else {
          __nanosleep(64);
          if (clock64() - idle0 > prm.wait_cycles) *s_abort = 1;
        }
      }
      if (*s_abort) {
        const long long lim = prm.wait_cycles / 4;
        for (int s = 0; s < 2; ++s)
          if (issued[s]) mbar_wait(&bars[B_LD0 + s], (issued[s] - 1) & 1, lim);
      }
    }
  } else if (warp == W_MMA) {
    // =========================== MMA issuer =====================================
    if (lane == 0) {
      const uint32_t idUT = idesc_f16(128, 64, true, true);
      const uint32_t ones = smem_u32(smem + OFF_ONES);
      bool issued = false;
      Step st;
      st.item = blockIdx.x;
      if (st.valid(prm)) st.set_item(prm, st.item);
      for (int n = 0; st.valid(prm); ++n, st.next(prm)) {
        const int s = n & 1, nk = nk_of(st.c);
        const bool first = st.c == st.c_hi - 1;   // the segment's summary starts here
        if (!waitb(B_KVR, n & 1)) break;
        if (n >= 1 && !waitb(B_CU, (n - 1) & 1)) break;   // U^B (and at an item's end the summary) read
        tc_fence_after();
        const uint32_t a = smem_u32(Vt(s));
        const uint32_t bb = smem_u32(MASK == MASK_LIT ? Kt(s) : KBt);
        const uint32_t bf = smem_u32(MASK == MASK_LIT ? Kt(s) : KFt);
        const uint64_t da0 = mnmaj(a, 0, ones - a);
        uint64_t da = da0, db = mnmaj(bb, 0, 0);
        for (int k = 0; k < nk; ++k, da += kMnmajOnesStep, db += kMnmajStep)
          mma_bf16(tbase + T_U, da, db, idUT, k > 0 ? 1u : 0u);
        if (prm.nseg > 1) {   // the forward summary only feeds the segment chaining
          da = da0;
          db = mnmaj(bf, 0, 0);
          for (int k = 0; k < nk; ++k, da += kMnmajOnesStep, db += kMnmajStep)
            mma_bf16(tbase + T_FA, da, db, idUT, (k > 0 || !first) ? 1u : 0u);
        }
        mma_commit(&bars[B_U]);
        mma_commit(&bars[B_KWE]);
        mma_commit(&bars[B_KVE0 + s]);
        issued = true;
      }
      if (*s_abort && issued) {
        mma_commit(&bars[B_DRAIN]);
        mbar_wait(&bars[B_DRAIN], 0, prm.wait_cycles / 4);
      }
    }
  } else if (warp < W_EPI) {
    // =========================== prep: four threads per token ====================
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
    float D = 0.f;   // sum of l over the item's chunks right of this one
    for (int n = 0; st.valid(prm); ++n) {
      const int s = n & 1, tok = kC * st.c + t;
      float ell[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) ell[r] = ell_next[r];
      const float lnext = lnext_next;
      if (st.c == st.c_hi - 1) D = 0.f;
      // ---- chunk-local inclusive prefix
      float p, T, pfirst;
      chunk_prefix_warp(ell, t, &p, &T, &pfirst);
      {
        // the next step's decays, loaded a whole step ahead of their use
        Step nx = st;
        nx.next(prm);
        if (nx.valid(prm)) load_ell(nx, ell_next, &lnext_next);
      }
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
      // ---- phi(k); the weighted copies once the previous chunk's MMAs read them
      //      (every mask waits, so that prep never runs two chunks ahead of the
      //      MMA issuer's wait on its arrival)
      float kv[16];
      if (good && live) {
        const uint8_t* kt = Kt(s);
#pragma unroll
        for (int j = 0; j < 2; ++j)
          unpack8_bf(*reinterpret_cast<const uint4*>(kt + sw128_offset(t, j0 + j)), kv + 8 * j);
        phi_part<PHI, 16, 4>(kv, peers);
      }
      if (n >= 1 && !waitb(B_KWE, (n - 1) & 1)) good = false;
      good = __all_sync(0xffffffffu, good);
      if (good) {
        if (MASK == MASK_LIT) {
          // rows past the sequence keep the zeros the copy engine filled in
          if (live) {
            uint8_t* kt = Kt(s);
#pragma unroll
            for (int j = 0; j < 2; ++j) *reinterpret_cast<uint4*>(kt + sw128_offset(t, j0 + j)) = pack8_h(kv + 8 * j);
          }
        } else {
          const float wb = live ? ex2((p - pfirst) * kLog2e) : 0.f;
          const float2 wb2 = make_float2(wb, wb);
          // the forward-summary copy only feeds the segment chaining
          const bool fsum = prm.nseg > 1;
          const float wf = live && fsum ? ex2((D + T - p) * kLog2e) : 0.f;
          const float2 wf2 = make_float2(wf, wf);
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            float yb[8], yf[8];
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
              const float2 k2 = live ? make_float2(kv[8 * j + e], kv[8 * j + e + 1]) : make_float2(0.f, 0.f);
              const float2 ub = mul2(k2, wb2);
              yb[e] = ub.x;
              yb[e + 1] = ub.y;
              if (fsum) {
                const float2 uf = mul2(k2, wf2);
                yf[e] = uf.x;
                yf[e + 1] = uf.y;
              }
            }
            *reinterpret_cast<uint4*>(KBt + sw128_offset(t, j0 + j)) = pack8_h(yb);
            if (fsum) *reinterpret_cast<uint4*>(KFt + sw128_offset(t, j0 + j)) = pack8_h(yf);
          }
        }
        if (pt == 0) {
          float* in = info(s);
          in[I_T] = T;
          in[I_DEC] = MASK == MASK_LIT ? 1.f : __expf(T - pfirst + lnext);
        }
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_KVR]);
      D += T;
      st.next(prm);
    }
  } else {
    // =========================== epi: two warps per TMEM lane quarter =============
    const int ew = warp - W_EPI;
    const int q = warp & 3;                  // TMEM lane quarter: lanes 32q..32q+31
    const int hc = ew >> 2;                  // half of the state columns m
    const int i = 32 * q + lane;             // TMEM lane = state column n (64: z)
    const uint32_t lane_off = (uint32_t)(32 * q) << 16;
    bool good = true;
    Step st;
    st.item = blockIdx.x;
    if (st.valid(prm)) st.set_item(prm, st.item);
    float tsum = 0.f;
    for (int n = 0; st.valid(prm); ++n) {
      const int s = n & 1, c = st.c, bh = st.bh;
      const bool first = c == st.c_hi - 1, last = c == st.c_lo;
      if (first) tsum = 0.f;
      // ---- the state entering this chunk from the right, out as its fp16 tile
      //      (16 columns m at a time)
      if (q < 3) {
        uint8_t* row = prm.gst + ((size_t)bh * nch + c) * kGstBytes + (size_t)i * 128;
#pragma unroll 1
        for (int h2 = 0; h2 < 2; ++h2) {
          float g[16];
          if (first) {
#pragma unroll
            for (int e = 0; e < 16; ++e) g[e] = 0.f;
          } else {
            tmem_ld16(tbase + lane_off + T_G + 32 * hc + 16 * h2, g);
            tmem_wait_ld();
            reg_fence16(g);
          }
          if (i < 65) {
#pragma unroll
            for (int j = 0; j < 2; ++j)
              *reinterpret_cast<uint4*>(row + (((4 * hc + 2 * h2 + j) ^ (i & 7)) << 4)) = pack8_h(g + 8 * j);
          }
        }
      }
      // ---- G <- exp(P_{s_{c+1}} - P_{s_c}) G + U^B_c (the U commit also means
      //      prep's scalars of this chunk are written)
      if (!waitb(B_U, n & 1)) good = false;
      good = __all_sync(0xffffffffu, good);
      tc_fence_after();
      tsum += good ? info(s)[I_T] : 0.f;
      if (good && q < 3) {
        const float dec = info(s)[I_DEC];
        float* ss = prm.segsum + (size_t)st.item * kSegSumFloats;   // [64 m][80] summaries
#pragma unroll 1
        for (int h2 = 0; h2 < 2; ++h2) {
          const int m0 = 32 * hc + 16 * h2;
          float g[16], u[16];
          tmem_ld16(tbase + lane_off + T_U + m0, u);
          if (!first) tmem_ld16(tbase + lane_off + T_G + m0, g);
          tmem_wait_ld();
          reg_fence16(u);
          if (first) {
#pragma unroll
            for (int e = 0; e < 16; ++e) g[e] = u[e];
          } else {
            reg_fence16(g);
#pragma unroll
            for (int e = 0; e < 16; ++e) g[e] = fmaf(dec, g[e], u[e]);
          }
          tmem_st16(tbase + lane_off + T_G + m0, g);
          if (last && prm.nseg > 1 && i < kLongStateCols) {
            // column i of the backward summary is this lane's G (anchored at the
            // segment's first token), of the forward one its forward sum
            // (anchored at the segment's last token)
#pragma unroll
            for (int e = 0; e < 16; ++e) ss[64 * kLongStateCols + (m0 + e) * kLongStateCols + i] = g[e];
          }
          if (last && prm.nseg > 1) {
            tmem_ld16(tbase + lane_off + T_FA + m0, u);
            tmem_wait_ld();
            reg_fence16(u);
            if (i < kLongStateCols) {
#pragma unroll
              for (int e = 0; e < 16; ++e) ss[(m0 + e) * kLongStateCols + i] = u[e];
            }
          }
        }
        if (last && prm.nseg > 1 && i == 0 && hc == 0) ss[2 * 64 * kLongStateCols] = tsum;
        tmem_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_CU]);
      // leave together
      if (!bar_and(2, kEpiWarps * 32, good)) break;
      st.next(prm);
    }
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

cudaError_t launch_chunk128_pre(const Problem& p, const LongPlan& plan, uint8_t* gst, float* segsum, int* status,
                                cudaStream_t s) {
  CUtensorMap mk, mv;
  const int BH = p.B * p.H;
  if (!make_map128(&mk, p.k, p.L, BH) || !make_map128(&mv, p.v, p.L, BH)) return cudaErrorInvalidValue;
  PreParams prm;
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
  void (*kern)(const CUtensorMap, const CUtensorMap, PreParams) = nullptr;
#define LION_C128P_CASE(M, F) \
  if (p.mask_kind == M && p.phi == F) kern = lion_chunk128_pre_kernel<M, F>;
  LION_C128P_CASE(MASK_LIT, PHI_ELU1)
  LION_C128P_CASE(MASK_LIT, PHI_SILU_L2)
  LION_C128P_CASE(MASK_LIT, PHI_IDENTITY)
  LION_C128P_CASE(MASK_D, PHI_ELU1)
  LION_C128P_CASE(MASK_D, PHI_SILU_L2)
  LION_C128P_CASE(MASK_D, PHI_IDENTITY)
  LION_C128P_CASE(MASK_S, PHI_ELU1)
  LION_C128P_CASE(MASK_S, PHI_SILU_L2)
  LION_C128P_CASE(MASK_S, PHI_IDENTITY)
#undef LION_C128P_CASE
  if (!kern) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const int items = BH * plan.nseg;
  const int grid = items < sm_count() ? items : sm_count();
  kern<<<grid, kThreads, kSmemBytes, s>>>(mk, mv, prm);
  return cudaGetLastError();
}

}  // namespace lion
