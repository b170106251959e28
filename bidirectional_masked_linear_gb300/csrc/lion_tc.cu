// lion_tc.cu -- chunkwise LION forward on the 5th-generation tensor cores
// (tcgen05 + TMEM + TMA), bfloat16 inputs, head dim 64, chunk 64, any L.
//
// Chunkwise form ("LION Part IV - Results", "LION Chunk"; rebuttal page
// "LION: A bidirectional framework ...", reply "4: Practicality of Recurrent
// Inference" -- chunking).  Per head, chunk c covers tokens [s_c, e_c]; p is
// the chunk-local inclusive prefix of l = log(lambda):
//
//   intra     num_i += sum_{j in c} M_ij s_ij [v_j; 1],  M_ij = exp(p_max - p_min)
//   states    U^F_c = sum_j exp(p_e - p_j) phi(k_j) [v_j; 1]^T
//             U^B_c = sum_j exp(p_j - p_s) phi(k_j) [v_j; 1]^T
//   scans     F_{c+1} = exp(T_c) F_c + U^F_c            (F_c anchored at e_{c-1})
//             G_{c-1} = exp(P_{s_{c+1}} - P_{s_c}) G_c + U^B_c   (G_c at s_{c+1})
//   apply     num_i += a_i phi(q_i) [F_c z^F_c] + b_i phi(q_i) [G_c z^G_c]
//             a_i = exp(P_i - P_{e_{c-1}}),  b_i = exp(P_{s_{c+1}} - P_i)
//   y_i = num_i[0:d] / num_i[d]
//
// The same recurrences chain 256-token blocks (four chunks) and segments of
// blocks: the state leaving one block is the state entering the next.
//
// Normalisers ride on the tensor cores: products with V use B = [V_c | 1]
// (N = 80; a constant tile whose first column is 1 is the second atom), so
// U carries z as its column 64 and A V carries the intra-chunk row sum; the
// scanned z vectors sit in one small operand tile.
//
// Precision: MMA operands are fp16 (11-bit significand) with fp32
// accumulation; phi(K), the decay-weighted phi(K), phi(Q), the chunk states,
// z, V and the masked scores are each rounded once to fp16, and so are the
// block boundary states exchanged through global memory for long sequences.
// (One bf16 rounding of the unit-norm SiLU features costs ~5e-3 relative
// error; fp16 stays within about half of the 2e-3 budget.)  Precondition:
// |phi(q)|, |phi(k)|, |v| and the chunk states below the fp16 range (65504);
// a v past it, or a non-finite row sum, is reported in `status` as
// kStatusRange.
//
// Work split.  Persistent CTAs (one per SM) walk work items.  An item is a
// segment of one head: up to SEGB consecutive 256-token blocks.  Warp 16
// issues TMA and tcgen05 MMAs; warps 0-15 do the CUDA-core stages and hand
// tiles to it through mbarriers.  Per block:
//   A  per chunk: phi(K_c) -> fp16 in place, V_c -> fp16 in place, the
//      decay-weighted copies Kf_c, Kb_c; one M=128 MMA per chunk computes
//      U^F_c (TMEM lanes 0-63) and U^B_c (lanes 64-127):
//      A = [Kf_c ; Kb_c]^T (MN-major, two atoms), B = [V_c | 1] (MN-major).
//   B  scans over chunks (lanes 0-63 forward, 64-127 backward), starting
//      from the states entering the block, writing fp16 operand tiles.
//   C  (main pass only) a two-deep pipeline over chunks:
//      S = phi(Q_c) phi(K_c)^T, O_F = phi(Q_c) F_c, O_G = phi(Q_c) G_c,
//      Z = phi(Q_c) [z tiles] (M=64 MMAs) overlap the previous chunk's
//      epilogue; the decay mask is applied to S on the CUDA cores
//      (factorised as exp(p_i - p_0) exp(p_0 - p_j) when the chunk's decay
//      range allows); O_I = A [V_c | 1]; the epilogue combines, normalises
//      and stores fp32.  Retired K/V tiles are refilled with the next
//      block's chunks; Q streams through a four-slot ring.
// Sequences longer than one block take three launches:
//   pre-pass  blocks of each segment right to left (phases A and B only):
//             writes the backward state entering each block from the right
//             within its segment, and the segment's two summary states;
//   scan      a small CUDA-core kernel chains the segment summaries into the
//             states entering each segment;
//   main      blocks left to right, the forward state carried in registers,
//             the backward state entering each block rebuilt from the
//             pre-pass state plus the decayed segment-level state.
//
// Every mbarrier wait is bounded; on timeout the kernel records an error in
// `status`, releases its TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "lion_common.cuh"
#include "lion_internal.h"
#include "tc_ptx.cuh"

namespace lion {
namespace {

using namespace tc;

constexpr int kC = 64;            // chunk length
constexpr int kD = 64;            // head dim
constexpr int kMaxChunks = 4;     // chunks per block
constexpr int kBlock = kC * kMaxChunks;   // 256 tokens
constexpr int kWorkerWarps = 16;  // CUDA-core stages
constexpr int kThreads = (kWorkerWarps + 1) * 32;  // + one TMA/MMA issuer warp
constexpr int kTile = kC * 128;   // bytes of one 64-row x 64-element 16-bit swizzled tile
constexpr int kQSlots = 4;
constexpr uint32_t kSleepNs = 20000u;            // longest sleep inside one try_wait
constexpr float kMaxFactorRange = 80.f;          // exp(80) stays finite in fp32
constexpr int kStateCols = 80;                   // global state rows: 64 values, z, padding

enum { MODE_MAIN = 0, MODE_PRE = 1 };

// shared-memory map (bytes from a 1024-aligned base)
constexpr int OFF_K = 0;                               // phi(K) tiles, one per chunk
constexpr int OFF_V = OFF_K + kMaxChunks * kTile;      // V tiles
constexpr int OFF_ONES = OFF_V + kMaxChunks * kTile;   // column 0 = 1: the normaliser atom
constexpr int OFF_WORK = OFF_ONES + kTile;             // A: Kf/Kb tiles; B/C: F, G tiles + z
constexpr int OFF_A = OFF_WORK + (2 * kMaxChunks + 1) * kTile;  // masked scores, 2 buffers
constexpr int OFF_Q = OFF_A + 2 * kTile;               // Q ring
constexpr int OFF_P = OFF_Q + kQSlots * kTile;         // float[256] chunk-local prefix
constexpr int OFF_E = OFF_P + kBlock * 4;              // float[3][2][64] mask factors, by chunk % 3
constexpr int OFF_MISC = OFF_E + 3 * 2 * kC * 4;       // float[8]: l at chunk starts
constexpr int OFF_UNI = OFF_MISC + 8 * 4;              // CTA-uniform worker bookkeeping
constexpr int OFF_BAR = OFF_UNI + 16 * 4;
constexpr int OFF_TSLOT = OFF_BAR + 24 * 8;
constexpr int kSmemBytes = OFF_TSLOT + 16 + 1024;      // + alignment slack
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

// work tiles in phases B/C: F_c at c, G_c at 4 + c, the z tile at 8
// (column 2c: z^F_c, column 2c+1: z^G_c)
constexpr int W_F = 0, W_G = 4, W_Z = 8;

// mbarriers: TMA completions (count 1, transaction bytes), tensor-core
// commits (count 1) and worker hand-offs (one arrival per worker warp)
constexpr int BAR_KV = 0;    // + chunk slot: K_c, V_c landed
constexpr int BAR_Q = 4;     // + Q slot: Q chunk landed
constexpr int BAR_RA = 8;    // + chunk slot: phase-A operand tiles written
constexpr int BAR_DA = 12;   // phase-A MMAs done
constexpr int BAR_RB = 13;   // state tiles written
constexpr int BAR_RP = 14;   // + region: phi(Q_c) written
constexpr int BAR_M1 = 16;   // + region: S, O_F, O_G, Z done
constexpr int BAR_RE = 18;   // + region: masked scores written
constexpr int BAR_M2 = 20;   // + region: O_I done
constexpr int BAR_FR = 22;   // + region: chunk retired (TMEM region, K/V tiles free)
constexpr int kNumBars = 24;
__host__ __device__ constexpr uint32_t bar_count(int b) {
  return (b >= BAR_RA && b < BAR_DA) || b == BAR_RB || (b >= BAR_RP && b < BAR_M1) ||
                 (b >= BAR_RE && b < BAR_M2) || b >= BAR_FR
             ? (uint32_t)kWorkerWarps
             : 1u;
}

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSlot = 80;       // phase A/B: chunk-state slot (64 values + z + 15 zero)
constexpr uint32_t kRegion = 216;    // phase C: per in-flight chunk
constexpr uint32_t R_SI = 0, R_OF = 80, R_OG = 144, R_Z = 208;
// state kept across the blocks of a segment (80 columns; lanes 0-63 forward
// direction, 64-127 backward):
//   main: forward state entering the next block / backward state entering the segment
//   pre:  the segment's forward summary / backward state entering the next block
constexpr uint32_t TM_KEEP = 2 * kRegion;   // 432

// long-sequence exchange buffers (global, per block / per segment): the
// backward state entering each block, fp16 [64 m][64 n] then fp32 z[64];
// segment summaries and entering states as declared in lion_internal.h
constexpr int kGlocBytes = kD * kD * 2 + kD * 4;
static_assert(kLongStateCols == kStateCols && kSegSumFloats == 2 * kD * kStateCols + 4 &&
                  kSegInFloats == 2 * kD * kStateCols,
              "exchange-buffer layout");

struct TcParams {
  float* out;
  const float* log_lambda;
  int BH, H, L;
  int NBL;        // 256-token blocks per head
  int SEGB;       // blocks per segment
  int nseg;       // segments per head
  uint8_t* gloc;       // [BH][NBL] backward state entering each block (within its segment)
  float* segsum;       // [BH][nseg] segment summaries (pre-pass output)
  const float* segin;  // [BH][nseg] states entering each segment (scan output)
  int* status;
  long long wait_cycles;   // bound of every mbarrier wait, in clock cycles
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

// Raises `flag` (the CTA's range flag in shared memory) when one of n fp32
// values about to become an fp16 operand lies past the fp16 range (65504).
template <int N>
__device__ __forceinline__ void check_f16(const float* x, volatile int* flag) {
  float m = 0.f;
#pragma unroll
  for (int e = 0; e < N; ++e) m = fmaxf(m, fabsf(x[e]));
  if (!(m <= 65504.f)) *flag = 1;
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

__device__ __forceinline__ int nchunks_of(int L, int b) {
  return min(kMaxChunks, (L - b * kBlock + kC - 1) / kC);
}

// Walks this CTA's blocks in processing order: items (segments of heads)
// blockIdx.x, + gridDim.x, ...; blocks of a segment left to right (main) or
// right to left (pre-pass).
struct BlockCursor {
  int item, b;
  __device__ void first_of_item(const TcParams& p, int mode) {
    const int seg = item % p.nseg;
    b = mode == MODE_MAIN ? seg * p.SEGB : min(p.NBL, (seg + 1) * p.SEGB) - 1;
  }
  __device__ void begin(const TcParams& p, int mode) {
    item = blockIdx.x;
    if (item < p.BH * p.nseg) first_of_item(p, mode);
  }
  __device__ bool valid(const TcParams& p) const { return item < p.BH * p.nseg; }
  __device__ void next(const TcParams& p, int mode) {
    const int seg = item % p.nseg;
    const int lo = seg * p.SEGB, hi = min(p.NBL, (seg + 1) * p.SEGB) - 1;
    if (mode == MODE_MAIN ? b < hi : b > lo) {
      b += mode == MODE_MAIN ? 1 : -1;
    } else {
      item += gridDim.x;
      if (valid(p)) first_of_item(p, mode);
    }
  }
};

template <int MASK>
__device__ __forceinline__ float ell_at(const TcParams& p, int bh, int t, float lh) {
  if (t >= p.L) return 0.f;
  if (MASK == MASK_S) return p.log_lambda[(size_t)bh * p.L + t];
  if (MASK == MASK_D) return lh;
  return 0.f;
}

template <int MASK, int PHI, int MODE>
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
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + OFF_TSLOT + 8);
  volatile int* s_range = reinterpret_cast<volatile int*>(smem + OFF_TSLOT + 12);
  auto Kt = [&](int c) { return smem + OFF_K + c * kTile; };
  auto Vt = [&](int c) { return smem + OFF_V + c * kTile; };
  auto Wt = [&](int i) { return sWork + i * kTile; };
  auto At = [&](int r) { return smem + OFF_A + r * kTile; };
  auto Qt = [&](int slot) { return smem + OFF_Q + slot * kTile; };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int L = prm.L;
  const int quarter = warp & 3, wg = (warp >> 2) & 3;   // TMEM lane quarter, column group

  if (tid == 0) {
    prefetch_tmap(&mapK);
    prefetch_tmap(&mapV);
    if (MODE == MODE_MAIN) prefetch_tmap(&mapQ);
    for (int b = 0; b < kNumBars; ++b) mbar_init(&bars[b], bar_count(b));
    *s_abort = 0;
    *s_range = 0;
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

  // bounded wait on a barrier phase; any timeout makes every later wait return at once
  auto waitb = [&](int b, uint32_t parity) -> bool {
    return mbar_wait_or_abort(&bars[b], parity, prm.wait_cycles, kSleepNs, s_abort);
  };

  if (warp == kWorkerWarps) {
    // =================== issuer warp: TMA and MMA =============================
    if (lane == 0) {
      int kvn[kMaxChunks] = {0, 0, 0, 0};   // loads issued per K/V slot
      int ran[kMaxChunks] = {0, 0, 0, 0};   // phase-A hand-offs consumed per slot
      auto issue_kv = [&](const BlockCursor& cur, int c) {
        const int bh_ = cur.item / prm.nseg;
        mbar_arrive_expect_tx(&bars[BAR_KV + c], (uint32_t)(2 * kTile));
        tma_load_3d(Kt(c), &mapK, &bars[BAR_KV + c], 0, cur.b * kBlock + c * kC, bh_);
        tma_load_3d(Vt(c), &mapV, &bars[BAR_KV + c], 0, cur.b * kBlock + c * kC, bh_);
        ++kvn[c];
      };
      // Q ring: a second cursor runs kQSlots chunks ahead of consumption
      BlockCursor qcur;
      qcur.begin(prm, MODE);
      int qc = 0, qg = 0;
      auto issue_q_next = [&]() {
        if (!qcur.valid(prm)) return;
        const int sl = qg % kQSlots;
        mbar_arrive_expect_tx(&bars[BAR_Q + sl], (uint32_t)kTile);
        tma_load_3d(Qt(sl), &mapQ, &bars[BAR_Q + sl], 0, qcur.b * kBlock + qc * kC, qcur.item / prm.nseg);
        ++qg;
        if (++qc == nchunks_of(L, qcur.b)) {
          qc = 0;
          qcur.next(prm, MODE);
        }
      };
      const uint32_t idA = idesc_f16(128, 80, true, true);
      const uint32_t idS = idesc_f16(64, 64, false, false);
      const uint32_t idO = idesc_f16(64, 64, false, true);
      const uint32_t idI = idesc_f16(64, 80, false, true);
      const uint32_t idZ = idesc_f16(64, 8, false, true);
      auto mma1 = [&](int c, int g, bool hasF, bool hasG) {
        const int rg = g & 1, sl = g % kQSlots;
        const uint32_t base = tbase + kRegion * rg;
        const uint8_t* qt = Qt(sl);
#pragma unroll
        for (int k = 0; k < 4; ++k) mma_bf16(base + R_SI, kmaj(qt, k), kmaj(Kt(c), k), idS, k > 0 ? 1u : 0u);
        if (hasF) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_bf16(base + R_OF, kmaj(qt, k), mnmaj(Wt(W_F + c), k, kTile), idO, k > 0 ? 1u : 0u);
        }
        if (hasG) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_bf16(base + R_OG, kmaj(qt, k), mnmaj(Wt(W_G + c), k, kTile), idO, k > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) mma_bf16(base + R_Z, kmaj(qt, k), mnmaj(Wt(W_Z), k, kTile), idZ, k > 0 ? 1u : 0u);
        mma_commit(&bars[BAR_M1 + rg]);
      };
      auto mma2 = [&](int c, int g) {
        const int rg = g & 1;
        const uint32_t base = tbase + kRegion * rg;
        const uint32_t lbo_v = (uint32_t)(sOnes - Vt(c));
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_bf16(base + R_SI, kmaj(At(rg), k), mnmaj(Vt(c), k, lbo_v), idI, k > 0 ? 1u : 0u);
        mma_commit(&bars[BAR_M2 + rg]);
      };

      BlockCursor cur;
      cur.begin(prm, MODE);
      if (cur.valid(prm))
        for (int c = 0; c < nchunks_of(L, cur.b); ++c) issue_kv(cur, c);
      if (MODE == MODE_MAIN)
        for (int i = 0; i < kQSlots; ++i) issue_q_next();
      int g = 0, nb = 0;   // chunks through phase C, blocks done
      bool good = true;
      while (cur.valid(prm) && good) {
        const int NC = nchunks_of(L, cur.b);
        BlockCursor nxt = cur;
        nxt.next(prm, MODE);
        const bool has_next = nxt.valid(prm);
        const int NCn = has_next ? nchunks_of(L, nxt.b) : 0;
        // K/V slots this block does not use are free now: start the next block's loads
        if (has_next)
          for (int c = NC; c < NCn; ++c) issue_kv(nxt, c);
        // phase A: one stacked MMA per chunk as soon as its tiles are ready
        for (int c = 0; c < NC && good; ++c) {
          good = waitb(BAR_RA + c, ran[c] & 1);
          ++ran[c];
          if (!good) break;
          tc_fence_after();
          const uint32_t lbo_v = (uint32_t)(sOnes - Vt(c));
          // LIT: both directions weigh every token by 1, so the stacked A is
          // phi(K_c) twice (second atom at offset 0)
          const uint8_t* a_tile = MASK == MASK_LIT ? Kt(c) : Wt(2 * c);
          const uint32_t lbo_a = MASK == MASK_LIT ? 0u : (uint32_t)kTile;
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_bf16(tbase + kSlot * c, mnmaj(a_tile, k, lbo_a), mnmaj(Vt(c), k, lbo_v), idA, k > 0 ? 1u : 0u);
        }
        if (!good) break;
        mma_commit(&bars[BAR_DA]);
        if (MODE == MODE_PRE) {
          // the K/V tiles are free once the phase-A MMAs have read them
          good = waitb(BAR_DA, nb & 1);
          if (!good) break;
          if (has_next)
            for (int c = 0; c < min(NC, NCn); ++c) issue_kv(nxt, c);
        } else {
          const bool hasFin = cur.b > 0, hasGin = cur.b < prm.NBL - 1;
          good = waitb(BAR_RB, nb & 1);
          if (!good) break;
          tc_fence_after();
          // phase C, in the order the workers produce their hand-offs
          auto hf = [&](int c) { return c > 0 || hasFin; };
          auto hg = [&](int c) { return c < NC - 1 || hasGin; };
          good = waitb(BAR_RP + (g & 1), (g >> 1) & 1);
          if (!good) break;
          tc_fence_after();
          mma1(0, g, hf(0), hg(0));
          if (NC > 1) {
            good = waitb(BAR_RP + ((g + 1) & 1), ((g + 1) >> 1) & 1);
            if (!good) break;
            tc_fence_after();
            mma1(1, g + 1, hf(1), hg(1));
          }
          good = waitb(BAR_RE + (g & 1), (g >> 1) & 1);
          if (!good) break;
          tc_fence_after();
          mma2(0, g);
          issue_q_next();
          for (int c = 1; c < NC && good; ++c) {
            const int gc = g + c;
            // chunk c-1 retired: its TMEM region takes chunk c+1's first MMA group
            good = waitb(BAR_FR + ((gc - 1) & 1), ((gc - 1) >> 1) & 1);
            if (!good) break;
            if (c - 1 < NCn) issue_kv(nxt, c - 1);
            if (c + 1 < NC) {
              good = waitb(BAR_RP + ((gc + 1) & 1), ((gc + 1) >> 1) & 1);
              if (!good) break;
              tc_fence_after();
              mma1(c + 1, gc + 1, hf(c + 1), hg(c + 1));
            }
            good = waitb(BAR_RE + (gc & 1), (gc >> 1) & 1);
            if (!good) break;
            tc_fence_after();
            mma2(c, gc);
            issue_q_next();
          }
          if (!good) break;
          good = waitb(BAR_FR + ((g + NC - 1) & 1), ((g + NC - 1) >> 1) & 1);
          if (!good) break;
          if (NC - 1 < NCn) issue_kv(nxt, NC - 1);
          g += NC;
        }
        ++nb;
        cur = nxt;
      }
    }
  } else {
    // =================== worker warps: CUDA-core stages =======================
    // (the main pass of a long sequence reads the pre-pass's and the scan's
    // output: it may have been launched before they ended)
    if (MODE == MODE_MAIN) pdl_wait();
    auto arrive = [&](int b) {   // every worker warp arrives once
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[b]);
    };
    auto worker_sync = [&]() { asm volatile("bar.sync 1, %0;" ::"n"(kWorkerWarps * 32) : "memory"); };
    // row-parallel stages: thread -> (row tid / 8, 16-byte column chunk tid % 8)
    const uint32_t off_rc = sw128_offset(tid >> 3, tid & 7);
    // CTA-uniform bookkeeping lives in shared memory (register budget):
    // [0..3] K/V loads consumed per slot, [4] rsum, [5] tseg, [6] lseg_after, [7] tcum
    int* uni_i = reinterpret_cast<int*>(smem + OFF_UNI);
    float* uni_f = reinterpret_cast<float*>(smem + OFF_UNI);
    if (tid < 8) uni_i[tid] = 0;
    worker_sync();
    bool good = true;
    int g = 0, nb = 0;
    // phase-B thread role: state row m of the forward (quarters 0-1) or
    // backward (2-3) direction, columns 16*wg.. (+ the z column for wg 3)
    const bool fwd = quarter < 2;
    const int m = 32 * (quarter & 1) + lane;
    // the kept state (TM_KEEP) of this thread's row and columns
    const uint32_t keep_addr = lane_addr(tbase, warp, TM_KEEP + 16 * wg);
    const uint32_t keepz_addr = lane_addr(tbase, warp, TM_KEEP + 64);
    auto keep_load = [&](float* v, float* vz) {
      tmem_ld16(keep_addr, v);
      float zz[16];
      if (wg == 3) tmem_ld16(keepz_addr, zz);
      tmem_wait_ld();
      *vz = wg == 3 ? zz[0] : 0.f;
    };
    auto keep_store = [&](const float* v, float vz) {
      tmem_st16(keep_addr, v);
      if (wg == 3) {
        float zz[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) zz[e] = 0.f;
        zz[0] = vz;
        tmem_st16(keepz_addr, zz);
      }
      tmem_wait_st();
    };
    BlockCursor cur;
    cur.begin(prm, MODE);
    int item_prev = -1;
    while (cur.valid(prm) && good) {
      const int bh = cur.item / prm.nseg, seg = cur.item % prm.nseg, b = cur.b;
      const int h = bh % prm.H;
      const float lh = MASK == MASK_D ? prm.log_lambda[h] : 0.f;
      const int NC = nchunks_of(L, b);
      const int bs = b * kBlock;
      const bool hasFin = b > 0, hasGin = b < prm.NBL - 1;
      const bool new_item = cur.item != item_prev;
      item_prev = cur.item;
      if (new_item) {
        // per-segment starting states (long sequences only)
        const size_t so = (size_t)cur.item;
        float kv[16], kz = 0.f;
#pragma unroll
        for (int e = 0; e < 16; ++e) kv[e] = 0.f;
        float tseg = 0.f, lseg_after = 0.f;
        // (one segment a head: zero entering states, no scan output to read)
        if (MODE == MODE_MAIN && prm.NBL > 1 && prm.nseg > 1) {
          const float* sin = prm.segin + so * kSegInFloats;
          const float* src = sin + (fwd ? 0 : kD * kStateCols) + m * kStateCols;
#pragma unroll
          for (int e = 0; e < 16; ++e) kv[e] = src[16 * wg + e];
          if (wg == 3) kz = src[64];
          tseg = prm.segsum[so * kSegSumFloats + 2 * kD * kStateCols];
          lseg_after = ell_at<MASK>(prm, bh, min(prm.NBL, (seg + 1) * prm.SEGB) * kBlock, lh);
        }
        keep_store(kv, kz);
        worker_sync();   // every worker has read the previous item's bookkeeping
        if (tid == 0) {
          uni_f[4] = 0.f;
          uni_f[5] = tseg;
          uni_f[6] = lseg_after;
          uni_f[7] = 0.f;
        }
      }
      // chunk-local inclusive prefixes (one warp per chunk, 2 tokens per lane)
      if (warp < NC) {
        const int c = warp, s = bs + c * kC;
        const int t0 = s + 2 * lane, t1 = t0 + 1;
        const float l0 = ell_at<MASK>(prm, bh, t0, lh), l1 = ell_at<MASK>(prm, bh, t1, lh);
        const float pair = l0 + l1;
        float x = pair;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, x, o);
          if (lane >= o) x += y;
        }
        const float excl = x - pair;
        sP[c * kC + 2 * lane] = excl + l0;
        sP[c * kC + 2 * lane + 1] = excl + l0 + l1;
        if (lane == 0) sMisc[c] = l0;   // l at s_c
      }
      if (tid == 0) sMisc[NC] = ell_at<MASK>(prm, bh, bs + NC * kC, lh);   // l after the block
      worker_sync();
      float tblk = 0.f;   // sum of l over the block
      for (int c = 0; c < NC; ++c) tblk += sP[c * kC + min(kC, L - bs - c * kC) - 1];

      // ---------------- phase A: phi(K), V, decay-weighted copies ---------
      for (int c = 0; c < NC; ++c) {
        good = waitb(BAR_KV + c, uni_i[c] & 1);
        if (!good) break;
        const int len = min(kC, L - bs - c * kC);
        const int r = tid >> 3;
        uint8_t* kp = Kt(c) + off_rc;
        uint8_t* vp = Vt(c) + off_rc;
        uint8_t* fp = Wt(2 * c) + off_rc;
        uint8_t* bp = Wt(2 * c + 1) + off_rc;
        if (4 * warp < len) {   // rows of this warp that hold tokens (the rest arrive as zeros)
          float x[8];
          unpack8_bf(*reinterpret_cast<const uint4*>(kp), x);
          phi8<PHI>(x);      // every lane: phi8 shuffles within the row's 8 lanes
          if (r >= len) {    // padding tokens contribute nothing
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = 0.f;
          }
          const uint4 kh = pack8_h(x);
          *reinterpret_cast<uint4*>(kp) = kh;
          if (MASK != MASK_LIT) {
            unpack8_h(kh, x);  // the decay weights multiply the fp16 phi(k) that S sees
            const float pj = sP[c * kC + r];
            const float wf = r < len ? __expf(sP[c * kC + len - 1] - pj) : 0.f;
            const float wb = r < len ? __expf(pj - sP[c * kC]) : 0.f;
            float y[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) y[e] = wf * x[e];
            *reinterpret_cast<uint4*>(fp) = pack8_h(y);
#pragma unroll
            for (int e = 0; e < 8; ++e) y[e] = wb * x[e];
            *reinterpret_cast<uint4*>(bp) = pack8_h(y);
          }
          float v8[8];
          unpack8_bf(*reinterpret_cast<const uint4*>(vp), v8);
          check_f16<8>(v8, s_range);
          *reinterpret_cast<uint4*>(vp) = pack8_h(v8);
        } else if (MASK != MASK_LIT) {
          // K and V rows past the sequence arrived as zeros (bf16 0 == fp16 0);
          // the weighted copies still hold an older block's data
          *reinterpret_cast<uint4*>(fp) = make_uint4(0u, 0u, 0u, 0u);
          *reinterpret_cast<uint4*>(bp) = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_async_smem();
        arrive(BAR_RA + c);
      }
      if (!good) break;

      // ---------------- phase B: scans -> fp16 state operand tiles --------
      good = waitb(BAR_DA, nb & 1);
      if (!good) break;
      tc_fence_after();
      if (MODE == MODE_MAIN && tid < 2 * kC) *chunk16(Wt(W_Z), tid >> 1, tid & 1) = make_uint4(0u, 0u, 0u, 0u);
      worker_sync();   // z tile cleared; every worker has read this block's K/V counters
      if (tid == 0)
        for (int c = 0; c < NC; ++c) ++uni_i[c];
      {
        // the state entering the block from this thread's direction: 16
        // columns (st) plus, for column group 3, the normaliser z (stz)
        float st[16], stz;
        {
          float kv[16], kz;
          keep_load(kv, &kz);
          if (MODE == MODE_MAIN) {
            if (fwd) {
#pragma unroll
              for (int e = 0; e < 16; ++e) st[e] = kv[e];
              stz = kz;
            } else {
#pragma unroll
              for (int e = 0; e < 16; ++e) st[e] = 0.f;
              stz = 0.f;
              if (hasGin) {
                // G entering block b = G_loc(b) + exp(P_{s_seg_end} - P_{s_{b+1}}) G_in(seg)
                const uint8_t* gl = prm.gloc + ((size_t)bh * prm.NBL + b) * kGlocBytes;
                const __half* gv = reinterpret_cast<const __half*>(gl) + m * kD + 16 * wg;
                const float rb = uni_f[5] - uni_f[7] - tblk;   // sum of l over this segment's blocks after b
                // (one segment a head: no entering state, and rb is not a
                // segment's sum then, so the factor is not evaluated)
                const float f = prm.nseg > 1 ? __expf(rb - sMisc[NC] + uni_f[6]) : 0.f;
#pragma unroll
                for (int e = 0; e < 16; ++e) st[e] = __half2float(gv[e]) + f * kv[e];
                if (wg == 3) stz = reinterpret_cast<const float*>(gl + kD * kD * 2)[m] + f * kz;
              }
            }
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) st[e] = fwd ? 0.f : kv[e];
            stz = fwd ? 0.f : kz;
            if (!fwd) {
              // the pre-pass records the backward state entering block b
              uint8_t* gl = prm.gloc + ((size_t)bh * prm.NBL + b) * kGlocBytes;
              __half* gv = reinterpret_cast<__half*>(gl) + m * kD + 16 * wg;
#pragma unroll
              for (int e = 0; e < 16; e += 2)
                *reinterpret_cast<__half2*>(gv + e) = __floats2half2_rn(st[e], st[e + 1]);
              if (wg == 3) reinterpret_cast<float*>(gl + kD * kD * 2)[m] = stz;
            }
          }
        }
        for (int cc = 0; cc < NC; ++cc) {
          const int c = fwd ? cc : NC - 1 - cc;
          const int len = min(kC, L - bs - c * kC);
          float u[16];
          tmem_ld16(lane_addr(tbase, warp, kSlot * c + 16 * wg), u);
          float uz = 0.f;
          if (wg == 3) uz = tmem_ld1(lane_addr(tbase, warp, kSlot * c + 64));
          if (MODE == MODE_MAIN && (fwd ? (c > 0 || hasFin) : (c < NC - 1 || hasGin))) {
            uint8_t* dst = fwd ? Wt(W_F + c) : Wt(W_G + c);   // state entering chunk c
            *chunk16(dst, m, 2 * wg) = pack8_h(st);
            *chunk16(dst, m, 2 * wg + 1) = pack8_h(st + 8);
            if (wg == 3) *elem16(Wt(W_Z), m, 2 * c + (fwd ? 0 : 1)) = __float2half_rn(stz);
          }
          tmem_wait_ld();
          float decay = 1.f;
          if (MASK != MASK_LIT) {
            const float T = sP[c * kC + len - 1];
            decay = fwd ? __expf(T) : __expf(T - sMisc[c] + sMisc[c + 1]);
          }
#pragma unroll
          for (int e = 0; e < 16; ++e) st[e] = decay * st[e] + u[e];
          stz = decay * stz + uz;
        }
        // states leaving the block
        if (MODE == MODE_MAIN) {
          if (fwd) keep_store(st, stz);
        } else {
          if (fwd) {
            // U^F of the block, decayed to the segment end
            float kv[16], kz;
            keep_load(kv, &kz);
            const float f = __expf(uni_f[4]);
#pragma unroll
            for (int e = 0; e < 16; ++e) kv[e] += f * st[e];
            keep_store(kv, kz + f * stz);
          } else {
            keep_store(st, stz);
          }
        }
      }
      tc_fence_before();
      if (MODE == MODE_PRE) {
        // segment summaries once the leftmost block is done
        const int seg_lo = seg * prm.SEGB;
        if (b == seg_lo && prm.nseg > 1) {
          float* ss = prm.segsum + (size_t)cur.item * kSegSumFloats;
          float* dst = ss + (fwd ? 0 : kD * kStateCols) + m * kStateCols;
          float sv[16], sz;
          keep_load(sv, &sz);
#pragma unroll
          for (int e = 0; e < 16; ++e) dst[16 * wg + e] = sv[e];
          if (wg == 3) {
            dst[64] = sz;
#pragma unroll
            for (int e = 65; e < kStateCols; ++e) dst[e] = 0.f;
          }
          if (tid == 0) ss[2 * kD * kStateCols] = uni_f[4] + tblk;
        }
        // TMEM slots are rewritten by the next block's phase A only after
        // every worker passed this point
        worker_sync();
        if (tid == 0) uni_f[4] += tblk;
      } else {
        fence_async_smem();
        arrive(BAR_RB);

        // ---------------- phase C: two-deep pipeline over chunks ----------
        auto hf = [&](int c) { return c > 0 || hasFin; };
        auto hg = [&](int c) { return c < NC - 1 || hasGin; };
        auto prep = [&](int c, int gg) -> bool {
          const int sl = gg % kQSlots;
          if (!waitb(BAR_Q + sl, (gg / kQSlots) & 1)) return false;
          const int len = min(kC, L - bs - c * kC);
          if (4 * warp < len) {   // padding rows arrive as zeros and stay unused
            uint8_t* qp = Qt(sl) + off_rc;
            float x[8];
            unpack8_bf(*reinterpret_cast<const uint4*>(qp), x);
            phi8<PHI>(x);
            *reinterpret_cast<uint4*>(qp) = pack8_h(x);
          }
          if (MASK != MASK_LIT && tid < 2 * kC) {
            // E[t] = exp(p_t - p_0), Einv[t] = exp(p_0 - p_t)
            const int t = tid & 63;
            const float d = sP[c * kC + t] - sP[c * kC];
            sE[((gg % 3) * 2 + (tid >> 6)) * kC + t] = tid < 64 ? __expf(d) : __expf(-d);
          }
          fence_async_smem();
          arrive(BAR_RP + (gg & 1));
          if (MASK != MASK_LIT) worker_sync();   // mask factors visible to every worker
          return true;
        };
        // Epilogues read the M=64 accumulators with the 16x256b shape: this
        // warp's 16 rows (lane quarter) x its 16 columns, spread over all 32
        // lanes -- thread t: rows i0 = t/4, i1 = t/4 + 8 of the quarter,
        // columns j0, j0 + 1, j0 + 8, j0 + 9 with j0 = 16 wg + 2 (t % 4).
        const int i0 = 16 * quarter + (lane >> 2), i1 = i0 + 8;
        const int jq = 2 * (lane & 3);
        const uint32_t a_off0 = sw128_offset(i0, 2 * wg) + 4 * (lane & 3);
        const uint32_t a_off1 = sw128_offset(i1, 2 * wg) + 4 * (lane & 3);
        const uint32_t a_off2 = sw128_offset(i0, 2 * wg + 1) + 4 * (lane & 3);
        const uint32_t a_off3 = sw128_offset(i1, 2 * wg + 1) + 4 * (lane & 3);
        auto epi1 = [&](int c, int gg) -> bool {
          const int rg = gg & 1;
          if (!waitb(BAR_M1 + rg, (gg >> 1) & 1)) return false;
          tc_fence_after();
          const int len = min(kC, L - bs - c * kC);
          const uint32_t base = tbase + kRegion * rg;
          float w[8];
          tmem_ld_16x256b_x2(lane_addr(base, warp, R_SI + 16 * wg), w);
          tmem_wait_ld();
          const int j0 = 16 * wg + jq;
          // register r: row (r & 2 ? i1 : i0), column j0 + (r & 1) + (r & 4 ? 8 : 0)
          if (i0 < len) {
            if (MASK == MASK_LIT) {
              if (len < kC) {
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                  const int i = (r & 2) ? i1 : i0, j = j0 + (r & 1) + ((r & 4) ? 8 : 0);
                  if (i >= len || j >= len) w[r] = 0.f;
                }
              }
            } else {
              const float* E = sE + ((gg % 3) * 2) * kC;
              const float* Einv = E + kC;
              const bool factor = sP[c * kC] - sP[c * kC + len - 1] < kMaxFactorRange;
              if (factor) {
                const float2 ej0 = *reinterpret_cast<const float2*>(E + j0);
                const float2 ej8 = *reinterpret_cast<const float2*>(E + j0 + 8);
                const float2 nj0 = *reinterpret_cast<const float2*>(Einv + j0);
                const float2 nj8 = *reinterpret_cast<const float2*>(Einv + j0 + 8);
                const float Ej[4] = {ej0.x, ej0.y, ej8.x, ej8.y};
                const float Nj[4] = {nj0.x, nj0.y, nj8.x, nj8.y};
                const float Ei[2] = {E[i0], E[i1]}, Ni[2] = {Einv[i0], Einv[i1]};
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                  const int ri = (r >> 1) & 1, cj = (r & 1) + ((r >> 1) & 2);
                  const int i = ri ? i1 : i0, j = j0 + (r & 1) + ((r & 4) ? 8 : 0);
                  w[r] *= j <= i ? Ei[ri] * Nj[cj] : Ni[ri] * Ej[cj];
                }
              } else {
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                  const int i = (r & 2) ? i1 : i0, j = j0 + (r & 1) + ((r & 4) ? 8 : 0);
                  const float pi = sP[c * kC + i], pj = sP[c * kC + j];
                  w[r] *= __expf(j <= i ? pi - pj : pj - pi);
                }
              }
              if (len < kC) {
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                  const int i = (r & 2) ? i1 : i0, j = j0 + (r & 1) + ((r & 4) ? 8 : 0);
                  if (i >= len || j >= len) w[r] = 0.f;
                }
              }
            }
            uint8_t* at = At(rg);
            *reinterpret_cast<uint32_t*>(at + a_off0) = pack_h2(w[0], w[1]);
            *reinterpret_cast<uint32_t*>(at + a_off1) = pack_h2(w[2], w[3]);
            *reinterpret_cast<uint32_t*>(at + a_off2) = pack_h2(w[4], w[5]);
            *reinterpret_cast<uint32_t*>(at + a_off3) = pack_h2(w[6], w[7]);
          }
          fence_async_smem();
          tc_fence_before();
          arrive(BAR_RE + rg);
          return true;
        };
        auto epi2 = [&](int c, int gg) -> bool {
          const int rg = gg & 1;
          if (!waitb(BAR_M2 + rg, (gg >> 1) & 1)) return false;
          tc_fence_after();
          const int s = c * kC, len = min(kC, L - bs - s);
          const bool hasF = hf(c), hasG = hg(c);
          const uint32_t base = tbase + kRegion * rg;
          float oi[8], of[8], og[8], dd[4], zz[4];
          tmem_ld_16x256b_x2(lane_addr(base, warp, R_SI + 16 * wg), oi);
          tmem_ld_16x256b(lane_addr(base, warp, R_SI + 64), dd);   // column 64: intra row sums
          if (hasF) tmem_ld_16x256b_x2(lane_addr(base, warp, R_OF + 16 * wg), of);
          if (hasG) tmem_ld_16x256b_x2(lane_addr(base, warp, R_OG + 16 * wg), og);
          tmem_ld_16x256b(lane_addr(base, warp, R_Z), zz);          // columns 2c, 2c+1: z terms
          tmem_wait_ld();
          tc_fence_before();
          arrive(BAR_FR + rg);   // this region (and chunk c's K/V tiles) may be reused
          // the row sums of rows i0, i1 sit in the quad's first lane (column 64)
          // and the z terms in the quad lane c (columns 2c, 2c+1)
          const int qbase = lane & ~3;
          float* out_c = prm.out + ((size_t)bh * L + bs + s) * kD + 16 * wg + jq;
          const float dI0 = __shfl_sync(0xffffffffu, dd[0], qbase);
          const float dI1 = __shfl_sync(0xffffffffu, dd[2], qbase);
          const float dF0 = __shfl_sync(0xffffffffu, zz[0], qbase + c);
          const float dG0 = __shfl_sync(0xffffffffu, zz[1], qbase + c);
          const float dF1 = __shfl_sync(0xffffffffu, zz[2], qbase + c);
          const float dG1 = __shfl_sync(0xffffffffu, zz[3], qbase + c);
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const int i = half ? i1 : i0;
            if (i < len) {
              const float pi = sP[s + i];
              float a = 0.f, bb = 0.f;
              if (hasF) a = MASK == MASK_LIT ? 1.f : __expf(pi);
              if (hasG) bb = MASK == MASK_LIT ? 1.f : __expf(sP[s + len - 1] - pi + sMisc[c + 1]);
              float den = half ? dI1 : dI0;
              if (hasF) den += a * (half ? dF1 : dF0);
              if (hasG) den += bb * (half ? dG1 : dG0);
              // a score past the fp16 range (unbounded features) leaves the row
              // sum non-finite: fp16 operands cannot make an fp32 sum overflow
              if (!(fabsf(den) <= 3.0e38f)) *s_range = 1;
              const float inv = 1.f / den;
              float y[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int r = 2 * half + (e & 1) + ((e & 2) ? 4 : 0);
                float acc = oi[r];
                if (hasF) acc += a * of[r];
                if (hasG) acc += bb * og[r];
                y[e] = acc * inv;
              }
              float* orow = out_c + (size_t)i * kD;
              *reinterpret_cast<float2*>(orow) = make_float2(y[0], y[1]);
              *reinterpret_cast<float2*>(orow + 8) = make_float2(y[2], y[3]);
            }
          }
          return true;
        };

        // phi(Q) prep runs two chunks ahead so each MMA group overlaps a full
        // epilogue: prep c+2 | epi2 c-1, epi1 c | ...
        good = prep(0, g);
        if (good && NC > 1) good = prep(1, g + 1);
        if (good) good = epi1(0, g);
        if (good && NC > 2) good = prep(2, g + 2);
        for (int c = 1; c < NC && good; ++c) {
          good = epi2(c - 1, g + c - 1);
          if (good) good = epi1(c, g + c);
          if (good && c + 2 < NC) good = prep(c + 2, g + c + 2);
        }
        if (good) good = epi2(NC - 1, g + NC - 1);
        g += NC;
        // the next block's prefix overwrites sP/sMisc: every worker must be done reading them
        worker_sync();
        if (tid == 0) uni_f[7] += tblk;
      }
      ++nb;
      cur.next(prm, MODE);
    }
  }

  __syncthreads();
  if (tid == 0 && *s_abort) atomicExch(prm.status, kStatusTimeout);
  if (tid == 0 && !*s_abort && *s_range) atomicExch(prm.status, kStatusRange);
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
    tmem_relinquish();
  }
}

// Chains segment summaries into the states entering each segment:
//   F_in(s+1) = exp(T_seg(s)) F_in(s) + U^F_seg(s),            F_in(0) = 0
//   G_in(s-1) = exp(P_{s_seg(s+1)} - P_{s_seg(s)}) G_in(s) + U^B_seg(s), G_in(last) = 0
// One thread per (head, state element, direction); the summaries it reads do
// not depend on the running state, so their loads go out ahead of the chain.
constexpr int kScanThreads = 128;
template <int MASK>
__global__ void __launch_bounds__(kScanThreads) lion_segment_scan_kernel(TcParams prm, float* segin) {
  pdl_wait();   // the summaries come from the pre-pass, the grid before this one
  const int bh = blockIdx.y, h = bh % prm.H;
  const int x = blockIdx.x * kScanThreads + threadIdx.x;     // [0, 2 * kD * kStateCols)
  if (x >= 2 * kD * kStateCols) return;
  const bool fwd = x < kD * kStateCols;
  const int e = fwd ? x : x - kD * kStateCols;
  const float lh = MASK == MASK_D ? prm.log_lambda[h] : 0.f;
  const int segtok = prm.SEGB * kBlock;
  const size_t base = (size_t)bh * prm.nseg;
  float st = 0.f;
  if (fwd) {
#pragma unroll 4
    for (int sg = 0; sg < prm.nseg; ++sg) {
      const float* ss = prm.segsum + (base + sg) * kSegSumFloats;
      const float t = __ldg(ss + 2 * kD * kStateCols), u = __ldg(ss + e);
      segin[(base + sg) * kSegInFloats + e] = st;
      st = __expf(t) * st + u;
    }
  } else {
#pragma unroll 4
    for (int sg = prm.nseg - 1; sg >= 0; --sg) {
      const float* ss = prm.segsum + (base + sg) * kSegSumFloats;
      const float t = __ldg(ss + 2 * kD * kStateCols), u = __ldg(ss + kD * kStateCols + e);
      const float lfirst = ell_at<MASK>(prm, bh, sg * segtok, lh);
      const float lnext = ell_at<MASK>(prm, bh, (sg + 1) * segtok, lh);
      segin[(base + sg) * kSegInFloats + kD * kStateCols + e] = st;
      st = __expf(t - lfirst + lnext) * st + u;
    }
  }
}

__device__ int g_lion_status;

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
  return p.dtype == DT_BF16 && p.d == kD && p.chunk == kC;
}

namespace {

int num_sms() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}

struct TcPlan {
  int NBL, SEGB, nseg;
  size_t gloc_bytes, segsum_bytes, segin_bytes;
};

TcPlan plan_tc(int B, int H, int L) {
  TcPlan t;
  const int BH = B * H;
  t.NBL = (L + kBlock - 1) / kBlock;
  t.nseg = 1;
  if (t.NBL > 1 && BH < num_sms()) t.nseg = min(t.NBL, max(1, num_sms() / BH));
  t.SEGB = (t.NBL + t.nseg - 1) / t.nseg;
  t.nseg = (t.NBL + t.SEGB - 1) / t.SEGB;
  t.gloc_bytes = t.NBL > 1 ? (size_t)BH * t.NBL * kGlocBytes : 0;
  t.segsum_bytes = t.NBL > 1 ? (size_t)BH * t.nseg * kSegSumFloats * 4 : 0;
  t.segin_bytes = t.NBL > 1 ? (size_t)BH * t.nseg * kSegInFloats * 4 : 0;
  return t;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

template <int MODE>
cudaError_t launch_mode(const Problem& p, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                        const TcParams& prm, int grid, cudaStream_t s) {
  void (*kern)(const CUtensorMap, const CUtensorMap, const CUtensorMap, TcParams) = nullptr;
#define LION_TC_CASE(M, F) \
  if (p.mask_kind == M && p.phi == F) kern = lion_chunk64_tc_kernel<M, F, MODE>;
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
  if (MODE == MODE_PRE || prm.NBL == 1) {
    kern<<<grid, kThreads, kSmemBytes, s>>>(mq, mk, mv, prm);
    return cudaGetLastError();
  }
  // the main pass after a pre-pass (and scan): launched as a programmatic
  // dependent, so that its launch and set-up overlap the end of the grid
  // before; its worker warps wait for that grid (pdl_wait) before they read
  // its output
  return launch_dependent(kern, dim3(grid), dim3(kThreads), kSmemBytes, s, mq, mk, mv, prm);
}

}  // namespace

LongPlan long_plan(int B, int H, int L) {
  const TcPlan t = plan_tc(B, H, L);
  LongPlan lp;
  lp.NBL = t.NBL;
  lp.SEGB = t.SEGB;
  lp.nseg = t.nseg;
  return lp;
}

size_t chunk_tc_workspace_bytes(int B, int H, int L) {
  const TcPlan t = plan_tc(B, H, L);
  if (t.NBL == 1) return 0;
  return align256(t.gloc_bytes) + align256(t.segsum_bytes) + align256(t.segin_bytes);
}

int chunk_tc_launches(int B, int H, int L) { return plan_tc(B, H, L).NBL > 1 ? 3 : 1; }

cudaError_t launch_chunk_tc(const Problem& p, void* ws, int* status, cudaStream_t s) {
  CUtensorMap mq, mk, mv;
  const int BH = p.B * p.H;
  if (!make_map(&mq, p.q, p.L, BH) || !make_map(&mk, p.k, p.L, BH) || !make_map(&mv, p.v, p.L, BH))
    return cudaErrorInvalidValue;
  const TcPlan t = plan_tc(p.B, p.H, p.L);
  TcParams prm;
  prm.out = p.out;
  prm.log_lambda = p.log_lambda;
  prm.BH = BH;
  prm.H = p.H;
  prm.L = p.L;
  prm.NBL = t.NBL;
  prm.SEGB = t.SEGB;
  prm.nseg = t.nseg;
  prm.gloc = nullptr;
  prm.segsum = nullptr;
  prm.segin = nullptr;
  prm.status = status;
  prm.wait_cycles = wait_limit_cycles();
  const int items = BH * t.nseg;
  const int grid = items < num_sms() ? items : num_sms();
  if (t.NBL > 1) {
    if (!ws) return cudaErrorInvalidValue;
    uint8_t* w = static_cast<uint8_t*>(ws);
    prm.gloc = w;
    prm.segsum = reinterpret_cast<float*>(w + align256(t.gloc_bytes));
    float* segin = reinterpret_cast<float*>(w + align256(t.gloc_bytes) + align256(t.segsum_bytes));
    prm.segin = segin;
    cudaError_t e = launch_mode<MODE_PRE>(p, mq, mk, mv, prm, grid, s);
    if (e != cudaSuccess) return e;
    const dim3 sgrid((2 * kD * kStateCols + kScanThreads - 1) / kScanThreads, BH);
    // with one segment a head there is nothing to chain
    if (t.nseg > 1) {
      void (*scan)(TcParams, float*) = p.mask_kind == MASK_LIT ? lion_segment_scan_kernel<MASK_LIT>
                                       : p.mask_kind == MASK_D ? lion_segment_scan_kernel<MASK_D>
                                                               : lion_segment_scan_kernel<MASK_S>;
      cudaError_t es = launch_dependent(scan, sgrid, dim3(kScanThreads), 0, s, prm, segin);
      if (es != cudaSuccess) return es;
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return launch_mode<MODE_MAIN>(p, mq, mk, mv, prm, grid, s);
}

}  // namespace lion
