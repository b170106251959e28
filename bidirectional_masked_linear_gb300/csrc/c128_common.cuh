// c128_common.cuh -- pieces shared by the 128-token-chunk tensor-core
// kernels (lion_c128.cu for sequences of at most 256 tokens, lion_c128L.cu
// for longer ones): 16-bit packing, packed fp32 arithmetic, the feature maps
// on a thread's share of a row, the factorised decay mask on a 16-column block
// of S, operand descriptors and tensor maps.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "lion_common.cuh"
#include "tc_ptx.cuh"

namespace lion {
namespace c128 {

using namespace tc;

constexpr int kC = 128;                 // chunk length
constexpr int kD = 64;                  // head dim
constexpr int kTile = kC * 128;         // 128 rows x 64 16-bit values, 128-byte swizzle
constexpr float kMaxFactorRange = 80.f; // exp(80) stays finite in fp32
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ uint32_t pack_h2(float a, float b) { return h2u(__floats2half2_rn(a, b)); }
__device__ __forceinline__ uint4 pack8_h(const float* x) {
  return make_uint4(pack_h2(x[0], x[1]), pack_h2(x[2], x[3]), pack_h2(x[4], x[5]), pack_h2(x[6], x[7]));
}
// 8 fp32 values rounded to nearest even bfloat16, low address first
__device__ __forceinline__ uint32_t pack_bf2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint4 pack8_bf(const float* x) {
  return make_uint4(pack_bf2(x[0], x[1]), pack_bf2(x[2], x[3]), pack_bf2(x[4], x[5]), pack_bf2(x[6], x[7]));
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
constexpr float kF16Max = 65504.f;   // the largest fp16
// The same, raising `flag` (the CTA's range flag in shared memory) when a
// value lies past the fp16 range: it would become an infinity in the tile.
__device__ __forceinline__ uint4 bf8_to_h8_chk(uint4 v, volatile int* flag) {
  float x[8];
  unpack8_bf(v, x);
  float m = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(x[e]));
  if (!(m <= kF16Max)) *flag = 1;
  return pack8_h(x);
}

// packed two-lane fp32 arithmetic (one instruction for both lanes)
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;"
      : "=l"(d)
      : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)));
  return *reinterpret_cast<float2*>(&d);
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;"
      : "=l"(d)
      : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)));
  return *reinterpret_cast<float2*>(&d);
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(d)
      : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)),
        "l"(*reinterpret_cast<uint64_t*>(&c)));
  return *reinterpret_cast<float2*>(&d);
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// phi over the N features of a row held by this thread; `peers` is the
// shuffle mask of the threads holding the rest of the row, `nshare` how many
// of them (SiLU's norm runs over the whole row; lanes of a row are adjacent).
template <int PHI, int N, int NSHARE>
__device__ __forceinline__ void phi_part(float* x, uint32_t peers) {
  if (PHI == PHI_ELU1) {
#pragma unroll
    for (int e = 0; e < N; ++e) x[e] = x[e] > 0.f ? x[e] + 1.f : ex2(x[e] * kLog2e);
  } else if (PHI == PHI_SILU_L2) {
    float2 ss = make_float2(0.f, 0.f);
#pragma unroll
    for (int e = 0; e < N; e += 2) {
      const float2 xx = make_float2(x[e], x[e + 1]);
      const float2 t = mul2(xx, make_float2(-kLog2e, -kLog2e));
      const float2 d = add2(make_float2(ex2(t.x), ex2(t.y)), make_float2(1.f, 1.f));
      const float2 u = mul2(xx, make_float2(rcp(d.x), rcp(d.y)));   // silu; -0 when exp overflows
      ss = fma2(u, u, ss);
      x[e] = u.x;
      x[e + 1] = u.y;
    }
    float s = ss.x + ss.y;
#pragma unroll
    for (int o = 1; o < NSHARE; o <<= 1) s += __shfl_xor_sync(peers, s, o);
    const float inv = rsqrtf(fmaxf(s, 1e-24f));
    const float2 inv2 = make_float2(inv, inv);
#pragma unroll
    for (int e = 0; e < N; e += 2) {
      const float2 u = mul2(make_float2(x[e], x[e + 1]), inv2);
      x[e] = u.x;
      x[e + 1] = u.y;
    }
  }
}

// The inclusive prefix of l over a 128-token chunk, taken by one warp on its
// own: lane w holds l of tokens 4w .. 4w + 3 in e[0..3].  Returns in *p the
// prefix at token t (any token of the chunk), in *T the chunk's sum and in
// *first l at its first token.
__device__ __forceinline__ void chunk_prefix_warp(const float* e, int t, float* p, float* T, float* first) {
  const int lane = threadIdx.x & 31;
  const float a0 = e[0], a1 = a0 + e[1], a2 = a1 + e[2], a3 = a2 + e[3];
  float x = a3;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  float ex = __shfl_up_sync(0xffffffffu, x, 1);
  if (lane == 0) ex = 0.f;
  const int sl = t >> 2, r = t & 3;
  const float v0 = __shfl_sync(0xffffffffu, ex + a0, sl);
  const float v1 = __shfl_sync(0xffffffffu, ex + a1, sl);
  const float v2 = __shfl_sync(0xffffffffu, ex + a2, sl);
  const float v3 = __shfl_sync(0xffffffffu, ex + a3, sl);
  *p = r == 0 ? v0 : r == 1 ? v1 : r == 2 ? v2 : v3;
  *T = __shfl_sync(0xffffffffu, x, 31);
  *first = __shfl_sync(0xffffffffu, e[0], 0);
}

// Orders every later use of v[0..15] after the preceding tcgen05.wait::ld
// (the TMEM load writes its registers asynchronously).
__device__ __forceinline__ void reg_fence16(float* v) {
  asm volatile("" : "+f"(v[0]), "+f"(v[1]), "+f"(v[2]), "+f"(v[3]), "+f"(v[4]), "+f"(v[5]), "+f"(v[6]),
               "+f"(v[7]), "+f"(v[8]), "+f"(v[9]), "+f"(v[10]), "+f"(v[11]), "+f"(v[12]), "+f"(v[13]),
               "+f"(v[14]), "+f"(v[15]));
}

__device__ __forceinline__ void reg_fence8(float* v) {
  asm volatile("" : "+f"(v[0]), "+f"(v[1]), "+f"(v[2]), "+f"(v[3]), "+f"(v[4]), "+f"(v[5]), "+f"(v[6]),
               "+f"(v[7]));
}

__device__ __forceinline__ uint64_t kmaj(const uint8_t* tile, int k) {
  return desc_sw128(smem_u32(tile) + 32 * k, 16, 1024);
}
// MN-major operand, K step k (16 rows of the tile); the second 64-wide atom
// along MN sits `lbo` bytes after the first.
__device__ __forceinline__ uint64_t mnmaj(uint32_t addr, int k, uint32_t lbo) {
  return desc_sw128(addr + 2048 * k, lbo, 1024);
}
// One K step (16 rows of K) is a constant added to a descriptor, whose fields
// count 16-byte units: 32 bytes of a K-major tile, one 2048-byte block of an
// MN-major one, and for the [V | 1] operand (second MN atom = the ones tile,
// reached through the leading byte offset) the offset shrinks by as much.
// The ones tile lies above every V block, so the offset stays positive.
constexpr uint64_t kKmajStep = 32 >> 4;
constexpr uint64_t kMnmajStep = 2048 >> 4;
constexpr uint64_t kMnmajOnesStep = (2048 >> 4) - ((uint64_t)(2048 >> 4) << 16);

// One 16-column block of the decay mask on a row of S (row i of its chunk,
// columns j0..j0+15), in place.  Blocks entirely left (right) of every row
// of the warp (rows row_lo..row_lo+31) take the lower (upper) factor pair
// without a select.  A row scale 2^lrow, already folded into the row
// factors ai and ri, enters the per-element exponential of the exact branch.
template <int MASK>
__device__ __forceinline__ void mask_block(float* sv, int j0, int i, int row_lo, bool exact, float ai, float ri,
                                           float pi, const float* alpha, const float* rho, const float* pp,
                                           float lrow = 0.f) {
  if (MASK == MASK_LIT) return;
  if (exact) {
#pragma unroll
    for (int e = 0; e < 16; ++e) sv[e] *= ex2(fmaf(-fabsf(pi - pp[j0 + e]), kLog2e, lrow));
    return;
  }
  if (j0 + 15 < row_lo) {
    const float2 a2 = make_float2(ai, ai);
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const float4 r4 = *reinterpret_cast<const float4*>(rho + j0 + 4 * v);
      const float2 p0 = mul2(mul2(make_float2(sv[4 * v], sv[4 * v + 1]), make_float2(r4.x, r4.y)), a2);
      const float2 p1 = mul2(mul2(make_float2(sv[4 * v + 2], sv[4 * v + 3]), make_float2(r4.z, r4.w)), a2);
      sv[4 * v] = p0.x;
      sv[4 * v + 1] = p0.y;
      sv[4 * v + 2] = p1.x;
      sv[4 * v + 3] = p1.y;
    }
  } else if (j0 > row_lo + 31) {
    const float2 r2 = make_float2(ri, ri);
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const float4 a4 = *reinterpret_cast<const float4*>(alpha + j0 + 4 * v);
      const float2 p0 = mul2(mul2(make_float2(sv[4 * v], sv[4 * v + 1]), make_float2(a4.x, a4.y)), r2);
      const float2 p1 = mul2(mul2(make_float2(sv[4 * v + 2], sv[4 * v + 3]), make_float2(a4.z, a4.w)), r2);
      sv[4 * v] = p0.x;
      sv[4 * v + 1] = p0.y;
      sv[4 * v + 2] = p1.x;
      sv[4 * v + 3] = p1.y;
    }
  } else {
    const float2 a2 = make_float2(ai, ai), r2 = make_float2(ri, ri);
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const float4 r4 = *reinterpret_cast<const float4*>(rho + j0 + 4 * v);
      const float4 a4 = *reinterpret_cast<const float4*>(alpha + j0 + 4 * v);
#pragma unroll
      for (int e = 0; e < 4; e += 2) {
        const int j = j0 + 4 * v + e;
        const float2 lo = mul2(a2, e == 0 ? make_float2(r4.x, r4.y) : make_float2(r4.z, r4.w));
        const float2 up = mul2(r2, e == 0 ? make_float2(a4.x, a4.y) : make_float2(a4.z, a4.w));
        const float2 fct = make_float2(j <= i ? lo.x : up.x, j + 1 <= i ? lo.y : up.y);
        const float2 pv = mul2(make_float2(sv[4 * v + e], sv[4 * v + e + 1]), fct);
        sv[4 * v + e] = pv.x;
        sv[4 * v + e + 1] = pv.y;
      }
    }
  }
}


typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
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
inline bool make_map128(CUtensorMap* m, const void* base, int L, int BH) {
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

// out: [BH][L][64] fp32; box = 32 columns (128 bytes, 128-byte swizzle) x
// 32 rows x 1 (rows past L are not written).
inline bool make_out_map(CUtensorMap* m, float* base, int L, int BH) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)L, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)kD * 4, (cuuint64_t)L * kD * 4};
  cuuint32_t box[3] = {32, 32, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// y as bfloat16 [BH][L][64]: a box of `cols` columns x 32 rows, the
// 128-byte swizzle when a box row is 128 bytes (cols = 64), none otherwise.
inline bool make_out_map_bf16(CUtensorMap* m, void* base, int L, int BH, int cols) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)L, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)L * kD * 2};
  cuuint32_t box[3] = {(cuuint32_t)cols, 32, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            cols == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline int sm_count() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}


}  // namespace c128
}  // namespace lion
