// Shared device helpers for the NVFP4 W4A16 MoE kernels (sm_103a).
#pragma once
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>

namespace nvfp4moe {

// ---------------------------------------------------------------------------
// Device status word (one per handle, in device memory).
// ---------------------------------------------------------------------------
struct DeviceStatus {
  unsigned int flags;       // bit 0: bounded wait timed out, bit 1: bounds check fired
  unsigned int nan_logits;  // NaN router logits seen
  unsigned int where;       // first failing site (for the log)
  unsigned int pad;
};
constexpr unsigned int kFlagTimeout = 1u;
constexpr unsigned int kFlagBounds = 2u;

__device__ __forceinline__ void report(DeviceStatus* st, unsigned int flag, unsigned int where) {
  if (atomicOr(&st->flags, flag) == 0u) st->where = where;
}

// ---------------------------------------------------------------------------
// Packed-weight layout constants.
//   Matrix W [N][K], N % 128 == 0, K % 64 == 0.  A "chunk" is 64 K-elements.
//   The matrix is a sequence of 4608-byte tiles, one per (row block rb of 128
//   rows, chunk c), tile rb*nch + c: 4096 bytes of codes, then 512 of scales,
//   so that any run of chunks of one row block is one contiguous range.
//   Codes: for sub-block sb (16 rows), lane t (0..31): 16 bytes at
//   sb*512 + P(t)*16 of the tile, holding
//     bytes 0..7 : row rb*128+sb*16+t/4,   K elements 64c+16(t%4) .. +15
//     bytes 8..15: the row 8 below, same K elements
//   (byte j of each half holds elements 2j / 2j+1 in its low / high nibble).
//   Scales: 2 bytes at 4096 + sb*64 + P(t)*2 of the tile: the E4M3 scale of
//   the two rows' 16-element group.
//   P(t) = 8*(t%4) + (t/4 + 2*(t%4)) % 8 orders a sub-block's segments by K
//   group (group q in 16-byte slots 8q .. 8q+7, rotated by 2q): each 8-lane
//   phase of a 16-byte fragment read (segments t = 8p .. 8p+7) and each
//   thread-per-row read of one group (rows r, r+8 of group q) cover all 32
//   shared-memory banks once.
//   Segment s = ((rb*nch + c)*8 + sb)*32 + t names one lane's 16 code bytes
//   and 2 scale bytes (code_byte / scale_byte below).
//   The gate/up matrix is stored row-interleaved: packed row 16g+r is gate
//   feature 8g+r for r < 8 and up feature 8g+r-8 for r >= 8.
// ---------------------------------------------------------------------------
constexpr int kChunk = 64;
constexpr int kSegBytes = 16;
constexpr int kBlockRows = 128;
constexpr int kTileCodes = 4096;  // one tile's codes
constexpr int kTileBytes = 4608;  // codes + scales

__host__ __device__ inline int seg_pos(int t) { return 8 * (t & 3) + (((t >> 2) + 2 * (t & 3)) & 7); }  // P(t)
__host__ __device__ inline size_t code_byte(size_t s) {
  return (s >> 8) * kTileBytes + ((s >> 5) & 7) * 512 + (size_t)seg_pos((int)(s & 31)) * 16;
}
__host__ __device__ inline size_t scale_byte(size_t s) {
  return (s >> 8) * kTileBytes + kTileCodes + ((s >> 5) & 7) * 64 + (size_t)seg_pos((int)(s & 31)) * 2;
}

struct ExpertLayout {
  // byte offsets inside one expert's blob: the gate/up matrix, the down matrix
  size_t w13, w2, stride;
};

// A dense linear W [N][K] packed on its own, like an expert's down matrix
// (N output rows, K reduction): codes, then scales; no gate/up part.
__host__ __device__ inline ExpertLayout linear_layout(int N, int K) {
  ExpertLayout L;
  const size_t n = (size_t)N * K;
  L.w13 = 0;
  L.w2 = 0;
  L.stride = n / 2 + n / 16;
  return L;
}

__host__ __device__ inline ExpertLayout expert_layout(int H, int I) {
  ExpertLayout L;
  size_t n13 = (size_t)2 * I * H, n2 = (size_t)H * I;
  L.w13 = 0;
  L.w2 = n13 / 2 + n13 / 16;
  L.stride = L.w2 + n2 / 2 + n2 / 16;
  return L;
}

// ---------------------------------------------------------------------------
// Format conversions.  The E2M1 and E4M3 conversions use the hardware cvt
// instructions of sm_100-family GPUs; the product e2m1 * e4m3 (at most 5
// significant bits, magnitude in [2^-10, 2688]) is exact in FP16.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte_in_low_bits) {
  uint32_t r;
  asm("{\n .reg .b8 b;\n cvt.u8.u32 b, %1;\n cvt.rn.f16x2.e2m1x2 %0, b;\n}" : "=r"(r) : "r"(byte_in_low_bits));
  return r;
}

// Two E4M3 bytes (lo = bits 0..7, hi = bits 8..15) -> f16x2 {lo, hi}.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
  uint32_t r;
  unsigned short s = (unsigned short)two_bytes;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(s));
  return r;
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// {x.lo, x.lo} and {x.hi, x.hi}
__device__ __forceinline__ uint32_t dup_lo(uint32_t x) { return __byte_perm(x, 0, 0x1010); }
__device__ __forceinline__ uint32_t dup_hi(uint32_t x) { return __byte_perm(x, 0, 0x3232); }

// f16x2 (exact dequantised values) -> bf16x2, exact for these values.
__device__ __forceinline__ uint32_t f16x2_to_bf16x2(uint32_t v) {
  __half2 h = *reinterpret_cast<__half2*>(&v);
  float2 f = __half22float2(h);
  __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
  return *reinterpret_cast<uint32_t*>(&b);
}

// 8 E2M1 codes (nibble j = element j) -> 4 f16x2 {element 2j, element 2j+1}.
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t (&o)[4]) {
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
      : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
      : "r"(w));
}

// ---------------------------------------------------------------------------
// W4A4 activation quantisation (NVFP4 activations with a per-module input
// scale is, the stock routed-expert format: "tenhkspark/GLM-5.3-Flash-NVFP4-
// Wabi", opening summary).  With inv6 = fl(1 / fl(6 is)) per module, per
// block of 16 values: scale = E4M3(fl(amax * inv6)), r = fl(1 / fl(scale *
// is)), code = E2M1(fl(v * r)); both conversions round to nearest even and
// saturate.  The values returned are code * scale, exact in FP16 and BF16;
// the input scale is applied after the dot product.
// ---------------------------------------------------------------------------
struct ActBlockScale {
  uint32_t s2;  // f16x2 {scale, scale}
  float r;      // 1 / (scale * is), 0 when the scale is 0
};
__device__ __forceinline__ float act_inv6(float is) { return __frcp_rn(__fmul_rn(6.0f, is)); }
__device__ __forceinline__ ActBlockScale act_block_scale(float amax, float inv6, float is) {
  const float st = __fmul_rn(amax, inv6);
  unsigned short sc;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %1;" : "=h"(sc) : "f"(st));
  const uint32_t s2 = e4m3x2_to_f16x2(sc);
  const float sv = __half2float(__ushort_as_half((unsigned short)(s2 & 0xFFFFu)));
  const float step = __fmul_rn(sv, is);
  return ActBlockScale{s2, step > 0.f ? __frcp_rn(step) : 0.f};
}

// E2M1 codes of v[0..7] (already multiplied by r), nibble j = code of v[j].
__device__ __forceinline__ uint32_t e2m1x8_rn(const float* v) {
  uint32_t r;
  asm("{\n .reg .b8 b0, b1, b2, b3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
      " mov.b32 %0, {b0, b1, b2, b3};\n}"
      : "=r"(r)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  return r;
}

// One block of 16 values -> 8 f16x2 of code * scale (in element order).
__device__ __forceinline__ void act_quant16_f16(const float (&v)[16], float is, float inv6, uint32_t (&out)[8]) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const ActBlockScale bs = act_block_scale(amax, inv6, is);
  float q[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) q[i] = __fmul_rn(v[i], bs.r);
  uint32_t c[4];
  e2m1x8_to_f16x2x4(e2m1x8_rn(q), c);
#pragma unroll
  for (int z = 0; z < 4; ++z) out[z] = hmul2_u32(c[z], bs.s2);
  e2m1x8_to_f16x2x4(e2m1x8_rn(q + 8), c);
#pragma unroll
  for (int z = 0; z < 4; ++z) out[4 + z] = hmul2_u32(c[z], bs.s2);
}

// One value of a block whose scale is bs -> code * scale.
__device__ __forceinline__ float act_quant1(float v, const ActBlockScale& bs) {
  uint32_t b;
  asm("{\n .reg .b8 c;\n cvt.rn.satfinite.e2m1x2.f32 c, %1, %1;\n cvt.u32.u8 %0, c;\n}"
      : "=r"(b)
      : "f"(__fmul_rn(v, bs.r)));
  const uint32_t f = hmul2_u32(e2m1x2_to_f16x2(b), bs.s2);
  return __half2float(__ushort_as_half((unsigned short)(f & 0xFFFFu)));
}

// Order-preserving key of a float: larger float -> larger key; NaN -> 0
// (below -inf, whose key is 0x007FFFFF); -0 and +0 share one key, as they
// compare equal.
__device__ __forceinline__ uint32_t float_key(float f) {
  if (f != f) return 0u;
  if (f == 0.0f) return 0x80000000u;
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

// Power-of-two exponent p such that max * 2^-p lies in [2^13, 2^14): the
// scaled row fits FP16 with headroom for the products' partial sums.
__device__ __forceinline__ int prescale_exp(float amax) {
  if (!(amax > 0.0f) || !isfinite(amax)) return 0;
  return ilogbf(amax) - 13;
}

// ---------------------------------------------------------------------------
// Warp MMA m16n8k16, FP16 inputs, FP32 accumulate.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

}  // namespace nvfp4moe
