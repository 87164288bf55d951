// Packer: canonical NVFP4 bytes -> the tile-ordered device layout, and the
// dequantisation check that reads the packed layout back.
//
// Format: weight-only NVFP4 experts, 4-bit E2M1 values with one E4M3 scale per
// 16 weights along K and an FP32 scale per tensor ("tenhkspark/GLM-5.3-Flash-
// NVFP4-Wabi", Config expectations: group_size = 16, weight_scale_2).  The
// packed byte map is described in common.cuh.
#include "common.cuh"
#include "kernels.h"

namespace nvfp4moe {

// One thread per 16-byte packed segment (32 weights, two rows x 16).
__global__ void pack_matrix_kernel(const uint8_t* __restrict__ src_q, const uint8_t* __restrict__ src_s,
                                   uint8_t* __restrict__ blob, size_t expert_stride, size_t mat_off,
                                   int N, int K, int interleave_gate_up,
                                   size_t src_q_expert_stride, size_t src_s_expert_stride, int n_valid) {
  const int e = blockIdx.y;
  const size_t nseg = (size_t)N * K / 32;
  const size_t s = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= nseg) return;
  const int nch = K / kChunk;
  const int t = (int)(s % 32);
  const int sb = (int)((s / 32) % 8);
  const int c = (int)((s / 256) % nch);
  const int rb = (int)(s / (256 * (size_t)nch));
  const int q = t & 3;
  const int R0 = rb * kBlockRows + sb * 16 + (t >> 2);
  int crow0, crow1;
  if (interleave_gate_up) {
    const int I = N / 2;
    const int f0 = 8 * (R0 / 16) + (t >> 2);
    crow0 = f0;       // gate feature f0
    crow1 = I + f0;   // up feature f0
  } else {
    crow0 = R0;
    crow1 = R0 + 8;
  }
  const uint8_t* q_e = src_q + (size_t)e * src_q_expert_stride;
  const uint8_t* s_e = src_s + (size_t)e * src_s_expert_stride;
  const size_t kb = (size_t)K / 2, ks = (size_t)K / 16;
  // rows >= n_valid (padding up to a whole 128-row block) are zero codes and zero scales
  const bool v0 = crow0 < n_valid, v1 = crow1 < n_valid;
  const uint2 lo = v0 ? *reinterpret_cast<const uint2*>(q_e + crow0 * kb + 32 * c + 8 * q) : make_uint2(0u, 0u);
  const uint2 hi = v1 ? *reinterpret_cast<const uint2*>(q_e + crow1 * kb + 32 * c + 8 * q) : make_uint2(0u, 0u);
  uint8_t* dst = blob + (size_t)e * expert_stride + mat_off;
  *reinterpret_cast<uint4*>(dst + code_byte(s)) = make_uint4(lo.x, lo.y, hi.x, hi.y);
  const uint8_t s0 = v0 ? s_e[crow0 * ks + 4 * c + q] : 0;
  const uint8_t s1 = v1 ? s_e[crow1 * ks + 4 * c + q] : 0;
  *reinterpret_cast<uint16_t*>(dst + scale_byte(s)) = (uint16_t)(s0 | (s1 << 8));
}

// Dequantise one tensor of one expert from the packed blob:
// out[n][k] = fp32(e2m1 * e4m3) * gs.  via_bf16 routes the exact FP16 product
// through BF16 as the tensor-core path does; both must be bit-identical.
__global__ void debug_dequant_kernel(const uint8_t* __restrict__ blob_e, const float* __restrict__ gs_e,
                                     int H, int I, int which, int via_bf16, float* __restrict__ out) {
  const ExpertLayout L = expert_layout(H, I);
  const bool down = which == 2;
  const int N = down ? H : 2 * I, K = down ? I : H;
  const size_t nseg = (size_t)N * K / 32;
  const size_t s = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= nseg) return;
  const int nch = K / kChunk;
  const int t = (int)(s % 32);
  const int sb = (int)((s / 32) % 8);
  const int c = (int)((s / 256) % nch);
  const int rb = (int)(s / (256 * (size_t)nch));
  const int q = t & 3;
  const int R0 = rb * kBlockRows + sb * 16 + (t >> 2);
  const uint8_t* nib = blob_e + (down ? L.w2 : L.w13) + code_byte(s);
  const uint8_t* sc = blob_e + (down ? L.w2 : L.w13) + scale_byte(s);
  const uint4 raw = *reinterpret_cast<const uint4*>(nib);
  const uint32_t s2 = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(sc));
  const float g = gs_e[which];
  const uint32_t words[4] = {raw.x, raw.y, raw.z, raw.w};
  for (int half = 0; half < 2; ++half) {
    int row;
    if (down) {
      row = R0 + 8 * half;
    } else {
      const int f0 = 8 * (R0 / 16) + (t >> 2);
      if ((which == 0) != (half == 0)) continue;  // gate rows are the first half
      row = f0;
    }
    const uint32_t sx2 = half ? dup_hi(s2) : dup_lo(s2);
    for (int j = 0; j < 8; ++j) {
      const uint32_t byte = (words[2 * half + j / 4] >> (8 * (j % 4))) & 0xFFu;
      uint32_t v = hmul2_u32(e2m1x2_to_f16x2(byte), sx2);
      float f0v, f1v;
      if (via_bf16) {
        const uint32_t b = f16x2_to_bf16x2(v);
        f0v = __uint_as_float(b << 16);
        f1v = __uint_as_float(b & 0xFFFF0000u);
      } else {
        const float2 f = __half22float2(*reinterpret_cast<__half2*>(&v));
        f0v = f.x;
        f1v = f.y;
      }
      const size_t k = (size_t)64 * c + 16 * q + 2 * j;
      out[(size_t)row * K + k] = __fmul_rn(f0v, g);
      out[(size_t)row * K + k + 1] = __fmul_rn(f1v, g);
    }
  }
}

// Per expert e: the largest product ||Wg_f|| ||Wu_f|| (Euclidean norms of the
// dequantised gate and up rows of feature f, e2m1 * e4m3 without the tensor
// scales) over its features, written as float bits by atomicMax (hb starts
// at zero).  With the tensor scales and ||x||^2 it bounds every |h| of a
// routed row: |silu(g)| <= |g| <= gs_g ||Wg_f|| ||x|| (Cauchy-Schwarz) and
// |u| <= gs_u ||Wu_f|| ||x||, which sizes the power-of-two prescale of h for
// the prefill down GEMM's FP16 operand.  One warp per (expert, feature);
// canonical layout: gate rows 0..I-1, up rows I..2I-1.
__global__ void gateup_bound_kernel(const uint8_t* __restrict__ w13_q, const uint8_t* __restrict__ w13_s, int E,
                                    int H, int I, float* __restrict__ hb) {
  const size_t wid = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid >= (size_t)E * I) return;
  const int e = (int)(wid / I), f = (int)(wid - (size_t)e * I);
  float ss[2];
#pragma unroll
  for (int w = 0; w < 2; ++w) {
    const size_t row = (size_t)e * 2 * I + (size_t)w * I + f;
    const uint8_t* q = w13_q + row * (H / 2);
    const uint8_t* sc = w13_s + row * (H / 16);
    float acc = 0.f;
    for (int j = lane; j < H / 2; j += 32) {  // byte j: elements 2j, 2j+1 of group j / 8
      const uint32_t v = e2m1x2_to_f16x2(q[j]);
      const uint32_t s2 = e4m3x2_to_f16x2(sc[j >> 3]);
      const float s = __half2float(__ushort_as_half((unsigned short)(s2 & 0xFFFFu)));
      const float a0 = __half2float(__ushort_as_half((unsigned short)(v & 0xFFFFu))) * s;
      const float a1 = __half2float(__ushort_as_half((unsigned short)(v >> 16))) * s;
      acc = fmaf(a0, a0, fmaf(a1, a1, acc));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    ss[w] = acc;
  }
  // FP32 sums of at most 16384 exact squares: a relative margin of 2^-10 keeps it an upper bound
  const float b = sqrtf(ss[0]) * sqrtf(ss[1]) * (1.0f + 1.0f / 1024.0f);
  if (lane == 0 && b > 0.f) atomicMax(reinterpret_cast<unsigned*>(hb + e), __float_as_uint(b));
}

cudaError_t launch_gateup_bound(const uint8_t* w13_q, const uint8_t* w13_s, int E, int H, int I, float* hb,
                                cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(hb, 0, sizeof(float) * E, st);
  if (e != cudaSuccess) return e;
  const size_t warps = (size_t)E * I;
  gateup_bound_kernel<<<(unsigned)((warps + 7) / 8), 256, 0, st>>>(w13_q, w13_s, E, H, I, hb);
  return cudaGetLastError();
}

cudaError_t launch_pack(const uint8_t* w13_q, const uint8_t* w13_s, const uint8_t* w2_q,
                        const uint8_t* w2_s, uint8_t* blob, int E, int H, int I, cudaStream_t st) {
  const ExpertLayout L = expert_layout(H, I);
  const int thr = 256;
  {
    const size_t nseg = (size_t)2 * I * H / 32;
    dim3 grid((unsigned)((nseg + thr - 1) / thr), E);
    pack_matrix_kernel<<<grid, thr, 0, st>>>(w13_q, w13_s, blob, L.stride, L.w13, 2 * I, H, 1,
                                             (size_t)2 * I * H / 2, (size_t)2 * I * H / 16, 2 * I);
  }
  {
    const size_t nseg = (size_t)H * I / 32;
    dim3 grid((unsigned)((nseg + thr - 1) / thr), E);
    pack_matrix_kernel<<<grid, thr, 0, st>>>(w2_q, w2_s, blob, L.stride, L.w2, H, I, 0,
                                             (size_t)H * I / 2, (size_t)H * I / 16, H);
  }
  return cudaGetLastError();
}

cudaError_t launch_pack_linear(const uint8_t* w_q, const uint8_t* w_s, uint8_t* blob, int N, int Np, int K,
                               cudaStream_t st) {
  const ExpertLayout L = linear_layout(Np, K);
  const int thr = 256;
  const size_t nseg = (size_t)Np * K / 32;
  pack_matrix_kernel<<<(unsigned)((nseg + thr - 1) / thr), thr, 0, st>>>(w_q, w_s, blob, L.stride, L.w2,
                                                                         Np, K, 0, 0, 0, N);
  return cudaGetLastError();
}

cudaError_t launch_debug_dequant(const uint8_t* blob, const float* gscale, int H, int I, int expert,
                                 int which, int via_bf16, float* out, cudaStream_t st) {
  const ExpertLayout L = expert_layout(H, I);
  const bool down = which == 2;
  const size_t nseg = (size_t)(down ? H : 2 * I) * (down ? I : H) / 32;
  const int thr = 256;
  debug_dequant_kernel<<<(unsigned)((nseg + thr - 1) / thr), thr, 0, st>>>(
      blob + (size_t)expert * L.stride, gscale + 3 * expert, H, I, which, via_bf16, out);
  return cudaGetLastError();
}

}  // namespace nvfp4moe
