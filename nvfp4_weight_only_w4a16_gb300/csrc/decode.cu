// Decode path (1..16 tokens): bandwidth-bound grouped GEMV over the touched
// experts, dequantising NVFP4 in registers.
//
// At decode sizes every expert a token picks is streamed from HBM once per
// step, which is why the GLM-5.3-Flash serving pages call single-stream decode
// "the memory-bandwidth wall for an 18B-active model" ("GLM-5.3-Flash on
// Blackwell", Two deployments, and the lever that reverses between them).  The
// weight-only path never takes an activation scale: weights are dequantised to
// 16-bit and multiplied with the 16-bit activations (same page, The model
// loaded, served an API, and produced garbage).
//
// Design (GB300):
//  * stream-K work split: the flat list of (touched expert, row block, 64-wide
//    K chunk) items is cut into equal contiguous ranges, one per warp, so
//    every SM streams the same number of bytes whatever the routing;
//    partial sums of a row block split across warps meet in an FP32 buffer
//    and the last warp to arrive (atomic counter) finishes the block;
//  * each lane issues one 16-byte, L1-bypassing load per 32 weights;
//  * dequantisation: hardware E2M1->FP16 convert, times the E4M3 group scale
//    in FP16 (exact); the dot products run on mma.sync m16n8k16 (FP16 in,
//    FP32 accumulate), which retires 16x8x16 products per instruction and
//    keeps the ALU cost per weight near one instruction;
//  * the K axis of every 64-chunk is permuted identically for weights and
//    activations so that each lane's 16-byte load covers exactly its fragment
//    (the sum over K is order-independent);
//  * activations enter as FP16 after a per-row power-of-two prescale (exact
//    for the BF16 inputs), undone in FP32 when the block is finished.
#include "common.cuh"
#include "kernels.h"

namespace nvfp4moe {

constexpr int kDecWarps = 8;       // warps per CTA
constexpr int kDecRG = 4;          // 16-row groups per block
constexpr int kPartFloats = 1024;  // [rg 4][row 16][token 16]

struct DecodeArgs {
  const uint8_t* blob;
  size_t expert_stride;
  size_t nib_off, sc_off;  // offsets of this matrix inside an expert blob
  const float* gscale;
  int K;        // reduction length
  int nblk;     // row blocks (64 rows) per expert
  int k;        // top_k
  int H, I;
  const int32_t* num_touched;
  const int32_t* tch_expert;
  const int32_t* tch_row0;
  const int32_t* tch_rows;
  const int32_t* perm;
  const __half* x16;
  const int32_t* xexp;
  __nv_bfloat16* h;
  uint32_t* hmax;
  float* y;
  float* part;
  int32_t* cnt;
};

// A operand for one 16x16 (logical) k-tile kt from a lane's 16-byte segment.
__device__ __forceinline__ void make_a(const uint4& raw, uint32_t s0, uint32_t s1, int kt, uint32_t& a0,
                                       uint32_t& a1, uint32_t& a2, uint32_t& a3) {
  const uint32_t wr0 = kt < 2 ? raw.x : raw.y;
  const uint32_t wr1 = kt < 2 ? raw.z : raw.w;
  const int sh = (kt & 1) * 16;
  a0 = hmul2_u32(e2m1x2_to_f16x2(wr0 >> sh), s0);
  a2 = hmul2_u32(e2m1x2_to_f16x2(wr0 >> (sh + 8)), s0);
  a1 = hmul2_u32(e2m1x2_to_f16x2(wr1 >> sh), s1);
  a3 = hmul2_u32(e2m1x2_to_f16x2(wr1 >> (sh + 8)), s1);
}

// B (activations) for the decode gate/up: 16 FP16 values of one token.
struct BFrag {
  uint32_t w[8];
};

__device__ __forceinline__ void load_b_f16(BFrag& b, const __half* row, int col) {
  const uint4* p = reinterpret_cast<const uint4*>(row + col);
  const uint4 u0 = __ldg(p), u1 = __ldg(p + 1);
  b.w[0] = u0.x; b.w[1] = u0.y; b.w[2] = u0.z; b.w[3] = u0.w;
  b.w[4] = u1.x; b.w[5] = u1.y; b.w[6] = u1.z; b.w[7] = u1.w;
}

// B for the down projection: 16 BF16 values of h, scaled by 2^-p into FP16.
__device__ __forceinline__ void load_b_bf16_scaled(BFrag& b, const __nv_bfloat16* row, int col, float sc) {
  const uint4* p = reinterpret_cast<const uint4*>(row + col);
  const uint4 u0 = p[0], u1 = p[1];
  const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const __half2 hh = __floats2half2_rn(__uint_as_float(w[i] << 16) * sc, __uint_as_float(w[i] & 0xFFFF0000u) * sc);
    b.w[i] = *reinterpret_cast<const uint32_t*>(&hh);
  }
}

__device__ __forceinline__ float pow2f(int p) {
  p = max(-126, min(127, p));
  return __int_as_float((127 + p) << 23);
}

template <bool kGateUp>
__device__ void finish_block(const DecodeArgs& a, int e, int row0, int m, int b, float (&acc)[kDecRG][2][4], int lane) {
  const int r0 = lane >> 2, q = lane & 3;
  const float* gs = a.gscale + 3 * e;
#pragma unroll
  for (int rg = 0; rg < kDecRG; ++rg) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int j = 8 * i + 2 * q + c;
        if (j >= m) continue;
        const int row = row0 + j;
        if (kGateUp) {
          const int t = a.perm[row] / a.k;
          const float s = pow2f(a.xexp[t]);
          const float g = gs[0] * (acc[rg][i][c] * s);
          const float u = gs[1] * (acc[rg][i][2 + c] * s);
          const __nv_bfloat16 hb = __float2bfloat16_rn(silu(g) * u);
          const int f = 8 * (kDecRG * b + rg) + r0;
          a.h[(size_t)row * a.I + f] = hb;
          atomicMax(&a.hmax[row], __float_as_uint(fabsf(__bfloat162float(hb))));
        } else {
          const float s = pow2f(prescale_exp(__uint_as_float(a.hmax[row])));
          const int d = 16 * (kDecRG * b + rg) + r0;
          a.y[(size_t)row * a.H + d] = gs[2] * (acc[rg][i][c] * s);
          a.y[(size_t)row * a.H + d + 8] = gs[2] * (acc[rg][i][2 + c] * s);
        }
      }
    }
  }
}

template <bool kGateUp>
__global__ void __launch_bounds__(kDecWarps * 32, 2) decode_gemv_kernel(DecodeArgs a) {
  const int lane = threadIdx.x & 31;
  const int warp_global = blockIdx.x * kDecWarps + (threadIdx.x >> 5);
  const long long W = (long long)gridDim.x * kDecWarps;
  const int U = *a.num_touched;
  const int nch = a.K / kChunk;
  const long long F = (long long)U * a.nblk * nch;
  long long f = F * warp_global / W;
  const long long fend = F * (warp_global + 1) / W;
  const int q = lane & 3, r0 = lane >> 2;

  while (f < fend) {
    const int blk = (int)(f / nch);
    const int c0 = (int)(f % nch);
    const int c1 = (int)min((long long)nch, c0 + (fend - f));
    f += c1 - c0;
    const int u = blk / a.nblk, b = blk % a.nblk;
    const int e = a.tch_expert[u], row0 = a.tch_row0[u], m = a.tch_rows[u];
    const int ng = (m + 7) >> 3;
    const uint8_t* nib = a.blob + (size_t)e * a.expert_stride + a.nib_off;
    const uint8_t* sc = a.blob + (size_t)e * a.expert_stride + a.sc_off;

    // the lane's B rows (token r0 of each 8-token group)
    const __half* xrow[2] = {nullptr, nullptr};
    const __nv_bfloat16* hrow[2] = {nullptr, nullptr};
    float hsc[2] = {1.f, 1.f};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int j = 8 * i + r0;
      if (j < m) {
        const int row = row0 + j;
        if (kGateUp) {
          xrow[i] = a.x16 + (size_t)(a.perm[row] / a.k) * a.H;
        } else {
          hrow[i] = a.h + (size_t)row * a.I;
          hsc[i] = pow2f(-prescale_exp(__uint_as_float(a.hmax[row])));
        }
      }
    }

    float acc[kDecRG][2][4];
#pragma unroll
    for (int rg = 0; rg < kDecRG; ++rg)
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int z = 0; z < 4; ++z) acc[rg][i][z] = 0.f;

    for (int c = c0; c < c1; ++c) {
      uint4 raw[kDecRG];
      uint32_t s2[kDecRG];
#pragma unroll
      for (int rg = 0; rg < kDecRG; ++rg) {
        const int g = kDecRG * b + rg;           // global 16-row group
        const size_t seg = ((size_t)(g >> 3) * nch + c) * 8 + (g & 7);
        raw[rg] = ldg_nc_na(nib + seg * 512 + lane * 16);
        s2[rg] = ldg_nc_u16(sc + seg * 64 + lane * 2);
      }
      BFrag bf[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        if (i < ng) {
          const int col = kChunk * c + 16 * q;
          if (kGateUp) {
            if (xrow[i]) load_b_f16(bf[i], xrow[i], col);
            else for (int z = 0; z < 8; ++z) bf[i].w[z] = 0u;
          } else {
            if (hrow[i]) load_b_bf16_scaled(bf[i], hrow[i], col, hsc[i]);
            else for (int z = 0; z < 8; ++z) bf[i].w[z] = 0u;
          }
        }
      }
#pragma unroll
      for (int rg = 0; rg < kDecRG; ++rg) {
        const uint32_t sx = e4m3x2_to_f16x2(s2[rg]);
        const uint32_t s0 = dup_lo(sx), s1 = dup_hi(sx);
#pragma unroll
        for (int kt = 0; kt < 4; ++kt) {
          uint32_t a0, a1, a2, a3;
          make_a(raw[rg], s0, s1, kt, a0, a1, a2, a3);
          mma_f16_16816(acc[rg][0], a0, a1, a2, a3, bf[0].w[2 * kt], bf[0].w[2 * kt + 1]);
          if (ng > 1) mma_f16_16816(acc[rg][1], a0, a1, a2, a3, bf[1].w[2 * kt], bf[1].w[2 * kt + 1]);
        }
      }
    }

    if (c0 == 0 && c1 == nch) {
      finish_block<kGateUp>(a, e, row0, m, b, acc, lane);
      continue;
    }
    // partial block: add into the shared FP32 buffer, last arriver finishes
    float* part = a.part + (size_t)blk * kPartFloats;
#pragma unroll
    for (int rg = 0; rg < kDecRG; ++rg)
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int j = 8 * i + 2 * q + c;
          if (j < m) {
            atomicAdd(part + rg * 256 + r0 * 16 + j, acc[rg][i][c]);
            atomicAdd(part + rg * 256 + (r0 + 8) * 16 + j, acc[rg][i][2 + c]);
          }
        }
    __threadfence();
    __syncwarp();
    int last = 0;
    if (lane == 0) {
      const int add = c1 - c0;
      const int old = atomicAdd(a.cnt + blk, add);
      last = (old + add == nch);
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (!last) continue;
    __threadfence();
#pragma unroll
    for (int rg = 0; rg < kDecRG; ++rg)
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int j = 8 * i + 2 * q + c;
          if (j < m) {
            float* p0 = part + rg * 256 + r0 * 16 + j;
            float* p1 = part + rg * 256 + (r0 + 8) * 16 + j;
            acc[rg][i][c] = __ldcg(p0);
            acc[rg][i][2 + c] = __ldcg(p1);
            __stcg(p0, 0.f);
            __stcg(p1, 0.f);
          }
        }
    if (lane == 0) a.cnt[blk] = 0;
    finish_block<kGateUp>(a, e, row0, m, b, acc, lane);
  }
}

cudaError_t launch_decode_ffn(const LayerDims& d, const uint8_t* blob, const float* gscale, int T, int k,
                              cudaEvent_t mid, int num_sms, const Workspace& ws, cudaStream_t st) {
  (void)T;
  const ExpertLayout L = expert_layout(d.H, d.I);
  DecodeArgs a{};
  a.blob = blob;
  a.expert_stride = L.stride;
  a.gscale = gscale;
  a.k = k;
  a.H = d.H;
  a.I = d.I;
  a.num_touched = ws.num_touched;
  a.tch_expert = ws.tch_expert;
  a.tch_row0 = ws.tch_row0;
  a.tch_rows = ws.tch_rows;
  a.perm = ws.perm;
  a.x16 = ws.x16;
  a.xexp = ws.xexp;
  a.h = ws.h;
  a.hmax = ws.hmax;
  a.y = ws.y;
  const int grid = 2 * num_sms;
  // gate/up: matrix rows 2I (interleaved), K = H, blocks of 64 rows = 32 features
  a.nib_off = L.w13_nib;
  a.sc_off = L.w13_sc;
  a.K = d.H;
  a.nblk = 2 * d.I / 64;
  a.part = ws.part_gu;
  a.cnt = ws.cnt_gu;
  decode_gemv_kernel<true><<<grid, kDecWarps * 32, 0, st>>>(a);
  if (mid) cudaEventRecord(mid, st);
  // down: rows H, K = I
  a.nib_off = L.w2_nib;
  a.sc_off = L.w2_sc;
  a.K = d.I;
  a.nblk = d.H / 64;
  a.part = ws.part_dn;
  a.cnt = ws.cnt_dn;
  decode_gemv_kernel<false><<<grid, kDecWarps * 32, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace nvfp4moe
