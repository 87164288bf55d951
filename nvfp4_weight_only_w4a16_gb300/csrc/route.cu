// Prefill routing (top-k + softmax over the chosen logits, per-CTA
// histograms, one-CTA scan into offsets and m-tiles, stable scatter and x
// gather) and the weighted combine of the prefill path.  The decode path
// routes inside its kernel (decode_stream.cu; decode.cu for the W4A4 variant)
// with the same primitives (route_common.cuh).
#include "common.cuh"
#include "kernels.h"
#include "route_common.cuh"

namespace nvfp4moe {

// ---------------------------------------------------------------------------
// Prefill: multi-CTA route, one-CTA scan, multi-CTA scatter + gather.
// ---------------------------------------------------------------------------
// K1: one warp per token (8 tokens per CTA): ids, weights, NaN count.  A
// token has k slots: its topk routed choices over the Er routed experts, then
// (k > topk) the shared expert, id Er, with weight 1.
__global__ void __launch_bounds__(256) route_topk_kernel(const void* __restrict__ logits, int bf16, int T, int k,
                                                         int topk, int Er, RouteParams rp, Workspace ws) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int nan_total = 0;
  {
    const int t = blockIdx.x * 8 + warp;
    if (t >= T) return;
    int id;
    float w;
    nan_total += warp_topk(logits, bf16, Er, topk, t, rp, &id, &w);
    if (lane < topk) {
      ws.ids[(size_t)t * k + lane] = id;
      ws.wts[(size_t)t * k + lane] = w;
    } else if (lane < k) {
      ws.ids[(size_t)t * k + lane] = Er;
      ws.wts[(size_t)t * k + lane] = 1.0f;
    }
  }
  if (lane == 0 && nan_total) atomicAdd(&ws.status->nan_logits, (unsigned)nan_total);
}

// K2: stable rank of every routed row inside its block of kRankTokens tokens,
// and the block's per-expert counts.  Rows of one expert are ordered by token
// (a token picks an expert at most once), so the rank of (t, j) is the number
// of earlier tokens of the block that picked the same expert.
__global__ void __launch_bounds__(256) route_rank_kernel(int T, int k, int E, Workspace ws) {
  __shared__ int32_t cnt[8][256];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < 8 * 256; i += blockDim.x) (&cnt[0][0])[i] = 0;
  __syncthreads();
  // kRankTokens / 8 tokens per warp, one per lane: the turn-taking loop below
  // is serial, so a short one (and more blocks) routes a chunk faster
  constexpr int kPerWarp = kRankTokens / 8;
  const int t = blockIdx.x * kRankTokens + warp * kPerWarp + lane;
  const bool valid = lane < kPerWarp && t < T;
  int ids[16], rank[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) ids[j] = (valid && j < k) ? ws.ids[(size_t)t * k + j] : -1;
  // lanes take turns in token order; each bumps its experts' counters
  for (int l = 0; l < kPerWarp; ++l) {
    if (lane == l) {
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (ids[j] >= 0) rank[j] = cnt[warp][ids[j]]++;
    }
    __syncwarp();
  }
  __syncthreads();
  // per-expert prefix over the 8 warps of the block
  if ((int)threadIdx.x < E) {
    int running = 0;
    for (int w = 0; w < 8; ++w) {
      const int c = cnt[w][threadIdx.x];
      cnt[w][threadIdx.x] = running;
      running += c;
    }
    ws.blk_counts[(size_t)blockIdx.x * E + threadIdx.x] = running;
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < 16; ++j)
    if (ids[j] >= 0) ws.local_rank[(size_t)t * k + j] = cnt[warp][ids[j]] + rank[j];
}

// K3 (one CTA): per-expert base of every rank block, expert offsets, and the
// list of m-tiles (<= kTileRows routed rows of one expert each).
__global__ void __launch_bounds__(1024) route_scan_kernel(int nblocks, int E, Workspace ws) {
  __shared__ int scan_tmp[32];
  const int e = threadIdx.x;
  int running = 0;
  if (e < E) {
    int c = 0;
    for (; c + 8 <= nblocks; c += 8) {  // eight loads in flight, then the running sums
      int v[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) v[q] = ws.blk_counts[(size_t)(c + q) * E + e];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        ws.blk_base[(size_t)(c + q) * E + e] = running;
        running += v[q];
      }
    }
    for (; c < nblocks; ++c) {
      const int v = ws.blk_counts[(size_t)c * E + e];
      ws.blk_base[(size_t)c * E + e] = running;
      running += v;
    }
  }
  int total = 0, ntiles = 0;
  const int off = block_exclusive_scan(e < E ? running : 0, scan_tmp, &total);
  const int nt = e < E ? (running + kTileRows - 1) / kTileRows : 0;
  const int tb = block_exclusive_scan(nt, scan_tmp, &ntiles);
  if (e < E) {
    ws.offsets[e] = off;
    for (int i = 0; i < nt; ++i) {
      ws.tile_expert[tb + i] = e;
      ws.tile_row0[tb + i] = off + i * kTileRows;
      ws.tile_rows[tb + i] = min(kTileRows, running - i * kTileRows);
    }
  }
  if (threadIdx.x == 0) {
    ws.offsets[E] = total;
    *ws.num_tiles = ntiles;
  }
}

// K4: one warp per routed row: its position, perm/inv, and (unless only
// routing) the copy of x[t] into position order as the FP16 operand of the
// grouped GEMMs:
//  * W4A16 experts: x times 2^-px, px such that the row's largest magnitude
//    lands in [2^13, 2^14) (exact for every BF16 value within 2^31 of it);
//    and the exponent ph of the row's h: the bound B = gs_g gs_u hb[e] ||x||^2
//    on every |h| of the row (|silu(g)| <= |g| <= gs_g ||Wg_f|| ||x|| and
//    |u| <= gs_u ||Wu_f|| ||x||, Cauchy-Schwarz; hb from launch_gateup_bound)
//    times 2^-ph stays below 2^13, so h times 2^-ph fits FP16;
//  * W4A4 experts (in_scale set, e < Er): x quantised to NVFP4 with the
//    expert's w13 input scale, code * scale (exact in FP16), px = ph = 0.
__global__ void __launch_bounds__(256) route_scatter_kernel(const __nv_bfloat16* __restrict__ x, int T, int k,
                                                            int E, int H, const float* __restrict__ in_scale,
                                                            int Er, const float* __restrict__ gs,
                                                            const float* __restrict__ hbound, Workspace ws) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t i = (size_t)blockIdx.x * 8 + warp;
  if (i >= (size_t)T * k) return;
  const int t = (int)(i / k);
  const int e = ws.ids[i];
  const int pos = ws.offsets[e] + ws.blk_base[(size_t)(t / kRankTokens) * E + e] + ws.local_rank[i];
  if (lane == 0) {
    ws.perm[pos] = (int)i;
    ws.inv[i] = pos;
  }
  if (x == nullptr) return;
  const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * H);
  uint4* dst = reinterpret_cast<uint4*>(ws.x_perm + (size_t)pos * H);
  if (in_scale == nullptr || e >= Er) {
    // pass 1: the row's largest magnitude and squared norm
    float m = 0.f, n2 = 0.f;
    for (int v = lane; v < H / 8; v += 32) {
      const uint4 u = __ldg(src + v);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int z = 0; z < 4; ++z) {
        const float lo = __uint_as_float(w[z] << 16), hi = __uint_as_float(w[z] & 0xFFFF0000u);
        m = fmaxf(m, fmaxf(fabsf(lo), fabsf(hi)));
        n2 = fmaf(lo, lo, fmaf(hi, hi, n2));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      n2 += __shfl_xor_sync(0xffffffffu, n2, o);
    }
    const int px = max(-126, min(126, prescale_exp(m)));
    // FP32 sums and products: a factor 2 of margin keeps B an upper bound
    const float B = 2.0f * __ldg(gs + 3 * e) * __ldg(gs + 3 * e + 1) * __ldg(hbound + e) * n2;
    const int ph = B > 3.0e38f ? 126 : max(-126, min(126, prescale_exp(B)));
    if (lane == 0) {
      ws.pexp_x[pos] = px;
      ws.pexp_h[pos] = ph;
    }
    const float sc = __int_as_float((127 - px) << 23);
    // pass 2: the scaled FP16 row (the source is in L1/L2 now)
    for (int v = lane; v < H / 8; v += 32) {
      const uint4 u = __ldg(src + v);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
      uint32_t o[4];
#pragma unroll
      for (int z = 0; z < 4; ++z) {
        const __half2 hh = __floats2half2_rn(__uint_as_float(w[z] << 16) * sc, __uint_as_float(w[z] & 0xFFFF0000u) * sc);
        o[z] = *reinterpret_cast<const uint32_t*>(&hh);
      }
      dst[v] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    return;
  }
  if (lane == 0) {
    ws.pexp_x[pos] = 0;
    ws.pexp_h[pos] = 0;
  }
  const float is = __ldg(in_scale + 2 * e), inv6 = act_inv6(is);
  for (int bk = lane; bk < H / 16; bk += 32) {  // one 16-element block per lane
    const uint4 u0 = __ldg(src + 2 * bk), u1 = __ldg(src + 2 * bk + 1);
    const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
    float v[16];
#pragma unroll
    for (int z = 0; z < 8; ++z) {
      v[2 * z] = __uint_as_float(w[z] << 16);
      v[2 * z + 1] = __uint_as_float(w[z] & 0xFFFF0000u);
    }
    uint32_t o[8];
    act_quant16_f16(v, is, inv6, o);
    dst[2 * bk] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[2 * bk + 1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

cudaError_t launch_route_prefill(const LayerDims& d, const void* logits, const void* x, int T, int top_k,
                                 const Workspace& ws, cudaStream_t st) {
  const int nrb = (T + kRankTokens - 1) / kRankTokens;
  const int k = top_k + d.S;  // slots per token
  route_topk_kernel<<<(T + 7) / 8, 256, 0, st>>>(logits, d.logits_bf16, T, k, top_k, d.Er, d.rp, ws);
  route_rank_kernel<<<nrb, 256, 0, st>>>(T, k, d.E, ws);
  route_scan_kernel<<<1, 1024, 0, st>>>(nrb, d.E, ws);
  const size_t rows = (size_t)T * k;
  route_scatter_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(x), T,
                                                                   k, d.E, d.H, d.in_scale, d.Er, d.gs, d.hbound, ws);
  return cudaGetLastError();
}

// A dense linear: identity tables and m-tiles of tile_rows (<= 128) rows in
// token order.
__global__ void __launch_bounds__(256) route_linear_kernel(int T, int tile_rows, Workspace ws) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < T) {
    ws.ids[i] = 0;
    ws.wts[i] = 1.0f;
    ws.perm[i] = i;
    ws.inv[i] = i;
  }
  const int ntiles = (T + tile_rows - 1) / tile_rows;
  if (i < ntiles) {
    ws.tile_expert[i] = 0;
    ws.tile_row0[i] = i * tile_rows;
    ws.tile_rows[i] = min(tile_rows, T - i * tile_rows);
  }
  if (i == 0) {
    ws.offsets[0] = 0;
    ws.offsets[1] = T;
    *ws.num_tiles = ntiles;
  }
}

cudaError_t launch_route_linear(int T, int tile_rows, const Workspace& ws, cudaStream_t st) {
  if (tile_rows < 16 || tile_rows > kTileRows || tile_rows % 16) return cudaErrorInvalidValue;
  const int n = max(T, (T + tile_rows - 1) / tile_rows);
  route_linear_kernel<<<(n + 255) / 256, 256, 0, st>>>(T, tile_rows, ws);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Router linear for a few tokens (T <= 16): logits[t][e] = x[t] . W[e] in
// FP32 from BF16 x [T][H] and W [E][H].  One CTA per expert; each thread takes
// 16-byte pieces of the row (8 columns), the 8 warps' partial sums are added
// in warp order.  The routers stay BF16 ("GLM-5.3-Flash on Blackwell", The
// quantization).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) router_gemv_kernel(const __nv_bfloat16* __restrict__ x,
                                                          const __nv_bfloat16* __restrict__ w, int T, int H,
                                                          float* __restrict__ logits, int E) {
  __shared__ float part[8][16];
  const int e = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float acc[16];
#pragma unroll
  for (int t = 0; t < 16; ++t) acc[t] = 0.f;
  const uint4* wr = reinterpret_cast<const uint4*>(w + (size_t)e * H);
  for (int p = threadIdx.x; p < H / 8; p += blockDim.x) {
    const uint4 wv = __ldg(wr + p);
    const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      if (t >= T) break;
      const uint4 xv = __ldg(reinterpret_cast<const uint4*>(x + (size_t)t * H) + p);
      const uint32_t xx[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        acc[t] = fmaf(__uint_as_float(xx[q] << 16), __uint_as_float(ww[q] << 16), acc[t]);
        acc[t] = fmaf(__uint_as_float(xx[q] & 0xFFFF0000u), __uint_as_float(ww[q] & 0xFFFF0000u), acc[t]);
      }
    }
  }
#pragma unroll
  for (int t = 0; t < 16; ++t) {
    float v = acc[t];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) part[warp][t] = v;
  }
  __syncthreads();
  if (threadIdx.x < T) {
    float v = 0.f;
    for (int j = 0; j < 8; ++j) v += part[j][threadIdx.x];
    logits[(size_t)threadIdx.x * E + e] = v;
  }
}

cudaError_t launch_router_gemv(const void* x, const void* w, int T, int E, int H, float* logits, cudaStream_t st) {
  if (T < 1 || T > 16) return cudaErrorInvalidValue;
  router_gemv_kernel<<<E, 256, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(x),
                                        reinterpret_cast<const __nv_bfloat16*>(w), T, H, logits, E);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Weighted combine: out[t][d] = sum_{j<k} w[t][j] * y[pos(t,j)][d] in FP32,
// slot order j = 0..k-1 (a shared expert is the last slot, weight 1),
// rounded once to BF16.  One thread per 8 outputs.
// ---------------------------------------------------------------------------
template <bool kOutF32>
__global__ void __launch_bounds__(256) combine_kernel(int T, int k, int H, const float* __restrict__ y,
                                                      const float* __restrict__ wts, const int32_t* __restrict__ inv,
                                                      void* __restrict__ out) {
  const int per_row = H / 8;
  const size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (size_t)T * per_row) return;
  const int t = (int)(idx / per_row), d8 = (int)(idx % per_row);
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int j = 0; j < k; ++j) {
    const float w = wts[(size_t)t * k + j];
    const float4* yr = reinterpret_cast<const float4*>(y + (size_t)inv[(size_t)t * k + j] * H) + 2 * d8;
    const float4 a = yr[0], b = yr[1];
    acc[0] = fmaf(w, a.x, acc[0]);
    acc[1] = fmaf(w, a.y, acc[1]);
    acc[2] = fmaf(w, a.z, acc[2]);
    acc[3] = fmaf(w, a.w, acc[3]);
    acc[4] = fmaf(w, b.x, acc[4]);
    acc[5] = fmaf(w, b.y, acc[5]);
    acc[6] = fmaf(w, b.z, acc[6]);
    acc[7] = fmaf(w, b.w, acc[7]);
  }
  if constexpr (kOutF32) {
    float4* o = reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + (size_t)t * H) + 2 * d8;
    o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  } else {
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]);
      o[q] = *reinterpret_cast<const uint32_t*>(&b2);
    }
    reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(out) + (size_t)t * H)[d8] =
        make_uint4(o[0], o[1], o[2], o[3]);
  }
}

cudaError_t launch_combine(const LayerDims& d, int T, int top_k, const Workspace& ws, void* out, cudaStream_t st) {
  const size_t n = (size_t)T * (d.H / 8);
  const int k = top_k + d.S;  // slots per token; the shared expert's is last
  if (d.out_f32)
    combine_kernel<true><<<(unsigned)((n + 255) / 256), 256, 0, st>>>(T, k, d.H, ws.y, ws.wts, ws.inv, out);
  else
    combine_kernel<false><<<(unsigned)((n + 255) / 256), 256, 0, st>>>(T, k, d.H, ws.y, ws.wts, ws.inv, out);
  return cudaGetLastError();
}

}  // namespace nvfp4moe
