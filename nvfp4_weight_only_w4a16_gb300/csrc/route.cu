// Route (top-k + softmax over the chosen logits) and permute (stable,
// expert-major) kernels, plus the weighted combine.
//
// The routers of the GLM-5.3-Flash experts stay BF16 linears ("GLM-5.3-Flash
// on Blackwell", The quantization), so their logits arrive here as an input.
// Readings (the pages do not state the scoring rule): top-k by logit, equal
// logits -> lower expert index, NaN below -inf; weights = softmax over the k
// chosen logits; rows ordered expert-major, ascending t*k+j inside an expert.
#include "common.cuh"
#include "kernels.h"

namespace nvfp4moe {

__device__ __forceinline__ float load_logit(const void* logits, int bf16, size_t i) {
  if (bf16) {
    const unsigned short b = reinterpret_cast<const unsigned short*>(logits)[i];
    return __uint_as_float((uint32_t)b << 16);
  }
  return reinterpret_cast<const float*>(logits)[i];
}

// One warp routes one token.  Lane l owns experts l, l+32, ... (E <= 256).
// Writes ids[t*k + j], wts[t*k + j] for j < k (lanes j < k write).
__device__ void warp_topk(const void* logits, int bf16, int E, int k, int t, int32_t* ids, float* wts,
                          int32_t* ids_smem, DeviceStatus* st) {
  const int lane = threadIdx.x & 31;
  unsigned long long key[8];
  float val[8];
  int nan_count = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = lane + 32 * i;
    if (e < E) {
      const float v = load_logit(logits, bf16, (size_t)t * E + e);
      nan_count += (v != v);
      val[i] = v;
      key[i] = ((unsigned long long)float_key(v) << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)e);
    } else {
      val[i] = 0.f;
      key[i] = 0ull;
    }
  }
  int my_id = -1;
  float my_logit = 0.f;
  for (int j = 0; j < k; ++j) {
    unsigned long long best = 0ull;
#pragma unroll
    for (int i = 0; i < 8; ++i) best = key[i] > best ? key[i] : best;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
      best = other > best ? other : best;
    }
    const int e = (int)(0xFFFFFFFFu - (uint32_t)(best & 0xFFFFFFFFull));
    float v = 0.f;
    if ((e & 31) == lane) {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (lane + 32 * i == e) {
          key[i] = 0ull;
          v = val[i];
        }
    }
    v = __shfl_sync(0xffffffffu, v, e & 31);
    if (lane == j) {
      my_id = e;
      my_logit = v;
    }
  }
  // softmax over the chosen logits; NaN counts as -inf
  float l = (lane < k) ? (my_logit != my_logit ? -INFINITY : my_logit) : -INFINITY;
  float m = l;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float ex;
  if (m == -INFINITY) {
    ex = (lane < k) ? 1.0f : 0.0f;
  } else if (m == INFINITY) {
    ex = (lane < k && l == INFINITY) ? 1.0f : 0.0f;
  } else {
    ex = (lane < k) ? expf(l - m) : 0.0f;
  }
  // sum in slot order: lane 0 accumulates j = 0..k-1
  float sum = 0.f;
  for (int j = 0; j < k; ++j) sum += __shfl_sync(0xffffffffu, ex, j);
  if (lane < k) {
    ids[(size_t)t * k + lane] = my_id;
    wts[(size_t)t * k + lane] = ex / sum;
    if (ids_smem) ids_smem[lane] = my_id;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) nan_count += __shfl_xor_sync(0xffffffffu, nan_count, o);
  if (lane == 0 && nan_count) atomicAdd(&st->nan_logits, (unsigned)nan_count);
}

// Exclusive scan of v over the first n (<= 1024) threads of the block;
// returns the exclusive prefix, *total receives the sum.  All threads call.
__device__ int block_exclusive_scan(int v, int* smem_warp /*[32]*/, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) smem_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    const int nw = (blockDim.x + 31) >> 5;
    int w = lane < nw ? smem_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    smem_warp[lane] = w;  // inclusive
  }
  __syncthreads();
  const int before = warp ? smem_warp[warp - 1] : 0;
  *total = smem_warp[((blockDim.x + 31) >> 5) - 1];
  __syncthreads();
  return before + x - v;
}

// ---------------------------------------------------------------------------
// Decode: one CTA of 512 threads routes, permutes and converts x for T <= 16.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(512) route_decode_kernel(const void* __restrict__ logits, int bf16,
                                                           const __nv_bfloat16* __restrict__ x, int T, int k,
                                                           int E, int H, Workspace ws) {
  __shared__ int32_t ids_s[kDecodeMaxTokens * 16];
  __shared__ int32_t off_s[257];
  __shared__ int scan_tmp[32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nrows = T * k;
  if (warp < T) warp_topk(logits, bf16, E, k, warp, ws.ids, ws.wts, ids_s + warp * k, ws.status);
  __syncthreads();
  // histogram (every thread below E counts its expert)
  int c = 0;
  if ((int)threadIdx.x < E)
    for (int i = 0; i < nrows; ++i) c += (ids_s[i] == (int)threadIdx.x);
  int total = 0, touched_total = 0;
  const int off = block_exclusive_scan((int)threadIdx.x < E ? c : 0, scan_tmp, &total);
  const int tch = block_exclusive_scan(((int)threadIdx.x < E && c > 0) ? 1 : 0, scan_tmp, &touched_total);
  if ((int)threadIdx.x < E) {
    off_s[threadIdx.x] = off;
    ws.offsets[threadIdx.x] = off;
    if (c > 0) {
      ws.tch_expert[tch] = threadIdx.x;
      ws.tch_row0[tch] = off;
      ws.tch_rows[tch] = c;
    }
  }
  if (threadIdx.x == 0) {
    ws.offsets[E] = total;
    *ws.num_touched = touched_total;
  }
  __syncthreads();
  if ((int)threadIdx.x < nrows) {
    const int i = threadIdx.x, e = ids_s[i];
    int rank = 0;
    for (int j = 0; j < i; ++j) rank += (ids_s[j] == e);
    const int pos = off_s[e] + rank;
    ws.perm[pos] = i;
    ws.inv[i] = pos;
    ws.hmax[i] = 0u;  // row maxima of h, accumulated by the gate/up kernel
  }
  // x -> FP16 with a per-token power-of-two prescale (skipped when only routing)
  for (int t = warp; x != nullptr && t < T; t += blockDim.x >> 5) {
    const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)t * H);
    float amax = 0.f;
    for (int i = lane; i < H / 8; i += 32) {
      const uint4 v = xr[i];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        amax = fmaxf(amax, fabsf(__uint_as_float(w[q] << 16)));
        amax = fmaxf(amax, fabsf(__uint_as_float(w[q] & 0xFFFF0000u)));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    int p = prescale_exp(amax);
    p = max(-126, min(126, p));
    const float sc = __int_as_float((127 - p) << 23);  // 2^-p
    uint4* xo = reinterpret_cast<uint4*>(ws.x16 + (size_t)t * H);
    for (int i = lane; i < H / 8; i += 32) {
      const uint4 v = xr[i];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      uint32_t o4[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const __half2 hh = __floats2half2_rn(__uint_as_float(w[q] << 16) * sc,
                                             __uint_as_float(w[q] & 0xFFFF0000u) * sc);
        o4[q] = *reinterpret_cast<const uint32_t*>(&hh);
      }
      xo[i] = make_uint4(o4[0], o4[1], o4[2], o4[3]);
    }
    if (lane == 0) ws.xexp[t] = p;
  }
}

cudaError_t launch_route_decode(const LayerDims& d, const void* logits, const void* x, int T, int k,
                                const Workspace& ws, cudaStream_t st) {
  route_decode_kernel<<<1, 512, 0, st>>>(logits, d.logits_bf16, reinterpret_cast<const __nv_bfloat16*>(x), T, k,
                                         d.E, d.H, ws);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Prefill: multi-CTA route, one-CTA scan, multi-CTA scatter + gather.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) route_topk_kernel(const void* __restrict__ logits, int bf16, int T, int k,
                                                         int E, Workspace ws) {
  __shared__ int32_t hist[256];
  __shared__ int32_t ids_s[kRouteTokPerCta * 16];
  const int warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < E; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const int t0 = blockIdx.x * kRouteTokPerCta;
  for (int tt = warp; tt < kRouteTokPerCta; tt += 8) {
    const int t = t0 + tt;
    if (t < T) warp_topk(logits, bf16, E, k, t, ws.ids, ws.wts, ids_s + tt * k, ws.status);
  }
  __syncthreads();
  const int nloc = min(kRouteTokPerCta, T - t0) * k;
  for (int i = threadIdx.x; i < nloc; i += blockDim.x) atomicAdd(&hist[ids_s[i]], 1);
  __syncthreads();
  for (int i = threadIdx.x; i < E; i += blockDim.x) ws.blk_counts[(size_t)blockIdx.x * E + i] = hist[i];
}

__global__ void __launch_bounds__(1024) route_scan_kernel(int ncta, int E, Workspace ws) {
  __shared__ int scan_tmp[32];
  const int e = threadIdx.x;
  int running = 0;
  if (e < E) {
    for (int c = 0; c < ncta; ++c) {
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

__global__ void __launch_bounds__(256) route_scatter_kernel(const __nv_bfloat16* __restrict__ x, int T, int k,
                                                            int E, int H, Workspace ws) {
  __shared__ int32_t ids_s[kRouteTokPerCta * 16];
  __shared__ int32_t pos_s[kRouteTokPerCta * 16];
  const int t0 = blockIdx.x * kRouteTokPerCta;
  const int nloc = min(kRouteTokPerCta, T - t0) * k;
  const size_t i0 = (size_t)t0 * k;
  for (int i = threadIdx.x; i < nloc; i += blockDim.x) ids_s[i] = ws.ids[i0 + i];
  __syncthreads();
  for (int i = threadIdx.x; i < nloc; i += blockDim.x) {
    const int e = ids_s[i];
    int rank = 0;
    for (int j = 0; j < i; ++j) rank += (ids_s[j] == e);
    const int pos = ws.offsets[e] + ws.blk_base[(size_t)blockIdx.x * E + e] + rank;
    ws.perm[pos] = (int)(i0 + i);
    ws.inv[i0 + i] = pos;
    pos_s[i] = pos;
  }
  __syncthreads();
  if (x == nullptr) return;  // routing only
  // gather x rows into position order (16-byte copies)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nvec = H / 8;
  for (int i = warp; i < nloc; i += 8) {
    const int t = t0 + i / k;
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * H);
    uint4* dst = reinterpret_cast<uint4*>(ws.x_perm + (size_t)pos_s[i] * H);
    for (int v = lane; v < nvec; v += 32) dst[v] = src[v];
  }
}

cudaError_t launch_route_prefill(const LayerDims& d, const void* logits, const void* x, int T, int k,
                                 const Workspace& ws, cudaStream_t st) {
  const int ncta = (T + kRouteTokPerCta - 1) / kRouteTokPerCta;
  route_topk_kernel<<<ncta, 256, 0, st>>>(logits, d.logits_bf16, T, k, d.E, ws);
  route_scan_kernel<<<1, 1024, 0, st>>>(ncta, d.E, ws);
  route_scatter_kernel<<<ncta, 256, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(x), T, k, d.E, d.H, ws);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Weighted combine: out[t][d] = sum_{j<k} w[t][j] * y[pos(t,j)][d] in FP32,
// slot order j = 0..k-1, rounded once to BF16.  One thread per 8 outputs.
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
  if (kOutF32) {
    float4* o = reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + (size_t)t * H) + 2 * d8;
    o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    return;
  }
  uint32_t o[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]);
    o[q] = *reinterpret_cast<const uint32_t*>(&b2);
  }
  reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(out) + (size_t)t * H)[d8] = make_uint4(o[0], o[1], o[2], o[3]);
}

cudaError_t launch_combine(const LayerDims& d, int T, int k, const Workspace& ws, void* out, cudaStream_t st) {
  const size_t n = (size_t)T * (d.H / 8);
  if (d.out_f32)
    combine_kernel<true><<<(unsigned)((n + 255) / 256), 256, 0, st>>>(T, k, d.H, ws.y, ws.wts, ws.inv, out);
  else
    combine_kernel<false><<<(unsigned)((n + 255) / 256), 256, 0, st>>>(T, k, d.H, ws.y, ws.wts, ws.inv, out);
  return cudaGetLastError();
}

}  // namespace nvfp4moe
