// Routing primitives shared by the decode and prefill kernels.
//
// Readings (the pages do not state the scoring rule): top-k by logit, equal
// logits -> lower expert index, NaN below -inf; weights = softmax over the k
// chosen logits (NaN as -inf; all chosen -inf -> 1/k each; any +inf -> the +inf
// entries share weight 1); rows ordered expert-major, ascending t*k+j inside
// an expert.  The routers are BF16 linears ("GLM-5.3-Flash on Blackwell",
// The quantization), so their logits are this layer's input.
#pragma once
#include "common.cuh"

namespace nvfp4moe {

__device__ __forceinline__ float load_logit(const void* logits, int bf16, size_t i) {
  if (bf16) {
    const unsigned short b = reinterpret_cast<const unsigned short*>(logits)[i];
    return __uint_as_float((uint32_t)b << 16);
  }
  return reinterpret_cast<const float*>(logits)[i];
}

// Softmax over the k chosen logits of one token: lane j < k holds logit j
// (NaN counts as -inf; all -inf -> 1/k each; any +inf -> the +inf entries
// share weight 1).  Returns lane j's weight; the sum runs in slot order
// j = 0..k-1 on every lane.
__device__ __forceinline__ float warp_softmax_k(float logit, int k) {
  const int lane = threadIdx.x & 31;
  const float l = (lane < k) ? (logit != logit ? -INFINITY : logit) : -INFINITY;
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
  float sum = 0.f;
  for (int j = 0; j < k; ++j) sum += __shfl_sync(0xffffffffu, ex, j);
  return ex / sum;
}

// Lane l of a warp takes the logits e = l + 32 i (i < 8, e < E <= 256) of
// token t as order keys (float_key: larger value -> larger key, NaN lowest).
// The loads are only issued here; nothing waits for them.
__device__ __forceinline__ void warp_load_logits(const void* logits, int bf16, int E, int t, uint32_t (&key)[8],
                                                 float (&val)[8]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = lane + 32 * i;
    val[i] = e < E ? load_logit(logits, bf16, (size_t)t * E + e) : 0.f;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) key[i] = float_key(val[i]);
}

// The k largest keys of the warp (k <= min(E, 16)) in order: largest value
// first, the lower expert index first among equal values.  Each round takes
// the warp maximum key (redux.sync), then the lowest index holding it.  Lane
// j < k receives choice j in (*my_id, *my_logit); returns the token's NaN
// count.
__device__ __forceinline__ int warp_select_topk(const uint32_t (&key)[8], const float (&val)[8], int E, int k,
                                                int* my_id, float* my_logit) {
  const int lane = threadIdx.x & 31;
  unsigned avail = 0;
  int nan = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i)
    if (lane + 32 * i < E) {
      avail |= 1u << i;
      nan += (val[i] != val[i]);
    }
  int id = -1;
  float logit = 0.f;
  for (int j = 0; j < k; ++j) {
    uint32_t bk = 0;
    int bi = -1;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (((avail >> i) & 1u) && (bi < 0 || key[i] > bk)) {
        bk = key[i];
        bi = i;
      }
    const uint32_t M = __reduce_max_sync(0xffffffffu, bk);
    const uint32_t cand = (bi >= 0 && bk == M) ? (uint32_t)(lane + 32 * bi) : 0xFFFFu;
    const uint32_t win = __reduce_min_sync(0xffffffffu, cand);
    float v = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (bi == i) v = val[i];
    v = __shfl_sync(0xffffffffu, v, (int)(win & 31u));
    if (lane == (int)(win & 31u)) avail &= ~(1u << (win >> 5));
    if (lane == j) {
      id = (int)win;
      logit = v;
    }
  }
  *my_id = id;
  *my_logit = logit;
  return (int)__reduce_add_sync(0xffffffffu, (unsigned)nan);
}

// One warp routes token t (E <= 256, k <= 16).  Lane j < k receives the j-th
// choice in (*my_id, *my_w); returns the number of NaN logits of the token.
__device__ __forceinline__ int warp_topk(const void* logits, int bf16, int E, int k, int t, int* my_id,
                                         float* my_w) {
  uint32_t key[8];
  float val[8];
  warp_load_logits(logits, bf16, E, t, key, val);
  float logit;
  const int nan = warp_select_topk(key, val, E, k, my_id, &logit);
  *my_w = warp_softmax_k(logit, k);
  return nan;
}

// Exclusive scan of v over the block (<= 1024 threads, all call); *total gets
// the sum.
__device__ __forceinline__ int block_exclusive_scan(int v, int* smem_warp /*[32]*/, int* total) {
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

}  // namespace nvfp4moe
