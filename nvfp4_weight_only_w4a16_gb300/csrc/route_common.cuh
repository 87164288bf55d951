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
#include "kernels.h"

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

// The same in two steps, so that other loads can be issued in between.
__device__ __forceinline__ void warp_issue_logits(const void* logits, int bf16, int E, int t, float (&val)[8]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = lane + 32 * i;
    val[i] = e < E ? load_logit(logits, bf16, (size_t)t * E + e) : 0.f;
  }
}
__device__ __forceinline__ void warp_logit_keys(const float (&val)[8], uint32_t (&key)[8]) {
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

// ---------------------------------------------------------------------------
// Scoring variants (RouteParams).  s_e = softmax over all E logits, or
// sigmoid(l_e).  The choice runs on s_e + bias_e when a bias is given, else
// on the logits themselves (both scores are strictly increasing in the logit,
// so that is their exact order).  Weights: the chosen s (no bias), divided by
// their sum over the k slots when renorm (softmax: softmax over the chosen
// logits; sigmoid: 1/k each if the sum is 0), then times scale.  NaN logits
// count as -inf in the scores.
// ---------------------------------------------------------------------------
struct SoftmaxStats {
  float m;    // max logit (NaN as -inf)
  float sum;  // sum of exp(l - m) over all E (m finite)
  int ninf;   // logits equal to +inf
};

__device__ __forceinline__ SoftmaxStats warp_softmax_stats(const float (&val)[8], int E) {
  const int lane = threadIdx.x & 31;
  float m = -INFINITY;
  int ninf = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i)
    if (lane + 32 * i < E && val[i] == val[i]) {
      m = fmaxf(m, val[i]);
      ninf += val[i] == INFINITY;
    }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float sum = 0.f;
  if (m != INFINITY && m != -INFINITY) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (lane + 32 * i < E && val[i] == val[i]) sum += expf(val[i] - m);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  return SoftmaxStats{m, sum, (int)__reduce_add_sync(0xffffffffu, (unsigned)ninf)};
}

// s of one logit under the full softmax (stats over all E experts)
__device__ __forceinline__ float softmax_score(float l, const SoftmaxStats& st, int E) {
  if (l != l) return 0.f;
  if (st.m == -INFINITY) return 1.0f / (float)E;
  if (st.m == INFINITY) return l == INFINITY ? 1.0f / (float)st.ninf : 0.f;
  return expf(l - st.m) / st.sum;
}

__device__ __forceinline__ float sigmoid_score(float l) {
  if (l != l) return 0.f;
  return 1.0f / (1.0f + expf(-l));
}

// With a bias, re-key the warp's logits by s_e + bias_e (NaN logits keep the
// lowest key).  Without one the logit keys stand.
__device__ __forceinline__ void warp_bias_keys(const RouteParams& rp, int E, const float (&val)[8],
                                               uint32_t (&key)[8], const SoftmaxStats& st) {
  if (!rp.bias) return;
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = lane + 32 * i;
    if (e < E && val[i] == val[i]) {
      const float sc = rp.score ? sigmoid_score(val[i]) : softmax_score(val[i], st, E);
      key[i] = float_key(sc + __ldg(rp.bias + e));
    }
  }
}

// Lane j < k holds its chosen logit; returns its final weight (all lanes call).
__device__ __forceinline__ float warp_route_weight(const RouteParams& rp, float logit, int k, int E,
                                                   const SoftmaxStats& st) {
  const int lane = threadIdx.x & 31;
  float w;
  if (rp.score == 0 && rp.renorm) {
    w = warp_softmax_k(logit, k);
  } else {
    float s = 0.f;
    if (lane < k) s = rp.score ? sigmoid_score(logit) : softmax_score(logit, st, E);
    w = s;
    if (rp.renorm) {
      float sum = 0.f;
      for (int j = 0; j < k; ++j) sum += __shfl_sync(0xffffffffu, s, j);
      w = sum > 0.f ? s / sum : 1.0f / (float)k;
    }
  }
  return w * rp.scale;
}

// One warp routes token t (E <= 256, k <= 16).  Lane j < k receives the j-th
// choice in (*my_id, *my_w); returns the number of NaN logits of the token.
__device__ __forceinline__ int warp_topk(const void* logits, int bf16, int E, int k, int t, const RouteParams& rp,
                                         int* my_id, float* my_w) {
  uint32_t key[8];
  float val[8];
  warp_load_logits(logits, bf16, E, t, key, val);
  SoftmaxStats st{0.f, 0.f, 0};
  if (rp.score == 0 && (rp.bias || !rp.renorm)) st = warp_softmax_stats(val, E);
  warp_bias_keys(rp, E, val, key, st);
  float logit;
  const int nan = warp_select_topk(key, val, E, k, my_id, &logit);
  *my_w = warp_route_weight(rp, logit, k, E, st);
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
