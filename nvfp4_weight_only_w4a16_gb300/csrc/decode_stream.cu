// Decode path (1..16 tokens): one cooperative persistent kernel, one CTA per
// SM, that routes the tokens and streams every touched expert's NVFP4 weights
// from HBM once, through the gate/up GEMV with SwiGLU, the down GEMV and the
// weighted combine.
//
// At decode sizes the layer is a weight stream: every expert a token picks is
// read from HBM once per step -- "the memory-bandwidth wall for an 18B-active
// model" ("GLM-5.3-Flash on Blackwell", Two deployments, and the lever that
// reverses between them).  The weight-only path never takes an activation
// scale: weights are dequantised to 16-bit and multiplied with the 16-bit
// activations (same page, The model loaded, served an API, and produced
// garbage).
//
// Design (GB300):
//  * routing first, in every CTA: the logits (or, with a router weight, the
//    router linear itself, each CTA a share of the experts, counted in) go
//    through a warp top-k per token; one warp's scan builds the touched-expert
//    list, and the producer starts on it while the other warps finish the
//    permutation tables; warps that route no token meanwhile convert this
//    CTA's share of x into 16-bit chunk rows in global memory;
//  * work items are claimed dynamically from one global counter: first every
//    gate/up item (expert u, 128 packed rows = 64 features, all of K = H),
//    then every down item (expert u, 128 output rows, all of K = I), each
//    group expert-major.  A CTA's first item is its index, later ones come
//    from the counter (claimed one item ahead, so the atomic's latency hides
//    behind the current item).  Fast SMs simply take more items; a down item
//    waits (bounded) until every chunk of its expert's h is published;
//  * one producer warp per CTA streams each item through a shared-memory ring
//    of stages of eight 64-wide K chunks: one cp.async.bulk of the chunks'
//    packed tiles (codes and scales, 36 KB, with an L2 evict_first hint: the
//    weights are read once per step) and one of their activation rows,
//    completed on mbarriers;
//  * two groups of 8 consumer warps take alternate stages; warp sb of a group
//    takes 16-row group sb of each chunk, dequantises in registers (hardware
//    E2M1 -> FP16 converts times the E4M3 group scale, exact) and runs
//    mma.sync m16n8k16 (FP16 in, FP32 accumulate); at an item's end the two
//    groups' partial sums meet in shared memory and one warp runs the
//    epilogue (gate/up: SwiGLU into h rows; down: FP32 y rows);
//  * activations enter the MMA as FP16 rows of one 64-wide chunk with their
//    own power-of-two scale (the chunk's largest magnitude in [2^13, 2^14):
//    exact for every value within 2^31 of it that has at most 11 significant
//    bits), stored next to the row; each chunk's partial sums are multiplied
//    back by the scale in FP32.  The gate/up epilogue of an item produces one
//    whole chunk of h (its 64 features) in that form: FP16, 11 significant
//    bits;
//  * gate/up columns are the step's tokens (every token through every touched
//    expert's MMA columns; only the routed ones are kept), down columns are
//    the expert's routed rows;
//  * a signal warp publishes finished items (a fence, then a count per
//    (expert, chunk) of h or per 128-wide output slice), so no consumer waits
//    on its own fence; up to 4 tokens the signal warp that completes a slice
//    for the last touched expert combines it, above that every consumer warp
//    takes (slice, token) tasks once the work runs out; the k slots are summed
//    in slot order;
//  * every wait is bounded (2 s): a wait that gives up records a timeout in the
//    status word and the kernel unwinds without a trap.
#include <cstdlib>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "route_common.cuh"

namespace nvfp4moe {

namespace dstr {
constexpr int kGroupWarps = 8;                    // consumer warps of a group: one per 16-row group of a block
constexpr int kGroups = 2;                        // consumer groups, taking alternate stages
constexpr int kConsumers = kGroups * kGroupWarps;
constexpr int kThreads = (kConsumers + 2) * 32;   // + one producer warp + one signal warp
constexpr int kProducer = kConsumers;             // the producer's warp index
constexpr int kSignaller = kConsumers + 1;        // the signal warp's index
constexpr int kSig = 8;                           // depth of each group's completion queue
constexpr int kSigCombineT = 4;                   // up to this many tokens the signal warp that completes
                                                  // an output slice combines it; beyond, every consumer warp
#ifndef NVFP4_MOE_DEC_CPS
#define NVFP4_MOE_DEC_CPS 8
#endif
constexpr int kCPS = NVFP4_MOE_DEC_CPS;           // 64-wide K chunks per stage (at most): 4 or 8
constexpr int kAct = kCPS * kTileBytes;          // after the stage's weight tiles (codes + scales): its activation rows
constexpr int kRow = 144;                         // one activation row of a chunk: 64 FP16, float scale at +128
constexpr int kMaxSlots = 17;                     // slots per token: top_k <= 16 + one shared expert
constexpr int kMaxR = kDecodeMaxTokens * kMaxSlots;
constexpr int kMaxE = 288;                        // routed + shared experts (9 per lane in the scan)
constexpr int kMaxStages = 12;
constexpr int kXChunks = 8;                       // chunks of x one CTA converts with its loads issued up front
constexpr uint64_t kTimeoutNs = 2000000000ull;
}  // namespace dstr

struct StreamSmem {
  int ids[dstr::kMaxR];
  float wts[dstr::kMaxR];
  int perm[dstr::kMaxR];
  int inv[dstr::kMaxR];
  int off[dstr::kMaxE + 1];
  int slot_of[dstr::kMaxE];  // expert -> touched slot
  int tch_e[dstr::kMaxE];
  int tch_r0[dstr::kMaxE];
  int tch_m[dstr::kMaxE];
  unsigned tch_mask[dstr::kMaxE];  // tokens routed to the touched expert
  float cmax[2][2][8][16];          // gate/up epilogue, [parity][group]: per 16-row group, per column, max |h|
  int epi_cnt[2];                   // per group: warps arrived at its gate/up epilogues (8 per epilogue)
  int meta[dstr::kMaxStages][4];   // item, stage within the item, chunks in the stage
  float rpart[dstr::kConsumers][16];  // router linear: per consumer warp, per token
  int sig[2][dstr::kSig];          // per group: completed items for the signal warp (-1: no more)
  int U, nan, last_cta;
  alignas(8) uint64_t full[dstr::kMaxStages];
  alignas(8) uint64_t empty[dstr::kMaxStages];
  alignas(8) uint64_t sig_full[2][dstr::kSig];   // the group's warps are done with the item
  alignas(8) uint64_t sig_empty[2][dstr::kSig];  // the signal warp has published it
  alignas(8) uint64_t red_full[2][8];            // [item parity][16-row group]: the helper's half is in
  alignas(8) uint64_t red_empty[2][8];           // the owner has taken it
};

struct StreamArgs {
  const uint8_t* blob;
  size_t expert_stride, w13, w2;  // an expert's bytes; its gate/up and down matrices' offsets
  const float* gscale;
  int E, Er, H, I, T, k, topk;  // E experts in the blob, k slots per token (top_k + shared)
  RouteParams rp;
  const void* logits;
  int logits_bf16;
  int linear;                     // 1: a dense linear out = gs W x (one "expert", down matrix only, x [T][I])
  int n_out;                      // a dense linear's output features (out is [T][n_out])
  const __nv_bfloat16* router_w;  // BF16 [Er][H]: the kernel computes the logits (else NULL)
  float* logits_w;                // [T][Er] FP32: where it writes them
  int32_t* logit_ready;           // experts whose logits are written (reset by the last CTA)
  const __nv_bfloat16* x;
  void* out;
  int out_f32;
  int route_only;
  int32_t* ids;
  float* wts;
  int32_t* offsets;
  int32_t* perm;
  int32_t* inv;
  uint8_t* act_h;     // h rows, FP16 with their scale: touched expert u's m rows from row0 form
                      // block [I/64][m][kRow] at row0 * I/64 rows
  uint8_t* act_x;     // [H/64][T][kRow]: x rows per chunk
  int rdec;           // rows of act_h per chunk
  float* y;           // [R][H] expert outputs, position order
  int32_t* wctr;      // claimed items beyond the first gridDim.x
  int32_t* done_c;    // [maxU][I/64]: 1 once (touched expert, chunk of h) is written
  int32_t* cmb;       // finished down items per 128-wide output slice
  int32_t* x_ready;   // tokens converted per chunk of x (act_x)
  int32_t* exit_cnt;
  DeviceStatus* st;
  DeviceStatus* st_sticky;
  int fault;          // 1: the producer issues nothing (tests the bounded waits)
  int stages, stage_bytes;
  int checks;         // 1: check table-derived indices (kFlagBounds; the access is skipped)
  int cps;            // 64-wide K chunks per stage (kCPS, or fewer for small H and I: two or more stages per item)
  unsigned long long* trace;  // optional: [cta][16] phase stamps (see decode_stream_kernel)
};

namespace {

__device__ __forceinline__ uint32_t saddr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void mb_init(uint64_t* b, uint32_t n) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(b)), "r"(n) : "memory");
}
__device__ __forceinline__ void mb_arrive(uint64_t* b) {
  asm volatile("{\n .reg .b64 s;\n mbarrier.arrive.shared::cta.b64 s, [%0];\n}" ::"r"(saddr(b)) : "memory");
}
__device__ __forceinline__ void mb_expect(uint64_t* b, uint32_t bytes) {
  asm volatile("{\n .reg .b64 s;\n mbarrier.arrive.expect_tx.shared::cta.b64 s, [%0], %1;\n}" ::"r"(saddr(b)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mb_try(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(saddr(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   saddr(dst)),
               "l"(src), "r"(bytes), "r"(saddr(bar))
               : "memory");
}
// The same copy with an L2 eviction-priority hint.  The weight tiles are read once per
// step, so they take evict_first: L2 gives up their lines before those of the rows every
// CTA keeps re-reading (x, h, the routing tables).  Measured on the MTP and 16-token steps:
// ~2-3 us less per step than with the default policy.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          saddr(dst)),
      "l"(src), "r"(bytes), "r"(saddr(bar)), "l"(pol)
      : "memory");
}
__device__ __forceinline__ uint64_t gtime() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ int ld_acq(const int32_t* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ bool is_aborted(const DeviceStatus* st) {
  return (*reinterpret_cast<const volatile unsigned*>(&st->flags) & kFlagTimeout) != 0;
}
__device__ __forceinline__ float exp2i(int p) { return __int_as_float((127 + max(-126, min(127, p))) << 23); }

// Bounded wait on an mbarrier phase; false after a timeout (recorded at
// `where`) or once another thread has recorded one.  A phase that has
// completed is always seen, even after an abort.
__device__ bool wait_phase(uint64_t* b, uint32_t parity, DeviceStatus* st, unsigned where) {
  if (mb_try(b, parity)) return true;
  const uint64_t t0 = gtime();
  for (uint32_t i = 0;; ++i) {
    if (mb_try(b, parity)) return true;
    if ((i & 31u) == 31u) {
      if (is_aborted(st)) return false;
      if (gtime() - t0 > dstr::kTimeoutNs) {
        report(st, kFlagTimeout, where);
        return false;
      }
    }
  }
}

// Bounded wait until *p >= target (acquire).  False after a timeout or abort.
__device__ bool wait_count(const int32_t* p, int target, DeviceStatus* st, unsigned where) {
  if (ld_acq(p) >= target) return true;
  const uint64_t t0 = gtime();
  for (;;) {
    if (ld_acq(p) >= target) return true;
    if (is_aborted(st)) return false;
    if (gtime() - t0 > dstr::kTimeoutNs) {
      report(st, kFlagTimeout, where);
      return false;
    }
    __nanosleep(64);
  }
}

// Bounded wait, by the whole warp, until p[i] >= target for every i < n: each
// lane polls its own flags (acquire), so all of them cost one round trip.
// Warp-uniform result; false after a timeout or abort.
__device__ bool warp_wait_all(const int32_t* p, int n, int target, DeviceStatus* st, unsigned where) {
  const int lane = threadIdx.x & 31;
  bool ok = true;
  for (int i = lane; i < n && ok; i += 32) ok = wait_count(p + i, target, st, where);
  return __all_sync(0xffffffffu, ok);
}

// One 64-element chunk of an activation row -> FP16 scaled by 2^-p, with p
// such that the chunk's largest magnitude lands in [2^13, 2^14); lane l holds
// elements 2l and 2l+1 (BF16 bits in one word).  Writes the row (128 B) and
// its scale 2^p (float at +128) to dst.
__device__ __forceinline__ void convert_chunk_row(uint32_t two_bf16, uint8_t* dst, int lane) {
  const float lo = __uint_as_float(two_bf16 << 16), hi = __uint_as_float(two_bf16 & 0xFFFF0000u);
  const unsigned m = __reduce_max_sync(0xffffffffu, max(__float_as_uint(fabsf(lo)), __float_as_uint(fabsf(hi))));
  const int p = max(-126, min(126, prescale_exp(__uint_as_float(m))));
  const float s = exp2i(-p);
  const __half2 hh = __floats2half2_rn(lo * s, hi * s);
  *reinterpret_cast<__half2*>(dst + 4 * lane) = hh;
  if (lane == 0) *reinterpret_cast<float*>(dst + 128) = exp2i(p);
}

}  // namespace

// ---------------------------------------------------------------------------
// Routing: every CTA routes the T tokens into shared memory (warp w picks the
// experts of tokens w, w + 9), builds the expert-major tables and the
// touched-expert list with each expert's token mask.  CTA 0 also writes the
// tables out.
// ---------------------------------------------------------------------------
// The router linear inside the kernel: CTA c computes the logits of experts
// c, c + grid, ... for every token (logit = sum_h x[t][h] * W_r[e][h] in FP32,
// BF16 inputs; the 16 consumer warps split H, then sum in warp order), writes
// them to logits_w, and counts them in; every CTA then waits (bounded) until
// all Er experts' logits are in.  All threads of the CTA call it.
__device__ void stream_router(const StreamArgs& a, StreamSmem& ss) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, T = a.T, H = a.H;
  int mine = 0;
  for (int e = blockIdx.x; e < a.Er; e += gridDim.x, ++mine) {
    if (warp < dstr::kConsumers) {
      float acc[16];
#pragma unroll
      for (int t = 0; t < 16; ++t) acc[t] = 0.f;
      const uint4* wr = reinterpret_cast<const uint4*>(a.router_w + (size_t)e * H);
      for (int p = tid; p < H / 8; p += dstr::kConsumers * 32) {
        const uint4 wv = __ldg(wr + p);
        const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
        for (int t = 0; t < 16; ++t) {
          if (t >= T) break;
          const uint4 xv = __ldg(reinterpret_cast<const uint4*>(a.x + (size_t)t * H) + p);
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
        if (t >= T) break;
        float v = acc[t];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) ss.rpart[warp][t] = v;
      }
    }
    __syncthreads();
    if (tid < T) {
      float v = 0.f;
      for (int w = 0; w < dstr::kConsumers; ++w) v += ss.rpart[w][tid];
      a.logits_w[(size_t)tid * a.Er + e] = v;
      __threadfence();
    }
    __syncthreads();
  }
  if (tid == 0) {
    if (mine) atomicAdd(a.logit_ready, mine);
    wait_count(a.logit_ready, a.Er, a.st, 900);
  }
  __syncthreads();
}

// A dense linear's tables, every CTA: one touched "expert" holding all T rows in token
// order with weight 1.  `mid` as in stream_route.
template <class Mid>
__device__ void stream_route_linear(const StreamArgs& a, StreamSmem& ss, Mid&& mid) {
  const int tid = threadIdx.x, T = a.T;
  if (tid == 0) {
    ss.U = 1;
    ss.nan = 0;
    ss.off[0] = 0;
    ss.off[1] = T;
    ss.slot_of[0] = 0;
    ss.tch_e[0] = 0;
    ss.tch_r0[0] = 0;
    ss.tch_m[0] = T;
    ss.tch_mask[0] = T >= 32 ? ~0u : (1u << T) - 1u;
  }
  if (tid < T) {
    ss.ids[tid] = 0;
    ss.wts[tid] = 1.0f;
    ss.perm[tid] = tid;
    ss.inv[tid] = tid;
  }
  mid();
  __syncthreads();
}

// The logit loads of this warp's tokens (issued first thing, so their latency
// overlaps everything else the kernel does before routing).
__device__ __forceinline__ void stream_route_issue(const StreamArgs& a, float (&val)[2][8]) {
  const int warp = threadIdx.x >> 5, nw = blockDim.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int t = warp + r * nw;
    if (t >= a.T) continue;
    if (a.router_w) {  // written by this kernel's other CTAs: read from L2
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int e = lane + 32 * i;
        val[r][i] = e < a.Er ? __ldcg(a.logits_w + (size_t)t * a.Er + e) : 0.f;
      }
    } else {
      warp_issue_logits(a.logits, a.logits_bf16, a.Er, t, val[r]);
    }
  }
}

// `mid` runs on every thread between the expert choice and the tables (the
// warps that choose no experts do their other early work there).  Warp
// `early` (or none: -1) leaves as soon as the touched-expert list is built --
// the weight producer needs nothing else -- and the other warps finish the
// tables behind a named barrier.
template <class Mid>
__device__ void stream_route(const StreamArgs& a, StreamSmem& ss, float (&val)[2][8], unsigned long long* tr,
                             Mid&& mid, int early) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nw = blockDim.x >> 5;
  const int T = a.T, k = a.k, E = a.E, Er = a.Er, topk = a.topk, R = T * k;
  uint32_t key[2][8];
  for (int i = tid; i <= E; i += blockDim.x) ss.off[i] = 0;
  if (tid == 0) ss.nan = 0;
  __syncthreads();
  if (tr && tid == 0) tr[14] = gtime();
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int t = warp + r * nw;
    if (t >= T) continue;
    warp_logit_keys(val[r], key[r]);
    int id;
    float logit;
    SoftmaxStats sst{0.f, 0.f, 0};
    if (a.rp.score == 0 && (a.rp.bias || !a.rp.renorm)) sst = warp_softmax_stats(val[r], Er);
    warp_bias_keys(a.rp, Er, val[r], key[r], sst);
    const int nt = warp_select_topk(key[r], val[r], Er, topk, &id, &logit);
    const float w = warp_route_weight(a.rp, logit, topk, Er, sst);
    if (a.checks && lane < topk && (id < 0 || id >= Er)) {
      report(a.st, kFlagBounds, 800);
      id = 0;
    }
    if (lane < topk) {
      ss.ids[t * k + lane] = id;
      ss.wts[t * k + lane] = w;
      atomicAdd(&ss.off[id], 1);
    } else if (lane < k) {  // the shared expert: every token, weight 1
      ss.ids[t * k + lane] = Er;
      ss.wts[t * k + lane] = 1.0f;
      atomicAdd(&ss.off[Er], 1);
    }
    if (lane == 0 && nt) atomicAdd(&ss.nan, nt);
  }
  mid();
  __syncthreads();
  if (tr && tid == 0) tr[15] = gtime();
  if (warp == 0) {
    // offsets (low 16 bits) and touched slots (high 16 bits) in one warp scan;
    // lane l owns experts 9l .. 9l+8
    int cnt[9], s = 0, tc = 0;
#pragma unroll
    for (int i = 0; i < 9; ++i) {
      const int e = 9 * lane + i;
      cnt[i] = e < E ? ss.off[e] : 0;
      s += cnt[i];
      tc += cnt[i] > 0;
    }
    const int v = s | (tc << 16);
    int inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    const int ex = inc - v;
    int off = ex & 0xFFFF, slot = ex >> 16;
#pragma unroll
    for (int i = 0; i < 9; ++i) {
      const int e = 9 * lane + i;
      if (e < E) {
        ss.off[e] = off;
        if (cnt[i] > 0) {
          ss.slot_of[e] = slot;
          ss.tch_e[slot] = e;
          ss.tch_r0[slot] = off;
          ss.tch_m[slot] = cnt[i];
          ss.tch_mask[slot] = 0u;
          ++slot;
        }
        off += cnt[i];
      }
    }
    if (lane == 31) {
      ss.off[E] = inc & 0xFFFF;
      ss.U = inc >> 16;
    }
  }
  __syncthreads();
  if (warp == early) return;
  // the remaining threads, renumbered without warp `early`
  const int nthr = (int)blockDim.x - (early >= 0 ? 32 : 0);
  const int idx = (early >= 0 && warp > early) ? tid - 32 : tid;
  for (int r = idx; r < R; r += nthr) {  // expert-major position: rank among the earlier rows of the same expert
    const int e = ss.ids[r];
    int rank = 0;
    for (int j = 0; j < r; ++j) rank += (ss.ids[j] == e);
    const int pos = ss.off[e] + rank;
    ss.perm[pos] = r;
    ss.inv[r] = pos;
    atomicOr(&ss.tch_mask[ss.slot_of[e]], 1u << (r / k));
  }
  if (early >= 0) asm volatile("bar.sync 3, %0;" ::"r"(nthr) : "memory");
  else __syncthreads();
  if (blockIdx.x == 0) {  // the tables, for inspection
    for (int i = idx; i < R; i += nthr) {
      a.ids[i] = ss.ids[i];
      a.wts[i] = ss.wts[i];
      a.perm[i] = ss.perm[i];
      a.inv[i] = ss.inv[i];
    }
    for (int i = idx; i <= E; i += nthr) a.offsets[i] = ss.off[i];
    if (idx == 0 && ss.nan) atomicAdd(&a.st->nan_logits, (unsigned)ss.nan);
  }
}

// ---------------------------------------------------------------------------
// One consumer warp's share of a stage: its 16-row group of each chunk,
// dequantised and multiplied with the chunk's activation rows.
// ---------------------------------------------------------------------------
// The A side of one chunk: the lane's 16-byte MMA fragment of codes times its
// two E4M3 group scales, as 16 FP16 pairs (rows g and g+8, K elements 16q..+15).
struct AFrag {
  uint32_t x[4], y[4], z[4], w[4];
};
__device__ __forceinline__ void load_a(const uint8_t* codes, const uint8_t* scales, int lane, AFrag& f) {
  const uint4 raw = *reinterpret_cast<const uint4*>(codes + lane * 16);
  const uint32_t s2 = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(scales + lane * 2));
  const uint32_t s0 = dup_lo(s2), s1 = dup_hi(s2);
  e2m1x8_to_f16x2x4(raw.x, f.x);
  e2m1x8_to_f16x2x4(raw.y, f.y);
  e2m1x8_to_f16x2x4(raw.z, f.z);
  e2m1x8_to_f16x2x4(raw.w, f.w);
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    f.x[t] = hmul2_u32(f.x[t], s0);
    f.y[t] = hmul2_u32(f.y[t], s0);
    f.z[t] = hmul2_u32(f.z[t], s1);
    f.w[t] = hmul2_u32(f.w[t], s1);
  }
}

// tile: the chunk's activation rows, kRow bytes apart, 8 NG of them.  Rows
// past the valid ones hold whatever the buffer held (in shared memory: any
// bits); they only ever reach their own MMA columns, which no epilogue keeps
// (an MMA's output column n depends on column n of B alone).
template <int NG>
__device__ __forceinline__ void mma_tile(const AFrag& f, const uint8_t* tile, float (&acc)[NG][4], int lane) {
  const int g = lane >> 2, q = lane & 3;
#pragma unroll
  for (int gi = 0; gi < NG; ++gi) {
    const uint8_t* pb = tile + (8 * gi + g) * dstr::kRow + q * 32;
    const uint4 b0 = *reinterpret_cast<const uint4*>(pb), b1 = *reinterpret_cast<const uint4*>(pb + 16);
    const int c0 = 8 * gi + 2 * q;
    const float sc0 = *reinterpret_cast<const float*>(tile + c0 * dstr::kRow + 128);
    const float sc1 = *reinterpret_cast<const float*>(tile + (c0 + 1) * dstr::kRow + 128);
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    mma_f16_16816(d, f.x[0], f.z[0], f.x[1], f.z[1], b0.x, b0.y);
    mma_f16_16816(d, f.x[2], f.z[2], f.x[3], f.z[3], b0.z, b0.w);
    mma_f16_16816(d, f.y[0], f.w[0], f.y[1], f.w[1], b1.x, b1.y);
    mma_f16_16816(d, f.y[2], f.w[2], f.y[3], f.w[3], b1.z, b1.w);
    acc[gi][0] = fmaf(d[0], sc0, acc[gi][0]);
    acc[gi][1] = fmaf(d[1], sc1, acc[gi][1]);
    acc[gi][2] = fmaf(d[2], sc0, acc[gi][2]);
    acc[gi][3] = fmaf(d[3], sc1, acc[gi][3]);
  }
}

// One stage's raw operands for consumer warp sb, in registers: its 16-row
// group's codes and scales of each of the NC chunks, and each chunk's
// activation fragments (B) with their column scales.  Once they are loaded
// the stage's shared memory can be refilled while the warp computes.
template <int NG, int NC>
struct StageRegs {
  uint4 raw[NC];
  uint16_t sc[NC];
  uint4 b[NC][NG][2];
  float cs[NC][NG][2];
};
// The stage carries each chunk's activation rows, `pitch` bytes apart (T rows
// of kRow bytes); reads past a chunk's rows land in the next chunk's rows or
// the ring's tail pad -- MMA columns that no epilogue keeps.
template <int NG, int NC>
__device__ __forceinline__ void load_stage(const uint8_t* stg, int cb, int pitch, int sb, int lane,
                                           StageRegs<NG, NC>& r) {
  const int g = lane >> 2, q = lane & 3;
#pragma unroll
  for (int c = 0; c < NC; ++c) {  // the stage's chunk cb + c
    r.raw[c] = *reinterpret_cast<const uint4*>(stg + (cb + c) * kTileBytes + sb * 512 + seg_pos(lane) * 16);
    r.sc[c] =
        *reinterpret_cast<const uint16_t*>(stg + (cb + c) * kTileBytes + kTileCodes + sb * 64 + seg_pos(lane) * 2);
    const uint8_t* tile = stg + dstr::kAct + (cb + c) * pitch;
#pragma unroll
    for (int gi = 0; gi < NG; ++gi) {
      const uint8_t* pb = tile + (8 * gi + g) * dstr::kRow + q * 32;
      r.b[c][gi][0] = *reinterpret_cast<const uint4*>(pb);
      r.b[c][gi][1] = *reinterpret_cast<const uint4*>(pb + 16);
      const int c0 = 8 * gi + 2 * q;
      r.cs[c][gi][0] = *reinterpret_cast<const float*>(tile + c0 * dstr::kRow + 128);
      r.cs[c][gi][1] = *reinterpret_cast<const float*>(tile + (c0 + 1) * dstr::kRow + 128);
    }
  }
}
template <int NG, int NC>
__device__ __forceinline__ void compute_stage(const StageRegs<NG, NC>& r, float (&acc)[NG][4]) {
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    AFrag f;
    const uint32_t s2 = e4m3x2_to_f16x2(r.sc[c]);
    const uint32_t s0 = dup_lo(s2), s1 = dup_hi(s2);
    e2m1x8_to_f16x2x4(r.raw[c].x, f.x);
    e2m1x8_to_f16x2x4(r.raw[c].y, f.y);
    e2m1x8_to_f16x2x4(r.raw[c].z, f.z);
    e2m1x8_to_f16x2x4(r.raw[c].w, f.w);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      f.x[t] = hmul2_u32(f.x[t], s0);
      f.y[t] = hmul2_u32(f.y[t], s0);
      f.z[t] = hmul2_u32(f.z[t], s1);
      f.w[t] = hmul2_u32(f.w[t], s1);
    }
#pragma unroll
    for (int gi = 0; gi < NG; ++gi) {
      const uint4 b0 = r.b[c][gi][0], b1 = r.b[c][gi][1];
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      mma_f16_16816(d, f.x[0], f.z[0], f.x[1], f.z[1], b0.x, b0.y);
      mma_f16_16816(d, f.x[2], f.z[2], f.x[3], f.z[3], b0.z, b0.w);
      mma_f16_16816(d, f.y[0], f.w[0], f.y[1], f.w[1], b1.x, b1.y);
      mma_f16_16816(d, f.y[2], f.w[2], f.y[3], f.w[3], b1.z, b1.w);
      acc[gi][0] = fmaf(d[0], r.cs[c][gi][0], acc[gi][0]);
      acc[gi][1] = fmaf(d[1], r.cs[c][gi][1], acc[gi][1]);
      acc[gi][2] = fmaf(d[2], r.cs[c][gi][0], acc[gi][2]);
      acc[gi][3] = fmaf(d[3], r.cs[c][gi][1], acc[gi][3]);
    }
  }
}

// Gate/up epilogue of item (u, b) on the 8 consumer warps (16-row group sb):
// h for the 64 features of chunk b, kept for the routed tokens, as the FP16
// chunk rows with their scale in act_h (published by the signal warp).
template <int NG>
__device__ void epilogue_gateup(const StreamArgs& a, StreamSmem& ss, int u, int b, int sb, int grp,
                                const float (&acc)[NG][4], int lane, uint32_t nepi) {
  const int par = (int)(nepi & 1u);  // this group's nepi-th gate/up epilogue
  const int e = ss.tch_e[u], row0 = ss.tch_r0[u], m_u = ss.tch_m[u];
  const unsigned mask = ss.tch_mask[u];
  const int g = lane >> 2, q = lane & 3;
  const float gsg = __ldg(a.gscale + 3 * e), gsu = __ldg(a.gscale + 3 * e + 1);
  float hv[NG][2];
#pragma unroll
  for (int gi = 0; gi < NG; ++gi)
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int t = 8 * gi + 2 * q + c;
      const bool keep = t < a.T && ((mask >> t) & 1u);
      // packed rows 16 sb + r: gate feature 8 sb + r (r < 8), up feature 8 sb + r - 8
      const float gg = gsg * acc[gi][c], uu = gsu * acc[gi][2 + c];
      hv[gi][c] = silu(gg) * uu;
      float m = keep ? fabsf(hv[gi][c]) : 0.f;
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
      if (g == 0) ss.cmax[par][grp][sb][t] = m;
    }
  // every warp of the group has written its maxima: an arrival count in shared memory, with a
  // bounded wait (a peer that gave up on a timed-out stage must not hang the others); the
  // maxima alternate between two buffers, so a warp one epilogue ahead writes the other one
  __threadfence_block();
  __syncwarp();
  if (lane == 0) {
    atomicAdd(&ss.epi_cnt[grp], 1);
    const int target = dstr::kGroupWarps * (int)(nepi + 1u);
    const uint64_t t0 = gtime();
    while (*reinterpret_cast<volatile int*>(&ss.epi_cnt[grp]) < target) {
      if (gtime() - t0 > dstr::kTimeoutNs) {
        report(a.st, kFlagTimeout, 340);
        break;
      }
    }
  }
  __syncwarp();
  __threadfence_block();
#pragma unroll
  for (int gi = 0; gi < NG; ++gi)
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int t = 8 * gi + 2 * q + c;
      if (t >= a.T || !((mask >> t) & 1u)) continue;
      float m = 0.f;
#pragma unroll
      for (int s = 0; s < 8; ++s) m = fmaxf(m, ss.cmax[par][grp][s][t]);
      const int p = max(-126, min(126, prescale_exp(m)));
      const int pos = row0 + __popc(mask & ((1u << t) - 1u));
      if (a.checks && (pos < 0 || pos >= a.T * a.k || pos - row0 >= m_u)) {
        report(a.st, kFlagBounds, 802);
        continue;
      }
      const int f = 8 * sb + g;  // feature within the chunk
      // the expert's rows are one block, chunk-major: [I/64][m][row]
      uint8_t* row = a.act_h + ((size_t)row0 * (a.I / 64) + (size_t)b * m_u + (pos - row0)) * dstr::kRow;
      *reinterpret_cast<__half*>(row + 2 * f) = __float2half_rn(hv[gi][c] * exp2i(-p));
      if (sb == 0 && g == 0) *reinterpret_cast<float*>(row + 128) = exp2i(p);
    }
  // the rows are read by other CTAs' bulk copies (the async proxy)
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Down epilogue of item (u, b): y rows 128 b + 16 sb + g (+8) for the
// expert's routed rows (counted in for output slice b by the signal warp);
// a dense linear (kLin) writes its output rows instead.
template <int NG, bool kLin>
__device__ void epilogue_down(const StreamArgs& a, const StreamSmem& ss, int u, int b, int sb,
                              const float (&acc)[NG][4], int lane) {
  const int e = ss.tch_e[u], row0 = ss.tch_r0[u], m = ss.tch_m[u];
  const int g = lane >> 2, q = lane & 3;
  const float gsd = __ldg(a.gscale + 3 * e + 2);
  const int d0 = 128 * b + 16 * sb + g;
#pragma unroll
  for (int gi = 0; gi < NG; ++gi)
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int j = 8 * gi + 2 * q + c;
      if (kLin && j < m) {  // a dense linear: row j is token j, written straight to out
#pragma unroll
        for (int h8 = 0; h8 < 2; ++h8) {
          const int d = d0 + 8 * h8;
          if (d >= a.n_out) continue;
          const float v = acc[gi][2 * h8 + c] * gsd;
          if (a.out_f32) reinterpret_cast<float*>(a.out)[(size_t)j * a.n_out + d] = v;
          else reinterpret_cast<__nv_bfloat16*>(a.out)[(size_t)j * a.n_out + d] = __float2bfloat16_rn(v);
        }
      } else if (!kLin && j < m) {
        float* yr = a.y + (size_t)(row0 + j) * a.H;
        yr[d0] = acc[gi][c] * gsd;
        yr[d0 + 8] = acc[gi][2 + c] * gsd;
      }
    }
}

// The combine of one 128-wide output slice b for token t, on one warp (lane l:
// features 128 b + 4l .. 4l+3): out[t][slice] = sum_j w[t][j] * y[pos(t, j)][slice]
// in slot order j = 0..k-1.  The caller has seen slice b complete for every
// touched expert (U down items counted in, then a fence).
__device__ void combine_slice(const StreamArgs& a, const StreamSmem& ss, int b, int t, int lane) {
  const int d = 128 * b + 4 * lane;
  float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
  for (int j0 = 0; j0 < a.k; j0 += 4) {  // four slots' loads in flight at a time
    float4 yy[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (j0 + u < a.k) {
        int pos = ss.inv[t * a.k + j0 + u];
        if (a.checks && (pos < 0 || pos >= a.T * a.k)) {
          report(a.st, kFlagBounds, 803);
          pos = 0;
        }
        yy[u] = __ldcg(reinterpret_cast<const float4*>(a.y + (size_t)pos * a.H + d));
      }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (j0 + u < a.k) {
        const float w = ss.wts[t * a.k + j0 + u];
        s0 = fmaf(w, yy[u].x, s0);
        s1 = fmaf(w, yy[u].y, s1);
        s2 = fmaf(w, yy[u].z, s2);
        s3 = fmaf(w, yy[u].w, s3);
      }
  }
  if (a.out_f32) {
    *reinterpret_cast<float4*>(reinterpret_cast<float*>(a.out) + (size_t)t * a.H + d) = make_float4(s0, s1, s2, s3);
  } else {
    const __nv_bfloat162 p0 = __floats2bfloat162_rn(s0, s1), p1 = __floats2bfloat162_rn(s2, s3);
    uint2 v;
    v.x = *reinterpret_cast<const uint32_t*>(&p0);
    v.y = *reinterpret_cast<const uint32_t*>(&p1);
    *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(a.out) + (size_t)t * a.H + d) = v;
  }
}

// For more than kSigCombineT tokens the combine is spread over every consumer
// warp of the grid instead: task (slice b, token t) waits until slice b is
// complete for every touched expert, then combines it.
__device__ void combine_tasks(const StreamArgs& a, const StreamSmem& ss, int wg, int W, int lane) {
  const int nsl = a.H / 128;
  for (int task = wg; task < nsl * a.T; task += W) {
    const int t = task / nsl, b = task - t * nsl;
    int ok = 1;
    if (lane == 0) ok = wait_count(a.cmb + b, ss.U, a.st, 400 + (unsigned)b);
    if (!__shfl_sync(0xffffffffu, ok, 0)) return;
    __threadfence();
    combine_slice(a, ss, b, t, lane);
  }
}

// ---------------------------------------------------------------------------
// The kernel.  Shared memory: StreamSmem | pair sums | ring
// [stages][stage_bytes].
// ---------------------------------------------------------------------------
// kLin: a dense linear (down-only, no routing); the MoE instantiations carry none of its code.
template <int NG, bool kLin>
__global__ void __launch_bounds__(dstr::kThreads, 1) decode_stream_kernel(StreamArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  StreamSmem& ss = *reinterpret_cast<StreamSmem*>(smem);
  const size_t base = (sizeof(StreamSmem) + 127) & ~size_t(127);
  const int nchH = a.H / 64, nchI = a.I / 64;
  float* red = reinterpret_cast<float*>(smem + base);  // [2][8][32][4 NG]
  uint8_t* ring = reinterpret_cast<uint8_t*>(red) + 2 * 8 * 32 * 4 * NG * sizeof(float);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = a.T, S = a.stages;
  constexpr int rows_pad = 8 * NG;
  const int apitch = T * dstr::kRow;  // a stage's activation rows per chunk
  // trace (NVFP4_MOE_TRACE=1): [0] entry, [1] routed, [2] first stage issued, [3] first stage
  // consumed (warp 0), [4] last stage posted, [5] warp 0 done, [6] exit, [7] items, [8] producer ns
  // waiting for free stages, [9] producer ns waiting for h / x, [10] warp 0 ns waiting for full
  // stages, [11] warp 0 ns in epilogues, [12] down items, [13] first down item started, [14] routing:
  // logits requested, [15] routing: experts chosen
  unsigned long long* tr = a.trace ? a.trace + (size_t)blockIdx.x * 16 : nullptr;
  // per-stage timeline of the first 8 CTAs (256 stages each, 8 words): producer before the
  // empty wait, after it, after the weight copies, after the activation copies, item<<8|stage;
  // the consumer group's wait end, its release
  unsigned long long* tl = (a.trace && blockIdx.x < 8) ? a.trace + (size_t)gridDim.x * 16 + blockIdx.x * 2048 : nullptr;
  if (tr && tid == 0) tr[0] = gtime();
  float lval[2][8];
  if (!kLin && !a.router_w) stream_route_issue(a, lval);

  // this CTA's share of the x conversion: token tx = 15 - warp of its chunks (chunk
  // blockIdx.x + i * gridDim.x), on the consumer warps from the top down -- for T <= 8
  // none of them chooses experts, so the conversion runs beside the routing; the loads
  // are issued first thing.  A dense linear's x ([T][I]) becomes the h rows of its one
  // "expert" (act_h, counted in done_c); the layer's x ([T][H]) the gate/up rows (act_x,
  // counted in x_ready)
  const int tx = dstr::kConsumers - 1 - warp;
  const bool xconv = !a.route_only && a.x && tx >= 0 && tx < T;
  const int xlen = kLin ? a.I : a.H, nchX = kLin ? nchI : nchH;
  uint8_t* const xdst = kLin ? a.act_h : a.act_x;
  int32_t* const xcnt = kLin ? a.done_c : a.x_ready;
  uint32_t xw[dstr::kXChunks];
  if (xconv) {
#pragma unroll
    for (int i = 0; i < dstr::kXChunks; ++i) {
      const int c = blockIdx.x + i * gridDim.x;
      if (c < nchX) xw[i] = __ldg(reinterpret_cast<const uint32_t*>(a.x + (size_t)tx * xlen + 64 * c) + lane);
    }
  }
  if (tid == 0 && !a.route_only) {
    ss.epi_cnt[0] = ss.epi_cnt[1] = 0;
    for (int s = 0; s < S; ++s) {
      mb_init(&ss.full[s], 1);
      mb_init(&ss.empty[s], dstr::kGroupWarps);  // each stage goes to one group
    }
    for (int g = 0; g < 2; ++g)
      for (int q = 0; q < dstr::kSig; ++q) {
        mb_init(&ss.sig_full[g][q], dstr::kGroupWarps);
        mb_init(&ss.sig_empty[g][q], 1);
      }
    for (int p = 0; p < 2; ++p)
      for (int q = 0; q < 8; ++q) {
        mb_init(&ss.red_full[p][q], 1);
        mb_init(&ss.red_empty[p][q], 1);
      }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (a.router_w) {  // the router linear first, then the logits it wrote
    stream_router(a, ss);
    stream_route_issue(a, lval);
  }
  auto convert_x = [&] {
    if (!xconv) return;
#pragma unroll
    for (int i = 0; i < dstr::kXChunks; ++i) {
      const int c = blockIdx.x + i * gridDim.x;
      if (c < nchX) convert_chunk_row(xw[i], xdst + ((size_t)c * T + tx) * dstr::kRow, lane);
    }
    // (chunks beyond the ones loaded above: only when the grid is small)
    for (int c = blockIdx.x + dstr::kXChunks * gridDim.x; c < nchX; c += gridDim.x) {
      const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(a.x + (size_t)tx * xlen + 64 * c) + lane);
      convert_chunk_row(w, xdst + ((size_t)c * T + tx) * dstr::kRow, lane);
    }
    // the rows are read by other CTAs' bulk copies (the async proxy) once counted in
    asm volatile("fence.proxy.async.global;" ::: "memory");
    __syncwarp();
    if (lane == 0) {
      __threadfence();
      for (int c = blockIdx.x; c < nchX; c += gridDim.x) atomicAdd(xcnt + c, 1);
    }
  };
  if (kLin) stream_route_linear(a, ss, convert_x);
  else stream_route(a, ss, lval, tr, convert_x, a.route_only ? -1 : dstr::kProducer);
  // the barriers and the touched-expert list are ready; except in the producer warp, so
  // are the positions, masks and (CTA 0) the tables written out
  if (a.route_only) return;
  if (tr && tid == 0) tr[1] = gtime();

  const int U = ss.U;
  const int gu_per = kLin ? 0 : nchI, dn_per = a.H / 128;  // items per expert (a linear: down only)
  const int n_gu = U * gu_per, n_items = n_gu + U * dn_per;
  const int cps = a.cps;
  const int nst_gu = (nchH + cps - 1) / cps, nst_dn = (nchI + cps - 1) / cps;  // both >= 2

  if (warp == dstr::kProducer) {
    // ---------------- producer ----------------
    uint32_t it = 0;
    int slot = 0;
    uint32_t ph = 0;  // phase parity of the ring's current lap
    bool dead = false;
    if (a.fault) {
      // issue nothing: the consumers' waits expire and record the timeout
      if (lane == 0) {
        const uint64_t t0 = gtime();
        while (!is_aborted(a.st) && gtime() - t0 < 2 * dstr::kTimeoutNs) __nanosleep(1000);
      }
      __syncwarp();
    } else {
      int item = blockIdx.x;
      const uint64_t once = l2_evict_first_policy();  // the weight tiles' L2 policy
      unsigned long long w_empty = 0, w_dep = 0, n_items_done = 0, n_dn = 0;
      bool x_ok = false;      // every chunk of act_x converted (known once, then for good)
      int ready_u = -1;       // the last expert whose h is known complete
      while (!dead) {
        if (item >= n_items) {  // no work left: a stage for each group that tells it to stop
          if (lane == 0) {
            for (int r = 0; r < 2; ++r) {
              if (!wait_phase(&ss.empty[slot], ph ^ 1u, a.st, 500)) break;
              ss.meta[slot][0] = -1;
              mb_arrive(&ss.full[slot]);
              if (++slot == S) {
                slot = 0;
                ph ^= 1u;
              }
            }
            if (tr) {
              tr[4] = gtime();
              tr[7] = n_items_done;
              tr[8] = w_empty;
              tr[9] = w_dep;
              tr[12] = n_dn;
            }
          }
          __syncwarp();
          ++it;
          break;
        }
        int nxt = 0;
        if (lane == 0) nxt = atomicAdd(a.wctr, 1);  // used after this item's stages: latency hidden
        const bool gu = item < n_gu;
        const int ii = gu ? item : item - n_gu;
        const int u = gu ? ii / gu_per : ii / dn_per, b = gu ? ii - u * gu_per : ii - u * dn_per;
        const int e = ss.tch_e[u], row0 = ss.tch_r0[u], m = ss.tch_m[u];
        const int nst = gu ? nst_gu : nst_dn, nch = gu ? nchH : nchI;
        if (a.checks && (e < 0 || e >= a.E || u >= U || row0 < 0 || m < 1 || row0 + m > a.rdec || m > rows_pad)) {
          if (lane == 0) report(a.st, kFlagBounds, 801);
          dead = true;
          break;
        }
        const uint8_t* eb = a.blob + (size_t)e * a.expert_stride;
        const uint8_t* tiles = eb + (gu ? a.w13 : a.w2) + (size_t)b * nch * kTileBytes;  // row block b's tiles
        const int32_t* dep = a.done_c + (size_t)u * nchI;
        // the item's inputs: a down item needs all of its expert's h (every chunk), a gate/up
        // item every chunk of act_x -- one parallel check, made once the first stage's weight
        // copies (which need nothing) are on their way
        bool need = gu ? !x_ok : ready_u != u;
        for (int s = 0; s < nst && !dead; ++s) {
          uint8_t* stg = ring + (size_t)slot * a.stage_bytes;
          uint64_t* full = &ss.full[slot];
          const int c0 = cps * s, nc = min(cps, nch - c0);
          int ok = 1;
          if (lane == 0) {
            const uint64_t t0 = tr ? gtime() : 0;
            if (tl && it < 256) tl[8 * it] = t0;
            ok = wait_phase(&ss.empty[slot], ph ^ 1u, a.st, 501);
            const uint64_t t1 = tr ? gtime() : 0;
            w_empty += t1 - t0;
            (void)t1;
            if (tr && it == 0) tr[2] = gtime();
            if (tl && it < 256) {
              tl[8 * it + 1] = gtime();
              tl[8 * it + 4] = ((unsigned long long)item << 8) | (unsigned)s;
            }
            if (ok) {
              ss.meta[slot][0] = item;
              ss.meta[slot][1] = s;
              ss.meta[slot][2] = nc;
              // the stage's activation rows: nc chunks x (T tokens or the expert's m rows)
              mb_expect(full, (uint32_t)(nc * kTileBytes + nc * (gu ? T : m) * dstr::kRow));
              bulk_g2s_hint(stg, tiles + (size_t)c0 * kTileBytes, (uint32_t)(nc * kTileBytes), full, once);
              if (tl && it < 256) tl[8 * it + 2] = gtime();
            }
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
          bool late = false;  // the inputs never became ready (the run is aborted)
          if (ok && need) {  // the readiness check, by the whole warp
            const uint64_t td0 = tr ? gtime() : 0;
            if (!gu && tr && n_dn == 0 && lane == 0) tr[13] = td0;
            late = !(gu ? warp_wait_all(a.x_ready, nchH, T, a.st, 700)
                        : warp_wait_all(dep, nchI, kLin ? T : 1, a.st, 600 + (unsigned)u));
            if (!late) {
              if (gu) x_ok = true;
              else ready_u = u;
            }
            need = false;
            // the inputs were written through the generic proxy; the copies read them through the async proxy
            asm volatile("fence.proxy.async.global;" ::: "memory");
            if (tr && lane == 0) w_dep += gtime() - td0;
          }
          // issued even when late: the rows are in the workspace either way, and the stage's
          // transaction count must complete so that the drain below ends
          if (ok && lane == 0) {
            if (gu) {
              bulk_g2s(stg + dstr::kAct, a.act_x + (size_t)c0 * apitch, (uint32_t)(nc * apitch), full);
            } else {  // the expert's h rows of chunks c0.. are one range
              bulk_g2s(stg + dstr::kAct, a.act_h + ((size_t)row0 * nchI + (size_t)c0 * m) * dstr::kRow,
                       (uint32_t)(nc * m * dstr::kRow), full);
            }
            if (tl && it < 256) tl[8 * it + 3] = gtime();
          }
          if (!ok) {
            dead = true;
          } else {
            ++it;
            if (++slot == S) {
              slot = 0;
              ph ^= 1u;
            }
            dead = late;
          }
        }
        ++n_items_done;
        n_dn += gu ? 0 : 1;
        item = (int)gridDim.x + __shfl_sync(0xffffffffu, nxt, 0);
      }
      // after an abort, copies may still be in flight: let them land first
      if (dead && lane == 0) {
        const uint64_t t0 = gtime();
        for (uint32_t i = it > (uint32_t)S ? it - S : 0; i < it; ++i) {
          const int sl = (int)(i % (uint32_t)S);
          while (!mb_try(&ss.full[sl], (i / S) & 1u) && gtime() - t0 < dstr::kTimeoutNs) {
          }
        }
      }
      __syncwarp();
    }
  } else if (warp == dstr::kSignaller) {
    // ---------------- signal warp: publishes what the consumers completed ----------------
    // The consumers' stores come before their arrivals on sig_full (release,
    // CTA scope); this warp's fence then orders them before the count that
    // other CTAs acquire, so no consumer ever waits for its own stores.  It
    // serves both groups' queues, each in order, until both have ended.
    uint32_t n[2] = {0, 0};
    bool open[2] = {true, true};
    uint64_t t0 = gtime();
    while (open[0] || open[1]) {
      bool any = false;
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        if (!open[g]) continue;
        const int q = (int)(n[g] % dstr::kSig);
        if (!mb_try(&ss.sig_full[g][q], (n[g] / dstr::kSig) & 1u)) continue;
        any = true;
        const int v = ss.sig[g][q];
        if (v < 0) {
          open[g] = false;
          continue;
        }
        // a down item completes output slice b for its expert; the item that completes
        // it for the last touched expert combines the slice here, at once
        const int b = v < n_gu ? -1 : (v - n_gu) % dn_per;
        int last = 0;
        if (lane == 0) {
          __threadfence();
          if (b < 0) atomicAdd(a.done_c + (size_t)(v / gu_per) * nchI + (v % gu_per), 1);
          else last = atomicAdd(a.cmb + b, 1) == ss.U - 1;
          mb_arrive(&ss.sig_empty[g][q]);
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (!kLin && last && T <= dstr::kSigCombineT) {
          __threadfence();  // the other CTAs' y rows, fenced before their counts
          for (int t = 0; t < T; ++t) combine_slice(a, ss, b, t, lane);
        }
        ++n[g];
      }
      if (any) {
        t0 = gtime();
      } else {
        if (is_aborted(a.st)) break;
        if (gtime() - t0 > dstr::kTimeoutNs) {
          if (lane == 0) report(a.st, kFlagTimeout, 320);
          break;
        }
        __nanosleep(32);
      }
    }
  } else {
    // ---------------- consumers ----------------
    // group grp takes the stages of even (0) or odd (1) global index; warp sb
    // of a group takes 16-row group sb of each of its stages
    const int grp = warp / dstr::kGroupWarps, sb = warp % dstr::kGroupWarps;

    float acc[NG][4];
    int slot = grp;
    uint32_t ph = 0, it = 0, nsig = 0, nitem = 0, nepi = 0;
    unsigned long long w_full = 0, w_epi = 0;
    // hands item v (or -1: the end) to the signal warp through the group's
    // queue: warp 0 of the group fills the entry once the signal warp has
    // freed it, then every warp of the group arrives
    auto post = [&](int v) {
      const int q = (int)(nsig % dstr::kSig);
      if (sb == 0 && lane == 0) {
        wait_phase(&ss.sig_empty[grp][q], ((nsig / dstr::kSig) & 1u) ^ 1u, a.st, 330);
        ss.sig[grp][q] = v;
      }
      __syncwarp();
      if (lane == 0) mb_arrive(&ss.sig_full[grp][q]);
      ++nsig;
    };
    for (;;) {
      const uint64_t tw0 = (tr && warp == 0) ? gtime() : 0;
      if (!wait_phase(&ss.full[slot], ph, a.st, 300)) break;
      if (tr && warp == 0 && lane == 0) {
        const uint64_t tw1 = gtime();
        w_full += tw1 - tw0;
        if (it == 0) tr[3] = tw1;
      }
      if (tl && sb == 0 && lane == 0 && 2 * it + grp < 256) tl[8 * (2 * it + grp) + 5] = gtime();
      const int item = ss.meta[slot][0];
      if (item < 0) break;
      const int s = ss.meta[slot][1], nc = ss.meta[slot][2];
      const bool gu = item < n_gu;
      if (s < 2) {  // this group's first stage of the item
#pragma unroll
        for (int gi = 0; gi < NG; ++gi)
#pragma unroll
          for (int z = 0; z < 4; ++z) acc[gi][z] = 0.f;
      }
      const uint8_t* stg = ring + (size_t)slot * a.stage_bytes;
      // a chunk's activation rows: the T tokens, or the down item's expert's m rows
      const int pitch = gu ? apitch : ss.tch_m[(item - n_gu) / dn_per] * dstr::kRow;
      // operands into registers, the math (4, 2 or 1 chunks at a time), then the stage back to the producer
      for (int cb = 0; cb < nc;) {
        if (nc - cb >= 4) {
          StageRegs<NG, 4> r;
          load_stage<NG, 4>(stg, cb, pitch, sb, lane, r);
          compute_stage<NG, 4>(r, acc);
          cb += 4;
        } else if (nc - cb >= 2) {
          StageRegs<NG, 2> r;
          load_stage<NG, 2>(stg, cb, pitch, sb, lane, r);
          compute_stage<NG, 2>(r, acc);
          cb += 2;
        } else {
          StageRegs<NG, 1> r;
          load_stage<NG, 1>(stg, cb, pitch, sb, lane, r);
          compute_stage<NG, 1>(r, acc);
          cb += 1;
        }
      }
      __syncwarp();
      if (lane == 0) mb_arrive(&ss.empty[slot]);
      if (tl && sb == 0 && lane == 0 && 2 * it + grp < 256) tl[8 * (2 * it + grp) + 6] = gtime();
      ++it;
      slot += 2;
      if (slot >= S) {
        slot -= S;
        ph ^= 1u;
      }
      const int nst = gu ? nst_gu : nst_dn;
      if (s + 2 < nst) continue;
      // this group's last stage of the item: the two warps of the 16-row group
      // (one per group) add their halves; the one with the item's last stage
      // finishes it
      const int par = nitem & 1;
      const uint32_t use = nitem >> 1;
      ++nitem;
      float* rb = red + ((size_t)(par * 8 + sb) * 32 + lane) * 4 * NG;
      if (s != nst - 1) {
        wait_phase(&ss.red_empty[par][sb], (use & 1u) ^ 1u, a.st, 310);
#pragma unroll
        for (int gi = 0; gi < NG; ++gi)
#pragma unroll
          for (int z = 0; z < 4; ++z) rb[4 * gi + z] = acc[gi][z];
        __syncwarp();
        if (lane == 0) mb_arrive(&ss.red_full[par][sb]);
        continue;
      }
      wait_phase(&ss.red_full[par][sb], use & 1u, a.st, 311);
#pragma unroll
      for (int gi = 0; gi < NG; ++gi)
#pragma unroll
        for (int z = 0; z < 4; ++z) acc[gi][z] += rb[4 * gi + z];
      __syncwarp();
      if (lane == 0) mb_arrive(&ss.red_empty[par][sb]);
      const int ii = gu ? item : item - n_gu;
      const int u = gu ? ii / gu_per : ii / dn_per;
      const int b = gu ? ii - u * gu_per : ii - u * dn_per;
      const uint64_t te0 = (tr && warp == 0) ? gtime() : 0;
      if (gu) epilogue_gateup<NG>(a, ss, u, b, sb, grp, acc, lane, nepi++);
      else epilogue_down<NG, kLin>(a, ss, u, b, sb, acc, lane);
      post(item);
      if (tr && warp == 0) w_epi += gtime() - te0;
    }
    post(-1);
    if (tr && warp == 0 && lane == 0) {
      tr[5] = gtime();
      tr[10] = w_full;
      tr[11] = w_epi;
    }
    if (!kLin && T > dstr::kSigCombineT && !is_aborted(a.st))
      combine_tasks(a, ss, (int)blockIdx.x * dstr::kConsumers + warp, (int)gridDim.x * dstr::kConsumers, lane);
  }

  // the last CTA out carries the status over and resets the per-forward counters
  __syncthreads();
  if (tr && tid == 0) tr[6] = gtime();
  if (tid == 0) {
    __threadfence();
    ss.last_cta = atomicAdd(a.exit_cnt, 1) == (int)gridDim.x - 1;
  }
  __syncthreads();
  if (!ss.last_cta) return;
  __threadfence();
  if (a.st_sticky && tid == 0) {
    const unsigned f = atomicOr(&a.st->flags, 0u), n = atomicAdd(&a.st->nan_logits, 0u);
    if (f && atomicOr(&a.st_sticky->flags, f) == 0u) a.st_sticky->where = *reinterpret_cast<volatile unsigned*>(&a.st->where);
    if (n) atomicAdd(&a.st_sticky->nan_logits, n);
  }
  for (int i = tid; i < U * nchI; i += blockDim.x) a.done_c[i] = 0;
  for (int i = tid; i < a.H / 128; i += blockDim.x) a.cmb[i] = 0;
  for (int i = tid; i < nchH; i += blockDim.x) a.x_ready[i] = 0;
  __syncthreads();
  if (tid == 0) {
    *a.wctr = 0;
    *a.exit_cnt = 0;
    if (a.router_w) *a.logit_ready = 0;
  }
}

// The hidden activations a forward consumed, as FP32 [R][I] (inspection):
// src 0 -- BF16 rows in h; src 1 -- the streaming decode kernel's FP16 chunk
// rows with their scale (act_h); src 2 -- the prefill GEMMs' FP16 rows in h,
// row p scaled by 2^-pexp_h[p].
__global__ void hidden_to_f32_kernel(const __nv_bfloat16* h, const uint8_t* act_h, const int32_t* pexp_h,
                                     const int32_t* ids, const int32_t* perm, const int32_t* offsets, int src, int R,
                                     int I, float* out) {
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (size_t)R * I) return;
  const int r = (int)(i / I), f = (int)(i - (size_t)r * I);
  if (src == 0) {
    out[i] = __bfloat162float(h[i]);
  } else if (src == 2) {
    out[i] = __half2float(reinterpret_cast<const __half*>(h)[i]) * __int_as_float((127 + pexp_h[r]) << 23);
  } else {
    // row r's expert block: rows offsets[e] .. offsets[e + 1], chunk-major
    const int e = ids[perm[r]], row0 = offsets[e], m = offsets[e + 1] - row0;
    const uint8_t* row = act_h + ((size_t)row0 * (I / 64) + (size_t)(f / 64) * m + (r - row0)) * dstr::kRow;
    out[i] = __half2float(*reinterpret_cast<const __half*>(row + 2 * (f % 64))) * *reinterpret_cast<const float*>(row + 128);
  }
}

cudaError_t launch_hidden_to_f32(const Workspace& ws, int src, int R, int I, float* out, cudaStream_t st) {
  const size_t n = (size_t)R * I;
  hidden_to_f32_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(ws.h, ws.act_h, ws.pexp_h, ws.ids, ws.perm,
                                                                    ws.offsets, src, R, I, out);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
bool stream_supported(const LayerDims& d, int T, int k) {
  return d.in_scale == nullptr && T >= 1 && T <= kDecodeMaxTokens && k + d.S <= dstr::kMaxSlots &&
         d.E <= dstr::kMaxE && d.H % 128 == 0 && d.I % 128 == 0 && d.H <= 16384 && d.I <= 16384;
}

size_t stream_act_h_bytes(int I, int rows) { return (size_t)(I / 64) * rows * dstr::kRow; }
size_t stream_act_x_bytes(int H) { return (size_t)(H / 64) * kDecodeMaxTokens * dstr::kRow; }

struct StreamPlan {
  int stages, stage_bytes;
  size_t smem;
};

static StreamPlan stream_plan(int T, int H, int smem_max) {
  const int NG = T <= 8 ? 1 : 2;
  (void)H;
  StreamPlan p{};
  // codes, scales, and T activation rows per chunk
  p.stage_bytes = (dstr::kAct + dstr::kCPS * T * dstr::kRow + 15) / 16 * 16;
  // + the pair sums, and a tail pad: the last stage's reads past its rows stay inside
  const size_t fixed = ((sizeof(StreamSmem) + 127) & ~size_t(127)) + 2 * 8 * 32 * 4 * NG * 4 + 8 * NG * dstr::kRow;
  const int room = (int)(((size_t)smem_max > fixed ? (size_t)smem_max - fixed : 0) / p.stage_bytes);
  p.stages = room < dstr::kMaxStages ? room : dstr::kMaxStages;
  p.smem = fixed + (size_t)p.stages * p.stage_bytes;
  return p;
}

cudaError_t stream_prepare_device(int dev, int* smem_max) {
  constexpr int kCached = 64;
  static std::mutex mu;
  static int cached[kCached] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (dev >= 0 && dev < kCached && cached[dev]) {
    *smem_max = cached[dev];
    return cudaSuccess;
  }
  int optin = 0;
  cudaError_t e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute((const void*)decode_stream_kernel<1, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute((const void*)decode_stream_kernel<1, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute((const void*)decode_stream_kernel<2, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute((const void*)decode_stream_kernel<2, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < kCached) cached[dev] = optin;
  *smem_max = optin;
  return cudaSuccess;
}

cudaError_t launch_decode_stream(const LayerDims& d, const uint8_t* blob, const float* gscale, const void* logits,
                                 const void* x, int T, int k, void* out, int route_only, int num_sms,
                                 const Workspace& ws, int fault, cudaStream_t st, const void* router_w) {
  if (!stream_supported(d, T, k)) return cudaErrorInvalidValue;
  int dev = 0, smem_max = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = stream_prepare_device(dev, &smem_max);
  if (e != cudaSuccess) return e;
  const StreamPlan plan = stream_plan(T, d.H, smem_max);
  if (plan.stages < 3 || plan.smem > (size_t)smem_max) return cudaErrorInvalidConfiguration;
  const ExpertLayout L = d.linear ? linear_layout(d.H, d.I) : expert_layout(d.H, d.I);
  StreamArgs a{};
  a.blob = blob;
  a.expert_stride = L.stride;
  a.w13 = L.w13;
  a.w2 = L.w2;
  a.gscale = gscale;
  a.E = d.E;
  a.Er = d.Er;
  a.H = d.H;
  a.I = d.I;
  a.T = T;
  a.k = k + d.S;
  a.topk = k;
  a.rp = d.rp;
  a.logits = logits;
  a.logits_bf16 = d.logits_bf16;
  a.linear = d.linear;
  a.n_out = d.n_out;
  if (d.linear && (router_w || route_only || !x)) return cudaErrorInvalidValue;
  if (router_w) {
    if (!x || route_only || !ws.logits || !ws.logit_ready) return cudaErrorInvalidValue;
    a.router_w = reinterpret_cast<const __nv_bfloat16*>(router_w);
    a.logits_w = ws.logits;
    a.logit_ready = ws.logit_ready;
    a.logits = ws.logits;
    a.logits_bf16 = 0;
  }
  a.x = reinterpret_cast<const __nv_bfloat16*>(x);
  a.out = out;
  a.out_f32 = d.out_f32;
  a.route_only = route_only;
  a.ids = ws.ids;
  a.wts = ws.wts;
  a.offsets = ws.offsets;
  a.perm = ws.perm;
  a.inv = ws.inv;
  a.act_h = ws.act_h;
  a.act_x = ws.act_x;
  a.rdec = ws.act_rows;
  a.y = ws.y;
  a.wctr = ws.wctr;
  a.done_c = ws.done_c;
  a.cmb = ws.cmb;
  a.x_ready = ws.x_ready;
  a.exit_cnt = ws.exit_cnt;
  a.st = ws.status;
  a.st_sticky = ws.status_sticky;
  a.fault = fault;
  a.stages = plan.stages;
  a.stage_bytes = plan.stage_bytes;
  // chunks per stage: 4, or fewer so that every item has at least two stages (one per consumer group)
  a.cps = (d.H / 64 >= 2 * dstr::kCPS && d.I / 64 >= 2 * dstr::kCPS) ? dstr::kCPS
          : (d.H / 64 >= 8 && d.I / 64 >= 8)                        ? 4
          : (d.H / 64 >= 4 && d.I / 64 >= 4)                        ? 2
                                                                     : 1;
  a.checks = d.checks;
  a.trace = ws.trace;
  if (!route_only && T * (k + d.S) > ws.act_rows) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(route_only ? 1 : num_sms);
  cfg.blockDim = dim3(dstr::kThreads);
  cfg.dynamicSmemBytes = plan.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = route_only ? 0 : 1;
  if (d.linear)
    return T <= 8 ? cudaLaunchKernelEx(&cfg, decode_stream_kernel<1, true>, a)
                  : cudaLaunchKernelEx(&cfg, decode_stream_kernel<2, true>, a);
  return T <= 8 ? cudaLaunchKernelEx(&cfg, decode_stream_kernel<1, false>, a)
                : cudaLaunchKernelEx(&cfg, decode_stream_kernel<2, false>, a);
}

}  // namespace nvfp4moe
