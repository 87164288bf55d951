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
//  * work items are claimed dynamically from one global counter: first every
//    gate/up item (expert u, 128 packed rows = 64 features, all of K = H),
//    then every down item (expert u, 128 output rows, all of K = I), each
//    group expert-major.  A CTA's first item is its index, later ones come
//    from the counter (claimed one item ahead, so the atomic's latency hides
//    behind the current item).  Fast SMs simply take more items, and a down
//    item waits only for the chunks of h it reads, chunk by chunk, so the
//    phases overlap instead of meeting at a barrier;
//  * one producer warp per CTA streams each item through a shared-memory ring
//    of stages (four 64-wide K chunks of one 128-row block: 16 KB of codes
//    and 2 KB of scales, each one contiguous cp.async.bulk, plus the chunks'
//    activation rows) completed on mbarriers; 8 consumer warps each take one
//    16-row group of a stage, all four chunks (four independent MMA chains),
//    dequantise in registers (hardware E2M1 -> FP16 converts times the E4M3
//    group scale, exact) and run mma.sync m16n8k16 (FP16 in, FP32
//    accumulate);
//  * activations enter the MMA as FP16 rows of one 64-wide chunk with their
//    own power-of-two scale (the chunk's largest magnitude in [2^13, 2^14):
//    exact for every value within 2^31 of it that has at most 11 significant
//    bits), stored next to the row; each chunk's partial sums are multiplied
//    back by the scale in FP32.  x is converted once per CTA into shared
//    memory (few tokens) or once per chunk by one CTA into global memory; the
//    gate/up epilogue of an item produces one whole chunk of h (its 64
//    features), so it writes h in that form: FP16, 11 significant bits;
//  * gate/up columns are the step's tokens (every token through every touched
//    expert's MMA columns; only the routed ones are kept), down columns are
//    the expert's routed rows;
//  * the combine: once the work runs out, every warp of the grid takes
//    (128-wide output slice, token) tasks, each starting when its slice is
//    complete for every touched expert, and sums the k slots in slot order;
//  * every wait is bounded (2 s): a wait that gives up records a timeout in the
//    status word and the kernel unwinds without a trap.
#include <cstdlib>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "route_common.cuh"

namespace nvfp4moe {

namespace dstr {
constexpr int kConsumers = 8;                     // consumer warps: one per 16-row group of a 128-row block
constexpr int kThreads = (kConsumers + 1) * 32;   // + one producer warp
constexpr int kProducer = kConsumers;             // the producer's warp index
constexpr int kCPS = 4;                           // 64-wide K chunks per stage
constexpr int kCodes = kCPS * 4096;               // 128 rows x 4 chunks of E2M1 codes
constexpr int kScales = kCPS * 512;               // their E4M3 scales
constexpr int kAct = kCodes + kScales;            // activation rows of the stage's chunks
constexpr int kRow = 144;                         // one activation row of a chunk: 64 FP16, float scale at +128
constexpr int kMaxSlots = 17;                     // slots per token: top_k <= 16 + one shared expert
constexpr int kMaxR = kDecodeMaxTokens * kMaxSlots;
constexpr int kMaxE = 288;                        // routed + shared experts (9 per lane in the scan)
constexpr int kMaxStages = 12;
constexpr int kXsPairs = 16;                      // (token, chunk) pairs per consumer warp in the shared x copy
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
  float cmax[8][16];               // gate/up epilogue: per 16-row group, per column, max |h|
  int meta[dstr::kMaxStages][4];   // item, stage within the item, chunks in the stage
  int U, nan, last_cta;
  alignas(8) uint64_t full[dstr::kMaxStages];
  alignas(8) uint64_t empty[dstr::kMaxStages];
};

struct StreamArgs {
  const uint8_t* blob;
  size_t expert_stride, nib13, sc13, nib2, sc2;
  const float* gscale;
  int E, Er, H, I, T, k, topk;  // E experts in the blob, k slots per token (top_k + shared)
  RouteParams rp;
  const void* logits;
  int logits_bf16;
  const __nv_bfloat16* x;
  void* out;
  int out_f32;
  int route_only;
  int32_t* ids;
  float* wts;
  int32_t* offsets;
  int32_t* perm;
  int32_t* inv;
  uint8_t* act_h;     // [I/64][rdec][kRow]: h rows per chunk, FP16 with their scale
  uint8_t* act_x;     // [H/64][8 NG][kRow]: x rows per chunk (when not kept in shared memory)
  int rdec;           // rows of act_h per chunk
  float* y;           // [R][H] expert outputs, position order
  int32_t* wctr;      // claimed items beyond the first gridDim.x
  int32_t* done_c;    // [maxU][I/64]: gate/up epilogue warps done per (touched expert, chunk of h)
  int32_t* cmb;       // finished down epilogue warps per 128-wide output slice
  int32_t* x_ready;   // tokens converted per chunk of x (act_x)
  int32_t* exit_cnt;
  DeviceStatus* st;
  DeviceStatus* st_sticky;
  int fault;          // 1: the producer issues nothing (tests the bounded waits)
  int stages, stage_bytes;
  int xs;             // 1: x is converted into shared memory by every CTA
  int checks;         // 1: check table-derived indices (kFlagBounds; the access is skipped)
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
__device__ __forceinline__ void named_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
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
__device__ void stream_route(const StreamArgs& a, StreamSmem& ss, unsigned long long* tr) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nw = blockDim.x >> 5;
  const int T = a.T, k = a.k, E = a.E, Er = a.Er, topk = a.topk, R = T * k;
  float val[2][8];
  uint32_t key[2][8];
#pragma unroll
  for (int r = 0; r < 2; ++r)
    if (warp + r * nw < T) warp_issue_logits(a.logits, a.logits_bf16, Er, warp + r * nw, val[r]);
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
  for (int r = tid; r < R; r += blockDim.x) {  // expert-major position: rank among the earlier rows of the same expert
    const int e = ss.ids[r];
    int rank = 0;
    for (int j = 0; j < r; ++j) rank += (ss.ids[j] == e);
    const int pos = ss.off[e] + rank;
    ss.perm[pos] = r;
    ss.inv[r] = pos;
    atomicOr(&ss.tch_mask[ss.slot_of[e]], 1u << (r / k));
  }
  __syncthreads();
  if (blockIdx.x == 0) {  // the tables, for inspection
    for (int i = tid; i < R; i += blockDim.x) {
      a.ids[i] = ss.ids[i];
      a.wts[i] = ss.wts[i];
      a.perm[i] = ss.perm[i];
      a.inv[i] = ss.inv[i];
    }
    for (int i = tid; i <= E; i += blockDim.x) a.offsets[i] = ss.off[i];
    if (tid == 0 && ss.nan) atomicAdd(&a.st->nan_logits, (unsigned)ss.nan);
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

// One stage's work of consumer warp sb: its 16-row group of NC chunks (all
// fragments loaded first, so the NC chains overlap).  xtile: the first
// chunk's activation rows when x sits in shared memory (rows `xpitch` chunks
// apart), else null (the stage carries them, rows_pad rows per chunk).
template <int NG, int NC>
__device__ __forceinline__ void consume_stage(const uint8_t* stg, const uint8_t* xtile, size_t xpitch, int sb,
                                              float (&acc)[NG][4], int lane) {
  AFrag f[NC];
#pragma unroll
  for (int cs = 0; cs < NC; ++cs) load_a(stg + cs * 4096 + sb * 512, stg + dstr::kCodes + cs * 512 + sb * 64, lane, f[cs]);
#pragma unroll
  for (int cs = 0; cs < NC; ++cs)
    mma_tile<NG>(f[cs], xtile ? xtile + cs * xpitch : stg + dstr::kAct + cs * (8 * NG) * dstr::kRow, acc, lane);
}

// Gate/up epilogue of item (u, b) on the 8 consumer warps (16-row group sb):
// h for the 64 features of chunk b, kept for the routed tokens, as the FP16
// chunk rows with their scale in act_h; then each warp counts itself in for
// (u, chunk b).
template <int NG>
__device__ void epilogue_gateup(const StreamArgs& a, StreamSmem& ss, int u, int b, int sb, const float (&acc)[NG][4],
                                int lane) {
  const int e = ss.tch_e[u], row0 = ss.tch_r0[u];
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
      if (g == 0) ss.cmax[sb][t] = m;
    }
  named_sync(1, dstr::kConsumers * 32);
#pragma unroll
  for (int gi = 0; gi < NG; ++gi)
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int t = 8 * gi + 2 * q + c;
      if (t >= a.T || !((mask >> t) & 1u)) continue;
      float m = 0.f;
#pragma unroll
      for (int s = 0; s < 8; ++s) m = fmaxf(m, ss.cmax[s][t]);
      const int p = max(-126, min(126, prescale_exp(m)));
      const int pos = row0 + __popc(mask & ((1u << t) - 1u));
      if (a.checks && (pos < 0 || pos >= a.T * a.k)) {
        report(a.st, kFlagBounds, 802);
        continue;
      }
      const int f = 8 * sb + g;  // feature within the chunk
      uint8_t* row = a.act_h + ((size_t)b * a.rdec + pos) * dstr::kRow;
      *reinterpret_cast<__half*>(row + 2 * f) = __float2half_rn(hv[gi][c] * exp2i(-p));
      if (sb == 0 && g == 0) *reinterpret_cast<float*>(row + 128) = exp2i(p);
    }
  // the rows are read by other CTAs' bulk copies (the async proxy)
  asm volatile("fence.proxy.async.global;" ::: "memory");
  __syncwarp();
  if (lane == 0) {
    __threadfence();
    atomicAdd(a.done_c + (size_t)u * (a.I / 64) + b, 1);
  }
}

// Down epilogue of item (u, b): y rows 128 b + 16 sb + g (+8) for the
// expert's routed rows; each warp counts itself in for output slice b.
template <int NG>
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
      if (j < m) {
        float* yr = a.y + (size_t)(row0 + j) * a.H;
        yr[d0] = acc[gi][c] * gsd;
        yr[d0 + 8] = acc[gi][2 + c] * gsd;
      }
    }
  __syncwarp();
  if (lane == 0) {
    __threadfence();
    atomicAdd(a.cmb + b, 1);
  }
}

// The combine, spread over every consumer warp of the grid: task (128-wide
// slice b, token t) waits until slice b is complete for every touched expert
// (8 U down epilogue warps), then out[t][slice] = sum_j w[t][j] *
// y[pos(t, j)][slice] in slot order j = 0..k-1 (lane l: features 4l..4l+3).
__device__ void combine_tasks(const StreamArgs& a, const StreamSmem& ss, int wg, int W, int lane) {
  const int nsl = a.H / 128, target = dstr::kConsumers * ss.U;
  for (int task = wg; task < nsl * a.T; task += W) {
    const int t = task / nsl, b = task - t * nsl;
    int ok = 1;
    if (lane == 0) ok = wait_count(a.cmb + b, target, a.st, 400 + (unsigned)b);
    if (!__shfl_sync(0xffffffffu, ok, 0)) return;
    __threadfence();
    const int d = 128 * b + 4 * lane;
    float4 yy[dstr::kMaxSlots];
#pragma unroll
    for (int j = 0; j < dstr::kMaxSlots; ++j)
      if (j < a.k) {
        int pos = ss.inv[t * a.k + j];
        if (a.checks && (pos < 0 || pos >= a.T * a.k)) {
          report(a.st, kFlagBounds, 803);
          pos = 0;
        }
        yy[j] = __ldcg(reinterpret_cast<const float4*>(a.y + (size_t)pos * a.H + d));
      }
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
    for (int j = 0; j < dstr::kMaxSlots; ++j)
      if (j < a.k) {
        const float w = ss.wts[t * a.k + j];
        s0 = fmaf(w, yy[j].x, s0);
        s1 = fmaf(w, yy[j].y, s1);
        s2 = fmaf(w, yy[j].z, s2);
        s3 = fmaf(w, yy[j].w, s3);
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
}

// ---------------------------------------------------------------------------
// The kernel.  Shared memory: StreamSmem | x rows (xs mode) | ring
// [stages][stage_bytes].
// ---------------------------------------------------------------------------
template <int NG>
__global__ void __launch_bounds__(dstr::kThreads, 1) decode_stream_kernel(StreamArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  StreamSmem& ss = *reinterpret_cast<StreamSmem*>(smem);
  const size_t base = (sizeof(StreamSmem) + 127) & ~size_t(127);
  const int nchH = a.H / 64, nchI = a.I / 64;
  const size_t xs_bytes = a.xs ? (size_t)nchH * a.T * dstr::kRow : 0;
  uint8_t* xs = smem + base;
  uint8_t* ring = smem + base + ((xs_bytes + 127) & ~size_t(127));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = a.T, S = a.stages;
  constexpr int rows_pad = 8 * NG;
  // trace (NVFP4_MOE_TRACE=1): [0] entry, [1] routed, [2] first stage issued, [3] first stage
  // consumed (warp 0), [4] last stage posted, [5] warp 0 done, [6] exit, [7] items, [8] producer ns
  // waiting for free stages, [9] producer ns waiting for h / x, [10] warp 0 ns waiting for full
  // stages, [11] warp 0 ns in epilogues, [12] down items, [13] first down item started, [14] routing:
  // logits requested, [15] routing: experts chosen
  unsigned long long* tr = a.trace ? a.trace + (size_t)blockIdx.x * 16 : nullptr;
  if (tr && tid == 0) tr[0] = gtime();

  // x words this warp converts (loads issued before routing so their latency overlaps it)
  uint32_t xw[dstr::kXsPairs];
  const int npairs = T * nchH;
  if (!a.route_only && a.x && warp < dstr::kConsumers) {
    if (a.xs) {
#pragma unroll
      for (int i = 0; i < dstr::kXsPairs; ++i) {
        const int p = warp + dstr::kConsumers * i;  // pair p: token p % T, chunk p / T
        if (p < npairs)
          xw[i] = __ldg(reinterpret_cast<const uint32_t*>(a.x + (size_t)(p % T) * a.H + 64 * (p / T)) + lane);
      }
    } else {
#pragma unroll
      for (int i = 0; i < dstr::kXsPairs; ++i) {
        // this CTA's chunks of x: chunk blockIdx.x + (i / 2) * gridDim.x, token warp + 8 (i % 2)
        const int c = blockIdx.x + (i >> 1) * gridDim.x, t = warp + dstr::kConsumers * (i & 1);
        if (c < nchH && t < T) xw[i] = __ldg(reinterpret_cast<const uint32_t*>(a.x + (size_t)t * a.H + 64 * c) + lane);
      }
    }
  }
  if (tid == 0 && !a.route_only) {
    for (int s = 0; s < S; ++s) {
      mb_init(&ss.full[s], 1);
      mb_init(&ss.empty[s], dstr::kConsumers);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  stream_route(a, ss, tr);  // ends with __syncthreads: tables and barriers are ready
  if (a.route_only) return;
  if (tr && tid == 0) tr[1] = gtime();

  const int U = ss.U;
  const int gu_per = nchI, dn_per = a.H / 128;  // items per expert
  const int n_gu = U * gu_per, n_items = n_gu + U * dn_per;
  const int nst_gu = (nchH + dstr::kCPS - 1) / dstr::kCPS, nst_dn = (nchI + dstr::kCPS - 1) / dstr::kCPS;

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
      unsigned long long w_empty = 0, w_dep = 0, n_items_done = 0, n_dn = 0;
      bool x_ok = a.xs != 0;  // every chunk of act_x converted (known once, then for good)
      int ready_u = -1;       // the last expert whose h is known complete
      while (!dead) {
        if (item >= n_items) {  // no work left: a stage that tells the consumers to stop
          if (lane == 0) {
            if (wait_phase(&ss.empty[slot], ph ^ 1u, a.st, 500)) {
              ss.meta[slot][0] = -1;
              mb_arrive(&ss.full[slot]);
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
        const uint8_t* codes = eb + (gu ? a.nib13 : a.nib2) + (size_t)b * nch * 4096;
        const uint8_t* scl = eb + (gu ? a.sc13 : a.sc2) + (size_t)b * nch * 512;
        const int32_t* dep = a.done_c + (size_t)u * nchI;
        // the item's inputs: a down item needs all of its expert's h (every gate/up epilogue warp of
        // each chunk), a gate/up item every chunk of act_x; one parallel check, then never again
        {
          const uint64_t td0 = tr ? gtime() : 0;
          if (!gu && ready_u != u) {
            if (tr && n_dn == 0 && lane == 0) tr[13] = gtime();
            if (warp_wait_all(dep, nchI, dstr::kConsumers, a.st, 600 + (unsigned)u)) ready_u = u;
            else dead = true;
          } else if (gu && !x_ok) {
            if (warp_wait_all(a.x_ready, nchH, T, a.st, 700)) x_ok = true;
            else dead = true;
          }
          // the inputs were written through the generic proxy; the copies read them through the async proxy
          asm volatile("fence.proxy.async.global;" ::: "memory");
          if (tr && lane == 0) w_dep += gtime() - td0;
        }
        for (int s = 0; s < nst && !dead; ++s) {
          uint8_t* stg = ring + (size_t)slot * a.stage_bytes;
          uint64_t* full = &ss.full[slot];
          const int c0 = dstr::kCPS * s, nc = min(dstr::kCPS, nch - c0);
          int ok = 1;
          if (lane == 0) {
            const uint64_t t0 = tr ? gtime() : 0;
            ok = wait_phase(&ss.empty[slot], ph ^ 1u, a.st, 501);
            const uint64_t t1 = tr ? gtime() : 0;
            w_empty += t1 - t0;
            // activation rows of the stage's chunks (none when x is in shared memory)
            const uint32_t act = !gu ? (uint32_t)(nc * m * dstr::kRow) : a.xs ? 0u : (uint32_t)(nc * rows_pad * dstr::kRow);
            (void)t1;
            if (tr && it == 0) tr[2] = gtime();
            if (ok) {
              ss.meta[slot][0] = item;
              ss.meta[slot][1] = s;
              ss.meta[slot][2] = nc;
              mb_expect(full, (uint32_t)nc * (4096u + 512u) + act);
              bulk_g2s(stg, codes + (size_t)c0 * 4096, (uint32_t)nc * 4096u, full);
              bulk_g2s(stg + dstr::kCodes, scl + (size_t)c0 * 512, (uint32_t)nc * 512u, full);
              if (act && gu) {
                bulk_g2s(stg + dstr::kAct, a.act_x + (size_t)c0 * rows_pad * dstr::kRow, act, full);
              } else if (act) {
                for (int c = 0; c < nc; ++c)
                  bulk_g2s(stg + dstr::kAct + c * rows_pad * dstr::kRow,
                           a.act_h + ((size_t)(c0 + c) * a.rdec + row0) * dstr::kRow, (uint32_t)(m * dstr::kRow), full);
              }
            }
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) {
            dead = true;
          } else {
            ++it;
            if (++slot == S) {
              slot = 0;
              ph ^= 1u;
            }
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
  } else {
    // ---------------- consumers ----------------
    const int sb = warp;
    if (a.x) {  // this CTA's share of the x conversion
      if (a.xs) {
#pragma unroll
        for (int i = 0; i < dstr::kXsPairs; ++i) {
          const int p = warp + dstr::kConsumers * i;
          if (p < npairs) convert_chunk_row(xw[i], xs + ((size_t)(p / T) * T + p % T) * dstr::kRow, lane);
        }
      } else {
        bool any = false;
#pragma unroll
        for (int i = 0; i < dstr::kXsPairs; ++i) {
          const int c = blockIdx.x + (i >> 1) * gridDim.x, t = warp + dstr::kConsumers * (i & 1);
          if (c < nchH && t < T) {
            convert_chunk_row(xw[i], a.act_x + ((size_t)c * rows_pad + t) * dstr::kRow, lane);
            any = true;
          }
        }
        // (chunks beyond the ones loaded above: only when the grid is small)
        for (int c = blockIdx.x + (dstr::kXsPairs / 2) * gridDim.x; c < nchH; c += gridDim.x)
          for (int t = warp; t < T; t += dstr::kConsumers) {
            const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(a.x + (size_t)t * a.H + 64 * c) + lane);
            convert_chunk_row(w, a.act_x + ((size_t)c * rows_pad + t) * dstr::kRow, lane);
            any = true;
          }
        if (any) {
          asm volatile("fence.proxy.async.global;" ::: "memory");
          __syncwarp();
          if (lane == 0) {
            __threadfence();
            for (int c = blockIdx.x; c < nchH; c += gridDim.x)
              for (int t = warp; t < T; t += dstr::kConsumers) atomicAdd(a.x_ready + c, 1);
          }
        }
      }
    }
    named_sync(2, dstr::kConsumers * 32);  // the shared x rows are complete

    float acc[NG][4];
    int slot = 0;
    uint32_t ph = 0, it = 0;
    unsigned long long w_full = 0, w_epi = 0;
    for (;;) {
      const uint64_t tw0 = (tr && warp == 0) ? gtime() : 0;
      if (!wait_phase(&ss.full[slot], ph, a.st, 300)) break;
      if (tr && warp == 0 && lane == 0) {
        const uint64_t tw1 = gtime();
        w_full += tw1 - tw0;
        if (it == 0) tr[3] = tw1;
      }
      const int item = ss.meta[slot][0];
      if (item < 0) break;
      const int s = ss.meta[slot][1], nc = ss.meta[slot][2];
      const bool gu = item < n_gu;
      if (s == 0) {
#pragma unroll
        for (int gi = 0; gi < NG; ++gi)
#pragma unroll
          for (int z = 0; z < 4; ++z) acc[gi][z] = 0.f;
      }
      const uint8_t* stg = ring + (size_t)slot * a.stage_bytes;
      const size_t xpitch = (size_t)T * dstr::kRow;
      const uint8_t* xtile = (gu && a.xs) ? xs + (size_t)(dstr::kCPS * s) * xpitch : nullptr;
      if (nc == dstr::kCPS) {
        consume_stage<NG, dstr::kCPS>(stg, xtile, xpitch, sb, acc, lane);
      } else {  // an item's last stage with two chunks (K/64 is even, not a multiple of 4)
        consume_stage<NG, 2>(stg, xtile, xpitch, sb, acc, lane);
      }
      __syncwarp();
      if (lane == 0) mb_arrive(&ss.empty[slot]);
      ++it;
      if (++slot == S) {
        slot = 0;
        ph ^= 1u;
      }
      if (s != (gu ? nst_gu : nst_dn) - 1) continue;
      // the item's last stage: this warp's 16-row group is complete
      const int ii = gu ? item : item - n_gu;
      const int u = gu ? ii / gu_per : ii / dn_per;
      const int b = gu ? ii - u * gu_per : ii - u * dn_per;
      const uint64_t te0 = (tr && warp == 0) ? gtime() : 0;
      if (gu) epilogue_gateup<NG>(a, ss, u, b, sb, acc, lane);
      else epilogue_down<NG>(a, ss, u, b, sb, acc, lane);
      if (tr && warp == 0) w_epi += gtime() - te0;
    }
    if (tr && warp == 0 && lane == 0) {
      tr[5] = gtime();
      tr[10] = w_full;
      tr[11] = w_epi;
    }
    if (!is_aborted(a.st))
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
  }
}

// The hidden activations a forward consumed, as FP32 [R][I] (inspection):
// src 0 -- BF16 rows in h; src 1 -- the streaming decode kernel's FP16 chunk
// rows with their scale (act_h); src 2 -- the prefill GEMMs' FP16 rows in h,
// row p scaled by 2^-pexp_h[p].
__global__ void hidden_to_f32_kernel(const __nv_bfloat16* h, const uint8_t* act_h, const int32_t* pexp_h, int rdec,
                                     int src, int R, int I, float* out) {
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (size_t)R * I) return;
  const int r = (int)(i / I), f = (int)(i - (size_t)r * I);
  if (src == 0) {
    out[i] = __bfloat162float(h[i]);
  } else if (src == 2) {
    out[i] = __half2float(reinterpret_cast<const __half*>(h)[i]) * __int_as_float((127 + pexp_h[r]) << 23);
  } else {
    const uint8_t* row = act_h + ((size_t)(f / 64) * rdec + r) * dstr::kRow;
    out[i] = __half2float(*reinterpret_cast<const __half*>(row + 2 * (f % 64))) * *reinterpret_cast<const float*>(row + 128);
  }
}

cudaError_t launch_hidden_to_f32(const Workspace& ws, int src, int R, int I, float* out, cudaStream_t st) {
  const size_t n = (size_t)R * I;
  hidden_to_f32_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(ws.h, ws.act_h, ws.pexp_h, ws.act_rows, src, R, I,
                                                                    out);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
bool stream_supported(const LayerDims& d, int T, int k) {
  return !d.linear && d.in_scale == nullptr && T >= 1 && T <= kDecodeMaxTokens && k + d.S <= dstr::kMaxSlots &&
         d.E <= dstr::kMaxE && d.H % 128 == 0 && d.I % 128 == 0 && d.H <= 16384 && d.I <= 16384;
}

size_t stream_act_h_bytes(int I, int rows) { return (size_t)(I / 64) * rows * dstr::kRow; }
size_t stream_act_x_bytes(int H) { return (size_t)(H / 64) * kDecodeMaxTokens * dstr::kRow; }

struct StreamPlan {
  int xs, stages, stage_bytes;
  size_t smem;
};

static StreamPlan stream_plan(int T, int H, int smem_max) {
  const int NG = T <= 8 ? 1 : 2;
  StreamPlan p{};
  const int nch = H / 64;
  p.xs = T * nch <= dstr::kConsumers * dstr::kXsPairs;
  p.stage_bytes = dstr::kAct + dstr::kCPS * 8 * NG * dstr::kRow;
  const size_t fixed = ((sizeof(StreamSmem) + 127) & ~size_t(127)) +
                       ((p.xs ? (size_t)nch * T * dstr::kRow : 0) + 127) / 128 * 128;
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
    e = cudaFuncSetAttribute((const void*)decode_stream_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute((const void*)decode_stream_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < kCached) cached[dev] = optin;
  *smem_max = optin;
  return cudaSuccess;
}

cudaError_t launch_decode_stream(const LayerDims& d, const uint8_t* blob, const float* gscale, const void* logits,
                                 const void* x, int T, int k, void* out, int route_only, int num_sms,
                                 const Workspace& ws, int fault, cudaStream_t st) {
  if (!stream_supported(d, T, k)) return cudaErrorInvalidValue;
  int dev = 0, smem_max = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = stream_prepare_device(dev, &smem_max);
  if (e != cudaSuccess) return e;
  const StreamPlan plan = stream_plan(T, d.H, smem_max);
  if (plan.stages < 3 || plan.smem > (size_t)smem_max) return cudaErrorInvalidConfiguration;
  const ExpertLayout L = expert_layout(d.H, d.I);
  StreamArgs a{};
  a.blob = blob;
  a.expert_stride = L.stride;
  a.nib13 = L.w13_nib;
  a.sc13 = L.w13_sc;
  a.nib2 = L.w2_nib;
  a.sc2 = L.w2_sc;
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
  a.xs = plan.xs;
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
  return T <= 8 ? cudaLaunchKernelEx(&cfg, decode_stream_kernel<1>, a)
                : cudaLaunchKernelEx(&cfg, decode_stream_kernel<2>, a);
}

}  // namespace nvfp4moe
