// The earlier decode kernel (1..16 tokens): one cooperative persistent kernel
// that routes, runs the grouped gate/up GEMV with SwiGLU, the grouped down GEMV
// and the weighted combine, dequantising NVFP4 in registers.  The W4A16 decode
// path runs the streaming kernel (decode_stream.cu); this one serves the W4A4
// comparison variant's decode and any shape the streaming kernel does not take.
//
// At decode sizes every expert a token picks is streamed from HBM once per
// step -- "the memory-bandwidth wall for an 18B-active model" ("GLM-5.3-Flash
// on Blackwell", Two deployments, and the lever that reverses between them).
// The weight-only path never takes an activation scale: weights are
// dequantised to 16-bit and multiplied with the 16-bit activations (same page,
// The model loaded, served an API, and produced garbage).
//
// Design (GB300):
//  * one launch per forward, one 16-warp CTA per SM (cooperative, so all CTAs
//    are resident); every CTA routes the <= 16 tokens itself (one warp per
//    token: redux.sync top-k over its logits, then the scoring rule), so no
//    routing tables cross CTAs before the GEMVs start;
//  * work split in two levels, so every SM streams the same number of weight
//    bytes whatever the routing: each CTA takes an equal share of the 16-row
//    groups of the touched experts' matrices over the whole K axis (no row's
//    sum crosses CTAs); inside the CTA the (64-row piece, 64-wide K chunk)
//    items are cut into contiguous ranges of equal estimated time, one per
//    warp, and partial sums of a piece split across warps meet in shared
//    memory (FP32 slots; global slots when the shared ones do not fit), the
//    last warp to arrive finishing the piece;
//  * each warp runs its own ring in shared memory (2 to 5 stages, as deep as
//    the shared memory left allows): one lane issues cp.async.bulk copies of
//    a chunk's codes (up to 2 KB), scales and -- unless the tokens'
//    activations are staged once per CTA in shared memory (few tokens) --
//    the routed rows' activation slices (128 B each) onto the stage's
//    mbarrier;
//  * dequantisation: hardware E2M1->FP16 converts (two weights each) times the
//    E4M3 group scale in FP16 (exact); the dot products run on mma.sync
//    m16n8k16 (FP16 in, FP32 accumulate) -- about one instruction per weight;
//  * the K axis of each 64-chunk is permuted identically for weights and
//    activations, so a lane's 16-byte load is exactly its MMA fragment;
//  * activations (x, then h) enter as FP16 after a per-row power-of-two
//    prescale (exact for BF16 values within 2^31 of the row maximum), undone
//    in FP32;
//  * the down GEMV of expert u starts once all gate/up rows of u are done
//    (per-expert counter, bounded wait); the combine is spread over every
//    warp as (64-wide slice of H, token) tasks, each starting once its slice
//    is finished for every expert, summing in slot order;
//  * the same kernel runs a dense linear (one matrix, no routing, the down
//    phase alone, rows written straight to out) and, as separate template
//    instantiations, the W4A4 comparison variant (each lane quantises its
//    16-element activation block to NVFP4 before the MMA).
#include <cstdlib>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "route_common.cuh"

namespace nvfp4moe {

namespace dec {
constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kRG = 4;               // 16-row groups per 64-row block
constexpr int kStA = 0;              // 4 x 512 B weight codes
constexpr int kStS = 2048;           // 4 x 64 B scales
constexpr int kStB = 2304;           // NG token groups x 8 rows x 144 B (BF16 x 64, padded: no bank conflicts)
constexpr int kRowPitch = 144;
constexpr int kSlots = kWarps - 1;   // shared-memory split-K slots: one per boundary between warps
// a stage holds activation rows for min(T, 8) tokens (one group) or 16 (two)
__host__ __device__ constexpr int stage_rows(int T) { return T <= 8 ? T : 16; }
__host__ __device__ constexpr int stage_bytes_for(int T) { return kStB + kRowPitch * stage_rows(T); }
// global split-K partial sums: per warp, two slots (its first and its last
// segment), each [rg 4][row 16][mslot] FP32 with mslot = min(T, 16)
constexpr uint64_t kTimeoutNs = 2000000000ull;
}  // namespace dec

struct RouteSmem {
  int ids[256];
  float wts[256];
  int perm[256];
  int inv[256];
  int off[257];
  int tch_e[256];
  int tch_r0[256];
  int tch_m[256];
  int U;
  int nan;
  int last_cta;
  unsigned xmax[16];
  int xexp[16];
};

struct FusedArgs {
  const uint8_t* blob;
  size_t expert_stride;
  size_t w13, w2;  // byte offsets of the gate/up and down matrices in an expert's blob
  const float* gscale;
  int E, H, I, T, k;  // E experts (routed + shared), k slots per token (top_k + shared)
  int Er, topk;       // routed experts (logits per token), routed choices per token
  int linear;         // 1: a dense linear: no routing, no gate/up; x [T][I] feeds the down GEMV
  RouteParams rp;     // scoring rule of the route step
  const float* in_scale;  // W4A4 routed experts: [E][2] input scales (w13, w2), else nullptr
  int n_out;          // a dense linear's output features (<= H; rows past it are padding)
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
  __nv_bfloat16* h;
  uint32_t* hmax;
  float* y;
  float* part_gu;
  int32_t* cnt_gu;
  float* part_dn;
  int32_t* cnt_dn;
  int mslot;      // token columns of a global partial-sum slot
  int no_split;   // 1: no global partial-sum buffers
  int slot_cols;  // token columns of a shared-memory split-K slot (0: none)
  int slot_sets;  // 2: separate shared-memory slots per phase; 1: one set, cleared between phases
  int xs_pitch;   // > 0: the tokens' FP16 activations are staged in shared memory, rows this many bytes apart
  int stage_bytes;  // bytes of one ring stage
  int32_t* done_gu;
  int32_t* cmb;
  int32_t* exit_cnt;
  DeviceStatus* st;
  DeviceStatus* st_sticky;    // optional: the last CTA ORs this launch's status into it
  int fault;                  // 1: no weight or activation copy is issued (tests the bounded waits)
  unsigned long long* trace;  // optional: [cta][warp][16] globaltimer stamps
};

__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// global -> shared bulk copy completing on an mbarrier (16-byte aligned, size % 16 == 0)
__device__ __forceinline__ void bulk_copy(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_addr(dst)),
               "l"(src), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}
__device__ __forceinline__ uint64_t now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ int ld_acquire(const int32_t* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ bool aborted(const DeviceStatus* st) {
  return (*reinterpret_cast<const volatile unsigned*>(&st->flags) & kFlagTimeout) != 0;
}

// Bounded wait on a ring stage; false if this or another warp gave up.
__device__ __forceinline__ bool ring_wait(uint64_t* bar, uint32_t parity, DeviceStatus* st) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = now_ns();
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 63u) {
      if (aborted(st)) return false;
      if (now_ns() - t0 > dec::kTimeoutNs) {
        report(st, kFlagTimeout, 300);
        return false;
      }
    }
  }
}

// 8 E2M1 codes (one 32-bit word, element 2j in the low nibble of byte j) ->
// four f16x2 registers {byte0, byte1, byte2, byte3}.
__device__ __forceinline__ void e2m1x8_to_f16(uint32_t w, uint32_t (&o)[4]) {
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
      : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
      : "r"(w));
}

__device__ __forceinline__ float pow2f(int p) {
  p = max(-126, min(127, p));
  return __int_as_float((127 + p) << 23);
}

// ---------------------------------------------------------------------------
// Phase 0: every CTA routes the T tokens into shared memory (warp t picks
// token t's experts), and takes each token's max |x| for the FP16 prescale
// (16/T warps per token).
// ---------------------------------------------------------------------------
// xs != nullptr: the tokens' activations are also left in shared memory as
// FP16 rows (xs_pitch bytes apart) after the per-token prescale.
__device__ void route_block(const FusedArgs& a, RouteSmem& rs, uint8_t* xs, unsigned long long* tr0) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // k slots per token: top_k routed choices, then the shared expert (id Er)
  // when the layer has one; E experts in all
  const int T = a.T, k = a.k, E = a.E, Er = a.Er, topk = a.topk, R = T * k;
  // loads first: token `warp`'s logits, and this warp's share of one x row
  uint32_t key[8];
  float val[8];
  // the logit loads are only issued here; their keys are taken after the x loads below are issued too
  if (warp < T && !a.linear) warp_issue_logits(a.logits, a.logits_bf16, Er, warp, val);
  const int wpt = dec::kWarps / T;  // warps per token row of x
  const int xt = warp / wpt, xpart = warp - xt * wpt;
  const int xcols = a.linear ? a.I : a.H;  // a linear's x rows have its K = I columns
  const int per_row = xcols / 8;           // 16-byte pieces per row
  float xm = 0.f;
  if (a.x && xt < T) {
    const uint4* row = reinterpret_cast<const uint4*>(a.x + (size_t)xt * xcols);
    for (int base = xpart * 32; base < per_row; base += 32 * wpt * 8) {
      uint4 v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int i = base + lane + j * 32 * wpt;
        if (i < per_row) v[j] = __ldg(row + i);
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int i = base + lane + j * 32 * wpt;
        if (i < per_row) {
          const uint32_t wv[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
          for (int q = 0; q < 4; ++q)
            xm = fmaxf(xm, fmaxf(fabsf(__uint_as_float(wv[q] << 16)), fabsf(__uint_as_float(wv[q] & 0xFFFF0000u))));
          if (xs) *reinterpret_cast<uint4*>(xs + (size_t)xt * a.xs_pitch + (size_t)i * 16) = v[j];
        }
      }
    }
  }
  if (warp < T && !a.linear) warp_logit_keys(val, key);
  if (tid < 16) rs.xmax[tid] = 0u;
  if (tid <= E) rs.off[tid] = 0;  // rows per expert, then offsets
  if (tid == 0) rs.nan = 0;
  __syncthreads();
  if (tr0 && tid == 0) tr0[8] = now_ns();
  if (a.x && xt < T) {  // |x| >= 0: its bits order like the values
    const unsigned m = __reduce_max_sync(0xffffffffu, __float_as_uint(xm));
    if (lane == 0) atomicMax(&rs.xmax[xt], m);
  }
  if (warp < T && a.linear) {  // a dense linear: every token to its one matrix, weight 1
    if (lane == 0) {
      rs.ids[warp] = 0;
      rs.wts[warp] = 1.0f;
      atomicAdd(&rs.off[0], 1);
    }
  } else if (warp < T) {
    int id;
    float logit;
    SoftmaxStats sst{0.f, 0.f, 0};
    if (a.rp.score == 0 && (a.rp.bias || !a.rp.renorm)) sst = warp_softmax_stats(val, Er);
    warp_bias_keys(a.rp, Er, val, key, sst);
    const int nt = warp_select_topk(key, val, Er, topk, &id, &logit);
    const float w = warp_route_weight(a.rp, logit, topk, Er, sst);
    if (lane < topk) {
      rs.ids[warp * k + lane] = id;
      rs.wts[warp * k + lane] = w;
      atomicAdd(&rs.off[id], 1);
    } else if (lane < k) {  // the shared expert: every token, weight 1
      rs.ids[warp * k + lane] = Er;
      rs.wts[warp * k + lane] = 1.0f;
      atomicAdd(&rs.off[Er], 1);
    }
    if (lane == 0 && nt) atomicAdd(&rs.nan, nt);
  }
  __syncthreads();
  if (tr0 && tid == 0) tr0[9] = now_ns();
  if (warp == 0) {
    // offsets (low 16 bits) and touched-expert slots (high 16 bits) in one
    // warp scan; lane l owns experts 8l .. 8l+7 (E <= 256, R <= 256)
    int cnt[8], s = 0, tc = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = 8 * lane + i;
      cnt[i] = e < E ? rs.off[e] : 0;
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
    for (int i = 0; i < 8; ++i) {
      const int e = 8 * lane + i;
      if (e < E) {
        rs.off[e] = off;
        if (cnt[i] > 0) {
          rs.tch_e[slot] = e;
          rs.tch_r0[slot] = off;
          rs.tch_m[slot] = cnt[i];
          ++slot;
        }
        off += cnt[i];
      }
    }
    if (lane == 31) {
      rs.off[E] = inc & 0xFFFF;
      rs.U = inc >> 16;
    }
  } else if (warp == 1 && lane < T) {
    rs.xexp[lane] = max(-126, min(126, prescale_exp(__uint_as_float(rs.xmax[lane]))));
  }
  __syncthreads();
  if (tr0 && tid == 0) tr0[10] = now_ns();
  if (tid < R) {  // expert-major position: rank among the earlier rows of the same expert
    const int e = rs.ids[tid];
    int rank = 0, j = 0;
    const int4* ids4 = reinterpret_cast<const int4*>(rs.ids);
    for (; j + 4 <= tid; j += 4) {
      const int4 q4 = ids4[j >> 2];
      rank += (q4.x == e) + (q4.y == e) + (q4.z == e) + (q4.w == e);
    }
    for (; j < tid; ++j) rank += (rs.ids[j] == e);
    const int pos = rs.off[e] + rank;
    rs.perm[pos] = tid;
    rs.inv[tid] = pos;
  }
  if (xs) {  // BF16 -> FP16 in place, times 2^-xexp[t] (exact)
    for (int i = tid; i < T * per_row; i += blockDim.x) {
      const int t = i / per_row;
      uint4* p = reinterpret_cast<uint4*>(xs + (size_t)t * a.xs_pitch + (size_t)(i - t * per_row) * 16);
      const float sc = pow2f(-rs.xexp[t]);
      const uint4 v = *p;
      uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int z = 0; z < 4; ++z) {
        const __half2 hh = __floats2half2_rn(__uint_as_float(w[z] << 16) * sc, __uint_as_float(w[z] & 0xFFFF0000u) * sc);
        w[z] = *reinterpret_cast<const uint32_t*>(&hh);
      }
      *p = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
  __syncthreads();
  if (blockIdx.x == 0) {  // the tables, for inspection
    if (tid < R) {
      a.ids[tid] = rs.ids[tid];
      a.wts[tid] = rs.wts[tid];
      a.perm[tid] = rs.perm[tid];
      a.inv[tid] = rs.inv[tid];
    }
    if (tid <= E) a.offsets[tid] = rs.off[tid];
    if (tid == 0 && rs.nan) atomicAdd(&a.st->nan_logits, (unsigned)rs.nan);
  }
}

// ---------------------------------------------------------------------------
// Piece finishing.  A piece is the 16-row groups [rg0, rg0 + cnt) of 64-row
// block b of touched expert u; acc[rg] holds group rg0 + rg.
// ---------------------------------------------------------------------------
__device__ void finish_gateup(const FusedArgs& a, const RouteSmem& rs, int u, int b, int rg0, int cnt,
                              float (&acc)[dec::kRG][2][4], int lane) {
  const int e = rs.tch_e[u], row0 = rs.tch_r0[u], m = rs.tch_m[u];
  const int r0 = lane >> 2, q = lane & 3;
  const float gsg = a.gscale[3 * e], gsu = a.gscale[3 * e + 1];
  float hmax[2][2] = {{0.f, 0.f}, {0.f, 0.f}};  // per token slot (i, c) of this lane
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int j = 8 * i + 2 * q + c;
      if (j >= m) continue;
      const int row = row0 + j;
      // W4A4 routed experts take unscaled quantised activations (no prescale)
      const float s = (a.in_scale && e < a.Er) ? 1.0f : pow2f(rs.xexp[rs.perm[row] / a.k]);
#pragma unroll
      for (int rg = 0; rg < dec::kRG; ++rg) {
        if (rg >= cnt) break;
        // packed rows 16g + r: gate row 8g + r (r < 8), up row 8g + r - 8
        const float g = gsg * (acc[rg][i][c] * s);
        const float uu = gsu * (acc[rg][i][2 + c] * s);
        const __nv_bfloat16 hb = __float2bfloat16_rn(silu(g) * uu);
        const int f = 8 * (dec::kRG * b + rg0 + rg) + r0;
        a.h[(size_t)row * a.I + f] = hb;
        hmax[i][c] = fmaxf(hmax[i][c], fabsf(__bfloat162float(hb)));
      }
    }
  // row maxima: reduce over the 8 lanes that share a token slot, then one
  // atomic per row from this piece
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      float v = hmax[i][c];
      v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
      v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
      v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
      const int j = 8 * i + 2 * q + c;
      if (r0 == 0 && j < m) atomicMax(&a.hmax[row0 + j], __float_as_uint(v));
    }
}

__device__ void finish_down(const FusedArgs& a, const RouteSmem& rs, int u, int b, int rg0, int cnt,
                            float (&acc)[dec::kRG][2][4], int lane) {
  const int e = rs.tch_e[u], row0 = rs.tch_r0[u], m = rs.tch_m[u];
  const int r0 = lane >> 2, q = lane & 3;
  const float gsd = a.gscale[3 * e + 2];
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int j = 8 * i + 2 * q + c;
      if (j >= m) continue;
      const int row = row0 + j;
      const float s = (a.in_scale && e < a.Er)
                          ? gsd
                          : gsd * pow2f(a.linear ? rs.xexp[rs.perm[row]]
                                                 : prescale_exp(__uint_as_float(__ldcg(a.hmax + row))));
      if (a.linear) {  // one slot per token, weight 1: the result is the output row itself
        const size_t o = (size_t)rs.perm[row] * a.n_out;
#pragma unroll
        for (int rg = 0; rg < dec::kRG; ++rg) {
          if (rg >= cnt) break;
          const int d = 16 * (dec::kRG * b + rg0 + rg) + r0;
          if (d >= a.n_out) break;  // a 16-row group is all padding or all real: n_out % 16 == 0
          if (a.out_f32) {
            reinterpret_cast<float*>(a.out)[o + d] = acc[rg][i][c] * s;
            reinterpret_cast<float*>(a.out)[o + d + 8] = acc[rg][i][2 + c] * s;
          } else {
            reinterpret_cast<__nv_bfloat16*>(a.out)[o + d] = __float2bfloat16_rn(acc[rg][i][c] * s);
            reinterpret_cast<__nv_bfloat16*>(a.out)[o + d + 8] = __float2bfloat16_rn(acc[rg][i][2 + c] * s);
          }
        }
        continue;
      }
#pragma unroll
      for (int rg = 0; rg < dec::kRG; ++rg) {
        if (rg >= cnt) break;
        const int d = 16 * (dec::kRG * b + rg0 + rg) + r0;
        a.y[(size_t)row * a.H + d] = acc[rg][i][c] * s;
        a.y[(size_t)row * a.H + d + 8] = acc[rg][i][2 + c] * s;
      }
    }
}

// Token t's 64-wide slice b of the output, once slice b is complete for
// every expert: out[t][slice] = sum_j w[t][j] * y[pos(t,j)][slice], slot
// order j = 0..k-1.  All k loads are issued before the first use (k <= 16).
__device__ void combine_slice_token(const FusedArgs& a, const RouteSmem& rs, int b, int t, int lane) {
  const int d = 64 * b + 2 * lane;
  float2 yy[16];
#pragma unroll
  for (int j = 0; j < 16; ++j)
    if (j < a.k) yy[j] = __ldcg(reinterpret_cast<const float2*>(a.y + (size_t)rs.inv[t * a.k + j] * a.H + d));
  float s0 = 0.f, s1 = 0.f;
#pragma unroll
  for (int j = 0; j < 16; ++j)
    if (j < a.k) {
      const float w = rs.wts[t * a.k + j];
      s0 = fmaf(w, yy[j].x, s0);
      s1 = fmaf(w, yy[j].y, s1);
    }
  if (a.out_f32) {
    *reinterpret_cast<float2*>(reinterpret_cast<float*>(a.out) + (size_t)t * a.H + d) = make_float2(s0, s1);
  } else {
    *reinterpret_cast<__nv_bfloat162*>(reinterpret_cast<__nv_bfloat16*>(a.out) + (size_t)t * a.H + d) =
        __floats2bfloat162_rn(s0, s1);
  }
}

// The combine, spread over every warp of the grid: task (slice b, token t),
// warp wg takes tasks wg, wg + W, ...; a task starts once all 4U 16-row groups
// of slice b are finished (counter cmb[b], bounded wait).
__device__ void combine_tasks(const FusedArgs& a, const RouteSmem& rs, long long wg, long long W, int lane) {
  const int nslices = a.H / 64;
  const int target = dec::kRG * rs.U;
  for (long long task = wg; task < (long long)nslices * a.T; task += W) {
    const int t = (int)(task / nslices), b = (int)(task - (long long)t * nslices);
    if (lane == 0) {
      const uint64_t t0 = now_ns();
      while (ld_acquire(a.cmb + b) < target) {
        if (aborted(a.st)) break;
        if (now_ns() - t0 > dec::kTimeoutNs) {
          report(a.st, kFlagTimeout, 400 + (unsigned)b);
          break;
        }
        __nanosleep(128);
      }
    }
    __syncwarp();
    if (aborted(a.st)) return;
    __threadfence();
    combine_slice_token(a, rs, b, t, lane);
  }
}

// ---------------------------------------------------------------------------
// Phases 1 and 2.  Work split: the units of a phase are the 16-row groups of
// the touched experts' matrices (gate/up: 2I/16 per expert, down: H/16),
// numbered expert-major.  CTA c takes units [g0, g1) (equal counts) over the
// whole K axis, so no output row's sum crosses CTAs.  Inside the CTA, the
// units of one 64-row block form a piece of nch 64-wide K chunks, and the
// (piece, chunk) items are cut into 16 equal contiguous warp ranges: split-K
// inside the CTA only.
// ---------------------------------------------------------------------------
struct CtaWork {
  int g0, g1;     // this CTA's units
  int B0;         // global 64-row block of piece 0
  int nch, nblk;  // chunks per piece; 64-row blocks per expert
  int nit;        // items: pieces x nch
  __device__ __forceinline__ void piece(int p, int* u, int* b, int* rg0, int* cnt) const {
    const int B = B0 + p;
    const int lo = max(g0, 4 * B), hi = min(g1, 4 * B + 4);
    *u = B / nblk;
    *b = B - *u * nblk;
    *rg0 = lo - 4 * B;
    *cnt = hi - lo;
  }
  __device__ __forceinline__ int unit_of(int p) const { return max(g0, 4 * (B0 + p)); }  // a piece's id
  // Warps split the CTA's items by an estimate of their time: a ring stage
  // costs about as much as four 16-row groups of a 64-wide chunk on top of
  // its bytes, so item i (piece p, chunk c) weighs kItemCost + cnt_p and
  // starts at cum(i) = nch * (units before p + kItemCost * p) + c * (kItemCost
  // + cnt_p); warp w takes the items with T_w <= cum(i) < T_w+1, T_w =
  // floor(cum(nit) * w / 16).
  static constexpr int kItemCost = 4;
  __device__ __forceinline__ long long cum(int i) const {
    const int p = i / nch;
    const int lo = unit_of(p), hi = min(g1, 4 * (B0 + p) + 4);
    return (long long)nch * ((lo - g0) + kItemCost * p) + (long long)(i - p * nch) * (kItemCost + hi - lo);
  }
  __device__ __forceinline__ long long total() const {
    return (long long)nch * ((g1 - g0) + kItemCost * (nit / nch));
  }
  __device__ __forceinline__ int range_lo(int w) const {
    if (w <= 0 || nit == 0) return 0;
    if (w >= dec::kWarps) return nit;
    const long long T = total() * w / dec::kWarps;
    int lo = 0, hi = nit;  // the first item with cum >= T (cum is increasing)
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (cum(mid) >= T) hi = mid;
      else lo = mid + 1;
    }
    return lo;
  }
  // the warp whose range [range_lo(w), range_lo(w + 1)) holds item i
  __device__ __forceinline__ int warp_of(int i) const {
    const long long tot = total();
    return (int)(((cum(i) + 1) * dec::kWarps + tot - 1) / tot) - 1;
  }
};

__device__ __forceinline__ CtaWork cta_work(long long units, int per_expert, int nch) {
  CtaWork w;
  const long long C = gridDim.x;
  w.g0 = (int)(units * blockIdx.x / C);
  w.g1 = (int)(units * (blockIdx.x + 1) / C);
  w.nch = nch;
  w.nblk = per_expert / 4;
  w.B0 = w.g0 >> 2;
  w.nit = w.g1 > w.g0 ? (((w.g1 - 1) >> 2) - w.B0 + 1) * nch : 0;
  return w;
}

// kXs: the routed tokens' activations are already in shared memory as
// prescaled FP16 rows (xs, xs_pitch bytes apart), so stages carry weights
// only (the gate/up phase of few-token steps, and a dense linear's one phase).  Every stage's weight copies are issued before its activation
// copies; at the start of the down phase all S-1 weight copies go out before
// the wait for the expert's h, so they land while the gate/up phase finishes.
// kQ4: the W4A4 variant is compiled in (the per-lane activation quantisation
// sits in the hot loop, so the W4A16 kernels leave it out).
template <bool kGateUp, int S, int NG, bool kXs, bool kQ4>
__device__ void run_phase(const FusedArgs& a, RouteSmem& rs, uint8_t* ring, uint64_t* bars, uint32_t& ring_it,
                          const CtaWork& cw, unsigned long long* tr, float* part_s, int* cnt_s,
                          const uint8_t* xs) {
  const int kStageBytes = a.stage_bytes;
  const int srows = dec::stage_rows(a.T);  // activation rows a stage holds
  constexpr bool kActCopies = !kXs;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, q = lane & 3, r0 = lane >> 2;
  const int nch = cw.nch;
  const int gu_units = 2 * a.I / 16;
  const int scol = a.slot_cols;  // token columns of a shared-memory slot
  const size_t mat_off = kGateUp ? a.w13 : a.w2;
  // without shared-memory slots or global partial buffers: whole pieces per warp
  const bool whole_only = a.no_split && part_s == nullptr;
  int ibeg, iend;
  if (whole_only) {
    const int np = cw.nit / nch;
    ibeg = np * warp / dec::kWarps * nch;
    iend = np * (warp + 1) / dec::kWarps * nch;
  } else {
    ibeg = cw.range_lo(warp);
    iend = cw.range_lo(warp + 1);
  }
  const int nf = iend - ibeg;
  if (nf <= 0) return;
  const uint32_t it0 = ring_it;
  bool dead = false;

  // ---- producer: weight copies (with the stage's byte count), then
  // activation copies, S-1 items ahead of the consumer ----
  int wpp = ibeg / nch, wpc = ibeg - (ibeg / nch) * nch, wp_cur = -1, w_cnt = 0, w_m = 0;
  size_t w_seg = 0;
  const uint8_t* w_mat = nullptr;
  auto issue_w = [&](uint32_t it) {
    if (wpp != wp_cur) {
      int u, b, rg0, cnt;
      cw.piece(wpp, &u, &b, &rg0, &cnt);
      const int e = rs.tch_e[u];
      w_m = kActCopies ? min(rs.tch_m[u], 8 * NG) : 0;
      w_mat = a.blob + (size_t)e * a.expert_stride + mat_off;
      // 16-row group g of 128-row block B2 at K chunk c is 512-byte segment
      // (B2 * nch + c) * 8 + (g & 7); 64-row block b is groups 4(b&1)..+3 of B2 = b >> 1
      w_seg = (size_t)(b >> 1) * nch * 8 + 4 * (b & 1) + rg0;
      w_cnt = cnt;
      wp_cur = wpp;
    }
    uint64_t* bar = bars + (int)(it % S);
    uint8_t* st = ring + (int)(it % S) * kStageBytes;
    const size_t seg0 = w_seg + (size_t)wpc * 8;
    // earlier generic reads and writes of this memory come before the copies
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (lane == 0 && !a.fault) {
      mbar_expect_tx(bar, (uint32_t)w_cnt * (512u + 64u) + 128u * (uint32_t)w_m);
      // the piece's 16-row groups (seg0 & 7 ..) lie inside tile seg0 >> 3: codes, then scales
      const uint8_t* tile = w_mat + (seg0 >> 3) * kTileBytes;
      bulk_copy(st + dec::kStA, tile + (seg0 & 7) * 512, 512u * (uint32_t)w_cnt, bar);
      bulk_copy(st + dec::kStS, tile + kTileCodes + (seg0 & 7) * 64, 64u * (uint32_t)w_cnt, bar);
    }
    if (++wpc == nch) {
      wpc = 0;
      ++wpp;
    }
  };
  int app = ibeg / nch, apc = ibeg - (ibeg / nch) * nch, ap_cur = -1, ap_u = -1, a_m = 0;
  const uint8_t* a_row = nullptr;  // lane j < m: its routed row's activations (bytes)
  auto issue_a = [&](uint32_t it) {
    if (!kActCopies) return;
    if (app != ap_cur) {
      int u, b, rg0, cnt;
      cw.piece(app, &u, &b, &rg0, &cnt);
      if (u != ap_u) {
        if (!kGateUp && !a.linear) {  // h of expert u must be complete
          if (lane == 0) {
            const uint64_t t0 = now_ns();
            while (ld_acquire(a.done_gu + u) < gu_units) {
              if (aborted(a.st)) break;
              if (now_ns() - t0 > dec::kTimeoutNs) {
                report(a.st, kFlagTimeout, 100 + (unsigned)u);
                break;
              }
              __nanosleep(64);
            }
          }
          __syncwarp();
          __threadfence();
          // h was written through the generic proxy; the copies read it through the async proxy
          asm volatile("fence.proxy.async.global;" ::: "memory");
          if (aborted(a.st)) dead = true;
          if (tr && lane == 0 && tr[3] == 0) tr[3] = now_ns();
        }
        const int row0 = rs.tch_r0[u];
        a_m = min(rs.tch_m[u], 8 * NG);
        a_row = nullptr;
        if (lane < a_m)
          a_row = kGateUp    ? reinterpret_cast<const uint8_t*>(a.x + (size_t)(rs.perm[row0 + lane] / a.k) * a.H)
                  : a.linear ? reinterpret_cast<const uint8_t*>(a.x + (size_t)rs.perm[row0 + lane] * a.I)
                             : reinterpret_cast<const uint8_t*>(a.h + (size_t)(row0 + lane) * a.I);
        ap_u = u;
      }
      ap_cur = app;
    }
    uint8_t* st = ring + (int)(it % S) * kStageBytes;
    __syncwarp();  // the stage's expect_tx (lane 0) comes first
    if (lane < a_m && !a.fault)
      bulk_copy(st + dec::kStB + (lane >> 3) * 8 * dec::kRowPitch + (lane & 7) * dec::kRowPitch,
                a_row + (size_t)apc * 128, 128, bars + (int)(it % S));
    if (++apc == nch) {
      apc = 0;
      ++app;
    }
  };

  // ---- consumer state ----
  int cpi = ibeg / nch, cc = ibeg - (ibeg / nch) * nch;
  float acc[dec::kRG][2][4];
  float bsc[2] = {1.f, 1.f};
  const uint8_t* xrow = nullptr;  // kXs: this lane's token row
  int seg_c0 = 0, m = 0, ng = 1, cu = 0, cb = 0, crg0 = 0, ccnt = 0;
  bool q4 = false;  // this piece's activations are quantised to NVFP4 (W4A4 routed expert)
  float q4_is = 0.f, q4_inv6 = 0.f;
  bool fin_head = false, fin_tail = false;  // split segments this warp finished in the loop
  int issued = 0, consumed = 0;

  const int pro = min(S - 1, nf);
  for (int j = 0; j < pro; ++j) issue_w(it0 + j);
  for (int j = 0; j < pro; ++j) issue_a(it0 + j);
  issued = pro;
  for (int i = 0; i < nf && !dead; ++i) {
    const uint32_t it = it0 + i;
    if (issued < nf) {
      issue_w(it0 + issued);
      issue_a(it0 + issued);
      ++issued;
    }
    if (dead) break;
    if (!ring_wait(bars + it % S, (it / S) & 1u, a.st)) {
      dead = true;
      break;
    }
    if (kGateUp && i == 0 && tr && lane == 0) tr[13] = now_ns();
    consumed = i + 1;
    const int c = cc, p = cpi;
    if (i == 0 || c == 0) {
      seg_c0 = c;
      cw.piece(p, &cu, &cb, &crg0, &ccnt);
      const int row0 = rs.tch_r0[cu];
      m = rs.tch_m[cu];
      q4 = kQ4 && a.in_scale != nullptr && rs.tch_e[cu] < a.Er;
      if (q4) {
        q4_is = __ldg(a.in_scale + 2 * rs.tch_e[cu] + (kGateUp ? 0 : 1));
        q4_inv6 = act_inv6(q4_is);
      }
      ng = (m + 7) >> 3;
#pragma unroll
      for (int rg = 0; rg < dec::kRG; ++rg)
#pragma unroll
        for (int gi = 0; gi < 2; ++gi)
#pragma unroll
          for (int z = 0; z < 4; ++z) acc[rg][gi][z] = 0.f;
      if (kXs) {
        // rows >= m read row 0's token (their MMA columns are never used)
        xrow = xs + (size_t)(rs.perm[row0 + (r0 < m ? r0 : 0)] / a.k) * a.xs_pitch + q * 32;
      } else {
#pragma unroll
        for (int gi = 0; gi < 2; ++gi) {
          const int j = 8 * gi + r0;
          int pe = 0;
          if (j < m) {
            const int row = row0 + j;
            pe = (kGateUp || a.linear) ? rs.xexp[rs.perm[row] / a.k]
                                       : max(-126, min(126, prescale_exp(__uint_as_float(__ldcg(a.hmax + row)))));
          }
          bsc[gi] = pow2f(-pe);
        }
      }
    }
    const uint8_t* st = ring + (int)(it % S) * kStageBytes;
    // activations: FP16 after the row prescale (rows >= m hold stale data;
    // their MMA columns are never read)
    uint32_t bw[2][8];
    if (kXs) {
      const uint4 u0 = *reinterpret_cast<const uint4*>(xrow + (size_t)c * 128);
      const uint4 u1 = *reinterpret_cast<const uint4*>(xrow + (size_t)c * 128 + 16);
      bw[0][0] = u0.x, bw[0][1] = u0.y, bw[0][2] = u0.z, bw[0][3] = u0.w;
      bw[0][4] = u1.x, bw[0][5] = u1.y, bw[0][6] = u1.z, bw[0][7] = u1.w;
    } else {
#pragma unroll
      for (int gi = 0; gi < NG; ++gi) {
        if (gi < ng) {
          const int srow = 8 * gi + r0 < srows ? 8 * gi + r0 : 0;  // rows past the stage's read row 0
          const uint8_t* pa = st + dec::kStB + srow * dec::kRowPitch + q * 32;
          const uint4 u0 = *reinterpret_cast<const uint4*>(pa), u1 = *reinterpret_cast<const uint4*>(pa + 16);
          const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
          if (kQ4 && q4) {  // this lane's 16 K elements are one NVFP4 block
            float v[16];
#pragma unroll
            for (int z = 0; z < 8; ++z) {
              v[2 * z] = __uint_as_float(w[z] << 16);
              v[2 * z + 1] = __uint_as_float(w[z] & 0xFFFF0000u);
            }
            act_quant16_f16(v, q4_is, q4_inv6, bw[gi]);
          } else {
#pragma unroll
            for (int z = 0; z < 8; ++z) {
              const __half2 hh = __floats2half2_rn(__uint_as_float(w[z] << 16) * bsc[gi],
                                                   __uint_as_float(w[z] & 0xFFFF0000u) * bsc[gi]);
              bw[gi][z] = *reinterpret_cast<const uint32_t*>(&hh);
            }
          }
        }
      }
    }
#pragma unroll
    for (int rg = 0; rg < dec::kRG; ++rg) {
      if (rg >= ccnt) break;
      const uint4 raw = *reinterpret_cast<const uint4*>(st + dec::kStA + rg * 512 + seg_pos(lane) * 16);
      const uint32_t s2 =
          e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(st + dec::kStS + rg * 64 + seg_pos(lane) * 2));
      const uint32_t s0 = dup_lo(s2), s1 = dup_hi(s2);
      uint32_t cx[4], cy[4], cz[4], cw4[4];
      e2m1x8_to_f16(raw.x, cx);
      e2m1x8_to_f16(raw.y, cy);
      e2m1x8_to_f16(raw.z, cz);
      e2m1x8_to_f16(raw.w, cw4);
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        cx[t] = hmul2_u32(cx[t], s0);
        cy[t] = hmul2_u32(cy[t], s0);
        cz[t] = hmul2_u32(cz[t], s1);
        cw4[t] = hmul2_u32(cw4[t], s1);
      }
#pragma unroll
      for (int kt = 0; kt < 4; ++kt) {
        const uint32_t* r0w = kt < 2 ? cx : cy;
        const uint32_t* r8w = kt < 2 ? cz : cw4;
        const int o = 2 * (kt & 1);
        mma_f16_16816(acc[rg][0], r0w[o], r8w[o], r0w[o + 1], r8w[o + 1], bw[0][2 * kt], bw[0][2 * kt + 1]);
        if (NG > 1 && ng > 1)
          mma_f16_16816(acc[rg][1], r0w[o], r8w[o], r0w[o + 1], r8w[o + 1], bw[1][2 * kt], bw[1][2 * kt + 1]);
      }
    }
    __syncwarp();  // every lane is done reading this stage before it is refilled
    if (++cc == nch) {
      cc = 0;
      ++cpi;
    }
    const bool seg_end = (c == nch - 1) || (i == nf - 1);
    if (!seg_end) continue;
    if (seg_c0 == 0 && c == nch - 1) {  // the whole piece is this warp's: finish it now, signal later
      if (kGateUp) finish_gateup(a, rs, cu, cb, crg0, ccnt, acc, lane);
      else finish_down(a, rs, cu, cb, crg0, ccnt, acc, lane);
      continue;
    }
    const bool head = (i - (c - seg_c0)) == 0;  // the segment starts this warp's range
    if (part_s != nullptr) {
      // split among warps of this CTA: shared-memory sum, the last one finishes
      const int slot = cw.warp_of(p * nch);  // the warp holding the piece's first chunk
      float* ps = part_s + slot * 64 * scol;
#pragma unroll
      for (int rg = 0; rg < dec::kRG; ++rg) {
        if (rg >= ccnt) break;
#pragma unroll
        for (int gi = 0; gi < NG; ++gi)
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            const int j = 8 * gi + 2 * q + h2;
            if (j < m) {
              atomicAdd(ps + (rg * 16 + r0) * scol + j, acc[rg][gi][h2]);
              atomicAdd(ps + (rg * 16 + r0 + 8) * scol + j, acc[rg][gi][2 + h2]);
            }
          }
      }
      __syncwarp();
      int last = 0;
      if (lane == 0) {
        __threadfence_block();
        const int add = c - seg_c0 + 1;
        last = (atomicAdd(cnt_s + slot, add) + add == nch);
      }
      last = __shfl_sync(0xffffffffu, last, 0);
      if (last) {
        __threadfence_block();
#pragma unroll
        for (int rg = 0; rg < dec::kRG; ++rg)
#pragma unroll
          for (int gi = 0; gi < 2; ++gi)
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              const int j = 8 * gi + 2 * q + h2;
              const bool ok = gi < NG && j < m && rg < ccnt;
              acc[rg][gi][h2] = ok ? ps[(rg * 16 + r0) * scol + j] : 0.f;
              acc[rg][gi][2 + h2] = ok ? ps[(rg * 16 + r0 + 8) * scol + j] : 0.f;
            }
        if (kGateUp) finish_gateup(a, rs, cu, cb, crg0, ccnt, acc, lane);
        else finish_down(a, rs, cu, cb, crg0, ccnt, acc, lane);
        if (head) fin_head = true;
        else fin_tail = true;
      }
      continue;
    }
    // no shared-memory slots: store the partial sums into this warp's global
    // slot (0: its first segment, 1: its last); counted in at the end of the phase
    {
      float* part = (kGateUp ? a.part_gu : a.part_dn) +
                    (((size_t)blockIdx.x * dec::kWarps + warp) * 2 + (head ? 0 : 1)) * 64 * a.mslot;
#pragma unroll
      for (int rg = 0; rg < dec::kRG; ++rg) {
        if (rg >= ccnt) break;
#pragma unroll
        for (int gi = 0; gi < 2; ++gi)
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            const int j = 8 * gi + 2 * q + h2;
            if (j < m) {
              __stcg(part + (rg * 16 + r0) * a.mslot + j, acc[rg][gi][h2]);
              __stcg(part + (rg * 16 + r0 + 8) * a.mslot + j, acc[rg][gi][2 + h2]);
            }
          }
      }
    }
  }
  if (tr && lane == 0) tr[kGateUp ? 11 : 12] = now_ns();

  // ---- end of phase: one fence covers every store and partial sum above ----
  if (!dead) {
    const uint64_t t_fin = tr ? now_ns() : 0;
    bool fin_global = false;
    __threadfence();
    __syncwarp();
    // pass 1: count the split segments that went through global slots in; the
    // last contributor of a piece finishes it
    for (int f = ibeg; f < iend;) {
      const int p = f / nch, c0 = f - (f / nch) * nch;
      const int c1 = min(nch, c0 + (iend - f));
      const bool head = f == ibeg;
      f += c1 - c0;
      if ((c0 == 0 && c1 == nch) || part_s != nullptr) continue;
      int32_t* cnt = (kGateUp ? a.cnt_gu : a.cnt_dn) + cw.unit_of(p);
      int last = 0;
      if (lane == 0) last = (atomicAdd(cnt, c1 - c0) + (c1 - c0) == nch);
      last = __shfl_sync(0xffffffffu, last, 0);
      if (!last) continue;
      __threadfence();
      int u, b, rg0, pcnt;
      cw.piece(p, &u, &b, &rg0, &pcnt);
      const int mm = rs.tch_m[u];
#pragma unroll
      for (int rg = 0; rg < dec::kRG; ++rg)
#pragma unroll
        for (int gi = 0; gi < 2; ++gi)
#pragma unroll
          for (int z = 0; z < 4; ++z) acc[rg][gi][z] = 0.f;
      // contributors: this CTA's warps whose ranges meet the piece's items
      const int i0 = p * nch, i1 = i0 + nch;
      for (int w = cw.warp_of(i0); w <= cw.warp_of(i1 - 1); ++w) {
        const int s0 = cw.range_lo(w), s1 = cw.range_lo(w + 1);
        if (s0 >= s1 || s1 <= i0 || s0 >= i1) continue;
        const float* part = (kGateUp ? a.part_gu : a.part_dn) +
                            (((size_t)blockIdx.x * dec::kWarps + w) * 2 + (s0 >= i0 ? 0 : 1)) * 64 * a.mslot;
#pragma unroll
        for (int rg = 0; rg < dec::kRG; ++rg) {
          if (rg >= pcnt) break;
#pragma unroll
          for (int gi = 0; gi < 2; ++gi)
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              const int j = 8 * gi + 2 * q + h2;
              if (j < mm) {
                acc[rg][gi][h2] += __ldcg(part + (rg * 16 + r0) * a.mslot + j);
                acc[rg][gi][2 + h2] += __ldcg(part + (rg * 16 + r0 + 8) * a.mslot + j);
              }
            }
        }
      }
      if (lane == 0) *cnt = 0;
      if (kGateUp) finish_gateup(a, rs, u, b, rg0, pcnt, acc, lane);
      else finish_down(a, rs, u, b, rg0, pcnt, acc, lane);
      if (head) fin_head = true;
      else fin_tail = true;
      fin_global = true;
    }
    // pass 2: after one more fence (only if pass 1 wrote results), signal
    // every piece this warp finished
    if (fin_global) {
      __threadfence();
      __syncwarp();
    }
    for (int f = ibeg; f < iend;) {
      const int p = f / nch, c0 = f - (f / nch) * nch;
      const int c1 = min(nch, c0 + (iend - f));
      const bool head = f == ibeg;
      f += c1 - c0;
      if (!((c0 == 0 && c1 == nch) || (head ? fin_head : fin_tail))) continue;
      int u, b, rg0, pcnt;
      cw.piece(p, &u, &b, &rg0, &pcnt);
      if (kGateUp) {
        if (lane == 0) atomicAdd(&a.done_gu[u], pcnt);
      } else {
        if (lane == 0) atomicAdd(&a.cmb[b], pcnt);
      }
    }
    if (tr && lane == 0) tr[kGateUp ? 6 : 7] += now_ns() - t_fin;
  }
  // on a normal exit every issued stage was consumed; after an abort, give the
  // copies still in flight a bounded chance to land before the ring is reused
  // (with the test fault set, no copy was ever issued)
  if (dead && !a.fault) {
    for (int i = consumed; i < issued; ++i) {
      const uint32_t it = it0 + i;
      const uint64_t t0 = now_ns();
      while (!mbar_try_wait(bars + it % S, (it / S) & 1u) && now_ns() - t0 < dec::kTimeoutNs) {
      }
    }
  }
  ring_it = it0 + (uint32_t)issued;
}

// kLin: a dense linear with its x staged in shared memory (its one phase reads
// the tokens' rows from there); the other linear cases run the general kernel.
template <int S, int NG, bool kQ4, bool kLin = false>
__global__ void __launch_bounds__(dec::kThreads, 1) decode_fused_kernel(FusedArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  const uint64_t t_start = now_ns();
  const long long c_start = clock64();
  // shared memory: routing tables | ring barriers | per-warp rings | split-K
  // slot counters [2][16] | slots [slot_sets][15][64 rows][slot_cols] | staged FP16 activations
  RouteSmem& rs = *reinterpret_cast<RouteSmem*>(smem);
  const size_t route_bytes = (sizeof(RouteSmem) + 127) & ~size_t(127);
  uint64_t* all_bars = reinterpret_cast<uint64_t*>(smem + route_bytes);
  uint8_t* rings = smem + route_bytes + 128 * 8;
  uint8_t* tail = rings + (size_t)dec::kWarps * S * a.stage_bytes;
  int* cnt_all = reinterpret_cast<int*>(tail);
  float* slots = reinterpret_cast<float*>(tail + 128);
  const int slot_floats = dec::kSlots * 64 * a.slot_cols;
  uint8_t* xs = a.xs_pitch > 0 ? tail + 128 + (size_t)a.slot_sets * slot_floats * 4 : nullptr;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* ring = rings + (size_t)warp * S * a.stage_bytes;
  uint64_t* bars = all_bars + warp * 8;
  auto clear_slots = [&](int sets) {
    for (int i = threadIdx.x; i < sets * slot_floats; i += blockDim.x) slots[i] = 0.f;
    if (threadIdx.x < 32) cnt_all[threadIdx.x] = 0;
  };
  // ring barriers and slots are set up while routing runs (its barriers order them)
  if (!a.route_only) {
    if (lane == 0) {
      for (int s = 0; s < S; ++s) mbar_init(bars + s, 1);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (a.slot_cols) clear_slots(a.slot_sets);
  }
  route_block(a, rs, xs, a.trace ? a.trace + (size_t)blockIdx.x * dec::kWarps * 16 : nullptr);
  if (a.route_only) return;
  unsigned long long* tr = a.trace ? a.trace + ((size_t)blockIdx.x * dec::kWarps + warp) * 16 : nullptr;
  if (tr && lane == 0) {
    tr[0] = t_start;
    tr[1] = now_ns();
    tr[14] = (unsigned long long)c_start;
    tr[15] = (unsigned long long)clock64();
  }
  __syncwarp();

  const int U = rs.U;
  uint32_t ring_it = 0;
  float* slots1 = a.slot_cols ? slots : nullptr;
  float* slots2 = slots1;
  if (!kLin && !a.linear) {  // a dense linear has no gate/up phase: its x goes straight to the down GEMV
    const CtaWork w1 = cta_work((long long)U * (2 * a.I / 16), 2 * a.I / 16, a.H / kChunk);
    if (xs)
      run_phase<true, S, NG, true, kQ4>(a, rs, ring, bars, ring_it, w1, tr, slots1, cnt_all, xs);
    else
      run_phase<true, S, NG, false, kQ4>(a, rs, ring, bars, ring_it, w1, tr, slots1, cnt_all, nullptr);
    if (tr && lane == 0) tr[2] = now_ns();
    if (a.slot_cols && a.slot_sets == 2) {
      slots2 = slots + slot_floats;  // the down phase has its own slots: no CTA barrier here
    } else if (a.slot_cols) {        // one set, reused by the down phase
      __syncthreads();
      clear_slots(1);
      __syncthreads();
    }
  }
  const CtaWork w2 = cta_work((long long)U * (a.H / 16), a.H / 16, a.I / kChunk);
  if constexpr (kLin)
    run_phase<false, S, NG, true, false>(a, rs, ring, bars, ring_it, w2, tr, slots2, cnt_all, xs);
  else
    run_phase<false, S, NG, false, kQ4>(a, rs, ring, bars, ring_it, w2, tr, slots2,
                                        cnt_all + (a.slot_sets == 2 ? 16 : 0), nullptr);
  if (tr && lane == 0) tr[4] = now_ns();
  if (!a.linear)
    combine_tasks(a, rs, (long long)blockIdx.x * dec::kWarps + warp, (long long)gridDim.x * dec::kWarps, lane);

  // the last CTA out resets the per-forward counters (and, after a timeout,
  // every arrival counter) for the next forward
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    rs.last_cta = atomicAdd(a.exit_cnt, 1) == (int)gridDim.x - 1;
  }
  __syncthreads();
  if (tr && lane == 0) tr[5] = now_ns();
  if (!rs.last_cta) return;
  __threadfence();
  if (a.st_sticky && threadIdx.x == 0) {  // every CTA's reports are in: carry them over
    const unsigned f = atomicOr(&a.st->flags, 0u), n = atomicAdd(&a.st->nan_logits, 0u);
    if (f && atomicOr(&a.st_sticky->flags, f) == 0u) a.st_sticky->where = *reinterpret_cast<volatile unsigned*>(&a.st->where);
    if (n) atomicAdd(&a.st_sticky->nan_logits, n);
  }
  const int R = a.T * a.k;
  for (int i = threadIdx.x; i < U; i += blockDim.x) a.done_gu[i] = 0;
  for (int i = threadIdx.x; i < R; i += blockDim.x) a.hmax[i] = 0u;
  for (int i = threadIdx.x; i < a.H / 64; i += blockDim.x) a.cmb[i] = 0;
  if (aborted(a.st)) {
    const size_t ngu = a.linear ? 0 : (size_t)U * (2 * a.I / 16), ndn = (size_t)U * (a.H / 16);
    for (size_t i = threadIdx.x; i < ngu; i += blockDim.x) a.cnt_gu[i] = 0;
    for (size_t i = threadIdx.x; i < ndn; i += blockDim.x) a.cnt_dn[i] = 0;
  }
  __syncthreads();
  if (threadIdx.x == 0) *a.exit_cnt = 0;
}

// Shared memory: T <= 8 (one token group per expert) adds split-K slots,
// one set per phase when both fit, and stages the tokens' activations when
// they fit too, with the deepest rings (3..5 stages per warp) that leave room
// for both; T <= 16 (two token groups): 2 stages and one set of split-K slots
// (cleared between the phases).  Environment variables (read once):
// NVFP4_MOE_DECODE_STAGES caps the ring depth, NVFP4_MOE_DECODE_STAGE_X=0
// turns activation staging off, NVFP4_MOE_DECODE_T16_SLOTS=0 gives T > 8
// three stages and global split-K slots instead.
struct DecodeSmemPlan {
  size_t bytes;
  int stages, slot_cols, slot_sets, xs_pitch;
};
static int decode_stage_cap() {
  static const int cap = [] {
    const char* s = getenv("NVFP4_MOE_DECODE_STAGES");
    const int v = s ? atoi(s) : 5;
    return v < 2 ? 2 : (v > 5 ? 5 : v);
  }();
  return cap;
}
static DecodeSmemPlan plan_smem(int T, int H, int linear, bool no_xs, int smem_max) {
  const size_t base = ((sizeof(RouteSmem) + 127) & ~size_t(127)) + 128 * 8 + 128;
  const size_t ring1 = (size_t)dec::kWarps * dec::stage_bytes_for(T);  // one stage per warp
  const int cap = decode_stage_cap();
  if (linear && T <= 8) {  // one phase: one set of slots; x staged (H = the linear's K) when it fits
    const size_t slot_b = (size_t)dec::kSlots * 64 * T * 4;
    const size_t xs_b = (size_t)T * (2 * H + 16);
    for (int S = cap; S >= 3; --S)
      if (base + S * ring1 + slot_b + xs_b <= (size_t)smem_max)
        return DecodeSmemPlan{base + S * ring1 + slot_b + xs_b, S, T, 1, 2 * H + 16};
    for (int S = cap; S > 3; --S)
      if (base + S * ring1 + slot_b <= (size_t)smem_max) return DecodeSmemPlan{base + S * ring1 + slot_b, S, T, 1, 0};
    return DecodeSmemPlan{base + 3 * ring1 + slot_b, cap < 3 ? cap : 3, T, 1, 0};
  }
  if (T > 8) {  // two ring stages and one set of shared-memory split-K slots, else three stages
    static const bool slots16 = [] {
      const char* s = getenv("NVFP4_MOE_DECODE_T16_SLOTS");
      return !(s && s[0] == '0');
    }();
    const size_t slot_b = (size_t)dec::kSlots * 64 * T * 4;
    if (slots16 && base + 2 * ring1 + slot_b <= (size_t)smem_max)
      return DecodeSmemPlan{base + 2 * ring1 + slot_b, 2, T, 1, 0};
    const int S = cap < 3 ? cap : 3;
    return DecodeSmemPlan{base + S * ring1, S, 0, 0, 0};
  }
  const size_t slot_b = (size_t)dec::kSlots * 64 * T * 4;
  const size_t xs_b = (size_t)T * (2 * H + 16);
  static const bool stage_x = [] {
    const char* s = getenv("NVFP4_MOE_DECODE_STAGE_X");
    return !(s && s[0] == '0');
  }();
  for (int S = cap; S >= 3 && stage_x && !no_xs; --S)
    if (base + S * ring1 + 2 * slot_b + xs_b <= (size_t)smem_max)
      return DecodeSmemPlan{base + S * ring1 + 2 * slot_b + xs_b, S, T, 2, 2 * H + 16};
  const int S = cap < 3 ? cap : 3;
  if (base + S * ring1 + 2 * slot_b <= (size_t)smem_max) return DecodeSmemPlan{base + S * ring1 + 2 * slot_b, S, T, 2, 0};
  return DecodeSmemPlan{base + S * ring1 + slot_b, S, T, 1, 0};
}

// The opt-in shared-memory size of every decode kernel instantiation,
// set once per device (function attributes belong to each device's context).
cudaError_t decode_prepare_device(int dev, int* smem_max) {
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
  const void* fns[] = {(const void*)decode_fused_kernel<2, 1, false>, (const void*)decode_fused_kernel<3, 1, false>,
                       (const void*)decode_fused_kernel<4, 1, false>, (const void*)decode_fused_kernel<5, 1, false>,
                       (const void*)decode_fused_kernel<2, 2, false>, (const void*)decode_fused_kernel<3, 2, false>,
                       (const void*)decode_fused_kernel<3, 1, true>,  (const void*)decode_fused_kernel<2, 2, true>,
                       (const void*)decode_fused_kernel<3, 2, true>,
                       (const void*)decode_fused_kernel<3, 1, false, true>,
                       (const void*)decode_fused_kernel<4, 1, false, true>,
                       (const void*)decode_fused_kernel<5, 1, false, true>};
  for (const void* f : fns)
    if (e == cudaSuccess) e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < kCached) cached[dev] = optin;
  *smem_max = optin;
  return cudaSuccess;
}

cudaError_t launch_decode_forward(const LayerDims& d, const uint8_t* blob, const float* gscale, const void* logits,
                                  const void* x, int T, int k, void* out, int route_only, int num_sms,
                                  const Workspace& ws, int fault, cudaStream_t st) {
  int dev = 0, smem_max = 0;
  cudaError_t de = cudaGetDevice(&dev);
  if (de == cudaSuccess) de = decode_prepare_device(dev, &smem_max);
  if (de != cudaSuccess) return de;
  const bool small = T <= 8;
  // W4A4 quantises activations from their BF16 values: no staged FP16 copy
  const DecodeSmemPlan plan = plan_smem(T, d.linear ? d.I : d.H, d.linear, d.in_scale != nullptr, smem_max);
  if (plan.bytes > (size_t)smem_max) return cudaErrorInvalidConfiguration;
  const ExpertLayout L = d.linear ? linear_layout(d.H, d.I) : expert_layout(d.H, d.I);
  FusedArgs a{};
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
  a.linear = d.linear;
  a.n_out = d.n_out;
  a.rp = d.rp;
  a.in_scale = d.in_scale;
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
  a.h = ws.h;
  a.hmax = ws.hmax;
  a.y = ws.y;
  a.part_gu = ws.part_gu;
  a.cnt_gu = ws.cnt_gu;
  a.part_dn = ws.part_dn;
  a.cnt_dn = ws.cnt_dn;
  a.mslot = T < 16 ? T : 16;
  a.no_split = ws.part_gu == nullptr;
  a.slot_cols = plan.slot_cols;
  a.slot_sets = plan.slot_sets;
  a.xs_pitch = plan.xs_pitch;
  a.stage_bytes = dec::stage_bytes_for(T);
  a.done_gu = ws.done_gu;
  a.cmb = ws.cmb;
  a.exit_cnt = ws.exit_cnt;
  a.st = ws.status;
  a.st_sticky = ws.status_sticky;
  a.fault = fault;
  a.trace = ws.trace;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(route_only ? 1 : num_sms);
  cfg.blockDim = dim3(dec::kThreads);
  cfg.dynamicSmemBytes = plan.bytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = route_only ? 0 : 1;
  if (d.linear && plan.xs_pitch > 0) {  // a dense linear with its x staged in shared memory
    switch (plan.stages) {
      case 3: return cudaLaunchKernelEx(&cfg, decode_fused_kernel<3, 1, false, true>, a);
      case 4: return cudaLaunchKernelEx(&cfg, decode_fused_kernel<4, 1, false, true>, a);
      case 5: return cudaLaunchKernelEx(&cfg, decode_fused_kernel<5, 1, false, true>, a);
      default: return cudaErrorInvalidConfiguration;  // the ring depth must match the kernel's
    }
  }
  if (d.in_scale) {  // W4A4: its own instantiations (three-stage rings for T <= 8)
    if (!small) return plan.stages == 2 ? cudaLaunchKernelEx(&cfg, decode_fused_kernel<2, 2, true>, a)
                                        : cudaLaunchKernelEx(&cfg, decode_fused_kernel<3, 2, true>, a);
    if (plan.stages != 3) return cudaErrorInvalidConfiguration;  // the ring depth must match the kernel's
    return cudaLaunchKernelEx(&cfg, decode_fused_kernel<3, 1, true>, a);
  }
  if (!small) return plan.stages == 2 ? cudaLaunchKernelEx(&cfg, decode_fused_kernel<2, 2, false>, a)
                                      : cudaLaunchKernelEx(&cfg, decode_fused_kernel<3, 2, false>, a);
  switch (plan.stages) {
    case 2: return cudaLaunchKernelEx(&cfg, decode_fused_kernel<2, 1, false>, a);
    case 3: return cudaLaunchKernelEx(&cfg, decode_fused_kernel<3, 1, false>, a);
    case 4: return cudaLaunchKernelEx(&cfg, decode_fused_kernel<4, 1, false>, a);
    default: return cudaLaunchKernelEx(&cfg, decode_fused_kernel<5, 1, false>, a);
  }
}

}  // namespace nvfp4moe
