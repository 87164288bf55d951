// Decode path (1..16 tokens): one cooperative persistent kernel that routes,
// runs the grouped gate/up GEMV with SwiGLU, the grouped down GEMV and the
// weighted combine, dequantising NVFP4 in registers.
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
//    are resident); every CTA routes the <= 16 tokens itself (a few KB of
//    logits; one thread per logit ranks it against its row in shared memory
//    when T*E <= 512), so no routing tables cross CTAs before the GEMVs start;
//  * stream-K work split: the flat list of (touched expert, 64-row block,
//    64-wide K chunk) items is cut into equal contiguous ranges, one per warp,
//    so every SM streams the same number of weight bytes whatever the
//    routing; partial sums of a block split across warps meet in an FP32
//    buffer and the last warp to arrive (atomic counter) finishes the block;
//  * each warp runs its own ring in shared memory (3-4 stages): one lane
//    issues cp.async.bulk copies of a chunk's codes (2 KB), scales (256 B) and
//    the routed rows' activation slices (128 B each) onto the stage's
//    mbarrier, so no per-thread copy is in flight when a warp fences;
//  * dequantisation: hardware E2M1->FP16 converts (two weights each) times the
//    E4M3 group scale in FP16 (exact); the dot products run on mma.sync
//    m16n8k16 (FP16 in, FP32 accumulate) -- about one instruction per weight;
//  * the K axis of each 64-chunk is permuted identically for weights and
//    activations, so a lane's 16-byte load is exactly its MMA fragment;
//  * activations (x, then h) enter as FP16 after a per-row power-of-two
//    prescale (exact for BF16 values within 2^31 of the row maximum), undone
//    in FP32;
//  * the down GEMV of expert u starts once all gate/up blocks of u are done
//    (per-expert counter, bounded wait); the last down block to finish a
//    64-wide slice of H combines that slice for every token, in slot order.
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
constexpr int kSlotFloats = 15 * 64 * 8;              // shared-memory split-K slots (T <= 8)
constexpr int kSlotBytes = kSlotFloats * 4 + 128;     // + 16 counters, padded
__host__ __device__ constexpr int stage_bytes(int ng) { return kStB + 8 * kRowPitch * ng; }
// split-K partial sums: per warp, two slots (its first and its last segment),
// each [rg 4][row 16][mslot] FP32 with mslot = min(T, 16)
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
  int scan[32];
};

struct FusedArgs {
  const uint8_t* blob;
  size_t expert_stride;
  size_t nib13, sc13, nib2, sc2;
  const float* gscale;
  int E, H, I, T, k;
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
  int mslot;     // token columns of a partial-sum slot
  int no_split;  // 1: every warp takes whole blocks (no split-K, no partial-sum buffers)
  int32_t* done_gu;
  int32_t* cmb;
  int32_t* exit_cnt;
  DeviceStatus* st;
  unsigned long long* trace;  // optional: [cta][warp][8] globaltimer stamps
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
// Phase 0: every CTA routes the T tokens into shared memory, and takes each
// token's max |x| for the FP16 prescale.  `scratch` (>= T*E*8 bytes) is the
// ring memory, free until the GEMVs start.
// ---------------------------------------------------------------------------
__device__ void route_block(const FusedArgs& a, RouteSmem& rs, uint8_t* scratch) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = a.T, k = a.k, E = a.E, R = T * k, TE = T * E;
  const bool by_rank = TE <= dec::kThreads;  // one thread per logit
  uint32_t* keys = reinterpret_cast<uint32_t*>(scratch);
  float* vals = reinterpret_cast<float*>(scratch + 4 * dec::kThreads);
  if (tid < 16) rs.xmax[tid] = 0u;
  if (tid == 0) rs.nan = 0;
  __syncthreads();
  // logits -> orderable keys (rank path); per-token max |x| on every thread
  int nan = 0;
  if (by_rank && tid < TE) {
    const float v = load_logit(a.logits, a.logits_bf16, tid);
    nan = (v != v);
    keys[tid] = float_key(v);
    vals[tid] = v;
  }
  if (a.x) {  // 8 independent 16-byte loads in flight per thread
    const int per_row = a.H / 8, n = T * per_row;
    for (int base = tid; base < n; base += 8 * blockDim.x) {
      uint4 v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int i = base + j * blockDim.x;
        if (i < n) {
          const int t = i / per_row;
          v[j] = __ldg(reinterpret_cast<const uint4*>(a.x + (size_t)t * a.H) + (i - t * per_row));
        }
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int i = base + j * blockDim.x;
        if (i < n) {
          const uint32_t wv[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
          float m = 0.f;
#pragma unroll
          for (int q = 0; q < 4; ++q)
            m = fmaxf(m, fmaxf(fabsf(__uint_as_float(wv[q] << 16)), fabsf(__uint_as_float(wv[q] & 0xFFFF0000u))));
          atomicMax(&rs.xmax[i / per_row], __float_as_uint(m));
        }
      }
    }
  }
  __syncthreads();
  if (by_rank) {
    // rank of logit (t, e) in its row: larger key first, lower index on ties
    if (tid < TE) {
      const int t = tid / E, e = tid - t * E;
      const uint32_t kk = keys[tid];
      const uint32_t* row = keys + t * E;
      int r = 0;
      for (int e2 = 0; e2 < E; ++e2) {
        const uint32_t k2 = row[e2];
        r += (k2 > kk) | ((k2 == kk) & (e2 < e));
      }
      if (r < k) {
        rs.ids[t * k + r] = e;
        rs.wts[t * k + r] = vals[tid];  // the chosen logit, turned into a weight below
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) nan += __shfl_xor_sync(0xffffffffu, nan, o);
    if (lane == 0 && nan) atomicAdd(&rs.nan, nan);
    __syncthreads();
    if (warp < T) {
      const float w = warp_softmax_k(lane < k ? rs.wts[warp * k + lane] : 0.f, k);
      __syncwarp();
      if (lane < k) rs.wts[warp * k + lane] = w;
    }
  } else if (warp < T) {
    int id;
    float w;
    const int nt = warp_topk(a.logits, a.logits_bf16, E, k, warp, &id, &w);
    if (lane < k) {
      rs.ids[warp * k + lane] = id;
      rs.wts[warp * k + lane] = w;
    }
    if (lane == 0 && nt) atomicAdd(&rs.nan, nt);
  }
  __syncthreads();
  int c = 0;
  if (tid < E)
    for (int i = 0; i < R; ++i) c += (rs.ids[i] == tid);
  int total = 0, touched = 0;
  const int off = block_exclusive_scan(tid < E ? c : 0, rs.scan, &total);
  const int slot = block_exclusive_scan((tid < E && c > 0) ? 1 : 0, rs.scan, &touched);
  if (tid < E) {
    rs.off[tid] = off;
    if (c > 0) {
      rs.tch_e[slot] = tid;
      rs.tch_r0[slot] = off;
      rs.tch_m[slot] = c;
    }
  }
  if (tid == 0) {
    rs.off[E] = total;
    rs.U = touched;
  }
  if (tid < T) rs.xexp[tid] = max(-126, min(126, prescale_exp(__uint_as_float(rs.xmax[tid]))));
  __syncthreads();
  if (tid < R) {
    const int e = rs.ids[tid];
    int rank = 0;
    for (int j = 0; j < tid; ++j) rank += (rs.ids[j] == e);
    const int pos = rs.off[e] + rank;
    rs.perm[pos] = tid;
    rs.inv[tid] = pos;
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
// Block finishing
// ---------------------------------------------------------------------------
__device__ void finish_gateup(const FusedArgs& a, const RouteSmem& rs, int u, int b, float (&acc)[dec::kRG][2][4],
                              int lane) {
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
      const float s = pow2f(rs.xexp[rs.perm[row] / a.k]);
#pragma unroll
      for (int rg = 0; rg < dec::kRG; ++rg) {
        const float g = gsg * (acc[rg][i][c] * s);
        const float uu = gsu * (acc[rg][i][2 + c] * s);
        const __nv_bfloat16 hb = __float2bfloat16_rn(silu(g) * uu);
        const int f = 8 * (dec::kRG * b + rg) + r0;
        a.h[(size_t)row * a.I + f] = hb;
        hmax[i][c] = fmaxf(hmax[i][c], fabsf(__bfloat162float(hb)));
      }
    }
  // row maxima: reduce over the 8 lanes that share a token slot, then one
  // atomic per row from this block
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

__device__ void finish_down(const FusedArgs& a, const RouteSmem& rs, int u, int b, float (&acc)[dec::kRG][2][4],
                            int lane) {
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
      const float s = gsd * pow2f(prescale_exp(__uint_as_float(__ldcg(a.hmax + row))));
#pragma unroll
      for (int rg = 0; rg < dec::kRG; ++rg) {
        const int d = 16 * (dec::kRG * b + rg) + r0;
        a.y[(size_t)row * a.H + d] = acc[rg][i][c] * s;
        a.y[(size_t)row * a.H + d + 8] = acc[rg][i][2 + c] * s;
      }
    }
}

// The 64-wide slice b of H is complete for every expert: out[t][slice] =
// sum_j w[t][j] * y[pos(t,j)][slice], slot order j = 0..k-1.
__device__ void combine_slice(const FusedArgs& a, const RouteSmem& rs, int b, int lane) {
  const int d = 64 * b + 2 * lane;
  for (int t = 0; t < a.T; ++t) {
    float s0 = 0.f, s1 = 0.f;
    for (int j = 0; j < a.k; ++j) {
      const float w = rs.wts[t * a.k + j];
      const float2 yy = __ldcg(reinterpret_cast<const float2*>(a.y + (size_t)rs.inv[t * a.k + j] * a.H + d));
      s0 = fmaf(w, yy.x, s0);
      s1 = fmaf(w, yy.y, s1);
    }
    if (a.out_f32) {
      *reinterpret_cast<float2*>(reinterpret_cast<float*>(a.out) + (size_t)t * a.H + d) = make_float2(s0, s1);
    } else {
      *reinterpret_cast<__nv_bfloat162*>(reinterpret_cast<__nv_bfloat16*>(a.out) + (size_t)t * a.H + d) =
          __floats2bfloat162_rn(s0, s1);
    }
  }
}

// ---------------------------------------------------------------------------
// Phases 1 and 2: stream-K GEMV over this warp's range of chunks.
// ---------------------------------------------------------------------------
// Position in the flat (touched expert u, 64-row block b, chunk c) list.
struct ItemPos {
  int u, b, c;
  __device__ __forceinline__ void next(int nch, int nblk) {
    if (++c == nch) {
      c = 0;
      if (++b == nblk) {
        b = 0;
        ++u;
      }
    }
  }
};

__device__ __forceinline__ ItemPos item_at(long long f, int nch, int nblk) {
  const int fi = (int)f;  // < 2^31: at most 256 experts x 512 blocks x 256 chunks
  const int blk = fi / nch;
  ItemPos p;
  p.c = fi - blk * nch;
  p.u = blk / nblk;
  p.b = blk - p.u * nblk;
  return p;
}

template <bool kGateUp, int S, int NG>
__device__ void run_phase(const FusedArgs& a, RouteSmem& rs, uint8_t* ring, uint64_t* bars, uint32_t& ring_it,
                          long long F, long long W, long long wg, unsigned long long* tr, float* part_s,
                          int* cnt_s) {
  const int nch_ = kGateUp ? a.H / kChunk : a.I / kChunk;
  // split-K: equal chunk ranges; no_split: equal ranges of whole blocks
  const long long fbeg = a.no_split ? (F / nch_) * wg / W * nch_ : F * wg / W;
  const long long fend = a.no_split ? (F / nch_) * (wg + 1) / W * nch_ : F * (wg + 1) / W;
  constexpr int kStageBytes = dec::stage_bytes(NG);
  const int lane = threadIdx.x & 31, q = lane & 3, r0 = lane >> 2;
  const int K = kGateUp ? a.H : a.I;
  const int nch = K / kChunk;
  const int nblk = kGateUp ? (2 * a.I / 64) : (a.H / 64);
  const int nblk_gu = 2 * a.I / 64;
  const size_t nib_off = kGateUp ? a.nib13 : a.nib2;
  const size_t sc_off = kGateUp ? a.sc13 : a.sc2;
  const int nf = (int)(fend - fbeg);
  if (nf <= 0) return;

  // ---- producer state (runs S-1 items ahead of the consumer) ----
  ItemPos ip = item_at(fbeg, nch, nblk);
  int ip_u = -1, ip_m = 0;
  const uint8_t* ip_nib = nullptr;
  const uint8_t* ip_sc = nullptr;
  const uint8_t* ip_row = nullptr;  // lane j < m: its routed row's activations (bytes)
  bool dead = false;

  auto issue = [&](uint32_t it) {
    if (ip.u != ip_u) {
      const int u = ip.u;
      if (!kGateUp) {  // h of expert u must be complete
        if (lane == 0) {
          const uint64_t t0 = now_ns();
          while (ld_acquire(a.done_gu + u) < nblk_gu) {
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
      const int e = rs.tch_e[u], row0 = rs.tch_r0[u];
      ip_m = min(rs.tch_m[u], 8 * NG);
      ip_row = nullptr;
      if (lane < ip_m)
        ip_row = kGateUp ? reinterpret_cast<const uint8_t*>(a.x + (size_t)(rs.perm[row0 + lane] / a.k) * a.H)
                         : reinterpret_cast<const uint8_t*>(a.h + (size_t)(row0 + lane) * a.I);
      ip_nib = a.blob + (size_t)e * a.expert_stride + nib_off;
      ip_sc = a.blob + (size_t)e * a.expert_stride + sc_off;
      ip_u = u;
    }
    const int slot = (int)(it % S);
    uint8_t* st = ring + slot * kStageBytes;
    uint64_t* bar = bars + slot;
    // the 4 row groups of block b are sub-blocks 4(b&1)..+3 of 128-row block b>>1
    const size_t seg0 = ((size_t)(ip.b >> 1) * nch + ip.c) * 8 + 4 * (ip.b & 1);
    // earlier generic reads and writes of this memory come before the copies
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (lane == 0) {
      mbar_expect_tx(bar, 2048u + 256u + 128u * (uint32_t)ip_m);
      bulk_copy(st + dec::kStA, ip_nib + seg0 * 512, 2048, bar);
      bulk_copy(st + dec::kStS, ip_sc + seg0 * 64, 256, bar);
    }
    __syncwarp();
    if (lane < ip_m)
      bulk_copy(st + dec::kStB + (lane >> 3) * 8 * dec::kRowPitch + (lane & 7) * dec::kRowPitch,
                ip_row + (size_t)ip.c * 128, 128, bar);
    ip.next(nch, nblk);
  };

  // ---- consumer state ----
  ItemPos cp = item_at(fbeg, nch, nblk);
  float acc[dec::kRG][2][4];
  float bsc[2] = {1.f, 1.f};
  int seg_c0 = 0, m = 0, ng = 1;
  const uint32_t it0 = ring_it;
  // blocks whose every contributor is a warp of this CTA reduce in shared memory
  const long long cta_w0 = wg - (wg % dec::kWarps);
  const long long cs0 = F * cta_w0 / W, cs1 = F * (cta_w0 + dec::kWarps) / W;
  int seg_idx = 0;
  uint64_t loop_fin = 0;  // CTA-internal blocks this warp finished during the loop
  int issued = 0, consumed = 0;

  for (; issued < S - 1 && issued < nf; ++issued) issue(it0 + issued);
  for (int i = 0; i < nf && !dead; ++i) {
    const uint32_t it = it0 + i;
    if (issued < nf) issue(it0 + issued++);
    if (dead) break;
    if (!ring_wait(bars + it % S, (it / S) & 1u, a.st)) {
      dead = true;
      break;
    }
    consumed = i + 1;
    const int u = cp.u, b = cp.b, c = cp.c;
    if (i == 0 || c == 0) {
      seg_c0 = c;
      const int row0 = rs.tch_r0[u];
      m = rs.tch_m[u];
      ng = (m + 7) >> 3;
#pragma unroll
      for (int rg = 0; rg < dec::kRG; ++rg)
#pragma unroll
        for (int gi = 0; gi < 2; ++gi)
#pragma unroll
          for (int z = 0; z < 4; ++z) acc[rg][gi][z] = 0.f;
#pragma unroll
      for (int gi = 0; gi < 2; ++gi) {
        const int j = 8 * gi + r0;
        int p = 0;
        if (j < m) {
          const int row = row0 + j;
          p = kGateUp ? rs.xexp[rs.perm[row] / a.k]
                      : max(-126, min(126, prescale_exp(__uint_as_float(__ldcg(a.hmax + row)))));
        }
        bsc[gi] = pow2f(-p);
      }
    }
    const uint8_t* st = ring + (int)(it % S) * kStageBytes;
    // activations: BF16 -> FP16 with the row prescale (rows >= m hold stale
    // data; their MMA columns are never read)
    uint32_t bw[2][8];
#pragma unroll
    for (int gi = 0; gi < NG; ++gi) {
      if (gi < ng) {
        const uint8_t* p = st + dec::kStB + gi * 8 * dec::kRowPitch + r0 * dec::kRowPitch + q * 32;
        const uint4 u0 = *reinterpret_cast<const uint4*>(p), u1 = *reinterpret_cast<const uint4*>(p + 16);
        const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
        for (int z = 0; z < 8; ++z) {
          const __half2 hh = __floats2half2_rn(__uint_as_float(w[z] << 16) * bsc[gi],
                                               __uint_as_float(w[z] & 0xFFFF0000u) * bsc[gi]);
          bw[gi][z] = *reinterpret_cast<const uint32_t*>(&hh);
        }
      }
    }
#pragma unroll
    for (int rg = 0; rg < dec::kRG; ++rg) {
      const uint4 raw = *reinterpret_cast<const uint4*>(st + dec::kStA + rg * 512 + lane * 16);
      const uint32_t s2 = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(st + dec::kStS + rg * 64 + lane * 2));
      const uint32_t s0 = dup_lo(s2), s1 = dup_hi(s2);
      uint32_t cx[4], cy[4], cz[4], cw[4];
      e2m1x8_to_f16(raw.x, cx);
      e2m1x8_to_f16(raw.y, cy);
      e2m1x8_to_f16(raw.z, cz);
      e2m1x8_to_f16(raw.w, cw);
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        cx[t] = hmul2_u32(cx[t], s0);
        cy[t] = hmul2_u32(cy[t], s0);
        cz[t] = hmul2_u32(cz[t], s1);
        cw[t] = hmul2_u32(cw[t], s1);
      }
#pragma unroll
      for (int kt = 0; kt < 4; ++kt) {
        const uint32_t* r0w = kt < 2 ? cx : cy;
        const uint32_t* r8w = kt < 2 ? cz : cw;
        const int o = 2 * (kt & 1);
        mma_f16_16816(acc[rg][0], r0w[o], r8w[o], r0w[o + 1], r8w[o + 1], bw[0][2 * kt], bw[0][2 * kt + 1]);
        if (NG > 1 && ng > 1)
          mma_f16_16816(acc[rg][1], r0w[o], r8w[o], r0w[o + 1], r8w[o + 1], bw[1][2 * kt], bw[1][2 * kt + 1]);
      }
    }
    __syncwarp();  // every lane is done reading this stage before it is refilled
    cp.next(nch, nblk);
    const bool seg_end = (c == nch - 1) || (i == nf - 1);
    if (!seg_end) continue;
    if (seg_c0 == 0 && c == nch - 1) {  // the whole block is this warp's: finish it now, signal later
      ++seg_idx;
      if (kGateUp) finish_gateup(a, rs, u, b, acc, lane);
      else finish_down(a, rs, u, b, acc, lane);
      continue;
    }
    const int seg_here = seg_idx++;
    const long long f0 = (long long)(u * nblk + b) * nch;
    if (part_s != nullptr && f0 >= cs0 && f0 + nch <= cs1) {
      // split among warps of this CTA: shared-memory sum, the last one finishes
      const long long wlo = ((f0 + 1) * W + F - 1) / F - 1;  // warp holding the block's first chunk
      const int slot = (int)(wlo - cta_w0);                    // its boundary with the next warp
      float* ps = part_s + slot * 64 * 8;
#pragma unroll
      for (int rg = 0; rg < dec::kRG; ++rg)
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int j = 2 * q + cc;
          if (j < m) {
            atomicAdd(ps + (rg * 16 + r0) * 8 + j, acc[rg][0][cc]);
            atomicAdd(ps + (rg * 16 + r0 + 8) * 8 + j, acc[rg][0][2 + cc]);
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
            for (int cc = 0; cc < 2; ++cc) {
              const int j = 2 * q + cc;
              acc[rg][gi][cc] = (gi == 0 && j < m) ? ps[(rg * 16 + r0) * 8 + j] : 0.f;
              acc[rg][gi][2 + cc] = (gi == 0 && j < m) ? ps[(rg * 16 + r0 + 8) * 8 + j] : 0.f;
            }
        if (kGateUp) finish_gateup(a, rs, u, b, acc, lane);
        else finish_down(a, rs, u, b, acc, lane);
        if (seg_here < 64) loop_fin |= 1ull << seg_here;
      }
      continue;
    }
    // split across CTAs: store the partial sums into this warp's global slot
    // (0: its first segment, 1: its last); counted at the end of the phase
    {
      const int slot = (i + 1 - (c - seg_c0 + 1) == 0) ? 0 : 1;  // did the segment start at the range start?
      float* part = (kGateUp ? a.part_gu : a.part_dn) + ((size_t)wg * 2 + slot) * 64 * a.mslot;
#pragma unroll
      for (int rg = 0; rg < dec::kRG; ++rg)
#pragma unroll
        for (int gi = 0; gi < 2; ++gi)
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const int j = 8 * gi + 2 * q + cc;
            if (j < m) {
              __stcg(part + (rg * 16 + r0) * a.mslot + j, acc[rg][gi][cc]);
              __stcg(part + (rg * 16 + r0 + 8) * a.mslot + j, acc[rg][gi][2 + cc]);
            }
          }
    }
  }

  // ---- end of phase: one fence covers every store and partial sum above ----
  if (!dead) {
    const uint64_t t_fin = tr ? now_ns() : 0;
    __threadfence();
    __syncwarp();
    // walk this warp's segments: count partial ones in; the last contributor
    // of a block finishes it
    uint64_t fin_mask = 0;
    int si = 0;
    // signals a finished block; used at once for segments past the 64-bit mask
    auto signal = [&](int blk) {
      const int u = blk / nblk, b = blk - (blk / nblk) * nblk;
      if (kGateUp) {
        if (lane == 0) atomicAdd(&a.done_gu[u], 1);
      } else {
        int lastc = 0;
        if (lane == 0) lastc = (atomicAdd(&a.cmb[b], 1) + 1 == rs.U);
        lastc = __shfl_sync(0xffffffffu, lastc, 0);
        if (lastc) {
          __threadfence();
          combine_slice(a, rs, b, lane);
          if (lane == 0) a.cmb[b] = 0;
        }
      }
    };
    for (long long f = fbeg; f < fend; ++si) {
      const int blk = (int)(f / nch), c0 = (int)(f % nch);
      const int c1 = (int)min((long long)nch, c0 + (fend - f));
      f += c1 - c0;
      if (c0 == 0 && c1 == nch) {
        if (si < 64) fin_mask |= 1ull << si;
        else signal(blk);
        continue;
      }
      if (part_s != nullptr && (long long)blk * nch >= cs0 && (long long)blk * nch + nch <= cs1) {
        if (si < 64 && ((loop_fin >> si) & 1ull)) fin_mask |= 1ull << si;
        continue;  // reduced in shared memory; finished (or not) by the loop
      }
      int last = 0;
      if (lane == 0) last = (atomicAdd((kGateUp ? a.cnt_gu : a.cnt_dn) + blk, c1 - c0) + (c1 - c0) == nch);
      last = __shfl_sync(0xffffffffu, last, 0);
      if (!last) continue;
      __threadfence();
      const int u = blk / nblk, b = blk - (blk / nblk) * nblk;
      const int mm = rs.tch_m[u];
#pragma unroll
      for (int rg = 0; rg < dec::kRG; ++rg)
#pragma unroll
        for (int gi = 0; gi < 2; ++gi)
#pragma unroll
          for (int z = 0; z < 4; ++z) acc[rg][gi][z] = 0.f;
      // contributors: the warps whose ranges meet [f0, f0 + nch)
      const long long f0 = (long long)blk * nch;
      const long long w_lo = ((f0 + 1) * W + F - 1) / F - 1, w_hi = ((f0 + nch) * W + F - 1) / F - 1;
      for (long long w = w_lo; w <= w_hi; ++w) {
        const long long s0 = F * w / W, s1 = F * (w + 1) / W;
        if (s0 >= s1 || s1 <= f0 || s0 >= f0 + nch) continue;
        const int slot = s0 >= f0 ? 0 : 1;
        const float* part = (kGateUp ? a.part_gu : a.part_dn) + ((size_t)w * 2 + slot) * 64 * a.mslot;
#pragma unroll
        for (int rg = 0; rg < dec::kRG; ++rg)
#pragma unroll
          for (int gi = 0; gi < 2; ++gi)
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
              const int j = 8 * gi + 2 * q + cc;
              if (j < mm) {
                acc[rg][gi][cc] += __ldcg(part + (rg * 16 + r0) * a.mslot + j);
                acc[rg][gi][2 + cc] += __ldcg(part + (rg * 16 + r0 + 8) * a.mslot + j);
              }
            }
      }
      if (lane == 0) (kGateUp ? a.cnt_gu : a.cnt_dn)[blk] = 0;
      if (kGateUp) finish_gateup(a, rs, u, b, acc, lane);
      else finish_down(a, rs, u, b, acc, lane);
      if (si < 64) {
        fin_mask |= 1ull << si;
      } else {
        __threadfence();
        __syncwarp();
        signal(blk);
      }
    }
    // signal the blocks this warp finished (after one more fence)
    if (fin_mask) {
      __threadfence();
      __syncwarp();
      si = 0;
      for (long long f = fbeg; f < fend && si < 64; ++si) {
        const int blk = (int)(f / nch), c0 = (int)(f % nch);
        const int c1 = (int)min((long long)nch, c0 + (fend - f));
        f += c1 - c0;
        if ((fin_mask >> si) & 1ull) signal(blk);
      }
    }
    if (tr && lane == 0) tr[kGateUp ? 6 : 7] += now_ns() - t_fin;
  }
  // on a normal exit every issued stage was consumed; after an abort, give the
  // copies still in flight a bounded chance to land before the ring is reused
  if (dead) {
    for (int i = consumed; i < issued; ++i) {
      const uint32_t it = it0 + i;
      const uint64_t t0 = now_ns();
      while (!mbar_try_wait(bars + it % S, (it / S) & 1u) && now_ns() - t0 < dec::kTimeoutNs) {
      }
    }
  }
  ring_it = it0 + (uint32_t)issued;
}

template <int S, int NG>
__global__ void __launch_bounds__(dec::kThreads, 1) decode_fused_kernel(FusedArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  RouteSmem& rs = *reinterpret_cast<RouteSmem*>(smem);
  const size_t route_bytes = (sizeof(RouteSmem) + 127) & ~size_t(127);
  uint64_t* all_bars = reinterpret_cast<uint64_t*>(smem + route_bytes);
  // NG == 1: shared-memory split-K slots, one per boundary between the CTA's warps
  float* part_s = NG == 1 ? reinterpret_cast<float*>(smem + route_bytes + 128 * 8) : nullptr;
  int* cnt_s = NG == 1 ? reinterpret_cast<int*>(smem + route_bytes + 128 * 8 + dec::kSlotFloats * 4) : nullptr;
  uint8_t* rings = smem + route_bytes + 128 * 8 + (NG == 1 ? dec::kSlotBytes : 0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* ring = rings + warp * S * dec::stage_bytes(NG);
  uint64_t* bars = all_bars + warp * 8;

  const uint64_t t_start = now_ns();
  route_block(a, rs, rings);
  if (a.route_only) return;
  auto clear_slots = [&]() {
    if (NG == 1) {
      for (int i = threadIdx.x; i < dec::kSlotFloats; i += blockDim.x) part_s[i] = 0.f;
      if (threadIdx.x < 16) cnt_s[threadIdx.x] = 0;
    }
  };
  clear_slots();
  __syncthreads();
  unsigned long long* tr = a.trace ? a.trace + ((size_t)blockIdx.x * dec::kWarps + warp) * 8 : nullptr;
  if (tr && lane == 0) {
    tr[0] = t_start;
    tr[1] = now_ns();
  }
  if (lane == 0) {
    for (int s = 0; s < S; ++s) mbar_init(bars + s, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();

  const long long W = (long long)gridDim.x * dec::kWarps;
  const long long wg = (long long)blockIdx.x * dec::kWarps + warp;
  const int U = rs.U;
  uint32_t ring_it = 0;
  const long long F1 = (long long)U * (2 * a.I / 64) * (a.H / kChunk);
  run_phase<true, S, NG>(a, rs, ring, bars, ring_it, F1, W, wg, tr, part_s, cnt_s);
  if (tr && lane == 0) tr[2] = now_ns();
  if (NG == 1) {  // phase 2 reuses the shared-memory slots
    __syncthreads();
    clear_slots();
    __syncthreads();
  }
  const long long F2 = (long long)U * (a.H / 64) * (a.I / kChunk);
  run_phase<false, S, NG>(a, rs, ring, bars, ring_it, F2, W, wg, tr, part_s, cnt_s);
  if (tr && lane == 0) tr[4] = now_ns();

  // the last CTA out resets the per-forward counters (and, after a timeout,
  // every partial sum) for the next forward
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    rs.last_cta = atomicAdd(a.exit_cnt, 1) == (int)gridDim.x - 1;
  }
  __syncthreads();
  if (tr && lane == 0) tr[5] = now_ns();
  if (!rs.last_cta) return;
  __threadfence();
  const int R = a.T * a.k;
  for (int i = threadIdx.x; i < U; i += blockDim.x) a.done_gu[i] = 0;
  for (int i = threadIdx.x; i < R; i += blockDim.x) a.hmax[i] = 0u;
  if (aborted(a.st)) {
    const size_t ngu = (size_t)U * (2 * a.I / 64), ndn = (size_t)U * (a.H / 64);
    for (size_t i = threadIdx.x; i < ngu; i += blockDim.x) a.cnt_gu[i] = 0;
    for (size_t i = threadIdx.x; i < ndn; i += blockDim.x) a.cnt_dn[i] = 0;
    for (int i = threadIdx.x; i < a.H / 64; i += blockDim.x) a.cmb[i] = 0;
  }
  __syncthreads();
  if (threadIdx.x == 0) *a.exit_cnt = 0;
}

// T <= 8: one token group per expert, shared-memory split-K slots, 3 stages;
// T <= 16: two groups, 3 stages, split-K through global slots only.
static size_t smem_for(int S, int NG) {
  return ((sizeof(RouteSmem) + 127) & ~size_t(127)) + 128 * 8 + (NG == 1 ? dec::kSlotBytes : 0) +
         (size_t)dec::kWarps * S * dec::stage_bytes(NG);
}
size_t decode_smem_bytes() { return smem_for(3, 2); }

cudaError_t launch_decode_forward(const LayerDims& d, const uint8_t* blob, const float* gscale, const void* logits,
                                  const void* x, int T, int k, void* out, int route_only, int num_sms,
                                  const Workspace& ws, cudaStream_t st) {
  static int attr_done = 0;
  const bool small = T <= 8;
  const size_t smem = small ? smem_for(3, 1) : smem_for(3, 2);
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(decode_fused_kernel<3, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem_for(3, 1));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(decode_fused_kernel<3, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem_for(3, 2));
    if (e != cudaSuccess) return e;
    attr_done = 1;
  }
  const ExpertLayout L = expert_layout(d.H, d.I);
  FusedArgs a{};
  a.blob = blob;
  a.expert_stride = L.stride;
  a.nib13 = L.w13_nib;
  a.sc13 = L.w13_sc;
  a.nib2 = L.w2_nib;
  a.sc2 = L.w2_sc;
  a.gscale = gscale;
  a.E = d.E;
  a.H = d.H;
  a.I = d.I;
  a.T = T;
  a.k = k;
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
  a.done_gu = ws.done_gu;
  a.cmb = ws.cmb;
  a.exit_cnt = ws.exit_cnt;
  a.st = ws.status;
  a.trace = ws.trace;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(route_only ? 1 : num_sms);
  cfg.blockDim = dim3(dec::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = route_only ? 0 : 1;
  return small ? cudaLaunchKernelEx(&cfg, decode_fused_kernel<3, 1>, a)
               : cudaLaunchKernelEx(&cfg, decode_fused_kernel<3, 2>, a);
}

}  // namespace nvfp4moe
