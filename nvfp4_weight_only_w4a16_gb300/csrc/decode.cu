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
//    logits), so no routing tables cross CTAs before the GEMVs start;
//  * stream-K work split: the flat list of (touched expert, 64-row block,
//    64-wide K chunk) items is cut into equal contiguous ranges, one per warp,
//    so every SM streams the same number of weight bytes whatever the
//    routing; partial sums of a block split across warps meet in an FP32
//    buffer and the last warp to arrive (atomic counter) finishes the block;
//  * each warp runs its own 3-stage cp.async ring in shared memory (weights,
//    scales and the activation slice of a chunk), ~110 KB in flight per SM;
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
constexpr int kStages = 3;
constexpr int kStA = 0;              // 4 x 512 B weight codes
constexpr int kStS = 2048;           // 4 x 64 B scales
constexpr int kStB = 2304;           // 2 token groups x 32 lanes x 32 B (BF16 activations)
constexpr int kStageBytes = 4352;
constexpr int kPartFloats = 1024;    // [rg 4][row 16][token 16]
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
  int32_t* done_gu;
  int32_t* cmb;
  int32_t* exit_cnt;
  DeviceStatus* st;
  unsigned long long* trace;  // optional: [cta][warp][8] globaltimer stamps
};

__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async16_zfill(void* dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
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
// Phase 0: every CTA routes the T tokens into shared memory.
// ---------------------------------------------------------------------------
__device__ void route_block(const FusedArgs& a, RouteSmem& rs) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = a.T, k = a.k, E = a.E, R = T * k;
  if (tid < 16) rs.xmax[tid] = 0u;
  if (tid == 0) rs.nan = 0;
  __syncthreads();
  if (warp < T) {
    int id;
    float w;
    const int nan = warp_topk(a.logits, a.logits_bf16, E, k, warp, &id, &w);
    if (lane < k) {
      rs.ids[warp * k + lane] = id;
      rs.wts[warp * k + lane] = w;
    }
    if (lane == 0 && nan) atomicAdd(&rs.nan, nan);
  }
  if (a.x) {  // per-token max |x| for the FP16 prescale
    const int per_row = a.H / 8;
    for (int i = tid; i < T * per_row; i += blockDim.x) {
      const int t = i / per_row;
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(a.x + (size_t)t * a.H) + (i - t * per_row));
      const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
      float m = 0.f;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        m = fmaxf(m, fmaxf(fabsf(__uint_as_float(wv[q] << 16)), fabsf(__uint_as_float(wv[q] & 0xFFFF0000u))));
      atomicMax(&rs.xmax[t], __float_as_uint(m));
    }
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
#pragma unroll
  for (int rg = 0; rg < dec::kRG; ++rg)
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int j = 8 * i + 2 * q + c;
        if (j >= m) continue;
        const int row = row0 + j;
        const float s = pow2f(rs.xexp[rs.perm[row] / a.k]);
        const float g = gsg * (acc[rg][i][c] * s);
        const float uu = gsu * (acc[rg][i][2 + c] * s);
        const __nv_bfloat16 hb = __float2bfloat16_rn(silu(g) * uu);
        const int f = 8 * (dec::kRG * b + rg) + r0;
        a.h[(size_t)row * a.I + f] = hb;
        atomicMax(&a.hmax[row], __float_as_uint(fabsf(__bfloat162float(hb))));
      }
  __threadfence();
  __syncwarp();
  if (lane == 0) atomicAdd(&a.done_gu[u], 1);
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
  __threadfence();
  __syncwarp();
  int last = 0;
  if (lane == 0) last = (atomicAdd(&a.cmb[b], 1) + 1 == rs.U);
  last = __shfl_sync(0xffffffffu, last, 0);
  if (!last) return;
  __threadfence();
  // combine the 64-wide slice of H for every token, slot order j = 0..k-1
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
  if (lane == 0) a.cmb[b] = 0;
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

template <bool kGateUp>
__device__ void run_phase(const FusedArgs& a, const RouteSmem& rs, uint8_t* ring, long long fbeg, long long fend,
                          unsigned long long* tr = nullptr) {
  const int lane = threadIdx.x & 31, q = lane & 3, r0 = lane >> 2;
  const int K = kGateUp ? a.H : a.I;
  const int nch = K / kChunk;
  const int nblk = kGateUp ? (2 * a.I / 64) : (a.H / 64);
  const int nblk_gu = 2 * a.I / 64;
  const size_t nib_off = kGateUp ? a.nib13 : a.nib2;
  const size_t sc_off = kGateUp ? a.sc13 : a.sc2;
  const int nf = (int)(fend - fbeg);
  if (nf <= 0) return;

  // ---- producer state (runs kStages-1 items ahead of the consumer) ----
  ItemPos ip = item_at(fbeg, nch, nblk);
  int ip_u = -1;                         // expert whose per-segment data is cached below
  const uint8_t* ip_nib = nullptr;       // lane's code pointer at chunk 0 of the block, per rg
  const uint8_t* ip_sc = nullptr;
  const __nv_bfloat16* ip_src[2] = {nullptr, nullptr};
  int ip_b = -1;
  bool dead = false;

  auto issue = [&](int slot) {
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
            __nanosleep(100);
          }
        }
        __syncwarp();
        __threadfence();
        if (aborted(a.st)) dead = true;
        if (tr && lane == 0 && tr[3] == 0) tr[3] = now_ns();
      }
      const int e = rs.tch_e[u], row0 = rs.tch_r0[u], m = rs.tch_m[u];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int j = 8 * i + r0;
        ip_src[i] = nullptr;
        if (j < m)
          ip_src[i] = kGateUp ? a.x + (size_t)(rs.perm[row0 + j] / a.k) * a.H + 16 * q
                              : a.h + (size_t)(row0 + j) * a.I + 16 * q;
      }
      ip_nib = a.blob + (size_t)e * a.expert_stride + nib_off;
      ip_sc = a.blob + (size_t)e * a.expert_stride + sc_off;
      ip_u = u;
      ip_b = -1;
    }
    // (rb, c, sb) -> segment; the 4 row groups of block b are sub-blocks 4(b&1)..+3 of row block b>>1
    const size_t seg0 = ((size_t)(ip.b >> 1) * nch + ip.c) * 8 + 4 * (ip.b & 1);
    uint8_t* st = ring + slot * dec::kStageBytes;
#pragma unroll
    for (int rg = 0; rg < dec::kRG; ++rg)
      cp_async16(st + dec::kStA + rg * 512 + lane * 16, ip_nib + (seg0 + rg) * 512 + lane * 16);
    if (lane < 16)
      cp_async16(st + dec::kStS + (lane >> 2) * 64 + (lane & 3) * 16,
                 ip_sc + (seg0 + (lane >> 2)) * 64 + (lane & 3) * 16);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const bool valid = ip_src[i] != nullptr;
      const __nv_bfloat16* src = valid ? ip_src[i] + kChunk * ip.c : a.x;
      // [group][half][lane] x 16 B: each 16-byte access of a warp is contiguous
      uint8_t* dst = st + dec::kStB + i * 1024 + lane * 16;
      cp_async16_zfill(dst, src, valid ? 16 : 0);
      cp_async16_zfill(dst + 512, valid ? src + 8 : src, valid ? 16 : 0);
    }
    cp_async_commit();
    ip.next(nch, nblk);
  };

  // ---- consumer state ----
  ItemPos cp = item_at(fbeg, nch, nblk);
  float acc[dec::kRG][2][4];
  float bsc[2] = {1.f, 1.f};
  int seg_c0 = 0, m = 0, ng = 1;

#pragma unroll
  for (int s = 0; s < dec::kStages - 1; ++s) {
    if (s < nf) issue(s);
    else cp_async_commit();
  }
  for (int i = 0; i < nf && !dead; ++i) {
    cp_async_wait<dec::kStages - 2>();
    __syncwarp();
    if (i + dec::kStages - 1 < nf) issue((i + dec::kStages - 1) % dec::kStages);
    else cp_async_commit();
    if (dead) break;
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
    const uint8_t* st = ring + (i % dec::kStages) * dec::kStageBytes;
    // activations: BF16 -> FP16 with the row prescale
    uint32_t bw[2][8];
#pragma unroll
    for (int gi = 0; gi < 2; ++gi) {
      if (gi < ng) {
        const uint8_t* p = st + dec::kStB + gi * 1024 + lane * 16;
        const uint4 u0 = *reinterpret_cast<const uint4*>(p), u1 = *reinterpret_cast<const uint4*>(p + 512);
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
        if (ng > 1)
          mma_f16_16816(acc[rg][1], r0w[o], r8w[o], r0w[o + 1], r8w[o + 1], bw[1][2 * kt], bw[1][2 * kt + 1]);
      }
    }
    cp.next(nch, nblk);
    const bool seg_end = (c == nch - 1) || (i == nf - 1);
    if (!seg_end) continue;
    if (seg_c0 == 0 && c == nch - 1) {
      if (kGateUp) finish_gateup(a, rs, u, b, acc, lane);
      else finish_down(a, rs, u, b, acc, lane);
      continue;
    }
    // partial block: add into the FP32 buffer; the last arriver finishes it
    const int blk = u * nblk + b;
    float* part = (kGateUp ? a.part_gu : a.part_dn) + (size_t)blk * dec::kPartFloats;
    int32_t* cnt = (kGateUp ? a.cnt_gu : a.cnt_dn) + blk;
#pragma unroll
    for (int rg = 0; rg < dec::kRG; ++rg)
#pragma unroll
      for (int gi = 0; gi < 2; ++gi)
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int j = 8 * gi + 2 * q + cc;
          if (j < m) {
            atomicAdd(part + rg * 256 + r0 * 16 + j, acc[rg][gi][cc]);
            atomicAdd(part + rg * 256 + (r0 + 8) * 16 + j, acc[rg][gi][2 + cc]);
          }
        }
    __threadfence();
    __syncwarp();
    int last = 0;
    if (lane == 0) {
      const int add = c - seg_c0 + 1;
      last = (atomicAdd(cnt, add) + add == nch);
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (!last) continue;
    __threadfence();
#pragma unroll
    for (int rg = 0; rg < dec::kRG; ++rg)
#pragma unroll
      for (int gi = 0; gi < 2; ++gi)
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int j = 8 * gi + 2 * q + cc;
          if (j < m) {
            float* p0 = part + rg * 256 + r0 * 16 + j;
            float* p1 = part + rg * 256 + (r0 + 8) * 16 + j;
            acc[rg][gi][cc] = __ldcg(p0);
            acc[rg][gi][2 + cc] = __ldcg(p1);
            __stcg(p0, 0.f);
            __stcg(p1, 0.f);
          }
        }
    if (lane == 0) *cnt = 0;
    if (kGateUp) finish_gateup(a, rs, u, b, acc, lane);
    else finish_down(a, rs, u, b, acc, lane);
  }
  cp_async_wait<0>();
  __syncwarp();
}

__global__ void __launch_bounds__(dec::kThreads, 1) decode_fused_kernel(FusedArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  RouteSmem& rs = *reinterpret_cast<RouteSmem*>(smem);
  uint8_t* rings = smem + ((sizeof(RouteSmem) + 127) & ~size_t(127));
  const int warp = threadIdx.x >> 5;
  uint8_t* ring = rings + warp * dec::kStages * dec::kStageBytes;

  const uint64_t t_start = now_ns();
  route_block(a, rs);
  if (a.route_only) return;
  unsigned long long* tr = a.trace ? a.trace + ((size_t)blockIdx.x * dec::kWarps + warp) * 8 : nullptr;
  const int lane0 = (threadIdx.x & 31) == 0;
  if (tr && lane0) {
    tr[0] = t_start;
    tr[1] = now_ns();
  }

  const long long W = (long long)gridDim.x * dec::kWarps;
  const long long wg = (long long)blockIdx.x * dec::kWarps + warp;
  const int U = rs.U;
  const long long F1 = (long long)U * (2 * a.I / 64) * (a.H / kChunk);
  run_phase<true>(a, rs, ring, F1 * wg / W, F1 * (wg + 1) / W);
  if (tr && lane0) tr[2] = now_ns();
  const long long F2 = (long long)U * (a.H / 64) * (a.I / kChunk);
  run_phase<false>(a, rs, ring, F2 * wg / W, F2 * (wg + 1) / W, tr);
  if (tr && lane0) tr[4] = now_ns();

  // the last CTA out resets the per-forward counters (and, after a timeout,
  // every partial sum) for the next forward
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    rs.last_cta = atomicAdd(a.exit_cnt, 1) == (int)gridDim.x - 1;
  }
  __syncthreads();
  if (tr && lane0) tr[5] = now_ns();
  if (!rs.last_cta) return;
  __threadfence();
  const int R = a.T * a.k;
  for (int i = threadIdx.x; i < U; i += blockDim.x) a.done_gu[i] = 0;
  for (int i = threadIdx.x; i < R; i += blockDim.x) a.hmax[i] = 0u;
  if (aborted(a.st)) {
    const size_t ngu = (size_t)U * (2 * a.I / 64), ndn = (size_t)U * (a.H / 64);
    for (size_t i = threadIdx.x; i < ngu * dec::kPartFloats; i += blockDim.x) a.part_gu[i] = 0.f;
    for (size_t i = threadIdx.x; i < ndn * dec::kPartFloats; i += blockDim.x) a.part_dn[i] = 0.f;
    for (size_t i = threadIdx.x; i < ngu; i += blockDim.x) a.cnt_gu[i] = 0;
    for (size_t i = threadIdx.x; i < ndn; i += blockDim.x) a.cnt_dn[i] = 0;
    for (int i = threadIdx.x; i < a.H / 64; i += blockDim.x) a.cmb[i] = 0;
  }
  __syncthreads();
  if (threadIdx.x == 0) *a.exit_cnt = 0;
}

size_t decode_smem_bytes() {
  return ((sizeof(RouteSmem) + 127) & ~size_t(127)) + (size_t)dec::kWarps * dec::kStages * dec::kStageBytes;
}

cudaError_t launch_decode_forward(const LayerDims& d, const uint8_t* blob, const float* gscale, const void* logits,
                                  const void* x, int T, int k, void* out, int route_only, int num_sms,
                                  const Workspace& ws, cudaStream_t st) {
  static int attr_done = 0;
  const size_t smem = decode_smem_bytes();
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(decode_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
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
  return cudaLaunchKernelEx(&cfg, decode_fused_kernel, a);
}

}  // namespace nvfp4moe
