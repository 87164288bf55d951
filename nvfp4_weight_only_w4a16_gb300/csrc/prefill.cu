// Prefill path: grouped GEMM over the routed rows of every expert on the
// 5th-generation tensor cores (tcgen05.mma, BF16 x BF16 -> FP32 in TMEM).
//
// The weight-only NVFP4 experts are dequantised to BF16 -- never through an
// activation scale ("GLM-5.3-Flash on Blackwell", The model loaded, served an
// API, and produced garbage: the working backend dequantises to bf16 and
// consumes no activation scale).
//
// The MoE's GEMMs run on FP16 operands (kF16): the dequantised weights
// (e2m1 * e4m3, exact in FP16), the gathered x rows and h, each row scaled by a
// power of two that the epilogues undo in FP32 (x: its largest magnitude in
// [2^13, 2^14); h: a Cauchy-Schwarz bound on its row, see route.cu), so h
// keeps 11 significant bits between the GEMMs.  The dense linear and the
// router GEMM stay on BF16 operands (the caller's BF16 x, the BF16 router).
//
// One persistent CTA per SM, 20 warps, warp-specialised:
//   warp 0      weight producer: cp.async.bulk of the packed FP4 chunks (codes +
//               scales) of a unit's two 128-row weight blocks into a 9-stage
//               ring, completion on mbarriers;
//   warps 1, 19 MMA issuers, one thread each, one per weight block: per stage of
//               two 64-wide K chunks 2 x 4 tcgen05.mma (K=16) with the weights
//               (A) from TMEM and the activation tile (B) from shared memory;
//               warp 1 also owns the TMEM allocation;
//   warp 2      activation producer: TMA (128B swizzle) boxes of 16 routed rows;
//   warps 3-10  dequantisers, one per (weight block, TMEM lane quarter), one
//               thread per weight row: E2M1 x E4M3 -> FP16 (BF16 for the W4A4
//               variant), exact, straight into the TMEM operand stage
//               (tcgen05.st);
//   warps 11-18 epilogue: tcgen05.ld of the accumulators, tensor scales,
//               SwiGLU (gate/up) or the down-projection store.
// (BF16 weights -- the router -- take a shared-memory operand ring filled by
// warp 0's TMA instead, one issuer, two accumulator buffers, no dequantisers.)
// Work unit = (m-tile of <= 128 routed rows of one expert, two 128-row weight
// blocks).  MMA orientation: weights are the 128-row M operand, routed tokens
// the N operand (16..128).  Two weight blocks per activation tile halve the
// activation bytes each MMA FLOP costs (shared memory and L2), and a
// tcgen05.commit -- which waits for the tensor pipe to drain the MMAs it
// covers -- is paid once per 8 MMAs instead of per 4.  The gate/up weight rows
// are interleaved in groups of 8 (gate f..f+7, up f..f+7), so each gate
// accumulator row and its up partner sit 8 TMEM lanes apart, inside one warp.
// Every mbarrier wait is bounded; on expiry the kernel records a timeout in
// the handle's status word and winds down instead of hanging.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace nvfp4moe {

namespace pf {
// Shared-memory rings (each stage is one 64-wide K chunk of one work unit):
//   A   : BF16 operand written by the dequantisers, read by tcgen05.mma
//   B   : routed activation rows (TMA, 128B swizzle), up to 128 rows
//   RAW : packed FP4 codes + scales of 128 weight rows (bulk copy) -- deep,
//         so the HBM latency of the weight stream is covered
#ifndef NVFP4_MOE_PF_STAGES_B
#define NVFP4_MOE_PF_STAGES_B 4
#endif
#ifndef NVFP4_MOE_PF_STAGES_RAW
#define NVFP4_MOE_PF_STAGES_RAW 9
#endif
// Packed weights: the dequantised operand lives in TMEM (tcgen05.mma with A
// from tensor memory), kAStagesT stages of two 64-wide K chunks x two blocks
// (32 columns per chunk and block: 64 16-bit values per row) in columns
// 256..511; the accumulator (two blocks x 128 columns) takes columns 0..255,
// one buffer.  The MMA issuer syncs once per stage (16 MMAs): every wait,
// fence and commit stalls its queue for a few hundred cycles.
// Shared memory: [B ring, kBStages x 2 chunks x 16 KB][RAW ring, one chunk
// per stage][row exponents][barriers].
// BF16 weights (the router) keep a shared-memory operand ring and two
// accumulator buffers: B takes 4 stages, operand stages 0, 1 the rest of the
// B region, 2, 3 the RAW region.
constexpr int kBStages = NVFP4_MOE_PF_STAGES_B;
constexpr int kBStagesW = 4;
constexpr int kRawStages = NVFP4_MOE_PF_STAGES_RAW;
constexpr int kBlocks = 2;                // 128-row weight blocks per work unit
constexpr int kABlockBytes = 16384;       // BF16 mode: one block's chunk, 128 rows x 128 B
constexpr int kAStageBytes = kBlocks * kABlockBytes;
constexpr int kBStageBytes = 16384;       // one chunk of up to 128 routed rows x 128 B
constexpr int kKS = 2;                    // packed weights: chunks per operand and activation stage
constexpr int kRawBlockBytes = 4608;      // one block's chunk: 4096 B codes + 512 B scales
constexpr int kRawStageBytes = kBlocks * kRawBlockBytes;
constexpr int kBOff = 0;
constexpr int kRawOff = kBOff + kBStages * kKS * kBStageBytes;
constexpr int kPexOff = kRawOff + kRawStages * kRawStageBytes;  // per epilogue warp [2][128] int: row exponents
constexpr int kBarOff = kPexOff + 8 * 1024;
constexpr int kSmemBytes = kBarOff + 512 + 1024;  // + barriers + alignment slack
constexpr int kAStagesW = 2 + (kRawStages * kRawStageBytes) / kAStageBytes;
static_assert(kBStagesW * kBStageBytes + 2 * kAStageBytes <= kRawOff, "BF16 mode: B and two operand stages fit the B region");
static_assert(kAStagesW <= kRawStages, "BF16-mode operand barriers reuse the packed ring's");
static_assert(kRawOff % 1024 == 0 && kAStageBytes % 1024 == 0, "128B-swizzled stages need 1024-byte alignment");
static_assert(kSmemBytes <= 232448, "shared memory");
__host__ __device__ constexpr int a_stage_off(int s) {
  return s < 2 ? kBStagesW * kBStageBytes + s * kAStageBytes : kRawOff + (s - 2) * kAStageBytes;
}
constexpr int kDequantWarps = 8;
constexpr int kEpiWarps = 8;                      // two per TMEM lane quarter: one per weight block
constexpr int kMma2Warp = 3 + kDequantWarps + kEpiWarps;       // packed weights: block 1's MMA issuer
constexpr int kThreads = (kMma2Warp + 1) * 32;                   // 20 warps
constexpr int kTmemCols = 512;
constexpr int kAStagesT = 2;
constexpr int kAColT = 256;
constexpr int kABars = kAStagesT;
static_assert(kBStages % kAStagesT == 0 && kBStages >= 2 * kAStagesT,
              "packed mode: a TMEM slot's previous stage is tracked on the B ring's barriers");
constexpr uint64_t kTimeoutNs = 2000000000ull;  // a wait longer than 2 s is a fault
}  // namespace pf

size_t prefill_smem_bytes() { return pf::kSmemBytes; }

struct PrefillArgs {
  const uint8_t* blob;
  size_t expert_stride;
  size_t mat_off;  // the matrix's byte offset in an expert's blob
  const float* gscale;
  int K;      // reduction length (H for gate/up, I for down)
  int NB;     // 128-row weight blocks per expert
  int H, I;
  const int32_t* tile_expert;
  const int32_t* tile_row0;
  const int32_t* tile_rows;
  const int32_t* num_tiles;
  __nv_bfloat16* h;
  float* y;
  void* out;     // a dense linear writes its rows here directly (row = token)
  int out_f32;   // out is FP32 (else BF16)
  int linear;    // 1: a dense linear (one matrix, rows in token order, weight 1)
  int n_out;     // a dense linear's output features: out is [T][n_out], rows d >= n_out are padding
  const float* in_scale;  // W4A4 routed experts (e < Er): [E][2] input scales, else nullptr
  int Er;
  DeviceStatus* st;
  int fault;  // 1: the producer issues nothing (tests the bounded waits)
  const int32_t* pexp_x;  // [R] FP16 operand rows: x row p was scaled by 2^-pexp_x[p] (kF16)
  const int32_t* pexp_h;  // [R] and h row p by 2^-pexp_h[p]
  int checks;             // 1: check the m-tile table against its ranges (kFlagBounds; the unit is skipped)
  int E, R;               // experts in the blob, routed rows (for the checks)
  // optional role timeline of CTA 0 (gate/up GEMM): per stage n < 256 at [4n] the MMA
  // issue, [4n+1] / [4n+2] dequantiser warp 3's start / end; per K chunk n < 256 at
  // [4n+3] the weight copy issue; per unit u < 16 at [1024 + 4u] the MMA's accumulator wait end, the epilogue's
  // start and end (block 0), the epilogue's end (block 1)
  unsigned long long* trace;
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.shared::cta.b64 st, [%0];\n}" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Bounded wait: false on timeout (recorded in the status word) or when
// another role has already aborted.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          DeviceStatus* st, unsigned where) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 63u) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > pf::kTimeoutNs) {
        *abort_flag = 1;
        report(st, kFlagTimeout, where);
        return false;
      }
    }
  }
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void tma_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// K-major operand, 128B swizzle, 8-row atoms 1024 B apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// kind::f16 instruction descriptor: D = F32, A = B = BF16 (or both F16), both K-major.
__device__ __forceinline__ uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ uint32_t idesc_f16(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(
          d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
// A from tensor memory (a_tmem: lane 0, the K step's first column), B from shared memory
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(
          d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld16_nw(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// One weight row's bytes of one packed chunk (a 4608-byte tile: codes, then
// scales): its four 16-element groups' codes and E4M3 scales.  Row r sits in
// 16-row group r / 16 as the low (r % 16 < 8) or high half of segments
// t = 4 (r % 8) + q, stored at slots seg_pos(t).
struct RowRaw {
  uint2 c[4];
  uint32_t s[4];
};
__device__ __forceinline__ void load_row_raw(const uint8_t* tile, int r, RowRaw& w) {
  const int g16 = r >> 4, hf = (r >> 3) & 1, rr = r & 7;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int p = seg_pos(4 * rr + q);
    w.c[q] = *reinterpret_cast<const uint2*>(tile + g16 * 512 + p * 16 + 8 * hf);
    w.s[q] = tile[4096 + g16 * 64 + p * 2 + hf];
  }
}
// Dequantise the row into 32 TMEM columns of the thread's lane: column c holds
// K elements 2c (low half) and 2c + 1 (high half) of the chunk, FP16 when
// kF16, else BF16 (both exact).  All 32 lanes of the warp call it; the caller
// waits for the store (tcgen05.wait::st).
template <bool kF16>
__device__ __forceinline__ void store_row_tmem(const RowRaw& raw, uint32_t taddr) {
  uint32_t w[32];
#pragma unroll
  for (int q = 0; q < 4; ++q) {  // K elements 16 q .. 16 q + 15
    const uint32_t sx = dup_lo(e4m3x2_to_f16x2(raw.s[q]));
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      const uint32_t v = hmul2_u32(e2m1x2_to_f16x2((b < 4 ? raw.c[q].x : raw.c[q].y) >> (8 * (b & 3))), sx);
      w[8 * q + b] = kF16 ? v : f16x2_to_bf16x2(v);
    }
  }
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7]), "r"(w[8]), "r"(w[9]),
      "r"(w[10]), "r"(w[11]), "r"(w[12]), "r"(w[13]), "r"(w[14]), "r"(w[15]), "r"(w[16]), "r"(w[17]), "r"(w[18]),
      "r"(w[19]), "r"(w[20]), "r"(w[21]), "r"(w[22]), "r"(w[23]), "r"(w[24]), "r"(w[25]), "r"(w[26]), "r"(w[27]),
      "r"(w[28]), "r"(w[29]), "r"(w[30]), "r"(w[31])
      : "memory");
}

// kBf16W: the weights are a plain BF16 matrix (the router): warp 0 moves its
// 128-row x 64-column tiles straight into the operand ring by TMA (128B
// swizzle, the layout the dequantisers write), and the dequantisers idle.
template <bool kGateUp, bool kBf16W = false, bool kF16 = false>
__global__ void __launch_bounds__(pf::kThreads, 1)
    prefill_gemm_kernel(const __grid_constant__ CUtensorMap tmap_b, const __grid_constant__ CUtensorMap tmap_w,
                        PrefillArgs a) {
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  uint64_t* raw_full = reinterpret_cast<uint64_t*>(smem + pf::kBarOff);
  uint64_t* raw_empty = raw_full + pf::kRawStages;
  uint64_t* a_full = raw_empty + pf::kRawStages;
  uint64_t* a_empty = a_full + pf::kABars;
  uint64_t* b_full = a_empty + pf::kABars;
  // the operand ring's barriers and depth (BF16 mode: the packed ring's barriers)
  uint64_t* af = kBf16W ? raw_full : a_full;
  uint64_t* ae = kBf16W ? raw_empty : a_empty;
  constexpr int nAS = kBf16W ? pf::kAStagesW : pf::kAStagesT;
  constexpr int nBS = kBf16W ? pf::kBStagesW : pf::kBStages;
  constexpr int kCS = kBf16W ? 1 : pf::kKS;  // K chunks per operand / activation stage
  static_assert(pf::kBStagesW <= pf::kBStages, "B barriers");
  // accumulator buffers: two with a shared-memory operand, one with the TMEM operand
  constexpr uint32_t nBuf = kBf16W ? 2u : 1u;
  uint64_t* b_empty = b_full + pf::kBStages;
  uint64_t* accfull = b_empty + pf::kBStages;
  uint64_t* accempty = accfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);


  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // epilogue warp w's copy of the unit's x and h row exponents (kF16)
  int* pex = reinterpret_cast<int*>(smem + pf::kPexOff) + 256 * max(0, warp - 3 - pf::kDequantWarps);
  int* peh = pex + 128;
  unsigned long long* tl = (kGateUp && a.trace && blockIdx.x == 0) ? a.trace : nullptr;
  if (threadIdx.x == 0) {
    for (int s = 0; s < pf::kRawStages; ++s) {
      mbar_init(raw_full + s, 1);
      mbar_init(raw_empty + s, kBf16W ? 1 : pf::kDequantWarps);
    }
    for (int s = 0; s < pf::kABars; ++s) {
      mbar_init(a_full + s, kBf16W ? 1 : pf::kDequantWarps);
      mbar_init(a_empty + s, 1);
    }
    for (int s = 0; s < nBS; ++s) {
      // packed weights: stage s is ready when its activation tiles have landed and all
      // eight dequantisers have filled its TMEM operand slot (one wait for the MMA
      // issuer); b_empty then also frees the TMEM slot (one commit per stage)
      mbar_init(b_full + s, kBf16W ? 1 : 1 + pf::kDequantWarps);
      mbar_init(b_empty + s, kBf16W ? 1 : 2);  // packed: one commit per MMA issuer
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accfull + b, kBf16W ? 1 : 2);
      mbar_init(accempty + b, pf::kEpiWarps);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(pf::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // work unit = (tile, pair of 128-row weight blocks 2p and 2p+1; the second
  // may not exist when the block count is odd)
  const int num_tiles = *a.num_tiles;
  const int NP = (a.NB + 1) / 2;
  const int total_units = num_tiles * NP;
  const int nch = a.K / kChunk;

  if (warp == 0 && kBf16W) {
    if (lane == 0) {
      // ---------------- weight producer (BF16 weights): TMA tiles into the operand ring ----------------
      uint32_t ia = 0;
      for (int unit = blockIdx.x; unit < total_units && !*abort_flag && a.fault != 1; unit += gridDim.x) {
        const int nb0 = 2 * (unit % NP);
        const int nblk = nb0 + 1 < a.NB ? 2 : 1;
        bool ok = true;
        for (int c = 0; c < nch; ++c, ++ia) {
          const int sa = ia % nAS;
          if (!mbar_wait(ae + sa, ((ia / nAS) & 1u) ^ 1u, abort_flag, a.st, 9)) {
            ok = false;
            break;
          }
          uint8_t* st = smem + pf::a_stage_off(sa);
          mbar_arrive_expect_tx(af + sa, (uint32_t)nblk * (uint32_t)pf::kABlockBytes);
          for (int j = 0; j < nblk; ++j)  // rows past the matrix read as zeros
            tma_2d(st + j * pf::kABlockBytes, &tmap_w, c * kChunk, (nb0 + j) * 128, af + sa);
        }
        if (!ok) break;
      }
    }
  } else if (warp == 0) {
    if (lane == 0) {
      // ---------------- weight producer: packed codes + scales of both blocks ----------------
      uint32_t it = 0;
      for (int unit = blockIdx.x; unit < total_units && !*abort_flag && a.fault != 1; unit += gridDim.x) {
        const int tile = unit / NP, nb0 = 2 * (unit % NP);
        const int nblk = nb0 + 1 < a.NB ? 2 : 1;
        const int e = a.tile_expert[tile];
        if (a.checks && (e < 0 || e >= a.E || a.tile_row0[tile] < 0 || a.tile_rows[tile] < 1 ||
                         a.tile_rows[tile] > kTileRows || a.tile_row0[tile] + a.tile_rows[tile] > a.R)) {
          report(a.st, kFlagBounds, 810);
          *abort_flag = 1;
          break;
        }
        const uint8_t* src = a.blob + (size_t)e * a.expert_stride + a.mat_off + (size_t)nb0 * nch * kTileBytes;
        for (int c = 0; c < nch; ++c, ++it) {
          const int s = it % pf::kRawStages;
          const uint32_t ph = (it / pf::kRawStages) & 1u;
          if (!mbar_wait(raw_empty + s, ph ^ 1u, abort_flag, a.st, 1)) break;
          if (tl && it < 256) tl[4 * it + 3] = globaltimer_ns();
          uint8_t* st = smem + pf::kRawOff + s * pf::kRawStageBytes;
          mbar_arrive_expect_tx(raw_full + s, (uint32_t)nblk * (4096u + 512u));
          for (int j = 0; j < nblk; ++j)  // block nb0 + j's chunk c: one tile, 4096 B codes + 512 B scales
            bulk_g2s(st + j * pf::kRawBlockBytes, src + ((size_t)j * nch + c) * kTileBytes, kTileBytes, raw_full + s);
        }
      }
    }
  } else if (warp == 1 || (!kBf16W && warp == pf::kMma2Warp)) {
    if (lane == 0) {
      // ---------------- MMA issuers ----------------
      // BF16 weights: warp 1 issues both blocks.  Packed weights: warp 1 issues block 0's
      // MMAs and warp kMma2Warp block 1's, into their own accumulators -- while one
      // issuer stalls on a wait or a commit, the other's MMAs keep the tensor pipe busy
      const int mb = warp == 1 ? 0 : 1;
      uint32_t ia = 0, ib = 0, j = 0;
      for (int unit = blockIdx.x; unit < total_units && !*abort_flag; unit += gridDim.x, ++j) {
        const int tile = unit / NP, nb0 = 2 * (unit % NP);
        const int nblk = nb0 + 1 < a.NB ? 2 : 1;
        const int rows = a.tile_rows[tile];
        const int N = (rows + 15) & ~15;
        const uint32_t idesc = kF16 ? idesc_f16(128, N) : idesc_bf16(128, N);
        const uint32_t buf = j % nBuf, aph = (j / nBuf) & 1u;
        if (!mbar_wait(accempty + buf, aph ^ 1u, abort_flag, a.st, 2)) break;
        if (tl && mb == 0 && j < 16) tl[1024 + 4 * j] = globaltimer_ns();
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * 256u;  // block b's accumulator at + 128 b
        bool ok = true;
        for (int c = 0; c < nch; c += kCS, ++ia, ++ib) {  // one stage: kCS chunks
          const int sa = ia % nAS, sb = ib % nBS;
          if ((kBf16W && !mbar_wait(af + sa, (ia / nAS) & 1u, abort_flag, a.st, 3)) ||
              !mbar_wait(b_full + sb, (ib / nBS) & 1u, abort_flag, a.st, 4)) {
            ok = false;
            break;
          }
          if (tl && mb == 0 && ia < 256) tl[4 * ia] = globaltimer_ns();
          tc_fence_after();
          const uint64_t bd = sw128_desc(smem_u32(smem + pf::kBOff + sb * kCS * pf::kBStageBytes));
          if (kBf16W) {
            const uint64_t ad = sw128_desc(smem_u32(smem + pf::a_stage_off(sa)));
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint32_t acc = (c | kk) != 0 ? 1u : 0u;
              umma_bf16(d_tmem, ad + 2u * kk, bd + 2u * kk, idesc, acc);
              if (nblk > 1)  // block 1's operand tile is 16 KB further (1024 in the 16-byte units)
                umma_bf16(d_tmem + 128u, ad + (uint64_t)(pf::kABlockBytes >> 4) + 2u * kk, bd + 2u * kk, idesc, acc);
            }
          } else if (mb < nblk) {
            // TMEM operand stage sa: chunk h, block mb, K step kk at columns + 64 h + 32 mb + 8 kk;
            // the stage's chunk h of B is 16 KB (1024 16-byte units) further
            const uint32_t at = tmem_base + (uint32_t)(pf::kAColT + sa * 64 * pf::kKS + 32 * mb);
            const uint32_t dt = d_tmem + 128u * (uint32_t)mb;
#pragma unroll
            for (int h = 0; h < pf::kKS; ++h)
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint32_t acc = (c | h | kk) != 0 ? 1u : 0u;
                umma_ts(dt, at + 64u * h + 8u * kk, bd + (uint64_t)(h * (pf::kBStageBytes >> 4)) + 2u * kk, idesc, acc);
              }
          }
          if (kBf16W) umma_commit(ae + sa);
          umma_commit(b_empty + sb);
        }
        if (!ok) break;
        umma_commit(accfull + buf);
      }
    }
  } else if (warp == 2) {
    // ---------------- activation producer: TMA boxes of 16 routed rows ----------------
    uint32_t it = 0;
    for (int unit = blockIdx.x; unit < total_units && !*abort_flag && a.fault != 1; unit += gridDim.x) {
      const int tile = unit / NP;
      const int row0 = a.tile_row0[tile], rows = a.tile_rows[tile];
      const int nbox = (rows + 15) >> 4;
      bool ok = true;
      for (int c = 0; c < nch; c += kCS, ++it) {  // one stage: kCS chunks
        const int s = it % nBS;
        const uint32_t ph = (it / nBS) & 1u;
        int got = 1;
        if (lane == 0) {
          got = mbar_wait(b_empty + s, ph ^ 1u, abort_flag, a.st, 7);
          if (got) mbar_arrive_expect_tx(b_full + s, (uint32_t)(kCS * nbox) * 2048u);
        }
        got = __shfl_sync(0xffffffffu, got, 0);
        if (!got) {
          ok = false;
          break;
        }
        uint8_t* st = smem + pf::kBOff + s * kCS * pf::kBStageBytes;
        if (lane < nbox)
#pragma unroll
          for (int h = 0; h < kCS; ++h)
            tma_2d(st + h * pf::kBStageBytes + lane * 2048, &tmap_b, (c + h) * kChunk, row0 + 16 * lane, b_full + s);
        __syncwarp();
      }
      if (!ok) break;
    }
  } else if (warp == pf::kMma2Warp || (kBf16W && warp < 3 + pf::kDequantWarps)) {
    // BF16 weights: one MMA issuer, nothing to dequantise
  } else if (warp < 3 + pf::kDequantWarps) {
    // ---------------- dequantisers: warp (block j, TMEM lane quarter Q); thread = one weight row ----------------
    const int j = (warp - 3) >> 2, Q = warp & 3;
    const int r = 32 * Q + lane;  // the row of block j this thread fills (its TMEM lane)
    const uint32_t t_row = tmem_base + ((uint32_t)(32 * Q) << 16) + (uint32_t)(pf::kAColT + 32 * j);
    uint32_t ir = 0, ia = 0;
    for (int unit = blockIdx.x; unit < total_units && !*abort_flag; unit += gridDim.x) {
      const int nblk = 2 * (unit % NP) + 1 < a.NB ? 2 : 1;
      bool ok = true;
      for (int c = 0; c < nch; c += pf::kKS, ++ia) {  // one TMEM stage: kKS chunks
        // the stage's packed chunks into registers first (their ring slots go straight back),
        // then the TMEM stage once the MMAs that read it last have completed
        RowRaw raw[pf::kKS];
        for (int h = 0; h < pf::kKS && ok; ++h, ++ir) {
          const int sr = ir % pf::kRawStages;
          if (!mbar_wait(raw_full + sr, (ir / pf::kRawStages) & 1u, abort_flag, a.st, 5)) {
            ok = false;
            break;
          }
          if (j < nblk) load_row_raw(smem + pf::kRawOff + sr * pf::kRawStageBytes + j * pf::kRawBlockBytes, r, raw[h]);
          __syncwarp();
          if (lane == 0) mbar_arrive(raw_empty + sr);
        }
        // TMEM slot sa last held stage ia - kAStagesT: wait until its MMAs have completed
        // (that stage's b_empty commit; B slots cycle kBStages >= kAStagesT, so the phase
        // parity is that stage's)
        const int sa = ia % pf::kAStagesT;
        const uint32_t prev = ia - pf::kAStagesT;
        if (!ok || (ia >= (uint32_t)pf::kAStagesT &&
                    !mbar_wait(b_empty + prev % pf::kBStages, (prev / pf::kBStages) & 1u, abort_flag, a.st, 8))) {
          ok = false;
          break;
        }
        if (tl && warp == 3 && lane == 0 && ia < 256) tl[4 * ia + 1] = globaltimer_ns();
        tc_fence_after();
        if (j < nblk) {
#pragma unroll
          for (int h = 0; h < pf::kKS; ++h) store_row_tmem<kF16>(raw[h], t_row + (uint32_t)(sa * 64 * pf::kKS + 64 * h));
          asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (tl && warp == 3 && ia < 256) tl[4 * ia + 2] = globaltimer_ns();
          mbar_arrive(b_full + ia % pf::kBStages);
        }
      }
      if (!ok) break;
    }
  } else {
    // ---------------- epilogue (256 threads; warp w reads TMEM lanes 32 (w % 4) .. of block (w - 11) / 4) ----------------
    const int quarter = warp & 3, blk = (warp - 3 - pf::kDequantWarps) >> 2;
    const int i = 32 * quarter + lane;  // accumulator row (TMEM lane)
    uint32_t j = 0;
    for (int unit = blockIdx.x; unit < total_units && !*abort_flag; unit += gridDim.x, ++j) {
      const int tile = unit / NP, nb0 = 2 * (unit % NP);
      const int nblk = nb0 + 1 < a.NB ? 2 : 1;
      const int e = a.tile_expert[tile], row0 = a.tile_row0[tile], rows = a.tile_rows[tile];
      const int N = (rows + 15) & ~15;
      const uint32_t buf = j % nBuf, aph = (j / nBuf) & 1u;
      if (!mbar_wait(accfull + buf, aph, abort_flag, a.st, 6)) break;
      if (tl && warp == 11 && lane == 0 && j < 16) tl[1024 + 4 * j + 1] = globaltimer_ns();
      tc_fence_after();
      const float* gs = a.gscale + 3 * e;
      if (kF16) {  // the tile's row exponents, once per unit, into this warp's shared-memory copy
        __syncwarp();  // done with the previous unit's
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int rr = 32 * q + lane;
          pex[rr] = rr < rows ? __ldg(a.pexp_x + row0 + rr) : 0;
          peh[rr] = rr < rows ? __ldg(a.pexp_h + row0 + rr) : 0;
        }
        __syncwarp();
      }
      if (blk < nblk) {
        const int nb = nb0 + blk;
        const uint32_t tbase = tmem_base + ((uint32_t)(32 * quarter) << 16) + buf * 256u + (uint32_t)(128 * blk);
        // 32 columns per TMEM round trip: two loads, one wait
        for (int col2 = 0; col2 < N; col2 += 32) {
          uint32_t vv[2][16];
          const bool two = col2 + 16 < N;
          tmem_ld16_nw(tbase + (uint32_t)col2, vv[0]);
          if (two) tmem_ld16_nw(tbase + (uint32_t)col2 + 16u, vv[1]);
          asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
          if (hh == 1 && !two) break;
          const int col = col2 + 16 * hh;
          const uint32_t* v = vv[hh];
          if (kGateUp) {
            const int R = 128 * nb + i;
            const int f = 8 * (R >> 4) + (R & 7);
            const bool is_gate = (R & 15) < 8;
            const float gsg = gs[0], gsu = gs[1];
            // W4A4 routed expert: h (rounded to BF16) is quantised to NVFP4 with the
            // w2 input scale; this warp's 16 gate lanes hold one 16-feature block
            // the x rows entered scaled by 2^-pexp_x (FP16 operands): undo it per column
            float sx[16];
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) sx[jj] = kF16 ? __int_as_float((127 + pex[col + jj]) << 23) : 1.0f;
            if (a.in_scale != nullptr && e < a.Er) {
              const float is1 = __ldg(a.in_scale + 2 * e + 1), inv6 = act_inv6(is1);
              float hv[16], am[16];
#pragma unroll
              for (int jj = 0; jj < 16; ++jj) {
                const float mine = __uint_as_float(v[jj]) * sx[jj];
                const float partner = __shfl_xor_sync(0xffffffffu, mine, 8);
                hv[jj] = is_gate ? __bfloat162float(__float2bfloat16_rn(silu(gsg * mine) * (gsu * partner))) : 0.f;
                am[jj] = fabsf(hv[jj]);
              }
              // block maxima over the 16 gate lanes (lane bit 3, gate / up, is never flipped)
#pragma unroll
              for (int o = 1; o <= 16; o <<= 1) {
                if (o == 8) continue;
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) am[jj] = fmaxf(am[jj], __shfl_xor_sync(0xffffffffu, am[jj], o));
              }
#pragma unroll
              for (int jj = 0; jj < 16; ++jj) {
                const float q = act_quant1(hv[jj], act_block_scale(am[jj], inv6, is1));
                if (is_gate && col + jj < rows) {
                  const size_t o = (size_t)(row0 + col + jj) * a.I + f;
                  if (kF16) reinterpret_cast<__half*>(a.h)[o] = __float2half_rn(q);  // code * scale: exact
                  else a.h[o] = __float2bfloat16_rn(q);
                }
              }
            } else {
              // every lane finishes 8 of the 16 tokens: the gate lane tokens 0..7 (its up
              // partner, 8 lanes away, sends those u), the up lane tokens 8..15
#pragma unroll
              for (int jj = 0; jj < 8; ++jj) {
                const float lo = __uint_as_float(v[jj]) * sx[jj], hi = __uint_as_float(v[8 + jj]) * sx[8 + jj];
                const float recv = __shfl_xor_sync(0xffffffffu, is_gate ? hi : lo, 8);
                const int t = is_gate ? jj : 8 + jj;
                if (col + t < rows) {
                  const float g = gsg * (is_gate ? lo : recv), u = gsu * (is_gate ? recv : hi);
                  const size_t o = (size_t)(row0 + col + t) * a.I + f;
                  // (fast exp and divide: a few FP32 ulp, far below h's FP16 / BF16 rounding)
                  const float sg = __fdividef(g, 1.0f + __expf(-g));
                  if (kF16)  // h times 2^-pexp_h as the down GEMM's FP16 operand (11 significant bits)
                    reinterpret_cast<__half*>(a.h)[o] = __float2half_rn(sg * u * __int_as_float((127 - peh[col + t]) << 23));
                  else
                    a.h[o] = __float2bfloat16_rn(sg * u);
                }
              }
            }
          } else {
            const int d = 128 * nb + i;
            const float gsd = gs[2];
            if (a.linear && a.out_f32) {
#pragma unroll
              for (int jj = 0; jj < 16; ++jj)
                if (col + jj < rows && d < a.n_out)
                  reinterpret_cast<float*>(a.out)[(size_t)(row0 + col + jj) * a.n_out + d] = gsd * __uint_as_float(v[jj]);
            } else if (a.linear) {
#pragma unroll
              for (int jj = 0; jj < 16; ++jj)
                if (col + jj < rows && d < a.n_out)
                  reinterpret_cast<__nv_bfloat16*>(a.out)[(size_t)(row0 + col + jj) * a.n_out + d] =
                      __float2bfloat16_rn(gsd * __uint_as_float(v[jj]));
            } else {
#pragma unroll
              for (int jj = 0; jj < 16; ++jj)
                if (col + jj < rows) {
                  // h row p entered scaled by 2^-pexp_h[p]
                  const float sh = kF16 ? __int_as_float((127 + peh[col + jj]) << 23) : 1.0f;
                  a.y[(size_t)(row0 + col + jj) * a.H + d] = gsd * (__uint_as_float(v[jj]) * sh);
                }
            }
          }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (tl && (warp == 11 || warp == 15) && lane == 0 && j < 16) tl[1024 + 4 * j + (warp == 11 ? 2 : 3)] = globaltimer_ns();
      if (lane == 0) mbar_arrive(accempty + buf);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(pf::kTmemCols)
                 : "memory");
  }
}

// The opt-in shared-memory size of every prefill kernel instantiation, set once
// per device (function attributes belong to each device's context).
static cudaError_t set_prefill_attrs() {
  constexpr int kCached = 64;
  static std::mutex mu;
  static bool done[kCached] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (dev >= 0 && dev < kCached && done[dev]) return cudaSuccess;
  const void* fns[] = {(const void*)prefill_gemm_kernel<true>, (const void*)prefill_gemm_kernel<false>,
                       (const void*)prefill_gemm_kernel<false, true>, (const void*)prefill_gemm_kernel<true, false, true>,
                       (const void*)prefill_gemm_kernel<false, false, true>};
  for (const void* f : fns) {
    e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, pf::kSmemBytes);
    if (e != cudaSuccess) return e;
  }
  if (dev >= 0 && dev < kCached) done[dev] = true;
  return cudaSuccess;
}

cudaError_t launch_prefill_ffn(const LayerDims& d, const uint8_t* blob, const float* gscale, int T, int k,
                               int num_sms, const PrefillMaps& maps, const Workspace& ws, int fault,
                               cudaEvent_t mid, void* out, cudaStream_t st) {
  cudaError_t ea = set_prefill_attrs();
  if (ea != cudaSuccess) return ea;
  const ExpertLayout L = d.linear ? linear_layout(d.H, d.I) : expert_layout(d.H, d.I);
  PrefillArgs a{};
  a.blob = blob;
  a.expert_stride = L.stride;
  a.gscale = gscale;
  a.H = d.H;
  a.I = d.I;
  a.tile_expert = ws.tile_expert;
  a.tile_row0 = ws.tile_row0;
  a.tile_rows = ws.tile_rows;
  a.num_tiles = ws.num_tiles;
  a.h = ws.h;
  a.y = ws.y;
  a.out = out;
  a.out_f32 = d.out_f32;
  a.linear = d.linear;
  a.n_out = d.n_out;
  a.in_scale = d.in_scale;
  a.Er = d.Er;
  a.st = ws.status;
  a.fault = fault;
  a.pexp_x = ws.pexp_x;
  a.pexp_h = ws.pexp_h;
  a.checks = d.checks;
  a.trace = ws.trace;
  a.E = d.E;
  a.R = T * (k + d.S);
  if (!d.linear) {  // gate/up: 2I interleaved rows, K = H (FP16 operands)
    a.mat_off = L.w13;
    a.K = d.H;
    a.NB = 2 * d.I / 128;
    prefill_gemm_kernel<true, false, true><<<num_sms, pf::kThreads, pf::kSmemBytes, st>>>(maps.x_perm, maps.x_perm, a);
  }
  if (mid) cudaEventRecord(mid, st);
  // down: H rows, K = I
  a.mat_off = L.w2;
  a.K = d.I;
  a.NB = d.H / 128;
  if (d.linear)  // the caller's BF16 x
    prefill_gemm_kernel<false><<<num_sms, pf::kThreads, pf::kSmemBytes, st>>>(maps.h, maps.h, a);
  else
    prefill_gemm_kernel<false, false, true><<<num_sms, pf::kThreads, pf::kSmemBytes, st>>>(maps.h, maps.h, a);
  return cudaGetLastError();
}

cudaError_t launch_router_gemm(const CUtensorMap& x_map, const CUtensorMap& w_map, int E, int H, int num_sms,
                               const float* ones3, const Workspace& ws, float* logits, cudaStream_t st) {
  cudaError_t ea = set_prefill_attrs();
  if (ea != cudaSuccess) return ea;
  PrefillArgs a{};
  a.gscale = ones3;  // "expert" 0, down-projection slot: 1.0
  a.K = H;
  a.NB = (E + 127) / 128;
  a.H = a.NB * 128;
  a.I = H;
  a.tile_expert = ws.tile_expert;
  a.tile_row0 = ws.tile_row0;
  a.tile_rows = ws.tile_rows;
  a.num_tiles = ws.num_tiles;
  a.out = logits;
  a.out_f32 = 1;
  a.linear = 1;
  a.n_out = E;
  a.st = ws.status;
  prefill_gemm_kernel<false, true><<<num_sms, pf::kThreads, pf::kSmemBytes, st>>>(x_map, w_map, a);
  return cudaGetLastError();
}

}  // namespace nvfp4moe
