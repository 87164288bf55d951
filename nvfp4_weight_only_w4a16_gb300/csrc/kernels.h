// Internal interface between the C-ABI layer (api.cu) and the kernels.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda.h>
#include "common.cuh"

namespace nvfp4moe {

// Device buffers of one handle.  R = max_tokens * max_top_k routed rows.
struct Workspace {
  int32_t* ids;        // [R]      expert of flattened row t*k+j
  float* wts;          // [R]      routing weight of flattened row
  int32_t* offsets;    // [E+1]    expert-major row offsets
  int32_t* perm;       // [R]      position -> flattened row
  int32_t* inv;        // [R]      flattened row -> position
  int32_t* tch_expert; // [E]      touched experts (decode), ascending
  int32_t* tch_row0;   // [E]
  int32_t* tch_rows;   // [E]
  int32_t* num_touched;// [1]
  __half* x16;         // [Tdec][H] FP16 activations, per-token power-of-two prescale
  int32_t* xexp;       // [Tdec]   prescale exponents
  __nv_bfloat16* h;    // [R][I]   silu(g)*u rounded to BF16, position order
  uint32_t* hmax;      // [R]      max |h| of each row (float bits, decode path)
  float* y;            // [R][H]   expert outputs, position order
  float* part_gu;      // split-K partial sums, gate/up: per decode warp 2 slots of [64][min(T,16)]
  int32_t* cnt_gu;     // arrival counters per gate/up 16-row group [maxU * I/8]
  float* part_dn;      // split-K partial sums, down: as part_gu
  int32_t* cnt_dn;     // arrival counters per down 16-row group    [maxU * H/16]
  int32_t* done_gu;    // finished gate/up 16-row groups per touched expert [maxU] (decode)
  int32_t* cmb;        // finished down 16-row groups per 64-wide slice of H [H/64] (decode)
  int32_t* exit_cnt;   // CTAs that finished the decode kernel [1]
  int32_t* blk_counts; // [nrb][E] per-rank-block histogram (prefill)
  int32_t* blk_base;   // [nrb][E] per-rank-block base inside each expert
  int32_t* local_rank; // [R] rank of a routed row inside its rank block (prefill)
  __nv_bfloat16* x_perm; // [R][H] gathered activations (prefill; the MoE's in FP16 times 2^-pexp_x[row])
  int32_t* pexp_x;       // [R] prefill: power-of-two prescale exponent of each gathered x row
  int32_t* pexp_h;       // [R] prefill: the same for each h row (FP16 in h), from the Cauchy-Schwarz bound
  int32_t* tile_expert;  // [max_tiles] prefill m-tiles
  int32_t* tile_row0;
  int32_t* tile_rows;
  int32_t* num_tiles;    // [1]
  // streaming decode kernel (decode_stream.cu)
  uint8_t* act_h;       // h rows of the streaming decode, 144 B per (row, 64-wide chunk): FP16 times 2^-p, float
                        // 2^p at +128; an expert's m rows from row0 form block [I/64][m] at row row0 * I/64
  uint8_t* act_x;       // [H/64][T <= 16][144 B] x rows per chunk, same form
  int act_rows;         // rows of act_h per chunk (>= T * slots of any decode step)
  int32_t* wctr;        // [1] work items claimed beyond the first one per CTA
  int32_t* done_c;      // [maxU][I/64] gate/up epilogue warps done per (touched expert, chunk of h)
  int32_t* x_ready;     // [H/64] tokens of act_x converted per chunk
  int32_t* logit_ready; // [1] router experts whose logits the streaming decode kernel has written
  DeviceStatus* status;
  DeviceStatus* status_sticky;  // optional (decode): a status word that outlives the launch's own
  float* logits;         // [max_tokens][Er] router logits (nvfp4_moe_forward_routed)
  float* ones3;          // [3] 1.0f: tensor scales of the BF16 router GEMM
  unsigned long long* trace;  // optional per-warp phase stamps of the decode kernel (NVFP4_MOE_TRACE=1)
};

// The route step's scoring rule (defaults: softmax over the chosen logits).
struct RouteParams {
  int score = 0;                 // 0: softmax over all experts, 1: sigmoid
  int renorm = 1;                // divide the chosen weights by their sum
  float scale = 1.0f;            // every final weight times this
  const float* bias = nullptr;   // [Er] device, added to the scores for the choice only
};

struct LayerDims {
  int E, H, I;     // E: experts in the blob (routed + shared)
  int logits_bf16;
  int out_f32;
  int Er;          // routed experts: router logits per token
  int S;           // shared experts (0 or 1): slots per token = top_k + S
  int linear;      // 1: a dense linear: one "expert" holding only a down matrix [H][I] (linear_layout),
                   // no routing and no gate/up; x [T][I] is the down GEMM's input
  int n_out;       // a dense linear's output features N <= H (H = N rounded up to 128; the
                   // padded rows are zero): out is [T][n_out]
  RouteParams rp;  // scoring rule of the route step
  const float* in_scale = nullptr;  // W4A4 routed experts: [E][2] input scales (w13, w2); the
                                    // caller passes tensor scales with them folded in
  const float* gs = nullptr;        // [E][3] the forward's tensor scales (prefill routing sizes h's prescale)
  const float* hbound = nullptr;    // [E] max_f ||Wg_f|| ||Wu_f|| (launch_gateup_bound)
  int checks = 0;                   // 1: kernels check table-derived indices (NVFP4_MOE_CHECKS=1)
};

constexpr int kRankTokens = 64;       // tokens per rank block in the prefill routing (8 per warp)
constexpr int kTileRows = 128;        // max routed rows per prefill m-tile (MMA N)
constexpr int kDecodeMaxTokens = 16;
constexpr int kDecodeWarpsPerSm = 16;  // warps of the decode kernel's one CTA per SM
// floats of the decode kernel's split-K partial-sum buffer (per phase)
inline size_t decode_part_floats(int num_sms, int T) {
  return (size_t)num_sms * kDecodeWarpsPerSm * 2 * 64 * (size_t)(T < 16 ? T : 16);
}

// W [N][K] into linear_layout(Np, K), Np = N rounded up to 128; rows N..Np-1 packed as zeros.
cudaError_t launch_pack_linear(const uint8_t* w_q, const uint8_t* w_s, uint8_t* blob, int N, int Np, int K,
                               cudaStream_t st);
// hb [E]: per expert, max over features f of ||Wg_f|| ||Wu_f|| (dequantised
// rows without the tensor scales) -- the bound that sizes h's FP16 prescale.
cudaError_t launch_gateup_bound(const uint8_t* w13_q, const uint8_t* w13_s, int E, int H, int I, float* hb,
                                cudaStream_t st);
cudaError_t launch_pack(const uint8_t* w13_q, const uint8_t* w13_s, const uint8_t* w2_q,
                        const uint8_t* w2_s, uint8_t* blob, int E, int H, int I, cudaStream_t st);
cudaError_t launch_debug_dequant(const uint8_t* blob, const float* gscale, int H, int I, int expert,
                                 int which, int via_bf16, float* out, cudaStream_t st);

cudaError_t launch_route_prefill(const LayerDims& d, const void* logits, const void* x, int T, int k,
                                 const Workspace& ws, cudaStream_t st);

// The whole decode forward (route, gate/up, down, combine) as one cooperative
// kernel; route_only = 1 runs the routing phase alone on one CTA and writes
// the tables (ids, wts, offsets, perm, inv) to the workspace.
// fault = 1 issues no copies, so the kernel's bounded waits expire (tests).
cudaError_t launch_decode_forward(const LayerDims& d, const uint8_t* blob, const float* gscale, const void* logits,
                                  const void* x, int T, int k, void* out, int route_only, int num_sms,
                                  const Workspace& ws, int fault, cudaStream_t st);
// Sets, once per device, the decode kernels' opt-in shared-memory size; returns it.
cudaError_t decode_prepare_device(int dev, int* smem_max);

// The streaming decode kernel (decode_stream.cu): the MoE decode forward for
// 1..16 tokens with dynamically claimed work items; route_only = 1 runs the
// routing alone on one CTA and writes the tables.  stream_supported says
// whether a layer and step can take it (W4A16 routed experts, not a dense
// linear, top_k + shared <= 17).
bool stream_supported(const LayerDims& d, int T, int k);
// router_w (BF16 [Er][H], or NULL): the kernel computes the router logits itself into ws.logits
// (logits is then ignored).
cudaError_t launch_decode_stream(const LayerDims& d, const uint8_t* blob, const float* gscale, const void* logits,
                                 const void* x, int T, int k, void* out, int route_only, int num_sms,
                                 const Workspace& ws, int fault, cudaStream_t st, const void* router_w = nullptr);
cudaError_t stream_prepare_device(int dev, int* smem_max);
size_t stream_act_h_bytes(int I, int rows);
// The hidden activations the last forward consumed, as FP32 [R][I]: src 0 --
// the BF16 rows in ws.h; src 1 -- the streaming decode kernel's chunk rows;
// src 2 -- the prefill GEMMs' FP16 rows in ws.h with pexp_h.
cudaError_t launch_hidden_to_f32(const Workspace& ws, int src, int R, int I, float* out, cudaStream_t st);
size_t stream_act_x_bytes(int H);

// A dense linear's tables: every token to matrix 0 with weight 1, identity
// perm/inv, offsets {0, T}, and m-tiles of tile_rows (16..128, a multiple of
// 16) rows in token order.
cudaError_t launch_route_linear(int T, int tile_rows, const Workspace& ws, cudaStream_t st);

// The router linear logits [T][E] = x [T][H] . W [E][H]^T (BF16 in, FP32 out):
// a GEMV kernel for T <= 16, else the tcgen05 GEMM over the m-tiles that
// launch_route_linear wrote (x_map: x [T][H], box {64, 16}; w_map: W [E][H],
// box {64, 128}; ones3: a device float[3] of ones).
cudaError_t launch_router_gemv(const void* x, const void* w, int T, int E, int H, float* logits, cudaStream_t st);
cudaError_t launch_router_gemm(const CUtensorMap& x_map, const CUtensorMap& w_map, int E, int H, int num_sms,
                               const float* ones3, const Workspace& ws, float* logits, cudaStream_t st);

struct PrefillMaps {
  CUtensorMap x_perm;  // [R][H] bf16, box {64, 16}, 128B swizzle
  CUtensorMap h;       // [R][I] bf16, box {64, 16}, 128B swizzle (a dense linear: its x [T][I])
};
// The grouped gate/up and down GEMMs; a dense linear (d.linear) runs the
// down GEMM alone and writes its rows to out (unused otherwise).
cudaError_t launch_prefill_ffn(const LayerDims& d, const uint8_t* blob, const float* gscale, int T, int k,
                               int num_sms, const PrefillMaps& maps, const Workspace& ws, int fault,
                               cudaEvent_t mid, void* out, cudaStream_t st);
size_t prefill_smem_bytes();

cudaError_t launch_combine(const LayerDims& d, int T, int k, const Workspace& ws, void* out,
                           cudaStream_t st);

}  // namespace nvfp4moe
