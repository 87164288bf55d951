/*
 * nvfp4_moe.h -- C ABI of the routed-expert MoE layer with weight-only NVFP4
 * (W4A16) experts, for one NVIDIA GB300 GPU (sm_103a).
 *
 * The layer (one call of nvfp4_moe_forward):
 *   route   : top-k of each token's router logits, weights = softmax over the
 *             k chosen logits;
 *   permute : group the T*k routed rows by expert (stable);
 *   gate/up : g = gs_g * (Wg x), u = gs_u * (Wu x), h = silu(g) * u;
 *   down    : y = gs_d * (Wd h);
 *   combine : out[t] = sum_j w[t][j] * y[t, j], rounded once to BF16.
 *
 * Sources.  The experts are "weight-only NVFP4": 4-bit values, one scale per
 * 16 weights and a per-tensor global scale ("tenhkspark/GLM-5.3-Flash-NVFP4-
 * Wabi", Config expectations: group_size = 16, weight_scale_2; "GLM-5.3-Flash
 * on Blackwell", The quantization).  Activations are BF16 and there is NO
 * activation scale anywhere in this interface: a weight-only MoE path that
 * consumes an input scale read an uninitialised 0.0 and zeroed every expert
 * ("GLM-5.3-Flash on Blackwell", The model loaded, served an API, and produced
 * garbage).  The 4-bit values are OCP MX E2M1, the group scales OCP E4M3.
 *
 * Beyond that forward the same kernels serve: a shared expert
 * (config.num_shared_experts), the routing variants (nvfp4_moe_set_scoring),
 * the BF16 router linear on the GPU (nvfp4_moe_set_router /
 * nvfp4_moe_forward_routed), the W4A4 comparison variant
 * (nvfp4_moe_set_act_quant), a dense W4A16 NVFP4 linear (nvfp4_linear_*), an
 * allocation-free decode forward (nvfp4_moe_forward_decode_static) and a
 * decode forward on pinned host buffers (nvfp4_moe_forward_host).
 *
 * Conventions for every call:
 *   - returns a status, never throws, never prints unless NVFP4_MOE_LOG=1;
 *   - device pointers are CUDA global-memory pointers on the handle's device
 *     (nvfp4_moe_forward_host alone takes host pointers);
 *     the caller keeps ownership of every pointer it passes;
 *   - work is enqueued on `stream`; only calls documented as synchronous
 *     wait for the GPU;
 *   - shape and pointer errors are detected on the host, before any launch.
 */
#ifndef NVFP4_MOE_H_
#define NVFP4_MOE_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum nvfp4_moe_status {
  NVFP4_MOE_OK = 0,
  NVFP4_MOE_ERR_INVALID_ARG = 1,       /* null handle/pointer, bad enum, misaligned pointer */
  NVFP4_MOE_ERR_UNSUPPORTED_SHAPE = 2, /* T, top_k, E, H or I outside the supported range   */
  NVFP4_MOE_ERR_NOT_PACKED = 3,        /* forward before a successful pack                  */
  NVFP4_MOE_ERR_WORKSPACE = 4,         /* device allocation failed in create                */
  NVFP4_MOE_ERR_CUDA = 5,              /* a CUDA runtime call failed (see status string)    */
  NVFP4_MOE_ERR_TIMEOUT = 6,           /* a bounded device-side wait gave up                */
  NVFP4_MOE_ERR_BAD_SCALE = 7,         /* tensor scale <= 0, NaN or Inf                     */
  NVFP4_MOE_ERR_NOT_IMPLEMENTED = 8,
  NVFP4_MOE_ERR_DEVICE_CHECK = 9       /* a device-side bounds check fired                  */
} nvfp4_moe_status;

typedef enum nvfp4_moe_logits_dtype {
  NVFP4_MOE_LOGITS_F32 = 0,
  NVFP4_MOE_LOGITS_BF16 = 1
} nvfp4_moe_logits_dtype;

typedef enum nvfp4_moe_out_dtype {
  NVFP4_MOE_OUT_BF16 = 0,      /* the layer's output rounded once to BF16 */
  NVFP4_MOE_OUT_F32 = 1        /* the FP32 combine result, unrounded      */
} nvfp4_moe_out_dtype;

typedef enum nvfp4_moe_score {
  NVFP4_MOE_SCORE_SOFTMAX = 0,
  NVFP4_MOE_SCORE_SIGMOID = 1
} nvfp4_moe_score;

typedef enum nvfp4_moe_path {
  NVFP4_MOE_PATH_AUTO = 0,     /* T <= decode_max_tokens -> decode, else prefill */
  NVFP4_MOE_PATH_DECODE = 1,   /* one streaming kernel, dequantised in registers  */
  NVFP4_MOE_PATH_PREFILL = 2   /* grouped tcgen05 GEMM, dequantised into TMEM     */
} nvfp4_moe_path;

/* Layer shape and limits, fixed at create.
 *   num_experts       E, 1..256
 *   hidden            H, multiple of 128, 128..16384
 *   inter             I (expert intermediate size), multiple of 128, 128..16384
 *   max_tokens        largest T a forward may pass (sizes the workspace), >= 1
 *   max_top_k         largest top_k a forward may pass, 1..min(E, 16)
 *   decode_max_tokens T at or below which AUTO picks the decode path, 0..16
 *   logits_dtype      nvfp4_moe_logits_dtype of router_logits
 *   device            CUDA device ordinal the handle lives on
 *   out_dtype         nvfp4_moe_out_dtype of out (BF16 unless set)
 *   num_shared_experts S, 0 or 1: the layer's single shared expert, used by
 *                     every token with weight 1 on top of its top_k routed
 *                     experts and added after them ("GLM-5.3-Flash on
 *                     Blackwell", The model loaded, served an API, and produced
 *                     garbage: "the single shared expert"; "GLM-5.3-Flash-NVFP4-h
 *                     — W4A16 dense-side quantization": shared experts in W4A16
 *                     NVFP4).  It has the routed experts' H and I, is packed as
 *                     expert E (after the E routed ones) and needs
 *                     E + S <= 256 and max_top_k + S <= 16.                     */
typedef struct nvfp4_moe_config {
  int num_experts;
  int hidden;
  int inter;
  int max_tokens;
  int max_top_k;
  int decode_max_tokens;
  int logits_dtype;
  int device;
  int out_dtype;
  int num_shared_experts;
} nvfp4_moe_config;

typedef struct nvfp4_moe* nvfp4_moe_t;

/* Allocate a handle: the packed-weight blob ((E + S) * 3*H*I * 9/16 bytes) and
 * the forward workspace (sized for max_tokens * (max_top_k + S) routed rows),
 * both on config->device.  Synchronous.  *out is NULL on failure. */
nvfp4_moe_status nvfp4_moe_create(const nvfp4_moe_config* config, nvfp4_moe_t* out);

/* Copy the experts into the handle's device layout: for every 128 weight rows
 * and 64-element K chunk, one 4608-byte tile of 4096 bytes of codes, ordered
 * so that each 16-byte vector holds two rows x 16 elements (one scale group
 * each; a 16-row group's vectors ordered by K group, then row), followed by
 * the matching 512 bytes of scales; a row block's tiles
 * follow one another along K, so any run of its chunks is one contiguous
 * bulk copy; the gate and up rows are interleaved in groups of 8.  Loads of
 * this layout are 16-byte vectorised and fully coalesced on both the decode
 * and the prefill path.
 * All inputs are DEVICE pointers in the canonical layout, per expert e (E
 * below counts the shared expert too when the handle has one: it is the last):
 *   w13_q [E][2I][H/2]  uint8  E2M1 codes, gate rows 0..I-1 then up rows
 *                              I..2I-1, row-major over K = H; element 2j in the
 *                              low nibble of byte j, element 2j+1 in the high
 *   w13_s [E][2I][H/16] uint8  E4M3 scale of elements 16g..16g+15 of the row
 *   w2_q  [E][H][I/2]   uint8  down projection, same rules with K = I
 *   w2_s  [E][H][I/16]  uint8
 *   gscale [E][3]       float  per-tensor scales (gate, up, down)
 * Every gscale must be finite and > 0, else NVFP4_MOE_ERR_BAD_SCALE and the
 * handle stays unpacked (this reads gscale back to the host: synchronous).
 * Inputs may be freed once the call returns. */
nvfp4_moe_status nvfp4_moe_pack(nvfp4_moe_t h, const uint8_t* w13_q, const uint8_t* w13_s,
                                const uint8_t* w2_q, const uint8_t* w2_s, const float* gscale,
                                cudaStream_t stream);

/* One forward of the layer, enqueued on `stream`; no host synchronisation and
 * no allocation, so the call can be captured into a CUDA graph.
 *   router_logits [T][E]  float or BF16 (config.logits_dtype), device
 *   x             [T][H]  BF16 activations, device, 16-byte aligned
 *   out           [T][H]  BF16 (or FP32, config.out_dtype) result, device,
 *                         16-byte aligned
 * 1 <= T <= max_tokens, 1 <= top_k <= max_top_k.  Ties between equal logits
 * go to the lower expert index; a NaN logit ranks below -inf and is counted
 * (see nvfp4_moe_get_status).  Concurrent forwards on one handle race on its
 * workspace: serialise them on one stream. */
nvfp4_moe_status nvfp4_moe_forward(nvfp4_moe_t h, const void* router_logits, int T, int top_k,
                                   const void* x, void* out, cudaStream_t stream);

/* The same forward (the layer above) with router_logits, x and out in HOST
 * memory that CUDA has mapped into the device's address space: page-locked
 * buffers from cudaHostAlloc / cudaMallocHost (mapped, at the same address,
 * whenever addressing is unified, as on every 64-bit system) or from
 * cudaHostRegister with cudaHostRegisterMapped.  Layouts, alignment and
 * ranges as for nvfp4_moe_forward.  The decode kernel reads the logits and x
 * and writes out in place -- on a Grace-Blackwell node over the coherent
 * CPU-GPU link -- so a step moves its inputs and its result without a
 * copy-engine transfer or a staging buffer.
 * Decode only: the W4A16 streaming decode kernel, T <= decode_max_tokens.  A
 * call that would take another path (T above that, a path forced to prefill,
 * W4A4 activation quantisation) returns NVFP4_MOE_ERR_UNSUPPORTED_SHAPE; a
 * pointer that is not mapped page-locked host memory (pageable, managed or
 * device memory) returns NVFP4_MOE_ERR_INVALID_ARG.  Both before anything is
 * enqueued.  Asynchronous like nvfp4_moe_forward: out holds the result once
 * `stream` has completed, and until then the host must neither write the
 * inputs nor read out. */
nvfp4_moe_status nvfp4_moe_forward_host(nvfp4_moe_t h, const void* router_logits, int T, int top_k,
                                        const void* x, void* out, cudaStream_t stream);

/* Synchronous: waits for the device, then reports the device-side status word
 * accumulated since the last call (and clears it).  Returns NVFP4_MOE_OK,
 * NVFP4_MOE_ERR_TIMEOUT or NVFP4_MOE_ERR_DEVICE_CHECK; *nan_logits (may be
 * NULL) receives the number of NaN router logits seen. */
nvfp4_moe_status nvfp4_moe_get_status(nvfp4_moe_t h, uint32_t* nan_logits);

/* Force a path (testing and measurement); AUTO by default.  The environment
 * variable NVFP4_MOE_FORCE_PATH=decode|prefill sets the default at create. */
nvfp4_moe_status nvfp4_moe_set_path(nvfp4_moe_t h, int path);

/* Decode forward that allocates nothing.  The GLM-5.3-Flash pages have no
 * counterpart to this call; it exists for callers that cannot call
 * cudaMalloc and so cannot create a handle: plugins whose host framework owns
 * and budgets every device byte, static-memory runtimes that forbid
 * allocation after start-up, and code that must not allocate while a graph
 * is being captured (no test in tests/ captures it).  It computes what
 * nvfp4_moe_forward computes on the decode path, from caller memory only:
 *   packed_experts  DEVICE, 16-byte aligned, E * 3*H*I*9/16 bytes in the
 *                   layout nvfp4_moe_pack writes (see nvfp4_moe_debug_packed_blob)
 *   gscale [E][3]   DEVICE float tensor scales (finite, > 0: not re-checked)
 *   router_logits [T][E] (logits_dtype), x [T][H] BF16, out [T][H] BF16
 * 1 <= T <= 16, 1 <= top_k <= min(E, 16); H, I as in nvfp4_moe_config.
 * All intermediates live in one static device array of 16 MiB that every GPU
 * loading this library holds until the process exits.  It needs about
 * T*top_k*(4.25*I + 4*H) + 36*H bytes plus small tables -- under 1 MiB for
 * E=128, H=4096, I=1536, T=2, top_k=8.
 * A shape needing more than the array returns
 * NVFP4_MOE_ERR_UNSUPPORTED_SHAPE before anything is enqueued.  The regions
 * that must start at zero are cleared by every call.  The first call on each
 * device looks up the array's device address and sets the decode kernels'
 * shared-memory attribute, with that device current: make it before any
 * stream capture.  Device ordinals 0..63 only (NVFP4_MOE_ERR_INVALID_ARG
 * above).  Calls whose GPU work overlaps (other streams, concurrent graph
 * replays) share the array and race: serialise them.  The call returns once
 * the work is enqueued; device-side errors (a bounded wait that gave up,
 * leaving a partial output; NaN router logits) are collected in a status word
 * inside the array that no call clears: read it with
 * nvfp4_moe_static_get_status. */
nvfp4_moe_status nvfp4_moe_forward_decode_static(const uint8_t* packed_experts, const float* gscale,
                                                 int num_experts, int hidden, int inter,
                                                 const void* router_logits, int logits_dtype, int T, int top_k,
                                                 const void* x, void* out, cudaStream_t stream);

/* Synchronous: waits for the current device, then reports and clears the
 * status word that nvfp4_moe_forward_decode_static calls on this device have
 * accumulated since the last read: NVFP4_MOE_OK, NVFP4_MOE_ERR_TIMEOUT (some
 * call's bounded wait gave up and its output is incomplete) or
 * NVFP4_MOE_ERR_DEVICE_CHECK; *nan_logits (may be NULL) receives the number
 * of NaN router logits those calls saw.  Like the forward it allocates
 * nothing; NVFP4_MOE_ERR_CUDA if a CUDA call fails. */
nvfp4_moe_status nvfp4_moe_static_get_status(uint32_t* nan_logits);

/* Fault injection for the allocation-free path's bounded-wait test, process-
 * wide: fault = 1 makes later nvfp4_moe_forward_decode_static calls issue no
 * weight copies, so their waits expire (after about 2 s) and report
 * NVFP4_MOE_ERR_TIMEOUT through nvfp4_moe_static_get_status; the GPU context
 * stays usable.  fault = 0 restores normal operation. */
nvfp4_moe_status nvfp4_moe_static_debug_set_fault(int fault);

/* Scoring rule of the route step (the router variants).  The pages keep the
 * routers as BF16 linears and do not state how their outputs become choices
 * and weights ("GLM-5.3-Flash on Blackwell", The quantization); the default
 * is softmax over the k chosen logits.  With s_e = softmax over all experts
 * (NVFP4_MOE_SCORE_SOFTMAX) or sigmoid(l_e) (NVFP4_MOE_SCORE_SIGMOID):
 *   choice : the k largest s_e + bias_e (bias NULL: the k largest logits,
 *            the same order), equal values -> lower expert index, NaN last;
 *   weights: the chosen s_e (never the bias); renormalize = 1 divides them
 *            by their sum over the k slots (softmax: the default rule;
 *            sigmoid: 1/k each if the sum is 0); then times scale.
 * bias: DEVICE float [num_experts] or NULL, copied on `stream` (the copy is
 * ordered before later forwards on that stream); scale finite and > 0.  A
 * shared expert keeps weight 1 under every rule.  Applies to later forwards
 * and nvfp4_moe_debug_route; a dense-linear handle returns
 * NVFP4_MOE_ERR_INVALID_ARG. */
nvfp4_moe_status nvfp4_moe_set_scoring(nvfp4_moe_t h, int score_func, int renormalize, float scale,
                                       const float* bias, cudaStream_t stream);

/* The router linear inside the library.  The routers stay BF16 linears
 * ("GLM-5.3-Flash on Blackwell", The quantization; "tenhkspark/GLM-5.3-Flash-
 * NVFP4-Wabi", Config expectations: the mlp.gate routers are excluded from
 * quantisation), so their logits can be computed here instead of passed in:
 *   nvfp4_moe_set_router copies w_router, DEVICE BF16 [num_experts][hidden]
 *   (16-byte aligned), into the handle (allocates once, then reuses; ordered
 *   on `stream`);
 *   nvfp4_moe_forward_routed is nvfp4_moe_forward with
 *   logits[t][e] = sum_h x[t][h] * w_router[e][h], accumulated in FP32 (no
 *   linear bias), computed on the GPU first: a GEMV kernel for T <= 16, the
 *   tcgen05 GEMM for larger T (its TMA descriptor over x is encoded on the
 *   host each call, so a captured graph replays with the x it was captured
 *   with).  Its time counts as route + permute in the stage times.
 *   nvfp4_moe_debug_logits copies the last forward_routed's logits
 *   [T][num_experts] FP32 to a DEVICE buffer.
 * NVFP4_MOE_ERR_INVALID_ARG: forward_routed before set_router, or a dense-
 * linear handle. */
nvfp4_moe_status nvfp4_moe_set_router(nvfp4_moe_t h, const void* w_router, cudaStream_t stream);
nvfp4_moe_status nvfp4_moe_forward_routed(nvfp4_moe_t h, int T, int top_k, const void* x, void* out,
                                          cudaStream_t stream);
nvfp4_moe_status nvfp4_moe_debug_logits(nvfp4_moe_t h, float* logits, cudaStream_t stream);

/* W4A4 comparison variant.  The stock checkpoint's routed experts are W4A4
 * NVFP4: activations are quantised to NVFP4 too, against a per-module FP32
 * input scale ("tenhkspark/GLM-5.3-Flash-NVFP4-Wabi", opening summary).
 * With input_scale set (DEVICE float [num_experts][2]: the gate/up input
 * scale, then the down input scale, of every routed expert; each finite and
 * > 0, else NVFP4_MOE_ERR_BAD_SCALE -- an input scale of 0 zeroes every expert,
 * "GLM-5.3-Flash on Blackwell", The model loaded, served an API, and produced
 * garbage), every routed expert quantises its input x and its hidden h
 * (rounded to BF16 first) per 16 elements: scale = E4M3(amax * fl(1/fl(6 is))),
 * code = E2M1(v * fl(1/fl(scale is))), round-to-nearest-even, saturating,
 * in FP32 in that order; the input scales multiply the tensor scales after
 * the dot products.  The shared
 * expert stays W4A16.  The quantised values are exact in BF16/FP16, so the
 * products run on the same tensor-core paths as W4A16.  NULL turns the
 * variant off.  Synchronous (reads the scales back to check them). */
nvfp4_moe_status nvfp4_moe_set_act_quant(nvfp4_moe_t h, const float* input_scale, cudaStream_t stream);

/* Per-stage timing.  With profiling on, every forward records CUDA events on
 * its stream before and after each stage.  nvfp4_moe_get_stage_times
 * (synchronous) returns in ms[0..3] the summed milliseconds of route+permute,
 * gate/up GEMM, down GEMM and combine over the forwards since profiling was
 * switched on or last read, and their number in *count; then it starts over.
 * Do not switch profiling on while capturing a CUDA graph. */
nvfp4_moe_status nvfp4_moe_set_profiling(nvfp4_moe_t h, int on);
nvfp4_moe_status nvfp4_moe_get_stage_times(nvfp4_moe_t h, float* ms, int* count);

/* Static text for a status code. */
const char* nvfp4_moe_status_string(nvfp4_moe_status s);

/* Text of the last error seen on this handle (CUDA error name, failed check). */
const char* nvfp4_moe_last_error(nvfp4_moe_t h);

/* Free the handle and its device memory (synchronises the device first). */
void nvfp4_moe_destroy(nvfp4_moe_t h);

/* ---- inspection entry points (same ABI; used by the parity tests) ------- */

/* Route and permute exactly as the forward of the chosen path does, into
 * caller DEVICE buffers, with K = top_k + S slots per token (the shared
 * expert, id E, weight 1, in the last): ids [T][K] int32, weights [T][K]
 * float, offsets [E+S+1] int32, perm [T*K] int32 (flattened index t*K+j of
 * the routed row at each expert-major position). */
nvfp4_moe_status nvfp4_moe_debug_route(nvfp4_moe_t h, const void* router_logits, int T, int top_k,
                                       int32_t* ids, float* weights, int32_t* offsets,
                                       int32_t* perm, cudaStream_t stream);

/* Copy the handle's packed expert blob (E * 3*H*I*9/16 bytes, the layout
 * described at nvfp4_moe_pack; per expert: the gate/up matrix's tiles
 * [2I/128][H/64][4608 B], then the down matrix's [H/128][I/64][4608 B]) into
 * a caller DEVICE buffer of at least that many bytes. */
nvfp4_moe_status nvfp4_moe_debug_packed_blob(nvfp4_moe_t h, void* dst, size_t dst_bytes, cudaStream_t stream);

/* Phase timeline of the decode kernel (handles created with the environment
 * variable NVFP4_MOE_TRACE=1 only).  Synchronous.  Copies up to n values into
 * host_dst: for each CTA c and warp w, 16 values at [(c*16 + w)*16]:
 * globaltimer nanosecond stamps 0 kernel start, 1 routed, 2 gate/up done,
 * 3 first down wait over, 4 down done, 5 exit barrier passed; durations (ns)
 * 6 gate/up and 7 down end-of-phase block finishing; stamps 8 inputs loaded,
 * 9 top-k chosen, 10 expert offsets scanned (warp 0 of each CTA only),
 * 11 gate/up stream ended, 12 down stream ended, 13 first gate/up stage
 * landed; 14 and 15: the SM clock counter (clock64) at stamps 0 and 1;
 * unused slots 0.  Clears the buffer. */
nvfp4_moe_status nvfp4_moe_debug_trace(nvfp4_moe_t h, uint64_t* host_dst, size_t n, size_t* n_written);

/* Dequantise one tensor of one expert from the PACKED blob into a caller
 * DEVICE buffer of float [N][K]: value = fp32(e2m1 * e4m3) * gscale, one
 * FP32 rounding.  which: 0 gate [I][H], 1 up [I][H], 2 down [H][I]. */
nvfp4_moe_status nvfp4_moe_debug_dequant(nvfp4_moe_t h, int expert, int which, float* w_out,
                                         cudaStream_t stream);

/* Copy the last forward's intermediates, in expert-major routed-row order
 * (row p = perm position p), into caller DEVICE buffers:
 *   hidden [T*K][I] float: h = silu(g)*u as the down GEMM consumed it, after
 *          its rounding to 16 bits (K = top_k + S),
 *   y      [T*K][H] float (expert output before the routing weight). */
nvfp4_moe_status nvfp4_moe_debug_intermediates(nvfp4_moe_t h, void* hidden, float* y,
                                               cudaStream_t stream);

/* Fault injection for the bounded-wait test: fault = 1 makes the prefill
 * producer and the decode kernel issue no copies, so the consumers' waits
 * expire (after about 2 s), the kernels record NVFP4_MOE_ERR_TIMEOUT in the
 * status word and return; the GPU context stays usable.  fault = 0 restores
 * normal operation. */
nvfp4_moe_status nvfp4_moe_debug_set_fault(nvfp4_moe_t h, int fault);

/* Fill every workspace buffer that each forward rewrites before it reads it
 * (routing tables, gathered and hidden activations, expert outputs, the
 * decode kernels' activation rows) with `byte`, on `stream`; the counters and
 * the status word keep their values.  A forward after it must give
 * bit-identical results: no kernel reads memory it has not written in the
 * same forward (the unused MMA columns that read such rows are never kept).
 * Tests use 0xFF (NaN in FP16, BF16 and FP32). */
nvfp4_moe_status nvfp4_moe_debug_poison_workspace(nvfp4_moe_t h, int byte, cudaStream_t stream);

/* Host only (no GPU needed): the status code a device status word stands for
 * -- bit 0 a bounded wait that gave up (NVFP4_MOE_ERR_TIMEOUT), bit 1 a
 * device-side bounds check that fired (NVFP4_MOE_ERR_DEVICE_CHECK; the checks
 * run when the handle was created with NVFP4_MOE_CHECKS=1), none
 * NVFP4_MOE_OK.  nvfp4_moe_get_status and nvfp4_moe_static_get_status decode
 * the words they read this way. */
nvfp4_moe_status nvfp4_moe_decode_status_word(uint32_t flags);

/* ---------------------------------------------------------------------------
 * Dense W4A16 NVFP4 linear: out[t] = gs * W x[t] for one weight matrix W
 * [N][K] in the same weight-only format as the experts (E2M1 codes, one E4M3
 * scale per 16 elements of a row, one FP32 tensor scale gs; activations
 * BF16, no activation scale).  The dense side of the model -- the attention
 * projections, the shared experts and lm_head -- is quantised this way
 * ("GLM-5.3-Flash-NVFP4-h — W4A16 dense-side quantization", opening summary
 * and Config expectations: W4A16_NVFP4 modules with group_size = 16).  It
 * runs on the same two paths as the MoE layer, as a one-matrix case: T <= 16
 * on the decode GEMV kernel, larger T on the tcgen05 GEMM kernel, both
 * writing out directly (no routing, no combine).
 *
 * A linear handle is an nvfp4_moe_t: nvfp4_moe_destroy, nvfp4_moe_set_path,
 * nvfp4_moe_get_status, nvfp4_moe_set_profiling / get_stage_times,
 * nvfp4_moe_debug_packed_blob and nvfp4_moe_debug_set_fault apply to it;
 * nvfp4_moe_pack, nvfp4_moe_forward, nvfp4_moe_debug_route and
 * nvfp4_moe_debug_intermediates return NVFP4_MOE_ERR_INVALID_ARG and
 * nvfp4_moe_debug_dequant NVFP4_MOE_ERR_NOT_IMPLEMENTED on it; the linear
 * calls below return NVFP4_MOE_ERR_INVALID_ARG on an MoE handle.
 * ------------------------------------------------------------------------- */
typedef struct nvfp4_linear_config {
  int out_features;      /* N: 16..16384, a multiple of 16 */
  int in_features;       /* K: 128..16384, a multiple of 128 */
  int max_tokens;        /* largest T of any forward, 1..2^20 */
  int decode_max_tokens; /* 0..16: T <= this takes the decode (GEMV) path */
  int out_dtype;         /* nvfp4_moe_out_dtype */
  int device;            /* CUDA device ordinal */
} nvfp4_linear_config;

/* Allocate a linear handle: the packed matrix (Np*K*9/16 bytes, Np = N
 * rounded up to a multiple of 128; the padding rows hold zeros and are never
 * written out) and a small workspace (tables for max_tokens rows; no
 * activation copies), on config->device.  Synchronous.  *out is NULL on
 * failure. */
nvfp4_moe_status nvfp4_linear_create(const nvfp4_linear_config* config, nvfp4_moe_t* out);

/* Copy W into the handle's device layout (the per-128-row, per-64-K-chunk
 * layout nvfp4_moe_pack writes for one down matrix).  DEVICE inputs:
 *   w_q [N][K/2]  uint8  E2M1 codes, row-major; element 2j in the low nibble
 *                        of byte j, element 2j+1 in the high (16-byte aligned)
 *   w_s [N][K/16] uint8  E4M3 scale of elements 16g..16g+15 of the row
 *   gscale [1]    float  the tensor scale: finite and > 0, else
 *                        NVFP4_MOE_ERR_BAD_SCALE and the handle stays unpacked
 * Synchronous (reads gscale back to the host).  Inputs may be freed once the
 * call returns. */
nvfp4_moe_status nvfp4_linear_pack(nvfp4_moe_t h, const uint8_t* w_q, const uint8_t* w_s, const float* gscale,
                                   cudaStream_t stream);

/* out [T][N] = gs * x [T][K] W^T, accumulated in FP32 and rounded once to
 * BF16 (or stored as FP32, config.out_dtype); x BF16 and out DEVICE, both
 * 16-byte aligned, 1 <= T <= max_tokens.  Enqueued on `stream`, no host
 * synchronisation and no allocation; the prefill path encodes a TMA
 * descriptor for x on the host each call, so a captured graph replays with
 * the x pointer it was captured with.  Concurrent forwards on one handle
 * race on its workspace: serialise them on one stream. */
nvfp4_moe_status nvfp4_linear_forward(nvfp4_moe_t h, int T, const void* x, void* out, cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* NVFP4_MOE_H_ */
