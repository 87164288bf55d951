// C ABI of the NVFP4 W4A16 MoE layer: handle, validation, dispatch.
// Every entry point returns a status and never throws; shape and pointer
// errors are caught here, before anything is enqueued.
#include <cstdio>
#include <cstdlib>
#include <algorithm>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "../../include/nvfp4_moe.h"
#include "kernels.h"

using namespace nvfp4moe;

struct nvfp4_moe {
  nvfp4_moe_config cfg;
  bool linear = false;  // a dense linear (nvfp4_linear_create): cfg holds E = 1, hidden = N padded to 128, inter = K
  int lin_n = 0;        // a dense linear's N (output features)
  RouteParams rp{};     // scoring rule (nvfp4_moe_set_scoring); rp.bias points at `bias` when set
  float* bias = nullptr;  // [num_experts] device copy of the choice bias
  void* w_router = nullptr;  // [num_experts][hidden] BF16 router weight (nvfp4_moe_set_router)
  CUtensorMap w_router_map{};  // over w_router, box {64, 128}, 128B swizzle
  bool have_router = false;
  // W4A4 comparison variant (nvfp4_moe_set_act_quant)
  bool w4a4 = false;
  float* in_scale = nullptr;     // [E][2] device input scales (w13, w2); shared expert's unused
  float* gs_eff = nullptr;       // [E][3] device tensor scales with the input scales folded in
  float* hbound = nullptr;       // [E] max_f ||Wg_f|| ||Wu_f|| (written at pack): sizes h's FP16 prescale
  std::vector<std::pair<uint8_t*, size_t>> data_regions;  // workspace buffers every forward rewrites
  int checks = 0;  // NVFP4_MOE_CHECKS=1 at create: kernels check table-derived indices
  std::vector<float> gs_host;    // [E][3] the packed tensor scales
  std::vector<float> is_host;    // [E][2]
  int path = NVFP4_MOE_PATH_AUTO;
  int num_sms = 0;
  bool packed = false;
  bool log = false;
  bool logged_path[3] = {false, false, false};
  uint8_t* blob = nullptr;
  float* gscale = nullptr;
  void* ws_mem = nullptr;
  size_t ws_bytes = 0;
  Workspace ws{};
  PrefillMaps maps{};
  int last_T = 0, last_k = 0;
  int last_hsrc = 0;  // where the last forward's hidden activations are (launch_hidden_to_f32's src)
  bool last_routed = false;
  int fault = 0;
  bool profiling = false;
  std::vector<cudaEvent_t> ev_pool;  // 5 events per profiled forward
  size_t ev_used = 0;
  char last_error[256] = {0};
};

namespace {

struct DeviceGuard {
  int prev = -1;
  bool changed = false;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) == cudaSuccess && prev != dev) changed = cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceGuard() {
    if (changed) cudaSetDevice(prev);
  }
};

nvfp4_moe_status fail(nvfp4_moe* h, nvfp4_moe_status s, const std::string& msg) {
  if (h) snprintf(h->last_error, sizeof(h->last_error), "%s", msg.c_str());
  if (h && h->log) fprintf(stderr, "[nvfp4_moe] %s\n", msg.c_str());
  return s;
}

nvfp4_moe_status cuda_fail(nvfp4_moe* h, cudaError_t e, const char* where) {
  return fail(h, NVFP4_MOE_ERR_CUDA, std::string(where) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")");
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 2D BF16 [rows][cols] row-major, box = 64 columns x box_rows rows, 128B swizzle.
bool encode_rows_map(CUtensorMap* map, void* base, uint64_t rows, uint64_t cols, uint32_t box_rows = 16) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct Carver {
  size_t off = 0;
  std::vector<std::pair<void**, size_t>> items;
  std::vector<bool> is_data;  // rewritten by every forward before it is read (no counter, no constant)
  template <class T>
  void add(T** p, size_t count, bool data = false) {
    items.push_back({reinterpret_cast<void**>(p), count * sizeof(T)});
    is_data.push_back(data);
  }
  size_t layout() {
    off = 0;
    for (auto& it : items) off = ((off + 255) & ~size_t(255)) + it.second;
    return off + 256;
  }
  void assign(uint8_t* base) {
    size_t o = 0;
    for (auto& it : items) {
      o = (o + 255) & ~size_t(255);
      *it.first = base + o;
      o += it.second;
    }
  }
};

int choose_path(const nvfp4_moe* h, int T, int k) {
  if (h->path != NVFP4_MOE_PATH_AUTO) return h->path;
  return (T <= h->cfg.decode_max_tokens && T <= kDecodeMaxTokens &&
          T * (k + h->cfg.num_shared_experts) <= kDecodeMaxTokens * 16)
             ? NVFP4_MOE_PATH_DECODE
             : NVFP4_MOE_PATH_PREFILL;
}

nvfp4_moe_status check_forward_args(nvfp4_moe* h, const void* logits, int T, int top_k, int path) {
  if (!h) return NVFP4_MOE_ERR_INVALID_ARG;
  if (h->linear) return fail(h, NVFP4_MOE_ERR_INVALID_ARG, "a dense-linear handle: call nvfp4_linear_forward");
  if (!h->packed) return fail(h, NVFP4_MOE_ERR_NOT_PACKED, "forward before a successful pack");
  if (!logits) return fail(h, NVFP4_MOE_ERR_INVALID_ARG, "router_logits is NULL");
  if (!aligned(logits, h->cfg.logits_dtype == NVFP4_MOE_LOGITS_BF16 ? 2 : 4))
    return fail(h, NVFP4_MOE_ERR_INVALID_ARG, "router_logits misaligned");
  if (T < 1 || T > h->cfg.max_tokens) return fail(h, NVFP4_MOE_ERR_UNSUPPORTED_SHAPE, "T outside 1..max_tokens");
  if (top_k < 1 || top_k > h->cfg.max_top_k || top_k > h->cfg.num_experts)
    return fail(h, NVFP4_MOE_ERR_UNSUPPORTED_SHAPE, "top_k outside 1..min(max_top_k, E)");
  if (path == NVFP4_MOE_PATH_DECODE && (T > kDecodeMaxTokens))
    return fail(h, NVFP4_MOE_ERR_UNSUPPORTED_SHAPE, "decode path takes at most 16 tokens");
  if (path == NVFP4_MOE_PATH_DECODE && T * (top_k + h->cfg.num_shared_experts) > kDecodeMaxTokens * 16)
    return fail(h, NVFP4_MOE_ERR_UNSUPPORTED_SHAPE, "decode path takes at most 256 routed rows");
  return NVFP4_MOE_OK;
}

LayerDims dims_of(const nvfp4_moe* h) {
  LayerDims d{h->cfg.num_experts + h->cfg.num_shared_experts, h->cfg.hidden, h->cfg.inter,
              h->cfg.logits_dtype == NVFP4_MOE_LOGITS_BF16, h->cfg.out_dtype == NVFP4_MOE_OUT_F32,
              h->cfg.num_experts, h->cfg.num_shared_experts, h->linear ? 1 : 0, h->lin_n};
  d.rp = h->rp;
  d.in_scale = h->w4a4 ? h->in_scale : nullptr;
  d.gs = h->w4a4 ? h->gs_eff : h->gscale;
  d.hbound = h->hbound;
  d.checks = h->checks;
  return d;
}

size_t blob_bytes_of(const nvfp4_moe_config& c, bool linear) {
  return linear ? linear_layout(c.hidden, c.inter).stride
                : (size_t)(c.num_experts + c.num_shared_experts) * expert_layout(c.hidden, c.inter).stride;
}

// Handle allocation shared by the MoE layer and the dense linear (c already
// validated; a linear's c holds one expert with hidden = N and inter = K).
nvfp4_moe_status create_handle(const nvfp4_moe_config* c, bool linear, int lin_n, nvfp4_moe_t* out);

// W4A4: tensor scales with the input scales folded in (routed experts: gate and
// up times is_w13, down times is_w2; the shared expert keeps its own).
nvfp4_moe_status upload_gs_eff(nvfp4_moe* h, cudaStream_t st) {
  const int E = h->cfg.num_experts + h->cfg.num_shared_experts, Er = h->cfg.num_experts;
  if (h->gs_host.size() != (size_t)3 * E) return NVFP4_MOE_OK;  // not packed yet: pack uploads it
  std::vector<float> g(h->gs_host);
  for (int e = 0; e < Er; ++e) {
    g[3 * e] *= h->is_host[2 * e];
    g[3 * e + 1] *= h->is_host[2 * e];
    g[3 * e + 2] *= h->is_host[2 * e + 1];
  }
  cudaError_t err = cudaMemcpyAsync(h->gs_eff, g.data(), sizeof(float) * g.size(), cudaMemcpyHostToDevice, st);
  if (err == cudaSuccess) err = cudaStreamSynchronize(st);  // g lives on this frame
  if (err != cudaSuccess) return cuda_fail(h, err, "W4A4 tensor scales upload");
  return NVFP4_MOE_OK;
}

// Forward events: 5 per profiled forward (ev[i] stays NULL when profiling is off).
nvfp4_moe_status take_events(nvfp4_moe* h, cudaEvent_t (&ev)[5]) {
  if (!h->profiling) return NVFP4_MOE_OK;
  for (int i = 0; i < 5; ++i) {
    if (h->ev_used == h->ev_pool.size()) {
      cudaEvent_t e0;
      if (cudaEventCreate(&e0) != cudaSuccess) return cuda_fail(h, cudaGetLastError(), "event create");
      h->ev_pool.push_back(e0);
    }
    ev[i] = h->ev_pool[h->ev_used++];
  }
  return NVFP4_MOE_OK;
}

// The decode forward takes the streaming kernel wherever it applies (W4A16
// routed experts); NVFP4_MOE_DECODE_KERNEL=fused keeps the earlier fused
// kernel for comparison.
bool use_stream(const nvfp4_moe* h, const LayerDims& d, int T, int k) {
  static const bool fused = [] {
    const char* s = getenv("NVFP4_MOE_DECODE_KERNEL");
    return s && !strcmp(s, "fused");
  }();
  (void)h;
  return !fused && stream_supported(d, T, k);
}

nvfp4_moe_status run_route(nvfp4_moe* h, const void* logits, const void* x, int T, int k, int path,
                           cudaStream_t st, int logits_bf16 = -1) {
  LayerDims d = dims_of(h);
  if (logits_bf16 >= 0) d.logits_bf16 = logits_bf16;
  cudaError_t e = path != NVFP4_MOE_PATH_DECODE ? launch_route_prefill(d, logits, x, T, k, h->ws, st)
                   : use_stream(h, d, T, k)
                       ? launch_decode_stream(d, h->blob, h->gscale, logits, nullptr, T, k, nullptr, 1, h->num_sms,
                                              h->ws, 0, st)
                       : launch_decode_forward(d, h->blob, h->gscale, logits, nullptr, T, k, nullptr, 1, h->num_sms,
                                               h->ws, 0, st);
  if (e != cudaSuccess) return cuda_fail(h, e, "route launch");
  return NVFP4_MOE_OK;
}

}  // namespace

extern "C" {

const char* nvfp4_moe_status_string(nvfp4_moe_status s) {
  switch (s) {
    case NVFP4_MOE_OK: return "ok";
    case NVFP4_MOE_ERR_INVALID_ARG: return "invalid argument";
    case NVFP4_MOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case NVFP4_MOE_ERR_NOT_PACKED: return "weights not packed";
    case NVFP4_MOE_ERR_WORKSPACE: return "device allocation failed";
    case NVFP4_MOE_ERR_CUDA: return "CUDA error";
    case NVFP4_MOE_ERR_TIMEOUT: return "device-side wait timed out";
    case NVFP4_MOE_ERR_BAD_SCALE: return "tensor scale is zero, negative, NaN or Inf";
    case NVFP4_MOE_ERR_NOT_IMPLEMENTED: return "not implemented";
    case NVFP4_MOE_ERR_DEVICE_CHECK: return "device-side bounds check fired";
  }
  return "unknown status";
}

const char* nvfp4_moe_last_error(nvfp4_moe_t h) { return h ? h->last_error : "null handle"; }

nvfp4_moe_status nvfp4_moe_create(const nvfp4_moe_config* c, nvfp4_moe_t* out) {
  if (!out) return NVFP4_MOE_ERR_INVALID_ARG;
  *out = nullptr;
  if (!c) return NVFP4_MOE_ERR_INVALID_ARG;
  if (c->num_experts < 1 || c->num_experts > 256) return NVFP4_MOE_ERR_UNSUPPORTED_SHAPE;
  if (c->hidden < 128 || c->hidden > 16384 || c->hidden % 128) return NVFP4_MOE_ERR_UNSUPPORTED_SHAPE;
  if (c->inter < 128 || c->inter > 16384 || c->inter % 128) return NVFP4_MOE_ERR_UNSUPPORTED_SHAPE;
  if (c->max_tokens < 1 || c->max_tokens > (1 << 20)) return NVFP4_MOE_ERR_UNSUPPORTED_SHAPE;
  if (c->max_top_k < 1 || c->max_top_k > 16 || c->max_top_k > c->num_experts) return NVFP4_MOE_ERR_UNSUPPORTED_SHAPE;
  if (c->decode_max_tokens < 0 || c->decode_max_tokens > kDecodeMaxTokens) return NVFP4_MOE_ERR_UNSUPPORTED_SHAPE;
  if (c->logits_dtype != NVFP4_MOE_LOGITS_F32 && c->logits_dtype != NVFP4_MOE_LOGITS_BF16)
    return NVFP4_MOE_ERR_INVALID_ARG;
  if (c->out_dtype != NVFP4_MOE_OUT_BF16 && c->out_dtype != NVFP4_MOE_OUT_F32) return NVFP4_MOE_ERR_INVALID_ARG;
  if (c->num_shared_experts < 0 || c->num_shared_experts > 1) return NVFP4_MOE_ERR_UNSUPPORTED_SHAPE;
  if (c->num_experts + c->num_shared_experts > 256 || c->max_top_k + c->num_shared_experts > 16)
    return NVFP4_MOE_ERR_UNSUPPORTED_SHAPE;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || c->device < 0 || c->device >= ndev) return NVFP4_MOE_ERR_INVALID_ARG;
  return create_handle(c, false, 0, out);
}

}  // extern "C"

namespace {
nvfp4_moe_status create_handle(const nvfp4_moe_config* c, bool linear, int lin_n, nvfp4_moe_t* out) {
  nvfp4_moe* h = new (std::nothrow) nvfp4_moe();
  if (!h) return NVFP4_MOE_ERR_WORKSPACE;
  h->cfg = *c;
  h->linear = linear;
  h->lin_n = lin_n;
  const char* lg = getenv("NVFP4_MOE_LOG");
  h->log = lg && lg[0] == '1';
  const char* ck = getenv("NVFP4_MOE_CHECKS");
  h->checks = ck && ck[0] == '1';
  const char* fp = getenv("NVFP4_MOE_FORCE_PATH");
  if (fp && !strcmp(fp, "decode")) h->path = NVFP4_MOE_PATH_DECODE;
  if (fp && !strcmp(fp, "prefill")) h->path = NVFP4_MOE_PATH_PREFILL;

  DeviceGuard g(c->device);
  cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, c->device);
  // E: experts in the blob (routed + shared); K: routed-row slots per token
  const int E = c->num_experts + c->num_shared_experts, H = c->hidden, I = c->inter;
  const int K = c->max_top_k + c->num_shared_experts;
  const size_t R = (size_t)c->max_tokens * K;
  const size_t Rm = R < 256 ? 256 : R;
  const size_t maxU = (size_t)std::min(E, kDecodeMaxTokens * K);
  const size_t ncta = ((size_t)c->max_tokens + kRankTokens - 1) / kRankTokens;
  // m-tiles: the MoE's (<= R/128 + E + 1) and the router GEMM's (<= one per SM)
  const size_t max_tiles = std::max(R / kTileRows + E + 1, (size_t)h->num_sms + 2);
  const size_t blob_bytes = blob_bytes_of(*c, linear);
  // a dense linear reads x and writes out directly: no permuted copies, no
  // hidden rows, no FP32 expert outputs
  const size_t RmH = linear ? 1 : Rm * H, RmI = linear ? 1 : Rm * I;

  Carver cv;
  Workspace& w = h->ws;
  cv.add(&w.ids, Rm, true);
  cv.add(&w.wts, Rm, true);
  cv.add(&w.offsets, E + 1, true);
  cv.add(&w.perm, Rm, true);
  cv.add(&w.inv, Rm, true);
  cv.add(&w.tch_expert, E, true);
  cv.add(&w.tch_row0, E, true);
  cv.add(&w.tch_rows, E, true);
  cv.add(&w.num_touched, 1);
  cv.add(&w.x16, (size_t)kDecodeMaxTokens * H, true);
  cv.add(&w.xexp, kDecodeMaxTokens, true);
  cv.add(&w.h, RmI, true);
  cv.add(&w.hmax, Rm);
  cv.add(&w.y, RmH, true);
  cv.add(&w.part_gu, decode_part_floats(h->num_sms, kDecodeMaxTokens), true);
  cv.add(&w.cnt_gu, maxU * (2 * I / 16));
  cv.add(&w.part_dn, decode_part_floats(h->num_sms, kDecodeMaxTokens), true);
  cv.add(&w.cnt_dn, maxU * (H / 16));
  cv.add(&w.done_gu, maxU);
  cv.add(&w.cmb, H / 64);
  cv.add(&w.exit_cnt, 1);
  w.act_rows = kDecodeMaxTokens * K;  // a dense linear: K = 1, its x rows as the "h" rows
  cv.add(&w.act_h, stream_act_h_bytes(I, w.act_rows), true);
  cv.add(&w.act_x, linear ? 16 : stream_act_x_bytes(H), true);
  cv.add(&w.wctr, 1);
  cv.add(&w.done_c, maxU * (I / 64));
  cv.add(&w.x_ready, H / 64);
  cv.add(&w.logit_ready, 1);
  cv.add(&w.blk_counts, ncta * E, true);
  cv.add(&w.blk_base, ncta * E, true);
  cv.add(&w.local_rank, Rm, true);
  cv.add(&w.x_perm, RmH, true);
  cv.add(&w.pexp_x, Rm, true);
  cv.add(&w.pexp_h, Rm, true);
  cv.add(&w.tile_expert, max_tiles, true);
  cv.add(&w.tile_row0, max_tiles, true);
  cv.add(&w.tile_rows, max_tiles, true);
  cv.add(&w.num_tiles, 1, true);
  cv.add(&w.status, 1);
  cv.add(&w.logits, linear ? 1 : (size_t)c->max_tokens * c->num_experts, true);
  cv.add(&w.ones3, 3);
  const char* tr = getenv("NVFP4_MOE_TRACE");
  const bool trace = tr && tr[0] == '1';
  if (trace) cv.add(&w.trace, (size_t)h->num_sms * 16 * 16);
  h->ws_bytes = cv.layout();

  if (cudaMalloc(&h->blob, blob_bytes) != cudaSuccess || cudaMalloc(&h->gscale, sizeof(float) * 3 * E) != cudaSuccess ||
      cudaMalloc(&h->bias, sizeof(float) * E) != cudaSuccess || cudaMalloc(&h->in_scale, sizeof(float) * 2 * E) != cudaSuccess ||
      cudaMalloc(&h->gs_eff, sizeof(float) * 3 * E) != cudaSuccess || cudaMalloc(&h->hbound, sizeof(float) * E) != cudaSuccess ||
      cudaMalloc(&h->ws_mem, h->ws_bytes) != cudaSuccess) {
    cudaGetLastError();
    nvfp4_moe_destroy(h);
    return NVFP4_MOE_ERR_WORKSPACE;
  }
  cv.assign(static_cast<uint8_t*>(h->ws_mem));
  for (size_t i = 0; i < cv.items.size(); ++i)
    if (cv.is_data[i]) h->data_regions.push_back({static_cast<uint8_t*>(*cv.items[i].first), cv.items[i].second});
  const float ones[3] = {1.0f, 1.0f, 1.0f};
  if (cudaMemset(h->ws_mem, 0, h->ws_bytes) != cudaSuccess ||
      cudaMemcpy(w.ones3, ones, sizeof(ones), cudaMemcpyHostToDevice) != cudaSuccess) {
    nvfp4_moe_destroy(h);
    return NVFP4_MOE_ERR_CUDA;
  }
  if (!linear && (!encode_rows_map(&h->maps.x_perm, w.x_perm, Rm, H) || !encode_rows_map(&h->maps.h, w.h, Rm, I))) {
    nvfp4_moe_destroy(h);
    return NVFP4_MOE_ERR_CUDA;
  }
  *out = h;
  return NVFP4_MOE_OK;
}
}  // namespace

extern "C" {

void nvfp4_moe_destroy(nvfp4_moe_t h) {
  if (!h) return;
  {
    DeviceGuard g(h->cfg.device);
    cudaDeviceSynchronize();
    for (cudaEvent_t ev : h->ev_pool) cudaEventDestroy(ev);
    if (h->blob) cudaFree(h->blob);
    if (h->gscale) cudaFree(h->gscale);
    if (h->bias) cudaFree(h->bias);
    if (h->w_router) cudaFree(h->w_router);
    if (h->in_scale) cudaFree(h->in_scale);
    if (h->gs_eff) cudaFree(h->gs_eff);
    if (h->hbound) cudaFree(h->hbound);
    if (h->ws_mem) cudaFree(h->ws_mem);
  }
  delete h;
}

nvfp4_moe_status nvfp4_moe_set_path(nvfp4_moe_t h, int path) {
  if (!h) return NVFP4_MOE_ERR_INVALID_ARG;
  if (path < NVFP4_MOE_PATH_AUTO || path > NVFP4_MOE_PATH_PREFILL) return NVFP4_MOE_ERR_INVALID_ARG;
  h->path = path;
  return NVFP4_MOE_OK;
}

nvfp4_moe_status nvfp4_moe_set_profiling(nvfp4_moe_t h, int on) {
  if (!h) return NVFP4_MOE_ERR_INVALID_ARG;
  h->profiling = on != 0;
  h->ev_used = 0;
  return NVFP4_MOE_OK;
}

nvfp4_moe_status nvfp4_moe_get_stage_times(nvfp4_moe_t h, float* ms, int* count) {
  if (!h || !ms || !count) return NVFP4_MOE_ERR_INVALID_ARG;
  DeviceGuard g(h->cfg.device);
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(h, e, "get_stage_times");
  for (int i = 0; i < 4; ++i) ms[i] = 0.f;
  const int n = (int)(h->ev_used / 5);
  for (int f = 0; f < n; ++f)
    for (int i = 0; i < 4; ++i) {
      float t = 0.f;
      e = cudaEventElapsedTime(&t, h->ev_pool[5 * f + i], h->ev_pool[5 * f + i + 1]);
      if (e != cudaSuccess) return cuda_fail(h, e, "get_stage_times elapsed");
      ms[i] += t;
    }
  *count = n;
  h->ev_used = 0;
  return NVFP4_MOE_OK;
}

nvfp4_moe_status nvfp4_moe_set_scoring(nvfp4_moe_t h, int score_func, int renormalize, float scale,
                                       const float* bias, cudaStream_t st) {
  if (!h) return NVFP4_MOE_ERR_INVALID_ARG;
  if (h->linear) return fail(h, NVFP4_MOE_ERR_INVALID_ARG, "set_scoring: a dense linear has no routing");
  if (score_func != NVFP4_MOE_SCORE_SOFTMAX && score_func != NVFP4_MOE_SCORE_SIGMOID)
    return fail(h, NVFP4_MOE_ERR_INVALID_ARG, "set_scoring: unknown score function");
  if (renormalize != 0 && renormalize != 1) return fail(h, NVFP4_MOE_ERR_INVALID_ARG, "set_scoring: renormalize is 0 or 1");
  if (!(scale > 0.0f) || scale > 3.4e38f) return fail(h, NVFP4_MOE_ERR_INVALID_ARG, "set_scoring: scale must be finite > 0");
  if (bias && !aligned(bias, 4)) return fail(h, NVFP4_MOE_ERR_INVALID_ARG, "set_scoring: bias misaligned");
  DeviceGuard g(h->cfg.device);
  if (bias) {
    cudaError_t e = cudaMemcpyAsync(h->bias, bias, sizeof(float) * h->cfg.num_experts, cudaMemcpyDeviceToDevice, st);
    if (e != cudaSuccess) return cuda_fail(h, e, "set_scoring: bias copy");
  }
  h->rp.score = score_func;
  h->rp.renorm = renormalize;
  h->rp.scale = scale;
  h->rp.bias = bias ? h->bias : nullptr;
  return NVFP4_MOE_OK;
}

nvfp4_moe_status nvfp4_moe_set_act_quant(nvfp4_moe_t h, const float* input_scale, cudaStream_t st) {
  if (!h) return NVFP4_MOE_ERR_INVALID_ARG;
  if (h->linear) return fail(h, NVFP4_MOE_ERR_INVALID_ARG, "set_act_quant: not for a dense-linear handle");
  if (!input_scale) {
    h->w4a4 = false;
    return NVFP4_MOE_OK;
  }
  if (!aligned(input_scale, 4)) return fail(h, NVFP4_MOE_ERR_INVALID_ARG, "set_act_quant: misaligned input_scale");
  DeviceGuard g(h->cfg.device);
  const int E = h->cfg.num_experts + h->cfg.num_shared_experts, Er = h->cfg.num_experts;
  std::vector<float> is((size_t)2 * E, 0.0f);
  cudaError_t e = cudaMemcpyAsync(is.data(), input_scale, sizeof(float) * 2 * Er, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(h, e, "set_act_quant: reading input_scale");
  for (int i = 0; i < 2 * Er; ++i) {
    const float v = is[i];
    if (!(v > 0.0f) || v != v || v > 3.4e38f) {
      h->w4a4 = false;
      return fail(h, NVFP4_MOE_ERR_BAD_SCALE, "set_act_quant: input scale " + std::to_string(i % 2) + " of expert " +
                                                  std::to_string(i / 2) + " is not finite > 0");
    }
  }
  e = cudaMemcpyAsync(h->in_scale, is.data(), sizeof(float) * is.size(), cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(h, e, "set_act_quant: input_scale upload");
  h->is_host = is;
  h->w4a4 = true;
  return upload_gs_eff(h, st);
}

nvfp4_moe_status nvfp4_moe_debug_poison_workspace(nvfp4_moe_t h, int byte, cudaStream_t st) {
  if (!h) return NVFP4_MOE_ERR_INVALID_ARG;
  if (byte < 0 || byte > 255) return fail(h, NVFP4_MOE_ERR_INVALID_ARG, "debug_poison_workspace: byte out of range");
  DeviceGuard g(h->cfg.device);
  for (const auto& r : h->data_regions) {
    const cudaError_t e = cudaMemsetAsync(r.first, byte, r.second, st);
    if (e != cudaSuccess) return cuda_fail(h, e, "debug_poison_workspace");
  }
  return NVFP4_MOE_OK;
}

nvfp4_moe_status nvfp4_moe_decode_status_word(uint32_t flags) {
  if (flags & kFlagTimeout) return NVFP4_MOE_ERR_TIMEOUT;
  if (flags & kFlagBounds) return NVFP4_MOE_ERR_DEVICE_CHECK;
  return NVFP4_MOE_OK;
}

nvfp4_moe_status nvfp4_moe_debug_set_fault(nvfp4_moe_t h, int fault) {
  if (!h) return NVFP4_MOE_ERR_INVALID_ARG;
  if (fault < 0 || fault > 1) return fail(h, NVFP4_MOE_ERR_INVALID_ARG, "debug_set_fault: unknown fault");
  h->fault = fault;
  return NVFP4_MOE_OK;
}

nvfp4_moe_status nvfp4_moe_pack(nvfp4_moe_t h, const uint8_t* w13_q, const uint8_t* w13_s, const uint8_t* w2_q,
                                const uint8_t* w2_s, const float* gscale, cudaStream_t st) {
  if (!h) return NVFP4_MOE_ERR_INVALID_ARG;
  if (h->linear) return fail(h, NVFP4_MOE_ERR_INVALID_ARG, "a dense-linear handle: call nvfp4_linear_pack");
  if (!w13_q || !w13_s || !w2_q || !w2_s || !gscale) return fail(h, NVFP4_MOE_ERR_INVALID_ARG, "pack: NULL input");
  if (!aligned(w13_q, 16) || !aligned(w2_q, 16) || !aligned(w13_s, 4) || !aligned(w2_s, 4) || !aligned(gscale, 4))
    return fail(h, NVFP4_MOE_ERR_INVALID_ARG, "pack: misaligned input");
  DeviceGuard g(h->cfg.device);
  const int E = h->cfg.num_experts + h->cfg.num_shared_experts;
  std::vector<float> gs((size_t)3 * E);
  cudaError_t e = cudaMemcpyAsync(gs.data(), gscale, sizeof(float) * gs.size(), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(h, e, "pack: reading gscale");
  for (size_t i = 0; i < gs.size(); ++i) {
    const float v = gs[i];
    if (!(v > 0.0f) || v != v || v > 3.4e38f) {
      h->packed = false;
      return fail(h, NVFP4_MOE_ERR_BAD_SCALE,
                  "pack: tensor scale " + std::to_string(i % 3) + " of expert " + std::to_string(i / 3) + " is not finite > 0");
    }
  }
  e = cudaMemcpyAsync(h->gscale, gscale, sizeof(float) * gs.size(), cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess) e = launch_pack(w13_q, w13_s, w2_q, w2_s, h->blob, E, h->cfg.hidden, h->cfg.inter, st);
  if (e == cudaSuccess) e = launch_gateup_bound(w13_q, w13_s, E, h->cfg.hidden, h->cfg.inter, h->hbound, st);
  if (e != cudaSuccess) return cuda_fail(h, e, "pack launch");
  h->gs_host = gs;
  if (h->w4a4) {
    nvfp4_moe_status s2 = upload_gs_eff(h, st);
    if (s2 != NVFP4_MOE_OK) return s2;
  }
  h->packed = true;
  return NVFP4_MOE_OK;
}

}  // extern "C"

namespace {
// One forward.  routed: the logits are computed here from x and the router
// weight (into the workspace) instead of being passed in.
nvfp4_moe_status forward_impl(nvfp4_moe* h, const void* logits, int T, int top_k, const void* x, void* out,
                              cudaStream_t st, bool routed) {
  const int path = choose_path(h, T, top_k);
  nvfp4_moe_status s = check_forward_args(h, routed ? h->ws.logits : logits, T, top_k, path);
  if (s != NVFP4_MOE_OK) return s;
  if (!x || !out) return fail(h, NVFP4_MOE_ERR_INVALID_ARG, "x or out is NULL");
  if (!aligned(x, 16) || !aligned(out, 16)) return fail(h, NVFP4_MOE_ERR_INVALID_ARG, "x or out not 16-byte aligned");
  if (routed && !h->have_router) return fail(h, NVFP4_MOE_ERR_INVALID_ARG, "forward_routed before set_router");
  DeviceGuard g(h->cfg.device);
  CUtensorMap x_map{};
  if (routed && T > kDecodeMaxTokens &&
      !encode_rows_map(&x_map, const_cast<void*>(x), (uint64_t)T, (uint64_t)h->cfg.hidden))
    return fail(h, NVFP4_MOE_ERR_CUDA, "forward_routed: cuTensorMapEncodeTiled failed for x");
  if (h->log && !h->logged_path[path]) {
    h->logged_path[path] = true;
    fprintf(stderr, "[nvfp4_moe] forward T=%d top_k=%d -> %s path\n", T, top_k,
            path == NVFP4_MOE_PATH_DECODE ? "decode (grouped GEMV)" : "prefill (tcgen05 grouped GEMM)");
  }
  cudaEvent_t ev[5] = {nullptr, nullptr, nullptr, nullptr, nullptr};
  s = take_events(h, ev);
  if (s != NVFP4_MOE_OK) return s;
  if (ev[0]) cudaEventRecord(ev[0], st);
  LayerDims d = dims_of(h);
  const float* gsc = h->w4a4 ? h->gs_eff : h->gscale;  // W4A4: input scales folded in
  cudaError_t e;
  // the streaming decode kernel computes the router logits itself (one launch for the layer)
  const bool fused_router = routed && path == NVFP4_MOE_PATH_DECODE && use_stream(h, d, T, top_k);
  if (routed && !fused_router) {  // the router linear, timed with route + permute
    const int Er = h->cfg.num_experts, H = h->cfg.hidden;
    if (T <= kDecodeMaxTokens) {
      e = launch_router_gemv(x, h->w_router, T, Er, H, h->ws.logits, st);
    } else {
      // token tiles small enough to give every SM a unit (16..128 rows)
      int rows = (T + h->num_sms - 1) / h->num_sms;
      rows = std::min(kTileRows, std::max(16, (rows + 15) / 16 * 16));
      e = launch_route_linear(T, rows, h->ws, st);
      if (e == cudaSuccess)
        e = launch_router_gemm(x_map, h->w_router_map, Er, H, h->num_sms, h->ws.ones3, h->ws, h->ws.logits, st);
    }
    if (e != cudaSuccess) return cuda_fail(h, e, "router launch");
  }
  if (routed) {
    logits = h->ws.logits;
    d.logits_bf16 = 0;
  }
  if (path == NVFP4_MOE_PATH_DECODE) {
    // one fused kernel: its time is reported as the gate/up stage
    if (ev[1]) cudaEventRecord(ev[1], st);
    const bool stream = use_stream(h, d, T, top_k);
    e = stream ? launch_decode_stream(d, h->blob, gsc, logits, x, T, top_k, out, 0, h->num_sms, h->ws, h->fault, st,
                                      fused_router ? h->w_router : nullptr)
               : launch_decode_forward(d, h->blob, gsc, logits, x, T, top_k, out, 0, h->num_sms, h->ws, h->fault, st);
    h->last_hsrc = stream ? 1 : 0;
    if (e != cudaSuccess) return cuda_fail(h, e, "decode launch");
    if (ev[2]) cudaEventRecord(ev[2], st);
    if (ev[3]) cudaEventRecord(ev[3], st);
  } else {
    s = run_route(h, logits, x, T, top_k, path, st, d.logits_bf16);
    if (s != NVFP4_MOE_OK) return s;
    if (ev[1]) cudaEventRecord(ev[1], st);
    e = launch_prefill_ffn(d, h->blob, gsc, T, top_k, h->num_sms, h->maps, h->ws, h->fault, ev[2],
                           nullptr, st);
    if (e != cudaSuccess) return cuda_fail(h, e, "expert FFN launch");
    if (ev[3]) cudaEventRecord(ev[3], st);
    e = launch_combine(d, T, top_k, h->ws, out, st);
    if (e != cudaSuccess) return cuda_fail(h, e, "combine launch");
    h->last_hsrc = 2;
  }
  if (ev[4]) cudaEventRecord(ev[4], st);
  h->last_T = T;
  h->last_k = top_k + h->cfg.num_shared_experts;  // routed-row slots per token
  h->last_routed = routed;
  return NVFP4_MOE_OK;
}
}  // namespace

extern "C" {

nvfp4_moe_status nvfp4_moe_forward(nvfp4_moe_t h, const void* logits, int T, int top_k, const void* x, void* out,
                                   cudaStream_t st) {
  if (!h) return NVFP4_MOE_ERR_INVALID_ARG;
  return forward_impl(h, logits, T, top_k, x, out, st, false);
}

}  // extern "C"

namespace {
// The device address of host memory the device may read and write in place: page-locked memory
// that CUDA has mapped into the device's address space (under unified addressing, the same
// pointer).  NULL for pageable, managed or device memory.
const void* mapped_host(const void* p) {
  if (!p) return nullptr;
  cudaPointerAttributes attr{};
  if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  return attr.type == cudaMemoryTypeHost ? attr.devicePointer : nullptr;
}
}  // namespace

extern "C" {

nvfp4_moe_status nvfp4_moe_forward_host(nvfp4_moe_t h, const void* logits, int T, int top_k, const void* x,
                                        void* out, cudaStream_t st) {
  if (!h) return NVFP4_MOE_ERR_INVALID_ARG;
  if (h->linear) return fail(h, NVFP4_MOE_ERR_INVALID_ARG, "forward_host: the handle is a dense linear");
  DeviceGuard g(h->cfg.device);
  // the streaming decode kernel reads logits and x and writes out with plain loads and stores
  // only, so those may live in host memory; the other paths copy x and logits in bulk
  if (choose_path(h, T, top_k) != NVFP4_MOE_PATH_DECODE || !use_stream(h, dims_of(h), T, top_k))
    return fail(h, NVFP4_MOE_ERR_UNSUPPORTED_SHAPE,
                "forward_host: host buffers are read in place by the W4A16 decode kernel only (T <= decode_max_tokens)");
  const void* dl = mapped_host(logits);
  const void* dx = mapped_host(x);
  void* dout = const_cast<void*>(mapped_host(out));
  if (!dl || !dx || !dout)
    return fail(h, NVFP4_MOE_ERR_INVALID_ARG, "forward_host: logits, x and out must be mapped page-locked host memory");
  return forward_impl(h, dl, T, top_k, dx, dout, st, false);
}

nvfp4_moe_status nvfp4_moe_set_router(nvfp4_moe_t h, const void* w_router, cudaStream_t st) {
  if (!h) return NVFP4_MOE_ERR_INVALID_ARG;
  if (h->linear) return fail(h, NVFP4_MOE_ERR_INVALID_ARG, "set_router: a dense linear has no router");
  if (!w_router || !aligned(w_router, 16)) return fail(h, NVFP4_MOE_ERR_INVALID_ARG, "set_router: NULL or misaligned");
  DeviceGuard g(h->cfg.device);
  const size_t n = (size_t)h->cfg.num_experts * h->cfg.hidden * 2;
  if (!h->w_router && cudaMalloc(&h->w_router, n) != cudaSuccess) {
    cudaGetLastError();
    h->w_router = nullptr;
    return fail(h, NVFP4_MOE_ERR_WORKSPACE, "set_router: device allocation failed");
  }
  cudaError_t e = cudaMemcpyAsync(h->w_router, w_router, n, cudaMemcpyDeviceToDevice, st);
  if (e != cudaSuccess) return cuda_fail(h, e, "set_router copy");
  if (!encode_rows_map(&h->w_router_map, h->w_router, (uint64_t)h->cfg.num_experts, (uint64_t)h->cfg.hidden, 128))
    return fail(h, NVFP4_MOE_ERR_CUDA, "set_router: cuTensorMapEncodeTiled failed");
  h->have_router = true;
  return NVFP4_MOE_OK;
}

nvfp4_moe_status nvfp4_moe_forward_routed(nvfp4_moe_t h, int T, int top_k, const void* x, void* out,
                                          cudaStream_t st) {
  if (!h) return NVFP4_MOE_ERR_INVALID_ARG;
  return forward_impl(h, nullptr, T, top_k, x, out, st, true);
}

nvfp4_moe_status nvfp4_moe_debug_logits(nvfp4_moe_t h, float* logits, cudaStream_t st) {
  if (!h) return NVFP4_MOE_ERR_INVALID_ARG;
  if (!h->last_T || !h->last_routed)
    return fail(h, NVFP4_MOE_ERR_INVALID_ARG, "debug_logits: no nvfp4_moe_forward_routed yet");
  if (!logits) return fail(h, NVFP4_MOE_ERR_INVALID_ARG, "debug_logits: NULL output");
  DeviceGuard g(h->cfg.device);
  cudaError_t e = cudaMemcpyAsync(logits, h->ws.logits, (size_t)h->last_T * h->cfg.num_experts * 4,
                                  cudaMemcpyDeviceToDevice, st);
  if (e != cudaSuccess) return cuda_fail(h, e, "debug_logits copy");
  return NVFP4_MOE_OK;
}

nvfp4_moe_status nvfp4_moe_get_status(nvfp4_moe_t h, uint32_t* nan_logits) {
  if (!h) return NVFP4_MOE_ERR_INVALID_ARG;
  DeviceGuard g(h->cfg.device);
  DeviceStatus ds{};
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(&ds, h->ws.status, sizeof(ds), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(h->ws.status, 0, sizeof(ds));
  if (e != cudaSuccess) return cuda_fail(h, e, "get_status");
  if (nan_logits) *nan_logits = ds.nan_logits;
  if (ds.flags & kFlagTimeout)
    return fail(h, NVFP4_MOE_ERR_TIMEOUT, "device wait timed out at site " + std::to_string(ds.where));
  if (ds.flags & kFlagBounds)
    return fail(h, NVFP4_MOE_ERR_DEVICE_CHECK, "device bounds check at site " + std::to_string(ds.where));
  return NVFP4_MOE_OK;
}

nvfp4_moe_status nvfp4_moe_debug_route(nvfp4_moe_t h, const void* logits, int T, int top_k, int32_t* ids,
                                       float* weights, int32_t* offsets, int32_t* perm, cudaStream_t st) {
  if (!h) return NVFP4_MOE_ERR_INVALID_ARG;
  const int path = choose_path(h, T, top_k);
  nvfp4_moe_status s = check_forward_args(h, logits, T, top_k, path);
  if (s != NVFP4_MOE_OK) return s;
  if (!ids || !weights || !offsets || !perm) return fail(h, NVFP4_MOE_ERR_INVALID_ARG, "debug_route: NULL output");
  DeviceGuard g(h->cfg.device);
  s = run_route(h, logits, nullptr, T, top_k, path, st);
  if (s != NVFP4_MOE_OK) return s;
  const size_t n = (size_t)T * (top_k + h->cfg.num_shared_experts);
  cudaError_t e = cudaMemcpyAsync(ids, h->ws.ids, n * 4, cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(weights, h->ws.wts, n * 4, cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(offsets, h->ws.offsets, (h->cfg.num_experts + h->cfg.num_shared_experts + 1) * 4,
                        cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(perm, h->ws.perm, n * 4, cudaMemcpyDeviceToDevice, st);
  if (e != cudaSuccess) return cuda_fail(h, e, "debug_route copy");
  return NVFP4_MOE_OK;
}

nvfp4_moe_status nvfp4_moe_debug_trace(nvfp4_moe_t h, uint64_t* host_dst, size_t n, size_t* n_written) {
  if (!h || !host_dst || !n_written) return NVFP4_MOE_ERR_INVALID_ARG;
  *n_written = 0;
  if (!h->ws.trace) return fail(h, NVFP4_MOE_ERR_INVALID_ARG, "debug_trace: create the handle with NVFP4_MOE_TRACE=1");
  DeviceGuard g(h->cfg.device);
  const size_t total = (size_t)h->num_sms * 16 * 16;
  const size_t m = n < total ? n : total;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(host_dst, h->ws.trace, m * 8, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(h->ws.trace, 0, total * 8);
  if (e != cudaSuccess) return cuda_fail(h, e, "debug_trace");
  *n_written = m;
  return NVFP4_MOE_OK;
}

nvfp4_moe_status nvfp4_moe_debug_packed_blob(nvfp4_moe_t h, void* dst, size_t dst_bytes, cudaStream_t st) {
  if (!h) return NVFP4_MOE_ERR_INVALID_ARG;
  if (!h->packed) return fail(h, NVFP4_MOE_ERR_NOT_PACKED, "debug_packed_blob before pack");
  const size_t n = blob_bytes_of(h->cfg, h->linear);
  if (!dst || dst_bytes < n) return fail(h, NVFP4_MOE_ERR_INVALID_ARG, "debug_packed_blob: destination too small");
  DeviceGuard g(h->cfg.device);
  cudaError_t e = cudaMemcpyAsync(dst, h->blob, n, cudaMemcpyDeviceToDevice, st);
  if (e != cudaSuccess) return cuda_fail(h, e, "debug_packed_blob copy");
  return NVFP4_MOE_OK;
}

nvfp4_moe_status nvfp4_moe_debug_dequant(nvfp4_moe_t h, int expert, int which, float* w_out, cudaStream_t st) {
  if (!h) return NVFP4_MOE_ERR_INVALID_ARG;
  if (h->linear) return fail(h, NVFP4_MOE_ERR_NOT_IMPLEMENTED, "debug_dequant: not for a dense-linear handle");
  if (!h->packed) return fail(h, NVFP4_MOE_ERR_NOT_PACKED, "debug_dequant before pack");
  const int base = which & 3, via_bf16 = (which >> 2) & 1;
  if (expert < 0 || expert >= h->cfg.num_experts + h->cfg.num_shared_experts || base > 2 || (which & ~7) || !w_out)
    return fail(h, NVFP4_MOE_ERR_INVALID_ARG, "debug_dequant: bad expert/which/out");
  DeviceGuard g(h->cfg.device);
  cudaError_t e = launch_debug_dequant(h->blob, h->gscale, h->cfg.hidden, h->cfg.inter, expert, base, via_bf16, w_out, st);
  if (e != cudaSuccess) return cuda_fail(h, e, "debug_dequant launch");
  return NVFP4_MOE_OK;
}

nvfp4_moe_status nvfp4_moe_debug_intermediates(nvfp4_moe_t h, void* hidden, float* y, cudaStream_t st) {
  if (!h) return NVFP4_MOE_ERR_INVALID_ARG;
  if (h->linear) return fail(h, NVFP4_MOE_ERR_INVALID_ARG, "debug_intermediates: a dense linear has none");
  if (!h->last_T) return fail(h, NVFP4_MOE_ERR_INVALID_ARG, "debug_intermediates before any forward");
  if (!hidden || !y) return fail(h, NVFP4_MOE_ERR_INVALID_ARG, "debug_intermediates: NULL output");
  DeviceGuard g(h->cfg.device);
  const size_t n = (size_t)h->last_T * h->last_k;
  cudaError_t e = launch_hidden_to_f32(h->ws, h->last_hsrc, (int)n, h->cfg.inter, static_cast<float*>(hidden), st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(y, h->ws.y, n * h->cfg.hidden * 4, cudaMemcpyDeviceToDevice, st);
  if (e != cudaSuccess) return cuda_fail(h, e, "debug_intermediates copy");
  return NVFP4_MOE_OK;
}

// ---------------------------------------------------------------------------
// Dense W4A16 NVFP4 linear: one matrix, every token, no routing.
// ---------------------------------------------------------------------------
nvfp4_moe_status nvfp4_linear_create(const nvfp4_linear_config* c, nvfp4_moe_t* out) {
  if (!out) return NVFP4_MOE_ERR_INVALID_ARG;
  *out = nullptr;
  if (!c) return NVFP4_MOE_ERR_INVALID_ARG;
  if (c->out_features < 16 || c->out_features > 16384 || c->out_features % 16) return NVFP4_MOE_ERR_UNSUPPORTED_SHAPE;
  if (c->in_features < 128 || c->in_features > 16384 || c->in_features % 128) return NVFP4_MOE_ERR_UNSUPPORTED_SHAPE;
  if (c->max_tokens < 1 || c->max_tokens > (1 << 20)) return NVFP4_MOE_ERR_UNSUPPORTED_SHAPE;
  if (c->decode_max_tokens < 0 || c->decode_max_tokens > kDecodeMaxTokens) return NVFP4_MOE_ERR_UNSUPPORTED_SHAPE;
  if (c->out_dtype != NVFP4_MOE_OUT_BF16 && c->out_dtype != NVFP4_MOE_OUT_F32) return NVFP4_MOE_ERR_INVALID_ARG;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || c->device < 0 || c->device >= ndev) return NVFP4_MOE_ERR_INVALID_ARG;
  nvfp4_moe_config m{};
  m.num_experts = 1;
  m.hidden = (c->out_features + 127) / 128 * 128;  // whole 128-row blocks; the padding rows are zero
  m.inter = c->in_features;
  m.max_tokens = c->max_tokens;
  m.max_top_k = 1;
  m.decode_max_tokens = c->decode_max_tokens;
  m.logits_dtype = NVFP4_MOE_LOGITS_F32;
  m.out_dtype = c->out_dtype;
  m.device = c->device;
  m.num_shared_experts = 0;
  return create_handle(&m, true, c->out_features, out);
}

nvfp4_moe_status nvfp4_linear_pack(nvfp4_moe_t h, const uint8_t* w_q, const uint8_t* w_s, const float* gscale,
                                   cudaStream_t st) {
  if (!h) return NVFP4_MOE_ERR_INVALID_ARG;
  if (!h->linear) return fail(h, NVFP4_MOE_ERR_INVALID_ARG, "not a dense-linear handle: call nvfp4_moe_pack");
  if (!w_q || !w_s || !gscale) return fail(h, NVFP4_MOE_ERR_INVALID_ARG, "linear_pack: NULL input");
  if (!aligned(w_q, 16) || !aligned(w_s, 4) || !aligned(gscale, 4))
    return fail(h, NVFP4_MOE_ERR_INVALID_ARG, "linear_pack: misaligned input");
  DeviceGuard g(h->cfg.device);
  float gs = 0.f;
  cudaError_t e = cudaMemcpyAsync(&gs, gscale, sizeof(float), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(h, e, "linear_pack: reading gscale");
  if (!(gs > 0.0f) || gs != gs || gs > 3.4e38f) {
    h->packed = false;
    return fail(h, NVFP4_MOE_ERR_BAD_SCALE, "linear_pack: the tensor scale is not finite > 0");
  }
  // the kernels read the down-projection scale of "expert" 0: slot 2 of 3
  const float gs3[3] = {gs, gs, gs};
  e = cudaMemcpyAsync(h->gscale, gs3, sizeof(gs3), cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = launch_pack_linear(w_q, w_s, h->blob, h->lin_n, h->cfg.hidden, h->cfg.inter, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);  // gs3 lives on this frame
  if (e != cudaSuccess) return cuda_fail(h, e, "linear_pack launch");
  h->packed = true;
  return NVFP4_MOE_OK;
}

nvfp4_moe_status nvfp4_linear_forward(nvfp4_moe_t h, int T, const void* x, void* out, cudaStream_t st) {
  if (!h) return NVFP4_MOE_ERR_INVALID_ARG;
  if (!h->linear) return fail(h, NVFP4_MOE_ERR_INVALID_ARG, "not a dense-linear handle: call nvfp4_moe_forward");
  if (!h->packed) return fail(h, NVFP4_MOE_ERR_NOT_PACKED, "linear_forward before a successful pack");
  if (T < 1 || T > h->cfg.max_tokens) return fail(h, NVFP4_MOE_ERR_UNSUPPORTED_SHAPE, "T outside 1..max_tokens");
  if (!x || !out) return fail(h, NVFP4_MOE_ERR_INVALID_ARG, "x or out is NULL");
  if (!aligned(x, 16) || !aligned(out, 16)) return fail(h, NVFP4_MOE_ERR_INVALID_ARG, "x or out not 16-byte aligned");
  const int path = choose_path(h, T, 1);
  if (path == NVFP4_MOE_PATH_DECODE && T > kDecodeMaxTokens)
    return fail(h, NVFP4_MOE_ERR_UNSUPPORTED_SHAPE, "decode path takes at most 16 tokens");
  DeviceGuard g(h->cfg.device);
  PrefillMaps maps{};
  if (path == NVFP4_MOE_PATH_PREFILL && !encode_rows_map(&maps.h, const_cast<void*>(x), (uint64_t)T, h->cfg.inter))
    return fail(h, NVFP4_MOE_ERR_CUDA, "linear_forward: cuTensorMapEncodeTiled failed for x");
  if (h->log && !h->logged_path[path]) {
    h->logged_path[path] = true;
    fprintf(stderr, "[nvfp4_moe] linear forward T=%d -> %s path\n", T,
            path == NVFP4_MOE_PATH_DECODE ? "decode (GEMV)" : "prefill (tcgen05 GEMM)");
  }
  cudaEvent_t ev[5] = {nullptr, nullptr, nullptr, nullptr, nullptr};
  nvfp4_moe_status s = take_events(h, ev);
  if (s != NVFP4_MOE_OK) return s;
  if (ev[0]) cudaEventRecord(ev[0], st);
  const LayerDims d = dims_of(h);
  cudaError_t e;
  if (path == NVFP4_MOE_PATH_DECODE) {
    if (ev[1]) cudaEventRecord(ev[1], st);
    if (ev[2]) cudaEventRecord(ev[2], st);
    e = stream_supported(d, T, 1)
            ? launch_decode_stream(d, h->blob, h->gscale, nullptr, x, T, 1, out, 0, h->num_sms, h->ws, h->fault, st)
            : launch_decode_forward(d, h->blob, h->gscale, nullptr, x, T, 1, out, 0, h->num_sms, h->ws, h->fault, st);
    if (e != cudaSuccess) return cuda_fail(h, e, "linear decode launch");
  } else {
    e = launch_route_linear(T, kTileRows, h->ws, st);
    if (e != cudaSuccess) return cuda_fail(h, e, "linear tables launch");
    if (ev[1]) cudaEventRecord(ev[1], st);
    e = launch_prefill_ffn(d, h->blob, h->gscale, T, 1, h->num_sms, maps, h->ws, h->fault, ev[2], out, st);
    if (e != cudaSuccess) return cuda_fail(h, e, "linear GEMM launch");
  }
  if (ev[3]) cudaEventRecord(ev[3], st);
  if (ev[4]) cudaEventRecord(ev[4], st);
  h->last_T = T;
  h->last_k = 1;
  h->last_routed = false;
  return NVFP4_MOE_OK;
}

}  // extern "C"
