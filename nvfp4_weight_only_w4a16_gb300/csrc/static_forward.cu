// Allocation-free decode forward.
//
// Some callers cannot call cudaMalloc: code that runs while a CUDA graph is
// being captured in global mode, plugins whose host framework owns every
// device byte (a serving engine with its own memory pool and allocation
// budget), and static-memory runtimes that allocate everything once at start
// and forbid allocation afterwards.  They cannot create a handle, because
// nvfp4_moe_create allocates the weight blob and the workspace.  This entry
// point runs the decode path (the streaming decode kernel: route, gate/up,
// down, combine, in one launch) with the caller's own weight blob, activations
// and output; every intermediate (routing tables, x and h rows, y, counters)
// lives in one file-scope __device__ array of kStaticScratchBytes.
//
// Consequences a caller must know:
//  * every GPU that loads this library reserves the array until the process
//    exits, whether or not this entry point is ever called;
//  * on each device, the first call looks up the array's device address
//    (cudaGetSymbolAddress) with that device current; make that first call
//    before any stream capture;
//  * all calls on a device share the array: calls whose work overlaps on the
//    GPU (different streams, or graphs replayed concurrently) race and give
//    wrong results; serialise them;
//  * the array keeps the last call's contents; the regions that must start at
//    zero are cleared (cudaMemsetAsync) by every call;
//  * device-side errors (a bounded wait that gave up, NaN router logits) of
//    every call are carried into a status word at the start of the array,
//    which no call clears: nvfp4_moe_static_get_status reads and clears it.
#include <algorithm>
#include <atomic>
#include <mutex>
#include <string>

#include "../../include/nvfp4_moe.h"
#include "kernels.h"

namespace nvfp4moe {

constexpr size_t kStaticScratchBytes = 16u << 20;  // 16 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

namespace {

struct StaticSetup {
  uint8_t* scratch = nullptr;  // device address of g_static_scratch on this device
  int num_sms = 0;
};

std::mutex g_setup_mutex;
StaticSetup g_setup[kMaxDevices];
std::atomic<int> g_fault{0};  // test hook: 1 makes the next calls issue no weight copies

// Once per device, with that device current: the array's device address, the
// SM count and the decode kernels' shared-memory attribute.
cudaError_t static_setup(int dev, StaticSetup* out) {
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_setup[dev].scratch) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return e;
    int sms = 0, smem = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = decode_prepare_device(dev, &smem);
    if (e == cudaSuccess) e = stream_prepare_device(dev, &smem);
    if (e != cudaSuccess) return e;
    g_setup[dev].scratch = static_cast<uint8_t*>(p);
    g_setup[dev].num_sms = sms;
  }
  *out = g_setup[dev];
  return cudaSuccess;
}

struct Region {
  size_t off = 0;
  template <class T>
  T* take(uint8_t* base, size_t count) {
    off = (off + 255) & ~size_t(255);
    T* p = reinterpret_cast<T*>(base + off);
    off += count * sizeof(T);
    return p;
  }
};

// The status word that outlives each call, at the start of the array.
constexpr size_t kStickyBytes = 256;

// Carves the decode workspace out of `base`; returns the bytes it needs.
// With base == nullptr only the size is computed.  [0, kStickyBytes) holds the
// status word carried across calls; the regions every call zeroes (counters,
// the call's own status) follow contiguously: [kStickyBytes, *zero_end).
size_t carve(uint8_t* base, int E, int H, int I, int T, int k, int num_sms, Workspace* ws, size_t* zero_end) {
  const size_t R = (size_t)T * k;
  const size_t maxU = std::min<size_t>((size_t)E, R);
  uint8_t* b = base ? base : reinterpret_cast<uint8_t*>(0x100);
  Region r;
  Workspace w{};
  w.status_sticky = r.take<DeviceStatus>(b, 1);
  r.off = kStickyBytes;
  w.cnt_gu = r.take<int32_t>(b, maxU * (2 * I / 16));
  w.cnt_dn = r.take<int32_t>(b, maxU * (H / 16));
  w.done_gu = r.take<int32_t>(b, maxU);
  w.cmb = r.take<int32_t>(b, H / 64);
  w.exit_cnt = r.take<int32_t>(b, 1);
  w.hmax = r.take<uint32_t>(b, R);
  w.wctr = r.take<int32_t>(b, 1);
  w.done_c = r.take<int32_t>(b, maxU * (I / 64));
  w.x_ready = r.take<int32_t>(b, H / 64);
  w.logit_ready = r.take<int32_t>(b, 1);
  w.status = r.take<DeviceStatus>(b, 1);
  *zero_end = (r.off + 255) & ~size_t(255);
  // no split-K partial-sum buffers here: with part_gu == nullptr the earlier
  // decode kernel (the fallback for shapes the streaming kernel does not take)
  // gives every warp whole blocks
  w.part_gu = nullptr;
  w.part_dn = nullptr;
  (void)num_sms;
  w.ids = r.take<int32_t>(b, R);
  w.wts = r.take<float>(b, R);
  w.offsets = r.take<int32_t>(b, E + 1);
  w.perm = r.take<int32_t>(b, R);
  w.inv = r.take<int32_t>(b, R);
  w.tch_expert = r.take<int32_t>(b, E);
  w.tch_row0 = r.take<int32_t>(b, E);
  w.tch_rows = r.take<int32_t>(b, E);
  w.num_touched = r.take<int32_t>(b, 1);
  w.x16 = r.take<__half>(b, (size_t)T * H);
  w.xexp = r.take<int32_t>(b, T);
  w.h = r.take<__nv_bfloat16>(b, R * I);
  w.y = r.take<float>(b, R * H);
  w.act_rows = (int)R;
  w.act_h = r.take<uint8_t>(b, stream_act_h_bytes(I, (int)R));
  w.act_x = r.take<uint8_t>(b, stream_act_x_bytes(H));
  if (base && ws) *ws = w;
  return r.off;
}

bool aligned_to(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace
}  // namespace nvfp4moe

using namespace nvfp4moe;

extern "C" nvfp4_moe_status nvfp4_moe_forward_decode_static(const uint8_t* packed_experts, const float* gscale,
                                                            int num_experts, int hidden, int inter,
                                                            const void* router_logits, int logits_dtype, int T,
                                                            int top_k, const void* x, void* out,
                                                            cudaStream_t stream) {
  const int E = num_experts, H = hidden, I = inter;
  if (E < 1 || E > 256 || H < 128 || H > 16384 || H % 128 || I < 128 || I > 16384 || I % 128)
    return NVFP4_MOE_ERR_UNSUPPORTED_SHAPE;
  if (T < 1 || T > kDecodeMaxTokens || top_k < 1 || top_k > 16 || top_k > E) return NVFP4_MOE_ERR_UNSUPPORTED_SHAPE;
  if (logits_dtype != NVFP4_MOE_LOGITS_F32 && logits_dtype != NVFP4_MOE_LOGITS_BF16) return NVFP4_MOE_ERR_INVALID_ARG;
  if (!packed_experts || !gscale || !router_logits || !x || !out) return NVFP4_MOE_ERR_INVALID_ARG;
  if (!aligned_to(packed_experts, 16) || !aligned_to(x, 16) || !aligned_to(out, 16) || !aligned_to(gscale, 4) ||
      !aligned_to(router_logits, logits_dtype == NVFP4_MOE_LOGITS_BF16 ? 2 : 4))
    return NVFP4_MOE_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return NVFP4_MOE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return NVFP4_MOE_ERR_INVALID_ARG;  // device ordinals 0..63 only
  StaticSetup setup;
  if (static_setup(dev, &setup) != cudaSuccess) return NVFP4_MOE_ERR_CUDA;
  size_t zero_end = 0;
  if (carve(nullptr, E, H, I, T, top_k, setup.num_sms, nullptr, &zero_end) > kStaticScratchBytes)
    return NVFP4_MOE_ERR_UNSUPPORTED_SHAPE;  // needs more than the static scratch holds

  Workspace ws{};
  carve(setup.scratch, E, H, I, T, top_k, setup.num_sms, &ws, &zero_end);
  const LayerDims d{E, H, I, logits_dtype == NVFP4_MOE_LOGITS_BF16, 0, E, 0, 0, 0};
  cudaError_t e = cudaMemsetAsync(setup.scratch + kStickyBytes, 0, zero_end - kStickyBytes, stream);
  if (e == cudaSuccess)
    e = stream_supported(d, T, top_k)
            ? launch_decode_stream(d, packed_experts, gscale, router_logits, x, T, top_k, out, 0, setup.num_sms, ws,
                                   g_fault.load(), stream)
            : launch_decode_forward(d, packed_experts, gscale, router_logits, x, T, top_k, out, 0, setup.num_sms, ws,
                                    g_fault.load(), stream);
  return e == cudaSuccess ? NVFP4_MOE_OK : NVFP4_MOE_ERR_CUDA;
}

extern "C" nvfp4_moe_status nvfp4_moe_static_get_status(uint32_t* nan_logits) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return NVFP4_MOE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return NVFP4_MOE_ERR_INVALID_ARG;
  StaticSetup setup;
  if (static_setup(dev, &setup) != cudaSuccess) return NVFP4_MOE_ERR_CUDA;
  DeviceStatus ds{};
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(&ds, setup.scratch, sizeof(ds), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(setup.scratch, 0, sizeof(ds));
  if (e != cudaSuccess) return NVFP4_MOE_ERR_CUDA;
  if (nan_logits) *nan_logits = ds.nan_logits;
  return nvfp4_moe_decode_status_word(ds.flags);
}

extern "C" nvfp4_moe_status nvfp4_moe_static_debug_set_fault(int fault) {
  if (fault < 0 || fault > 1) return NVFP4_MOE_ERR_INVALID_ARG;
  g_fault.store(fault);
  return NVFP4_MOE_OK;
}
