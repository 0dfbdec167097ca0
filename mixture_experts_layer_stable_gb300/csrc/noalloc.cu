// noalloc.cu -- moe_schedule_noalloc: the routing + schedule-table call for
// callers that cannot allocate device memory and cannot hand the library a
// workspace.  Its scratch lives in a fixed-size array in the library's own
// device data, so the call needs nothing beyond its inputs and outputs.
#include <mutex>

#include "moe_internal.h"

namespace moe {

namespace {

// Scratch of the schedule kernels (status/ticket words, per-block histograms,
// padded offsets, row positions).  Every GPU that loads the library holds it
// until the process exits.
constexpr size_t kNoAllocScratchBytes = 1536u * 1024u;
static __device__ __align__(256) unsigned char g_sched_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};
unsigned long long g_scratch_ctx[kMaxDevices] = {0};  // context id the address belongs to

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current CUDA context (ids are never
// reused within a process, unlike context handles), or 0 if unknown.
unsigned long long current_ctx_id() {
  static CtxGetCurrentFn get_cur = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static bool looked = false;
  if (!looked) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_cur = reinterpret_cast<CtxGetCurrentFn>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
    looked = true;
  }
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_cur == nullptr || get_id == nullptr || get_cur(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of g_sched_scratch on the current device, looked up with
// that device current and cached per device for as long as the device's
// context stays the same (a device reset or a new primary context loads the
// module again, and the array may then sit elsewhere).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  const unsigned long long id = current_ctx_id();  // 0 before the first runtime call made one
  if (g_scratch_ptr[dev] == nullptr || id == 0 || id != g_scratch_ctx[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_sched_scratch);  // makes the device's context current
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
    g_scratch_ctx[dev] = current_ctx_id();
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

}  // namespace moe

using namespace moe;

static bool ok_ptr(const void* p) {
  return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 127) == 0;
}

extern "C" moe_status moe_schedule_noalloc(const moe_config* cfg, const float* logits,
                                           moe_sched sched, moe_stream_t stream) {
  if (!config_valid(cfg) || !ok_ptr(logits) || !ok_ptr(sched.topk_ids) ||
      !ok_ptr(sched.topk_w) || !ok_ptr(sched.counts) || !ok_ptr(sched.offsets) ||
      !ok_ptr(sched.perm) || !ok_ptr(sched.inv))
    return MOE_ERR_INVALID_ARG;
  Ws w;
  w.L = ws_layout(cfg);
  // the schedule kernels use the layout up to the first FFN buffer
  if (w.L.Xp > kNoAllocScratchBytes) return MOE_ERR_INVALID_ARG;
  void* base = nullptr;
  if (scratch_address(&base) != cudaSuccess) return MOE_ERR_CUDA;
  w.base = static_cast<uint8_t*>(base);
  const cudaError_t e =
      launch_schedule(*cfg, logits, sched, w, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
