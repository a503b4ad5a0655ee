// moe_route_noalloc: the router and top-k selection for callers that cannot allocate device
// memory.
//
// Some callers of this library cannot call cudaMalloc: a host runtime that owns every byte of
// device memory through its own pool and forbids side allocations, or a latency-critical
// serving loop in which an allocation (which may synchronise the device) is not allowed.
// moe_route needs a caller-provided workspace for the fp32 logits; this variant keeps that
// scratch in a fixed array compiled into the library instead, so the caller passes only its
// inputs and outputs.
//
// The array lives in device memory of every GPU that loads the library, for the life of the
// process (kNoAllocBytes below).  Every call on a device uses the same array, so calls whose
// work overlaps on the GPU (two streams, or two host threads) overwrite each other's logits:
// serialise them.  The array keeps whatever the previous call left; the part that must start
// at zero (the status record) is cleared by each call, the logits are fully rewritten.  Free
// routing has no forced ids and the SIMT router kernels used here have no device-side waits,
// so no device-side error can arise: the status record is never read back.
#include <cuda.h>

#include <mutex>

#include "common.cuh"

namespace {

constexpr size_t kNoAllocStatusBytes = sizeof(moe::DevStatus);
constexpr size_t kNoAllocMaxLogits = size_t(1) << 20;  // limit on T * n_experts
constexpr size_t kNoAllocBytes = kNoAllocStatusBytes + kNoAllocMaxLogits * sizeof(float);  // 4 MiB + 768 B
static_assert(kNoAllocStatusBytes % 256 == 0, "the logits start 256-byte aligned");

// The scratch: status record, then T x n_experts fp32 logits.
static __device__ __align__(256) unsigned char g_route_scratch[kNoAllocBytes];

// Device address of g_route_scratch per device, looked up at set-up with that device current
// and kept with the identity of the CUDA context it was taken in.  In host code the symbol is
// only a host-side stand-in, never a device address.  The library's module is loaded once per
// context, so after a device reset (or under another context on the same device) the array
// sits at a new address: a call that finds a different current context looks it up again.
constexpr int kMaxDevices = 128;
struct ScratchAddr {
  unsigned long long ctx_id;
  void* addr;
};
std::mutex g_scratch_mu;
ScratchAddr g_scratch_addr[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// The current context's process-unique id (0 if the driver cannot say).
cudaError_t current_context_id(unsigned long long* id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  *id = 0;
  if (!get_current || !get_id) return cudaSuccess;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS) return cudaErrorUnknown;
  if (!ctx) {  // no context current yet on this thread: make the device's primary context current
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaSetDevice(dev);
    if (e != cudaSuccess) return e;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return cudaErrorUnknown;
  }
  return get_id(ctx, id) == CUDA_SUCCESS ? cudaSuccess : cudaErrorUnknown;
}

cudaError_t scratch_on_current_device(char** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  unsigned long long ctx_id = 0;
  e = current_context_id(&ctx_id);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  ScratchAddr& slot = g_scratch_addr[dev];
  // without a context id (old driver) the address is looked up on every call
  if (!slot.addr || ctx_id == 0 || slot.ctx_id != ctx_id) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_route_scratch);
    if (e != cudaSuccess) return e;
    slot.addr = p;
    slot.ctx_id = ctx_id;
  }
  *out = static_cast<char*>(slot.addr);
  return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" moe_status moe_route_noalloc(const void* x, moe_dtype x_dtype, int T, const moe_layer* layer, int k,
                                        int32_t* ids_out, float* w_out, moe_stream_t stream) {
  if (!layer) return MOE_ERR_INVALID_ARG;
  if (layer->top_k != moe::kTopK || k != layer->top_k) return MOE_ERR_UNSUPPORTED;
  if (layer->n_experts < moe::kTopK || layer->n_experts > moe::kMaxExperts) return MOE_ERR_INVALID_ARG;
  if (layer->d_model <= 0 || layer->d_model % 128 != 0) return MOE_ERR_UNSUPPORTED;
  if (!layer->w_router || !aligned16(layer->w_router)) return MOE_ERR_INVALID_ARG;
  if (layer->bias_mode != MOE_BIAS_SCORE && layer->bias_mode != MOE_BIAS_SELECT) return MOE_ERR_INVALID_ARG;
  if (T < 0) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (size_t(T) * size_t(layer->n_experts) > kNoAllocMaxLogits) return MOE_ERR_WORKSPACE;
  if (!x || !ids_out || !w_out || !aligned16(x)) return MOE_ERR_INVALID_ARG;
  if (x_dtype != MOE_F32 && x_dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;

  char* scratch = nullptr;
  if (scratch_on_current_device(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  moe::DevStatus* st = reinterpret_cast<moe::DevStatus*>(scratch);
  float* logits = reinterpret_cast<float*>(scratch + kNoAllocStatusBytes);

  moe::LayerDev L{};
  L.d = layer->d_model;
  L.F = layer->ffn;
  L.E = layer->n_experts;
  L.k = layer->top_k;
  L.fp8 = layer->w_dtype == MOE_E4M3 || layer->w_dtype == MOE_E2M1;
  L.w4 = layer->w_dtype == MOE_E2M1;
  L.Wr = layer->w_router;
  L.bias = layer->router_bias;
  L.bias_sel = layer->bias_mode == MOE_BIAS_SELECT && layer->router_bias != nullptr;

  if (cudaMemsetAsync(st, 0, kNoAllocStatusBytes, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (moe::launch_router_logits(x, x_dtype == MOE_BF16, T, L, logits, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (moe::launch_select(logits, nullptr, nullptr, T, L, ids_out, w_out, st, s) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}
