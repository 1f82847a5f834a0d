// noalloc.cu -- fp4gemv_moe_down_combine_noalloc: down_combine without a
// caller-provided workspace.
//
// Some callers cannot allocate device memory when they call this library:
// a serving process whose device memory is planned and handed out once at
// start-up (allocating on the request path would break that budget, and
// cudaMalloc can synchronize the device), or a plug-in that only receives
// the tensors it works on and owns no allocator.  This entry point needs no
// allocation at all: its scratch is a file-scope device array of fixed size
// that lives as long as the library is loaded on a device.
//
// The array's name is only a host-side stand-in in host code, so the device
// address is obtained once per device with cudaGetSymbolAddress (with that
// device current) and handed to the existing down_combine entry point as its
// workspace.  Every call shares the array; its contents carry nothing from
// one call to the next (the arrival counters are tagged per call), but calls
// that overlap on the GPU race on it.
#include <atomic>

#include "fp4gemv.h"

namespace {

constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[FP4GEMV_NOALLOC_SCRATCH_BYTES];

std::atomic<void*> g_scratch_addr[kMaxDevices];

// Device address of g_noalloc_scratch on the current device (set up on the
// first call per device).
fp4gemv_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FP4GEMV_ERR_CUDA;
  void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (!p) {
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return FP4GEMV_ERR_CUDA;
    g_scratch_addr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return FP4GEMV_OK;
}

}  // namespace

extern "C" fp4gemv_status fp4gemv_moe_down_combine_noalloc(
    const void* act, const int32_t* ids, const float* tw, int M, int topk, const uint8_t* w2, const uint8_t* w2_sf,
    const float* alpha2, int E, int H, int I, const void* sact, const uint8_t* wsd, const uint8_t* ssd,
    const float* gssd, int SI, void* out, int pdl, cudaStream_t stream) {
  if (M < 1 || topk < 1 || H < 1) return FP4GEMV_ERR_INVALID_ARG;
  const size_t need = fp4gemv_moe_down_combine_workspace_bytes(M, topk, H);
  if (need == 0) return FP4GEMV_ERR_INVALID_ARG;
  if (need > static_cast<size_t>(FP4GEMV_NOALLOC_SCRATCH_BYTES)) return FP4GEMV_ERR_UNSUPPORTED_SHAPE;
  void* scratch = nullptr;
  const fp4gemv_status st = scratch_address(&scratch);
  if (st != FP4GEMV_OK) return st;
  return fp4gemv_moe_down_combine(act, ids, tw, M, topk, w2, w2_sf, alpha2, E, H, I, sact, wsd, ssd, gssd, SI, out,
                                  scratch, FP4GEMV_NOALLOC_SCRATCH_BYTES, pdl, stream);
}
