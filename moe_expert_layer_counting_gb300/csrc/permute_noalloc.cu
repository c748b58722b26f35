// permute_noalloc.cu -- moe_permute for callers that cannot allocate device memory.
//
// Some callers have no way to obtain a workspace: plugins running inside a
// host framework that owns every device allocation, or serving loops that
// must not call cudaMalloc once they are running (it can synchronise the
// device and it eats into a fixed memory budget).  This entry point runs the
// same two permute kernels as moe_permute, but their scratch (the status
// words and the per-block expert histogram) lives in a file-scope device
// array that the library carries, so the caller passes only inputs and
// outputs and nothing is allocated.
//
// The array is 256 bytes of status words plus kHistBytes (64 KiB) of
// histogram: every GPU that loads the library holds it until the process
// exits.  Problems whose histogram does not fit (blocks x experts x 4 bytes
// above 64 KiB, e.g. E = 1024 with more than 32768 pairs) are rejected with
// MOE_ERR_UNSUPPORTED_SHAPE.  All calls on a device share the one array and
// it keeps the last call's contents, so calls that overlap on the GPU (on
// different streams without ordering) race with each other.
#include <mutex>

#include "host_common.h"

namespace mxq {

namespace {

constexpr size_t kHistBytes = 64 * 1024;
constexpr int kMaxDevices = 64;

// Status words [0, 256) then the histogram.  Host code must not use this name
// as an address: it is a host-side stand-in; the device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_permute_scratch[kStatusBytes + kHistBytes];

std::mutex g_setup_mutex;
struct CachedAddress {
  unsigned long long ctx_id;   // context the address belongs to (0: none yet)
  void *ptr;
};
CachedAddress g_scratch[kMaxDevices] = {};

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);

// Id of the current context, or 0 if the driver does not report one.  A
// device reset (cudaDeviceReset, or a framework that resets the device)
// replaces the context, and with it the array's device address.
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Looks up the device address of the scratch array with the device current:
// once per device and context (again after a reset replaced the context;
// on every call while the driver reports no context id, e.g. before the
// runtime created the device's context, which the lookup itself does).  Returns nullptr if the
// lookup fails.
void *scratch_for_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  CachedAddress &c = g_scratch[dev];
  if (ctx == 0 || c.ctx_id != ctx || !c.ptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_permute_scratch) != cudaSuccess || !p) return nullptr;
    c.ctx_id = ctx;
    c.ptr = p;
  }
  return c.ptr;
}

}  // namespace

}  // namespace mxq

using namespace mxq;

extern "C" int moe_permute_noalloc(const int32_t *topk_idx, int64_t T, int32_t E, int32_t k, int32_t *counts,
                                   int32_t *offsets, int32_t *perm, int32_t *inv_perm, int32_t *device_status,
                                   cudaStream_t stream) {
  if (T < 0 || E <= 0 || k <= 0) return MOE_ERR_INVALID_ARG;
  if (E > 1024 || k > E || k > 32 || T * (int64_t)k >= ((int64_t)1 << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!topk_idx || !perm || !inv_perm)) return MOE_ERR_INVALID_ARG;
  if (permute_scratch_bytes(T, E, k) > kHistBytes) return MOE_ERR_UNSUPPORTED_SHAPE;
  char *scratch = reinterpret_cast<char *>(scratch_for_current_device());
  if (!scratch) return MOE_ERR_CUDA;
  // the status words must start at zero: the kernels only ever raise them
  if (cudaMemsetAsync(scratch, 0, 32, stream) != cudaSuccess) return MOE_ERR_CUDA;
  int *status = reinterpret_cast<int *>(scratch);
  if (device_status) {
    if (cudaMemsetAsync(device_status, 0, sizeof(int32_t), stream) != cudaSuccess) return MOE_ERR_CUDA;
    status = device_status;
  }
  return launch_permute(topk_idx, T, E, k, counts, offsets, perm, inv_perm, status, scratch + kStatusBytes,
                        stream);
}
