// gdn_frame_fwd_noalloc: the forward scan for callers that cannot allocate
// device memory.
//
// It runs the split form (the kernels that use scratch), but its scratch is a
// fixed array in the library's own device memory instead of memory taken from
// an allocator.  It exists for callers that cannot call cudaMalloc: code
// plugged into another runtime that owns the device memory (its caching
// allocator has reserved the HBM, so a raw cudaMalloc fails or fragments the
// pool), and latency-critical loops in which an allocation or free that
// synchronises the device would stall unrelated streams.
//
// The array lives in this translation unit alone, so it is a module of its own:
// with CUDA's lazy module loading (the default) a device only reserves its
// 64 MiB when this entry point is first called there, not when the library's
// other entry points are.
#include "../../include/gdn.h"
#include "gdn_internal.h"

namespace gdn {
namespace {

// Every GPU on which this entry point has been called holds this array until
// the process exits.
constexpr size_t kStaticScratchBytes = size_t(64) << 20;  // 64 MiB
__device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Device address of g_static_scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up with
// cudaGetSymbolAddress once per device (and context), with that device
// current, and cached.
void* static_scratch_address() {
  static SymbolAddressCache cache;
  return cache.get(reinterpret_cast<const void*>(&g_static_scratch));
}

}  // namespace
}  // namespace gdn

extern "C" int gdn_frame_fwd_noalloc(const void* q, const void* k, const void* v, const float* g,
                                     const float* beta, const float* state_in, void* out, float* state_out, int B,
                                     int H, int T, int S, int D, int dtype, void* stream) {
  gdn::Problem p{};
  int rc = gdn::check_args(q, k, v, g, beta, state_in, out, state_out, B, H, T, S, D, dtype, GDN_MODE_SPLIT, &p);
  if (rc != gdn::kOk) return rc;
  // Every stage writes its scratch before reading it, so the previous call's
  // contents never need clearing.
  const size_t need = gdn::scratch_bytes(p);
  if (need > gdn::kStaticScratchBytes) return GDN_ERR_WORKSPACE;
  void* ws = nullptr;
  if (need > 0) {
    ws = gdn::static_scratch_address();
    if (!ws) return GDN_ERR_CUDA;
  }
  return gdn::run_forward(p, ws, static_cast<cudaStream_t>(stream));
}

extern "C" size_t gdn_noalloc_scratch_bytes(void) { return gdn::kStaticScratchBytes; }
