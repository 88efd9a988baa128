// C ABI of libgdn (declared in include/gdn.h): argument validation, workspace
// management and dispatch to the float32 SIMT path or the bf16 tensor-core path.
#include <cuda.h>

#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/gdn.h"
#include "gdn_internal.h"

namespace gdn {

__device__ unsigned int g_device_status = 0;

// The driver context current on this thread (nullptr if none or on failure).
// A symbol's device address belongs to the context the module was loaded in: a
// cudaDeviceReset or a primary-context teardown unloads the module, and the next
// context loads it again, possibly elsewhere.
void* current_context() {
  using Fn = CUresult (*)(CUcontext*);
  static Fn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<Fn>(ptr);
  });
  CUcontext ctx = nullptr;
  if (!fn || fn(&ctx) != CUDA_SUCCESS) return nullptr;
  return ctx;
}

void* SymbolAddressCache::get(const void* symbol) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  void* ctx = current_context();
  if (!ctx) {  // no context current yet: the runtime makes the device's primary one current
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, symbol) != cudaSuccess) return nullptr;
    ctx = current_context();
    if (!ctx) return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu_);
  if (ctx_[dev] != ctx || !ptr_[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, symbol) != cudaSuccess) return nullptr;
    ctx_[dev] = ctx;
    ptr_[dev] = ptr;
  }
  return ptr_[dev];
}

namespace {

// Device address of the status word in the current device's current context.
unsigned int* status_word() {
  static SymbolAddressCache cache;
  return static_cast<unsigned int*>(cache.get(reinterpret_cast<const void*>(&g_device_status)));
}

// Validates everything that can be checked on the host.  Fills `p`.
int validate(const void* q, const void* k, const void* v, const float* g, const float* beta,
             const float* state_in, void* out, float* state_out, int B, int H, int T, int S, int D, int dtype,
             int mode, Problem* p, bool need_gates = true) {
  if (B < 1 || H < 1 || T < 0 || S < 1 || D < 1) return kInvalidArg;
  if (dtype != GDN_F32 && dtype != GDN_BF16) return kInvalidArg;
  if (mode < GDN_MODE_SEQUENTIAL || mode > GDN_MODE_SPLIT) return kInvalidArg;
  if (D % 16 != 0 || D > 128) return kUnsupported;
  // Counts must stay inside what the kernels index with 64-bit offsets and
  // 32-bit grid dimensions / tensor-map extents.
  const long long bht = (long long)B * H * T;
  if ((long long)B * H > (1LL << 31) - 1 || bht > (1LL << 31) - 1) return kInvalidArg;
  if ((long long)S * D > (1LL << 31) - 1) return kInvalidArg;
  if (T > 0) {
    if (!q || !k || !v || !out) return kInvalidArg;
    if (need_gates && (!g || !beta)) return kInvalidArg;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16)) return kMisaligned;
    if (!aligned(g, 4) || !aligned(beta, 4)) return kMisaligned;
  }
  if (state_in && !aligned(state_in, 16)) return kMisaligned;
  if (state_out && !aligned(state_out, 16)) return kMisaligned;
  p->q = q;
  p->k = k;
  p->v = v;
  p->g = g;
  p->beta = beta;
  p->state_in = state_in;
  p->out = out;
  p->state_out = state_out;
  p->B = B;
  p->H = H;
  p->T = T;
  p->S = S;
  p->D = D;
  p->dtype = dtype;
  p->mode = mode;
  p->key_scale = (float)(1.0 / std::sqrt((double)D * (double)S));
  p->out_scale = (float)(1.0 / std::sqrt((double)D));
  return kOk;
}

size_t workspace_for(const Problem& p) {
  if (p.T == 0) return 0;
  return p.dtype == GDN_F32 ? simt_workspace_bytes(p, p.mode) : tc_workspace_bytes(p, p.mode);
}

// T = 0: the final state is the initial state.
int copy_state(const Problem& p, cudaStream_t st) {
  if (!p.state_out) return kOk;
  const size_t bytes = (size_t)p.BH() * p.D * p.D * sizeof(float);
  cudaError_t e;
  if (!p.state_in)
    e = cudaMemsetAsync(p.state_out, 0, bytes, st);
  else if (p.state_in != p.state_out)
    e = cudaMemcpyAsync(p.state_out, p.state_in, bytes, cudaMemcpyDeviceToDevice, st);
  else
    e = cudaSuccess;
  return e == cudaSuccess ? kOk : kCuda;
}

int forward(Problem p, void* ws, cudaStream_t st) {
  if (p.T == 0) return copy_state(p, st);
  p.status = status_word();
  if (!p.status) return kCuda;
  return p.dtype == GDN_F32 ? simt_forward(p, ws, st) : tc_forward(p, ws, st);
}

// ---- per-kernel event profiler --------------------------------------------------
struct ProfRec {
  const char* name;
  cudaEvent_t a, b;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<ProfRec> g_prof_recs;
std::vector<cudaEvent_t> g_prof_pool;

cudaEvent_t prof_event() {
  if (!g_prof_pool.empty()) {
    cudaEvent_t e = g_prof_pool.back();
    g_prof_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// gdn_frame_fwd_ex and gdn_frame_fwd_from_logits: validation, workspace check, launch.
int forward_ex(const void* q, const void* k, const void* v, const float* g, const float* beta, const float* state_in,
               void* out, float* state_out, int B, int H, int T, int S, int D, int dtype, int mode, void* workspace,
               size_t workspace_bytes, void* stream, int gate_logits) {
  Problem p{};
  int rc = validate(q, k, v, g, beta, state_in, out, state_out, B, H, T, S, D, dtype, mode, &p);
  if (rc != kOk) return rc;
  p.gate_logits = gate_logits;
  const size_t need = workspace_for(p);
  if (need > 0) {
    if (!workspace || workspace_bytes < need) return kWorkspace;
    if (!aligned(workspace, 256)) return kMisaligned;
  }
  return forward(p, workspace, static_cast<cudaStream_t>(stream));
}

}  // namespace

int check_args(const void* q, const void* k, const void* v, const float* g, const float* beta,
               const float* state_in, void* out, float* state_out, int B, int H, int T, int S, int D, int dtype,
               int mode, Problem* p, bool need_gates) {
  return validate(q, k, v, g, beta, state_in, out, state_out, B, H, T, S, D, dtype, mode, p, need_gates);
}
size_t scratch_bytes(const Problem& p) { return workspace_for(p); }

size_t debug_shrink() {
#if GDN_DEBUG
  const char* e = std::getenv("GDN_DEBUG_SHRINK");
  return e ? (size_t)std::strtoull(e, nullptr, 10) : 0;
#else
  return 0;
#endif
}
unsigned int* device_status_word() { return status_word(); }
int run_forward(const Problem& p, void* ws, cudaStream_t st) { return forward(p, ws, st); }

ProfScope::ProfScope(cudaStream_t st, const char* name) : st_(st), idx_(-1) {
  std::lock_guard<std::mutex> lock(g_prof_mu);
  if (!g_prof_on) return;
  ProfRec r{name, prof_event(), prof_event()};
  if (!r.a || !r.b) return;
  if (cudaEventRecord(r.a, st) != cudaSuccess) return;
  g_prof_recs.push_back(r);
  idx_ = (int)g_prof_recs.size() - 1;
}

ProfScope::~ProfScope() {
  if (idx_ < 0) return;
  std::lock_guard<std::mutex> lock(g_prof_mu);
  if (idx_ < (int)g_prof_recs.size()) cudaEventRecord(g_prof_recs[idx_].b, st_);
}

}  // namespace gdn

using namespace gdn;

extern "C" {

int gdn_frame_fwd_ex(const void* q, const void* k, const void* v, const float* g, const float* beta,
                     const float* state_in, void* out, float* state_out, int B, int H, int T, int S, int D,
                     int dtype, int mode, void* workspace, size_t workspace_bytes, void* stream) {
  return gdn::forward_ex(q, k, v, g, beta, state_in, out, state_out, B, H, T, S, D, dtype, mode, workspace,
                         workspace_bytes, stream, 0);
}

int gdn_relu_linear_fwd(const void* q, const void* k, const void* v, const float* state_in, void* out,
                        float* state_out, int B, int H, int T, int S, int D, int dtype, int mode, void* workspace,
                        size_t workspace_bytes, void* stream) {
  Problem p{};
  int rc = validate(q, k, v, nullptr, nullptr, state_in, out, state_out, B, H, T, S, D, dtype, mode, &p, false);
  if (rc != kOk) return rc;
  p.variant = kReluLinear;
  const size_t need = workspace_for(p);
  if (need > 0) {
    if (!workspace || workspace_bytes < need) return kWorkspace;
    if (!aligned(workspace, 256)) return kMisaligned;
  }
  return forward(p, workspace, static_cast<cudaStream_t>(stream));
}

int gdn_frame_fwd_from_logits(const void* q, const void* k, const void* v, const float* g_logit,
                              const float* beta_logit, const float* state_in, void* out, float* state_out, int B,
                              int H, int T, int S, int D, int dtype, int mode, void* workspace,
                              size_t workspace_bytes, void* stream) {
  return gdn::forward_ex(q, k, v, g_logit, beta_logit, state_in, out, state_out, B, H, T, S, D, dtype, mode,
                         workspace, workspace_bytes, stream, 1);
}

int gdn_frame_fwd(const void* q, const void* k, const void* v, const float* g, const float* beta,
                  const float* state_in, void* out, float* state_out, int B, int H, int T, int S, int D, int dtype,
                  void* stream) {
  Problem p{};
  int rc = validate(q, k, v, g, beta, state_in, out, state_out, B, H, T, S, D, dtype, GDN_MODE_SEQUENTIAL, &p);
  if (rc != kOk) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t need = workspace_for(p);
  void* ws = nullptr;
  if (need > 0 && cudaMallocAsync(&ws, need, st) != cudaSuccess) return kCuda;
  rc = forward(p, ws, st);
  if (ws && cudaFreeAsync(ws, st) != cudaSuccess && rc == kOk) rc = kCuda;
  return rc;
}

size_t gdn_workspace_bytes(int B, int H, int T, int S, int D, int dtype, int mode) {
  Problem p{};
  // Pointers are irrelevant here: validate as if T = 0 for the pointer checks.
  static const char dummy[16] __attribute__((aligned(16))) = {0};
  const void* d = dummy;
  if (validate(d, d, d, (const float*)d, (const float*)d, nullptr, (void*)d, nullptr, B, H, T, S, D, dtype, mode,
               &p) != kOk)
    return 0;
  return workspace_for(p);
}

int gdn_last_error(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return kCuda;
  unsigned int status = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&status, g_device_status, sizeof(status)) != cudaSuccess) return kCuda;
  if (status != 0 && cudaMemcpyToSymbol(g_device_status, &zero, sizeof(zero)) != cudaSuccess) return kCuda;
  return (int)status;
}

const char* gdn_status_string(int status) {
  switch (status) {
    case GDN_OK: return "GDN_OK";
    case GDN_ERR_INVALID_ARG: return "GDN_ERR_INVALID_ARG";
    case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED";
    case GDN_ERR_MISALIGNED: return "GDN_ERR_MISALIGNED";
    case GDN_ERR_CUDA: return "GDN_ERR_CUDA";
    case GDN_ERR_TIMEOUT: return "GDN_ERR_TIMEOUT";
    case GDN_ERR_WORKSPACE: return "GDN_ERR_WORKSPACE";
    case GDN_ERR_BOUNDS: return "GDN_ERR_BOUNDS";
    default: return "GDN_ERR_UNKNOWN";
  }
}

int gdn_version(void) { return 100; }

int gdn_profile_begin(void) {
  std::lock_guard<std::mutex> lock(g_prof_mu);
  g_prof_on = true;
  return GDN_OK;
}

int gdn_profile_end(gdn_kernel_stat_t* stats, int max_stats, int* n_stats) {
  if (!n_stats || (max_stats > 0 && !stats)) return GDN_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_prof_mu);
  g_prof_on = false;
  int rc = GDN_OK;
  std::vector<gdn_kernel_stat_t> agg;
  for (const ProfRec& r : g_prof_recs) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) {
      rc = GDN_ERR_CUDA;
      ms = 0.f;
    }
    size_t i = 0;
    while (i < agg.size() && std::strncmp(agg[i].name, r.name, sizeof(agg[i].name)) != 0) ++i;
    if (i == agg.size()) {
      gdn_kernel_stat_t z{};
      std::strncpy(z.name, r.name, sizeof(z.name) - 1);
      agg.push_back(z);
    }
    agg[i].launches += 1;
    agg[i].total_ms += ms;
    g_prof_pool.push_back(r.a);
    g_prof_pool.push_back(r.b);
  }
  g_prof_recs.clear();
  *n_stats = (int)agg.size();
  for (int i = 0; i < (int)agg.size() && i < max_stats; ++i) stats[i] = agg[i];
  return rc;
}

}  // extern "C"
