// Internal declarations shared by the libgdn translation units.
//
// Every path computes the scan in its affine ("transition") form, which is the
// residual-form update multiplied out:
//
//   S_t = g_t S_{t-1} + K~^T diag(beta) (V - g_t K~ S_{t-1})
//       = g_t (S_{t-1} - M_t S_{t-1}) + b_t,
//   M_t = K~^T diag(beta) K~   (D x D, symmetric PSD),   b_t = K~^T diag(beta) V_t.
//
// M_t and b_t depend only on frame t's inputs, so they are formed for every
// frame in parallel ("gram" stage); only the D x D x D recurrence is serial
// ("scan" stage); the read-out O_t = Q_t S_t / sqrt(D) is parallel again
// ("readout" stage).  The same maps (A_t = g_t (I - M_t), b_t) are what the
// prefix mode composes (zhichai.net SANA-WM summary, training Stage 3).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <mutex>

namespace gdn {

struct Problem {
  const void* q;
  const void* k;
  const void* v;
  const float* g;
  const float* beta;
  const float* state_in;
  void* out;
  float* state_out;
  int B, H, T, S, D;
  int dtype;  // gdn_dtype_t
  int mode;   // gdn_mode_t
  int gate_logits;  // 1: g and beta hold raw logits, mapped by decay_of / beta_of where loaded
  int variant;      // kGdn, or kReluLinear: the cumulative ReLU linear attention baseline
  float key_scale;  // 1/sqrt(D*S)
  float out_scale;  // 1/sqrt(D)
  unsigned int* status;  // device-side status word (first error wins)
  long long BH() const { return (long long)B * H; }
  long long BHT() const { return (long long)B * H * T; }
};

// Status codes (mirror gdn_status_t).
enum Status {
  kOk = 0, kInvalidArg = 1, kUnsupported = 2, kMisaligned = 3, kCuda = 4, kTimeout = 5, kWorkspace = 6, kBounds = 7
};

// The gate prologue fused into the kernels (gdn_frame_fwd_from_logits): raw
// logits x become the per-frame decay g = exp(-softplus(x)) = 1 / (1 + e^x) and
// the per-token delta-rule weight beta = sigmoid(x) = 1 / (1 + e^-x) where the
// kernels load them.
__device__ __forceinline__ float decay_of(float x, int logits) { return logits ? 1.f / (1.f + expf(x)) : x; }
__device__ __forceinline__ float beta_of(float x, int logits) { return logits ? 1.f / (1.f + expf(-x)) : x; }

// Recurrence computed by the kernels.  kReluLinear is the SANA-Video baseline the
// pages contrast GDN with (cumulative ReLU-based linear attention): no decay
// (g = 1), no delta-rule correction (the M_t term dropped, beta = 1), ReLU
// applied to queries and keys:  S_t = S_{t-1} + relu(K_t)~^T V_t,
// O_t = relu(Q_t) S_t / sqrt(D), with the same 1/sqrt(D*S) key scale.
enum Variant { kGdn = 0, kReluLinear = 1 };
__device__ __forceinline__ float relu_if(float x, int variant) { return variant == kReluLinear ? fmaxf(x, 0.f) : x; }

// Element loads and stores of the I/O dtypes (float32 arithmetic inside).
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void from_f32(float& d, float x) { d = x; }
__device__ __forceinline__ void from_f32(__nv_bfloat16& d, float x) { d = __float2bfloat16_rn(x); }

// Records a device-side error in the status word; the first error wins.
__device__ __forceinline__ void report_device_error(unsigned int* status, unsigned int code) {
  atomicCAS(status, 0u, code);
}

// The debug build (nvcc -DGDN_DEBUG=1: libgdn_debug.so) checks every scratch
// offset a kernel computes against the extent of its region as the host's
// layout gives it: `end`, one past the last byte the access touches relative to
// the region's start, must not pass `span` (0: not given, not checked).  A failed
// check records GDN_ERR_BOUNDS and the access is skipped (a skipped copy then
// ends in a bounded wait that gives up); nothing traps.  Compiled out otherwise.
#ifndef GDN_DEBUG
#define GDN_DEBUG 0
#endif
__device__ __forceinline__ bool in_region(size_t end, size_t span, unsigned int* status) {
#if GDN_DEBUG
  if (span != 0 && end > span) {
    if (status) report_device_error(status, kBounds);
    return false;
  }
#else
  (void)end;
  (void)span;
  (void)status;
#endif
  return true;
}

// Debug build only: bytes taken off the read-out's image region extent before it
// is passed to the kernel (GDN_DEBUG_SHRINK in the environment), so that a test
// can see a check fire; 0 in the release build.
size_t debug_shrink();

// ---- argument checks and dispatch (gdn_api.cu), for the other C-ABI files -------
// Validates the arguments of a forward call and fills `p` (returns a Status).
int check_args(const void* q, const void* k, const void* v, const float* g, const float* beta,
               const float* state_in, void* out, float* state_out, int B, int H, int T, int S, int D, int dtype,
               int mode, Problem* p, bool need_gates = true);
// Enqueues the call on `st` (scratch `ws` of scratch_bytes(p) bytes).
int run_forward(const Problem& p, void* ws, cudaStream_t st);
// Device address of the status word on the current device (nullptr on failure).
unsigned int* device_status_word();
// Scratch bytes the call `p` needs.
size_t scratch_bytes(const Problem& p);

// Device addresses of a __device__ variable, looked up (cudaGetSymbolAddress)
// once per device and context and cached: a symbol's name in host code is only
// a host-side stand-in, and its address changes if the context is torn down
// and re-created.  Thread-safe.
class SymbolAddressCache {
 public:
  // The address of `symbol` (the address of the __device__ variable as host
  // code names it) in the current device's current context; nullptr on failure.
  void* get(const void* symbol);
 private:
  static constexpr int kMaxDevices = 64;
  std::mutex mu_;
  void* ctx_[kMaxDevices] = {nullptr};
  void* ptr_[kMaxDevices] = {nullptr};
};

// ---- SIMT path (float32 arithmetic; used for float32 I/O) --------------------
size_t simt_workspace_bytes(const Problem& p, int mode);
int simt_forward(const Problem& p, void* ws, cudaStream_t st);
// M_t, b_t and the state S_t after every frame (each BHT x D x D float32, frame-head
// major), by the sequential scan; writes p.state_out when it is not null.
int simt_states(const Problem& p, float* Mws, float* bws, float* Sws, cudaStream_t st);

// Per-chunk composed maps [A_c | b_c] (BH x nchunks x D x 2D float32, in `ws`,
// which holds at least simt_workspace_bytes(p, GDN_MODE_PREFIX) bytes) of
// 16-frame chunks: the float32 gram and composition.
int simt_chunk_maps(const Problem& p, void* ws, float** maps, int* nchunks, cudaStream_t st);

// Fold of affine maps over chunks in float32 (gdn_simt.cu): per head,
// x_{c+1} = A_c x_c + b_c for c = 0 .. nchunks - 1, with A_c at A + (head *
// nchunks + c) * chunk_stride (rows `ld` floats apart) and b_c likewise from b.
// Boundary form (A_out null): x_0 = state_in (zeros if null); x_c -> starts (if
// set), the last x -> x_out (if set; may alias state_in).  Summary form: the
// composed map of all chunks -> A_out, b_out ([BH][D][D] each).
int launch_chunk_fold(const float* A, const float* b, long long chunk_stride, int ld, int nchunks,
                      const float* state_in, float* starts, float* x_out, float* A_out, float* b_out, long long BH,
                      int D, cudaStream_t st, size_t a_span = 0, size_t b_span = 0, size_t starts_span = 0);

// ---- tensor-core path (bf16 I/O) ------------------------------------------------
size_t tc_workspace_bytes(const Problem& p, int mode);
int tc_forward(const Problem& p, void* ws, cudaStream_t st);
// Per-chunk composed maps [A_c | b_c] of kTcChunkFrames-frame chunks on the tensor
// cores (the gram, then the chunked scan's summary form), in `ws` of at least
// tc_workspace_bytes(p, GDN_MODE_PREFIX) bytes.
int tc_chunk_maps(const Problem& p, void* ws, float** maps, int* nchunks, cudaStream_t st);

// ---- backward pass (gdn_bwd.cu; the bf16 kernels in gdn_tc.cu) -------------------
struct BwdGrads {
  const void* dout;
  const float* dstate_out;
  void *dq, *dk, *dv;
  float *dg, *dbeta, *dstate_in;
};
// Tensor-core backward (bf16 I/O): workspace bytes, and the call.  Writes dq, dk,
// dv, dbeta and dstate_in, and per (frame-head, 128-token tile) partial sums of dg
// into `dg_part` (*ntiles tiles per frame-head), which launch_dg_sum reduces.
// With states_ready the workspace already holds the M_t image, b_t blocks and S_t
// images of a forward split-form call over the same inputs (the first three regions
// of the backward layout are the forward's), and their recomputation is skipped.
size_t tc_bwd_workspace_bytes(const Problem& p);
int tc_backward(const Problem& p, const BwdGrads& gr, void* ws, cudaStream_t st, bool states_ready);
// dg[f] = sum of dg_part[f * ntiles .. + ntiles) (times dg/dlogit for logits).
int launch_dg_sum(const float* dg_part, const float* g, float* dg, long long nframes, int ntiles, int logits,
                  cudaStream_t st);

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Brackets one kernel launch with CUDA events while gdn_profile_begin() is in
// effect (no-op otherwise).  Construct immediately before the launch.
class ProfScope {
 public:
  ProfScope(cudaStream_t st, const char* name);
  ~ProfScope();
 private:
  cudaStream_t st_;
  int idx_;
};

}  // namespace gdn
