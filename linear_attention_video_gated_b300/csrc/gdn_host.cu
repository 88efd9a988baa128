// Host-buffer entry point (gdn_frame_fwd_host): the forward scan over inputs and
// outputs in host memory.  The frames are processed in chunks (the state carried
// from chunk to chunk on the device, as in a chunk-causal rollout); the copies in
// of chunk c + 1, the kernels of chunk c and the copies out of chunk c - 1 run at
// the same time on three streams, so a long clip costs about its host-to-device
// copy time rather than the sum of copies and kernels.
#include <cstring>

#include "../../include/gdn.h"
#include "gdn_internal.h"

namespace gdn {
namespace {

struct HostPlan {
  int C;                           // frames per chunk
  size_t q_bytes, g_bytes, b_bytes;  // one chunk buffer of q (= k = v = out), g, beta
  size_t off_q[2], off_k[2], off_v[2], off_o[2], off_g[2], off_b[2], off_state, off_ws;
  size_t ws_bytes, total;
};

// Device buffers: two chunk buffers of every tensor, the carried state and the
// scratch of one chunk call.  Returns false for arguments the entry point rejects.
bool host_plan(int B, int H, int T, int S, int D, int dtype, int chunk, HostPlan* pl) {
  if (B < 1 || H < 1 || T < 0 || S < 1 || chunk < 1) return false;
  if (dtype != GDN_F32 && dtype != GDN_BF16) return false;
  const int C = T < chunk ? (T > 0 ? T : 1) : chunk;
  static const char dummy[16] __attribute__((aligned(16))) = {0};
  const void* d = dummy;
  Problem p{};
  if (check_args(d, d, d, (const float*)d, (const float*)d, nullptr, (void*)d, nullptr, B, H, C, S, D, dtype,
                 GDN_MODE_SEQUENTIAL, &p) != kOk)
    return false;
  const size_t bh = (size_t)B * H, e = dtype == GDN_BF16 ? 2 : 4;
  pl->C = C;
  pl->q_bytes = align_up(bh * C * S * D * e, 256);
  pl->g_bytes = align_up(bh * C * 4, 256);
  pl->b_bytes = align_up(bh * C * S * 4, 256);
  pl->ws_bytes = align_up(scratch_bytes(p), 256);
  size_t o = 0;
  for (int i = 0; i < 2; ++i) {
    pl->off_q[i] = o; o += pl->q_bytes;
    pl->off_k[i] = o; o += pl->q_bytes;
    pl->off_v[i] = o; o += pl->q_bytes;
    pl->off_o[i] = o; o += pl->q_bytes;
    pl->off_g[i] = o; o += pl->g_bytes;
    pl->off_b[i] = o; o += pl->b_bytes;
  }
  pl->off_state = o;
  o += align_up(bh * D * D * 4, 256);
  pl->off_ws = o;
  pl->total = o + pl->ws_bytes;
  return true;
}

struct Streams {
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t start = nullptr, in[2] = {nullptr, nullptr}, comp[2] = {nullptr, nullptr},
              outd[2] = {nullptr, nullptr};
  ~Streams() {  // released once their work completes; nothing waits here
    if (h2d) cudaStreamDestroy(h2d);
    if (d2h) cudaStreamDestroy(d2h);
    for (cudaEvent_t ev : {start, in[0], in[1], comp[0], comp[1], outd[0], outd[1]})
      if (ev) cudaEventDestroy(ev);
  }
  bool create() {
    if (cudaStreamCreateWithFlags(&h2d, cudaStreamNonBlocking) != cudaSuccess) return false;
    if (cudaStreamCreateWithFlags(&d2h, cudaStreamNonBlocking) != cudaSuccess) return false;
    for (cudaEvent_t* ev : {&start, &in[0], &in[1], &comp[0], &comp[1], &outd[0], &outd[1]})
      if (cudaEventCreateWithFlags(ev, cudaEventDisableTiming) != cudaSuccess) return false;
    return true;
  }
};

#define GDN_TRY(x)                       \
  do {                                   \
    if ((x) != cudaSuccess) return kCuda; \
  } while (0)

}  // namespace
}  // namespace gdn

using namespace gdn;

extern "C" size_t gdn_host_workspace_bytes(int B, int H, int T, int S, int D, int dtype, int chunk_frames) {
  HostPlan pl;
  return host_plan(B, H, T, S, D, dtype, chunk_frames, &pl) ? pl.total : 0;
}

extern "C" int gdn_frame_fwd_host(const void* q, const void* k, const void* v, const float* g, const float* beta,
                                  const float* state_in, void* out, float* state_out, int B, int H, int T, int S,
                                  int D, int dtype, int chunk_frames, void* workspace, size_t workspace_bytes,
                                  void* stream) {
  HostPlan pl;
  if (!host_plan(B, H, T, S, D, dtype, chunk_frames, &pl)) {
    // report the same status the device entry points give for these arguments
    if (B < 1 || H < 1 || T < 0 || S < 1 || chunk_frames < 1 || (dtype != GDN_F32 && dtype != GDN_BF16))
      return GDN_ERR_INVALID_ARG;
    return (D % 16 != 0 || D < 16 || D > 128) ? GDN_ERR_UNSUPPORTED : GDN_ERR_INVALID_ARG;
  }
  if (T > 0 && (!q || !k || !v || !g || !beta || !out)) return GDN_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < pl.total) return GDN_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return GDN_ERR_MISALIGNED;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(workspace);
  const size_t bh = (size_t)B * H, e = dtype == GDN_BF16 ? 2 : 4;
  const size_t row = (size_t)S * D * e;  // one frame of q / k / v / out, bytes
  float* state = reinterpret_cast<float*>(w + pl.off_state);
  const size_t state_bytes = bh * D * D * 4;

  if (state_in)
    GDN_TRY(cudaMemcpyAsync(state, state_in, state_bytes, cudaMemcpyHostToDevice, st));
  else
    GDN_TRY(cudaMemsetAsync(state, 0, state_bytes, st));
  if (T > 0) {
    Streams ss;
    if (!ss.create()) return kCuda;
    GDN_TRY(cudaEventRecord(ss.start, st));  // after the caller's earlier work on `stream`
    GDN_TRY(cudaStreamWaitEvent(ss.h2d, ss.start, 0));
    GDN_TRY(cudaStreamWaitEvent(ss.d2h, ss.start, 0));
    const int nchunks = (T + pl.C - 1) / pl.C;
    for (int c = 0; c < nchunks; ++c) {
      const int b = c & 1, t0 = c * pl.C, tc = (T - t0) < pl.C ? (T - t0) : pl.C;
      // copies in: chunk c into buffer b, once chunk c - 2's kernels have read it
      if (c >= 2) GDN_TRY(cudaStreamWaitEvent(ss.h2d, ss.comp[b], 0));
      const struct {
        const void* src;
        size_t off, frame;
      } ins[5] = {{q, pl.off_q[b], row}, {k, pl.off_k[b], row}, {v, pl.off_v[b], row},
                  {g, pl.off_g[b], 4}, {beta, pl.off_b[b], (size_t)S * 4}};
      for (const auto& in : ins)
        GDN_TRY(cudaMemcpy2DAsync(w + in.off, tc * in.frame, static_cast<const uint8_t*>(in.src) + t0 * in.frame,
                                  (size_t)T * in.frame, tc * in.frame, bh, cudaMemcpyHostToDevice, ss.h2d));
      GDN_TRY(cudaEventRecord(ss.in[b], ss.h2d));
      // kernels: chunk c on the caller's stream, the state carried in place
      GDN_TRY(cudaStreamWaitEvent(st, ss.in[b], 0));
      if (c >= 2) GDN_TRY(cudaStreamWaitEvent(st, ss.outd[b], 0));  // out buffer b copied out
      Problem p{};
      int rc = check_args(w + pl.off_q[b], w + pl.off_k[b], w + pl.off_v[b],
                          reinterpret_cast<const float*>(w + pl.off_g[b]),
                          reinterpret_cast<const float*>(w + pl.off_b[b]), state, w + pl.off_o[b], state, B, H, tc,
                          S, D, dtype, GDN_MODE_SEQUENTIAL, &p);
      if (rc != kOk) return rc;
      if (scratch_bytes(p) > pl.ws_bytes) return kWorkspace;
      rc = run_forward(p, w + pl.off_ws, st);
      if (rc != kOk) return rc;
      GDN_TRY(cudaEventRecord(ss.comp[b], st));
      // copies out: chunk c's outputs
      GDN_TRY(cudaStreamWaitEvent(ss.d2h, ss.comp[b], 0));
      GDN_TRY(cudaMemcpy2DAsync(static_cast<uint8_t*>(out) + t0 * row, (size_t)T * row, w + pl.off_o[b], tc * row,
                                tc * row, bh, cudaMemcpyDeviceToHost, ss.d2h));
      GDN_TRY(cudaEventRecord(ss.outd[b], ss.d2h));
    }
    // the call is complete on `stream` once every copy out is
    GDN_TRY(cudaStreamWaitEvent(st, ss.outd[(nchunks - 1) & 1], 0));
  }
  if (state_out) GDN_TRY(cudaMemcpyAsync(state_out, state, state_bytes, cudaMemcpyDeviceToHost, st));
  return kOk;
}
