// C ABI of the context-parallel pieces (declared in include/gdn.h): the affine
// map a range of frames applies to the state, and its application.  The pages'
// context-parallel training cuts the latent sequence into frame ranges, one per
// GPU, and recovers each range's initial state by composing the GDN transition
// maps of the ranges before it, exactly (zhichai.net SANA-WM summary, training
// pipeline Stage 3).  Per head, frames [t0, t1) map a state S to
//     A S + b,   A = A_{t1-1} ... A_{t0},  A_t = g_t (I - K~_t^T diag(beta_t) K~_t),
// and b is the state the range produces from a zero initial state.
#include <cstdint>

#include "../../include/gdn.h"
#include "gdn_internal.h"

namespace gdn {
namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Validation of gdn_frame_summary's arguments (everything but the workspace).
int check_summary(const void* k, const void* v, const float* g, const float* beta, float* A_out, float* b_out,
                  int B, int H, int T, int S, int D, int dtype, int flags, Problem* p) {
  if (flags & ~GDN_SUMMARY_GATE_LOGITS) return kInvalidArg;
  if (!A_out || !b_out) return kInvalidArg;
  if (!aligned16(A_out) || !aligned16(b_out)) return kMisaligned;
  // q and out take no part: k and A_out stand in for them in the shared checks
  const int rc = check_args(k, k, v, g, beta, nullptr, A_out, nullptr, B, H, T, S, D, dtype, GDN_MODE_PREFIX, p);
  if (rc != kOk) return rc;
  p->q = nullptr;
  p->out = nullptr;
  p->gate_logits = (flags & GDN_SUMMARY_GATE_LOGITS) ? 1 : 0;
  return kOk;
}

}  // namespace
}  // namespace gdn

using namespace gdn;

extern "C" size_t gdn_summary_workspace_bytes(int B, int H, int T, int S, int D, int dtype) {
  return gdn_workspace_bytes(B, H, T, S, D, dtype, GDN_MODE_PREFIX);
}

extern "C" int gdn_frame_summary(const void* k, const void* v, const float* g, const float* beta, float* A_out,
                                 float* b_out, int B, int H, int T, int S, int D, int dtype, int flags,
                                 void* workspace, size_t workspace_bytes, void* stream) {
  Problem p{};
  int rc = check_summary(k, v, g, beta, A_out, b_out, B, H, T, S, D, dtype, flags, &p);
  if (rc != kOk) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (T == 0)  // no frames: the identity map
    return launch_chunk_fold(nullptr, nullptr, 0, 0, 0, nullptr, nullptr, nullptr, A_out, b_out, p.BH(), D, st);
  const size_t need = scratch_bytes(p);
  if (!workspace || workspace_bytes < need) return kWorkspace;
  if (!aligned(workspace, 256)) return kMisaligned;
  p.status = device_status_word();
  if (!p.status) return kCuda;
  float* maps = nullptr;
  int nch = 0;
  rc = dtype == GDN_BF16 ? tc_chunk_maps(p, workspace, &maps, &nch, st)
                         : simt_chunk_maps(p, workspace, &maps, &nch, st);
  if (rc != kOk) return rc;
  return launch_chunk_fold(maps, maps + D, 2LL * D * D, 2 * D, nch, nullptr, nullptr, nullptr, A_out, b_out, p.BH(),
                           D, st);
}

extern "C" int gdn_summary_apply(const float* A, const float* b, const float* state_in, float* state_out, int B,
                                 int H, int D, void* stream) {
  if (B < 1 || H < 1 || (long long)B * H > (1LL << 31) - 1) return kInvalidArg;
  if (D % 16 != 0 || D < 16 || D > 128) return kUnsupported;
  if (!A || !b || !state_out) return kInvalidArg;
  if (!aligned16(A) || !aligned16(b) || !aligned16(state_out) || (state_in && !aligned16(state_in)))
    return kMisaligned;
  const size_t span = (size_t)B * H * D * D * sizeof(float);
  return launch_chunk_fold(A, b, (long long)D * D, D, 1, state_in, nullptr, state_out, nullptr, nullptr,
                           (long long)B * H, D, static_cast<cudaStream_t>(stream), span, span, 0);
}
