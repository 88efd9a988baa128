/*
 * gdn.h -- C ABI of libgdn: the frame-wise Gated DeltaNet (GDN) forward scan on
 * NVIDIA B300 (sm_103a).
 *
 * The operation (SANA-WM's frame-wise GDN sequence mixer).  Per head (b, h),
 * for frames t = 0 .. T-1, with S tokens per frame and head dim D:
 *
 *     K~_t = K_t / sqrt(D*S)                                   (key scaling)
 *     S_t  = g_t S_{t-1} + K~_t^T diag(beta_t) (V_t - g_t K~_t S_{t-1})
 *     O_t  = Q_t S_t / sqrt(D)
 *
 * Sources, by page and section:
 *   - frame-wise recurrence, one step per latent frame: bilibili SANA-WM
 *     article, fourth key point (frame-wise Gated DeltaNet replacing most
 *     attention blocks; decay g in the update rule);
 *   - decay gate multiplies the previous state by a scalar; beta delta rule
 *     writes only the residual between target and prediction; constant D x D
 *     state; keys scaled by 1/sqrt(D*S): zhichai.net SANA-WM summary, section
 *     "四大工程设计" item 1 (Hybrid Linear Attention -- Gated DeltaNet + Softmax);
 *   - state carried across chunk-causal autoregressive calls: bilibili article,
 *     second key point (chunk-causal autoregressive generator), and zhichai.net
 *     summary, training pipeline Stage 4;
 *   - composition of the per-frame transition maps by prefix sums, exact:
 *     zhichai.net summary, training pipeline Stage 3 (context parallel).
 * The pages print no equation; the 1/sqrt(D) read-out scale is not on them.
 *
 * Conventions for every entry point below:
 *   - Tensors are dense, row-major, contiguous:
 *       q, k, v, out : [B, H, T, S, D]  elements of `dtype` (GDN_F32 or GDN_BF16)
 *       g            : [B, H, T]        float32, the per-frame decay, in [0, 1]
 *       beta         : [B, H, T, S]     float32, the per-token delta-rule weight
 *       state_in/out : [B, H, D, D]     float32, S[i][j]: i = key dim, j = value dim
 *   - Every pointer is a DEVICE pointer on the current CUDA device, owned by the
 *     caller.  The library allocates no persistent memory and keeps no state
 *     beyond cached function attributes and one device-side status word.
 *   - q, k, v, out, state_in, state_out and workspace must be 16-byte aligned
 *     (TMA requirement); g and beta 4-byte aligned.  Otherwise GDN_ERR_MISALIGNED.
 *   - Supported shapes: B >= 1, H >= 1, T >= 0, S >= 1, D in {16, 32, ..., 128}.
 *     Other D -> GDN_ERR_UNSUPPORTED.  T = 0 copies state_in to state_out (zeros
 *     if state_in is NULL) and touches nothing else.
 *   - state_in == NULL means a zero initial state; state_out == NULL means the
 *     final state is not written; state_in == state_out is allowed (the kernel
 *     reads a head's state before it writes it).  No other overlap is allowed.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls are
 *     asynchronous: the return code covers argument validation and launch
 *     errors only.  Faults detected on the device (a bounded wait that timed
 *     out) are reported by gdn_last_error().
 *   - Returns 0 (GDN_OK) or a gdn_status_t code; gdn_status_string() names it.
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GDN_F32 = 0,  /* q, k, v, out are float32 */
  GDN_BF16 = 1  /* q, k, v, out are bfloat16 (the state stays float32) */
} gdn_dtype_t;

typedef enum {
  GDN_OK = 0,
  GDN_ERR_INVALID_ARG = 1, /* NULL pointer, bad count, bad dtype/mode     */
  GDN_ERR_UNSUPPORTED = 2, /* D not a multiple of 16 in [16, 128]         */
  GDN_ERR_MISALIGNED = 3,  /* a pointer misses its alignment              */
  GDN_ERR_CUDA = 4,        /* a CUDA runtime/driver call or launch failed */
  GDN_ERR_TIMEOUT = 5,     /* a bounded device-side wait gave up          */
  GDN_ERR_WORKSPACE = 6,   /* workspace NULL or smaller than required     */
  GDN_ERR_BOUNDS = 7       /* debug build only (libgdn_debug.so, compiled
                            * with -DGDN_DEBUG=1): a kernel's scratch offset
                            * fell outside its region; the access was
                            * skipped and the call's results are invalid  */
} gdn_status_t;

typedef enum {
  /* One pass over the frames per head: the library's fastest form for the
   * shape and dtype (currently the split form below). */
  GDN_MODE_SEQUENTIAL = 0,
  /* Chunked prefix composition of the affine maps (A_t, b_t) across frames:
   * per-chunk composed maps in parallel, a short scan over chunk boundaries,
   * then every chunk replayed from its true initial state (zhichai.net summary,
   * training pipeline Stage 3).  Same result up to rounding. */
  GDN_MODE_PREFIX = 1,
  /* Three kernels through a workspace: the per-frame transition terms
   * (M_t = K~^T diag(beta) K~, b_t = K~^T diag(beta) V_t) for all frames in
   * parallel, the serial D x D recurrence, then the read-out for all frames in
   * parallel. */
  GDN_MODE_SPLIT = 2
  /* Any other value gives GDN_ERR_INVALID_ARG. */
} gdn_mode_t;

/*
 * gdn_frame_fwd -- the forward scan over T frames of every (b, h) head.
 *   q, k, v   : inputs, see conventions.  K is scaled by 1/sqrt(D*S) inside.
 *   g, beta   : decay per frame, delta-rule weight per token.
 *   state_in  : initial state or NULL (zeros).
 *   out       : output O_t for every frame, same dtype as q.
 *   state_out : final state S_{T-1} or NULL.
 *   dtype     : gdn_dtype_t.
 * Uses GDN_MODE_SEQUENTIAL.  Its scratch memory (gdn_workspace_bytes()) is
 * taken with cudaMallocAsync on
 * `stream` and released with cudaFreeAsync on the same stream, so nothing
 * persists past the call.
 */
int gdn_frame_fwd(const void* q, const void* k, const void* v,
                  const float* g, const float* beta, const float* state_in,
                  void* out, float* state_out,
                  int B, int H, int T, int S, int D, int dtype, void* stream);

/*
 * gdn_workspace_bytes -- scratch bytes gdn_frame_fwd_ex needs for this shape,
 * dtype and mode (0 for T = 0).  Returns 0 for arguments gdn_frame_fwd_ex would
 * reject.  The result is a pure function of the arguments.
 */
size_t gdn_workspace_bytes(int B, int H, int T, int S, int D, int dtype, int mode);

/*
 * gdn_frame_fwd_ex -- gdn_frame_fwd with an explicit algorithm form and a
 * caller-owned device workspace of at least gdn_workspace_bytes() bytes,
 * 256-byte aligned.  The workspace is not read before it is written.  After a
 * call it holds the per-frame states that gdn_frame_bwd_ex reads with
 * GDN_BWD_STATES_IN_WORKSPACE.  Two calls in flight at the same time must not share a workspace.
 *   mode : gdn_mode_t.
 */
int gdn_frame_fwd_ex(const void* q, const void* k, const void* v,
                     const float* g, const float* beta, const float* state_in,
                     void* out, float* state_out,
                     int B, int H, int T, int S, int D, int dtype, int mode,
                     void* workspace, size_t workspace_bytes, void* stream);

/*
 * gdn_frame_fwd_from_logits -- gdn_frame_fwd_ex with the gate computations fused
 * into the scan's kernels (the pages fuse the "GDN scan and gate ops"; zhichai.net
 * summary, the paragraph after training Stage 4).  g_logit [B,H,T] and
 * beta_logit [B,H,T,S] hold raw float32 logits; where the kernels load them they
 * become the decay g = exp(-softplus(g_logit)) = 1 / (1 + e^g_logit), in (0, 1),
 * and the delta-rule weight beta = sigmoid(beta_logit), in (0, 1).  The pages do
 * not state the gates' parameterisation: these are the maps the one-minute
 * workload's gates are drawn through.  Everything else (arguments, workspace,
 * modes, errors) is as gdn_frame_fwd_ex.
 */
int gdn_frame_fwd_from_logits(const void* q, const void* k, const void* v,
                              const float* g_logit, const float* beta_logit, const float* state_in,
                              void* out, float* state_out,
                              int B, int H, int T, int S, int D, int dtype, int mode,
                              void* workspace, size_t workspace_bytes, void* stream);

/*
 * gdn_relu_linear_fwd -- the baseline the pages contrast GDN with: SANA-Video's
 * cumulative ReLU-based linear attention (zhichai.net summary, section 1, the
 * paragraph on SANA-Video; bilibili article, third key point), run through the
 * same kernels.  Per head, with no decay, no delta-rule correction and no gates:
 *     S_t = S_{t-1} + relu(K_t)^T V_t / sqrt(D*S),   O_t = relu(Q_t) S_t / sqrt(D).
 * (The pages give no formula; this is the plainest reading with the GDN scan's
 * own scalings, so the two differ only in the decay, the delta rule and the
 * feature map.)  Arguments, layouts, workspace (gdn_workspace_bytes with the same
 * mode) and errors as gdn_frame_fwd_ex without g and beta.
 */
int gdn_relu_linear_fwd(const void* q, const void* k, const void* v, const float* state_in,
                        void* out, float* state_out,
                        int B, int H, int T, int S, int D, int dtype, int mode,
                        void* workspace, size_t workspace_bytes, void* stream);

/*
 * gdn_frame_bwd -- the gradients of gdn_frame_fwd with respect to all of its
 * inputs, for training.  The pages train the model with this layer (zhichai.net
 * SANA-WM summary, training pipeline, Stages 1-4) but give no backward pass: it
 * is the forward definition differentiated.  Per head, with U_t the gradient with
 * respect to the state after frame t and M_t = K~_t^T diag(beta_t) K~_t:
 *     U_{T-1} = dstate_out + Q_{T-1}^T dO_{T-1} / sqrt(D)
 *     U_{t-1} = Q_{t-1}^T dO_{t-1} / sqrt(D) + g_t (U_t - M_t U_t)
 *     dstate_in = g_0 (U_0 - M_0 U_0)
 * (the forward's affine map, adjoint, from the last frame to the first), and per
 * frame, with P = K~_t S_{t-1} and dR = K~_t U_t:
 *     dQ_t = dO_t S_t^T / sqrt(D)
 *     dV_t = diag(beta_t) dR
 *     dbeta_t[s] = <dR_s, V_s - g_t P_s>
 *     dK_t = ( diag(beta_t)(V_t - g_t P) U_t^T - g_t diag(beta_t) dR S_{t-1}^T ) / sqrt(D*S)
 *     dg_t = <U_t, S_{t-1}> - sum_s beta_t[s] <dR_s, P_s>
 *   q, k, v, g, beta, state_in : the forward call's inputs, as gdn_frame_fwd takes
 *       them (the states S_t are recomputed, not passed in).
 *   dout       : [B,H,T,S,D] `dtype`, the gradient of the loss with respect to out.
 *   dstate_out : [B,H,D,D] float32, the gradient with respect to state_out, or NULL
 *                (zeros: the final state does not enter the loss).
 *   dq, dk, dv : [B,H,T,S,D] `dtype`, written (bf16 results rounded to nearest even).
 *   dg         : [B,H,T] float32, written.
 *   dbeta      : [B,H,T,S] float32, written.
 *   dstate_in  : [B,H,D,D] float32, written, or NULL (not written).
 *   workspace  : device memory of at least gdn_bwd_workspace_bytes() bytes,
 *                256-byte aligned, owned by the caller; not read before it is
 *                written.  Per frame-head: M_t, the read-out term Q^T dO, S_t and
 *                U_t (float32 matrices for GDN_F32; for GDN_BF16 M_t as a bf16
 *                image and S_t, U_t as bf16 hi + lo images) and a few partial sums.
 * All pointers are device pointers with the alignment rules of the conventions
 * (dq, dk, dv, dout, dstate_* 16 bytes; dg, dbeta 4 bytes).  No output may overlap
 * an input or another output.  GDN_F32 computes in float32 on CUDA cores;
 * GDN_BF16 runs the dense products on the tensor cores (bf16 operands, the states
 * and state gradients split into bf16 hi + lo parts, float32 accumulation) and
 * the element-wise steps in float32.  T = 0 copies dstate_out to dstate_in (zeros
 * if NULL) and touches nothing else.  Returns as gdn_frame_fwd_ex (GDN_ERR_INVALID_ARG for a NULL
 * gradient output other than dstate_in).
 */
int gdn_frame_bwd(const void* q, const void* k, const void* v,
                  const float* g, const float* beta, const float* state_in,
                  const void* dout, const float* dstate_out,
                  void* dq, void* dk, void* dv, float* dg, float* dbeta, float* dstate_in,
                  int B, int H, int T, int S, int D, int dtype,
                  void* workspace, size_t workspace_bytes, void* stream);

/*
 * gdn_frame_bwd_from_logits -- gdn_frame_bwd for gdn_frame_fwd_from_logits: the
 * gates are given as logits, and dg_logit / dbeta_logit receive the gradients of
 * the logits (the chain rule through g = exp(-softplus(x)), dg/dx = -g (1 - g),
 * and beta = sigmoid(y), dbeta/dy = beta (1 - beta), applied inside the kernels).
 */
int gdn_frame_bwd_from_logits(const void* q, const void* k, const void* v,
                              const float* g_logit, const float* beta_logit, const float* state_in,
                              const void* dout, const float* dstate_out,
                              void* dq, void* dk, void* dv, float* dg_logit, float* dbeta_logit,
                              float* dstate_in, int B, int H, int T, int S, int D, int dtype,
                              void* workspace, size_t workspace_bytes, void* stream);

/* gdn_bwd_workspace_bytes -- workspace gdn_frame_bwd needs (0 for T = 0 and for
 * arguments it rejects).  It is never smaller than gdn_workspace_bytes() of any
 * forward form for the same shape and dtype. */
size_t gdn_bwd_workspace_bytes(int B, int H, int T, int S, int D, int dtype);

/* Flags of gdn_frame_bwd_ex. */
#define GDN_BWD_STATES_IN_WORKSPACE 1 /* reuse the states a forward call left in the workspace */
#define GDN_BWD_GATE_LOGITS 2         /* g and beta are logits (as gdn_frame_bwd_from_logits) */

/*
 * gdn_frame_bwd_ex -- gdn_frame_bwd / gdn_frame_bwd_from_logits with flags.
 * (No counterpart on the pages: it saves recomputing the forward states in a
 * training step that has just run the forward.)
 *   GDN_BWD_STATES_IN_WORKSPACE : `workspace` (at least gdn_bwd_workspace_bytes())
 *       already holds what a gdn_frame_fwd_ex call left in it -- GDN_MODE_SEQUENTIAL
 *       or GDN_MODE_SPLIT (for GDN_F32 also GDN_MODE_PREFIX) -- over the same q, k,
 *       v, g, beta, state_in, shape and dtype, with gates given the same way (a
 *       logit forward for GDN_BWD_GATE_LOGITS), and nothing has written to the
 *       workspace since.  The backward then skips recomputing the per-frame
 *       states; its results are bit for bit those of the call without the flag.
 *       The library cannot check that the workspace holds such states: a
 *       workspace that does not gives wrong gradients, not an error.
 *   GDN_BWD_GATE_LOGITS : g and beta are logits; dg and dbeta are the logits'
 *       gradients (as gdn_frame_bwd_from_logits).
 * Other flag bits give GDN_ERR_INVALID_ARG.  Everything else as gdn_frame_bwd.
 * For the GDN_MODE_PREFIX forward the states are the prefix composition's, so
 * the gradients agree with the recomputing call's up to rounding, not bit for bit.
 */
int gdn_frame_bwd_ex(const void* q, const void* k, const void* v,
                     const float* g, const float* beta, const float* state_in,
                     const void* dout, const float* dstate_out,
                     void* dq, void* dk, void* dv, float* dg, float* dbeta, float* dstate_in,
                     int B, int H, int T, int S, int D, int dtype, int flags,
                     void* workspace, size_t workspace_bytes, void* stream);

/*
 * gdn_frame_fwd_host -- the forward scan over inputs and outputs in HOST memory.
 * (No counterpart on the pages: a streaming runtime around the scan.)
 *   q, k, v, g, beta, state_in, out, state_out : host pointers with the layouts of
 *       gdn_frame_fwd; page-locked (pinned) memory lets the copies overlap the
 *       kernels, pageable memory works but serialises them.  state_in / state_out
 *       may be NULL as in gdn_frame_fwd.
 *   chunk_frames : frames per chunk (>= 1).  The frames are processed chunk by
 *       chunk, the state carried from one chunk to the next on the device as in a
 *       chunk-causal rollout (the bilibili SANA-WM article, second key point), so
 *       the result equals gdn_frame_fwd's bit for bit.  The copies in of chunk
 *       c + 1, the kernels of chunk c and the copies out of chunk c - 1 run at the
 *       same time: the kernels on `stream`, the copies on two streams the call
 *       creates and releases.
 *   workspace : DEVICE memory of at least gdn_host_workspace_bytes() bytes,
 *       256-byte aligned, owned by the caller: two chunk buffers of every tensor,
 *       the carried state and one chunk call's scratch.
 * Asynchronous like gdn_frame_fwd: the host buffers must stay valid and unchanged
 * until `stream` reaches the end of the call (synchronise the stream before reading
 * out / state_out).  Returns GDN_OK, GDN_ERR_INVALID_ARG (bad counts, NULL inputs,
 * chunk_frames < 1), GDN_ERR_UNSUPPORTED (D), GDN_ERR_WORKSPACE, GDN_ERR_MISALIGNED
 * (workspace) or GDN_ERR_CUDA.
 */
int gdn_frame_fwd_host(const void* q, const void* k, const void* v,
                       const float* g, const float* beta, const float* state_in,
                       void* out, float* state_out,
                       int B, int H, int T, int S, int D, int dtype, int chunk_frames,
                       void* workspace, size_t workspace_bytes, void* stream);

/* gdn_host_workspace_bytes -- device workspace gdn_frame_fwd_host needs (0 for
 * arguments it rejects). */
size_t gdn_host_workspace_bytes(int B, int H, int T, int S, int D, int dtype, int chunk_frames);

/*
 * Context parallelism over frames (zhichai.net SANA-WM summary, training pipeline
 * Stage 3: the latent sequence is split across GPUs and the GDN transition maps
 * are composed by prefix sums, exactly).  Per head, a range of frames maps any
 * state S entering it to
 *     A S + b,   A = A_{T-1} ... A_1 A_0,   A_t = g_t (I - K~_t^T diag(beta_t) K~_t),
 * with b the state the range produces from a zero initial state.  A rank holding
 * frames [t0, t1) of a sequence computes its range's (A, b) with
 * gdn_frame_summary, the ranks exchange them (2 D^2 floats per head), each rank
 * folds the maps of the ranges before its own onto the sequence's initial state
 * with gdn_summary_apply, and then runs gdn_frame_fwd_ex on its frames from that
 * state: its outputs are those of one call over the whole sequence up to
 * rounding (the replayed frames take the same arithmetic; only the entering
 * state is reached through composed maps).
 */

/* Flags of gdn_frame_summary. */
#define GDN_SUMMARY_GATE_LOGITS 1 /* g and beta are logits (as gdn_frame_fwd_from_logits) */

/*
 * gdn_frame_summary -- the affine map (A, b) the T frames of every head apply to
 * the state.
 *   k, v, g, beta : as gdn_frame_fwd (q takes no part); with
 *                   GDN_SUMMARY_GATE_LOGITS, g and beta are logits.
 *   A_out, b_out  : [B, H, D, D] float32 each, written: A_out[i][j] maps key
 *                   dim j of the entering state to key dim i of the leaving one;
 *                   b_out is laid out as a state.  T = 0 gives A = I, b = 0.
 *   workspace     : device memory of gdn_summary_workspace_bytes() bytes,
 *                   256-byte aligned, owned by the caller (not read before it is
 *                   written).
 * The frames are cut into chunks of 16 whose maps are formed in parallel (for
 * GDN_BF16 on the tensor cores, as the prefix form's summaries; for GDN_F32 on
 * CUDA cores) and then composed in float32.  Returns GDN_OK, GDN_ERR_INVALID_ARG
 * (bad counts, NULL pointers, unknown flags), GDN_ERR_UNSUPPORTED (D),
 * GDN_ERR_MISALIGNED, GDN_ERR_WORKSPACE or GDN_ERR_CUDA; device-side timeouts
 * through gdn_last_error.
 */
int gdn_frame_summary(const void* k, const void* v, const float* g, const float* beta,
                      float* A_out, float* b_out,
                      int B, int H, int T, int S, int D, int dtype, int flags,
                      void* workspace, size_t workspace_bytes, void* stream);

/* gdn_summary_workspace_bytes -- workspace gdn_frame_summary needs (0 for T = 0
 * and for arguments it rejects). */
size_t gdn_summary_workspace_bytes(int B, int H, int T, int S, int D, int dtype);

/*
 * gdn_summary_apply -- state_out = A state_in + b for every head, in float32:
 * the state after a range of frames whose map gdn_frame_summary returned.
 *   A, b      : [B, H, D, D] float32 (device).
 *   state_in  : [B, H, D, D] float32, or NULL (zeros: state_out = b).
 *   state_out : [B, H, D, D] float32, written; may alias state_in (each
 *               head's block is read before it is written), not A or b.
 * All pointers 16-byte aligned.  Returns GDN_OK, GDN_ERR_INVALID_ARG,
 * GDN_ERR_UNSUPPORTED (D), GDN_ERR_MISALIGNED or GDN_ERR_CUDA.
 */
int gdn_summary_apply(const float* A, const float* b, const float* state_in, float* state_out,
                      int B, int H, int D, void* stream);

/*
 * gdn_last_error -- synchronises `stream`, then returns and clears the
 * device-side status word: GDN_OK, GDN_ERR_TIMEOUT (a kernel's bounded wait on
 * an mbarrier or a flag gave up; its results are invalid), GDN_ERR_BOUNDS (the
 * debug build's index check failed), or GDN_ERR_CUDA (the stream reported an
 * error).  The first error recorded since the last call wins.
 */
int gdn_last_error(void* stream);

/*
 * gdn_selftest_wait_timeout -- exercises the library's failure detection without
 * a fault (no counterpart on the pages).  Enqueues on `stream` one kernel whose
 * thread waits, with the bounded wait every kernel here uses, on a barrier that
 * nothing arrives on; after timeout_us microseconds (1 .. 10,000,000) it gives
 * up, records GDN_ERR_TIMEOUT in the device status word and returns normally.
 * The next gdn_last_error(stream) then reports GDN_ERR_TIMEOUT (and clears it),
 * and the context stays usable.  Returns GDN_OK, GDN_ERR_INVALID_ARG (timeout out
 * of range) or GDN_ERR_CUDA.
 */
int gdn_selftest_wait_timeout(unsigned int timeout_us, void* stream);

/* gdn_status_string -- a static, human-readable name for a status code. */
const char* gdn_status_string(int status);

/* gdn_version -- library version as major * 10000 + minor * 100 + patch. */
int gdn_version(void);

/*
 * gdn_frame_fwd_noalloc -- gdn_frame_fwd for callers that cannot allocate
 * device memory.  (No counterpart on the pages: this is a property of the
 * library, not of the method.)
 *
 * Some callers cannot call cudaMalloc: code plugged into another runtime whose
 * caching allocator already owns the GPU's memory (a raw cudaMalloc would fail
 * or fragment that pool), and latency-critical loops in which an allocation or
 * a free that synchronises the device would stall other streams.  This entry
 * point takes the same arguments as gdn_frame_fwd and runs the split form
 * (GDN_MODE_SPLIT, the form whose kernels use scratch memory), but it calls no
 * cudaMalloc, cudaFree or other allocating routine: its scratch is one fixed
 * array of gdn_noalloc_scratch_bytes() bytes (64 MiB) in the library's own
 * device memory.  The array sits in a module of its own: with CUDA's lazy
 * module loading (the default) a device reserves it when this entry point is
 * first called there, and holds it until the process exits; with eager loading
 * (CUDA_MODULE_LOADING=EAGER) every device the process uses reserves it when its
 * context is created.  So make the first call before a caching allocator has
 * taken the rest of the memory, or load eagerly.
 *   - Shapes whose scratch (gdn_workspace_bytes(..., GDN_MODE_SPLIT)) is
 *     larger than that are rejected with GDN_ERR_WORKSPACE before any CUDA call.
 *     At D = 112 that is about 490 frame-heads per call, e.g. 20 heads
 *     x 24 frames: chunk-causal rollouts of a few frames per call fit.
 *   - The first call on a device (and after a device reset, the first call in
 *     the new context) loads the array's module and looks up its device
 *     address with that device current, then caches it; make that first call
 *     before any stream capture.
 *   - Every call, on every stream, shares the one array, and it keeps the last
 *     call's contents (each call writes its scratch before reading it, so nothing
 *     needs clearing).  Calls that overlap on the GPU race on it: serialise them
 *     (one stream, or events between streams).
 * Returns as gdn_frame_fwd.
 */
int gdn_frame_fwd_noalloc(const void* q, const void* k, const void* v,
                          const float* g, const float* beta, const float* state_in,
                          void* out, float* state_out,
                          int B, int H, int T, int S, int D, int dtype, void* stream);

/* gdn_noalloc_scratch_bytes -- size of gdn_frame_fwd_noalloc's fixed scratch. */
size_t gdn_noalloc_scratch_bytes(void);

/*
 * Per-kernel timing (a tracing aid; no counterpart on the pages).
 * Between gdn_profile_begin() and gdn_profile_end(), every kernel launch the
 * library makes in this process is bracketed by two CUDA events recorded on
 * the launch stream.  gdn_profile_end() waits for those events, aggregates the
 * device time per kernel name into `stats` (at most `max_stats` entries, the
 * count in *n_stats) and stops recording.  Host-side cost: two event records
 * per launch.  Returns GDN_OK, GDN_ERR_INVALID_ARG (NULL n_stats or stats with
 * max_stats > 0) or GDN_ERR_CUDA.
 */
typedef struct {
  char name[32];   /* kernel name, NUL-terminated */
  int launches;    /* launches recorded */
  double total_ms; /* summed device time between each launch's two events */
} gdn_kernel_stat_t;

int gdn_profile_begin(void);
int gdn_profile_end(gdn_kernel_stat_t* stats, int max_stats, int* n_stats);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
