"""Thin Python binding of libgdn's C ABI (include/gdn.h).

Argument marshalling only: every step of the forward scan runs in the library's
CUDA kernels.  The raw functions take integer device addresses; ``frame_fwd``
additionally accepts torch tensors (torch is used for device memory and
streams only).  There is no fallback: if ``libgdn.so`` is missing or fails to
load, every call raises.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libgdn.so")
DEBUG_LIB_PATH = os.path.join(PKG, "libgdn_debug.so")

GDN_F32, GDN_BF16 = 0, 1
GDN_BWD_STATES_IN_WORKSPACE, GDN_BWD_GATE_LOGITS = 1, 2
GDN_SUMMARY_GATE_LOGITS = 1
GDN_MODE_SEQUENTIAL, GDN_MODE_PREFIX, GDN_MODE_SPLIT = 0, 1, 2
STATUS = {0: "GDN_OK", 1: "GDN_ERR_INVALID_ARG", 2: "GDN_ERR_UNSUPPORTED", 3: "GDN_ERR_MISALIGNED",
          4: "GDN_ERR_CUDA", 5: "GDN_ERR_TIMEOUT", 6: "GDN_ERR_WORKSPACE", 7: "GDN_ERR_BOUNDS"}

_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_SIGS = {
    "gdn_frame_fwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P]),
    "gdn_frame_fwd_ex": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P,
                              ctypes.c_size_t, _P]),
    "gdn_frame_fwd_from_logits": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P,
                                       ctypes.c_size_t, _P]),
    "gdn_workspace_bytes": (ctypes.c_size_t, [_I, _I, _I, _I, _I, _I, _I]),
    "gdn_relu_linear_fwd": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, ctypes.c_size_t, _P]),
    "gdn_frame_fwd_host": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, ctypes.c_size_t,
                                _P]),
    "gdn_host_workspace_bytes": (ctypes.c_size_t, [_I, _I, _I, _I, _I, _I, _I]),
    "gdn_frame_fwd_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P]),
    "gdn_noalloc_scratch_bytes": (ctypes.c_size_t, []),
    "gdn_frame_bwd": (_I, [_P] * 14 + [_I] * 6 + [_P, ctypes.c_size_t, _P]),
    "gdn_frame_bwd_from_logits": (_I, [_P] * 14 + [_I] * 6 + [_P, ctypes.c_size_t, _P]),
    "gdn_bwd_workspace_bytes": (ctypes.c_size_t, [_I, _I, _I, _I, _I, _I]),
    "gdn_frame_bwd_ex": (_I, [_P] * 14 + [_I] * 7 + [_P, ctypes.c_size_t, _P]),
    "gdn_frame_summary": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, ctypes.c_size_t, _P]),
    "gdn_summary_workspace_bytes": (ctypes.c_size_t, [_I, _I, _I, _I, _I, _I]),
    "gdn_summary_apply": (_I, [_P, _P, _P, _P, _I, _I, _I, _P]),
    "gdn_last_error": (_I, [_P]),
    "gdn_selftest_wait_timeout": (_I, [ctypes.c_uint, _P]),
    "gdn_status_string": (ctypes.c_char_p, [_I]),
    "gdn_version": (_I, []),
    "gdn_profile_begin": (_I, []),
    "gdn_profile_end": (_I, [_P, _I, ctypes.POINTER(_I)]),
}


class KernelStat(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 32), ("launches", ctypes.c_int), ("total_ms", ctypes.c_double)]


class GDNError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)}")


def _load(path) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with __graft_entry__.build()")
    handle = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(handle, name)
        fn.restype = res
        fn.argtypes = args
    return handle


def lib() -> ctypes.CDLL:
    """Loads libgdn.so (once).  Raises if it is not built."""
    global _lib
    if _lib is None:
        _lib = _load(LIB_PATH)
    return _lib


_debug_lib = None


def debug_lib() -> ctypes.CDLL:
    """Loads the debug build, libgdn_debug.so (once): the same entry points, with
    every kernel's scratch offsets checked (GDN_ERR_BOUNDS).  Its status word and
    module state are its own; call its functions through the returned handle."""
    global _debug_lib
    if _debug_lib is None:
        _debug_lib = _load(DEBUG_LIB_PATH)
    return _debug_lib


# ---- raw C-ABI calls (integer device addresses) ------------------------------------

def gdn_frame_fwd(q, k, v, g, beta, state_in, out, state_out, B, H, T, S, D, dtype, stream) -> int:
    return lib().gdn_frame_fwd(q, k, v, g, beta, state_in, out, state_out, B, H, T, S, D, dtype, stream)


def gdn_frame_fwd_ex(q, k, v, g, beta, state_in, out, state_out, B, H, T, S, D, dtype, mode,
                     workspace, workspace_bytes, stream) -> int:
    return lib().gdn_frame_fwd_ex(q, k, v, g, beta, state_in, out, state_out, B, H, T, S, D, dtype, mode,
                                  workspace, workspace_bytes, stream)


def gdn_frame_fwd_from_logits(q, k, v, g_logit, beta_logit, state_in, out, state_out, B, H, T, S, D, dtype, mode,
                              workspace, workspace_bytes, stream) -> int:
    return lib().gdn_frame_fwd_from_logits(q, k, v, g_logit, beta_logit, state_in, out, state_out, B, H, T, S, D,
                                           dtype, mode, workspace, workspace_bytes, stream)


def gdn_frame_fwd_host(q, k, v, g, beta, state_in, out, state_out, B, H, T, S, D, dtype, chunk_frames,
                       workspace, workspace_bytes, stream) -> int:
    return lib().gdn_frame_fwd_host(q, k, v, g, beta, state_in, out, state_out, B, H, T, S, D, dtype, chunk_frames,
                                    workspace, workspace_bytes, stream)


def gdn_host_workspace_bytes(B, H, T, S, D, dtype, chunk_frames) -> int:
    return lib().gdn_host_workspace_bytes(B, H, T, S, D, dtype, chunk_frames)


def gdn_relu_linear_fwd(q, k, v, state_in, out, state_out, B, H, T, S, D, dtype, mode, workspace, workspace_bytes,
                        stream) -> int:
    return lib().gdn_relu_linear_fwd(q, k, v, state_in, out, state_out, B, H, T, S, D, dtype, mode, workspace,
                                     workspace_bytes, stream)


def gdn_frame_fwd_noalloc(q, k, v, g, beta, state_in, out, state_out, B, H, T, S, D, dtype, stream) -> int:
    return lib().gdn_frame_fwd_noalloc(q, k, v, g, beta, state_in, out, state_out, B, H, T, S, D, dtype, stream)


def gdn_noalloc_scratch_bytes() -> int:
    return lib().gdn_noalloc_scratch_bytes()


def gdn_frame_bwd(q, k, v, g, beta, state_in, dout, dstate_out, dq, dk, dv, dg, dbeta, dstate_in, B, H, T, S, D,
                  dtype, workspace, workspace_bytes, stream) -> int:
    return lib().gdn_frame_bwd(q, k, v, g, beta, state_in, dout, dstate_out, dq, dk, dv, dg, dbeta, dstate_in, B, H,
                               T, S, D, dtype, workspace, workspace_bytes, stream)


def gdn_frame_bwd_from_logits(q, k, v, g_logit, beta_logit, state_in, dout, dstate_out, dq, dk, dv, dg_logit,
                              dbeta_logit, dstate_in, B, H, T, S, D, dtype, workspace, workspace_bytes,
                              stream) -> int:
    return lib().gdn_frame_bwd_from_logits(q, k, v, g_logit, beta_logit, state_in, dout, dstate_out, dq, dk, dv,
                                           dg_logit, dbeta_logit, dstate_in, B, H, T, S, D, dtype, workspace,
                                           workspace_bytes, stream)


def gdn_frame_bwd_ex(q, k, v, g, beta, state_in, dout, dstate_out, dq, dk, dv, dg, dbeta, dstate_in, B, H, T, S, D,
                     dtype, flags, workspace, workspace_bytes, stream) -> int:
    return lib().gdn_frame_bwd_ex(q, k, v, g, beta, state_in, dout, dstate_out, dq, dk, dv, dg, dbeta, dstate_in, B,
                                  H, T, S, D, dtype, flags, workspace, workspace_bytes, stream)


def gdn_bwd_workspace_bytes(B, H, T, S, D, dtype) -> int:
    return lib().gdn_bwd_workspace_bytes(B, H, T, S, D, dtype)


def gdn_workspace_bytes(B, H, T, S, D, dtype, mode) -> int:
    return lib().gdn_workspace_bytes(B, H, T, S, D, dtype, mode)


def gdn_frame_summary(k, v, g, beta, A_out, b_out, B, H, T, S, D, dtype, flags, workspace, workspace_bytes,
                      stream) -> int:
    return lib().gdn_frame_summary(k, v, g, beta, A_out, b_out, B, H, T, S, D, dtype, flags, workspace,
                                   workspace_bytes, stream)


def gdn_summary_workspace_bytes(B, H, T, S, D, dtype) -> int:
    return lib().gdn_summary_workspace_bytes(B, H, T, S, D, dtype)


def gdn_summary_apply(A, b, state_in, state_out, B, H, D, stream) -> int:
    return lib().gdn_summary_apply(A, b, state_in, state_out, B, H, D, stream)


def gdn_last_error(stream) -> int:
    return lib().gdn_last_error(stream)


def gdn_selftest_wait_timeout(timeout_us, stream) -> int:
    return lib().gdn_selftest_wait_timeout(timeout_us, stream)


def gdn_status_string(status: int) -> str:
    return lib().gdn_status_string(status).decode()


def gdn_version() -> int:
    return lib().gdn_version()


def gdn_profile_begin() -> int:
    return lib().gdn_profile_begin()


def gdn_profile_end(max_stats: int = 64) -> dict:
    """Stops per-kernel timing; returns {kernel name: (launches, total_ms)}."""
    arr = (KernelStat * max_stats)()
    n = ctypes.c_int(0)
    rc = lib().gdn_profile_end(ctypes.cast(arr, ctypes.c_void_p), max_stats, ctypes.byref(n))
    if rc != 0:
        raise GDNError(rc, "gdn_profile_end")
    return {arr[i].name.decode(): (arr[i].launches, arr[i].total_ms) for i in range(min(n.value, max_stats))}


# ---- torch marshalling -------------------------------------------------------------

def _ptr(t):
    return None if t is None else t.data_ptr()


def frame_fwd(q, k, v, g, beta, state_in=None, out=None, state_out=None, mode=None,
              workspace=None, stream=None, want_state=True, gate_logits=False):
    """Runs the forward scan on torch CUDA tensors through the C ABI.

    q, k, v: [B,H,T,S,D] float32 or bfloat16, contiguous; g: [B,H,T] float32;
    beta: [B,H,T,S] float32; state_in: [B,H,D,D] float32 or None.  ``out`` and
    ``state_out`` are allocated if not given (state_out only if want_state).
    mode=None calls gdn_frame_fwd (library-managed scratch); mode=0/1/2
    (sequential, prefix, split) calls gdn_frame_fwd_ex with ``workspace``
    (a uint8 CUDA tensor, allocated if None).
    gate_logits=True passes g and beta as raw logits to gdn_frame_fwd_from_logits
    (mode None then means the sequential form).
    Returns (out, state_out).  Raises GDNError on a non-zero status.
    """
    import torch

    B, H, T, S, D = q.shape
    dtype = {torch.float32: GDN_F32, torch.bfloat16: GDN_BF16}[q.dtype]
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.shape != q.shape or t.dtype != q.dtype or not t.is_contiguous() or not t.is_cuda:
            raise ValueError(f"{name}: expected a contiguous CUDA tensor like q")
    if g.dtype != torch.float32 or beta.dtype != torch.float32:
        raise ValueError("g and beta must be float32")
    if tuple(g.shape) != (B, H, T) or tuple(beta.shape) != (B, H, T, S):
        raise ValueError("g must be [B,H,T] and beta [B,H,T,S]")
    if not g.is_contiguous() or not beta.is_contiguous():
        raise ValueError("g and beta must be contiguous")
    if state_in is not None and (tuple(state_in.shape) != (B, H, D, D) or state_in.dtype != torch.float32
                                 or not state_in.is_contiguous()):
        raise ValueError("state_in must be a contiguous float32 [B,H,D,D] tensor")
    if out is None:
        out = torch.empty_like(q)
    if state_out is None and want_state:
        state_out = torch.empty((B, H, D, D), dtype=torch.float32, device=q.device)
    cur = torch.cuda.current_stream(q.device)
    strm = stream if stream is not None else cur
    st = strm.cuda_stream
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state_in), _ptr(out), _ptr(state_out),
            B, H, T, S, D, dtype)
    if gate_logits and mode is None:
        mode = GDN_MODE_SEQUENTIAL
    if mode is None:
        rc = gdn_frame_fwd(*args, st)
    else:
        need = gdn_workspace_bytes(B, H, T, S, D, dtype, mode)
        if workspace is None and need > 0:
            # allocated on the current stream; keep it alive for `strm` too
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
            if strm != cur:
                workspace.record_stream(strm)
        wbytes = 0 if workspace is None else workspace.numel()
        fn = gdn_frame_fwd_from_logits if gate_logits else gdn_frame_fwd_ex
        rc = fn(*args, mode, _ptr(workspace), wbytes, st)
    if rc != 0:
        raise GDNError(rc, "gdn_frame_fwd")
    return out, state_out


def frame_fwd_host(q, k, v, g, beta, state_in=None, chunk_frames=32, workspace=None, stream=None, out=None,
                   state_out=None):
    """gdn_frame_fwd_host on torch CPU tensors (pinned for overlap): q, k, v
    [B,H,T,S,D] float32 or bfloat16, g [B,H,T], beta [B,H,T,S], state_in [B,H,D,D]
    or None.  ``workspace`` is a uint8 CUDA tensor (allocated if None).  Waits for
    the stream and returns (out, state_out) as CPU tensors."""
    import torch

    B, H, T, S, D = q.shape
    dtype = {torch.float32: GDN_F32, torch.bfloat16: GDN_BF16}[q.dtype]
    for t in (q, k, v, g, beta) + (() if state_in is None else (state_in,)):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("gdn_frame_fwd_host takes contiguous host tensors")
    if out is None:
        out = torch.empty(tuple(q.shape), dtype=q.dtype, pin_memory=q.is_pinned())
    if state_out is None:
        state_out = torch.empty((B, H, D, D), dtype=torch.float32, pin_memory=q.is_pinned())
    need = gdn_host_workspace_bytes(B, H, T, S, D, dtype, chunk_frames)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
    strm = stream if stream is not None else torch.cuda.current_stream()
    rc = gdn_frame_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state_in), _ptr(out),
                            _ptr(state_out), B, H, T, S, D, dtype, chunk_frames, _ptr(workspace),
                            workspace.numel(), strm.cuda_stream)
    if rc != 0:
        raise GDNError(rc, "gdn_frame_fwd_host")
    strm.synchronize()
    return out, state_out


def relu_linear_fwd(q, k, v, state_in=None, mode=GDN_MODE_SEQUENTIAL, workspace=None, stream=None):
    """gdn_relu_linear_fwd on torch CUDA tensors (layouts as frame_fwd).  Returns (out, state_out)."""
    import torch

    B, H, T, S, D = q.shape
    dtype = {torch.float32: GDN_F32, torch.bfloat16: GDN_BF16}[q.dtype]
    out = torch.empty_like(q)
    state_out = torch.empty((B, H, D, D), dtype=torch.float32, device=q.device)
    need = gdn_workspace_bytes(B, H, T, S, D, dtype, mode)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    strm = stream if stream is not None else torch.cuda.current_stream(q.device)
    rc = gdn_relu_linear_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(state_in), _ptr(out), _ptr(state_out), B, H, T, S, D,
                             dtype, mode, _ptr(workspace), 0 if workspace is None else workspace.numel(),
                             strm.cuda_stream)
    if rc != 0:
        raise GDNError(rc, "gdn_relu_linear_fwd")
    return out, state_out


def frame_summary(k, v, g, beta, gate_logits=False, workspace=None, stream=None):
    """gdn_frame_summary on torch CUDA tensors (k, v [B,H,T,S,D], g [B,H,T], beta
    [B,H,T,S]): returns (A, b), each [B,H,D,D] float32, the map the frames apply
    to the state, S -> A S + b."""
    import torch

    B, H, T, S, D = k.shape
    dtype = {torch.float32: GDN_F32, torch.bfloat16: GDN_BF16}[k.dtype]
    A = torch.empty((B, H, D, D), dtype=torch.float32, device=k.device)
    b = torch.empty_like(A)
    need = gdn_summary_workspace_bytes(B, H, T, S, D, dtype)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=k.device)
    strm = stream if stream is not None else torch.cuda.current_stream(k.device)
    rc = gdn_frame_summary(_ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(A), _ptr(b), B, H, T, S, D, dtype,
                           GDN_SUMMARY_GATE_LOGITS if gate_logits else 0, _ptr(workspace),
                           0 if workspace is None else workspace.numel(), strm.cuda_stream)
    if rc != 0:
        raise GDNError(rc, "gdn_frame_summary")
    return A, b


def summary_apply(A, b, state_in=None, state_out=None, stream=None):
    """gdn_summary_apply on torch CUDA tensors: state_out = A state_in + b per head
    ([B,H,D,D] float32; state_in None means zeros).  Returns state_out."""
    import torch

    B, H, D, _ = A.shape
    if state_out is None:
        state_out = torch.empty_like(b)
    strm = stream if stream is not None else torch.cuda.current_stream(A.device)
    rc = gdn_summary_apply(_ptr(A), _ptr(b), _ptr(state_in), _ptr(state_out), B, H, D, strm.cuda_stream)
    if rc != 0:
        raise GDNError(rc, "gdn_summary_apply")
    return state_out


def frame_bwd(q, k, v, g, beta, dout, state_in=None, dstate_out=None, gate_logits=False, workspace=None,
              stream=None, want_dstate_in=True, states_in_workspace=False):
    """gdn_frame_bwd_ex on torch CUDA tensors: the forward's inputs (layouts as
    frame_fwd), dout like q, and dstate_out [B,H,D,D] float32 or None.  Returns a
    dict of dq, dk, dv (dtype of q), dg [B,H,T], dbeta [B,H,T,S] and dstate_in
    [B,H,D,D] (None unless want_dstate_in); with gate_logits the dg and dbeta
    entries are the logits' gradients.  states_in_workspace: ``workspace`` holds
    what a frame_fwd call (mode 0 or 2) over the same inputs left in it."""
    import torch

    if states_in_workspace and workspace is None:
        raise ValueError("states_in_workspace needs the forward call's workspace")
    B, H, T, S, D = q.shape
    dtype = {torch.float32: GDN_F32, torch.bfloat16: GDN_BF16}[q.dtype]
    for name, t in (("k", k), ("v", v), ("dout", dout)):
        if t.shape != q.shape or t.dtype != q.dtype or not t.is_contiguous() or not t.is_cuda:
            raise ValueError(f"{name}: expected a contiguous CUDA tensor like q")
    if tuple(g.shape) != (B, H, T) or tuple(beta.shape) != (B, H, T, S):
        raise ValueError("g must be [B,H,T] and beta [B,H,T,S]")
    out = {"dq": torch.empty_like(q), "dk": torch.empty_like(q), "dv": torch.empty_like(q),
           "dg": torch.empty((B, H, T), dtype=torch.float32, device=q.device),
           "dbeta": torch.empty((B, H, T, S), dtype=torch.float32, device=q.device),
           "dstate_in": torch.empty((B, H, D, D), dtype=torch.float32, device=q.device) if want_dstate_in else None}
    need = gdn_bwd_workspace_bytes(B, H, T, S, D, dtype)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    strm = stream if stream is not None else torch.cuda.current_stream(q.device)
    flags = (GDN_BWD_GATE_LOGITS if gate_logits else 0) | (GDN_BWD_STATES_IN_WORKSPACE if states_in_workspace else 0)
    rc = gdn_frame_bwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state_in), _ptr(dout),
                          _ptr(dstate_out), _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]), _ptr(out["dg"]),
                          _ptr(out["dbeta"]), _ptr(out["dstate_in"]), B, H, T, S, D, dtype, flags, _ptr(workspace),
                          0 if workspace is None else workspace.numel(), strm.cuda_stream)
    if rc != 0:
        raise GDNError(rc, "gdn_frame_bwd")
    return out


_FRAME_GDN = None


def _frame_gdn_function():
    """torch.autograd.Function over the forward and backward entry points (built
    on first use so that importing the binding does not import torch)."""
    global _FRAME_GDN
    if _FRAME_GDN is None:
        import torch

        class FrameGDN(torch.autograd.Function):
            @staticmethod
            def forward(ctx, q, k, v, g, beta, state_in, gate_logits):
                # the forward runs in a workspace sized for the backward, which then
                # reuses the per-frame states the forward left there
                B, H, T, S, D = q.shape
                dtype = {torch.float32: GDN_F32, torch.bfloat16: GDN_BF16}[q.dtype]
                need = gdn_bwd_workspace_bytes(B, H, T, S, D, dtype)
                ws = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
                out, st = frame_fwd(q, k, v, g, beta, state_in=state_in, mode=GDN_MODE_SEQUENTIAL,
                                    gate_logits=gate_logits, workspace=ws)
                ctx.save_for_backward(q, k, v, g, beta, state_in)
                ctx.gate_logits = gate_logits
                ctx.ws = ws if need > 0 else None
                return out, st

            @staticmethod
            def backward(ctx, dout, dstate):
                q, k, v, g, beta, state_in = ctx.saved_tensors
                res = frame_bwd(q, k, v, g, beta, dout.contiguous(), state_in=state_in,
                                dstate_out=dstate.contiguous(), gate_logits=ctx.gate_logits,
                                want_dstate_in=state_in is not None, workspace=ctx.ws,
                                states_in_workspace=ctx.ws is not None)
                ctx.ws = None
                return res["dq"], res["dk"], res["dv"], res["dg"], res["dbeta"], res["dstate_in"], None

        _FRAME_GDN = FrameGDN
    return _FRAME_GDN


def gdn(q, k, v, g, beta, state_in=None, gate_logits=False):
    """The scan as a differentiable torch op: (out, state_out) = gdn_frame_fwd(...),
    with gradients from gdn_frame_bwd (gdn_frame_*_from_logits when gate_logits).
    Layouts as frame_fwd; every input may require grad."""
    return _frame_gdn_function().apply(q, k, v, g, beta, state_in, gate_logits)

