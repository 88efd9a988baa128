"""C-ABI checks that need no GPU: the library builds and loads, exports every
function include/gdn.h declares, and rejects bad arguments on the host before
any CUDA call is made."""
import os
import re
import subprocess

import pytest

from linear_attention_video_gated_b300 import binding, build_lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include")))
           if f.endswith(".h")]

# Fake, never-dereferenced device addresses: every call below fails validation
# before the library touches CUDA.
A16 = 0x10000
MIS = 0x10002


@pytest.fixture(scope="module")
def lib():
    build_lib.build()
    return binding.lib()


def declared_functions():
    names = []
    for h in HEADERS:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w \*]*?\b(gdn_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("gdn_frame_fwd", "gdn_frame_fwd_ex", "gdn_workspace_bytes", "gdn_last_error",
                     "gdn_status_string"):
        assert required in names


@pytest.mark.parametrize("debug", [False, True], ids=["release", "debug"])
def test_library_exports_every_declared_symbol(lib, debug):
    path = binding.DEBUG_LIB_PATH if debug else binding.LIB_PATH
    if debug:
        build_lib.build(debug=True)
    handle = binding.debug_lib() if debug else lib
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (gdn_\w+)$", out, flags=re.M))
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(handle, name)


def test_status_strings(lib):
    for code, name in binding.STATUS.items():
        assert binding.gdn_status_string(code) == name
    assert binding.gdn_status_string(99) == "GDN_ERR_UNKNOWN"
    assert binding.gdn_version() >= 100


def _call(B=1, H=2, T=3, S=17, D=32, dtype=1, ptr=A16, g=A16, beta=A16, out=A16, state_in=None, state_out=None,
          mode=0, ws=A16, wsb=1 << 40):
    return binding.gdn_frame_fwd_ex(ptr, ptr, ptr, g, beta, state_in, out, state_out, B, H, T, S, D, dtype, mode,
                                    ws, wsb, None)


@pytest.mark.parametrize("kw,code", [
    (dict(B=0), 1), (dict(H=0), 1), (dict(T=-1), 1), (dict(S=0), 1), (dict(D=0), 1),
    (dict(dtype=2), 1), (dict(mode=4), 1), (dict(mode=-1), 1), (dict(mode=3), 1), (dict(mode=3, dtype=0), 1),
    (dict(D=24), 2), (dict(D=144), 2), (dict(D=8), 2),
    (dict(ptr=None), 1), (dict(g=None), 1), (dict(beta=None), 1), (dict(out=None), 1),
    (dict(ptr=MIS), 3), (dict(out=MIS), 3), (dict(g=A16 + 2), 3), (dict(state_in=MIS), 3),
    (dict(state_out=MIS), 3),
    (dict(ws=None, mode=2), 6), (dict(wsb=16, mode=2), 6), (dict(ws=A16 + 16, mode=2), 3),
    (dict(ws=None, mode=1), 6), (dict(ws=None, dtype=0), 6),
])
def test_validation_rejects(lib, kw, code):
    assert _call(**kw) == code


def test_validation_rejects_plain_entry(lib):
    assert binding.gdn_frame_fwd(A16, A16, A16, A16, A16, None, A16, None, 1, 1, 1, 1, 24, 1, None) == 2
    assert binding.gdn_frame_fwd(None, A16, A16, A16, A16, None, A16, None, 1, 1, 1, 1, 32, 1, None) == 1


def test_workspace_bytes_is_pure_and_scales(lib):
    a = binding.gdn_workspace_bytes(1, 20, 961, 880, 112, 1, 2)
    assert a > 0 and a == binding.gdn_workspace_bytes(1, 20, 961, 880, 112, 1, 2)
    assert binding.gdn_workspace_bytes(1, 20, 0, 880, 112, 1, 2) == 0
    assert binding.gdn_workspace_bytes(1, 20, 961, 880, 24, 1, 2) == 0
    assert binding.gdn_workspace_bytes(1, 20, 961, 880, 112, 1, 1) >= a
    assert binding.gdn_workspace_bytes(2, 20, 961, 880, 112, 1, 2) >= a
    assert binding.gdn_workspace_bytes(1, 2, 8, 16, 16, 0, 0) > 0


@pytest.mark.parametrize("D", [16, 32, 48, 64, 80, 96, 112, 128])
def test_every_form_needs_a_workspace_and_no_mode_3(lib, D):
    """Modes 0-2 need scratch; mode 3 (no such form) is rejected: 0 bytes, and
    GDN_ERR_INVALID_ARG from the entry points (test_host_validation)."""
    for mode in (0, 1, 2):
        assert binding.gdn_workspace_bytes(4, 16, 241, 3600, D, 1, mode) > 0
    assert binding.gdn_workspace_bytes(4, 16, 241, 3600, D, 1, 3) == 0


def test_no_gpu_call_fails_loudly_not_silently(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("GPU present")
    # with no device, a valid-looking call must report a CUDA error, never succeed
    assert binding.gdn_last_error(None) == 4


def _host(B=1, H=2, T=3, S=17, D=32, dtype=1, chunk=2, ptr=A16, ws=A16, wsb=1 << 40):
    return binding.gdn_frame_fwd_host(ptr, ptr, ptr, ptr, ptr, None, ptr, None, B, H, T, S, D, dtype, chunk, ws, wsb,
                                      None)


@pytest.mark.parametrize("kw,code", [
    (dict(chunk=0), 1), (dict(chunk=-3), 1), (dict(B=0), 1), (dict(T=-1), 1), (dict(dtype=7), 1),
    (dict(D=24), 2), (dict(D=144), 2), (dict(ptr=None), 1),
    (dict(ws=None), 6), (dict(wsb=16), 6), (dict(ws=A16 + 16), 3),
])
def test_host_entry_validation_rejects(lib, kw, code):
    assert _host(**kw) == code


def test_host_workspace_bytes(lib):
    a = binding.gdn_host_workspace_bytes(1, 20, 961, 880, 112, 1, 32)
    assert a > 0 and a == binding.gdn_host_workspace_bytes(1, 20, 961, 880, 112, 1, 32)
    # two chunk buffers of q, k, v, out dominate: grows with the chunk, capped by T
    assert binding.gdn_host_workspace_bytes(1, 20, 961, 880, 112, 1, 64) > a
    assert binding.gdn_host_workspace_bytes(1, 20, 10, 880, 112, 1, 64) == \
        binding.gdn_host_workspace_bytes(1, 20, 10, 880, 112, 1, 10)
    assert binding.gdn_host_workspace_bytes(1, 20, 961, 880, 112, 1, 0) == 0
    assert binding.gdn_host_workspace_bytes(1, 20, 961, 880, 24, 1, 32) == 0


def _bwd(B=1, H=2, T=3, S=17, D=32, dtype=1, ptr=A16, dout=A16, dq=A16, dk=A16, dv=A16, dg=A16, dbeta=A16,
         dstate_out=None, dstate_in=None, state_in=None, ws=A16, wsb=1 << 40, logits=False):
    fn = binding.gdn_frame_bwd_from_logits if logits else binding.gdn_frame_bwd
    return fn(ptr, ptr, ptr, ptr, ptr, state_in, dout, dstate_out, dq, dk, dv, dg, dbeta, dstate_in,
              B, H, T, S, D, dtype, ws, wsb, None)


@pytest.mark.parametrize("logits", [False, True])
@pytest.mark.parametrize("kw,code", [
    (dict(B=0), 1), (dict(T=-1), 1), (dict(S=0), 1), (dict(dtype=3), 1), (dict(D=24), 2), (dict(D=144), 2),
    (dict(ptr=None), 1), (dict(dout=None), 1), (dict(dq=None), 1), (dict(dk=None), 1), (dict(dv=None), 1),
    (dict(dg=None), 1), (dict(dbeta=None), 1),
    (dict(dout=MIS), 3), (dict(dq=MIS), 3), (dict(dk=MIS), 3), (dict(dv=MIS), 3), (dict(dg=A16 + 2), 3),
    (dict(dbeta=A16 + 1), 3), (dict(dstate_out=MIS), 3), (dict(dstate_in=MIS), 3), (dict(state_in=MIS), 3),
    (dict(ws=None), 6), (dict(wsb=16), 6), (dict(ws=A16 + 16), 3),
])
def test_backward_validation_rejects(lib, kw, code, logits):
    assert _bwd(logits=logits, **kw) == code


def test_backward_zero_frames_needs_no_gradient_outputs(lib):
    """T = 0 with no dstate_in: nothing to compute, nothing touched, no CUDA call."""
    assert _bwd(T=0, ptr=None, dout=None, dq=None, dk=None, dv=None, dg=None, dbeta=None, ws=None) == 0


def test_backward_workspace_bytes(lib):
    a = binding.gdn_bwd_workspace_bytes(1, 20, 961, 880, 112, 1)
    f = binding.gdn_bwd_workspace_bytes(1, 20, 961, 880, 112, 0)
    # float32 I/O: four D x D float32 matrices per frame-head plus one float per 32-token tile
    assert f >= 4 * 20 * 961 * 112 * 112 * 4 + 20 * 961 * 28 * 4
    # bf16 I/O: the M_t image, the E_t blocks and the S_t and U_t images (bf16 hi + lo)
    assert a >= 20 * 961 * (2 * 112 * 128 + 112 * 112 * 4 + 2 * 4 * 112 * 128)
    assert a == binding.gdn_bwd_workspace_bytes(1, 20, 961, 880, 112, 1)
    assert binding.gdn_bwd_workspace_bytes(1, 20, 0, 880, 112, 1) == 0
    assert binding.gdn_bwd_workspace_bytes(1, 20, 961, 880, 24, 1) == 0
    assert binding.gdn_bwd_workspace_bytes(1, 20, 961, 880, 112, 5) == 0
    assert binding.gdn_bwd_workspace_bytes(2, 20, 961, 880, 112, 1) > a


@pytest.mark.parametrize("flags", [4, 8, -1, 1 << 30])
def test_backward_ex_rejects_unknown_flags(lib, flags):
    assert binding.gdn_frame_bwd_ex(A16, A16, A16, A16, A16, None, A16, None, A16, A16, A16, A16, A16, None,
                                    1, 2, 3, 17, 32, 1, flags, A16, 1 << 40, None) == 1


def test_backward_workspace_holds_the_forward_scratch(lib):
    """The backward's workspace is never smaller than the forward's (sequential form),
    so one buffer serves a training step's forward and backward."""
    for dtype in (0, 1):
        for shape in ((1, 20, 961, 880, 112), (2, 3, 7, 129, 16), (4, 16, 241, 3600, 128)):
            assert binding.gdn_bwd_workspace_bytes(*shape, dtype) >= binding.gdn_workspace_bytes(*shape, dtype, 0)
            if dtype == 1:
                assert binding.gdn_bwd_workspace_bytes(*shape, dtype) >= binding.gdn_workspace_bytes(*shape, 1, 2)
