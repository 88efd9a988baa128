"""The debug build, libgdn_debug.so (compiled with -DGDN_DEBUG=1): every kernel
checks each scratch offset it computes against the extent of its region in the
host's workspace layout, and reports GDN_ERR_BOUNDS through gdn_last_error
instead of touching memory outside it.  On the tiny and odd shapes, in every
algorithm form and in the backward pass, no check fires and the results are
bit for bit those of the release library (the checks change no arithmetic).
With GDN_DEBUG_SHRINK the host reports the read-out's image region one frame-head
image short, and the check on the last frame-head fires (its copy is skipped,
nothing outside the workspace is touched, the bounded wait on it gives up)."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from linear_attention_video_gated_b300 import binding, build_lib, synth
from tests import parity

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _libs():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_lib.ensure_built()
    build_lib.ensure_built(debug=True)


def _fwd(handle, ins, S0, mode, ws):
    q, k, v, g, beta = ins
    B, H, T, S, D = q.shape
    dtype = binding.GDN_BF16 if q.dtype == torch.bfloat16 else binding.GDN_F32
    out = torch.full_like(q, float("nan"))
    st = torch.full((B, H, D, D), float("nan"), device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    rc = handle.gdn_frame_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), g.data_ptr(), beta.data_ptr(),
                                 None if S0 is None else S0.data_ptr(), out.data_ptr(), st.data_ptr(), B, H, T, S,
                                 D, dtype, mode, ws.data_ptr(), ws.numel(), stream)
    assert rc == 0
    return out, st, handle.gdn_last_error(stream)


SHAPES = [("bf16", 1, 1, 1, 1, 16, False), ("bf16", 1, 2, 5, 17, 32, True), ("bf16", 2, 1, 4, 129, 48, False),
          ("bf16", 1, 1, 17, 200, 96, True), ("bf16", 1, 1, 33, 64, 128, False), ("bf16", 1, 3, 6, 880, 112, True),
          ("f32", 2, 2, 5, 33, 128, True), ("f32", 1, 1, 20, 7, 64, False)]


@pytest.mark.parametrize("case", SHAPES, ids=lambda c: "-".join(map(str, c)))
def test_debug_build_checks_pass_and_change_nothing(case):
    dt, B, H, T, S, D, nz = case
    wl = synth.WORKLOADS["short" if dt == "bf16" else "tiny"].with_(B=B, H=H, T=T, S=S, D=D, seed=9700 + S + D)
    x = synth.full(wl)
    ins = parity.upload(wl, x)
    S0 = (torch.from_numpy(np.stack([np.stack([synth.state(wl, b, h, 0.3) for h in range(H)]) for b in range(B)]))
          .cuda() if nz else None)
    dbg, rel = binding.debug_lib(), binding.lib()
    for mode in (0, 1, 2):
        need = binding.gdn_workspace_bytes(B, H, T, S, D, binding.GDN_BF16 if dt == "bf16" else binding.GDN_F32,
                                           mode)
        ws = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")
        o1, s1, rc1 = _fwd(dbg, ins, S0, mode, ws)
        o2, s2, rc2 = _fwd(rel, ins, S0, mode, ws)
        assert rc1 == 0, f"debug build, mode {mode}: {binding.STATUS.get(rc1, rc1)}"
        assert rc2 == 0
        assert torch.equal(o1, o2) and torch.equal(s1, s2), f"mode {mode}"
    # backward: the debug build's gradients equal the release library's
    if dt == "bf16":
        q, k, v, g, beta = ins
        dout = torch.from_numpy(synth.full_grads(wl)["dout"]).cuda().to(q.dtype).contiguous()
        grads = {}
        for name, handle in (("debug", dbg), ("release", rel)):
            res = [torch.full_like(q, float("nan")) for _ in range(3)]
            dg = torch.full((B, H, T), float("nan"), device="cuda")
            dbeta = torch.full((B, H, T, S), float("nan"), device="cuda")
            ds0 = torch.full((B, H, D, D), float("nan"), device="cuda")
            need = binding.gdn_bwd_workspace_bytes(B, H, T, S, D, binding.GDN_BF16)
            ws = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")
            stream = torch.cuda.current_stream().cuda_stream
            rc = handle.gdn_frame_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), g.data_ptr(), beta.data_ptr(),
                                      None if S0 is None else S0.data_ptr(), dout.data_ptr(), None,
                                      res[0].data_ptr(), res[1].data_ptr(), res[2].data_ptr(), dg.data_ptr(),
                                      dbeta.data_ptr(), ds0.data_ptr(), B, H, T, S, D, binding.GDN_BF16,
                                      ws.data_ptr(), need, stream)
            assert rc == 0
            assert handle.gdn_last_error(stream) == 0, name
            grads[name] = res + [dg, dbeta, ds0]
        for a, b in zip(grads["debug"], grads["release"]):
            assert torch.equal(a, b)


_SHRINK = r"""
import sys, torch
sys.path.insert(0, {root!r})
from linear_attention_video_gated_b300 import binding, synth
from tests import parity
wl = synth.WORKLOADS["short"].with_(H=2, T=3, S=100, D=32, seed=9800)
ins = parity.upload(wl, synth.full(wl))
q, k, v, g, beta = ins
h = binding.debug_lib()
need = binding.gdn_workspace_bytes(1, 2, 3, 100, 32, binding.GDN_BF16, 0)
ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
out = torch.empty_like(q)
s = torch.cuda.current_stream().cuda_stream
rc = h.gdn_frame_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), g.data_ptr(), beta.data_ptr(), None,
                        out.data_ptr(), None, 1, 2, 3, 100, 32, binding.GDN_BF16, 0, ws.data_ptr(), need, s)
print("rc", rc, "status", h.gdn_last_error(s))
# the context is still usable
x = torch.ones(4, device="cuda"); torch.cuda.synchronize(); print("after", float(x.sum()))
"""


def test_a_failed_check_reports_bounds_without_touching_memory():
    """One frame-head image short (hi + lo of a d32 state, 8 KB): the read-out's check
    on the last frame-head fails, GDN_ERR_BOUNDS is reported, the process's CUDA
    context stays usable."""
    env = dict(os.environ, GDN_DEBUG_SHRINK=str(2 * 1 * 32 * 128))
    res = subprocess.run([sys.executable, "-c", _SHRINK.format(root=ROOT)], capture_output=True, text=True, env=env,
                         timeout=300, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    assert "rc 0 status 7" in res.stdout, res.stdout
    assert "after 4.0" in res.stdout
