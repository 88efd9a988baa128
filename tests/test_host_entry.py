"""gdn_frame_fwd_host: inputs and outputs in host memory, frames processed in
chunks with the copies overlapped with the kernels.  The chunked sequential form
does the same arithmetic per frame as one device call, so the two agree bit for
bit; these GPU tests check that on pinned and pageable buffers, with partial last
chunks, a carried initial state and T = 0."""
import numpy as np
import pytest
import torch

from linear_attention_video_gated_b300 import binding, build_lib, synth
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_lib.ensure_built()


def _host_inputs(wl, pinned):
    x = synth.full(wl)
    tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32

    def h(a, dt):
        t = torch.from_numpy(np.ascontiguousarray(a)).to(dt)
        return t.pin_memory() if pinned else t
    return x, h(x["q"], tdt), h(x["k"], tdt), h(x["v"], tdt), h(x["g"], torch.float32), h(x["beta"], torch.float32)


# (dtype, B, H, T, S, D, chunk, nonzero initial state, pinned)
CASES = [
    ("bf16", 1, 20, 21, 880, 112, 8, False, True),
    ("bf16", 2, 3, 9, 300, 64, 4, True, True),
    ("bf16", 1, 2, 9, 129, 48, 64, True, False),
    ("f32", 1, 2, 5, 33, 128, 2, True, True),
    ("bf16", 1, 1, 1, 16, 16, 1, False, True),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_host_entry_equals_device_call(case):
    dt, B, H, T, S, D, chunk, nz, pinned = case
    base = synth.WORKLOADS["short" if dt == "bf16" else "tiny"]
    wl = base.with_(B=B, H=H, T=T, S=S, D=D, seed=900 + 13 * S + D)
    x, q, k, v, g, beta = _host_inputs(wl, pinned)
    s0 = None
    if nz:
        s0 = torch.from_numpy(np.stack([np.stack([synth.state(wl, b, h) for h in range(H)]) for b in range(B)]))
    out_h, st_h = binding.frame_fwd_host(q, k, v, g, beta, state_in=s0, chunk_frames=chunk)
    parity.check_status()
    out_d, st_d = binding.frame_fwd(q.cuda(), k.cuda(), v.cuda(), g.cuda(), beta.cuda(),
                                    state_in=None if s0 is None else s0.cuda(), mode=0)
    torch.cuda.synchronize()
    assert torch.equal(out_h, out_d.cpu()) and torch.equal(st_h, st_d.cpu())


def test_host_entry_zero_frames_copies_state():
    wl = synth.WORKLOADS["short"].with_(H=2, T=1, S=16, D=32)
    _, q, k, v, g, beta = _host_inputs(wl, True)
    e = lambda t: t[:, :, :0].contiguous()  # noqa: E731
    s0 = torch.randn(1, 2, 32, 32)
    _, st = binding.frame_fwd_host(e(q), e(k), e(v), e(g), e(beta), state_in=s0, chunk_frames=4)
    assert torch.equal(st, s0)
