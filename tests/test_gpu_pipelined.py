"""The pipelined form (GDN_MODE_PIPELINED): the split form's gram and read-out over
32-frame chunks of every head on the caller's stream, the recurrence of each
chunk (one CTA per head, every column block in one MMA chain) on a second stream,
joined by events.  Compared with the fp64 oracle on the same seeded inputs
(tests/parity.py bounds), with the split form bit for bit (the per-element
arithmetic is the same: one K-step sequence per output element, the same fp32
update), on a workspace full of NaN bit patterns (no scratch read before it is
written), with the state aliased in place, and on the one-minute workload against
the single sequential call."""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_video_gated_b300 import binding, build_lib, synth
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_lib.ensure_built()
    binding.lib()


def np_(t):
    return t.float().cpu().numpy()


def run(ins, S0, mode, nan_ws=False, state_out=None):
    q = ins[0]
    B, H, T, S, D = q.shape
    need = binding.gdn_workspace_bytes(B, H, T, S, D, binding.GDN_BF16, mode)
    ws = torch.full((need,), 0xFF if nan_ws else 0, dtype=torch.uint8, device="cuda")
    out, st = binding.frame_fwd(*ins, state_in=S0, mode=mode, workspace=ws, state_out=state_out)
    torch.cuda.synchronize()
    parity.check_status()
    return out, st


# (B, H, T, S, D, nonzero initial state): every one takes the pipelined path
# (bf16, D <= 112, 4 B H <= the SM count, T > 32) -- a ragged last chunk, one or
# two atoms of D, several batch indices
SHAPES = [(1, 3, 70, 300, 112, True), (2, 2, 40, 129, 64, False), (1, 1, 33, 64, 32, True),
          (1, 20, 65, 880, 112, False), (1, 4, 97, 17, 16, True), (3, 1, 36, 200, 96, False)]


@pytest.mark.parametrize("case", SHAPES, ids=lambda c: "-".join(map(str, c)))
def test_pipelined_equals_split_and_matches_the_oracle(case):
    B, H, T, S, D, nz = case
    wl = synth.WORKLOADS["short"].with_(B=B, H=H, T=T, S=S, D=D, seed=9900 + T + D)
    x = synth.full(wl)
    ins = parity.upload(wl, x)
    S0n = (np.stack([np.stack([synth.state(wl, b, h, 0.3) for h in range(H)]) for b in range(B)])
           if nz else None)
    S0 = None if S0n is None else torch.from_numpy(S0n).cuda()
    out_p, st_p = run(ins, S0, binding.GDN_MODE_PIPELINED, nan_ws=True)
    out_s, st_s = run(ins, S0, binding.GDN_MODE_SPLIT, nan_ws=True)
    ro, rs = oracle.frame_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], S0n)
    eo, es = parity.assert_parity("bf16", np_(out_p), ro, np_(st_p), rs, f"pipelined {case}")
    print(f"pipelined {case}: out {eo} state {es}")
    assert torch.equal(out_p, out_s) and torch.equal(st_p, st_s), "pipelined and split forms differ"


def test_pipelined_state_in_place():
    wl = synth.WORKLOADS["short"].with_(H=3, T=45, S=300, seed=9950)
    ins = parity.upload(wl, synth.full(wl))
    S0 = torch.from_numpy(np.stack([np.stack([synth.state(wl, 0, h) for h in range(wl.H)])])).cuda()
    out_a, st_a = run(ins, S0.clone(), binding.GDN_MODE_PIPELINED)
    buf = S0.clone()
    out_b, _ = run(ins, buf, binding.GDN_MODE_PIPELINED, state_out=buf)
    assert torch.equal(out_a, out_b) and torch.equal(st_a, buf)


def test_pipelined_minute_equals_the_sequential_call():
    """961 frames x 880 tokens x 20 heads x d112 (31 chunks): bit for bit the split
    form's single call, which the every-head oracle test checks."""
    wl = synth.WORKLOADS["minute"]
    ins = parity.device_inputs(wl)
    out_p, st_p = run(ins, None, binding.GDN_MODE_PIPELINED)
    out_s, st_s = run(ins, None, binding.GDN_MODE_SPLIT)
    assert torch.equal(out_p, out_s) and torch.equal(st_p, st_s)
