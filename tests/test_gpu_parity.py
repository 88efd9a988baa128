"""GPU parity: the CUDA path through the C ABI against the fp64 oracle, on the
same seeded inputs.  Tolerances are in tests/parity.py."""
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


def run(q, k, v, g, beta, state_in=None, mode=None, **kw):
    out, st = binding.frame_fwd(q, k, v, g, beta, state_in=state_in, mode=mode, **kw)
    torch.cuda.synchronize()
    parity.check_status()
    return out, st


def np_(t):
    return t.float().cpu().numpy()


@pytest.mark.parametrize("mode", [None, 0, 1, 2])
def test_tiny_f32(mode):
    wl = synth.WORKLOADS["tiny"]
    x = synth.full(wl)
    out, st = run(*parity.upload(wl, x), mode=mode)
    ro, rs = oracle.frame_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"])
    parity.assert_parity("f32", np_(out), ro, np_(st), rs, f"tiny mode={mode}")


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_short_bf16(mode):
    wl = synth.WORKLOADS["short"]
    x = synth.full(wl)
    out, st = run(*parity.upload(wl, x), mode=mode)
    ro, rs = oracle.frame_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"])
    eo, es = parity.assert_parity("bf16", np_(out), ro, np_(st), rs, f"short mode={mode}")
    print(f"short mode={mode}: out {eo} state {es}")


# (dtype, B, H, T, S, D, nonzero initial state)
EDGE = [
    ("bf16", 1, 1, 1, 1, 16, False),
    ("bf16", 1, 2, 5, 17, 32, True),
    ("bf16", 2, 1, 4, 129, 48, False),
    ("bf16", 1, 1, 3, 300, 64, True),
    ("bf16", 1, 2, 2, 257, 80, False),
    ("bf16", 1, 1, 17, 200, 96, True),
    ("bf16", 1, 1, 33, 64, 128, False),
    ("bf16", 1, 3, 6, 880, 112, True),
    ("f32", 1, 1, 1, 1, 16, False),
    ("f32", 2, 2, 5, 33, 128, True),
    ("f32", 1, 1, 3, 100, 112, True),
    ("f32", 1, 1, 20, 7, 64, False),
]


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("case", EDGE, ids=lambda c: "-".join(map(str, c)))
def test_edge_shapes(case, mode):
    dt, B, H, T, S, D, nz = case
    base = synth.WORKLOADS["short" if dt == "bf16" else "tiny"]
    wl = base.with_(B=B, H=H, T=T, S=S, D=D, seed=base.seed + 17 * S + D)
    x = synth.full(wl)
    S0 = np.stack([np.stack([synth.state(wl, b, h, 0.3) for h in range(H)]) for b in range(B)]) if nz else None
    si = None if S0 is None else torch.from_numpy(S0).cuda()
    out, st = run(*parity.upload(wl, x), state_in=si, mode=mode)
    ro, rs = oracle.frame_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], S0)
    eo, es = parity.assert_parity(dt, np_(out), ro, np_(st), rs, f"edge {case} mode={mode}")
    print(f"edge {case} mode={mode}: out {eo} state {es}")


# (dtype, B, H, T, S, D): gates given as logits (the fused gate prologue)
LOGIT_CASES = [
    ("bf16", 1, 20, 21, 880, 112),
    ("bf16", 1, 2, 5, 17, 32),
    ("bf16", 2, 1, 4, 129, 48),
    ("bf16", 1, 1, 9, 64, 128),
    ("f32", 2, 2, 5, 33, 128),
    ("f32", 1, 1, 3, 100, 112),
]


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("case", LOGIT_CASES, ids=lambda c: "-".join(map(str, c)))
def test_gate_logits(case, mode):
    """gdn_frame_fwd_from_logits: g and beta computed from raw logits inside the
    kernels, against the oracle's gate prologue followed by its scan."""
    dt, B, H, T, S, D = case
    wl = synth.WORKLOADS["short"].with_(B=B, H=H, T=T, S=S, D=D, dtype=dt, seed=4000 + 7 * S + D)
    x = synth.full(wl)
    lg = synth.logits_full(wl)
    q, k, v, _, _ = parity.upload(wl, x)
    gl = torch.from_numpy(lg["g_logit"]).cuda()
    bl = torch.from_numpy(lg["beta_logit"]).cuda()
    out, st = run(q, k, v, gl, bl, mode=mode, gate_logits=True)
    ro, rs = oracle.frame_fwd_from_logits(x["q"], x["k"], x["v"], lg["g_logit"], lg["beta_logit"])
    eo, es = parity.assert_parity(dt, np_(out), ro, np_(st), rs, f"logits {case} mode={mode}")
    print(f"logits {case} mode={mode}: out {eo} state {es}")


# (dtype, B, H, T, S, D, nonzero initial state): the cumulative ReLU linear attention baseline
RELU_CASES = [
    ("bf16", 1, 20, 21, 880, 112, False),
    ("bf16", 1, 2, 5, 17, 32, True),
    ("bf16", 2, 1, 4, 129, 48, False),
    ("bf16", 1, 1, 9, 64, 128, True),
    ("f32", 2, 2, 5, 33, 128, True),
    ("f32", 1, 1, 3, 100, 112, False),
]


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("case", RELU_CASES, ids=lambda c: "-".join(map(str, c)))
def test_relu_linear_baseline(case, mode):
    """gdn_relu_linear_fwd against the oracle's cumulative ReLU linear attention."""
    dt, B, H, T, S, D, nz = case
    base = synth.WORKLOADS["short" if dt == "bf16" else "tiny"]
    wl = base.with_(B=B, H=H, T=T, S=S, D=D, seed=5000 + 3 * S + D)
    x = synth.full(wl)
    q, k, v, _, _ = parity.upload(wl, x)
    S0 = np.stack([np.stack([synth.state(wl, b, h, 0.3) for h in range(H)]) for b in range(B)]) if nz else None
    out, st = binding.relu_linear_fwd(q, k, v, state_in=None if S0 is None else torch.from_numpy(S0).cuda(),
                                      mode=mode)
    torch.cuda.synchronize()
    parity.check_status()
    ro, rs = oracle.relu_linear_fwd(x["q"], x["k"], x["v"], S0)
    eo, es = parity.assert_parity(dt, np_(out), ro, np_(st), rs, f"relu-linear {case} mode={mode}")
    print(f"relu-linear {case} mode={mode}: out {eo} state {es}")


def _small_bf16(T=21, H=3, S=300, D=112):
    wl = synth.WORKLOADS["short"].with_(H=H, T=T, S=S, D=D)
    return wl, synth.full(wl)


@pytest.mark.parametrize("mode", [0, 2])
def test_state_aliasing_is_bitwise_identical(mode):
    wl, x = _small_bf16()
    ins = parity.upload(wl, x)
    S0 = torch.from_numpy(np.stack([np.stack([synth.state(wl, 0, h) for h in range(wl.H)])])).cuda()
    out_a, st_a = run(*ins, state_in=S0.clone(), mode=mode)
    buf = S0.clone()
    out_b, st_b = run(*ins, state_in=buf, state_out=buf, mode=mode)
    assert torch.equal(out_a, out_b) and torch.equal(st_a, buf)


def test_zero_frames_copies_state():
    wl, x = _small_bf16(T=1)
    q, k, v, g, beta = parity.upload(wl, x)
    e = lambda t: t[:, :, :0].contiguous()  # noqa: E731
    S0 = torch.randn(1, wl.H, wl.D, wl.D, device="cuda")
    _, st = run(e(q), e(k), e(v), e(g), e(beta), state_in=S0, mode=0)
    assert torch.equal(st, S0)
    st2 = torch.full_like(S0, 7.0)
    run(e(q), e(k), e(v), e(g), e(beta), state_out=st2, mode=0)
    assert torch.count_nonzero(st2) == 0


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_chunked_calls_equal_single_call(mode):
    """Chunk-causal rollout: consecutive calls passing state_out -> state_in give the
    single call's outputs.  In the sequential and split forms the per-frame
    arithmetic does not depend on where the calls split, so the results are
    bitwise equal."""
    wl, x = _small_bf16(T=21)
    q, k, v, g, beta = parity.upload(wl, x)
    out1, st1 = run(q, k, v, g, beta, mode=mode)
    outs, st = [], None
    for a, b in ((0, 10), (10, 20), (20, 21)):
        sl = lambda t: t[:, :, a:b].contiguous()  # noqa: E731
        o, st = run(sl(q), sl(k), sl(v), sl(g), sl(beta), state_in=st, mode=mode)
        outs.append(o)
    out2 = torch.cat(outs, dim=2)
    if mode in (0, 2):
        assert torch.equal(out1, out2) and torch.equal(st1, st)
    else:
        ro, rs = oracle.frame_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"])
        parity.assert_parity("bf16", np_(out2), ro, np_(st), rs, "chunked prefix")


@pytest.mark.parametrize("mode", [0, 2])
def test_repeat_calls_are_deterministic(mode):
    wl, x = _small_bf16(T=9)
    ins = parity.upload(wl, x)
    a = run(*ins, mode=mode)
    b = run(*ins, mode=mode)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("shape", [(1, 20, 13, 880, 112), (2, 3, 9, 300, 64), (1, 1, 4, 129, 16), (1, 9, 5, 200, 128)])
def test_sequential_equals_split_bitwise(shape):
    """The sequential and split forms agree bit for bit, each run on a workspace
    filled with NaN bit patterns, so a read of scratch that no kernel has written
    (a transition term or a state block read before it is stored) cannot go
    unnoticed."""
    B, H, T, S, D = shape
    wl = synth.WORKLOADS["short"].with_(B=B, H=H, T=T, S=S, D=D, seed=777 + D)
    x = synth.full(wl)
    ins = parity.upload(wl, x)
    S0 = torch.from_numpy(np.stack([np.stack([synth.state(wl, b, h) for h in range(H)]) for b in range(B)])).cuda()
    results = []
    for mode in (0, 2):
        need = binding.gdn_workspace_bytes(B, H, T, S, D, binding.GDN_BF16, mode)
        ws = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")
        results.append(run(*ins, state_in=S0, mode=mode, workspace=ws))
    a, b = results
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_plain_entry_matches_explicit_workspace():
    wl, x = _small_bf16(T=5)
    ins = parity.upload(wl, x)
    a = run(*ins, mode=None)
    b = run(*ins, mode=0)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


# ------------------------------------------------------------------ full sizes

@pytest.fixture(scope="module")
def minute_inputs():
    wl = synth.WORKLOADS["minute"]
    return wl, parity.device_inputs(wl)


def _check_heads(wl, outs, ref_iter, what):
    """outs: {label: (out, state)} device results; every head ref_iter yields is
    compared, for every label, against the oracle."""
    n = 0
    for (b, h), ro, rs in ref_iter:
        for label, (out, st) in outs.items():
            eo, es = parity.assert_parity(wl.dtype, np_(out[b, h]), ro, np_(st[b, h]), rs,
                                          f"{what} {label} head {(b, h)}")
            print(f"{what} {label} head {(b, h)}: out {eo} state {es}")
        n += 1
    return n


def test_minute_every_head_single_call_and_chunked_rollout(minute_inputs):
    """961 frames x 880 tokens x 20 heads x d112: one call (the bench's launch
    configuration) and the same tensors as 97 chunk-causal calls of <= 10 frames
    carrying the state.  The rollout equals the single call bit for bit (the
    per-frame arithmetic does not depend on where calls split), and every one of
    the 20 heads of the single call is compared over every frame with the oracle."""
    wl, (q, k, v, g, beta) = minute_inputs
    out, st = run(q, k, v, g, beta, mode=0)
    cw = synth.WORKLOADS["chunked"]
    outs, stc, t0 = [], None, 0
    for n in cw.chunks:
        sl = lambda t: t[:, :, t0:t0 + n].contiguous()  # noqa: E731
        o, stc = run(sl(q), sl(k), sl(v), sl(g), sl(beta), state_in=stc, mode=0)
        outs.append(o)
        t0 += n
    assert t0 == wl.T
    outc = torch.cat(outs, dim=2)
    del outs
    same = torch.equal(out, outc) and torch.equal(st, stc)
    checked = {"single": (out, st)} if same else {"single": (out, st), "chunked": (outc, stc)}
    heads = [(b, h) for b in range(wl.B) for h in range(wl.H)]
    assert _check_heads(wl, checked, parity.oracle_heads(wl, heads), "minute") == len(heads)
    assert same, "the chunk-causal rollout differs from the single call"


def test_large_sequential_and_prefix_agree():
    """4 x 16 heads, 241 frames of 3600 tokens, d128: eight heads spread over all
    four batch indices, for both the sequential scan and the chunked prefix
    composition, match the oracle over every frame, and the two forms agree
    everywhere.

    Agreement of two bf16 outputs: each form rounds its own fp32 value, so the two
    may land on adjacent bf16 values even when both are within the bound of the
    exact result; one bf16 ulp of |out| is the smallest difference the output type
    can show.  The element-wise bound is therefore |a - b| <= ulp_bf16 + 2e-2 rms;
    the fp32 final states are held to the plain 2e-2 rms bound."""
    wl = synth.WORKLOADS["large"]
    ins = parity.device_inputs(wl)
    out0, st0 = run(*ins, mode=0)
    out1, st1 = run(*ins, mode=1)
    del ins
    heads = synth.head_sample(wl, 8)
    assert {b for b, _ in heads} == set(range(wl.B))
    n = _check_heads(wl, {"seq": (out0, st0), "prefix": (out1, st1)}, parity.oracle_heads(wl, heads), "large")
    assert n == len(heads)
    rms_o = torch.sqrt(torch.mean(out0.float() ** 2)).item()
    rms_s = torch.sqrt(torch.mean(st0 ** 2)).item()
    beyond, sq = 0.0, 0.0
    for b in range(wl.B):
        a, c = out0[b].float(), out1[b].float()
        m = torch.maximum(a.abs(), c.abs())
        ulp = torch.where(m > 0, torch.exp2(torch.floor(torch.log2(torch.where(m > 0, m, 1.0))) - 7), 0.0)
        d = (a - c).abs()
        beyond = max(beyond, (d - ulp).clamp_min(0.0).max().item())
        sq += (d.double() ** 2).sum().item()
    rms_d = (sq / out0.numel()) ** 0.5
    d_s = (st0 - st1).abs().max().item()
    print(f"large: seq vs prefix out beyond-1-ulp/rms {beyond / rms_o:.3e}, rms diff/rms {rms_d / rms_o:.3e}, "
          f"state max/rms {d_s / rms_s:.3e}")
    assert beyond / rms_o <= parity.BF16_MAX_ABS_OVER_RMS
    assert rms_d / rms_o <= parity.BF16_RMS_ERR_OVER_RMS
    assert d_s / rms_s <= parity.BF16_MAX_ABS_OVER_RMS


# (H, T, S): frame-head counts just below, at and above one and two rounds of the
# 148 persistent CTAs, token counts giving 1, 3 and 7 read-out tiles (the last one
# ragged), so the read-out's round-robin phase, its balanced tail and the
# boundary between them all run
ROUNDS = [(7, 21, 300), (4, 37, 129), (1, 149, 880), (3, 99, 250), (9, 33, 64), (2, 74, 700)]


@pytest.mark.parametrize("case", ROUNDS, ids=lambda c: "-".join(map(str, c)))
def test_readout_work_split_over_frame_head_counts(case):
    H, T, S = case
    wl = synth.WORKLOADS["short"].with_(H=H, T=T, S=S, D=64, seed=7300 + H * T)
    x = synth.full(wl)
    out, st = run(*parity.upload(wl, x), mode=0)
    ro, rs = oracle.frame_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"])
    eo, es = parity.assert_parity("bf16", np_(out), ro, np_(st), rs, f"read-out split {case}")
    print(f"read-out split {case} (F = {H * T}): out {eo} state {es}")
