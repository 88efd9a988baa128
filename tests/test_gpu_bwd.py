"""GPU parity of the backward pass (gdn_frame_bwd, gdn_frame_bwd_from_logits)
against the fp64 oracle's backward on the same seeded inputs and output
gradients.  Bounds are in tests/parity.py (assert_grad_parity)."""
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
    return None if t is None else t.float().cpu().numpy()


def _case_inputs(dt, B, H, T, S, D, nz_state, seed):
    base = synth.WORKLOADS["short" if dt == "bf16" else "tiny"]
    wl = base.with_(B=B, H=H, T=T, S=S, D=D, seed=seed)
    x = synth.full(wl)
    gr = synth.full_grads(wl)
    S0 = np.stack([np.stack([synth.state(wl, b, h, 0.3) for h in range(H)]) for b in range(B)]) if nz_state else None
    return wl, x, gr, S0


def _run_bwd(wl, x, dout, S0, dST, gate_logits=False, g=None, beta=None, **kw):
    q, k, v, g_t, b_t = parity.upload(wl, x)
    if g is not None:
        g_t, b_t = g, beta
    do = torch.from_numpy(np.ascontiguousarray(dout)).cuda().to(q.dtype).contiguous()
    si = None if S0 is None else torch.from_numpy(S0).cuda()
    ds = None if dST is None else torch.from_numpy(dST).cuda()
    res = binding.frame_bwd(q, k, v, g_t, b_t, do, state_in=si, dstate_out=ds, gate_logits=gate_logits, **kw)
    torch.cuda.synchronize()
    parity.check_status()
    return {key: np_(val) for key, val in res.items()}


# (dtype, B, H, T, S, D, nonzero initial state, final-state gradient)
CASES = [
    ("f32", 1, 2, 4, 37, 32, True, True),
    ("f32", 1, 1, 1, 1, 16, False, False),
    ("f32", 2, 1, 3, 70, 128, True, False),
    ("f32", 1, 1, 5, 33, 112, False, True),
    ("bf16", 1, 3, 6, 70, 48, True, True),
    ("bf16", 1, 2, 5, 880, 112, True, True),
    ("bf16", 1, 1, 9, 129, 64, False, False),
    ("bf16", 1, 1, 3, 200, 96, True, True),
    ("bf16", 1, 1, 2, 1, 16, False, True),
    ("bf16", 1, 1, 17, 31, 80, True, False),
    ("bf16", 1, 2, 4, 150, 128, True, True),
    ("bf16", 2, 1, 3, 257, 32, False, True),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_backward_matches_oracle(case):
    dt, B, H, T, S, D, nz, nd = case
    wl, x, gr, S0 = _case_inputs(dt, B, H, T, S, D, nz, seed=6000 + 5 * S + D)
    dST = gr["dstate"] if nd else None
    got = _run_bwd(wl, x, gr["dout"], S0, dST)
    ref = oracle.frame_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], S0, gr["dout"], dST)
    res = parity.assert_grad_parity(dt, got, ref, f"bwd {case}")
    print(f"bwd {case}: " + ", ".join(f"{k} max {v['max_abs_over_rms']:.2e} rms {v['rms_err_over_rms']:.2e}"
                                      for k, v in res.items()))


@pytest.mark.parametrize("case", [("bf16", 1, 2, 5, 70, 48), ("f32", 1, 2, 4, 37, 32)],
                         ids=lambda c: "-".join(map(str, c)))
def test_backward_from_logits_matches_oracle(case):
    dt, B, H, T, S, D = case
    wl = synth.WORKLOADS["short"].with_(B=B, H=H, T=T, S=S, D=D, dtype=dt, seed=6100 + S + D)
    x = synth.full(wl)
    lg = synth.logits_full(wl)
    gr = synth.full_grads(wl)
    S0 = np.stack([np.stack([synth.state(wl, b, h, 0.3) for h in range(H)]) for b in range(B)])
    gl = torch.from_numpy(lg["g_logit"]).cuda()
    bl = torch.from_numpy(lg["beta_logit"]).cuda()
    got = _run_bwd(wl, x, gr["dout"], S0, gr["dstate"], gate_logits=True, g=gl, beta=bl)
    ref = oracle.frame_bwd_from_logits(x["q"], x["k"], x["v"], lg["g_logit"], lg["beta_logit"], S0, gr["dout"],
                                       gr["dstate"])
    ref["dg"], ref["dbeta"] = ref.pop("dg_logit"), ref.pop("dbeta_logit")
    parity.assert_grad_parity(dt, got, ref, f"bwd logits {case}")


def test_backward_without_initial_state_gradient_output():
    """dstate_in = NULL: every other gradient is unchanged, bit for bit."""
    wl, x, gr, S0 = _case_inputs("bf16", 1, 2, 4, 50, 32, True, 6200)
    a = _run_bwd(wl, x, gr["dout"], S0, gr["dstate"])
    b = _run_bwd(wl, x, gr["dout"], S0, gr["dstate"], want_dstate_in=False)
    for key in ("dq", "dk", "dv", "dg", "dbeta"):
        np.testing.assert_array_equal(a[key], b[key])
    assert b["dstate_in"] is None


def test_backward_is_deterministic():
    wl, x, gr, S0 = _case_inputs("bf16", 1, 2, 6, 100, 64, True, 6300)
    a = _run_bwd(wl, x, gr["dout"], S0, gr["dstate"])
    b = _run_bwd(wl, x, gr["dout"], S0, gr["dstate"])
    for key in parity.GRAD_KEYS:
        np.testing.assert_array_equal(a[key], b[key])


def test_backward_zero_frames_passes_the_state_gradient_through():
    wl, x, gr, _ = _case_inputs("bf16", 1, 2, 1, 16, 32, False, 6400)
    q, k, v, g, beta = parity.upload(wl, x)
    e = lambda t: t[:, :, :0].contiguous()  # noqa: E731
    dST = torch.randn(1, 2, 32, 32, device="cuda")
    res = binding.frame_bwd(e(q), e(k), e(v), e(g), e(beta), e(q), dstate_out=dST)
    torch.cuda.synchronize()
    assert torch.equal(res["dstate_in"], dST)
    res = binding.frame_bwd(e(q), e(k), e(v), e(g), e(beta), e(q))
    torch.cuda.synchronize()
    assert torch.count_nonzero(res["dstate_in"]) == 0


def test_backward_on_nan_filled_workspace():
    """Every stage writes its scratch before reading it: a workspace full of NaN
    bit patterns gives the same gradients as a zeroed one."""
    wl, x, gr, S0 = _case_inputs("bf16", 1, 2, 5, 70, 48, True, 6500)
    need = binding.gdn_bwd_workspace_bytes(1, 2, 5, 70, 48, binding.GDN_BF16)
    a = _run_bwd(wl, x, gr["dout"], S0, gr["dstate"], workspace=torch.zeros(need, dtype=torch.uint8, device="cuda"))
    b = _run_bwd(wl, x, gr["dout"], S0, gr["dstate"],
                 workspace=torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda"))
    for key in parity.GRAD_KEYS:
        np.testing.assert_array_equal(a[key], b[key])


def test_backward_minute_every_head():
    """The one-minute workload (961 frames x 880 tokens x 20 heads x d112, bf16) in
    one backward call; every one of the 20 heads checked over every frame against
    the oracle."""
    wl = synth.WORKLOADS["minute"]
    q, k, v, g, beta = parity.device_inputs(wl)
    dout = parity.device_dout(wl)
    res = binding.frame_bwd(q, k, v, g, beta, dout)
    torch.cuda.synchronize()
    parity.check_status()
    del q, k, v, g, beta, dout

    def ref_of(b, h):
        x = synth.head(wl, b, h)
        ref = oracle.backward_head(x["q"], x["k"], x["v"], x["g"], x["beta"], None, synth.head_dout(wl, b, h))
        ref["dstate_in"] = ref.pop("dS0")
        return ref

    heads = [(b, h) for b in range(wl.B) for h in range(wl.H)]
    n, failures = 0, []
    for (b, h), ref in parity.oracle_heads(wl, heads, fn=ref_of, workers=2):
        n += 1
        got = {key: np_(res[key][b, h]) for key in parity.GRAD_KEYS}
        r = {key: parity.errors(got[key], ref[key]) for key in parity.GRAD_KEYS}
        print(f"minute bwd head {(b, h)}: " + ", ".join(
            f"{k} max {v['max_abs_over_rms']:.2e} beyond-half-ulp {v['max_beyond_half_ulp_over_rms']:.2e} "
            f"rms {v['rms_err_over_rms']:.2e}" for k, v in r.items()))
        try:
            parity.assert_grad_parity(wl.dtype, got, ref, f"minute bwd head {(b, h)}")
        except AssertionError as e:  # every head is checked before the test fails
            failures.append(str(e))
    assert n == len(heads)
    assert not failures, failures


@pytest.mark.parametrize("gate_logits", [False, True])
def test_autograd_op_matches_the_backward_entry(gate_logits):
    """binding.gdn under torch.autograd: a loss over both outputs gives exactly the
    gradients gdn_frame_bwd returns for that loss's output gradients."""
    wl, x, gr, S0 = _case_inputs("bf16", 1, 2, 4, 70, 48, True, 6600)
    q, k, v, g, beta = parity.upload(wl, x)
    if gate_logits:
        lg = synth.logits_full(wl)
        g, beta = torch.from_numpy(lg["g_logit"]).cuda(), torch.from_numpy(lg["beta_logit"]).cuda()
    s0 = torch.from_numpy(S0).cuda()
    leaves = [t.clone().requires_grad_(True) for t in (q, k, v, g, beta, s0)]
    out, st = binding.gdn(*leaves, gate_logits=gate_logits)
    w_out = torch.from_numpy(gr["dout"]).cuda().to(q.dtype)
    w_st = torch.from_numpy(gr["dstate"]).cuda()
    ((out.float() * w_out.float()).sum() + (st * w_st).sum()).backward()
    ref = binding.frame_bwd(q, k, v, g, beta, w_out.contiguous(), state_in=s0, dstate_out=w_st,
                            gate_logits=gate_logits)
    torch.cuda.synchronize()
    parity.check_status()
    for leaf, key in zip(leaves, ("dq", "dk", "dv", "dg", "dbeta", "dstate_in")):
        assert torch.equal(leaf.grad, ref[key]), key



# (dtype, forward mode, gate logits)
REUSE = [("bf16", 0, False), ("bf16", 2, False), ("bf16", 0, True), ("f32", 0, False), ("f32", 1, False)]


@pytest.mark.parametrize("case", REUSE, ids=lambda c: "-".join(map(str, c)))
def test_backward_reuses_the_forward_states(case):
    """GDN_BWD_STATES_IN_WORKSPACE: a backward that reads the states a forward call
    left in the workspace gives the recomputing backward's gradients bit for bit (the
    same kernels made the states), or, after the fp32 prefix form (whose states come
    from its own composition), gradients within the oracle bound."""
    dt, mode, logits = case
    wl, x, gr, S0 = _case_inputs(dt, 1, 2, 6, 150, 48, True, 6700 + mode)
    q, k, v, g, beta = parity.upload(wl, x)
    if logits:
        lg = synth.logits_full(wl)
        g, beta = torch.from_numpy(lg["g_logit"]).cuda(), torch.from_numpy(lg["beta_logit"]).cuda()
    s0 = torch.from_numpy(S0).cuda()
    dout = torch.from_numpy(gr["dout"]).cuda().to(q.dtype).contiguous()
    dst = torch.from_numpy(gr["dstate"]).cuda()
    need = binding.gdn_bwd_workspace_bytes(1, 2, 6, 150, 48, binding.GDN_BF16 if dt == "bf16" else binding.GDN_F32)
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")
    binding.frame_fwd(q, k, v, g, beta, state_in=s0, mode=mode, workspace=ws, gate_logits=logits)
    a = binding.frame_bwd(q, k, v, g, beta, dout, state_in=s0, dstate_out=dst, gate_logits=logits, workspace=ws,
                          states_in_workspace=True)
    b = binding.frame_bwd(q, k, v, g, beta, dout, state_in=s0, dstate_out=dst, gate_logits=logits)
    torch.cuda.synchronize()
    parity.check_status()
    if (dt, mode) == ("f32", 1):
        ref = oracle.frame_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], S0, gr["dout"], gr["dstate"])
        parity.assert_grad_parity(dt, {key: np_(val) for key, val in a.items()}, ref, f"reuse {case}")
    else:
        for key in parity.GRAD_KEYS:
            assert torch.equal(a[key], b[key]), key


def test_backward_outputs_only_16_byte_aligned():
    """dk and dv on 16- but not 32-byte boundaries (the kernel's 32-byte row stores
    fall back to 16-byte ones): the same gradients, bit for bit."""
    wl, x, gr, S0 = _case_inputs("bf16", 1, 2, 5, 130, 112, True, 6600)
    ref = _run_bwd(wl, x, gr["dout"], S0, gr["dstate"])
    q, k, v, g, beta = parity.upload(wl, x)
    do = torch.from_numpy(np.ascontiguousarray(gr["dout"])).cuda().to(q.dtype).contiguous()
    si = torch.from_numpy(S0).cuda()
    ds = torch.from_numpy(gr["dstate"]).cuda()
    n = q.numel()
    raw = [torch.empty(n + 16, dtype=q.dtype, device="cuda") for _ in range(2)]
    dk, dv = (r[8:8 + n] for r in raw)  # 16 bytes past a 256-byte boundary
    assert dk.data_ptr() % 32 == 16 and dv.data_ptr() % 32 == 16
    dq = torch.empty_like(q)
    dg = torch.empty(g.shape, device="cuda")
    db = torch.empty(beta.shape, device="cuda")
    dsi = torch.empty_like(si)
    B, H, T, S, D = q.shape
    need = binding.gdn_bwd_workspace_bytes(B, H, T, S, D, binding.GDN_BF16)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    rc = binding.gdn_frame_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), g.data_ptr(), beta.data_ptr(), si.data_ptr(),
                               do.data_ptr(), ds.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), dg.data_ptr(),
                               db.data_ptr(), dsi.data_ptr(), B, H, T, S, D, binding.GDN_BF16, ws.data_ptr(), need, st)
    assert rc == 0
    torch.cuda.synchronize()
    parity.check_status()
    np.testing.assert_array_equal(np_(dk.view(q.shape)), ref["dk"])
    np.testing.assert_array_equal(np_(dv.view(q.shape)), ref["dv"])
    np.testing.assert_array_equal(np_(dq), ref["dq"])
