"""Context parallelism over frame ranges on the GPU (zhichai.net SANA-WM summary,
training pipeline Stage 3: the transition maps of the frame ranges before a
rank's own compose, exactly, into the state entering its range).

  * gdn_frame_summary against the oracle's scan: a range's map is the scan's
    linear part and offset, A = S_T(S_0 = I) - S_T(S_0 = 0), b = S_T(S_0 = 0);
  * gdn_summary_apply against A S + b, in place too;
  * the whole scheme on one GPU in one process (ranges in turn: summary, fold,
    forward from the folded state) against the oracle's single pass, both I/O
    dtypes, every algorithm form;
  * the rank driver, context_parallel.frame_fwd_cp, with two processes sharing
    the GPU and exchanging their summaries through gloo on the host (the kernels
    of the two processes never wait on each other), against the oracle.
Tolerances as tests/parity.py (float32 I/O 1e-4 max-abs; bf16 outputs 2e-2 x rms
beyond their own representation; float32 maps of bf16 calls 2e-2 x rms)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from linear_attention_video_gated_b300 import binding, build_lib, context_parallel, synth
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


def _wl(dt, B, H, T, S, D, seed):
    base = synth.WORKLOADS["short" if dt == "bf16" else "tiny"]
    return base.with_(B=B, H=H, T=T, S=S, D=D, seed=seed)


def _oracle_map(x, b, h):
    """(A, b) of head (b, h) over all frames of x, through the oracle's scan."""
    D = x["k"].shape[-1]
    args = (x["q"][b, h], x["k"][b, h], x["v"][b, h], x["g"][b, h], x["beta"][b, h])
    _, s0 = oracle.scan_head(*args)
    _, s1 = oracle.scan_head(*args, S0=np.eye(D))
    return s1 - s0, s0


def _map_parity(dt, got, ref, what):
    e = parity.errors(got, ref)
    if dt == "f32":
        assert e["max_abs"] <= parity.F32_MAX_ABS, f"{what}: {e}"
    else:
        assert e["max_abs_over_rms"] <= parity.BF16_MAX_ABS_OVER_RMS, f"{what}: {e}"
    return e


SUMMARY = [("f32", 1, 2, 8, 16, 16), ("f32", 2, 1, 37, 33, 64), ("bf16", 1, 3, 21, 300, 112),
           ("bf16", 2, 2, 33, 129, 128), ("bf16", 1, 1, 5, 17, 32), ("bf16", 1, 20, 21, 880, 112)]


@pytest.mark.parametrize("case", SUMMARY, ids=lambda c: "-".join(map(str, c)))
def test_summary_is_the_scans_affine_map(case):
    dt, B, H, T, S, D = case
    wl = _wl(dt, B, H, T, S, D, 9300 + T + D)
    x = synth.full(wl)
    _, k, v, g, beta = parity.upload(wl, x)
    A, b = binding.frame_summary(k, v, g, beta)
    torch.cuda.synchronize()
    parity.check_status()
    for bb in range(B):
        for h in range(H):
            ra, rb = _oracle_map(x, bb, h)
            ea = _map_parity(dt, np_(A[bb, h]), ra, f"A {case} head {(bb, h)}")
            eb = _map_parity(dt, np_(b[bb, h]), rb, f"b {case} head {(bb, h)}")
    print(f"summary {case}: A {ea} b {eb}")


def test_summary_of_no_frames_is_the_identity():
    k = torch.empty((1, 2, 0, 5, 32), dtype=torch.bfloat16, device="cuda")
    A, b = binding.frame_summary(k, k, torch.empty((1, 2, 0), device="cuda"),
                                 torch.empty((1, 2, 0, 5), device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(A, torch.eye(32, device="cuda").expand(1, 2, 32, 32)) and not b.any()


@pytest.mark.parametrize("D", [16, 112, 128])
def test_apply_is_a_times_s_plus_b_in_place_too(D):
    gen = torch.Generator().manual_seed(D)
    A, b, s = (torch.randn((2, 3, D, D), generator=gen, dtype=torch.float64) for _ in range(3))
    ref = (A @ s + b).numpy()
    Ad, bd, sd = (t.float().cuda() for t in (A, b, s))
    out = binding.summary_apply(Ad, bd, sd)
    binding.summary_apply(Ad, bd, sd, state_out=sd)  # in place
    zero = binding.summary_apply(Ad, bd, None)
    torch.cuda.synchronize()
    # float32 products of D terms of N(0,1) values: |err| <~ D * 2^-24 * |terms| * few
    np.testing.assert_allclose(np_(out), ref, rtol=0, atol=2e-4 * np.sqrt(D))
    assert torch.equal(out, sd)
    assert torch.equal(zero, bd)


# (dtype, B, H, T, S, D, ranges, nonzero initial state, gate logits)
SCHEME = [("f32", 1, 2, 8, 16, 16, 2, False, False), ("f32", 2, 1, 23, 40, 64, 3, True, False),
          ("bf16", 1, 4, 21, 300, 112, 2, False, False), ("bf16", 1, 3, 17, 129, 128, 4, True, False),
          ("bf16", 1, 2, 9, 880, 112, 3, False, True)]


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("case", SCHEME, ids=lambda c: "-".join(map(str, c)))
def test_ranges_in_one_process_equal_the_single_pass(case, mode):
    dt, B, H, T, S, D, R, nz, logits = case
    wl = _wl(dt, B, H, T, S, D, 9400 + T + D)
    x = synth.full(wl)
    q, k, v, g, beta = parity.upload(wl, x)
    if logits:
        lg = synth.logits_full(wl)
        g, beta = torch.from_numpy(lg["g_logit"]).cuda(), torch.from_numpy(lg["beta_logit"]).cuda()
    S0 = (np.stack([np.stack([synth.state(wl, bb, h, 0.3) for h in range(H)]) for bb in range(B)])
          if nz else None)
    s0 = None if S0 is None else torch.from_numpy(S0).cuda()
    sl = lambda t, a, c: t[:, :, a:c].contiguous()  # noqa: E731
    ranges = context_parallel.frame_ranges(T, R)
    maps = [binding.frame_summary(sl(k, a, c), sl(v, a, c), sl(g, a, c), sl(beta, a, c), gate_logits=logits)
            for a, c in ranges]
    outs, state = [], None
    for r, (a, c) in enumerate(ranges):
        enter = s0
        for rr in range(r):
            enter = binding.summary_apply(*maps[rr], enter)
        o, state = binding.frame_fwd(sl(q, a, c), sl(k, a, c), sl(v, a, c), sl(g, a, c), sl(beta, a, c),
                                     state_in=enter, mode=mode, gate_logits=logits)
        outs.append(o)
    torch.cuda.synchronize()
    parity.check_status()
    out = torch.cat(outs, dim=2)
    if logits:
        ro, rs = oracle.frame_fwd_from_logits(x["q"], x["k"], x["v"], lg["g_logit"], lg["beta_logit"], S0)
    else:
        ro, rs = oracle.frame_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], S0)
    eo, es = parity.assert_parity(dt, np_(out), ro, np_(state), rs, f"ranges {case} mode={mode}")
    print(f"ranges {case} mode={mode}: out {eo} state {es}")


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _cp_worker(rank, world, port, case, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    torch.cuda.set_device(0)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dt, B, H, T, S, D, seed = case
        wl = _wl(dt, B, H, T, S, D, seed)
        t0, t1 = context_parallel.frame_ranges(T, world)[rank]
        q, k, v, g, beta = parity.device_inputs(wl, t0=t0, t1=t1)
        o, s = context_parallel.frame_fwd_cp(q, k, v, g, beta)
        torch.cuda.synchronize()
        out[rank] = (np_(o), np_(s), binding.gdn_last_error(torch.cuda.current_stream().cuda_stream))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("case", [("bf16", 1, 20, 21, 880, 112, 1001), ("f32", 1, 2, 9, 33, 64, 9500)],
                         ids=lambda c: "-".join(map(str, c)))
def test_two_processes_exchange_summaries_through_gloo(case):
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_cp_worker, args=(world, _free_port(), case, out), nprocs=world, join=True)
        res = dict(out)
    dt, B, H, T, S, D, seed = case
    wl = _wl(dt, B, H, T, S, D, seed)
    x = synth.full(wl)
    ro, rs = oracle.frame_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"])
    got = np.concatenate([res[r][0] for r in range(world)], axis=2)
    for r in range(world):
        assert res[r][2] == 0
        eo, es = parity.assert_parity(dt, got, ro, res[r][1], rs, f"cp {case} rank {r}")
        print(f"cp {case} rank {r}: out {eo} state {es}")
