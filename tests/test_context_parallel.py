"""Context parallelism over frame ranges on the CPU: the rank driver
(context_parallel.frame_fwd_cp) with gloo ranks, the exchange and the order of
composition checked against the oracle's single pass over the whole sequence
(zhichai.net SANA-WM summary, training pipeline Stage 3: the transition maps of
the ranges before a rank's compose, exactly, into the state entering its range).

The ranks here run the oracle in place of the CUDA entry points (the same three
operations: a range's map, a map applied to a state, the scan from a state), so
what is tested is the driver: which ranges' maps are folded, in which order,
onto which state, and the final state every rank returns.  The same driver on
the CUDA path is tested in tests/test_gpu_context_parallel.py.  Also here: the
C ABI of the two context-parallel entry points rejects bad arguments on the host."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from linear_attention_video_gated_b300 import binding, build_lib, context_parallel, synth  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class OracleOps:
    """The three operations, by the fp64 oracle, on float64 CPU tensors [B,H,...]."""

    def summary(self, k, v, g, beta, gate_logits):
        B, H, T, S, D = k.shape
        A = torch.zeros((B, H, D, D), dtype=torch.float64)
        b = torch.zeros_like(A)
        for bb in range(B):
            for h in range(H):
                m = (np.eye(D), np.zeros((D, D)))
                for t in range(T):
                    m = oracle.compose(oracle.transition(k[bb, h, t].numpy(), v[bb, h, t].numpy(),
                                                         float(g[bb, h, t]), beta[bb, h, t].numpy()), m)
                A[bb, h] = torch.from_numpy(m[0])
                b[bb, h] = torch.from_numpy(m[1])
        return A, b

    def apply(self, A, b, state):
        out = torch.empty_like(b)
        for bb in range(A.shape[0]):
            for h in range(A.shape[1]):
                S = np.zeros(tuple(b.shape[2:])) if state is None else state[bb, h].numpy()
                out[bb, h] = torch.from_numpy(oracle.apply_map((A[bb, h].numpy(), b[bb, h].numpy()), S))
        return out

    def forward(self, q, k, v, g, beta, state_in, gate_logits, mode):
        S0 = None if state_in is None else state_in.numpy()
        o, s = oracle.frame_fwd(q.numpy(), k.numpy(), v.numpy(), g.numpy(), beta.numpy(), S0)
        return torch.from_numpy(o), torch.from_numpy(s)


def _inputs(T, nonzero):
    wl = synth.WORKLOADS["tiny"].with_(T=T, seed=9100 + T)
    x = synth.full(wl)
    S0 = (np.stack([np.stack([synth.state(wl, b, h, 0.3) for h in range(wl.H)]) for b in range(wl.B)])
          if nonzero else None)
    return wl, x, S0


def _worker(rank, world, port, T, nonzero, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl, x, S0 = _inputs(T, nonzero)
        t0, t1 = context_parallel.frame_ranges(T, world)[rank]
        t = {key: torch.from_numpy(np.ascontiguousarray(x[key][:, :, t0:t1], np.float64))
             for key in ("q", "k", "v", "g", "beta")}
        si = None if S0 is None else torch.from_numpy(S0.astype(np.float64))
        o, s = context_parallel.frame_fwd_cp(t["q"], t["k"], t["v"], t["g"], t["beta"], state_in=si,
                                             ops=OracleOps())
        out[rank] = (o.numpy(), s.numpy())
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,T,nonzero", [(2, 8, False), (2, 7, True), (3, 8, True), (3, 2, False)])
def test_ranks_compose_into_the_single_pass(world, T, nonzero):
    """R gloo ranks, each with its contiguous frame range (T = 2 over 3 ranks gives
    one rank no frames): concatenated outputs and every rank's final state equal
    the oracle's one pass over all frames."""
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, _free_port(), T, nonzero, out), nprocs=world, join=True)
        res = dict(out)
    wl, x, S0 = _inputs(T, nonzero)
    ro, rs = oracle.frame_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], S0)
    got = np.concatenate([res[r][0] for r in range(world)], axis=2)
    np.testing.assert_allclose(got, ro, rtol=0, atol=1e-12)
    for r in range(world):
        np.testing.assert_allclose(res[r][1], rs, rtol=0, atol=1e-12)


def test_a_wrong_fold_order_is_caught():
    """The check above can fail: folding the earlier ranges' maps in reverse order
    (a plausible driver mistake) gives a different entering state."""
    wl, x, _ = _inputs(9, False)
    ops = OracleOps()
    parts = []
    for t0, t1 in context_parallel.frame_ranges(9, 3):
        t = {key: torch.from_numpy(np.ascontiguousarray(x[key][:, :, t0:t1], np.float64)) for key in ("k", "v", "g",
                                                                                                      "beta")}
        parts.append(ops.summary(t["k"], t["v"], t["g"], t["beta"], False))
    right, wrong = None, None
    for r in (0, 1):
        right = ops.apply(*parts[r], right)
    for r in (1, 0):
        wrong = ops.apply(*parts[r], wrong)
    _, rs = oracle.scan_head(x["q"][0, 0, :6], x["k"][0, 0, :6], x["v"][0, 0, :6], x["g"][0, 0, :6],
                             x["beta"][0, 0, :6])
    np.testing.assert_allclose(right[0, 0].numpy(), rs, atol=1e-12)
    assert np.abs(wrong[0, 0].numpy() - rs).max() > 1e-6


def test_frame_ranges_cover_the_sequence_in_order():
    for T in (0, 1, 5, 961):
        for world in (1, 2, 3, 8):
            rs = context_parallel.frame_ranges(T, world)
            assert len(rs) == world and rs[0][0] == 0 and rs[-1][1] == T
            assert all(a[1] == b[0] for a, b in zip(rs, rs[1:]))
            assert max(b - a for a, b in rs) - min(b - a for a, b in rs) <= 1


# ------------------------------------------------------------------ C ABI, host side

A16 = 0x10000
MIS = 0x10008


@pytest.fixture(scope="module")
def lib():
    build_lib.build()
    return binding.lib()


@pytest.mark.parametrize("kw,code", [
    (dict(B=0), 1), (dict(H=0), 1), (dict(T=-1), 1), (dict(S=0), 1), (dict(D=24), 2), (dict(D=144), 2),
    (dict(dtype=3), 1), (dict(flags=2), 1), (dict(A=None), 1), (dict(bo=None), 1), (dict(k=None), 1),
    (dict(A=MIS), 3), (dict(bo=MIS), 3), (dict(k=MIS), 3), (dict(g=A16 + 2), 3),
    (dict(ws=None), 6), (dict(wsb=16), 6), (dict(ws=A16 + 16), 3),
])
def test_summary_rejects(lib, kw, code):
    a = dict(k=A16, v=A16, g=A16, beta=A16, A=A16, bo=A16, B=1, H=2, T=3, S=17, D=32, dtype=1, flags=0, ws=A16,
             wsb=1 << 40)
    a.update(kw)
    rc = binding.gdn_frame_summary(a["k"], a["v"], a["g"], a["beta"], a["A"], a["bo"], a["B"], a["H"], a["T"],
                                   a["S"], a["D"], a["dtype"], a["flags"], a["ws"], a["wsb"], None)
    assert rc == code


@pytest.mark.parametrize("kw,code", [
    (dict(B=0), 1), (dict(H=0), 1), (dict(D=8), 2), (dict(D=136), 2), (dict(A=None), 1), (dict(b=None), 1),
    (dict(so=None), 1), (dict(A=MIS), 3), (dict(si=MIS), 3), (dict(so=MIS), 3),
])
def test_apply_rejects(lib, kw, code):
    a = dict(A=A16, b=A16, si=None, so=A16, B=1, H=2, D=32)
    a.update(kw)
    assert binding.gdn_summary_apply(a["A"], a["b"], a["si"], a["so"], a["B"], a["H"], a["D"], None) == code


def test_summary_workspace_is_the_prefix_forms(lib):
    for dt in (0, 1):
        n = binding.gdn_summary_workspace_bytes(1, 20, 961, 880, 112, dt)
        assert n > 0 and n == binding.gdn_workspace_bytes(1, 20, 961, 880, 112, dt, binding.GDN_MODE_PREFIX)
    assert binding.gdn_summary_workspace_bytes(1, 20, 0, 880, 112, 1) == 0
    assert binding.gdn_summary_workspace_bytes(1, 20, 9, 880, 24, 1) == 0
