"""bench.py's algorithmic work against the per-workload figures stated for the
measurement (each of q, k, v, out crossing HBM once, g and beta read once, the
state in and out once; 6 S D^2 flop per frame-head): 0.335 GB / 27.8 GF (short),
15.22 GB / 1.273 TF (minute), 57.09 GB / 5.459 TF (large).  Also the per-kernel
shares the roofline uses, and the backward's accounting."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from linear_attention_video_gated_b300 import synth  # noqa: E402


@pytest.mark.parametrize("name,gb,tf", [("short", 0.335, 0.0278), ("minute", 15.22, 1.273), ("large", 57.09, 5.459)])
def test_forward_work_matches_the_stated_figures(name, gb, tf):
    wl = synth.WORKLOADS[name]
    assert bench.alg_bytes(wl) / 1e9 == pytest.approx(gb, rel=2e-3)
    assert bench.alg_flops(wl) / 1e12 == pytest.approx(tf, rel=2e-3)


def test_tokens_per_call():
    assert synth.WORKLOADS["minute"].tokens == 845680
    assert synth.WORKLOADS["large"].tokens == 3470400


def test_kernel_shares_cover_the_call():
    """gram (k, v, beta, g) + read-out (q, out) = every algorithmic byte but the state's."""
    wl = synth.WORKLOADS["minute"]
    state = 2 * 4 * wl.B * wl.H * wl.D * wl.D
    assert bench.kernel_alg_bytes("tc_gram", wl) + bench.kernel_alg_bytes("tc_readout", wl) == \
        bench.alg_bytes(wl) - state
    assert bench.kernel_alg_bytes("tc_scan", wl) is None  # workspace traffic only


def test_backward_work():
    """Backward: seven S x D tensors cross HBM once (q, k, v, dout in; dq, dk, dv out),
    g and beta in, dg and dbeta out, the state and its two gradients; 14 S D^2 flop."""
    wl = synth.WORKLOADS["minute"]
    n = wl.B * wl.H * wl.T * wl.S * wl.D
    assert bench.alg_bytes_bwd(wl) - bench.alg_bytes(wl) == pytest.approx(3 * n * 2 + 4 * wl.B * wl.H * wl.T * (1 + wl.S)
                                                                          + 4 * wl.B * wl.H * wl.D * wl.D)
    assert bench.alg_bytes_bwd(wl) / 1e9 == pytest.approx(26.6, rel=5e-3)
    assert bench.alg_flops_bwd(wl) == pytest.approx(14 / 6 * bench.alg_flops(wl))
    fh = wl.B * wl.H * wl.T
    assert bench.kernel_alg_bytes("tc_bwd_kv_grad", wl) == fh * (4 * wl.S * wl.D * 2 + 8 * wl.S + 4)
    assert bench.kernel_alg_bytes("tc_bwd_q_grad", wl) == fh * 2 * wl.S * wl.D * 2


def test_link_bound_reduces_to_the_textbook_cases():
    # full duplex (each direction keeps its rate): the slower direction alone
    full = {"h2d_gbs": 50.0, "d2h_gbs": 40.0, "duplex_h2d_gbs": 50.0, "duplex_d2h_gbs": 40.0}
    assert abs(bench.link_bound_ms(10e9, 4e9, full) - 200.0) < 1e-9  # 10 GB at 50 GB/s
    assert abs(bench.link_bound_ms(1e9, 8e9, full) - 200.0) < 1e-9   # 8 GB at 40 GB/s
    # half duplex (the directions split one link): the bytes add up
    half = {"h2d_gbs": 50.0, "d2h_gbs": 50.0, "duplex_h2d_gbs": 25.0, "duplex_d2h_gbs": 25.0}
    assert abs(bench.link_bound_ms(3e9, 2e9, half) - 100.0) < 1e-9
    # one direction only
    assert abs(bench.link_bound_ms(5e9, 0.0, half) - 100.0) < 1e-9
    # in between (as measured on one B300 host): between the two extremes
    meas = {"h2d_gbs": 55.6, "d2h_gbs": 57.3, "duplex_h2d_gbs": 37.4, "duplex_d2h_gbs": 54.4}
    b = bench.link_bound_ms(11.43e9, 3.79e9, meas)
    assert 11.43e9 / 55.6e6 < b < 11.43e9 / 55.6e6 + 3.79e9 / 57.3e6
