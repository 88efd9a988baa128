"""Pins of the oracle's baseline: SANA-Video's cumulative ReLU linear attention,
S_t = S_{t-1} + relu(K_t)^T V_t / sqrt(D*S), O_t = relu(Q_t) S_t / sqrt(D).
Each pin computes the value another way than the oracle's frame loop."""
import numpy as np

import oracle
from linear_attention_video_gated_b300 import synth


def _x(T=5, S=12, D=16, H=2, seed=3):
    wl = synth.WORKLOADS["short"].with_(H=H, T=T, S=S, D=D, seed=seed)
    return wl, synth.full(wl)


def test_final_state_is_one_product_over_all_frames():
    """Accumulating every frame's write equals one product over the frames stacked."""
    wl, x = _x()
    _, st = oracle.relu_linear_fwd(x["q"], x["k"], x["v"])
    for h in range(wl.H):
        K = np.maximum(x["k"][0, h].reshape(-1, wl.D).astype(np.float64), 0) / np.sqrt(wl.D * wl.S)
        V = x["v"][0, h].reshape(-1, wl.D).astype(np.float64)
        np.testing.assert_allclose(st[0, h], K.T @ V, rtol=1e-12, atol=1e-13)


def test_outputs_are_cumulative_sums():
    """O_t = relu(Q_t) (sum over s <= t of the frame writes) / sqrt(D), with the sums
    taken by np.cumsum over per-frame products (einsum)."""
    wl, x = _x()
    out, _ = oracle.relu_linear_fwd(x["q"], x["k"], x["v"])
    for h in range(wl.H):
        k = np.maximum(x["k"][0, h].astype(np.float64), 0) / np.sqrt(wl.D * wl.S)
        writes = np.einsum("tsi,tsj->tij", k, x["v"][0, h].astype(np.float64))
        states = np.cumsum(writes, axis=0)
        ref = np.einsum("tsi,tij->tsj", np.maximum(x["q"][0, h].astype(np.float64), 0), states) / np.sqrt(wl.D)
        np.testing.assert_allclose(out[0, h], ref, rtol=1e-11, atol=1e-13)


def test_negative_keys_write_nothing():
    """relu zeroes negative keys: the state stays the initial state."""
    wl, x = _x()
    k = -np.abs(x["k"])
    S0 = np.stack([np.stack([synth.state(wl, 0, h) for h in range(wl.H)])])
    out, st = oracle.relu_linear_fwd(x["q"], k, x["v"], S0)
    np.testing.assert_allclose(st, S0, rtol=0, atol=0)
    ref = np.einsum("htsi,hij->htsj", np.maximum(x["q"][0].astype(np.float64), 0), S0[0].astype(np.float64))
    np.testing.assert_allclose(out[0], ref / np.sqrt(wl.D), rtol=1e-12, atol=1e-14)


def test_equals_gdn_without_decay_or_prediction():
    """With g = 1 and beta = 1, and each frame's keys nonnegative and on coordinates
    no other frame uses, GDN's prediction K~ S_{t-1} is zero, so GDN and the
    baseline agree exactly: the two differ only in the decay, the delta rule and
    the feature map."""
    T, S, D = 4, 6, 16
    rng = np.random.default_rng(11)
    k = np.zeros((1, 1, T, S, D))
    for t in range(T):
        k[0, 0, t, :, 4 * t:4 * t + 4] = np.abs(rng.standard_normal((S, 4)))
    q = rng.standard_normal((1, 1, T, S, D))
    v = rng.standard_normal((1, 1, T, S, D))
    g = np.ones((1, 1, T))
    beta = np.ones((1, 1, T, S))
    o1, s1 = oracle.frame_fwd(np.maximum(q, 0), k, v, g, beta)
    o2, s2 = oracle.relu_linear_fwd(q, k, v)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(s1, s2, rtol=1e-12, atol=1e-14)
