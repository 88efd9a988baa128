"""Pins of the oracle's gate prologue (raw logits -> decay g, delta-rule weight
beta), against values the mathematics fixes and an independent library routine:
scipy's expit (the logistic function), which the oracle does not use."""
import numpy as np
import pytest
from scipy.special import expit

import oracle
from linear_attention_video_gated_b300 import synth

XS = np.concatenate([np.linspace(-40, 40, 801), [-700.0, -100.0, 100.0, 700.0, 0.0]])


def test_gates_at_zero_are_one_half():
    assert oracle.decay_from_logit(0.0) == 0.5
    assert oracle.beta_from_logit(0.0) == 0.5


def test_gates_match_the_logistic_function():
    """exp(-softplus(x)) = 1 / (1 + e^x) = expit(-x); sigmoid(x) = expit(x)."""
    np.testing.assert_allclose(oracle.decay_from_logit(XS), expit(-XS), rtol=1e-13, atol=0)
    np.testing.assert_allclose(oracle.beta_from_logit(XS), expit(XS), rtol=1e-13, atol=0)


def test_gates_are_complementary_and_bounded():
    g, b = oracle.decay_from_logit(XS), oracle.beta_from_logit(XS)
    assert np.all((g >= 0) & (g <= 1) & (b >= 0) & (b <= 1))
    np.testing.assert_allclose(g + b, 1.0, rtol=0, atol=1e-15)


def test_softplus_identity():
    """softplus(x) - softplus(-x) = x, and softplus(x) > max(x, 0)."""
    np.testing.assert_allclose(oracle.softplus(XS) - oracle.softplus(-XS), XS, rtol=1e-12, atol=1e-12)
    assert np.all(oracle.softplus(XS) >= np.maximum(XS, 0.0))


def test_scan_from_logits_equals_scan_of_gates():
    """The logit entry point is the gate prologue followed by the scan: with the
    logits mapped by the independent routine the plain scan gives the same result."""
    wl = synth.WORKLOADS["short"].with_(H=2, T=4, S=24, D=16, seed=31)
    x = synth.full(wl)
    lg = synth.logits_full(wl)
    o1, s1 = oracle.frame_fwd_from_logits(x["q"], x["k"], x["v"], lg["g_logit"], lg["beta_logit"])
    o2, s2 = oracle.frame_fwd(x["q"], x["k"], x["v"], expit(-lg["g_logit"].astype(np.float64)),
                              expit(lg["beta_logit"].astype(np.float64)))
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(s1, s2, rtol=1e-12, atol=1e-14)


def test_workload_gates_are_the_mapped_logits():
    """synth's gates are the same draws as its logits, mapped (to float32)."""
    wl = synth.WORKLOADS["short"]
    for (b, h, t) in [(0, 0, 0), (0, 7, 3), (0, 19, 20)]:
        assert abs(float(synth.gate(wl, b, h, t)) - oracle.decay_from_logit(synth.gate_logit(wl, b, h, t))) < 1e-7
        np.testing.assert_allclose(synth.beta(wl, b, h, t), oracle.beta_from_logit(synth.beta_logit(wl, b, h, t)),
                                   rtol=1e-6, atol=1e-7)


def test_uniform_gates_have_no_logits():
    with pytest.raises(ValueError):
        synth.gate_logit(synth.WORKLOADS["tiny"], 0, 0, 0)
