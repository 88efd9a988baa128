"""Pins of the oracle's backward pass against what the mathematics fixes,
independently of the hand derivation it follows:

* central finite differences of the forward oracle, for every element of every
  input (q, k, v, g, beta, the initial state), on tiny inputs;
* Euler's identity for the parts of the scan that are linear: the outputs are
  linear in Q, and jointly linear in (S_0, V), so <dQ, Q> = <dO, O> and
  <dV, V> + <dS_0, S_0> = L exactly;
* special cases: beta = 0 writes nothing, so no gradient reaches K or V; g = 0
  in the first frame cuts the initial state off.

``test_planted_mistake_is_caught`` plants a dropped term, a wrong sign or a
transposed operand in each adjoint step (monkeypatched, on the CPU) and checks
that a pin fails for each.
"""
import numpy as np
import pytest

import oracle
import oracle.gdn_oracle as fw
import oracle.gdn_oracle_bwd as bw


def _inputs(seed=0, B=1, H=2, T=3, S=5, D=4, beta_zero=False, g0_zero=False):
    rng = np.random.default_rng(seed)
    x = {
        "q": rng.standard_normal((B, H, T, S, D)),
        "k": rng.standard_normal((B, H, T, S, D)),
        "v": rng.standard_normal((B, H, T, S, D)),
        "g": rng.uniform(0.3, 1.0, (B, H, T)),
        "beta": rng.uniform(0.0, 1.0, (B, H, T, S)),
        "state_in": 0.3 * rng.standard_normal((B, H, D, D)),
    }
    if beta_zero:
        x["beta"][:] = 0.0
    if g0_zero:
        x["g"][:, :, 0] = 0.0
    dout = rng.standard_normal((B, H, T, S, D))
    dst = 0.3 * rng.standard_normal((B, H, D, D))
    return x, dout, dst


def _loss(x, dout, dst):
    o, s = fw.frame_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["state_in"])
    return float(np.sum(dout * o) + np.sum(dst * s))


def _grads(x, dout, dst):
    return bw.frame_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["state_in"], dout, dst)


GRAD_OF = {"q": "dq", "k": "dk", "v": "dv", "g": "dg", "beta": "dbeta", "state_in": "dstate_in"}


def _fd_errors(x, dout, dst, eps=1e-6):
    """max |analytic - central difference| / (1 + |analytic|) per input."""
    gr = _grads(x, dout, dst)
    errs = {}
    for name, gname in GRAD_OF.items():
        a = x[name]
        num = np.zeros_like(a)
        for idx in np.ndindex(a.shape):
            old = a[idx]
            a[idx] = old + eps
            lp = _loss(x, dout, dst)
            a[idx] = old - eps
            lm = _loss(x, dout, dst)
            a[idx] = old
            num[idx] = (lp - lm) / (2 * eps)
        errs[name] = float(np.max(np.abs(gr[gname] - num) / (1.0 + np.abs(gr[gname]))))
    return errs


def pin_finite_differences():
    x, dout, dst = _inputs(seed=1)
    errs = _fd_errors(x, dout, dst)
    return all(e < 1e-6 for e in errs.values())


def pin_euler_identities():
    x, dout, dst = _inputs(seed=2, T=4, S=6, D=4)
    gr = _grads(x, dout, dst)
    L = _loss(x, dout, dst)
    o, _ = fw.frame_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["state_in"])
    lin_q = float(np.sum(gr["dq"] * x["q"]))
    lin_vs = float(np.sum(gr["dv"] * x["v"]) + np.sum(gr["dstate_in"] * x["state_in"]))
    return abs(lin_q - float(np.sum(dout * o))) < 1e-10 * (1 + abs(lin_q)) and abs(lin_vs - L) < 1e-10 * (1 + abs(L))


def pin_beta_zero_writes_nothing():
    x, dout, dst = _inputs(seed=3, beta_zero=True)
    gr = _grads(x, dout, dst)
    return not np.any(gr["dk"]) and not np.any(gr["dv"]) and np.any(gr["dbeta"])


def pin_first_gate_zero_cuts_initial_state():
    x, dout, dst = _inputs(seed=4, g0_zero=True)
    gr = _grads(x, dout, dst)
    return not np.any(gr["dstate_in"]) and np.any(gr["dg"][:, :, 0])


PINS = [pin_finite_differences, pin_euler_identities, pin_beta_zero_writes_nothing,
        pin_first_gate_zero_cuts_initial_state]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    assert pin()


def test_finite_differences_with_zero_initial_state_and_no_state_gradient():
    """The None defaults: zero initial state, no gradient on the final state."""
    x, dout, _ = _inputs(seed=5, H=1, T=2, S=3, D=4)
    gr = bw.frame_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], None, dout, None)
    x["state_in"][:] = 0.0
    gr2 = _grads(x, dout, np.zeros_like(x["state_in"]))
    for key in ("dq", "dk", "dv", "dg", "dbeta", "dstate_in"):
        np.testing.assert_array_equal(gr[key], gr2[key])
    errs = _fd_errors(x, dout, np.zeros_like(x["state_in"]))
    assert all(e < 1e-6 for e in errs.values()), errs


def test_logit_gradients_match_finite_differences():
    """Gradients of the logits of the gate prologue g = exp(-softplus(x)),
    beta = sigmoid(y), by central differences of frame_fwd_from_logits."""
    rng = np.random.default_rng(6)
    B, H, T, S, D = 1, 1, 3, 4, 4
    q, k, v = (rng.standard_normal((B, H, T, S, D)) for _ in range(3))
    xl = rng.standard_normal((B, H, T))
    yl = rng.standard_normal((B, H, T, S))
    s0 = 0.3 * rng.standard_normal((B, H, D, D))
    dout = rng.standard_normal((B, H, T, S, D))
    dst = 0.3 * rng.standard_normal((B, H, D, D))

    def loss():
        o, s = fw.frame_fwd_from_logits(q, k, v, xl, yl, s0)
        return float(np.sum(dout * o) + np.sum(dst * s))

    gr = oracle.frame_bwd_from_logits(q, k, v, xl, yl, s0, dout, dst)
    eps = 1e-6
    for a, key in ((xl, "dg_logit"), (yl, "dbeta_logit")):
        for idx in np.ndindex(a.shape):
            old = a[idx]
            a[idx] = old + eps
            lp = loss()
            a[idx] = old - eps
            lm = loss()
            a[idx] = old
            assert abs((lp - lm) / (2 * eps) - gr[key][idx]) < 1e-6 * (1 + abs(gr[key][idx]))


def test_gradients_are_linear_in_the_upstream_gradient():
    """The backward pass is a linear map of (dO, dS_T): scaling them scales every gradient."""
    x, dout, dst = _inputs(seed=7)
    g1 = _grads(x, dout, dst)
    g2 = _grads(x, 2.5 * dout, 2.5 * dst)
    for key in g1:
        np.testing.assert_allclose(g2[key], 2.5 * g1[key], rtol=1e-12, atol=1e-13)


# ---- planted mistakes -----------------------------------------------------------

_true_residual_adjoint = bw.residual_adjoint


def _mut_readout_untransposed(Qt, St, dO, D):
    c = fw.out_scale(D)
    return (dO @ St) * c, (Qt.T @ dO) * c


def _mut_readout_no_state_term(Qt, St, dO, D):
    c = fw.out_scale(D)
    return (dO @ St.T) * c, 0.0 * St


def _mut_write_no_decay(S_prev, Kt, R, g, dS):
    return dS, float(np.sum(dS * S_prev)), R @ dS.T, Kt @ dS


def _mut_write_gate_term_dropped(S_prev, Kt, R, g, dS):
    return g * dS, 0.0, R @ dS.T, Kt @ dS


def _mut_write_key_grad_transposed(S_prev, Kt, R, g, dS):
    return g * dS, float(np.sum(dS * S_prev)), R @ dS, Kt @ dS


def _mut_residual_sign(Vt, P, g, beta, dR):
    dV, dP, dbeta, dg = _true_residual_adjoint(Vt, P, g, beta, dR)
    return dV, -dP, dbeta, dg


def _mut_residual_beta_grad_no_gate(Vt, P, g, beta, dR):
    dV, dP, _, dg = _true_residual_adjoint(Vt, P, g, beta, dR)
    return dV, dP, np.sum(dR * (Vt - P), axis=1), dg


def _mut_predict_no_state_term(Kt, S_prev, dP):
    return dP @ S_prev.T, 0.0 * S_prev


def _mut_predict_untransposed(Kt, S_prev, dP):
    return dP @ S_prev, Kt.T @ dP


MUTATIONS = [
    ("readout_adjoint", _mut_readout_untransposed),
    ("readout_adjoint", _mut_readout_no_state_term),
    ("write_adjoint", _mut_write_no_decay),
    ("write_adjoint", _mut_write_gate_term_dropped),
    ("write_adjoint", _mut_write_key_grad_transposed),
    ("residual_adjoint", _mut_residual_sign),
    ("residual_adjoint", _mut_residual_beta_grad_no_gate),
    ("predict_adjoint", _mut_predict_no_state_term),
    ("predict_adjoint", _mut_predict_untransposed),
]


@pytest.mark.parametrize("target,fn", MUTATIONS, ids=[m[1].__name__ for m in MUTATIONS])
def test_planted_mistake_is_caught(monkeypatch, target, fn):
    monkeypatch.setattr(bw, target, fn)
    failed = []
    for pin in PINS:
        try:
            ok = pin()
        except Exception:  # a shape error also counts as caught
            ok = False
        if not ok:
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {fn.__name__}"
