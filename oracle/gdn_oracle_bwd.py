"""Backward pass of the frame-wise Gated DeltaNet scan: a plain, slow, fp64 oracle.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Plain numpy in float64.

The pages train SANA-WM with this layer (zhichai.net SANA-WM summary, training
pipeline, Stages 1-4, the 64-GPU run) but print no backward pass; the gradient
is fixed by the forward definition alone (``gdn_oracle.frame_step``).  This
module is that forward scan differentiated by reverse-mode calculus, one
adjoint per forward step, taken in the reverse of the forward order:

    forward, frame t              adjoint (dX is dLoss/dX)
    K~  = c K                     dK   = c dK~
    P   = K~ S_{t-1}              dK~ += dP S_{t-1}^T        dS_{t-1} += K~^T dP
    R   = diag(b)(V - g P)        dV   = diag(b) dR          dP = -g diag(b) dR
                                  db_s = <dR_s, V_s - g P_s> dg  -= sum_s b_s <dR_s, P_s>
    S_t = g S_{t-1} + K~^T R      dS_{t-1} += g dS_t         dg += <dS_t, S_{t-1}>
                                  dK~  = R dS_t^T            dR  = K~ dS_t
    O_t = Q S_t / sqrt(D)         dQ   = dO S_t^T / sqrt(D)  dS_t += Q^T dO / sqrt(D)

with c = 1/sqrt(D*S) and <X, Y> the sum of the elementwise product.  The loss
is any L whose gradient with respect to the outputs is (dO, dS_T): the caller
passes dO (the gradient of every frame's output) and dS_T (that of the final
state, or zero).  The state gradient flowing back through frame t is
dS_{t-1} = g (dS_t - M_t dS_t) with M_t = K~^T diag(b) K~: the same affine map
the forward applies, run from the last frame to the first.
"""
from __future__ import annotations

import numpy as np

from . import gdn_oracle as fw

F64 = np.float64


def readout_adjoint(Qt, St, dO, D):
    """O = Q S / sqrt(D): returns (dQ, the contribution to dS)."""
    c = fw.out_scale(D)
    return (dO @ St.T) * c, (Qt.T @ dO) * c


def write_adjoint(S_prev, Kt, R, g, dS):
    """S_t = g S_{t-1} + K~^T R: returns (dS_{t-1} part, dg part, dK~ part, dR)."""
    return g * dS, float(np.sum(dS * S_prev)), R @ dS.T, Kt @ dS


def residual_adjoint(Vt, P, g, beta, dR):
    """R = diag(beta) (V - g P): returns (dV, dP, dbeta, dg part)."""
    dV = beta[:, None] * dR
    dP = -g * beta[:, None] * dR
    dbeta = np.sum(dR * (Vt - g * P), axis=1)
    dg = -float(np.sum(beta[:, None] * dR * P))
    return dV, dP, dbeta, dg


def predict_adjoint(Kt, S_prev, dP):
    """P = K~ S_{t-1}: returns (dK~ part, dS_{t-1} part)."""
    return dP @ S_prev.T, Kt.T @ dP


def backward_head(q, k, v, g, beta, S0, dout, dS_T=None):
    """Gradients of one (b, h) head.

    q, k, v, dout: [T, S, D]; g: [T]; beta: [T, S]; S0: [D, D] or None (zeros);
    dS_T: [D, D] or None (zeros).  Returns a dict of dq, dk, dv [T, S, D],
    dg [T], dbeta [T, S] and dS0 [D, D], all float64.
    """
    q, k, v, dout = (np.asarray(a, F64) for a in (q, k, v, dout))
    g = np.asarray(g, F64)
    beta = np.asarray(beta, F64)
    T, S, D = k.shape
    S0 = np.zeros((D, D), F64) if S0 is None else np.array(S0, F64)
    # forward pass, keeping every state: states[t] is S_{t-1} (states[0] = S0)
    _, _, kept = fw.scan_head(q, k, v, g, beta, S0, keep_states=True)
    states = [S0] + kept
    c = fw.key_scale(D, S)
    grads = {"dq": np.zeros_like(q), "dk": np.zeros_like(k), "dv": np.zeros_like(v),
             "dg": np.zeros(T, F64), "dbeta": np.zeros((T, S), F64)}
    dS = np.zeros((D, D), F64) if dS_T is None else np.array(dS_T, F64)
    for t in reversed(range(T)):
        S_prev, S_t = states[t], states[t + 1]
        # recompute the frame's forward intermediates
        Kt = k[t] * c
        P = fw.predict(Kt, S_prev)
        R = fw.residual(v[t], P, g[t], beta[t])
        # read-out
        dQ, dS_read = readout_adjoint(q[t], S_t, dout[t], D)
        dS = dS + dS_read
        # write
        dS_prev, dg_w, dK, dR = write_adjoint(S_prev, Kt, R, g[t], dS)
        # residual
        dV, dP, dbeta, dg_r = residual_adjoint(v[t], P, g[t], beta[t], dR)
        # prediction
        dK_p, dS_prev_p = predict_adjoint(Kt, S_prev, dP)
        grads["dq"][t] = dQ
        grads["dk"][t] = (dK + dK_p) * c
        grads["dv"][t] = dV
        grads["dg"][t] = dg_w + dg_r
        grads["dbeta"][t] = dbeta
        dS = dS_prev + dS_prev_p
    grads["dS0"] = dS
    return grads


def frame_bwd(q, k, v, g, beta, state_in, dout, dstate_out=None):
    """Whole-tensor gradients: inputs as ``gdn_oracle.frame_fwd`` takes them plus
    dout [B,H,T,S,D] and dstate_out [B,H,D,D] (or None).  Returns a dict of
    dq, dk, dv [B,H,T,S,D], dg [B,H,T], dbeta [B,H,T,S], dstate_in [B,H,D,D]."""
    B, H, T, S, D = np.shape(k)
    out = {"dq": np.zeros((B, H, T, S, D), F64), "dk": np.zeros((B, H, T, S, D), F64),
           "dv": np.zeros((B, H, T, S, D), F64), "dg": np.zeros((B, H, T), F64),
           "dbeta": np.zeros((B, H, T, S), F64), "dstate_in": np.zeros((B, H, D, D), F64)}
    for b in range(B):
        for h in range(H):
            S0 = None if state_in is None else state_in[b, h]
            dST = None if dstate_out is None else dstate_out[b, h]
            gr = backward_head(q[b, h], k[b, h], v[b, h], g[b, h], beta[b, h], S0, dout[b, h], dST)
            for key in ("dq", "dk", "dv", "dg", "dbeta"):
                out[key][b, h] = gr[key]
            out["dstate_in"][b, h] = gr["dS0"]
    return out


def gate_logit_adjoint(g_logit, beta_logit, dg, dbeta):
    """Chain rule through the gate prologue g = exp(-softplus(x)), beta = sigmoid(y):
    dg/dx = -g sigmoid(x) = -g (1 - g) and dbeta/dy = beta (1 - beta).
    Returns (dx, dy)."""
    g = fw.decay_from_logit(g_logit)
    b = fw.beta_from_logit(beta_logit)
    return -np.asarray(dg, F64) * g * (1.0 - g), np.asarray(dbeta, F64) * b * (1.0 - b)


def frame_bwd_from_logits(q, k, v, g_logit, beta_logit, state_in, dout, dstate_out=None):
    """frame_bwd for the scan whose gates are given as logits: the gradients of
    the logits in place of those of g and beta (keys dg_logit, dbeta_logit)."""
    gr = frame_bwd(q, k, v, fw.decay_from_logit(g_logit), fw.beta_from_logit(beta_logit), state_in, dout,
                   dstate_out)
    gr["dg_logit"], gr["dbeta_logit"] = gate_logit_adjoint(g_logit, beta_logit, gr.pop("dg"), gr.pop("dbeta"))
    return gr
