"""Pins for the fp64 oracle: what the pages and the mathematics fix, checked
against something other than the oracle's own formula.

Each pin is a plain function ``pin_*(og)`` taking the oracle module, so that
``test_oracle_mutations.py`` can run every pin against an oracle with a planted
mistake and show that some pin fails.
"""
import json
import os

import numpy as np
import pytest

import oracle.gdn_oracle as ORACLE
from linear_attention_video_gated_b300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
TOL = 1e-11


def _rand_head(rng, T, S, D, Dv=None, g_lo=0.05, g_hi=1.0):
    Dv = D if Dv is None else Dv
    return dict(q=rng.standard_normal((T, S, D)), k=rng.standard_normal((T, S, D)),
                v=rng.standard_normal((T, S, Dv)), g=rng.uniform(g_lo, g_hi, T),
                beta=rng.uniform(0, 1, (T, S)))


def _close(a, b, tol=TOL):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    scale = max(1.0, float(np.max(np.abs(b))) if b.size else 1.0)
    return a.shape == b.shape and float(np.max(np.abs(a - b))) <= tol * scale if a.size else a.shape == b.shape


# --------------------------------------------------------------------------- pins

def pin_golden_hand_example(og):
    """Hand-derived two-frame example (tests/golden/hand_example_d2_s2_t2.json)."""
    with open(os.path.join(GOLDEN, "hand_example_d2_s2_t2.json")) as f:
        ex = json.load(f)
    i = ex["inputs"]
    out, ST, states = og.scan_head(i["q"], i["k"], i["v"], i["g"], i["beta"], keep_states=True)
    ok = _close(np.array(states), ex["expected"]["states"])
    ok &= _close(out * np.sqrt(2.0), ex["expected"]["out_times_sqrt_D"])
    ok &= _close(ST, ex["expected"]["states"][-1])
    return ok


def pin_delta_rule_exact_write(og):
    """S = 1 token, key of unit scaled norm (k = sqrt(D) u, |u| = 1), beta = 1:
    the delta rule stores the target exactly, u^T S_t = v_t, for any decay and any
    previous state."""
    rng = np.random.default_rng(11)
    D, T = 8, 6
    ok = True
    St = rng.standard_normal((D, D))
    for t in range(T):
        u = rng.standard_normal(D)
        u /= np.linalg.norm(u)
        k = (np.sqrt(D) * u)[None, :]
        v = rng.standard_normal((1, D))
        q = rng.standard_normal((1, D))
        g = rng.uniform(0.1, 1.0)
        _, St = og.scan_head(q[None], k[None], v[None], [g], [[1.0]], S0=St)
        ok &= _close(u @ St, v[0])
    return ok


def pin_beta_zero_pure_decay(og):
    """beta = 0: nothing is written; the state only decays, S_t = (prod g) S0,
    and with a zero initial state every output and the final state are 0."""
    rng = np.random.default_rng(12)
    T, S, D = 5, 7, 6
    h = _rand_head(rng, T, S, D)
    h["beta"] = np.zeros((T, S))
    out0, st0 = og.scan_head(**h)
    ok = _close(out0, np.zeros_like(out0)) and _close(st0, np.zeros((D, D)))
    S0 = rng.standard_normal((D, D))
    out, st, states = og.scan_head(**h, S0=S0, keep_states=True)
    decay = np.cumprod(h["g"])
    for t in range(T):
        ok &= _close(states[t], decay[t] * S0)
    return ok


def pin_gate_zero_memoryless(og):
    """g = 0: the previous state is forgotten and the prediction term vanishes, so
    frame t's state and output do not depend on any earlier frame or on S0."""
    rng = np.random.default_rng(13)
    T, S, D = 4, 9, 5
    h = _rand_head(rng, T, S, D)
    h["g"] = np.zeros(T)
    out, _, states = og.scan_head(**h, S0=rng.standard_normal((D, D)), keep_states=True)
    ok = True
    for t in range(T):
        one = {k: v[t:t + 1] for k, v in h.items()}
        o1, s1 = og.scan_head(**one, S0=rng.standard_normal((D, D)))
        ok &= _close(states[t], s1) and _close(out[t], o1[0])
    return ok


def _disjoint_keys(rng, T, S, D):
    """Frame t's keys live on coordinates {2t, 2t+1} only."""
    k = np.zeros((T, S, D))
    for t in range(T):
        k[t, :, 2 * t: 2 * t + 2] = rng.standard_normal((S, 2))
    return k


def pin_cumulative_linear_attention(og):
    """Keys of different frames on disjoint coordinates, zero initial state: every
    prediction K~_t S_{t-1} is exactly 0, so with g = 1 and beta = 1 the scan is
    textbook causal (cumulative) linear attention at frame granularity,
    O_t = Q_t (sum_{s<=t} K~_s^T V_s) / sqrt(D): computed here with a cumsum."""
    rng = np.random.default_rng(14)
    T, S, D = 8, 5, 16
    q = rng.standard_normal((T, S, D))
    v = rng.standard_normal((T, S, D))
    k = _disjoint_keys(rng, T, S, D)
    out, _ = og.scan_head(q, k, v, np.ones(T), np.ones((T, S)))
    kt = k / np.sqrt(D * S)
    kv = np.cumsum(np.einsum("tsi,tsj->tij", kt, v), axis=0)
    ref = np.einsum("tsi,tij->tsj", q, kv) / np.sqrt(D)
    return _close(out, ref)


def pin_gated_cumulative_linear_attention(og):
    """Same disjoint-key setting with per-frame decay and per-token beta: the scan is
    gated linear attention, S_t = sum_{s<=t} (prod_{s<r<=t} g_r) K~_s^T diag(beta_s) V_s."""
    rng = np.random.default_rng(15)
    T, S, D = 8, 6, 16
    q = rng.standard_normal((T, S, D))
    v = rng.standard_normal((T, S, D))
    k = _disjoint_keys(rng, T, S, D)
    g = rng.uniform(0.2, 1.0, T)
    beta = rng.uniform(0, 1, (T, S))
    out, _, states = og.scan_head(q, k, v, g, beta, keep_states=True)
    kt = k / np.sqrt(D * S)
    ok = True
    for t in range(T):
        ref = np.zeros((D, D))
        for s in range(t + 1):
            w = np.prod(g[s + 1: t + 1])
            ref += w * np.einsum("si,s,sj->ij", kt[s], beta[s], v[s])
        ok &= _close(states[t], ref)
    return ok


def pin_column_separability(og):
    """Columns of the state evolve independently: scanning value column j alone
    (V[:, :, j] and S0[:, j]) gives column j of the full result."""
    rng = np.random.default_rng(16)
    T, S, D = 4, 6, 5
    h = _rand_head(rng, T, S, D)
    S0 = rng.standard_normal((D, D))
    out, st = og.scan_head(**h, S0=S0)
    ok = True
    for j in range(D):
        hj = dict(h)
        hj["v"] = h["v"][:, :, j: j + 1]
        oj, sj = og.scan_head(**hj, S0=S0[:, j: j + 1])
        ok &= _close(oj[:, :, 0], out[:, :, j]) and _close(sj[:, 0], st[:, j])
    return ok


def pin_linearity(og):
    """Outputs and final state are jointly linear in (S0, V) for fixed Q, K, g, beta."""
    rng = np.random.default_rng(17)
    T, S, D = 4, 6, 5
    h = _rand_head(rng, T, S, D)
    v2 = rng.standard_normal(h["v"].shape)
    S0a, S0b = rng.standard_normal((2, D, D))
    a, b = 0.7, -1.3
    oa, sa = og.scan_head(**h, S0=S0a)
    hb = dict(h, v=v2)
    ob, sb = og.scan_head(**hb, S0=S0b)
    hc = dict(h, v=a * h["v"] + b * v2)
    oc, sc = og.scan_head(**hc, S0=a * S0a + b * S0b)
    return _close(oc, a * oa + b * ob) and _close(sc, a * sa + b * sb)


def pin_forms_agree(og):
    """Residual-form scan == brute-force products of the per-frame affine maps
    (A_t, b_t) == Hillis-Steele and Blelloch prefix compositions == a random
    bracketing of the total composition == chunked calls carrying the state."""
    rng = np.random.default_rng(18)
    T, S, D = 7, 5, 4
    h = _rand_head(rng, T, S, D)
    S0 = rng.standard_normal((D, D))
    out, st, states = og.scan_head(**h, S0=S0, keep_states=True)
    maps = [og.transition(h["k"][t], h["v"][t], h["g"][t], h["beta"][t]) for t in range(T)]
    As = [m[0] for m in maps]
    bs = [m[1] for m in maps]
    ok = True
    bf = og.brute_force_states(As, bs, S0)
    for t in range(T):
        ok &= _close(bf[t], states[t])
        ok &= _close(h["q"][t] @ bf[t] / np.sqrt(D), out[t])
    hs = og.states_from_maps(og.scan_hillis_steele(maps), S0)
    ok &= all(_close(hs[t], states[t]) for t in range(T))
    ex = og.scan_blelloch_exclusive(maps, D)
    ok &= _close(og.apply_map(ex[0], S0), S0)
    ok &= all(_close(og.apply_map(ex[t], S0), states[t - 1]) for t in range(1, T))
    for seed in range(3):
        tot = og.fold_random_bracketing(maps, np.random.default_rng(seed))
        ok &= _close(og.apply_map(tot, S0), st)
    # chunked calls: 3 + 1 + 3 frames, state carried
    Sc = S0
    outs = []
    for a, b in ((0, 3), (3, 4), (4, 7)):
        oc, Sc = og.scan_head(**{k: v[a:b] for k, v in h.items()}, S0=Sc)
        outs.append(oc)
    ok &= _close(np.concatenate(outs), out) and _close(Sc, st)
    return ok


def pin_transition_structure(og):
    """A_t is symmetric, g(I - M) with M = K~^T diag(beta) K~ positive semidefinite;
    with the 1/sqrt(D*S) scaling, tr(M) = sum_s beta_s |k_s|^2 / (D*S)."""
    rng = np.random.default_rng(19)
    S, D = 12, 6
    k = rng.standard_normal((S, D))
    v = rng.standard_normal((S, D))
    beta = rng.uniform(0, 1, S)
    g = 0.8
    A, _ = og.transition(k, v, g, beta)
    M = np.eye(D) - A / g
    ok = _close(A, A.T)
    ok &= float(np.min(np.linalg.eigvalsh(M))) >= -1e-12
    ok &= abs(np.trace(M) - np.sum(beta * np.sum(k * k, axis=1)) / (D * S)) < 1e-12
    return ok


PINS = [pin_golden_hand_example, pin_delta_rule_exact_write, pin_beta_zero_pure_decay,
        pin_gate_zero_memoryless, pin_cumulative_linear_attention,
        pin_gated_cumulative_linear_attention, pin_column_separability, pin_linearity,
        pin_forms_agree, pin_transition_structure]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    assert pin(ORACLE)


# ------------------------------------------------- invariants on the workloads' draws

def test_spectral_bound_tiny_workload():
    """The key scaling bounds the transition: ||A_t||_2 <= 1 on every frame of the
    tiny workload (and the norm-growth bound |S_t| <= |S_{t-1}| + |b_t| holds)."""
    wl = synth.WORKLOADS["tiny"]
    for b in range(wl.B):
        for h in range(wl.H):
            x = synth.head(wl, b, h)
            _, _, states = ORACLE.scan_head(x["q"], x["k"], x["v"], x["g"], x["beta"], keep_states=True)
            prev = np.zeros((wl.D, wl.D))
            for t in range(wl.T):
                A, bt = ORACLE.transition(x["k"][t], x["v"][t], x["g"][t], x["beta"][t])
                assert ORACLE.spectral_norm_sym(A) <= 1.0
                assert np.linalg.norm(states[t]) <= np.linalg.norm(prev) + np.linalg.norm(bt) + 1e-12
                prev = states[t]


@pytest.mark.parametrize("name", ["short", "large"])
def test_spectral_bound_sampled_frames(name):
    """||A_t||_2 <= 1 on sampled frames of the 720p-shaped workloads."""
    wl = synth.WORKLOADS[name]
    for (b, h) in synth.head_sample(wl, 2):
        for t in (0, wl.T // 2, wl.T - 1):
            k = synth.frame(wl, "k", b, h, t).astype(np.float64)
            bt = synth.beta(wl, b, h, t).astype(np.float64)
            g = float(synth.gate(wl, b, h, t))
            c = ORACLE.key_scale(wl.D, wl.S)
            M = (k * c).T @ (bt[:, None] * (k * c))
            lam = np.linalg.eigvalsh(M)
            assert lam.min() >= -1e-12 and lam.max() <= 2.0
            assert g * np.max(np.abs(1.0 - lam)) <= 1.0
