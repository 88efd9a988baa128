"""Frame-wise Gated DeltaNet (GDN) forward scan: a plain, slow, fp64 oracle.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Plain numpy in float64;
the only library primitive used as a step is the matrix product.  No blocking,
no fusion, no reordering beyond what the update states.

What it computes, and where each piece is stated:

* Each recurrent step consumes one whole latent frame of S tokens
  (bilibili article on SANA-WM, the paragraph on the fourth key point:
  frame-wise rather than token-wise GDN).
* The state has constant size D x D however many frames there are
  (zhichai.net SANA-WM summary, "四大工程设计" section 1, Hybrid Linear
  Attention -- Gated DeltaNet + Softmax).
* Decay gate g: each step multiplies the previous state by a learned scalar
  (same section, the gamma decay-gate bullet; bilibili article, decay g).
* Delta-rule correction beta: the write corrects only the residual between
  the target value and the value the state predicts (same section, the beta
  bullet).
* Keys are scaled by 1/sqrt(D*S), D the head dim and S the spatial tokens per
  frame (same section, the paragraph on training stability / algebraic key
  scaling).

The pages state these in words and print no equation.  The update written out
below is the one reading that satisfies all of them at once, with the key
scale applied to K wherever K appears (prediction and write), per-token beta
weighting the residual rows, and the read-out using the post-update state:

    K~_t = K_t / sqrt(D*S)
    P    = K~_t S_{t-1}                     (prediction of the frame's values)
    R    = diag(beta_t) (V_t - g_t P)       (beta-weighted residual)
    S_t  = g_t S_{t-1} + K~_t^T R           (gated delta-rule write)
    O_t  = Q_t S_t / sqrt(D)                (read-out)

State orientation: S[i, j], i = key dim, j = value dim, row-major [D_k][D_v].

The affine form of one step, S_t = A_t S_{t-1} + b_t with
A_t = g_t (I - K~^T diag(beta) K~) and b_t = K~^T diag(beta) V_t, is built only by
``transition`` for the independent cross-checks (brute-force products and the
prefix-composition forms: the pages' context-parallel training composes GDN
transition matrices by prefix sums, exactly -- zhichai.net summary, training
pipeline, Stage 3).  The scan itself (``scan_head``) never forms A_t.
"""
from __future__ import annotations

import numpy as np

F64 = np.float64


def key_scale(D: int, S: int) -> float:
    """1/sqrt(D*S): the algebraic key scaling (zhichai.net summary, section 1)."""
    return 1.0 / np.sqrt(float(D) * float(S))


def out_scale(D: int) -> float:
    """1/sqrt(D): read-out scale (not on the pages; the plain attention read-out scale)."""
    return 1.0 / np.sqrt(float(D))


def predict(Kt: np.ndarray, St: np.ndarray) -> np.ndarray:
    """Values the previous state predicts for the frame's (scaled) keys: K~ S_{t-1}."""
    return Kt @ St


def residual(Vt: np.ndarray, P: np.ndarray, g: float, beta: np.ndarray) -> np.ndarray:
    """beta-weighted residual between the target values and the decayed prediction."""
    return beta[:, None] * (Vt - g * P)


def write(St: np.ndarray, Kt: np.ndarray, R: np.ndarray, g: float) -> np.ndarray:
    """Gated delta-rule write: decay the old state, add K~^T R."""
    return g * St + Kt.T @ R


def readout(Qt: np.ndarray, St: np.ndarray, D: int) -> np.ndarray:
    """Frame output from the post-update state."""
    return (Qt @ St) * out_scale(D)


def frame_step(St, Qt, Kt_raw, Vt, g, beta, D, S):
    """One frame of the scan.  Returns (S_t, O_t).  All float64."""
    Kt = Kt_raw * key_scale(D, S)
    P = predict(Kt, St)
    R = residual(Vt, P, g, beta)
    St_new = write(St, Kt, R, g)
    return St_new, readout(Qt, St_new, D)


def scan_head(q, k, v, g, beta, S0=None, keep_states: bool = False):
    """The frame scan of one (b, h) head.

    q, k: [T, S, D]; v: [T, S, Dv]; g: [T]; beta: [T, S]; S0: [D, Dv] or None
    (zeros).  D is the head (key) dim; Dv defaults to D but may be any width,
    which the column-separability check uses.  Returns (out [T, S, Dv], S_T [D, Dv])
    and, with keep_states, the list of S_t.
    """
    q = np.asarray(q, F64)
    k = np.asarray(k, F64)
    v = np.asarray(v, F64)
    g = np.asarray(g, F64)
    beta = np.asarray(beta, F64)
    T, S, D = k.shape
    Dv = v.shape[2]
    St = np.zeros((D, Dv), F64) if S0 is None else np.array(S0, F64)
    out = np.zeros((T, S, Dv), F64)
    states = []
    for t in range(T):
        St, out[t] = frame_step(St, q[t], k[t], v[t], g[t], beta[t], D, S)
        if keep_states:
            states.append(St.copy())
    if keep_states:
        return out, St, states
    return out, St


def frame_fwd(q, k, v, g, beta, state_in=None):
    """Whole-tensor forward: q, k, v [B,H,T,S,D]; g [B,H,T]; beta [B,H,T,S];
    state_in [B,H,D,D] or None.  Returns (out [B,H,T,S,D], state_out [B,H,D,D]), fp64."""
    B, H, T, S, D = np.shape(k)
    out = np.zeros((B, H, T, S, D), F64)
    st = np.zeros((B, H, D, D), F64)
    for b in range(B):
        for h in range(H):
            S0 = None if state_in is None else state_in[b, h]
            out[b, h], st[b, h] = scan_head(q[b, h], k[b, h], v[b, h], g[b, h], beta[b, h], S0)
    return out, st


# ----------------------------------------------------------------------------
# Gate prologue: raw logits -> decay g and delta-rule weight beta.
#
# The pages fuse unnamed "gate ops" with the GDN scan (zhichai.net summary, the
# paragraph after training Stage 4) without stating their form.  The library's
# logit entry point takes the plainest parameterisation that keeps each gate in
# (0, 1) and matches how the workloads draw them: g = exp(-softplus(x)) for the
# decay (a positive forgetting rate), beta = sigmoid(x) for the write strength.
# ----------------------------------------------------------------------------

def softplus(x):
    """log(1 + e^x), written so that neither branch overflows."""
    x = np.asarray(x, F64)
    return np.maximum(x, 0.0) + np.log1p(np.exp(-np.abs(x)))


def decay_from_logit(x):
    """g = exp(-softplus(x)), in (0, 1)."""
    return np.exp(-softplus(x))


def beta_from_logit(x):
    """beta = sigmoid(x) = 1 / (1 + e^-x), in (0, 1); e^-x computed where it cannot overflow."""
    x = np.asarray(x, F64)
    e = np.exp(-np.abs(x))
    return np.where(x >= 0, 1.0 / (1.0 + e), e / (1.0 + e))


def frame_fwd_from_logits(q, k, v, g_logit, beta_logit, state_in=None):
    """The forward scan with its gates given as logits: the gate prologue, then frame_fwd."""
    return frame_fwd(q, k, v, decay_from_logit(g_logit), beta_from_logit(beta_logit), state_in)


# ----------------------------------------------------------------------------
# Baseline: SANA-Video's cumulative ReLU-based linear attention.
#
# The pages contrast GDN with the linear attention of its predecessor, which
# applies a ReLU feature map and keeps a recurrent state that only accumulates,
# with no decay and no delta-rule correction (zhichai.net summary, section 1, the paragraph on
# SANA-Video; bilibili article, third key point).  They give no formula; the
# plainest reading with the GDN scan's own scalings (so the two differ only in
# the decay, the delta rule and the feature map) is
#     S_t = S_{t-1} + relu(K_t)^T V_t / sqrt(D*S),   O_t = relu(Q_t) S_t / sqrt(D),
# with no normaliser (none is mentioned).
# ----------------------------------------------------------------------------

def relu(x):
    return np.maximum(np.asarray(x, F64), 0.0)


def relu_linear_head(q, k, v, S0=None):
    """The cumulative ReLU linear attention of one head: q, k, v [T, S, D]; S0 [D, D] or None."""
    q, k, v = (np.asarray(a, F64) for a in (q, k, v))
    T, S, D = k.shape
    St = np.zeros((D, D), F64) if S0 is None else np.array(S0, F64)
    out = np.zeros((T, S, D), F64)
    for t in range(T):
        St = St + (relu(k[t]) * key_scale(D, S)).T @ v[t]
        out[t] = (relu(q[t]) @ St) * out_scale(D)
    return out, St


def relu_linear_fwd(q, k, v, state_in=None):
    """Whole-tensor form of relu_linear_head: [B,H,T,S,D] inputs, (out, state_out)."""
    B, H, T, S, D = np.shape(k)
    out = np.zeros((B, H, T, S, D), F64)
    st = np.zeros((B, H, D, D), F64)
    for b in range(B):
        for h in range(H):
            S0 = None if state_in is None else state_in[b, h]
            out[b, h], st[b, h] = relu_linear_head(q[b, h], k[b, h], v[b, h], S0)
    return out, st


# ----------------------------------------------------------------------------
# Affine-map forms, used only to cross-check the scan.
# ----------------------------------------------------------------------------

def transition(Kt_raw, Vt, g, beta):
    """Explicit affine map of one frame: (A_t, b_t) with S_t = A_t S_{t-1} + b_t.

    A_t = g (I - K~^T diag(beta) K~),  b_t = K~^T diag(beta) V_t.
    Formed entry by entry from its definition as a sum over the frame's tokens
    (a plain loop over tokens of rank-one terms), deliberately not via the
    matrix-product route the scan uses.
    """
    Kt_raw = np.asarray(Kt_raw, F64)
    Vt = np.asarray(Vt, F64)
    beta = np.asarray(beta, F64)
    S, D = Kt_raw.shape
    c = key_scale(D, S)
    M = np.zeros((D, D), F64)
    b = np.zeros((D, D), F64)
    for s in range(S):
        ks = Kt_raw[s] * c
        M += beta[s] * np.outer(ks, ks)
        b += beta[s] * np.outer(ks, Vt[s])
    A = float(g) * (np.eye(D) - M)
    return A, b


def compose(later, earlier):
    """(A2, b2) o (A1, b1): apply the earlier map first.  = (A2 A1, A2 b1 + b2)."""
    A2, b2 = later
    A1, b1 = earlier
    return A2 @ A1, A2 @ b1 + b2


def apply_map(m, S):
    A, b = m
    return A @ S + b


def brute_force_states(As, bs, S0):
    """S_t for every t by explicit products: S_t = (prod_{r<=t} A_r) S0 + sum_{s<=t} (prod_{s<r<=t} A_r) b_s.

    Every product is formed from scratch (no reuse across t): O(T^2) matrix
    products, for tiny inputs only.
    """
    T = len(As)
    D = S0.shape[0]
    out = []
    for t in range(T):
        P = np.eye(D)
        for r in range(t + 1):
            P = As[r] @ P
        St = P @ S0
        for s in range(t + 1):
            Q = np.eye(D)
            for r in range(s + 1, t + 1):
                Q = As[r] @ Q
            St = St + Q @ bs[s]
        out.append(St)
    return out


def states_from_maps(prefix_maps, S0):
    """Apply inclusive prefix maps (frame 0..t composed) to S0."""
    return [apply_map(m, S0) for m in prefix_maps]


def scan_hillis_steele(maps):
    """Inclusive prefix composition, Hillis-Steele: log2(T) rounds of doubling."""
    cur = list(maps)
    n = len(cur)
    d = 1
    while d < n:
        nxt = list(cur)
        for i in range(d, n):
            nxt[i] = compose(cur[i], cur[i - d])
        cur = nxt
        d *= 2
    return cur


def scan_blelloch_exclusive(maps, D):
    """Exclusive prefix composition, Blelloch up-sweep / down-sweep (length padded
    to a power of two with identity maps).  Element t is frames 0..t-1 composed."""
    ident = (np.eye(D), np.zeros((D, D)))
    n = 1
    while n < len(maps):
        n *= 2
    a = list(maps) + [ident] * (n - len(maps))
    d = 1
    while d < n:  # up-sweep: a[i] accumulates its left sibling subtree
        for i in range(2 * d - 1, n, 2 * d):
            a[i] = compose(a[i], a[i - d])
        d *= 2
    a[n - 1] = ident
    d = n // 2
    while d >= 1:  # down-sweep
        for i in range(2 * d - 1, n, 2 * d):
            left = a[i - d]
            a[i - d] = a[i]
            a[i] = compose(left, a[i])
        d //= 2
    return a[: len(maps)]


def fold_random_bracketing(maps, rng):
    """Total composition of all maps under a random binary bracketing."""
    items = list(maps)
    while len(items) > 1:
        i = int(rng.integers(0, len(items) - 1))
        items[i: i + 2] = [compose(items[i + 1], items[i])]
    return items[0]


def spectral_norm_sym(A):
    """||A||_2 of a symmetric matrix: the largest |eigenvalue| (eigvalsh)."""
    return float(np.max(np.abs(np.linalg.eigvalsh(A))))
