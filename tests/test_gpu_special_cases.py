"""GPU parity on the method's special cases: inputs for which the update has an
exact, independently known result (zhichai.net SANA-WM summary, section
"四大工程设计" item 1: the decay gate scales the previous state, the delta rule
writes only the beta-weighted residual, keys are scaled by 1/sqrt(D*S)).

Each case runs through the CUDA path (every algorithm form, float32 and bf16
I/O) and is compared element by element with the fp64 oracle on the same
seeded inputs (tolerances in tests/parity.py: 1e-4 max-abs for float32 I/O,
2e-2 x rms beyond the output's own bf16 representation for bf16 I/O), and,
where the special case fixes the
result in closed form, with that closed form too (computed here in float64 from
the inputs, not through the oracle):

  * beta = 0, non-zero S_0: nothing is written, S_t = (prod g) S_0 and
    O_t = Q_t (prod_{s<=t} g_s) S_0 / sqrt(D);
  * g = 0: memoryless, S_t = K~_t^T diag(beta_t) V_t whatever S_0 is, so a call
    from a non-zero S_0 gives the zero-state call's results bit for bit;
  * g = 1, beta = 1, frames on disjoint key coordinates, S_0 = 0: the prediction
    K~_t S_{t-1} vanishes, so the scan is plain cumulative linear attention,
    S_t = sum_{s<=t} K~_s^T V_s;
  * one token per frame with entries +-1 (|k~| = 1), beta = 1, Q = K: the delta
    rule writes exactly, k~^T S_t = v_t, so every output equals V;
  * g ~ U(0.99, 1), beta = 1 over 961 frames of 880 tokens at d112: the largest
    transition norms |A_t| = g |I - M_t| that Gaussian keys give, where the
    single bf16 image of M_t is applied 961 times in a row.
"""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_video_gated_b300 import binding, build_lib, synth
from tests import parity

pytestmark = pytest.mark.gpu

MODES = [0, 1, 2]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_lib.ensure_built()
    binding.lib()


def np_(t):
    return t.float().cpu().numpy()


def base(dt):
    return synth.WORKLOADS["short" if dt == "bf16" else "tiny"]


def initial_states(wl, scale=0.3):
    return np.stack([np.stack([synth.state(wl, b, h, scale) for h in range(wl.H)]) for b in range(wl.B)])


def run(wl, x, S0, mode):
    ins = parity.upload(wl, x)
    si = None if S0 is None else torch.from_numpy(np.ascontiguousarray(S0, np.float32)).cuda()
    out, st = binding.frame_fwd(*ins, state_in=si, mode=mode)
    torch.cuda.synchronize()
    parity.check_status()
    return out, st


def check(wl, x, S0, mode, what, closed=None):
    """GPU vs oracle (and vs the closed form `closed` = (out, state), float64)."""
    out, st = run(wl, x, S0, mode)
    ro, rs = oracle.frame_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], S0)
    eo, es = parity.assert_parity(wl.dtype, np_(out), ro, np_(st), rs, f"{what} mode={mode} vs oracle")
    print(f"{what} mode={mode}: vs oracle out {eo} state {es}")
    if closed is not None:
        co, cs = closed
        eo, es = parity.assert_parity(wl.dtype, np_(out), co, np_(st), cs, f"{what} mode={mode} vs closed form")
        print(f"{what} mode={mode}: vs closed form out {eo} state {es}")
    return out, st


# ------------------------------------------------------------------ beta = 0

BETA0 = [("bf16", 1, 2, 9, 300, 112), ("bf16", 2, 1, 5, 129, 48), ("f32", 1, 2, 6, 33, 64), ("f32", 1, 1, 4, 17, 16)]


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("case", BETA0, ids=lambda c: "-".join(map(str, c)))
def test_beta_zero_only_decays_the_initial_state(case, mode):
    dt, B, H, T, S, D = case
    wl = base(dt).with_(B=B, H=H, T=T, S=S, D=D, beta_dist=("uniform", 0.0, 0.0), seed=8100 + S + D)
    x = synth.full(wl)
    assert not x["beta"].any()
    S0 = initial_states(wl)
    gcum = np.cumprod(x["g"].astype(np.float64), axis=2)  # [B,H,T]
    St = gcum[..., None, None] * S0[:, :, None].astype(np.float64)  # [B,H,T,D,D]
    co = np.einsum("bhtsi,bhtij->bhtsj", x["q"].astype(np.float64), St) / np.sqrt(D)
    check(wl, x, S0, mode, f"beta=0 {case}", closed=(co, St[:, :, -1]))


# ------------------------------------------------------------------ g = 0

G0 = [("bf16", 1, 3, 6, 880, 112), ("bf16", 1, 2, 4, 77, 32), ("f32", 2, 1, 5, 40, 128), ("f32", 1, 2, 3, 16, 16)]


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("case", G0, ids=lambda c: "-".join(map(str, c)))
def test_g_zero_is_memoryless(case, mode):
    dt, B, H, T, S, D = case
    wl = base(dt).with_(B=B, H=H, T=T, S=S, D=D, g_dist=("uniform", 0.0, 0.0), seed=8200 + S + D)
    x = synth.full(wl)
    assert not x["g"].any()
    S0 = initial_states(wl)
    kt = x["k"].astype(np.float64) / np.sqrt(D * S)
    St = np.einsum("bhtsi,bhts,bhtsj->bhtij", kt, x["beta"].astype(np.float64), x["v"].astype(np.float64))
    co = np.einsum("bhtsi,bhtij->bhtsj", x["q"].astype(np.float64), St) / np.sqrt(D)
    # S_0 has no effect: the call from S_0 equals the zero-state call bit for bit
    out_a, st_a = run(wl, x, S0, mode)
    out_b, st_b = check(wl, x, None, mode, f"g=0 {case}", closed=(co, St[:, :, -1]))
    assert torch.equal(out_a, out_b) and torch.equal(st_a, st_b), "the initial state leaked through g = 0"


# ------------------------------------------------------------------ disjoint keys, g = beta = 1

# (dtype, B, H, T, S, D): each frame's keys live on D / T coordinates of their own
DISJOINT = [("f32", 1, 2, 8, 16, 16), ("bf16", 1, 2, 8, 16, 16), ("bf16", 1, 2, 7, 300, 112),
            ("bf16", 2, 1, 4, 129, 128), ("f32", 1, 1, 4, 100, 64)]


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("case", DISJOINT, ids=lambda c: "-".join(map(str, c)))
def test_disjoint_keys_are_cumulative_linear_attention(case, mode):
    dt, B, H, T, S, D = case
    wl = base(dt).with_(B=B, H=H, T=T, S=S, D=D, g_dist=("uniform", 1.0, 1.0), beta_dist=("uniform", 1.0, 1.0),
                        seed=8300 + S + D)
    x = synth.full(wl)
    w = D // T
    for t in range(T):  # keys of frame t only on coordinates [w t, w t + w)
        x["k"][:, :, t, :, :w * t] = 0.0
        x["k"][:, :, t, :, w * (t + 1):] = 0.0
    kt = x["k"].astype(np.float64) / np.sqrt(D * S)
    St = np.cumsum(np.einsum("bhtsi,bhtsj->bhtij", kt, x["v"].astype(np.float64)), axis=2)
    co = np.einsum("bhtsi,bhtij->bhtsj", x["q"].astype(np.float64), St) / np.sqrt(D)
    check(wl, x, None, mode, f"disjoint {case}", closed=(co, St[:, :, -1]))


# ------------------------------------------------------------------ delta rule writes exactly

EXACT = [("bf16", 1, 2, 12, 112), ("bf16", 1, 1, 9, 64), ("f32", 1, 2, 12, 16), ("f32", 2, 1, 7, 128)]


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("case", EXACT, ids=lambda c: "-".join(map(str, c)))
def test_one_token_frames_write_exactly(case, mode):
    """S = 1, keys of +-1 entries (|k|^2 = D, so |k~| = 1, exact in bf16), beta = 1,
    queries equal to the keys: O_t = k S_t / sqrt(D) = k~^T S_t = v_t, from a
    non-zero initial state and whatever the decay."""
    dt, B, H, T, D = case
    wl = base(dt).with_(B=B, H=H, T=T, S=1, D=D, beta_dist=("uniform", 1.0, 1.0), seed=8400 + D)
    x = synth.full(wl)
    x["k"] = np.where(x["k"] >= 0, 1.0, -1.0).astype(np.float32)
    x["q"] = x["k"].copy()
    S0 = initial_states(wl)
    out, st = run(wl, x, S0, mode)
    ro, rs = oracle.frame_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], S0)
    eo, es = parity.assert_parity(wl.dtype, np_(out), ro, np_(st), rs, f"exact write {case} mode={mode}")
    print(f"exact write {case} mode={mode}: vs oracle out {eo} state {es}")
    # the closed form: every output is the frame's value row
    e = parity.errors(np_(out), x["v"])
    bound = parity.F32_MAX_ABS if dt == "f32" else parity.BF16_MAX_ABS_OVER_RMS * e["rms_ref"]
    print(f"exact write {case} mode={mode}: out vs V {e}")
    assert e["max_abs"] <= bound, e


# ------------------------------------------------------------------ largest transition norms, long

@pytest.fixture(scope="module")
def slow_decay():
    """One head of 961 frames x 880 tokens x d112, g ~ U(0.99, 1), beta = 1, in
    both I/O dtypes, with the oracle's result (the same inputs: bf16 values are
    exact in float32)."""
    res = {}
    for dt in ("bf16", "f32"):
        wl = synth.WORKLOADS["minute"].with_(H=1, dtype=dt, g_dist=("uniform", 0.99, 1.0),
                                             beta_dist=("uniform", 1.0, 1.0), seed=8500)
        res[dt] = wl
    x = synth.head(res["bf16"], 0, 0)
    ro, rs = oracle.scan_head(x["q"], x["k"], x["v"], x["g"], x["beta"])
    # |A_t| on a few frames: close to 1 (the longest memory Gaussian keys allow)
    norms = [oracle.spectral_norm_sym(oracle.transition(x["k"][t], x["v"][t], x["g"][t], x["beta"][t])[0])
             for t in (0, 480, 960)]
    print(f"slow decay |A_t|_2 on frames 0, 480, 960: {norms}")
    assert all(0.98 < n <= 1.0 for n in norms)
    return res, x, ro, rs


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_slow_decay_full_strength_writes_over_961_frames(slow_decay, dt, mode):
    res, x, ro, rs = slow_decay
    wl = res[dt]
    xx = {k_: v_[None, None] for k_, v_ in x.items()}
    out, st = run(wl, xx, None, mode)
    eo, es = parity.assert_parity(dt, np_(out[0, 0]), ro, np_(st[0, 0]), rs, f"slow decay {dt} mode={mode}")
    print(f"slow decay {dt} mode={mode}: out {eo} state {es}")
