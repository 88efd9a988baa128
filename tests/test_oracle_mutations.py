"""Plant plausible mistakes in the oracle (on the CPU, by monkeypatching one of its
step functions) and check that at least one pin catches each of them.

This is what shows the pins in ``test_oracle_pins.py`` are strong enough to trust
the oracle: a dropped term, a wrong sign, a wrong scale, a transposed operand or
an off-by-one-frame read-out each fail a pin.
"""
import numpy as np
import pytest

import oracle.gdn_oracle as og
from tests.test_oracle_pins import PINS


def _mut_residual_no_gate(Vt, P, g, beta):
    return beta[:, None] * (Vt - P)


def _mut_residual_sign(Vt, P, g, beta):
    return beta[:, None] * (Vt + g * P)


def _mut_residual_beta_on_target_only(Vt, P, g, beta):
    return beta[:, None] * Vt - g * P


def _mut_write_no_decay(St, Kt, R, g):
    return St + Kt.T @ R


def _mut_write_double_decay(St, Kt, R, g):
    return g * (g * St + Kt.T @ R)


def _mut_predict_transposed_state(Kt, St):
    return Kt @ St.T


def _mut_key_scale_head_dim_only(D, S):
    return 1.0 / np.sqrt(float(D))


def _mut_key_scale_tokens_only(D, S):
    return 1.0 / np.sqrt(float(S))


def _mut_out_scale_missing(D):
    return 1.0


def _mut_frame_step_reads_old_state(St, Qt, Kt_raw, Vt, g, beta, D, S):
    Kt = Kt_raw * og.key_scale(D, S)
    P = og.predict(Kt, St)
    R = og.residual(Vt, P, g, beta)
    return og.write(St, Kt, R, g), og.readout(Qt, St, D)


def _mut_frame_step_unscaled_write_key(St, Qt, Kt_raw, Vt, g, beta, D, S):
    Kt = Kt_raw * og.key_scale(D, S)
    P = og.predict(Kt, St)
    R = og.residual(Vt, P, g, beta)
    St_new = og.write(St, Kt_raw, R, g)
    return St_new, og.readout(Qt, St_new, D)


MUTATIONS = [
    ("residual", _mut_residual_no_gate),
    ("residual", _mut_residual_sign),
    ("residual", _mut_residual_beta_on_target_only),
    ("write", _mut_write_no_decay),
    ("write", _mut_write_double_decay),
    ("predict", _mut_predict_transposed_state),
    ("key_scale", _mut_key_scale_head_dim_only),
    ("key_scale", _mut_key_scale_tokens_only),
    ("out_scale", _mut_out_scale_missing),
    ("frame_step", _mut_frame_step_reads_old_state),
    ("frame_step", _mut_frame_step_unscaled_write_key),
]


@pytest.mark.parametrize("target,fn", MUTATIONS, ids=[m[1].__name__ for m in MUTATIONS])
def test_planted_mistake_is_caught(monkeypatch, target, fn):
    monkeypatch.setattr(og, target, fn)
    failed = []
    for pin in PINS:
        try:
            ok = pin(og)
        except Exception:  # a shape error also counts as caught
            ok = False
        if not ok:
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {fn.__name__}"


def test_unmutated_oracle_passes_all_pins():
    assert all(pin(og) for pin in PINS)
