"""fp64 CPU oracle for the frame-wise Gated DeltaNet scan (forward and backward).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may import or run it.  It shares no code with the CUDA path.
"""
from .gdn_oracle import (  # noqa: F401
    key_scale, out_scale, predict, residual, write, readout, frame_step,
    scan_head, frame_fwd, transition, compose, apply_map, brute_force_states,
    scan_hillis_steele, scan_blelloch_exclusive, fold_random_bracketing,
    spectral_norm_sym, states_from_maps,
    softplus, decay_from_logit, beta_from_logit, frame_fwd_from_logits,
    relu, relu_linear_head, relu_linear_fwd,
)
from .gdn_oracle_bwd import (  # noqa: F401
    backward_head, frame_bwd, gate_logit_adjoint, frame_bwd_from_logits,
)
