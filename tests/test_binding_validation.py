"""The Python binding rejects malformed tensors on the host, before any CUDA call
(runs without a GPU): CPU tensors where device tensors are expected, mismatched
shapes or dtypes, non-contiguous views, a state-reuse backward without a workspace."""
import pytest
import torch

from linear_attention_video_gated_b300 import binding

B, H, T, S, D = 1, 2, 3, 17, 32


def _inputs(dtype=torch.bfloat16):
    q, k, v = (torch.zeros(B, H, T, S, D, dtype=dtype) for _ in range(3))
    g = torch.full((B, H, T), 0.5)
    beta = torch.full((B, H, T, S), 0.5)
    return q, k, v, g, beta


def test_forward_rejects_host_tensors():
    with pytest.raises(ValueError):
        binding.frame_fwd(*_inputs())


def test_backward_rejects_host_tensors():
    q, k, v, g, beta = _inputs()
    with pytest.raises(ValueError):
        binding.frame_bwd(q, k, v, g, beta, torch.zeros_like(q))


def test_backward_rejects_a_mismatched_output_gradient():
    q, k, v, g, beta = _inputs()
    with pytest.raises(ValueError):
        binding.frame_bwd(q, k, v, g, beta, torch.zeros(B, H, T, S + 1, D, dtype=q.dtype))


def test_forward_rejects_mixed_dtypes_and_views():
    q, k, v, g, beta = _inputs()
    with pytest.raises(ValueError):
        binding.frame_fwd(q, k.float(), v, g, beta)
    with pytest.raises(ValueError):
        binding.frame_fwd(q, k.transpose(3, 4), v, g, beta)


def test_host_entry_rejects_device_style_misuse():
    q, k, v, g, beta = _inputs()
    with pytest.raises(ValueError):
        binding.frame_fwd_host(q, k.transpose(3, 4), v, g, beta)


def test_state_reuse_needs_the_workspace():
    q, k, v, g, beta = _inputs()
    with pytest.raises(ValueError, match="workspace"):
        binding.frame_bwd(q, k, v, g, beta, torch.zeros_like(q), states_in_workspace=True)
