"""gdn_frame_fwd_noalloc: the entry point for callers that cannot allocate device
memory (for example code running inside another runtime whose allocator owns the
GPU's memory).  It runs the split form (the kernels that use scratch) with its
scratch in one fixed array inside the library, so these tests check that

  * on the GPU, its results equal gdn_frame_fwd_ex's (caller-owned workspace, the
    same split-form kernels, so bit for bit), and both match the oracle within the
    parity tolerances of tests/parity.py, on calls in a row with different shapes
    and data (each later call reuses the array the one before left behind);
  * on the host, a shape whose scratch does not fit in the array is rejected with
    GDN_ERR_WORKSPACE before any CUDA call.

The file name sorts last so that a run stopping at the first failure has already
run every other test."""
import numpy as np
import pytest

from linear_attention_video_gated_b300 import binding, build_lib, synth


def test_oversized_shape_is_rejected_on_the_host():
    build_lib.build()
    cap = binding.gdn_noalloc_scratch_bytes()
    assert cap == 64 << 20
    # 20 heads x 961 frames x 880 tokens x d112 needs ~2.6 GB of scratch.
    need = binding.gdn_workspace_bytes(1, 20, 961, 880, 112, binding.GDN_BF16, binding.GDN_MODE_SPLIT)
    assert need > cap
    fake = 0x10000  # never dereferenced: the call fails before touching CUDA
    rc = binding.gdn_frame_fwd_noalloc(fake, fake, fake, fake, fake, None, fake, None,
                                       1, 20, 961, 880, 112, binding.GDN_BF16, None)
    assert rc == 6  # GDN_ERR_WORKSPACE


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_on_two_calls_in_a_row():
    import torch

    import oracle
    from tests import parity

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_lib.ensure_built()
    stream = torch.cuda.current_stream().cuda_stream
    cases = [
        # (workload, non-zero initial state): 20 heads x 21 frames fills ~57 MB of
        # the 64 MiB array; the second, smaller case then reuses it.
        (synth.WORKLOADS["short"], False),
        (synth.WORKLOADS["short"].with_(H=3, T=9, S=300, seed=4242), True),
        (synth.WORKLOADS["tiny"], True),
    ]
    for wl, nonzero in cases:
        dtype = binding.GDN_BF16 if wl.dtype == "bf16" else binding.GDN_F32
        need = binding.gdn_workspace_bytes(wl.B, wl.H, wl.T, wl.S, wl.D, dtype, binding.GDN_MODE_SPLIT)
        assert 0 < need <= binding.gdn_noalloc_scratch_bytes()
        x = synth.full(wl)
        q, k, v, g, beta = parity.upload(wl, x)
        s0 = None
        if nonzero:
            s0 = torch.from_numpy(np.stack([np.stack([synth.state(wl, b, h) for h in range(wl.H)])
                                            for b in range(wl.B)])).cuda()
        shape_args = (wl.B, wl.H, wl.T, wl.S, wl.D, dtype)

        def ptrs(out, st):
            return (q.data_ptr(), k.data_ptr(), v.data_ptr(), g.data_ptr(), beta.data_ptr(),
                    None if s0 is None else s0.data_ptr(), out.data_ptr(), st.data_ptr())

        out_ref = torch.empty_like(q)
        st_ref = torch.empty((wl.B, wl.H, wl.D, wl.D), dtype=torch.float32, device="cuda")
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        rc = binding.gdn_frame_fwd_ex(*ptrs(out_ref, st_ref), *shape_args, binding.GDN_MODE_SPLIT,
                                      ws.data_ptr(), need, stream)
        assert rc == 0
        out = torch.full_like(q, float("nan"))
        st = torch.full_like(st_ref, float("nan"))
        rc = binding.gdn_frame_fwd_noalloc(*ptrs(out, st), *shape_args, stream)
        assert rc == 0
        torch.cuda.synchronize()
        parity.check_status()
        assert torch.equal(out, out_ref) and torch.equal(st, st_ref), f"noalloc {wl.name} H={wl.H} T={wl.T}"
        S0 = None if s0 is None else s0.cpu().numpy()
        ro, rs = oracle.frame_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], S0)
        parity.assert_parity(wl.dtype, out.float().cpu().numpy(), ro, st.cpu().numpy(), rs,
                             f"noalloc {wl.name} H={wl.H} T={wl.T}")
