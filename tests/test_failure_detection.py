"""Failure detection, tested without a GPU fault: a bounded device-side wait that
runs out reports GDN_ERR_TIMEOUT through gdn_last_error and leaves the context
usable.  The wait is on a barrier nothing arrives on, with a 20 ms limit."""
import time

import numpy as np
import pytest

import oracle
from linear_attention_video_gated_b300 import binding, build_lib, synth


def test_selftest_rejects_bad_limits_on_the_host():
    build_lib.build()
    assert binding.gdn_selftest_wait_timeout(0, None) == 1
    assert binding.gdn_selftest_wait_timeout(10000001, None) == 1


@pytest.mark.gpu
def test_bounded_wait_reports_timeout_and_context_stays_usable():
    import torch

    from tests import parity

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_lib.ensure_built()
    stream = torch.cuda.current_stream().cuda_stream
    assert binding.gdn_last_error(stream) == 0
    t0 = time.perf_counter()
    assert binding.gdn_selftest_wait_timeout(20000, stream) == 0
    assert binding.gdn_last_error(stream) == 5  # GDN_ERR_TIMEOUT, after the wait gave up
    assert time.perf_counter() - t0 >= 0.02
    assert binding.gdn_last_error(stream) == 0  # reported once, then cleared
    # the context is still usable: a forward call after it matches the oracle
    wl = synth.WORKLOADS["short"].with_(H=2, T=3, S=100, D=32)
    x = synth.full(wl)
    out, st = binding.frame_fwd(*parity.upload(wl, x))
    torch.cuda.synchronize()
    parity.check_status()
    ro, rs = oracle.frame_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"])
    parity.assert_parity("bf16", out.float().cpu().numpy(), ro, st.cpu().numpy(), rs, "after timeout")
