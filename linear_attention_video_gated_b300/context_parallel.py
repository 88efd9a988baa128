"""Context-parallel forward over frame ranges: one rank per GPU, each holding a
contiguous range of a sequence's latent frames (the pages' context-parallel
training splits the latent sequence across GPUs and composes the GDN transition
maps by prefix sums, exactly: zhichai.net SANA-WM summary, training pipeline
Stage 3).

Per head, frames [t0, t1) map the state entering them to A S + b (A the product
of the frames' transition matrices, b the state the range reaches from zero).
Rank r of R:

  1. gdn_frame_summary: the (A_r, b_r) of its own frames (2 D^2 float32 per head);
  2. all_gather of the summaries over the process group: the one exchange step;
  3. gdn_summary_apply, folded in rank order: the state entering its range,
     S_r = A_{r-1}( ... (A_0 S_in + b_0) ... ) + b_{r-1};
  4. gdn_frame_fwd_ex on its frames from S_r: its outputs;
  5. the sequence's final state: its own final state with the later ranks' maps
     folded on (every rank returns it; on the last rank it is that rank's scan).

Steps 1, 3 and 4 run in the library's kernels; this module moves arguments and
the exchanged summaries only.  The summaries travel as one [2, B, H, D, D]
float32 tensor per rank, on the device under NCCL and through host memory under
gloo.
"""
from __future__ import annotations

from . import binding


class CudaOps:
    """The library's entry points (the CUDA path): summary, apply, forward."""

    def summary(self, k, v, g, beta, gate_logits):
        return binding.frame_summary(k, v, g, beta, gate_logits=gate_logits)

    def apply(self, A, b, state):
        return binding.summary_apply(A, b, state_in=state)

    def forward(self, q, k, v, g, beta, state_in, gate_logits, mode):
        return binding.frame_fwd(q, k, v, g, beta, state_in=state_in, mode=mode, gate_logits=gate_logits)


def frame_ranges(T: int, world: int) -> list:
    """Contiguous frame ranges [t0, t1) of a T-frame sequence over `world` ranks, in
    rank order, as even as possible (the first T % world ranks take one frame more)."""
    base, extra = divmod(T, world)
    out, t0 = [], 0
    for r in range(world):
        n = base + (1 if r < extra else 0)
        out.append((t0, t0 + n))
        t0 += n
    return out


def _all_gather(packed, group):
    import torch
    import torch.distributed as dist

    world = dist.get_world_size(group)
    backend = dist.get_backend(group)
    dev = packed.device
    send = packed.cpu() if (backend == "gloo" and packed.is_cuda) else packed
    parts = [torch.empty_like(send) for _ in range(world)]
    dist.all_gather(parts, send.contiguous(), group=group)
    return [p.to(dev) for p in parts]


def frame_fwd_cp(q, k, v, g, beta, state_in=None, group=None, gate_logits=False,
                 mode=binding.GDN_MODE_SEQUENTIAL, ops=None):
    """The forward scan of this rank's frames of a sequence split over the ranks of
    `group` (default: the world) in rank order.

    q, k, v: [B,H,T_r,S,D], g: [B,H,T_r], beta: [B,H,T_r,S] -- this rank's frames
    only, laid out as gdn_frame_fwd takes them; state_in: the sequence's initial
    state [B,H,D,D] float32 (None: zeros), the same on every rank.  Every rank
    must call this (the summaries are exchanged collectively).

    Returns (out, state_out): the outputs of this rank's frames, and the state
    after the sequence's last frame.
    """
    import torch
    import torch.distributed as dist

    ops = ops or CudaOps()
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    A, b = ops.summary(k, v, g, beta, gate_logits)
    parts = _all_gather(torch.stack([A, b]), group)
    state = state_in
    for r in range(rank):
        state = ops.apply(parts[r][0], parts[r][1], state)
    out, state_out = ops.forward(q, k, v, g, beta, state, gate_logits, mode)
    for r in range(rank + 1, world):
        state_out = ops.apply(parts[r][0], parts[r][1], state_out)
    return out, state_out
