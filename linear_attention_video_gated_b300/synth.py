"""Seeded synthetic inputs for the frame-wise Gated DeltaNet forward scan.

This module holds random-number generation and dtype rounding only: none of the
method's arithmetic.  Both the CUDA path (through the binding) and the fp64
oracle read their inputs from here.

Every frame (b, h, t) of every tensor is drawn from its own counter-based
Philox-4x64 stream (numpy's ``Philox`` bit generator, Salmon et al., SC'11),
keyed by ``(seed, tensor id, b, h, t)``.  Any single frame, or any single head,
can therefore be regenerated without drawing the rest of the workload, which is
what lets the oracle check sampled heads of workloads far too large to hold on
the host in fp64.

Values are drawn in float32.  For bf16 workloads each q/k/v value is rounded to
bf16 (round-to-nearest-even) and the oracle receives exactly the rounded value,
upcast, so both sides see identical inputs.  g and beta are float32 on both
sides.

Workload shapes follow the 720p latent geometry of the SANA-WM pages: a
60 s, 16 fps, 720p clip is 961 latent frames; a 2240-wide model with 20 heads
has head dim 112; a frame is a 22 x 40 latent grid, 880 tokens.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

# Tensor ids mixed into the Philox key.
TID = {"q": 1, "k": 2, "v": 3, "g": 4, "beta": 5, "state": 6, "dout": 7, "dstate": 8}


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: shapes, I/O dtype, gate distributions, seed."""

    name: str
    B: int
    H: int
    T: int
    S: int
    D: int
    dtype: str  # "f32" or "bf16": the dtype of q, k, v and out
    g_dist: tuple  # ("uniform", lo, hi) | ("exp_neg_softplus_normal",)
    beta_dist: tuple  # ("uniform", lo, hi) | ("sigmoid_normal",)
    seed: int
    chunks: tuple = field(default=())  # frames per call for chunk-causal rollouts

    @property
    def tokens(self) -> int:
        """Tokens per call: every (b, t, s) position, all H heads processed."""
        return self.B * self.T * self.S

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == "bf16" else 4

    def with_(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


_EXPNS = ("exp_neg_softplus_normal",)
_SIGN = ("sigmoid_normal",)

WORKLOADS = {
    # oracle-sized correctness case, fp32 I/O
    "tiny": Workload("tiny", 1, 2, 8, 16, 16, "f32", ("uniform", 0.9, 1.0), ("uniform", 0.0, 1.0), 1000),
    # 21-frame clip at the 720p latent geometry
    "short": Workload("short", 1, 20, 21, 880, 112, "bf16", _EXPNS, _SIGN, 1001),
    # one minute of 720p video: 961 latent frames, single call
    "minute": Workload("minute", 1, 20, 961, 880, 112, "bf16", _EXPNS, _SIGN, 1002),
    # the same tensors as "minute" (same seed), fed as 96 calls of 10 frames + 1 call of 1 frame
    "chunked": Workload("chunked", 1, 20, 961, 880, 112, "bf16", _EXPNS, _SIGN, 1002,
                        chunks=tuple([10] * 96 + [1])),
    # batched large-frame variant: 45 x 80 latent grid, head dim 128
    "large": Workload("large", 4, 16, 241, 3600, 128, "bf16", ("uniform", 0.8, 0.999), ("uniform", 0.0, 1.0), 1004),
}


def _rng(seed: int, tid: int, b: int, h: int, t: int) -> np.random.Generator:
    if not (0 <= b < (1 << 16) and 0 <= h < (1 << 16) and 0 <= t < (1 << 24)):
        raise ValueError("frame index out of key range")
    key = np.array([seed & ((1 << 64) - 1), (tid << 56) | (b << 40) | (h << 24) | t], dtype=np.uint64)
    return np.random.Generator(np.random.Philox(key=key))


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest, ties to even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> the exactly equal float32 values."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def round_to_dtype(x: np.ndarray, dtype: str) -> np.ndarray:
    """float32 values as the I/O dtype represents them (returned as float32)."""
    if dtype == "bf16":
        return bf16_to_f32(bf16_bits(x))
    return np.asarray(x, dtype=np.float32)


def frame_raw(wl: Workload, name: str, b: int, h: int, t: int) -> np.ndarray:
    """q/k/v (or dout, the gradient a loss sends back into the output) frame
    (b,h,t): [S, D] float32 N(0,1) draws, before dtype rounding."""
    rng = _rng(wl.seed, TID[name], b, h, t)
    return rng.standard_normal((wl.S, wl.D), dtype=np.float32)


def frame(wl: Workload, name: str, b: int, h: int, t: int) -> np.ndarray:
    """q/k/v frame (b,h,t) as float32 holding exactly the I/O-dtype values."""
    return round_to_dtype(frame_raw(wl, name, b, h, t), wl.dtype)


def _draw(rng: np.random.Generator, dist: tuple, n: int) -> np.ndarray:
    kind = dist[0]
    if kind == "uniform":
        return rng.uniform(dist[1], dist[2], size=n).astype(np.float32)
    x = rng.standard_normal(n)  # float64 draw, mapped in float64, stored float32
    if kind == "exp_neg_softplus_normal":
        # exp(-softplus(x)) = 1 / (1 + e^x), in (0, 1)
        return (1.0 / (1.0 + np.exp(x))).astype(np.float32)
    if kind == "sigmoid_normal":
        return (1.0 / (1.0 + np.exp(-x))).astype(np.float32)
    raise ValueError(f"unknown distribution {dist}")


def _logits(rng: np.random.Generator, dist: tuple, n: int) -> np.ndarray:
    """The N(0,1) draws the gate distributions map through, as float32 logits."""
    if dist[0] not in ("exp_neg_softplus_normal", "sigmoid_normal"):
        raise ValueError(f"{dist} is not drawn through a logit")
    return rng.standard_normal(n).astype(np.float32)


def gate_logit(wl: Workload, b: int, h: int, t: int) -> np.float32:
    """Per-frame decay logit for (b,h,t): the same draw gate() maps, float32."""
    return _logits(_rng(wl.seed, TID["g"], b, h, t), wl.g_dist, 1)[0]


def beta_logit(wl: Workload, b: int, h: int, t: int) -> np.ndarray:
    """Per-token beta logits for frame (b,h,t): the same draws beta() maps, float32."""
    return _logits(_rng(wl.seed, TID["beta"], b, h, t), wl.beta_dist, wl.S)


def logits_full(wl: Workload) -> dict:
    """g and beta logits of every frame: {"g_logit": [B,H,T], "beta_logit": [B,H,T,S]}."""
    gl = np.array([[[gate_logit(wl, b, h, t) for t in range(wl.T)] for h in range(wl.H)] for b in range(wl.B)],
                  dtype=np.float32).reshape(wl.B, wl.H, wl.T)
    bl = np.array([[[beta_logit(wl, b, h, t) for t in range(wl.T)] for h in range(wl.H)] for b in range(wl.B)],
                  dtype=np.float32).reshape(wl.B, wl.H, wl.T, wl.S)
    return {"g_logit": gl, "beta_logit": bl}


def gate(wl: Workload, b: int, h: int, t: int) -> np.float32:
    """Per-frame decay g for (b,h,t): one draw, float32."""
    return _draw(_rng(wl.seed, TID["g"], b, h, t), wl.g_dist, 1)[0]


def beta(wl: Workload, b: int, h: int, t: int) -> np.ndarray:
    """Per-token beta for frame (b,h,t): [S] float32."""
    return _draw(_rng(wl.seed, TID["beta"], b, h, t), wl.beta_dist, wl.S)


def state(wl: Workload, b: int, h: int, scale: float = 0.1) -> np.ndarray:
    """A non-zero initial state for (b,h): [D, D] float32, N(0, scale^2)."""
    rng = _rng(wl.seed, TID["state"], b, h, 0)
    return (scale * rng.standard_normal((wl.D, wl.D))).astype(np.float32)


def dstate(wl: Workload, b: int, h: int, scale: float = 0.1) -> np.ndarray:
    """A gradient for the final state of (b,h): [D, D] float32, N(0, scale^2)."""
    rng = _rng(wl.seed, TID["dstate"], b, h, 0)
    return (scale * rng.standard_normal((wl.D, wl.D))).astype(np.float32)


def head_dout(wl: Workload, b: int, h: int, t0: int = 0, t1: int | None = None) -> np.ndarray:
    """Output gradients of one head for frames [t0, t1): [T', S, D] float32 (dtype-rounded)."""
    t1 = wl.T if t1 is None else t1
    if t1 <= t0:
        return np.zeros((0, wl.S, wl.D), np.float32)
    return np.stack([frame(wl, "dout", b, h, t) for t in range(t0, t1)])


def head(wl: Workload, b: int, h: int, t0: int = 0, t1: int | None = None) -> dict:
    """All inputs of one head for frames [t0, t1), float32 arrays (dtype-rounded).

    Returns q, k, v: [T', S, D]; g: [T']; beta: [T', S].
    """
    t1 = wl.T if t1 is None else t1
    ts = range(t0, t1)
    return {
        "q": np.stack([frame(wl, "q", b, h, t) for t in ts]) if t1 > t0 else np.zeros((0, wl.S, wl.D), np.float32),
        "k": np.stack([frame(wl, "k", b, h, t) for t in ts]) if t1 > t0 else np.zeros((0, wl.S, wl.D), np.float32),
        "v": np.stack([frame(wl, "v", b, h, t) for t in ts]) if t1 > t0 else np.zeros((0, wl.S, wl.D), np.float32),
        "g": np.array([gate(wl, b, h, t) for t in ts], dtype=np.float32),
        "beta": np.stack([beta(wl, b, h, t) for t in ts]) if t1 > t0 else np.zeros((0, wl.S), np.float32),
    }


def full(wl: Workload) -> dict:
    """All inputs as float32 arrays [B,H,T,S,D] etc. (small workloads only)."""
    hs = [[head(wl, b, h) for h in range(wl.H)] for b in range(wl.B)]
    return {key: np.stack([np.stack([hs[b][h][key] for h in range(wl.H)]) for b in range(wl.B)])
            for key in ("q", "k", "v", "g", "beta")}


def full_grads(wl: Workload) -> dict:
    """dout [B,H,T,S,D] and dstate [B,H,D,D] float32 arrays (small workloads only)."""
    return {"dout": np.stack([np.stack([head_dout(wl, b, h) for h in range(wl.H)]) for b in range(wl.B)]),
            "dstate": np.stack([np.stack([dstate(wl, b, h) for h in range(wl.H)]) for b in range(wl.B)])}


def _threads() -> int:
    return max(1, len(os.sched_getaffinity(0)))


def fill_io(wl: Workload, q: np.ndarray, k: np.ndarray, v: np.ndarray,
            g: np.ndarray, bt: np.ndarray, t0: int = 0, b0: int = 0, threads: int | None = None,
            logits: bool = False) -> None:
    """Fill caller-owned host arrays with frames [t0, t0 + q.shape[2]) of batch
    indices [b0, b0 + q.shape[0]), every head.

    q, k, v: [B', H, T', S, D] uint16 (bf16 bits) for bf16 workloads or float32 for
    f32; g: [B', H, T'] float32; bt: [B', H, T', S] float32.  The arrays may be numpy
    views of pinned torch tensors.  Generation runs on a thread pool (numpy
    releases the GIL while drawing).
    """
    Bn, Hn, Tn = q.shape[0], q.shape[1], q.shape[2]
    jobs = [(bb, h, tt) for bb in range(Bn) for h in range(Hn) for tt in range(Tn)]
    nthreads = threads or _threads()

    def one(job):
        bb, h, tt = job
        b, t = b0 + bb, t0 + tt
        for name, dst in (("q", q), ("k", k), ("v", v)):
            x = frame_raw(wl, name, b, h, t)
            dst[bb, h, tt] = bf16_bits(x) if wl.dtype == "bf16" else x
        g[bb, h, tt] = gate_logit(wl, b, h, t) if logits else gate(wl, b, h, t)
        bt[bb, h, tt] = beta_logit(wl, b, h, t) if logits else beta(wl, b, h, t)

    with ThreadPoolExecutor(nthreads) as ex:
        for _ in ex.map(one, jobs, chunksize=max(1, len(jobs) // (16 * nthreads))):
            pass


def fill_dout(wl: Workload, dst: np.ndarray, t0: int = 0, b0: int = 0, threads: int | None = None) -> None:
    """Fill a caller-owned host array [B', H, T', S, D] (uint16 bf16 bits or float32)
    with the output gradients of frames [t0, t0 + T') of batch indices [b0, b0 + B')."""
    Bn, Hn, Tn = dst.shape[0], dst.shape[1], dst.shape[2]
    jobs = [(bb, h, tt) for bb in range(Bn) for h in range(Hn) for tt in range(Tn)]
    nthreads = threads or _threads()

    def one(job):
        bb, h, tt = job
        x = frame_raw(wl, "dout", b0 + bb, h, t0 + tt)
        dst[bb, h, tt] = bf16_bits(x) if wl.dtype == "bf16" else x

    with ThreadPoolExecutor(nthreads) as ex:
        for _ in ex.map(one, jobs, chunksize=max(1, len(jobs) // (16 * nthreads))):
            pass


def head_sample(wl: Workload, n: int) -> list:
    """n (b, h) heads spread over the workload (first and last always included)."""
    heads = [(b, h) for b in range(wl.B) for h in range(wl.H)]
    if n >= len(heads):
        return heads
    if n == 1:
        return [heads[0]]
    idx = sorted({round(i * (len(heads) - 1) / (n - 1)) for i in range(n)})
    return [heads[i] for i in idx]
