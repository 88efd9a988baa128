"""Shared helpers for the GPU parity tests: device upload of seeded inputs and the
tolerance checks.

Tolerances (written here, used by every parity test):
  * float32 I/O: max |gpu - oracle| <= 1e-4, for out and for the final state.
  * bf16 outputs: the error beyond the output type's own representation,
    max(|gpu - oracle| - 0.5 ulp_bf16(oracle)) <= 2e-2 x rms(oracle), per tensor.
    No bf16 output can be closer to the exact value than half an ulp, so the part
    of the error within half an ulp is the output type's, not the kernel's; where
    the largest outputs are many times the rms that part alone exceeds
    2e-2 x rms: on the one-minute workload, head (0, 6) has outputs of 8-16 x rms,
    the correctly rounded exact result itself misses the plain max-abs form, and
    the kernels' outputs there were 0.0225 x rms from the oracle of which
    6.4e-5 x rms lay beyond half an ulp.
  * bf16 outputs, also: rms(gpu - oracle) / rms(oracle) <= 5e-3.  Derivation: RNE
    rounding of the outputs gives ~1.6e-3 (uniform error of up to 2^-9 relative,
    averaged over the significand range); the kernels' bf16 hi+lo operand splits
    add < 1e-4; single-bf16 operands where a split is needed would add ~1e-3 on
    top and still pass, a wrong or dropped term would not.
  * The final state (float32) of a bf16 call: max |gpu - oracle| <= 2e-2 x rms and
    the plain form (no representation allowance).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from linear_attention_video_gated_b300 import binding, synth

F32_MAX_ABS = 1e-4
BF16_MAX_ABS_OVER_RMS = 2e-2
BF16_RMS_ERR_OVER_RMS = 5e-3


def torch_dtype(wl):
    return torch.bfloat16 if wl.dtype == "bf16" else torch.float32


def upload(wl, x, dev="cuda"):
    """float32 numpy inputs (already dtype-rounded) -> CUDA tensors."""
    tdt = torch_dtype(wl)
    q, k, v = (torch.from_numpy(np.ascontiguousarray(x[n])).to(dev).to(tdt).contiguous() for n in ("q", "k", "v"))
    g = torch.from_numpy(np.ascontiguousarray(x["g"], dtype=np.float32)).to(dev)
    beta = torch.from_numpy(np.ascontiguousarray(x["beta"], dtype=np.float32)).to(dev)
    return q, k, v, g, beta


def device_inputs(wl, dev="cuda", t0=0, t1=None):
    """Generates frames [t0, t1) of every head straight into CUDA tensors, one
    batch index at a time to bound host memory."""
    t1 = wl.T if t1 is None else t1
    Tn = t1 - t0
    tdt = torch_dtype(wl)
    shape = (wl.B, wl.H, Tn, wl.S, wl.D)
    q = torch.empty(shape, dtype=tdt, device=dev)
    k = torch.empty_like(q)
    v = torch.empty_like(q)
    g = torch.empty((wl.B, wl.H, Tn), dtype=torch.float32, device=dev)
    beta = torch.empty((wl.B, wl.H, Tn, wl.S), dtype=torch.float32, device=dev)
    hdt = np.uint16 if wl.dtype == "bf16" else np.float32
    for b in range(wl.B):
        hq = np.empty((1, wl.H, Tn, wl.S, wl.D), hdt)
        hk = np.empty_like(hq)
        hv = np.empty_like(hq)
        hg = np.empty((1, wl.H, Tn), np.float32)
        hb = np.empty((1, wl.H, Tn, wl.S), np.float32)
        synth.fill_io(wl, hq, hk, hv, hg, hb, t0=t0, b0=b)
        for dst, src in ((q, hq), (k, hk), (v, hv)):
            t = torch.from_numpy(src)
            if wl.dtype == "bf16":
                t = t.view(torch.bfloat16)
            dst[b:b + 1].copy_(t)
        g[b:b + 1].copy_(torch.from_numpy(hg))
        beta[b:b + 1].copy_(torch.from_numpy(hb))
    return q, k, v, g, beta


def device_dout(wl, dev="cuda"):
    """The output gradients of every frame, generated straight into a CUDA tensor
    one batch index at a time."""
    tdt = torch_dtype(wl)
    out = torch.empty((wl.B, wl.H, wl.T, wl.S, wl.D), dtype=tdt, device=dev)
    hdt = np.uint16 if wl.dtype == "bf16" else np.float32
    for b in range(wl.B):
        h = np.empty((1, wl.H, wl.T, wl.S, wl.D), hdt)
        synth.fill_dout(wl, h, b0=b)
        t = torch.from_numpy(h)
        out[b:b + 1].copy_(t.view(torch.bfloat16) if wl.dtype == "bf16" else t)
    return out


GRAD_KEYS = ("dq", "dk", "dv", "dg", "dbeta", "dstate_in")
F32_GRAD_MAX_ABS_OVER_RMS = 1e-4


def assert_grad_parity(wl_dtype, gpu, ref, what=""):
    """Backward-pass bound, per gradient tensor.

    float32 I/O (CUDA-core float32 arithmetic from exact inputs): every gradient
    within 1e-4 x rms(oracle) -- sums of up to ~1e5 products, typical relative
    error ~sqrt(n) x 2^-24 ~ 2e-5.
    bf16 I/O (tensor cores): dq, dk, dv are bf16 outputs and take the forward's
    bf16 bound for outputs with the half-ulp allowance.  dg, dbeta and dstate_in
    are float32 outputs, but computed through bf16 operands (the M_t image, R and
    dP rounded to bf16, the states and U split hi + lo): like the forward's final
    state they take max |err| <= 2e-2 x rms and rms(err) <= 5e-3 x rms."""
    res = {}
    for key in GRAD_KEYS:
        if key not in gpu or gpu[key] is None:
            continue
        e = errors(gpu[key], ref[key])
        res[key] = e
        assert e["finite"], f"{what} {key}: non-finite values"
        if e["rms_ref"] == 0:
            assert e["max_abs"] == 0.0, f"{what} {key}: {e}"
            continue
        if wl_dtype == "f32":
            assert e["max_abs_over_rms"] <= F32_GRAD_MAX_ABS_OVER_RMS, f"{what} {key}: {e}"
            continue
        key_max = "max_beyond_half_ulp_over_rms" if key in ("dq", "dk", "dv") else "max_abs_over_rms"
        assert e[key_max] <= BF16_MAX_ABS_OVER_RMS, f"{what} {key}: {e}"
        assert e["rms_err_over_rms"] <= BF16_RMS_ERR_OVER_RMS, f"{what} {key}: {e}"
    return res


def oracle_head(wl, b, h, S0=None):
    x = synth.head(wl, b, h)
    return oracle.scan_head(x["q"], x["k"], x["v"], x["g"], x["beta"], S0)


def half_ulp_bf16(x):
    """Half the bf16 spacing at |x| (bf16 has 8 significand bits)."""
    ax = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return np.where(ax > 0, 2.0 ** (e - 8), 0.0)


def errors(gpu, ref):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    d = np.abs(gpu - ref)
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    excess = np.maximum(d - half_ulp_bf16(ref), 0.0)
    return {"max_abs": float(d.max()) if d.size else 0.0, "rms_ref": rms,
            "max_abs_over_rms": float(d.max()) / rms if rms > 0 else 0.0,
            "max_beyond_half_ulp_over_rms": float(excess.max()) / rms if rms > 0 and d.size else 0.0,
            "rms_err_over_rms": float(np.sqrt(np.mean(d ** 2))) / rms if rms > 0 else 0.0,
            "finite": bool(np.all(np.isfinite(gpu)))}


def assert_parity(wl_dtype, out_gpu, out_ref, st_gpu, st_ref, what=""):
    """The bounds of the module docstring, for the outputs and the final state."""
    eo = errors(out_gpu, out_ref)
    es = errors(st_gpu, st_ref)
    assert eo["finite"] and es["finite"], f"{what}: non-finite values"
    if wl_dtype == "f32":
        assert eo["max_abs"] <= F32_MAX_ABS, f"{what}: out {eo}"
        assert es["max_abs"] <= F32_MAX_ABS, f"{what}: state {es}"
        return eo, es
    if eo["rms_ref"] > 0:
        assert eo["max_beyond_half_ulp_over_rms"] <= BF16_MAX_ABS_OVER_RMS, f"{what}: out {eo}"
        assert eo["rms_err_over_rms"] <= BF16_RMS_ERR_OVER_RMS, f"{what}: out {eo}"
    else:
        assert eo["max_abs"] == 0.0, f"{what}: out {eo}"
    if es["rms_ref"] > 0:
        assert es["max_abs_over_rms"] <= BF16_MAX_ABS_OVER_RMS, f"{what}: state {es}"
    else:
        assert es["max_abs"] == 0.0, f"{what}: state {es}"
    return eo, es


def check_status():
    rc = binding.gdn_last_error(torch.cuda.current_stream().cuda_stream)
    assert rc == 0, f"device status {binding.STATUS.get(rc, rc)}"


def oracle_heads(wl, heads, S0_of=None, workers=None, fn=None):
    """Yields ((b, h), out_ref, state_ref) for each head in `heads`, in order: the
    head's inputs regenerated from the seeded streams and run through the fp64
    oracle, a few heads at a time on a thread pool (numpy releases the GIL in its
    generators and matrix products), so a full-size workload's every head can be
    checked without holding more than `workers` heads' fp64 results in host
    memory.  S0_of(b, h) gives a head's initial state (None: zeros).  With `fn`,
    yields ((b, h), fn(b, h)) instead (any per-head oracle computation)."""
    import contextlib
    import os
    from concurrent.futures import ThreadPoolExecutor

    try:
        from threadpoolctl import threadpool_limits
    except ImportError:
        threadpool_limits = None
    cores = len(os.sched_getaffinity(0))
    workers = workers or max(1, min(4, cores))
    limits = threadpool_limits(max(1, cores // workers)) if threadpool_limits else contextlib.nullcontext()

    def one(bh):
        b, h = bh
        if fn is not None:
            return bh, fn(b, h)
        return bh, oracle_head(wl, b, h, None if S0_of is None else S0_of(b, h))

    with limits, ThreadPoolExecutor(workers) as ex:
        pending = []
        it = iter(heads)
        for bh in it:
            pending.append(ex.submit(one, bh))
            if len(pending) >= workers:
                break
        while pending:
            bh, res = pending.pop(0).result()
            nxt = next(it, None)
            if nxt is not None:
                pending.append(ex.submit(one, nxt))
            yield (bh, res) if fn is not None else (bh, res[0], res[1])
