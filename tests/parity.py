"""Shared helpers for the GPU parity tests: device upload of seeded inputs and the
tolerance checks.

Tolerances (written here, used by every parity test):
  * float32 I/O: max |gpu - oracle| <= 1e-4, for out and for the final state.
  * bf16 I/O: max |gpu - oracle| / rms(oracle) <= 2e-2, per tensor (out and the
    final state separately).  rms(gpu - oracle) / rms(oracle) is reported too.
    Rounding the outputs to bf16 alone costs up to 2^-8 relative at the largest
    elements (about 0.016 of the RMS on the 720p-shaped workloads), so the
    kernels' own error has to stay well below the remaining margin.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from linear_attention_video_gated_b300 import binding, synth

F32_MAX_ABS = 1e-4
BF16_MAX_ABS_OVER_RMS = 2e-2


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


def oracle_head(wl, b, h, S0=None):
    x = synth.head(wl, b, h)
    return oracle.scan_head(x["q"], x["k"], x["v"], x["g"], x["beta"], S0)


def errors(gpu, ref):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    d = np.abs(gpu - ref)
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    return {"max_abs": float(d.max()) if d.size else 0.0, "rms_ref": rms,
            "max_abs_over_rms": float(d.max()) / rms if rms > 0 else 0.0,
            "rms_err_over_rms": float(np.sqrt(np.mean(d ** 2))) / rms if rms > 0 else 0.0,
            "finite": bool(np.all(np.isfinite(gpu)))}


def assert_parity(wl_dtype, out_gpu, out_ref, st_gpu, st_ref, what=""):
    eo = errors(out_gpu, out_ref)
    es = errors(st_gpu, st_ref)
    assert eo["finite"] and es["finite"], f"{what}: non-finite values"
    if wl_dtype == "f32":
        assert eo["max_abs"] <= F32_MAX_ABS, f"{what}: out {eo}"
        assert es["max_abs"] <= F32_MAX_ABS, f"{what}: state {es}"
    else:
        if eo["rms_ref"] > 0:
            assert eo["max_abs_over_rms"] <= BF16_MAX_ABS_OVER_RMS, f"{what}: out {eo}"
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
