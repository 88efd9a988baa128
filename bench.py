"""Benchmark: frame-wise Gated DeltaNet forward tokens/s on the 961-frame,
880-token, 20-head, d112 bf16 workload (one minute of 720p-shaped latents), with
its fraction of the HBM roofline.

One step = one gdn_frame_fwd_ex call over the whole workload (every stage of
the path: key scale and beta, the per-frame transition terms, the D x D
recurrence over all frames, the read-out).  Inputs are resident in HBM when
the timed region starts and are larger than L2, so no flush is needed.  The
per-kernel device times behind the roofline come from a second pass over the
same steps with CUDA events around each of the library's launches.

    python bench.py [--gpus N --steps K --warmup W] [--impl reference]

``--backward`` times the backward pass instead (one gdn_frame_bwd call over the
same workload: every gradient, states recomputed), on its own metric line;
``--backward --reuse-forward`` the backward that reads the per-frame states a
forward call left in the shared workspace (gdn_frame_bwd_ex).

Under torchrun (N > 1) every rank runs its own full replica of the workload on
its own GPU (weak scaling; the path needs no cross-GPU exchange), the ranks
barrier around the timed region and the slowest rank's time is used.
"""
from __future__ import annotations

import argparse
import datetime as dt
import glob
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from linear_attention_video_gated_b300 import synth  # noqa: E402

METRIC = "frame-GDN fwd tokens/s at 961f×880tok×20h×d112; % of roofline"
METRIC_BWD = "frame-GDN bwd tokens/s at 961f×880tok×20h×d112; % of roofline"
UNIT = "tokens/s"


# ----------------------------------------------------------------- algorithmic work

def alg_bytes(wl) -> int:
    """q, k, v read once, out written once, g and beta read once, state in and out."""
    n = wl.B * wl.H * wl.T * wl.S * wl.D
    return 4 * n * wl.elem_bytes + 4 * wl.B * wl.H * wl.T * (1 + wl.S) + 2 * 4 * wl.B * wl.H * wl.D * wl.D


def alg_flops(wl) -> int:
    """Three S x D x D contractions per frame-head (prediction, write, read-out)."""
    return 6 * wl.B * wl.H * wl.T * wl.S * wl.D * wl.D


def alg_bytes_bwd(wl) -> int:
    """Backward: q, k, v and dout read once, dq, dk, dv written once, g and beta
    read once, dg and dbeta written once, state_in and dstate_out read, dstate_in
    written."""
    n = wl.B * wl.H * wl.T * wl.S * wl.D
    fh = wl.B * wl.H * wl.T
    return 7 * n * wl.elem_bytes + 2 * 4 * fh * (1 + wl.S) + 3 * 4 * wl.B * wl.H * wl.D * wl.D


def alg_flops_bwd(wl) -> int:
    """Seven S x D x D contractions per frame-head: the states again (prediction,
    write), Q^T dO, K~ U, the two halves of dK~, dO S^T."""
    return 14 * wl.B * wl.H * wl.T * wl.S * wl.D * wl.D


def kernel_alg_bytes(name: str, wl) -> int | None:
    """Algorithmic bytes each kernel is responsible for, per launch (one call).

    gram-type kernels read k, v, beta (and g); read-out kernels read q and write
    out.  Scratch traffic is not algorithmic.
    """
    fh = wl.B * wl.H * wl.T
    e = wl.elem_bytes
    if name.endswith("_gram"):
        return fh * (2 * wl.S * wl.D * e + 4 * wl.S + 4)
    if name.endswith("_readout") or name.endswith("_q_grad") or name.endswith("_qdo"):
        return fh * 2 * wl.S * wl.D * e  # q in, out out / dout in, dq out / q and dout in
    if name.endswith("_kv_grad"):
        return fh * (4 * wl.S * wl.D * e + 8 * wl.S + 4)  # k, v, beta, g in; dk, dv, dbeta out
    return None


# ----------------------------------------------------------------- multi-rank timing

def rank_max(value: float, world: int, device=None) -> float:
    """The maximum of `value` over all ranks (the slowest rank's time); the value
    itself when world == 1.  `device` is where the reduction tensor lives: the
    rank's GPU under NCCL, the CPU under gloo."""
    if world <= 1:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_value(units_per_rank: float, world: int, ms: float) -> float:
    """Whole-job throughput: the units every rank processed (each rank a full
    replica of the workload) divided by the slowest rank's time."""
    return units_per_rank * world / (ms / 1e3)


# ----------------------------------------------------------------- environment

def peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


def csrc_hash() -> str:
    h = hashlib.sha256()
    for p in sorted(glob.glob(os.path.join(ROOT, "linear_attention_video_gated_b300", "csrc", "*"))):
        h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, wl) -> float | None:
    """DRAM bytes per launch from profiles/ncu_traffic.txt, if taken on the current sources.

    Line format: <kernel> <dram bytes per launch> <csrc hash> <workload name>."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(p):
        return None
    cur = csrc_hash()
    for line in open(p):
        f = line.split()
        if len(f) >= 4 and not line.startswith("#") and f[0] == kernel and f[2] == cur and f[3] == wl.name:
            return float(f[1])
    return None


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons in the background."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id: str | None):
        self.rows = []
        self.proc = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50"]
        if bus_id:
            cmd += ["-i", bus_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = dt.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f")
            except ValueError:
                continue
            self.rows.append((ts, f))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: dt.datetime, t1: dt.datetime) -> dict | None:
        rows = [f for ts, f in self.rows if t0 <= ts <= t1] or [f for _, f in self.rows[-5:]]
        if not rows:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(f[2]) for f in rows if num(f[2]) is not None]
        mx = [num(f[3]) for f in rows if num(f[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for f in rows for n, v in zip(names, f[6:10]) if v.lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def host_link_gbs(dev, nbytes: int = 1 << 30, reps: int = 3) -> dict:
    """Measured pinned host <-> device copy bandwidth (GB/s): each direction alone
    (one cudaMemcpyAsync of `nbytes`, best of `reps`), and both directions at once
    on two streams (`duplex_*`: each direction's rate while the other runs), all
    timed with CUDA events."""
    import torch
    h = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    h2 = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d2 = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    res = {}
    for name, (dst, src) in (("h2d_gbs", (d, h)), ("d2h_gbs", (h, d))):
        best = float("inf")
        for _ in range(reps):
            e0, e1 = ev(), ev()
            e0.record()
            dst.copy_(src, non_blocking=True)
            e1.record()
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1))
        res[name] = nbytes / (best / 1e3) / 1e9
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    bi, bo = float("inf"), float("inf")
    for _ in range(reps):
        a0, a1, b0, b1 = ev(), ev(), ev(), ev()
        torch.cuda.synchronize()
        with torch.cuda.stream(s1):
            a0.record()
            d.copy_(h, non_blocking=True)
            a1.record()
        with torch.cuda.stream(s2):
            b0.record()
            h2.copy_(d2, non_blocking=True)
            b1.record()
        torch.cuda.synchronize()
        bi, bo = min(bi, a0.elapsed_time(a1)), min(bo, b0.elapsed_time(b1))
    res["duplex_h2d_gbs"] = nbytes / (bi / 1e3) / 1e9
    res["duplex_d2h_gbs"] = nbytes / (bo / 1e3) / 1e9
    res["bytes"] = nbytes
    return res


def link_bound_ms(h2d: float, d2h: float, link: dict) -> float:
    """The least time the host link needs for `h2d` bytes in and `d2h` bytes out
    when the two directions share it as measured: copies out overlap copies in as
    far as they can (each direction at its duplex rate), the rest of whichever
    direction has more to move runs alone."""
    ti = h2d / (link["duplex_h2d_gbs"] * 1e9)
    to = d2h / (link["duplex_d2h_gbs"] * 1e9)
    if to <= ti:  # copies out finish first; the rest of the copies in run alone
        rest = h2d - to * link["duplex_h2d_gbs"] * 1e9
        return (to + rest / (link["h2d_gbs"] * 1e9)) * 1e3
    rest = d2h - ti * link["duplex_d2h_gbs"] * 1e9
    return (ti + rest / (link["d2h_gbs"] * 1e9)) * 1e3


def bus_id(dev) -> str | None:
    import torch
    try:
        p = torch.cuda.get_device_properties(dev)
        return f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
    except Exception:
        return None


# ----------------------------------------------------------------- CPU oracle timing

def oracle_sample(wl, budget_s: float, max_heads: int | None = None, frames: int | None = None,
                  backward: bool = False, threads: int | None = None):
    """Times the fp64 oracle (its backward pass with ``backward``) on whole heads of
    the workload until `budget_s` of CPU work, with `threads` BLAS threads (all of
    the process's cores by default).  Returns (equivalent tokens/s, threads,
    sample description, seconds)."""
    import contextlib

    import oracle
    try:
        from threadpoolctl import threadpool_limits
    except ImportError:  # BLAS then runs on its default thread count: every core
        threadpool_limits = lambda n: contextlib.nullcontext()  # noqa: E731
    cores = threads or len(os.sched_getaffinity(0))
    T = wl.T if frames is None else min(frames, wl.T)
    max_heads = wl.B * wl.H if max_heads is None else max_heads
    spent, n = 0.0, 0
    with threadpool_limits(cores):
        while n < max_heads and (n == 0 or spent < budget_s):
            b, h = divmod(n, wl.H)
            one = wl.with_(B=1, H=1)
            hq = np.empty((1, 1, T, wl.S, wl.D), np.uint16 if wl.dtype == "bf16" else np.float32)
            hk, hv = np.empty_like(hq), np.empty_like(hq)
            hg = np.empty((1, 1, T), np.float32)
            hb = np.empty((1, 1, T, wl.S), np.float32)
            _fill_head(wl, b, h, hq, hk, hv, hg, hb)
            cvt = (lambda a: synth.bf16_to_f32(a[0, 0])) if wl.dtype == "bf16" else (lambda a: a[0, 0])
            q, k, v = cvt(hq), cvt(hk), cvt(hv)
            if backward:
                do = synth.head_dout(wl, b, h, 0, T)
                t0 = time.perf_counter()
                oracle.backward_head(q, k, v, hg[0, 0], hb[0, 0], None, do)
            else:
                t0 = time.perf_counter()
                oracle.scan_head(q, k, v, hg[0, 0], hb[0, 0])
            spent += time.perf_counter() - t0
            n += 1
            del one
    tokens = n * T * wl.S / wl.H  # a token of the workload spans all H heads
    desc = (f"{n} of {wl.B * wl.H} heads x {T} of {wl.T} frames x {wl.S} tokens (d{wl.D}) of the {wl.name} "
            f"workload, numpy fp64{' backward pass' if backward else ''}; tokens counted as heads/{wl.H}")
    return tokens / spent, cores, desc, spent


def _fill_head(wl, b, h, hq, hk, hv, hg, hb):
    from concurrent.futures import ThreadPoolExecutor
    T = hq.shape[2]

    def one(t):
        for name, dst in (("q", hq), ("k", hk), ("v", hv)):
            x = synth.frame_raw(wl, name, b, h, t)
            dst[0, 0, t] = synth.bf16_bits(x) if wl.dtype == "bf16" else x
        hg[0, 0, t] = synth.gate(wl, b, h, t)
        hb[0, 0, t] = synth.beta(wl, b, h, t)

    with ThreadPoolExecutor(len(os.sched_getaffinity(0))) as ex:
        list(ex.map(one, range(T)))


# ----------------------------------------------------------------- arms

def config_of(wl, mode, gate_logits=False, relu_linear=False, backward=False, rollout=False, reuse=False) -> dict:
    gates = ", gates from logits (fused gate prologue)" if gate_logits else ""
    if relu_linear:
        gates = ", cumulative ReLU linear attention baseline (no decay, no delta rule)"
    if backward:
        gates += (", BACKWARD pass (gdn_frame_bwd_ex: every gradient, the per-frame states read from the "
                  "forward call's workspace)" if reuse else
                  ", BACKWARD pass (gdn_frame_bwd: every gradient, states recomputed)")
    calls = (f"{len(wl.chunks)} chunk-causal calls of <= {max(wl.chunks)} frames carrying the state" if rollout
             else "single call over all frames")
    return {"workload": f"{wl.name}: B={wl.B} H={wl.H} T={wl.T} S={wl.S} D={wl.D} {wl.dtype} I/O, fp32 state, "
                        f"{calls}{gates}",
            "B": wl.B, "H": wl.H, "T": wl.T, "S": wl.S, "D": wl.D,
            "mode": "backward" if backward else {0: "sequential", 1: "prefix", 2: "split"}[mode],
            "l2": f"no flush: inputs larger than L2 "
                  f"({(alg_bytes_bwd(wl) if backward else alg_bytes(wl)) / 1e9:.1f} GB moved per step vs 126 MB L2)"}


def reference_arm(args, rank, world):
    if rank != 0:
        return
    wl = synth.WORKLOADS[args.workload]
    frames = min(wl.T, 240)
    times = []
    cores = len(os.sched_getaffinity(0))
    for i in range(args.warmup + args.steps):
        v, cores, desc, spent = oracle_sample(wl, 0.0, max_heads=1, frames=frames, backward=args.backward)
        if i >= args.warmup:
            times.append(spent)
    ms = 1e3 * float(np.mean(times))
    value = (frames * wl.S / wl.H) / (ms / 1e3)
    line = {"impl": "reference", "metric": METRIC_BWD if args.backward else METRIC, "value": value, "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(wl, args.mode, backward=args.backward),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def ours_arm(args, rank, world, local_rank):
    import torch

    from linear_attention_video_gated_b300 import binding, build_lib
    build_lib.ensure_built()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    wl = synth.WORKLOADS[args.workload]
    if args.frames:
        wl = wl.with_(T=min(args.frames, wl.T))
    mode = args.mode
    dtype = binding.GDN_BF16 if wl.dtype == "bf16" else binding.GDN_F32
    tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    hdt = torch.uint16 if wl.dtype == "bf16" else torch.float32

    # inputs: generated into pinned host memory, copied once to the device
    shape = (wl.B, wl.H, wl.T, wl.S, wl.D)
    hq, hk, hv = (torch.empty(shape, dtype=hdt, pin_memory=True) for _ in range(3))
    hg = torch.empty((wl.B, wl.H, wl.T), dtype=torch.float32, pin_memory=True)
    hb = torch.empty((wl.B, wl.H, wl.T, wl.S), dtype=torch.float32, pin_memory=True)
    synth.fill_io(wl, hq.numpy(), hk.numpy(), hv.numpy(), hg.numpy(), hb.numpy(), logits=args.gate_logits)
    if wl.dtype == "bf16":
        hq, hk, hv = (t.view(torch.bfloat16) for t in (hq, hk, hv))
    q, k, v = (t.to(dev) for t in (hq, hk, hv))
    g, beta = hg.to(dev), hb.to(dev)
    out = torch.empty(shape, dtype=tdt, device=dev)
    st_out = torch.empty((wl.B, wl.H, wl.D, wl.D), dtype=torch.float32, device=dev)
    need = binding.gdn_workspace_bytes(wl.B, wl.H, wl.T, wl.S, wl.D, dtype, mode)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream

    entry = binding.gdn_frame_fwd_from_logits if args.gate_logits else binding.gdn_frame_fwd_ex
    # chunk-causal rollout (a workload with chunks): one step = every chunk's call in
    # order, each chunk's tensors contiguous as a generator would produce them, the
    # state carried from call to call
    rollout = bool(wl.chunks) and not args.frames and not args.backward and not args.relu_linear
    if rollout:
        spans, t0 = [], 0
        for n in wl.chunks:
            spans.append((t0, n))
            t0 += n
        cut = lambda t, a, n: t[:, :, a:a + n].contiguous()  # noqa: E731
        chunk_in = [tuple(cut(t, a, n) for t in (q, k, v, g, beta)) + (cut(out, a, n),) for a, n in spans]
        need = max(binding.gdn_workspace_bytes(wl.B, wl.H, n, wl.S, wl.D, dtype, mode) for n in wl.chunks)
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
        states = [torch.empty((wl.B, wl.H, wl.D, wl.D), dtype=torch.float32, device=dev) for _ in range(2)]
    if args.backward:
        hdo = torch.empty(shape, dtype=hdt, pin_memory=True)
        synth.fill_dout(wl, hdo.numpy())
        dout = (hdo.view(torch.bfloat16) if wl.dtype == "bf16" else hdo).to(dev)
        grads = [torch.empty(shape, dtype=tdt, device=dev) for _ in range(3)]
        dg = torch.empty((wl.B, wl.H, wl.T), dtype=torch.float32, device=dev)
        dbeta = torch.empty((wl.B, wl.H, wl.T, wl.S), dtype=torch.float32, device=dev)
        need = binding.gdn_bwd_workspace_bytes(wl.B, wl.H, wl.T, wl.S, wl.D, dtype)
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
        bflags = ((binding.GDN_BWD_GATE_LOGITS if args.gate_logits else 0)
                  | (binding.GDN_BWD_STATES_IN_WORKSPACE if args.reuse_forward else 0))
        if args.reuse_forward:  # one forward call leaves the per-frame states in the workspace
            rc = entry(q.data_ptr(), k.data_ptr(), v.data_ptr(), g.data_ptr(), beta.data_ptr(), None,
                       out.data_ptr(), st_out.data_ptr(), wl.B, wl.H, wl.T, wl.S, wl.D, dtype, 0, ws.data_ptr(),
                       need, sp)
            if rc != 0:
                raise binding.GDNError(rc, "gdn_frame_fwd_ex")

    def step(qq=q, kk=k, vv=v, gg=g, bb=beta, so=st_out):
        if rollout:
            sin = None
            for i, ((_, n), (cq, ck, cv, cg, cb, co)) in enumerate(zip(spans, chunk_in)):
                sout = states[i & 1]
                rc = entry(cq.data_ptr(), ck.data_ptr(), cv.data_ptr(), cg.data_ptr(), cb.data_ptr(),
                           None if sin is None else sin.data_ptr(), co.data_ptr(), sout.data_ptr(), wl.B, wl.H, n,
                           wl.S, wl.D, dtype, mode, ws.data_ptr(), need, sp)
                if rc != 0:
                    raise binding.GDNError(rc, "gdn_frame_fwd_ex (rollout)")
                sin = sout
            return
        if args.backward:
            rc = binding.gdn_frame_bwd_ex(qq.data_ptr(), kk.data_ptr(), vv.data_ptr(), gg.data_ptr(),
                                          bb.data_ptr(), None, dout.data_ptr(), None, grads[0].data_ptr(),
                                          grads[1].data_ptr(), grads[2].data_ptr(), dg.data_ptr(),
                                          dbeta.data_ptr(), so.data_ptr(), wl.B, wl.H, wl.T, wl.S, wl.D, dtype,
                                          bflags, ws.data_ptr(), need, sp)
        elif args.relu_linear:
            rc = binding.gdn_relu_linear_fwd(qq.data_ptr(), kk.data_ptr(), vv.data_ptr(), None, out.data_ptr(),
                                             so.data_ptr(), wl.B, wl.H, wl.T, wl.S, wl.D, dtype, mode,
                                             ws.data_ptr(), need, sp)
        else:
            rc = entry(qq.data_ptr(), kk.data_ptr(), vv.data_ptr(), gg.data_ptr(), bb.data_ptr(),
                       None, out.data_ptr(), so.data_ptr(), wl.B, wl.H, wl.T, wl.S, wl.D, dtype,
                       mode, ws.data_ptr(), need, sp)
        if rc != 0:
            raise binding.GDNError(rc, "gdn_frame_fwd_ex")

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    rc = binding.gdn_last_error(sp)
    if rc != 0:
        raise binding.GDNError(rc, "warm-up")

    clocks = ClockSampler(bus_id(dev))
    time.sleep(0.3)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    w0 = dt.datetime.now()
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    w1 = dt.datetime.now()
    barrier()
    rc = binding.gdn_last_error(sp)
    if rc != 0:
        raise binding.GDNError(rc, "timed region")
    ms = rank_max(ev0.elapsed_time(ev1) / args.steps, world, dev)
    # Per-kernel device times: the same steps again, each launch of the library's
    # kernels between two CUDA events on its own stream (gdn_profile_begin/end).
    # The events between launches stop a kernel's prologue from overlapping the one
    # before, so this pass is a little slower than the timed region above.
    torch.cuda.synchronize()
    binding.gdn_profile_begin()
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    kstats = binding.gdn_profile_end()
    prof_ms = ev0.elapsed_time(ev1) / args.steps
    time.sleep(0.1)
    clocks.stop()
    clk = clocks.summary(w0, w1)
    rc = binding.gdn_last_error(sp)
    if rc != 0:
        raise binding.GDNError(rc, "profiled pass")
    value = job_value(wl.tokens, world, ms)
    pk = peaks()

    # roofline of the dominant kernel, from its own CUDA-event durations
    dom = max(kstats.items(), key=lambda kv: kv[1][1]) if kstats else None
    roof = None
    if dom is not None:
        name, (launches, tot) = dom
        avg = tot / launches
        ab = kernel_alg_bytes(name, wl)  # per call over the whole workload
        if ab is not None:
            # a rollout splits each call's work over one launch per chunk
            ab_launch = ab * args.steps / launches
            ach = ab_launch / (avg / 1e3) / 1e9
            traffic = ncu_traffic(name, wl) if launches == args.steps else None
            roof = {"bound": "hbm", "kernel": name, "achieved": ach, "peak": pk["hbm_gbs"], "unit": "GB/s",
                    "frac": ach / pk["hbm_gbs"], "traffic": traffic, "alg_bytes_per_launch": ab_launch,
                    "avg_launch_ms": avg, "peak_source": f"{pk['source']} (MEASURED_PEAKS.json hbm_gbs)"
                    if pk["source"] == "measured" else "fallback 6.4 TB/s"}
    call_gbs = (alg_bytes_bwd(wl) if args.backward else alg_bytes(wl)) / (ms / 1e3) / 1e9

    # end to end through the C ABI from pinned host buffers: gdn_frame_fwd_host,
    # which overlaps the copies of one chunk of frames with the kernels of another
    e2e = None
    if not args.no_e2e and not args.gate_logits and not args.relu_linear and not args.backward:
        ho = torch.empty(shape, dtype=tdt, pin_memory=True)
        hs = torch.empty((wl.B, wl.H, wl.D, wl.D), dtype=torch.float32, pin_memory=True)
        n_e2e = max(2, min(args.steps, args.e2e_steps))
        echunk = max(wl.chunks) if rollout else args.e2e_chunk
        hneed = binding.gdn_host_workspace_bytes(wl.B, wl.H, wl.T, wl.S, wl.D, dtype, echunk)
        hws = torch.empty(max(hneed, 1), dtype=torch.uint8, device=dev)

        def e2e_step():
            rc = binding.gdn_frame_fwd_host(hq.data_ptr(), hk.data_ptr(), hv.data_ptr(), hg.data_ptr(),
                                            hb.data_ptr(), None, ho.data_ptr(), hs.data_ptr(), wl.B, wl.H, wl.T,
                                            wl.S, wl.D, dtype, echunk, hws.data_ptr(), hneed, sp)
            if rc != 0:
                raise binding.GDNError(rc, "gdn_frame_fwd_host")

        e2e_step()
        torch.cuda.synchronize()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n_e2e):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        ems = rank_max(e0.elapsed_time(e1) / n_e2e, world, dev)
        h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hg, hb))
        d2h = ho.numel() * ho.element_size() + hs.numel() * hs.element_size()
        link = host_link_gbs(dev)
        # the copies overlap the kernels; the two copy directions share the link as
        # the duplex measurement found (copies in slow down while copies out run)
        bound_ms = max(link_bound_ms(h2d, d2h, link), ms)
        e2e = {"value": job_value(wl.tokens, world, ems), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": ems, "steps": n_e2e,
               "api": f"gdn_frame_fwd_host, {echunk}-frame chunks, pinned host buffers",
               "link": link, "bound_ms": bound_ms, "frac_of_bound": bound_ms / ems}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v_, cores, desc, spent = oracle_sample(wl, args.cpu_seconds, frames=240 if args.backward else None,
                                               backward=args.backward)
        cpu = {"value": v_, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc, "seconds": spent}
        # the oracle on one thread, on the 21-frame short clip (a whole head)
        v1, c1, d1, s1 = oracle_sample(synth.WORKLOADS["short"], 0.0, max_heads=1, backward=args.backward,
                                       threads=1)
        cpu["one_thread_short"] = {"value": v1, "unit": UNIT, "cores": c1, "sample": d1, "seconds": s1}

    if rank == 0:
        line = {"metric": METRIC_BWD if args.backward else METRIC, "value": value, "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
                "config": config_of(wl, mode, args.gate_logits, args.relu_linear, args.backward, rollout,
                                    args.reuse_forward),
                "roofline_pct": 100.0 * call_gbs / pk["hbm_gbs"],
                "call_achieved_gbs": call_gbs,
                "tflops": (alg_flops_bwd(wl) if args.backward else alg_flops(wl)) / (ms / 1e3) / 1e12,
                "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "clocks": clk,
                "gpu_launches": int(sum(n for n, _ in kstats.values())),
                "kernels": {k_: {"launches": n, "avg_ms": t / n} for k_, (n, t) in kstats.items()},
                "kernel_times_pass": {"ms_per_step": prof_ms, "how": "the same steps after the timed region, each "
                                      "library launch between two CUDA events on its stream"}}
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="minute", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--mode", type=int, default=0, choices=[0, 1, 2])
    ap.add_argument("--frames", type=int, default=None,
                    help="run the workload's first N frames only (small cases for profiling)")
    ap.add_argument("--gate-logits", action="store_true",
                    help="pass g and beta as logits (gdn_frame_fwd_from_logits)")
    ap.add_argument("--relu-linear", action="store_true",
                    help="time the cumulative ReLU linear attention baseline (gdn_relu_linear_fwd)")
    ap.add_argument("--backward", action="store_true",
                    help="time the backward pass (gdn_frame_bwd) instead of the forward scan")
    ap.add_argument("--reuse-forward", action="store_true",
                    help="with --backward: the backward reads the states a forward call left in its workspace")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--e2e-chunk", type=int, default=32, help="frames per chunk of the host-buffer entry point")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.reuse_forward and not args.backward:
        ap.error("--reuse-forward goes with --backward")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        reference_arm(args, rank, world)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    try:
        ours_arm(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
