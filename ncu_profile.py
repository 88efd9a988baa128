"""Nsight Compute evidence for the library's kernels: the commands behind every
summary under profiles/, as one script.

Three captures, each run through ``bench.py`` (the same launch configuration the
bench times), each preceded by the same command without ncu, which must exit 0:

  launches  every launch of the library's kernels with its device time
            (``gpu__time_duration.sum`` only: one pass, safe on the full
            workload).  Per kernel: launches, total time, share of the step.
  counters  one kernel (``--kernel``), a small case (``--frames``), at most two
            launches: DRAM bytes and throughput, tensor-pipe activity, warps
            active, L2 hit rate, registers, the top warp stalls.
  traffic   ``counters``' DRAM bytes per launch scaled from the small case to
            the full workload by frame-heads (the kernels stream whole
            frame-heads, so their traffic grows in proportion), as the line
            bench.py reads from profiles/ncu_traffic.txt.

Every ncu command carries ``--clock-control none`` (the GPU's clocks are left as
they are).  Raw reports and CSVs go to ``--out`` (default ncu_out/); the
markdown summary, headed by the exact commands, is printed and written beside
them.

    python ncu_profile.py launches [--workload minute] [--mode 0] [--backward]
    python ncu_profile.py counters --kernel tc_gram [--frames 128] [--workload minute]
    python ncu_profile.py traffic --kernel tc_gram [--frames 128]
"""
from __future__ import annotations

import argparse
import csv
import io
import os
import shlex
import subprocess
import sys

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

NCU = os.environ.get("NCU", "ncu")

# counters read from a capture (ncu raw page names)
COUNTERS = [
    "gpu__time_duration.sum",
    "dram__bytes_read.sum",
    "dram__bytes_write.sum",
    "gpu__dram_throughput.avg.pct_of_peak_sustained_elapsed",
    "sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_elapsed",
    "sm__warps_active.avg.pct_of_peak_sustained_active",
    "lts__t_sector_hit_rate.pct",
    "sm__throughput.avg.pct_of_peak_sustained_elapsed",
    "launch__registers_per_thread",
    "launch__grid_size",
]
STALL_PREFIX = "smsp__average_warps_issue_stalled_"
SECTIONS = ["SpeedOfLight", "MemoryWorkloadAnalysis", "ComputeWorkloadAnalysis", "WarpStateStats", "Occupancy",
            "LaunchStats"]


def bench_cmd(args, steps=2, warmup=3) -> list:
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--workload", args.workload, "--mode", str(args.mode),
           "--steps", str(steps), "--warmup", str(warmup), "--no-e2e", "--no-cpu-baseline"]
    if getattr(args, "frames", None):
        cmd += ["--frames", str(args.frames)]
    if args.backward:
        cmd += ["--backward"]
    return cmd


def shown(cmd) -> str:
    """The command as run from the repository root (interpreter and paths relative)."""
    out = []
    for c in cmd:
        c = "python" if c == sys.executable else c
        out.append(os.path.relpath(c, ROOT) if os.path.isabs(c) and c.startswith(ROOT + os.sep) else c)
    return shlex.join(out)


def run(cmd, log) -> int:
    with open(log, "w") as f:
        f.write("$ " + shown(cmd) + "\n")
        f.flush()
        return subprocess.run(cmd, stdout=f, stderr=subprocess.STDOUT, cwd=ROOT).returncode


def plain_then(cmd, ncu_cmd, out, tag) -> None:
    """The recipe's order: the command alone must exit 0 before ncu runs it."""
    rc = run(cmd, os.path.join(out, f"{tag}_plain.log"))
    if rc != 0:
        raise SystemExit(f"the plain run exited {rc}; not profiling (see {tag}_plain.log)")
    rc = run(ncu_cmd, os.path.join(out, f"{tag}_ncu.log"))
    if rc != 0:
        raise SystemExit(f"ncu exited {rc} (see {tag}_ncu.log)")


def read_csv(path) -> list:
    text = open(path).read()
    start = text.find('"ID"')
    if start < 0:
        start = text.find('"')
    return list(csv.reader(io.StringIO(text[start:])))


def num(x) -> float:
    try:
        return float(str(x).replace(",", ""))
    except ValueError:
        return float("nan")


def launches(args) -> str:
    cmd = bench_cmd(args)
    csv_path = os.path.join(args.out, f"launches_{args.workload}.csv")
    ncu_cmd = [NCU, "--metrics", "gpu__time_duration.sum", "--clock-control", "none", "--csv", "--log-file",
               csv_path] + cmd
    plain_then(cmd, ncu_cmd, args.out, f"launches_{args.workload}")
    rows = read_csv(csv_path)
    hdr = rows[0]
    ik, iv, iu = hdr.index("Kernel Name"), hdr.index("Metric Value"), hdr.index("Metric Unit")
    per = {}
    for r in rows[1:]:
        if len(r) <= iv:
            continue
        scale = {"nsecond": 1e-3, "ns": 1e-3, "usecond": 1.0, "us": 1.0, "msecond": 1e3, "ms": 1e3,
                 "second": 1e6, "s": 1e6}[r[iu]]
        name = r[ik].split("(")[0].split("<")[0]
        name = name.split("::")[-1]
        n, tot = per.get(name, (0, 0.0))
        per[name] = (n + 1, tot + num(r[iv]) * scale)
    total = sum(t for _, t in per.values())
    lines = [f"# Launch list: {args.workload} workload, mode {args.mode}{' (backward)' if args.backward else ''}",
             "", "Command (plain run first, exit 0, then):", "", "```", shown(ncu_cmd), "```", "",
             "Per-launch times are cold-cache and serialised under ncu: compare shares, not absolutes.", "",
             "| kernel | launches | total µs | share |", "|---|---|---|---|"]
    for name, (n, t) in sorted(per.items(), key=lambda kv: -kv[1][1]):
        lines.append(f"| {name} | {n} | {t:.1f} | {100 * t / total:.1f} % |")
    return "\n".join(lines) + "\n"


def capture(args):
    cmd = bench_cmd(args)
    rep = os.path.join(args.out, f"counters_{args.kernel}_{args.workload}{args.frames or ''}")
    ncu_cmd = [NCU, "--clock-control", "none", "-k", f"regex:^{args.kernel}", "-s", str(args.skip), "-c",
               str(args.count), "--metrics", "dram__bytes_read.sum,dram__bytes_write.sum"]
    for sec in SECTIONS:
        ncu_cmd += ["--section", sec]
    ncu_cmd += ["-o", rep, "-f"] + cmd
    plain_then(cmd, ncu_cmd, args.out, f"counters_{args.kernel}")
    raw = subprocess.run([NCU, "-i", rep + ".ncu-rep", "--page", "raw", "--csv"], capture_output=True, text=True,
                         check=True).stdout
    rows = list(csv.reader(io.StringIO(raw)))
    return ncu_cmd, rows[0], rows[1], rows[2:]


def counters(args) -> str:
    ncu_cmd, hdr, unit, vals = capture(args)
    lines = [f"# ncu counters: {args.kernel}, {args.workload} workload"
             f"{f', first {args.frames} frames' if args.frames else ''}", "",
             "Command (plain run first, exit 0, then):", "", "```", shown(ncu_cmd), "```", "",
             "| counter | " + " | ".join(f"launch {i}" for i in range(len(vals))) + " |",
             "|---|" + "---|" * len(vals)]
    for c in COUNTERS:
        if c in hdr:
            i = hdr.index(c)
            lines.append(f"| {c} ({unit[i]}) | " + " | ".join(v[i] for v in vals) + " |")
    stalls = [(h, num(vals[0][i])) for i, h in enumerate(hdr)
              if h.startswith(STALL_PREFIX) and h.endswith("_per_issue_active.ratio")]
    stalls.sort(key=lambda x: -x[1])
    lines += ["", "Top warp stalls (first launch, cycles per issued instruction):", ""]
    for h, v in stalls[:6]:
        lines.append(f"- {h[len(STALL_PREFIX):-len('_per_issue_active.ratio')]}: {v:.3f}")
    return "\n".join(lines) + "\n"


def traffic(args) -> str:
    from linear_attention_video_gated_b300 import synth
    import bench

    ncu_cmd, hdr, unit, vals = capture(args)
    scale_of = {"byte": 1.0, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "Tbyte": 1e12}
    ir, iw = hdr.index("dram__bytes_read.sum"), hdr.index("dram__bytes_write.sum")
    per = [num(v[ir]) * scale_of[unit[ir]] + num(v[iw]) * scale_of[unit[iw]] for v in vals]
    small = sum(per) / len(per)
    wl = synth.WORKLOADS[args.workload]
    scale = wl.T / min(args.frames or wl.T, wl.T)  # frame-heads of the full workload per frame-head captured
    full = small * scale
    line = f"{args.kernel} {full:.0f} {bench.csrc_hash()} {args.workload}"
    return (f"# DRAM traffic of {args.kernel}, {args.workload} workload\n\nCommand (plain run first, exit 0, then):"
            f"\n\n```\n{shown(ncu_cmd)}\n```\n\nDRAM bytes (read + write) per launch on the first "
            f"{args.frames} frames: {small:.4g}; scaled x{scale:.3f} by frame-heads to the full workload: "
            f"{full:.4g}\n\nprofiles/ncu_traffic.txt line:\n\n    {line}\n")


def main():
    from linear_attention_video_gated_b300 import synth

    ap = argparse.ArgumentParser()
    ap.add_argument("what", choices=["launches", "counters", "traffic"])
    ap.add_argument("--workload", default="minute", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--mode", type=int, default=0, choices=[0, 1, 2])
    ap.add_argument("--backward", action="store_true")
    ap.add_argument("--kernel", default="tc_gram", help="kernel function name prefix (counters, traffic)")
    ap.add_argument("--frames", type=int, default=None, help="first N frames only (counters, traffic)")
    ap.add_argument("--skip", type=int, default=3, help="launches of the kernel skipped before capturing")
    ap.add_argument("--count", type=int, default=1, help="launches captured (counters, traffic; at most 2)")
    ap.add_argument("--out", default=os.path.join(ROOT, "ncu_out"))
    args = ap.parse_args()
    if args.what != "launches" and args.frames is None:
        args.frames = 128  # a small case: a few GB on the device, larger than L2
    args.count = max(1, min(args.count, 2))
    os.makedirs(args.out, exist_ok=True)
    text = {"launches": launches, "counters": counters, "traffic": traffic}[args.what](args)
    name = f"{args.what}_{args.kernel if args.what != 'launches' else args.workload}.md"
    with open(os.path.join(args.out, name), "w") as f:
        f.write(text)
    print(text)


if __name__ == "__main__":
    main()
