#!/usr/bin/env python
"""B and W backward TFLOP/s of one pipeline stage on GB300 (bf16, float32 accumulation).

A step is one iteration of the stage over m microbatches in the ZB-H1 order
the library generates (stage 0 of a p = m pipeline: F of every microbatch,
then B and W alternating): F, B and W of every microbatch, all through the C
ABI on one CUDA stream.  CUDA events around every B call and every W call
(on that stream) give the B and W device time; F runs inside the step but is
not part of the metric.  ``value`` = (B GEMM FLOPs + W GEMM FLOPs) / (B time +
W time) over the K timed steps.  ``e2e`` is the same metric with host buffers:
each step copies x and dy of every microbatch from pinned host memory,
runs F / B / W and copies dx back, all inside the timed region.

Run: python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
     python bench.py --impl reference   (the float64 oracle on the host cores)
Under torchrun each rank runs its own replica (weak scaling, no collective on
the data path); the barrier and the max over ranks only frame the timing.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORKLOADS = {
    "llama8b_stage": dict(kind="transformer", n_layers=4, hidden=4096, ffn=14336, n_heads=32, n_kv_heads=8,
                          head_dim=128, tokens=4096, m=8),
    # the same stage with the causal softmax attention core (one 4096-token sequence per microbatch)
    "llama8b_stage_causal": dict(kind="transformer", n_layers=4, hidden=4096, ffn=14336, n_heads=32, n_kv_heads=8,
                                 head_dim=128, tokens=4096, m=8, attention="causal", seq_len=0),
    "llama70b_stage": dict(kind="transformer", n_layers=2, hidden=8192, ffn=28672, n_heads=64, n_kv_heads=8,
                           head_dim=128, tokens=4096, m=8),
    "tiny_stage": dict(kind="mlp", n_layers=2, hidden=256, ffn=1024, n_heads=0, n_kv_heads=0, head_dim=0,
                       tokens=128, m=4),
}
for _t in (512, 1024, 2048, 4096, 8192):
    WORKLOADS[f"wgrad_sweep_t{_t}"] = dict(kind="linear", n_layers=1, hidden=4096, ffn=14336, n_heads=0,
                                           n_kv_heads=0, head_dim=0, tokens=_t, m=4)

METRIC = "B and W backward TFLOP/s per stage (bf16, 1xGB300) and % of dense tensor peak"
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def gemm_flops_per_mb(w):
    """Algorithmic GEMM FLOPs of one microbatch for one pass (B or W): 2 T in out per linear."""
    t, h, f = w["tokens"], w["hidden"], w["ffn"]
    if w["kind"] == "linear":
        return 2.0 * t * h * f
    per_layer = 2.0 * t * (2 * f * h + h * f)
    if w["kind"] == "transformer":
        q = (w["n_heads"] + 2 * w["n_kv_heads"]) * w["head_dim"]
        per_layer += 2.0 * t * (q * h + h * h)
    return per_layer * w["n_layers"]


# ---------------------------------------------------------------- ncu summaries

GEMM_SOURCES = ("gemm.cu", "device_common.cuh", "launch.h")
ROW_SOURCES = ("rowops.cu", "device_common.cuh", "launch.h")
EPILOGUES = {0: "bf16 store", 1: "residual epilogue", 2: "SwiGLU backward epilogue", 3: "float32 TMA reduce-add epilogue",
             4: "SwiGLU forward epilogue"}


def _sources_sha(names):
    import hashlib

    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "backward_split_linear_gb300", "csrc", name), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def gemm_source_sha():
    """sha256 over the GEMM kernel sources: a stored traffic figure holds only for these bytes."""
    return _sources_sha(GEMM_SOURCES)


def row_source_sha():
    """sha256 over the row kernels' sources (see gemm_source_sha)."""
    return _sources_sha(ROW_SOURCES)


def kernel_label(name):
    """Readable label of a kernel name from an ncu CSV; GEMMs by pass (F, B, W) and epilogue."""
    import re

    m = re.search(r"(gemm_pair_kernel|gemm_kernel)<([^>]*)>", name)
    if not m:
        base = re.sub(r"^void ", "", name).replace("(anonymous namespace)::", "").replace("<unnamed>::", "").replace("unnamed>::", "")
        base = re.sub(r"^zbk::", "", base)
        return base.split("(")[0]
    args = [a.strip() for a in m.group(2).split(",")]
    if m.group(1) == "gemm_kernel":
        args = args[1:]  # leading tile width
    a_mn, b_mn, epi = args[0] in ("true", "1"), args[1] in ("true", "1"), int(args[2])
    pas = "W" if a_mn else ("B" if b_mn else "F")
    fam = "gemm_pair_kernel" if m.group(1) == "gemm_pair_kernel" else "gemm_kernel (one CTA)"
    return f"{fam} {pas} ({EPILOGUES.get(epi, epi)})"


def _ncu_value(value, unit):
    v = float(value.replace(",", ""))
    scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "Tbyte": 1e12,
             "nsecond": 1e-9, "usecond": 1e-6, "msecond": 1e-3, "second": 1.0,
             "ns": 1e-9, "us": 1e-6, "ms": 1e-3, "s": 1.0}
    return v * scale.get(unit, 1.0)


def read_ncu_csv(paths):
    """Launches of one or more ncu --csv logs (a list, or names joined by commas), in order:
    list of (kernel name, {metric: value in bytes or seconds})."""
    import csv

    if isinstance(paths, str):
        paths = paths.split(",")
    launches = {}
    for f, path in enumerate(paths):
        with open(path) as fh:
            lines = [l for l in fh if l.startswith('"')]
        for row in csv.DictReader(lines):
            if not (row.get("ID") or "").isdigit() or not row.get("Metric Name"):
                continue
            key = (f, int(row["ID"]))
            name, met = launches.setdefault(key, (row["Kernel Name"], {}))
            met[row["Metric Name"]] = _ncu_value(row["Metric Value"], row.get("Metric Unit", ""))
    return [launches[k] for k in sorted(launches)]


def summarize_ncu(path, command, title, bw_flops=None):
    """Markdown summary of an ncu CSV: launches, time and share per kernel; DRAM bytes if captured.

    When DRAM bytes are present and `bw_flops` (the algorithmic FLOPs of the captured B and W
    GEMM launches) is given, closing lines give the B/W GEMMs' DRAM bytes per FLOP with the
    sha256 of the GEMM sources; bench.py scales it by its own FLOPs per launch to report the
    roofline's traffic while the sources are unchanged."""
    rows = {}
    for name, met in read_ncu_csv(path):
        r = rows.setdefault(kernel_label(name), {"n": 0, "s": 0.0, "rd": 0.0, "wr": 0.0})
        r["n"] += 1
        r["s"] += met.get("gpu__time_duration.sum", 0.0)
        r["rd"] += met.get("dram__bytes_read.sum", 0.0)
        r["wr"] += met.get("dram__bytes_write.sum", 0.0)
    total = sum(r["s"] for r in rows.values()) or 1.0
    dram = any(r["rd"] or r["wr"] for r in rows.values())
    out = [f"# {title}", "", "Command (GB300, one GPU; the same command exited 0 without ncu just before):", "",
           "```", command, "```", "",
           "Per-launch times under ncu are serialised and cold-cache: compare shares, not absolutes.", ""]
    head = "| kernel | launches | total ms | share |" + (" DRAM read MB / launch | DRAM write MB / launch |" if dram else "")
    out += [head, "|---|---:|---:|---:|" + ("---:|---:|" if dram else "")]
    for label, r in sorted(rows.items(), key=lambda kv: -kv[1]["s"]):
        line = f"| {label} | {r['n']} | {1e3 * r['s']:.2f} | {100 * r['s'] / total:.1f} % |"
        if dram:
            line += f" {r['rd'] / r['n'] / 1e6:.1f} | {r['wr'] / r['n'] / 1e6:.1f} |"
        out.append(line)
    out.append(f"| **total** | {sum(r['n'] for r in rows.values())} | {1e3 * total:.2f} | 100 % |" +
               (" | |" if dram else ""))
    if dram and bw_flops:
        bw = [r for label, r in rows.items() if label.startswith("gemm") and (" B (" in label or " W (" in label)]
        total = sum(r["rd"] + r["wr"] for r in bw)
        if total:
            out += ["", f"B/W GEMM DRAM bytes per algorithmic FLOP: {total / bw_flops:.6e} "
                        f"(GEMM sources sha256 {gemm_source_sha()[:16]}...)"]
    return "\n".join(out) + "\n"


ROW_KERNELS = ("rmsnorm_bwd_kernel", "attn_bwd_kv_kernel", "dgamma_partial_kernel", "dgamma_final_kernel")


def row_traffic_record(path, command, algorithmic_bytes):
    """The data file bench.py reads for roofline_rows.traffic: DRAM bytes of the captured B/W row
    kernel launches per algorithmic byte (`algorithmic_bytes`: their total, counted as the
    library's tracing counts them)."""
    rows = [(kernel_label(n), m) for n, m in read_ncu_csv(path)]
    sel = [m for label, m in rows if label.split("<")[0] in ROW_KERNELS]
    total = sum(m.get("dram__bytes_read.sum", 0.0) + m.get("dram__bytes_write.sum", 0.0) for m in sel)
    return {"what": "DRAM bytes (read + write) of the captured B and W row-kernel launches per algorithmic byte",
            "dram_bytes_per_unit": total / algorithmic_bytes, "unit": "byte per algorithmic byte",
            "launches": len(sel), "algorithmic_bytes": algorithmic_bytes, "command": command,
            "source_sha256": row_source_sha()}


def gemm_traffic_record(path, command, bw_flops):
    """The data file bench.py reads for roofline.traffic: B/W GEMM DRAM bytes per algorithmic FLOP."""
    rows = [(kernel_label(n), m) for n, m in read_ncu_csv(path)]
    bw = [m for label, m in rows if label.startswith("gemm") and (" B (" in label or " W (" in label)]
    total = sum(m.get("dram__bytes_read.sum", 0.0) + m.get("dram__bytes_write.sum", 0.0) for m in bw)
    return {"what": "DRAM bytes (read + write) of the captured B and W GEMM launches per algorithmic FLOP",
            "dram_bytes_per_unit": total / bw_flops, "unit": "byte per FLOP", "launches": len(bw),
            "algorithmic_flops": bw_flops, "command": command, "source_sha256": gemm_source_sha()}


def profiled_traffic(name, workload, sources_sha):
    """DRAM bytes per algorithmic unit from the committed data file profiles/<name>_<workload>.json
    (written with --summarize-ncu --write-json from an ncu capture), or None when there is none or
    the kernel sources changed since it was taken."""
    path = os.path.join(ROOT, "profiles", f"{name}_{workload}.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
    except (OSError, ValueError):
        return None, "no capture"
    if d.get("source_sha256") != sources_sha or "dram_bytes_per_unit" not in d:
        return None, "kernel sources changed since the capture"
    return float(d["dram_bytes_per_unit"]), f"profiles/{name}_{workload}.json"


def profiled_gemm_traffic(workload, w_mode):
    """DRAM bytes per algorithmic FLOP of the B/W GEMMs (see profiled_traffic)."""
    if w_mode != "per-microbatch":
        return None, "no capture for this W mode"
    return profiled_traffic("gemm_traffic", workload, gemm_source_sha())


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            d = json.load(fh)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi samples every 200 ms while the timed region runs."""

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={CLOCK_FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            for line in open(self.path):
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                    rows.append(parts)
        except Exception:
            pass
        finally:
            if self.path:
                os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        sm = [float(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        loaded = [s for s in sm if s > 0.5 * max(sm)]
        return {"sm_mhz": statistics.median(loaded or sm), "sm_max_mhz": float(rows[0][2]),
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max(float(r[3]) for r in rows if r[3].replace(".", "").isdigit())}


# ---------------------------------------------------------------- multi-rank timing frame


def max_over_ranks(values, dist=None, device="cpu"):
    """Element-wise max of `values` over all ranks (each rank times its own replica)."""
    if dist is None:
        return list(values)
    import torch

    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_tflops(flops_per_rank, world, ms):
    """Throughput of all ranks together: every rank does `flops_per_rank` in at most `ms`."""
    return world * flops_per_rank / (ms * 1e-3) / 1e12


# ---------------------------------------------------------------- oracle (host) leg


def oracle_sample(w, sample_tokens, seed=0, params_f64=None):
    """Times the float64 oracle's B and W for one microbatch of `sample_tokens` tokens."""
    import numpy as np

    from backward_split_linear_gb300 import synth
    from oracle import stage as S

    shp = dict(kind=w["kind"], n_layers=w["n_layers"], hidden=w["hidden"], ffn=w["ffn"], n_heads=w["n_heads"],
               n_kv_heads=w["n_kv_heads"], head_dim=w["head_dim"], eps=1e-5,
               attention=w.get("attention", "standin"), seq_len=w.get("seq_len", 0))
    if params_f64 is None:
        inp = synth.stage_inputs(w["kind"], w["n_layers"], w["hidden"], w["ffn"], w["n_heads"], w["n_kv_heads"],
                                 w["head_dim"], tokens=sample_tokens, n_mb=1, seed=seed, gamma="ones")
        params_f64 = synth.params_f64(inp["params"])
        x, dy = synth.bf16_to_f64(inp["x"][0]), synth.bf16_to_f64(inp["dy"][0])
    else:
        rng = np.random.default_rng(seed + 1)
        out = w["ffn"] if w["kind"] == "linear" else w["hidden"]
        x = synth.bf16_to_f64(synth.bf16_bits(rng.standard_normal((sample_tokens, w["hidden"]), dtype=np.float32)))
        dy = synth.bf16_to_f64(synth.bf16_bits(rng.standard_normal((sample_tokens, out), dtype=np.float32)))
    _, saved = S.stage_forward(x, params_f64, shp)
    t0 = time.perf_counter()
    _, kept = S.stage_backward_input(dy, params_f64, saved, shp)
    t1 = time.perf_counter()
    acc = S.zero_grads(params_f64)
    S.stage_backward_weight(acc, saved, kept, shp)
    t2 = time.perf_counter()
    return t1 - t0, t2 - t1, params_f64


def blas_threads():
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var):
            return int(os.environ[var])
    return None


def cpu_baseline(w, sample_tokens):
    tb, tw, _ = oracle_sample(w, sample_tokens)
    flops = 2 * gemm_flops_per_mb(dict(w, tokens=sample_tokens))
    cores = len(os.sched_getaffinity(0))
    return {"value": flops / (tb + tw) / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "blas_threads": blas_threads(),
            "sample": f"B and W of one {sample_tokens}-token microbatch of the {w['n_layers']}-layer stage "
                      f"(float64 numpy, F untimed); B {tb:.2f} s, W {tw:.2f} s"}


def run_reference(args, w):
    """--impl reference: the float64 oracle timed on the host cores, same metric."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    sample = args.sample_tokens
    _, _, params = oracle_sample(w, sample)  # builds the parameters once (untimed)
    for _ in range(args.warmup):
        oracle_sample(w, sample, params_f64=params)
    tb = tw = 0.0
    t0 = time.perf_counter()
    for k in range(args.steps):
        b, wt, _ = oracle_sample(w, sample, seed=k, params_f64=params)
        tb += b
        tw += wt
    wall = time.perf_counter() - t0
    flops = 2 * gemm_flops_per_mb(dict(w, tokens=sample)) * args.steps
    value = flops / (tb + tw) / 1e12
    cores = len(os.sched_getaffinity(0))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * (tb + tw) / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, **{k: v for k, v in w.items()},
                       "timed": f"each step: B and W of one {sample}-token microbatch of this workload "
                                f"(a bounded sample), float64 on the host cores",
                       "sample_tokens_per_step": sample, "wall_s": wall},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "blas_threads": blas_threads(),
                             "sample": f"each step: B and W of one {sample}-token microbatch of the stage"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- GPU leg


def run_order(st, order, xs, ys, dys, dxs, stream, ev, record, before=None, after=None):
    """One step: the (kind, mb) ops of `order` through the stage ('X': one flush).  With
    `record`, CUDA events from `ev` bracket every B and W call on `stream`; returns the
    (pass, start, end) spans."""
    i_ev = 0
    spans = []
    for kind, mb in order:
        if before is not None:
            before(kind, mb)
        if kind == "F":
            st.forward(mb, xs[mb], ys[mb], stream)
            continue
        a, b = ev[i_ev]
        i_ev += 1
        if record:
            a.record(stream)
        if kind == "B":
            st.backward_input(mb, dys[mb], dxs[mb], stream)
        elif kind == "W":
            st.backward_weight(mb, stream)
        else:
            st.flush(stream)
        if record:
            b.record(stream)
            spans.append(("B" if kind == "B" else "W", a, b))
        if after is not None:
            after(kind, mb)
    return spans


def measure_config(w, order, steps, warmup, peaks, peak_key, params=None, seed=0):
    """A further workload of the list, timed like the headline on a stage of its own: `warmup`
    untimed steps, then `steps` steps with events around every B and W call.  Returns its
    B / W TFLOP/s, the GEMM fraction of `peak_key`'s peak, the row kernels' share and the
    stash it held.  `params` reuses device weights of the same shapes."""
    import torch

    from backward_split_linear_gb300 import synth
    from backward_split_linear_gb300.runtime import Stage, bf16_from_bits

    t = w["tokens"]
    n_mb = 1 + max(mb for _, mb in order if mb >= 0)
    slots = w.get("slots", n_mb)
    inp = synth.stage_inputs(w["kind"], w["n_layers"] if params is None else 0, w["hidden"], w["ffn"], w["n_heads"],
                             w["n_kv_heads"], w["head_dim"], tokens=t, n_mb=n_mb, seed=seed, gamma="ones")
    if params is None:
        st = Stage.from_synth(w["kind"], w["n_layers"], w["hidden"], w["ffn"], w["n_heads"], w["n_kv_heads"],
                              w["head_dim"], 1e-5, t, slots, inp["params"], attention=w.get("attention", "standin"),
                              seq_len=w.get("seq_len", 0))
    else:
        st = Stage(w["kind"], w["n_layers"], w["hidden"], w["ffn"], w["n_heads"], w["n_kv_heads"], w["head_dim"],
                   1e-5, t, slots, params, attention=w.get("attention", "standin"), seq_len=w.get("seq_len", 0))
    xs = [bf16_from_bits(b) for b in inp["x"]]
    dys = [bf16_from_bits(b) for b in inp["dy"]]
    ys = [torch.empty(t, st.out_dim, dtype=torch.bfloat16, device="cuda") for _ in range(n_mb)]
    dxs = [torch.empty(t, w["hidden"], dtype=torch.bfloat16, device="cuda") for _ in range(n_mb)]
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for k, _ in order if k != "F"]
    st.set_tracing(True)
    for _ in range(warmup):
        run_order(st, order, xs, ys, dys, dxs, stream, ev, False)
    st.sync()
    st.read_tracing(reset=True)
    torch.cuda.synchronize()
    b_ms = w_ms = 0.0
    n_b = n_w = 0
    for _ in range(steps):
        spans = run_order(st, order, xs, ys, dys, dxs, stream, ev, True)
        torch.cuda.synchronize()
        for kind, a, b in spans:
            if kind == "B":
                b_ms += a.elapsed_time(b)
                n_b += 1
            else:
                w_ms += a.elapsed_time(b)
                n_w += 1
    trace = st.read_tracing(reset=True)
    st.sync()
    peak_inflight = st.stats()[1]
    st.close()
    flops_mb = gemm_flops_per_mb(w)
    b_fl = w_fl = flops_mb * n_mb * steps
    gemm = [trace[k] for k in ("gemm_backward_input", "gemm_backward_weight")]
    g_ms = sum(c["ms"] for c in gemm)
    g_ach = sum(c["flops"] for c in gemm) / (g_ms * 1e-3) / 1e12
    rows = [trace[k] for k in ("row_backward_input", "row_backward_weight")]
    r_ms = sum(c["ms"] for c in rows)
    peak = peaks[peak_key]
    rec = {"value": (b_fl + w_fl) / ((b_ms + w_ms) * 1e-3) / 1e12,
           "b_tflops": b_fl / (b_ms * 1e-3) / 1e12, "w_tflops": w_fl / (w_ms * 1e-3) / 1e12,
           "pct_of_dense_bf16_peak": {"b": 100 * b_fl / (b_ms * 1e-3) / 1e12 / peak,
                                      "w": 100 * w_fl / (w_ms * 1e-3) / 1e12 / peak, "peak_tflops": peak,
                                      "peak_source": f"{peaks['source']} {peak_key}"},
           "gemm_roofline_frac": g_ach / peak,
           "row_kernels_share_of_bw_time": r_ms / (b_ms + w_ms),
           "ms_per_call": {"B": b_ms / max(1, n_b), "W": w_ms / max(1, n_w)},
           "peak_inflight": peak_inflight, "steps": steps, "warmup": warmup}
    if w.get("attention") == "causal":
        ab = trace["attn_backward"]
        rec["attention_bwd_tflops"] = ab["flops"] / (ab["ms"] * 1e-3) / 1e12 if ab["ms"] else None
        rec["attention_bwd_share_of_b_time"] = ab["ms"] / b_ms if b_ms else None
        rec["attention_bwd_roofline"] = attention_roofline(ab, peaks, peak_key)
    return rec


def attention_layer_alone(w, peaks, reps=5, warmup=3):
    """The causal attention of one layer of workload `w` through its C-ABI ops alone (seeded N(0, 1)
    qkv and da, the forward's a and lse): CUDA events around `reps` back-to-back calls of the forward
    and of the backward after `warmup` calls, against the burst bf16 peak (nothing else runs, so
    the clocks are the unloaded ones)."""
    import torch

    from backward_split_linear_gb300 import binding as zb

    t, nh, nkv, d = w["tokens"], w["n_heads"], w["n_kv_heads"], w["head_dim"]
    seq = w.get("seq_len", 0)
    g = torch.Generator(device="cuda").manual_seed(0)
    qkv = torch.randn(t, (nh + 2 * nkv) * d, device="cuda", generator=g).to(torch.bfloat16)
    da = torch.randn(t, nh * d, device="cuda", generator=g).to(torch.bfloat16)
    a = torch.empty(t, nh * d, device="cuda", dtype=torch.bfloat16)
    lse = torch.empty(nh, zb.zb_op_attention_stat_stride(t), device="cuda", dtype=torch.float32)
    dvec = torch.empty_like(lse)
    dqkv = torch.empty_like(qkv)
    fwd = lambda: zb.zb_op_attention_causal_forward(qkv, a, lse, t, nh, nkv, d, seq)
    bwd = lambda: zb.zb_op_attention_causal_backward(qkv, a, da, lse, dvec, dqkv, t, nh, nkv, d, seq)
    times = {}
    for name, fn in (("fwd", fwd), ("bwd", bwd)):
        for _ in range(warmup):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        times[name] = e0.elapsed_time(e1) / reps
    # visible (query, key) pairs and head: sum over sequences of L (L + 1) / 2, times the heads
    lens = [seq] * (t // seq) + ([t % seq] if t % seq else []) if seq else [t]
    pairs = nh * sum(n * (n + 1) // 2 for n in lens)
    fwd_tf = 4 * d * pairs / (times["fwd"] * 1e-3) / 1e12
    bwd_tf = 10 * d * pairs / (times["bwd"] * 1e-3) / 1e12
    return {"fwd_ms": times["fwd"], "bwd_ms": times["bwd"], "fwd_tflops": fwd_tf, "bwd_tflops": bwd_tf,
            "bwd_frac_of_burst_peak": bwd_tf / peaks["bf16_tflops"], "peak_source": f"{peaks['source']} bf16_tflops",
            "flops_counted": "4 d (forward) and 10 d (backward) per visible query-key pair and head"}


def attention_roofline(ab, peaks, peak_key):
    """The causal attention backward (row kernel, dK/dV and dQ kernels, events around each call) against
    the dense bf16 peak, on its algorithmic count (5 products of 2 d per visible query-key pair)."""
    if not ab["ms"]:
        return None
    achieved = ab["flops"] / (ab["ms"] * 1e-3) / 1e12
    return {"bound": "tensor", "achieved": achieved, "peak": peaks[peak_key], "unit": "TFLOP/s",
            "frac": achieved / peaks[peak_key], "peak_source": f"{peaks['source']} {peak_key}",
            "launches": ab["launches"], "ms_per_launch": ab["ms"] / max(1, ab["launches"])}


def wgrad_sweep_record(tokens, steps, warmup, peaks):
    """One linear (in 4096, out 14336), m = 4 microbatches of `tokens` tokens: W per microbatch
    (after each B) and W of all four batched by one flush, each against the roofline that binds
    it: tensor time 2 T in out / peak against DRAM time (2 T (in + out) + 8 in out) / HBM peak
    (the float32 dW read and written once per W)."""
    from backward_split_linear_gb300 import binding as zb

    m, n_in, n_out = 4, 4096, 14336
    w = dict(kind="linear", n_layers=1, hidden=n_in, ffn=n_out, n_heads=0, n_kv_heads=0, head_dim=0, tokens=tokens,
             m=m)
    out = {}
    for mode, order in (("per_microbatch", zb.zb_schedule("zbh1", 0, m, m)),
                        ("flush", [("F", i) for i in range(m)] + [("B", i) for i in range(m)] + [("X", -1)])):
        rec = measure_config(w, order, steps, warmup, peaks, "bf16_tflops")
        t_w = tokens if mode == "per_microbatch" else m * tokens
        flops = 2.0 * t_w * n_in * n_out
        nbytes = 2.0 * t_w * (n_in + n_out) + 8.0 * n_in * n_out
        t_tensor = flops / (peaks["bf16_tflops"] * 1e12)
        t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
        w_calls = m if mode == "per_microbatch" else 1
        t_meas = rec["ms_per_call"]["W"] * 1e-3
        out[mode] = {"w_tflops": rec["w_tflops"], "b_tflops": rec["b_tflops"],
                     "w_pct_of_dense_bf16_peak": rec["pct_of_dense_bf16_peak"]["w"],
                     "w_tokens_per_call": t_w, "w_calls_per_step": w_calls,
                     "binding_roofline": "hbm" if t_hbm > t_tensor else "tensor",
                     "w_frac_of_binding_roofline": max(t_hbm, t_tensor) / t_meas,
                     "w_hbm_gbs": nbytes / t_meas / 1e9}
    return out


def other_workloads(args, st, peaks):
    """The rest of the workload list, each timed on its own stage after the headline: the
    70B-shaped stage, the ZB-H1 order of stage 3 of p = 8 over 16 microbatches (on the
    headline's weights), the 8B-shaped stage with the causal attention core, and the wgrad
    token sweep.  Steps are capped at 5 (at least 3 warm-up steps each)."""
    import torch

    from backward_split_linear_gb300 import binding as zb

    steps, warmup = max(1, min(args.steps, 5)), 3
    params = st.params
    st.close()
    st.workspace = st.grads = None
    torch.cuda.empty_cache()
    out = {"note": "each workload on a stage of its own after the headline's timed region; same timing "
                   "(events around every B and W call, F untimed); stage GEMM fractions against the "
                   "sustained peak, the sweep against the burst peak (short steps)"}
    w8 = dict(WORKLOADS["llama8b_stage"], slots=8)
    rec = measure_config(w8, zb.zb_schedule("zbh1", 3, 8, 16), steps, warmup, peaks, "bf16_tflops_sustained",
                         params=params)
    rec["order"] = "ZB-H1 order of stage 3 of p = 8, m = 16 (library generator), 8 stash slots"
    out["zbh1_stage3_p8_m16"] = rec
    del params
    torch.cuda.empty_cache()
    w70 = WORKLOADS["llama70b_stage"]
    rec = measure_config(w70, zb.zb_schedule("zbh1", 0, w70["m"], w70["m"]), steps, warmup, peaks,
                         "bf16_tflops_sustained")
    rec["order"] = "ZB-H1 order of stage 0 of p = m = 8"
    out["llama70b_stage"] = rec
    torch.cuda.empty_cache()
    wc = WORKLOADS["llama8b_stage_causal"]
    rec = measure_config(wc, zb.zb_schedule("zbh1", 0, wc["m"], wc["m"]), steps, warmup, peaks,
                         "bf16_tflops_sustained")
    rec["order"] = "ZB-H1 order of stage 0 of p = m = 8"
    rec["attention_layer_alone"] = attention_layer_alone(wc, peaks)
    out["llama8b_stage_causal"] = rec
    torch.cuda.empty_cache()
    out["wgrad_sweep_in4096_out14336_m4"] = {f"t{t}": wgrad_sweep_record(t, steps, warmup, peaks)
                                              for t in (512, 1024, 2048, 4096, 8192)}
    return out


def run_ours(args, w):
    import numpy as np
    import torch

    import __graft_entry__
    from backward_split_linear_gb300 import binding as zb
    from backward_split_linear_gb300 import synth
    from backward_split_linear_gb300.runtime import Stage, bf16_from_bits

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA device (the library has no CPU path)")
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    __graft_entry__.build()

    t, m = w["tokens"], w["m"]
    inp = synth.stage_inputs(w["kind"], w["n_layers"], w["hidden"], w["ffn"], w["n_heads"], w["n_kv_heads"],
                             w["head_dim"], tokens=t, n_mb=m, seed=rank, gamma="ones")
    st = Stage.from_synth(w["kind"], w["n_layers"], w["hidden"], w["ffn"], w["n_heads"], w["n_kv_heads"],
                          w["head_dim"], 1e-5, t, m, inp["params"], attention=w.get("attention", "standin"),
                          seq_len=w.get("seq_len", 0))
    xs = [bf16_from_bits(b) for b in inp["x"]]
    dys = [bf16_from_bits(b) for b in inp["dy"]]
    out_dim = st.out_dim
    ys = [torch.empty(t, out_dim, dtype=torch.bfloat16, device="cuda") for _ in range(m)]
    dxs = [torch.empty(t, w["hidden"], dtype=torch.bfloat16, device="cuda") for _ in range(m)]
    if args.w_mode == "flush":
        # F and B of every microbatch, then one flush: the stage batches the W of
        # consecutive full stash slots into one W over their concatenated tokens.
        order = [("F", i) for i in range(m)] + [("B", i) for i in range(m)] + [("X", -1)]
    else:
        pipe = args.pipeline or m
        order = zb.zb_schedule("zbh1", args.stage, pipe, m)
    stream = torch.cuda.current_stream()
    n_b = sum(1 for k, _ in order if k != "F")
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_b)]

    def step(record, before=None, after=None):
        return run_order(st, order, xs, ys, dys, dxs, stream, ev, record, before, after)

    st.set_tracing(True)
    # stash bytes one microbatch holds between its F and its W
    st.forward(0, xs[0], ys[0], stream)
    stash_per_mb = st.stats()[2]
    dys0 = torch.empty_like(dxs[0])
    st.backward_input(0, dys[0], dys0, stream)
    st.backward_weight(0, stream)
    st.sync()
    for _ in range(args.warmup):
        step(False)
    st.sync()
    st.read_tracing(reset=True)
    st.zero_grads()

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    b_ms = w_ms = 0.0
    with ClockSampler(local) as clocks:
        barrier()
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        all_spans = []
        for _ in range(args.steps):
            all_spans.append(step(True))
        t_end.record(stream)
        barrier()
    total_ms = t_start.elapsed_time(t_end)
    for spans in all_spans:
        for kind, a, b in spans:
            if kind == "B":
                b_ms += a.elapsed_time(b)
            else:
                w_ms += a.elapsed_time(b)
    trace = st.read_tracing(reset=True)
    st.sync()
    launches = sum(c["launches"] for c in trace.values())

    flops_mb = gemm_flops_per_mb(w)
    b_flops = flops_mb * m * args.steps
    w_flops = flops_mb * m * args.steps
    bw_ms = b_ms + w_ms
    bw_ms, b_ms, w_ms, total_ms = max_over_ranks([bw_ms, b_ms, w_ms, total_ms], dist, "cuda")
    value = whole_job_tflops(b_flops + w_flops, world, bw_ms)

    # ---- end to end: host buffers, copies inside the timed region
    e2e = None
    if not args.no_e2e:
        hx = [torch.empty(t, w["hidden"], dtype=torch.bfloat16, pin_memory=True) for _ in range(m)]
        hdy = [torch.empty(t, out_dim, dtype=torch.bfloat16, pin_memory=True) for _ in range(m)]
        hdx = [torch.empty(t, w["hidden"], dtype=torch.bfloat16, pin_memory=True) for _ in range(m)]
        for i in range(m):
            hx[i].copy_(xs[i])
            hdy[i].copy_(dys[i])
        st.set_tracing(False)

        # Copies run on their own stream, overlapped with the F/B/W order: a
        # microbatch's x lands before its F and its dy before its B, and its dx
        # goes back as soon as its B is done.  The step ends when the last copy
        # has landed, so every copy stays inside the timed region.
        copy_stream = torch.cuda.Stream()
        x_ready = [torch.cuda.Event() for _ in range(m)]
        dy_ready = [torch.cuda.Event() for _ in range(m)]
        dx_ready = [torch.cuda.Event() for _ in range(m)]

        def e2e_step():
            copy_stream.wait_stream(stream)  # the previous step no longer reads xs / dys
            with torch.cuda.stream(copy_stream):
                for i in range(m):
                    xs[i].copy_(hx[i], non_blocking=True)
                    x_ready[i].record(copy_stream)
                for i in range(m):
                    dys[i].copy_(hdy[i], non_blocking=True)
                    dy_ready[i].record(copy_stream)

            def before(kind, mb):
                if kind == "F":
                    stream.wait_event(x_ready[mb])
                elif kind == "B":
                    stream.wait_event(dy_ready[mb])

            def after(kind, mb):
                if kind == "B":
                    dx_ready[mb].record(stream)
                    copy_stream.wait_event(dx_ready[mb])
                    with torch.cuda.stream(copy_stream):
                        hdx[mb].copy_(dxs[mb], non_blocking=True)

            step(False, before, after)
            stream.wait_stream(copy_stream)

        e2e_step()
        barrier()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        n_e2e = max(1, min(args.steps, 3))
        a.record(stream)
        for _ in range(n_e2e):
            e2e_step()
        b.record(stream)
        barrier()
        e_ms = a.elapsed_time(b) / n_e2e
        h2d = sum(x.numel() * 2 for x in hx) + sum(x.numel() * 2 for x in hdy)
        d2h = sum(x.numel() * 2 for x in hdx)
        e2e = {"value": world * 2 * flops_mb * m / (e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e_ms,
               "note": "B+W GEMM FLOPs over the whole step: H2D of x and dy, F, B, W, D2H of dx "
                       "(copies on a side stream, overlapped with the order)"}

    peaks = measured_peaks()
    bytes_per_flop, traffic_src = profiled_gemm_traffic(args.workload, args.w_mode) if not args.overridden else (
        None, "workload overridden")
    gemm = {k: trace[k] for k in ("gemm_backward_input", "gemm_backward_weight")}
    g_ms = sum(c["ms"] for c in gemm.values())
    g_launch = sum(c["launches"] for c in gemm.values())
    g_flops = sum(c["flops"] for c in gemm.values())
    g_ach = g_flops / (g_ms * 1e-3) / 1e12
    # DRAM bytes of an average B/W GEMM launch: the captured bytes per FLOP times this run's FLOPs per launch
    traffic = bytes_per_flop * g_flops / max(1, g_launch) if bytes_per_flop else None
    rows = {k: trace[k] for k in ("row_backward_input", "row_backward_weight")}
    r_ms = sum(c["ms"] for c in rows.values())
    r_bytes = sum(c["bytes"] for c in rows.values())
    r_ach = r_bytes / (r_ms * 1e-3) / 1e9 if r_ms > 0 else None
    roofline = {"bound": "tensor", "kernel": "gemm_kernel (B and W GEMMs, tcgen05)",
                "achieved": g_ach, "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s",
                "frac": g_ach / peaks["bf16_tflops_sustained"], "traffic": traffic,
                "traffic_source": traffic_src,
                "peak_source": f"{peaks['source']} bf16 sustained (kernel timed inside a long step)",
                "launches": g_launch, "flops_per_launch": g_flops / max(1, g_launch),
                "ms_per_launch": g_ms / max(1, g_launch)}
    roofline_rows = None
    if r_ach is not None:
        r_launch = sum(c["launches"] for c in rows.values())
        # DRAM bytes of an average row-kernel launch: the captured bytes per algorithmic byte times
        # this run's algorithmic bytes per launch
        row_ratio, row_src = profiled_traffic("row_traffic", args.workload, row_source_sha()) if not args.overridden \
            else (None, "workload overridden")
        roofline_rows = {"bound": "hbm", "kernel": "B/W row kernels (RMSNorm backward, stand-in backward, "
                                                   "gamma reduction)",
                         "achieved": r_ach, "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": r_ach / peaks["hbm_gbs"],
                         "traffic": row_ratio * r_bytes / max(1, r_launch) if row_ratio else None,
                         "traffic_source": row_src, "launches": r_launch,
                         "bytes_per_launch": r_bytes / max(1, r_launch), "share_of_bw_time": r_ms / bw_ms}
    copy = trace.get("stash_copy")
    stash_copy = None
    if copy and copy["ms"] > 0:
        stash_copy = {"what": "stash copies of the caller's x (F) and dy (B), cudaMemcpyAsync device to device",
                      "gbs": copy["bytes"] / (copy["ms"] * 1e-3) / 1e9, "ms": copy["ms"]}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, args.sample_tokens if w["kind"] != "mlp" else w["tokens"])

    if rank == 0:
        cs = clocks.summary()
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": bw_ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "b_tflops": whole_job_tflops(b_flops, world, b_ms),
            "w_tflops": whole_job_tflops(w_flops, world, w_ms),
            "pct_of_dense_bf16_peak": {
                "b": 100 * b_flops / (b_ms * 1e-3) / 1e12 / peaks["bf16_tflops_sustained"],
                "w": 100 * w_flops / (w_ms * 1e-3) / 1e12 / peaks["bf16_tflops_sustained"],
                "peak_tflops": peaks["bf16_tflops_sustained"], "peak_source": peaks["source"] + " sustained"},
            "step_ms_with_forward": total_ms / args.steps,
            # F, B and W of the whole order: the same GEMM FLOPs three times over the step
            "fbw_tflops": whole_job_tflops(3 * flops_mb * m * args.steps, world, total_ms),
            "config": {"workload": args.workload, **{k: v for k, v in w.items()},
                       "order": (f"ZB-H1 order of stage {args.stage} of p = {args.pipeline or m} (library generator)"
                                 if args.w_mode != "flush"
                                 else "F and B of every microbatch, then one flush (W batched over the "
                                      "concatenated tokens of consecutive full stash slots)"),
                       "w_mode": args.w_mode,
                       "timed": "CUDA events around each B and W call; F runs in the step, untimed",
                       "l2": "inputs larger than L2 (stash per microbatch far above 129 MB)",
                       "gamma": "ones", "seed": rank},
            "roofline": roofline, "roofline_rows": roofline_rows, "stash_copy": stash_copy,
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
            "clocks": {"sm_mhz": cs["sm_mhz"], "sm_max_mhz": cs["sm_max_mhz"], "reasons": cs["reasons"],
                       "samples": cs["samples"]},
            "trace": {k: {"launches": v["launches"], "ms": round(v["ms"], 3)} for k, v in trace.items()},
        }
        # the memory-limited order search fed with this run's per-microbatch F, B and W times
        f_ms = sum(trace[k]["ms"] for k in ("gemm_forward", "row_forward", "attn_forward"))
        n_mb = m * args.steps
        t_f, t_b, t_w = (max(1, round(1e3 * v / n_mb)) for v in (f_ms, b_ms, w_ms))
        search = {"p": 8, "m": 16, "t_us": {"F": t_f, "B": t_b, "W": t_w}, "by_memory_limit": {}}
        for mem in (8, 12, 16):
            _, limit, span = zb.zb_schedule_search(0, 8, 16, mem, t_f, t_b, t_w)
            work = 16 * (t_f + t_b + t_w)
            search["by_memory_limit"][mem] = {"ceiling": limit, "makespan_ms": span / 1e3,
                                              "bubble_over_wall": (span - work) / span}
        line["schedule_search"] = search
        if args.w_mode != "flush":
            # the order the step ran: its held microbatches and the unit-time model of the whole pipeline
            pipe = args.pipeline or m
            inflight, peak, _ = st.stats()
            span, over_compute, over_wall = zb.zb_schedule_bubble("zbh1", pipe, m)
            line["order_stats"] = {"stage": args.stage, "p": pipe, "m": m, "peak_inflight": peak,
                                   "stash_bytes_per_microbatch": stash_per_mb,
                                   "unit_model": {"makespan": span, "bubble_over_compute": over_compute,
                                                  "bubble_over_wall": over_wall}}
        if w.get("attention") == "causal":
            # the attention core's own work: not in the metric (which counts the linears), reported beside it
            af, ab = trace["attn_forward"], trace["attn_backward"]
            line["attention"] = {
                "kind": "causal softmax, grouped K/V heads", "seq_len": w.get("seq_len", 0) or t,
                "fwd_tflops": af["flops"] / (af["ms"] * 1e-3) / 1e12 if af["ms"] else None,
                "bwd_tflops": ab["flops"] / (ab["ms"] * 1e-3) / 1e12 if ab["ms"] else None,
                "bwd_flops_counted": "5 products of 2 d per visible query-key pair (the kernels do 7: "
                                     "dQ recomputes S and dP)",
                "bwd_share_of_b_time": ab["ms"] / b_ms if b_ms else None,
                "b_tflops_with_attention": (b_flops + ab["flops"]) / (b_ms * 1e-3) / 1e12,
                "bwd_roofline": attention_roofline(ab, peaks, "bf16_tflops_sustained"),
                "layer_alone": attention_layer_alone(w, peaks) if not args.overridden else None,
            }
        if (world == 1 and args.workload == "llama8b_stage" and args.w_mode == "per-microbatch"
                and not args.overridden and args.stage == 0 and not args.pipeline and not args.no_workloads):
            line["workloads"] = other_workloads(args, st, peaks)
        print(json.dumps(line), flush=True)
    st.close()
    if dist is not None:
        dist.destroy_process_group()
    return 0


def run_op(args):
    """--op: times repeated launches of one per-step op at one shape (profiling and the wgrad sweep)."""
    import torch

    import __graft_entry__
    from backward_split_linear_gb300 import binding as zb

    __graft_entry__.build()
    t, n_in, n_out = (int(v) for v in args.shape.split(","))
    g = torch.Generator(device="cuda").manual_seed(0)

    def rnd(*shape, std=1.0):
        return (torch.randn(*shape, generator=g, device="cuda") * std).to(torch.bfloat16)

    peaks = measured_peaks()
    flops = 2.0 * t * n_in * n_out
    if args.op == "backward_weight":
        dy, x = rnd(t, n_out), rnd(t, n_in)
        dw = torch.zeros(n_out, n_in, dtype=torch.float32, device="cuda")
        launch = lambda: zb.zb_op_backward_weight(dy, x, dw, t, n_in, n_out)
        nbytes = 2.0 * t * (n_in + n_out) + 8.0 * n_in * n_out
    elif args.op == "backward_input":
        dy, w = rnd(t, n_out), rnd(n_out, n_in, std=0.02)
        dx = torch.empty(t, n_in, dtype=torch.bfloat16, device="cuda")
        launch = lambda: zb.zb_op_backward_input(dy, w, dx, t, n_in, n_out)
        nbytes = 2.0 * (t * n_out + n_out * n_in + t * n_in)
    elif args.op == "rmsnorm_backward_gamma":  # shape T,H,unused
        dn, x = rnd(t, n_in), rnd(t, n_in)
        rstd = torch.ones(t, dtype=torch.float32, device="cuda")
        dg = torch.zeros(n_in, dtype=torch.float32, device="cuda")
        nb = zb.zb_op_rmsnorm_backward_gamma_scratch_bytes(t, n_in)
        scratch = torch.empty(nb // 4 + 4, dtype=torch.float32, device="cuda")
        launch = lambda: zb.zb_op_rmsnorm_backward_gamma(dn, x, rstd, dg, t, n_in, scratch, nb)
        flops = 3.0 * t * n_in
        nbytes = 4.0 * t * n_in + 4.0 * t + 8.0 * n_in
    elif args.op == "backward_input_swiglu":  # n_in = ffn, n_out = hidden
        dy, w, gu = rnd(t, n_out), rnd(n_out, n_in, std=0.02), rnd(t, 2 * n_in)
        launch = lambda: zb.zb_op_backward_input_swiglu(dy, w, gu, gu, t, n_out, n_in)
        nbytes = 2.0 * (t * n_out + n_out * n_in) + 8.0 * t * n_in
    else:
        x, w = rnd(t, n_in), rnd(n_out, n_in, std=0.02)
        y = torch.empty(t, n_out, dtype=torch.bfloat16, device="cuda")
        launch = lambda: zb.zb_op_linear_forward(x, w, None, y, t, n_in, n_out)
        nbytes = 2.0 * (t * n_in + n_out * n_in + t * n_out)
    for _ in range(args.warmup):
        launch()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    # Read (not write) 256 MiB before every launch: L2 then holds only clean
    # lines of another buffer, so the timed launch neither hits in L2 nor pays
    # for writing back someone else's dirty lines.
    flush = torch.ones(64 << 20, dtype=torch.int32, device="cuda")
    for a, b in ev:
        flush.sum()
        a.record()
        launch()
        b.record()
    torch.cuda.synchronize()
    ms = sum(a.elapsed_time(b) for a, b in ev) / args.steps
    tflops = flops / (ms * 1e-3) / 1e12
    gbs = nbytes / (ms * 1e-3) / 1e9
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    bound = "tensor" if flops / nbytes >= ridge and args.op != "rmsnorm_backward_gamma" else "hbm"
    frac = tflops / peaks["bf16_tflops"] if bound == "tensor" else gbs / peaks["hbm_gbs"]
    print(json.dumps({"op": args.op, "shape": {"tokens": t, "in": n_in, "out": n_out}, "ms": ms,
                      "tflops": tflops, "pct_of_burst_bf16": 100 * tflops / peaks["bf16_tflops"],
                      "gbs": gbs, "bound": bound, "frac_of_binding_roofline": frac,
                      "peak_source": peaks["source"] + " burst (kernel timed alone)",
                      "l2": "256 MiB buffer read before every launch"}), flush=True)
    assert zb.zb_device_status()[0] == 0
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="llama8b_stage")
    ap.add_argument("--sample-tokens", type=int, default=256,
                    help="tokens of the microbatch the host oracle runs (cpu_baseline / reference arm)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-workloads", "--no-configs", dest="no_workloads", action="store_true",
                    help="skip the sub-records of the other workloads (70B-shaped stage, ZB-H1 order of stage 3, causal, wgrad sweep)")
    ap.add_argument("--w-mode", choices=["per-microbatch", "flush"], default="per-microbatch",
                    help="W as one call per microbatch (the ZB-H1 order) or batched in one flush")
    ap.add_argument("--op", choices=["backward_weight", "backward_input", "backward_input_swiglu", "forward",
                                     "rmsnorm_backward_gamma"],
                    help="time one per-step op instead of the stage (with --shape T,IN,OUT)")
    ap.add_argument("--shape", default="4096,4096,14336")
    ap.add_argument("--stage", type=int, default=0, help="pipeline stage whose ZB-H1 order the step runs")
    ap.add_argument("--pipeline", type=int, default=0, help="pipeline depth p of that order (default: m)")
    ap.add_argument("--layers", type=int, help="override the workload's layer count (small ncu captures)")
    ap.add_argument("--microbatches", type=int, help="override the workload's microbatch count")
    ap.add_argument("--summarize-ncu", metavar="CSV[,CSV...]", help="print a markdown summary of ncu --csv logs")
    ap.add_argument("--ncu-command", default="", help="the command that wrote the CSV (for the summary)")
    ap.add_argument("--title", default="ncu launch list")
    ap.add_argument("--bw-flops", type=float, help="algorithmic FLOPs of the B/W GEMM launches in the CSV")
    ap.add_argument("--row-bytes", type=float, help="algorithmic bytes of the B/W row-kernel launches in the CSV")
    ap.add_argument("--write-json", metavar="PATH", help="with --summarize-ncu and --bw-flops: write the "
                                                         "bytes-per-FLOP data file that roofline.traffic reads")
    args = ap.parse_args()
    if args.summarize_ncu:
        sys.stdout.write(summarize_ncu(args.summarize_ncu, args.ncu_command, args.title, args.bw_flops))
        if args.write_json and (args.bw_flops or args.row_bytes):
            rec = (gemm_traffic_record(args.summarize_ncu, args.ncu_command, args.bw_flops) if args.bw_flops else
                   row_traffic_record(args.summarize_ncu, args.ncu_command, args.row_bytes))
            with open(args.write_json, "w") as fh:
                json.dump(rec, fh, indent=1)
                fh.write("\n")
        return 0
    if args.op:
        return run_op(args)
    w = dict(WORKLOADS[args.workload])
    args.overridden = False
    if args.layers:
        w["n_layers"] = args.layers
        args.overridden = True
    if args.microbatches:
        w["m"] = args.microbatches
        args.overridden = True
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
