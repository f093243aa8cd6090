"""Benchmark of the exact attention forward pass on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--splitkv S]

One step = one forward pass (S = QK^T, masking, online softmax, P V,
normalisation and L) over the whole workload, inputs resident in HBM.  The
default workload is the largest of the five named ones that fits one GPU,
b1h32n32768d128_causal (B=1, H=32, N=32768, d=128, causal, bf16).  The
metric is attention-forward TFLOPS = 4*B*H*N^2*d (halved for a causal mask)
/ kernel time.  L2 is flushed (a 256 MiB write) between timed iterations;
each iteration's kernel is timed with CUDA events on the launching stream.

The line also carries `per_config`: every named workload (the 128-token
single head as latency in microseconds, the others in TFLOPS and roofline
fraction) timed the same way, each with its outputs checked against the
float64 oracle (whole heads where affordable, else sampled rows), its
DRAM-traffic record and its exponentials per second against the MUFU rate,
and `bwd_per_config`: the backward (fa_bwd) on the same workloads (all but
the 128-token one), timed the same way in TFLOPS counted as 2.5x the
forward's FLOPs, each checked on sampled rows of two heads against the
oracle's gradients under the derived gradient bound; and `fp8_per_config`:
the 8-bit forward (fa_fwd_e4m3) on the same workloads from E4M3 codes made
once, timed the same way, with its ratio to the bf16 kernel and a check of
the codes and of sampled rows of O and L against the oracle.

Rank 0 prints one JSON line.  Under torchrun every rank runs the same
workload on its own GPU (independent replicas, no collective on the data
path); `value` is the total over ranks divided by the slowest rank's time.

--impl reference times the float64 CPU oracle instead (a deliberately slow
baseline), on a bounded sample of the same workload per step.

--bwd times the backward pass (fa_bwd: dQ, dK, dV from Q, K, V, O, L and dO;
three kernels per step: the row statistics, then the dK/dV and dQ walks on
two streams, joined back before the step's end event) on the same
workloads; the metric counts 2.5x the forward's FLOPs (five matrix products
instead of two; the dQ walk recomputes two of them, which it does not count).

--fp8 times the 8-bit forward (fa_fwd_e4m3) on E4M3 codes of the same
workload (quantised once per (batch, head) by fa_quantize_e4m3, outside the
timed region; that step's own time is reported beside it).  The roofline
peak is the measured bf16 peak times 2, the nominal FP8 / BF16 ratio.

--unfused times standard attention in three kernels (fa_attn_unfused: S
and P written to and read back from HBM) beside the fused forward on the
same workload (default b4h16n2048d128), with the DRAM traffic of both from
the committed ncu record and the arithmetic intensities.

--splitkv S times the split key/value forward (fa_fwd_splitkv: S key ranges
per query tile, 0 = the library's choice, then the logsumexp merge; two
kernels per step) on a few-heads, long-sequence workload
(default b1h1n8192d128), and reports the one-pass kernel's time on the same
workload beside it.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOPS (bf16) and % of GB300 dense BF16 peak, 1 GPU"
DEFAULT_WORKLOAD = "b1h32n32768d128_causal"
# ex2.approx.ftz.f32 throughput measured by a microbenchmark on GB300 (inputs
# changing every iteration): one warp instruction per ~4.3 cycles per SM
# sub-partition, i.e. 32 / 4.3 * 4 = ~29.8 results per clock per SM.
MUFU_EX2_PER_CLK_SM = 29.8
N_SMS = 152
# The files the forward pair kernel and its launch schedule (head groups,
# cluster count) come from: the committed DRAM traffic record is used only
# while they hash to the captured value.
KERNEL_SOURCES = ("exact_attention_forward_04_gb300/csrc/fa_fwd_pair.cuh",
                  "exact_attention_forward_04_gb300/csrc/sm103_ptx.cuh",
                  "exact_attention_forward_04_gb300/csrc/tmem_ldst.cuh",
                  "exact_attention_forward_04_gb300/csrc/fa_fwd.cu")
# The same for the unfused three-kernel path (records keyed "unfused:<workload>").
UNFUSED_KERNEL_SOURCES = ("exact_attention_forward_04_gb300/csrc/fa_unfused.cuh",
                          "exact_attention_forward_04_gb300/csrc/sm103_ptx.cuh",
                          "exact_attention_forward_04_gb300/csrc/tmem_ldst.cuh",
                          "exact_attention_forward_04_gb300/csrc/fa_fwd.cu")
# The same for the backward kernels and their launch (records keyed
# "bwd:<workload>": the three kernels of one step summed).
BWD_KERNEL_SOURCES = ("exact_attention_forward_04_gb300/csrc/fa_bwd.cuh",
                      "exact_attention_forward_04_gb300/csrc/sm103_ptx.cuh",
                      "exact_attention_forward_04_gb300/csrc/tmem_ldst.cuh",
                      "exact_attention_forward_04_gb300/csrc/fa_fwd.cu")


def _args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--workload", default=None,
                   help=f"workload name (default: {DEFAULT_WORKLOAD}; b4h16n2048d128 with --bwd, --fp8 or "
                        "--unfused; b1h1n8192d128 with --splitkv)")
    p.add_argument("--impl", default="ours", choices=("ours", "reference"))
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="budget of the CPU oracle sample")
    p.add_argument("--bwd", action="store_true",
                   help="time the backward (fa_bwd) instead of the forward")
    p.add_argument("--fp8", action="store_true",
                   help="time the 8-bit forward (fa_fwd_e4m3) on E4M3 codes")
    p.add_argument("--splitkv", type=int, default=-1,
                   help="time fa_fwd_splitkv with this many splits (0: library's choice)")
    p.add_argument("--unfused", action="store_true",
                   help="time standard three-kernel attention beside the fused forward")
    p.add_argument("--no-per-config", action="store_true",
                   help="skip the per_config block (every named workload)")
    return p.parse_args()


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}, "fallback"


def _kernel_hash(sources=KERNEL_SOURCES):
    h = hashlib.sha256()
    for rel in sources:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(os.path.basename(rel).encode() + f.read())
    return h.hexdigest()[:16]


def _traffic(workload_name):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    if workload_name.startswith("bwd:"):
        if d.get("bwd_kernel_hash") != _kernel_hash(BWD_KERNEL_SOURCES):
            return None
    elif workload_name.startswith("unfused:"):
        if d.get("unfused_kernel_hash") != _kernel_hash(UNFUSED_KERNEL_SOURCES):
            return None
    elif d.get("kernel_hash") != _kernel_hash():
        return None
    ent = d.get("per_launch_bytes", {}).get(workload_name)
    return ent


class ClockSampler:
    """nvidia-smi samples every 100 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = [ln for (t, ln) in self.lines if t0 - 0.15 <= t <= t1 + 0.15] or \
            [ln for (_, ln) in self.lines]
        sm, smax, reasons, power = [], [], set(), []
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in rows:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(n)
        return {
            "sm_mhz": statistics.median(sm) if sm else None,
            "sm_max_mhz": max(smax) if smax else None,
            "power_w_max": max(power) if power else None,
            "samples": len(sm),
            "reasons": sorted(reasons),
        }


def _dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _exps(w):
    """Exponentials the definition takes per launch: one per visible
    (query, key) pair."""
    per_head = w.N * (w.N + 1) // 2 if w.causal else w.N * w.N
    return w.B * w.H * per_head


def _mufu(w, mean_ms, peaks):
    """Secondary roofline: exponentials per second against the MUFU ex2 rate
    (microbenchmark figure x SMs x the maximum SM clock)."""
    clk = float(peaks.get("sm_max_mhz", 2070.0)) * 1e6
    peak = MUFU_EX2_PER_CLK_SM * N_SMS * clk
    rate = _exps(w) / (mean_ms * 1e-3)
    return {"exps_per_s": rate, "peak": peak, "frac": rate / peak, "unit": "exp/s",
            "peak_source": f"ex2.approx {MUFU_EX2_PER_CLK_SM}/clk/SM (microbenchmark) x "
                           f"{N_SMS} SMs x {clk / 1e6:.0f} MHz"}


def _time_launches(launch, stream, flush, n):
    """n launches, each after an L2 flush, each timed by CUDA events on the
    launching stream; returns the per-launch times in ms."""
    import torch
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n)]
    with torch.cuda.stream(stream):
        for a, b in ev:
            flush.zero_()
            a.record(stream)
            launch()
            b.record(stream)
    stream.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def _parity_sample(w, q, k, v, o_dev, l_dev):
    """The outputs against the float64 oracle (test infrastructure): whole
    heads where the oracle takes well under a second per head, else sampled
    rows (tile edges, first and last rows, random rows) of four heads."""
    import torch
    import oracle
    from tests.parity import compare
    torch.set_num_threads(os.cpu_count() or 1)
    o, lse = o_dev.cpu(), l_dev.cpu()
    BH = w.B * w.H
    head_cost = w.N * w.N * w.d * (2 if w.causal else 4)
    if head_cost <= 3e9:
        n_heads = BH if BH <= 8 else (3 if head_cost > 1e9 else 8)
        heads = sorted({(i * (BH - 1)) // max(1, n_heads - 1) for i in range(n_heads)})
        res = []
        for hh in heads:
            b, h = divmod(hh, w.H)
            sl = (slice(b, b + 1), slice(h, h + 1))
            O_ref, L_ref = oracle.attention_ref(q[sl], k[sl], v[sl], w.scale, w.causal)
            res.append(compare(o[sl], lse[sl], O_ref, L_ref))
        worst = {key: max(r[key] for r in res) for key in ("max_dO", "max_dO_over_bound", "max_dL")}
        worst["finite"] = all(r["finite"] for r in res)
        worst["ok"] = worst["finite"] and worst["max_dO_over_bound"] <= 1.0 and worst["max_dL"] <= 1e-3
        worst["sample"] = f"{len(heads)} of {BH} heads in full"
        return worst
    g = torch.Generator().manual_seed(w.seed + 12345)
    heads = sorted({0, BH - 1, BH // 3, (2 * BH) // 3})
    base_rows = {0, 1, 127, 128, 255, 256, w.N // 2, w.N - 2, w.N - 1}
    picks = []
    for hh in heads:
        b, h = divmod(hh, w.H)
        rnd = torch.randint(0, w.N, (8,), generator=g).tolist()
        picks += [(b, h, i) for i in sorted(base_rows | set(rnd)) if 0 <= i < w.N]
    O_ref, L_ref = oracle.attention_rows(q, k, v, w.scale, w.causal, picks)
    idx = torch.tensor(picks)
    r = compare(o[idx[:, 0], idx[:, 1], idx[:, 2]], lse[idx[:, 0], idx[:, 1], idx[:, 2]], O_ref, L_ref)
    r["sample"] = f"{len(picks)} rows of {len(heads)} heads (tile edges, ends, random)"
    return r


def _latency(lib, args, stream, n=200):
    """Latency of one call on a tiny workload: host enqueue time per call
    (back to back), the kernel's CUDA-event time, and call + stream
    synchronise, in microseconds."""
    import torch
    sh = stream.cuda_stream
    for _ in range(20):
        lib.fa_fwd(*args, sh)
    stream.synchronize()
    t0 = time.perf_counter()
    for _ in range(n):
        lib.fa_fwd(*args, sh)
    t1 = time.perf_counter()
    stream.synchronize()
    lat, ks = [], []
    for _ in range(n):
        a0 = time.perf_counter()
        lib.fa_fwd(*args, sh)
        stream.synchronize()
        lat.append(time.perf_counter() - a0)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(n):
        e0.record(stream)
        lib.fa_fwd(*args, sh)
        e1.record(stream)
        stream.synchronize()
        ks.append(e0.elapsed_time(e1))
    return {"host_enqueue_us": 1e6 * (t1 - t0) / n,
            "call_and_sync_us": 1e6 * statistics.median(lat),
            "kernel_us": 1e3 * statistics.median(ks), "calls": n}


def _per_config(a, lib, dev, stream, flush, peaks, main=None):
    """Every named workload, timed like the headline (L2 flushed, CUDA
    events), each checked against the oracle.  `main` carries the headline
    workload's own measurement so that it is not repeated."""
    import torch
    from exact_attention_forward_04_gb300.inputs import WORKLOADS, make_workload
    peak = peaks["bf16_tflops"]
    out = {}
    for w in WORKLOADS:
        q, k, v = make_workload(w)
        qd, kd, vd = (t.to(dev) for t in (q, k, v))
        o = torch.empty_like(qd)
        lse = torch.empty(w.B, w.H, w.N, dtype=torch.float32, device=dev)
        args = (qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), lse.data_ptr(),
                w.B, w.H, w.N, w.d, w.scale, int(w.causal))

        def launch():
            st = lib.fa_fwd(*args, stream.cuda_stream)
            if st != 0:
                raise RuntimeError(f"fa_fwd: status {st}")

        if main is not None and w.name == main["name"]:
            times = main["times"]  # the headline's own timing; one launch for the outputs
            _time_launches(launch, stream, flush, 1)
        else:
            _time_launches(launch, stream, flush, 3)
            times = _time_launches(launch, stream, flush, max(5, min(a.steps, 20)))
        st = lib.fa_check_errors(stream.cuda_stream)
        if st != 0:
            raise RuntimeError(f"per_config {w.name}: status {st}")
        mean_ms = sum(times) / len(times)
        ent = {"B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal,
               "kernel_ms_mean": mean_ms, "kernel_ms_median": statistics.median(times)}
        if w.N * w.N * w.B * w.H < 1e6:
            ent["latency"] = _latency(lib, args, stream)
            ent["note"] = "latency-bound (one 128-row block, one CTA): reported in microseconds"
        else:
            tf = w.flops / (mean_ms * 1e-3) / 1e12
            ent.update({"tflops": tf, "frac_of_bf16_peak": tf / peak,
                        "traffic_bytes": _traffic(w.name),
                        "algorithmic_bytes": w.B * w.H * (8 * w.N * w.d + 4 * w.N)})
        ent["mufu"] = _mufu(w, mean_ms, peaks)
        ent["parity"] = _parity_sample(w, q, k, v, o, lse)
        out[w.name] = ent
        del qd, kd, vd, o, lse
        torch.cuda.empty_cache()
    return out


def _bwd_per_config(a, lib, dev, stream, flush, peaks):
    """The backward (fa_bwd) on every named workload but the 128-token one,
    timed like the forward's per_config (L2 flushed, CUDA events on the
    launching stream, TFLOPS as 2.5x the forward's FLOPs), each checked on
    sampled rows of two heads against the oracle's row-by-row gradients under
    the derived gradient bound (test infrastructure)."""
    import torch
    import oracle
    from exact_attention_forward_04_gb300.inputs import WORKLOADS, make_qkv, make_workload
    from tests.parity import grad_compare, grad_row_term_scales
    torch.set_num_threads(os.cpu_count() or 1)
    peak = peaks["bf16_tflops"]
    sustained = peaks.get("bf16_tflops_sustained", peak)
    sh = stream.cuda_stream
    out = {}
    for w in WORKLOADS:
        if w.N * w.N * w.B * w.H < 1e6:
            continue
        q, k, v = make_workload(w)
        g = make_qkv(w.B, w.H, w.N, w.d, seed=w.seed + 100)[0]
        qd, kd, vd, gd = (t.to(dev) for t in (q, k, v, g))
        o = torch.empty_like(qd)
        lse = torch.empty(w.B, w.H, w.N, dtype=torch.float32, device=dev)
        dq, dk, dv = torch.empty_like(qd), torch.empty_like(qd), torch.empty_like(qd)
        ws_bytes = lib.fa_bwd_workspace_size(w.B, w.H, w.N, w.d)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        st = lib.fa_fwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), lse.data_ptr(),
                        w.B, w.H, w.N, w.d, w.scale, int(w.causal), sh)
        if st != 0:
            raise RuntimeError(f"bwd_per_config {w.name}: fa_fwd status {st}")

        def launch():
            st = lib.fa_bwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), lse.data_ptr(),
                            gd.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), w.B, w.H, w.N,
                            w.d, w.scale, int(w.causal), ws.data_ptr(), ws_bytes, sh)
            if st != 0:
                raise RuntimeError(f"fa_bwd: status {st}")

        _time_launches(launch, stream, flush, 3)
        times = _time_launches(launch, stream, flush, max(5, min(a.steps, 20)))
        st = lib.fa_check_errors(sh)
        if st != 0:
            raise RuntimeError(f"bwd_per_config {w.name}: status {st}")
        mean_ms = sum(times) / len(times)
        tf = 2.5 * w.flops / (mean_ms * 1e-3) / 1e12
        ent = {"B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal,
               "kernel_ms_mean": mean_ms, "kernel_ms_median": statistics.median(times),
               "tflops": tf, "frac_of_bf16_peak": tf / peak, "frac_of_sustained": tf / sustained,
               "traffic_bytes": _traffic("bwd:" + w.name)}
        # parity: dQ rows and dK, dV rows (tile edges, ends, middle) of the
        # first and the last head
        BH = w.B * w.H
        rows = sorted(i for i in {0, 1, 127, 128, w.N // 2, w.N - 2, w.N - 1} if 0 <= i < w.N)
        picks = [(hh // w.H, hh % w.H, i) for hh in sorted({0, BH - 1}) for i in rows]
        oc, lc = o.cpu(), lse.cpu()
        ref = oracle.attention_backward_rows(q, k, v, oc, lc, g, w.scale, w.causal, picks, picks)
        A = grad_row_term_scales(q, k, v, oc, lc, g, w.scale, w.causal, picks, picks)
        idx = torch.tensor(picks)
        par = {}
        for got, r, sc, nm in zip((dq, dk, dv), ref, A, ("dQ", "dK", "dV")):
            res = grad_compare(got.cpu()[idx[:, 0], idx[:, 1], idx[:, 2]], r, sc)
            par[nm] = {key: res[key] for key in ("max_over_bound", "max_rel", "ok")}
        par["ok"] = all(par[nm]["ok"] for nm in ("dQ", "dK", "dV"))
        par["sample"] = f"{len(picks)} rows of each gradient, 2 of {BH} heads"
        ent["parity"] = par
        out[w.name] = ent
        del qd, kd, vd, gd, o, lse, dq, dk, dv, ws
        torch.cuda.empty_cache()
    return out


def _fp8_per_config(a, lib, dev, stream, flush, peaks):
    """The 8-bit forward (fa_fwd_e4m3) on every named workload but the
    128-token one: E4M3 codes made once by fa_quantize_qkv_e4m3 (untimed),
    the forward timed like per_config, its TFLOPS against twice the bf16
    peak and against the bf16 kernel (fa_fwd) timed right before it on the
    same inputs with as many launches (so that both see the same clocks and
    power state; the headline's long run is power-capped), each checked
    as the --fp8 leg does (test infrastructure): head 0's codes bit for bit
    against the oracle's quantisation, and O and L of 64 of its rows against
    the oracle's attention of the dequantised codes (O within the 8-bit
    bound, L within 1e-3)."""
    import torch
    import oracle
    import exact_attention_forward_04_gb300 as fa
    from exact_attention_forward_04_gb300.inputs import WORKLOADS, make_workload
    from tests.parity import L_TOL, fp8_o_bound
    torch.set_num_threads(os.cpu_count() or 1)
    peak = 2.0 * peaks["bf16_tflops"]
    sustained = 2.0 * peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
    sh = stream.cuda_stream
    out = {}
    for w in WORKLOADS:
        if w.N * w.N * w.B * w.H < 1e6:
            continue
        q, k, v = make_workload(w)
        qd, kd, vd = (t.to(dev) for t in (q, k, v))
        with torch.cuda.stream(stream):
            q8, k8, vt8, dsq, dsk, dsv = fa.quantize_qkv_e4m3(qd, kd, vd, stream=stream)
            o = torch.empty(w.B, w.H, w.N, w.d, dtype=torch.bfloat16, device=dev)
            lse = torch.empty(w.B, w.H, w.N, dtype=torch.float32, device=dev)
        n_timed = max(5, min(a.steps, 20))

        def launch_bf16():
            st = lib.fa_fwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), lse.data_ptr(),
                            w.B, w.H, w.N, w.d, w.scale, int(w.causal), sh)
            if st != 0:
                raise RuntimeError(f"fa_fwd: status {st}")

        _time_launches(launch_bf16, stream, flush, 3)
        t16 = _time_launches(launch_bf16, stream, flush, n_timed)
        tf16 = w.flops / (sum(t16) / len(t16) * 1e-3) / 1e12

        def launch():
            st = lib.fa_fwd_e4m3(q8.data_ptr(), k8.data_ptr(), vt8.data_ptr(), dsq.data_ptr(),
                                 dsk.data_ptr(), dsv.data_ptr(), o.data_ptr(), lse.data_ptr(), w.B,
                                 w.H, w.N, w.d, w.scale, int(w.causal), sh)
            if st != 0:
                raise RuntimeError(f"fa_fwd_e4m3: status {st}")

        _time_launches(launch, stream, flush, 3)
        times = _time_launches(launch, stream, flush, n_timed)
        st = lib.fa_check_errors(sh)
        if st != 0:
            raise RuntimeError(f"fp8_per_config {w.name}: status {st}")
        mean_ms = sum(times) / len(times)
        tf = w.flops / (mean_ms * 1e-3) / 1e12
        ent = {"B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal,
               "kernel_ms_mean": mean_ms, "kernel_ms_median": statistics.median(times),
               "tflops": tf, "frac_of_fp8_peak": tf / peak, "frac_of_sustained": tf / sustained,
               "peak_source": "2 x bf16_tflops (nominal FP8/BF16 ratio 4.5/2.25)",
               "traffic_bytes": _traffic("e4m3:" + w.name),
               "bf16_kernel_tflops": tf16, "vs_bf16_kernel": tf / tf16}
        sl = (slice(0, 1), slice(0, 1))
        rows = torch.arange(0, w.N, max(1, w.N // 64))
        refs = [oracle.quantize_e4m3(t[sl]) for t in (q, k, v)]
        codes_ok = bool(torch.equal(q8.cpu()[sl], refs[0][0]) and torch.equal(k8.cpu()[sl], refs[1][0])
                        and torch.equal(vt8.cpu()[sl],
                                        oracle.transpose_keys_last(refs[2][0], vt8.shape[-1])))
        deq = [oracle.dequantize_e4m3(c, s_) for c, s_ in refs]
        if w.causal:
            per_row = [oracle.attention_ref(deq[0][:, :, r:r + 1], deq[1][:, :, :r + 1],
                                            deq[2][:, :, :r + 1], w.scale) for r in rows.tolist()]
            O_ref = torch.cat([x[0] for x in per_row], 2)
            L_ref = torch.cat([x[1] for x in per_row], 2)
        else:
            O_ref, L_ref = oracle.attention_ref(deq[0][:, :, rows], deq[1], deq[2], w.scale)
        bound = fp8_o_bound(deq[0], deq[1], deq[2], O_ref, w.scale, w.causal, rows)
        o_got = o.cpu()[sl][:, :, rows].double()
        l_got = lse.cpu()[sl][:, :, rows].double()
        r_o = ((o_got - O_ref).abs() / bound).max().item()
        r_l = (l_got - L_ref).abs().max().item()
        ent["parity"] = {"codes_bit_exact": codes_ok, "max_dO_over_bound": r_o, "max_dL": r_l,
                         "ok": codes_ok and r_o <= 1.0 and r_l <= L_TOL,
                         "sample": f"codes of head 0; O and L of {len(rows)} of its rows"}
        out[w.name] = ent
        del qd, kd, vd, q8, k8, vt8, dsq, dsk, dsv, o, lse
        torch.cuda.empty_cache()
    return out


# ----------------------------------------------------------------- oracle arm

def _oracle_sample(w, q, k, v, budget_s, max_heads=None):
    """Run the float64 oracle head by head on the workload until the time
    budget is spent; returns (metric flops done, seconds, heads)."""
    import torch
    import oracle
    torch.set_num_threads(os.cpu_count() or 1)
    per_head = w.flops / (w.B * w.H)
    done, t0, heads = 0, time.perf_counter(), 0
    for b in range(w.B):
        for h in range(w.H):
            oracle.attention_ref(q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1],
                                 v[b:b + 1, h:h + 1], w.scale, w.causal)
            heads += 1
            done += per_head
            el = time.perf_counter() - t0
            if el >= budget_s or (max_heads and heads >= max_heads):
                return done, el, heads
    return done, time.perf_counter() - t0, heads


def _oracle_rows(w, q, k, v, step, n_rows):
    """One oracle step on a bounded sample: n_rows consecutive query rows of
    head (step mod B*H), every key they see.  Returns (metric flops, s)."""
    import oracle
    bh = step % (w.B * w.H)
    b, h = divmod(bh, w.H)
    r0 = (step * 7919 * n_rows) % max(1, w.N - n_rows + 1)
    picks = [(b, h, i) for i in range(r0, r0 + n_rows)]
    t0 = time.perf_counter()
    oracle.attention_rows(q, k, v, w.scale, w.causal, picks)
    el = time.perf_counter() - t0
    # metric flops of these rows: 4*d per visible (query, key) pair, with the
    # causal workload counted as half the square like the metric itself
    per_row = w.flops / (w.B * w.H * w.N)
    return per_row * n_rows, el


def run_reference(a, w):
    import torch
    world, rank, _ = _dist_env()
    if rank != 0:
        return 0
    torch.set_num_threads(os.cpu_count() or 1)
    from exact_attention_forward_04_gb300.inputs import make_workload
    q, k, v = make_workload(w)
    # size each step so the whole run stays within about a minute of CPU time
    budget = max(10.0, min(60.0, a.cpu_seconds * 5))
    per_step = budget / max(1, a.steps + a.warmup)
    _, t1 = _oracle_rows(w, q, k, v, 0, 64)
    n_rows = int(max(1, min(w.N, 64 * per_step / max(t1, 1e-6))))
    for i in range(a.warmup):
        _oracle_rows(w, q, k, v, i, n_rows)
    flops = secs = 0.0
    for i in range(a.steps):
        f, s = _oracle_rows(w, q, k, v, a.warmup + i, n_rows)
        flops += f
        secs += s
    val = flops / secs / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOPS",
        "n_gpus": world, "steps": a.steps, "warmup": a.warmup,
        "ms_per_step": secs / a.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                   "causal": w.causal,
                   "sample": f"{n_rows} consecutive query rows of one head per step "
                             "(all keys they see), float64 oracle"},
        "cpu_baseline": {"value": val, "unit": "TFLOPS", "cores": os.cpu_count(),
                         "kind": "oracle",
                         "sample": f"{a.steps} steps x {n_rows} rows of {w.describe()}"},
        "e2e": {"value": val, "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ------------------------------------------------------------------- our arm

def replica_throughput(mean_ms, flops_per_rank, world, device):
    """Whole-job throughput of independent replicas: every rank ran the same
    workload; the job is as slow as its slowest rank.  Returns (max mean
    launch time over ranks in ms, total TFLOPS of all ranks).  Uses the
    default process group when world > 1 (NCCL on GPUs, gloo in tests)."""
    import torch
    if world > 1:
        import torch.distributed as dist
        tt = torch.tensor([float(mean_ms)], dtype=torch.float64, device=device)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        mean_ms = tt.item()
    return mean_ms, flops_per_rank * world / (mean_ms * 1e-3) / 1e12


def run_ours(a, w):
    import torch
    world, rank, local = _dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)

    import exact_attention_forward_04_gb300 as fa
    from exact_attention_forward_04_gb300 import _build
    from exact_attention_forward_04_gb300.inputs import make_workload
    if rank == 0 or world == 1:
        _build.build()
    if world > 1:
        dist.barrier()
    lib = fa.load_library()

    q, k, v = make_workload(w)
    qd, kd, vd = (t.to(dev) for t in (q, k, v))
    o = torch.empty_like(qd)
    lse = torch.empty(w.B, w.H, w.N, dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    sh = stream.cuda_stream
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    split = a.splitkv >= 0
    n_splits = None
    if split:
        n_splits = a.splitkv or fa.splitkv_num_splits(w.B, w.H, w.N, w.causal)
        ws_bytes = fa.splitkv_workspace_size(w.B, w.H, w.N, w.d, n_splits) if n_splits > 1 else 0
        ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)

    def launch_plain():
        st = lib.fa_fwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(),
                        lse.data_ptr(), w.B, w.H, w.N, w.d, w.scale, int(w.causal), sh)
        if st != 0:
            raise fa.FAError(st, "fa_fwd")

    def launch_split():
        st = lib.fa_fwd_splitkv(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(),
                                lse.data_ptr(), w.B, w.H, w.N, w.d, w.scale, int(w.causal),
                                n_splits, ws.data_ptr(), ws_bytes, sh)
        if st != 0:
            raise fa.FAError(st, "fa_fwd_splitkv")

    launch = launch_split if split else launch_plain

    with torch.cuda.stream(stream):
        for _ in range(a.warmup):
            flush.zero_()
            launch()
    stream.synchronize()
    st = lib.fa_check_errors(sh)
    if st != 0:
        raise fa.FAError(st, "warmup")

    # outputs of the warm-up launches, for the oracle's spot check in the
    # CPU-baseline leg below
    picks = [(0, 0, 0), (w.B - 1, w.H - 1, w.N - 1), (w.B // 2, w.H // 2, w.N // 2)]
    idx = torch.tensor(picks)
    o_s = o.cpu()[idx[:, 0], idx[:, 1], idx[:, 2]].double()
    l_s = lse.cpu()[idx[:, 0], idx[:, 1], idx[:, 2]].double()
    spot = None

    sampler = ClockSampler(dev.index)
    sampler.start()
    time.sleep(0.3)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(a.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(a.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t0 = time.time()
    region0 = torch.cuda.Event(enable_timing=True)
    region1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        region0.record(stream)
        for i in range(a.steps):
            flush.zero_()
            starts[i].record(stream)
            launch()
            ends[i].record(stream)
        region1.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    t1 = time.time()
    clocks = sampler.stop(t0, t1)
    st = lib.fa_check_errors(sh)
    if st != 0:
        raise fa.FAError(st, "timed region")
    times = [s.elapsed_time(e) for s, e in zip(starts, ends)]  # ms
    mean_ms = sum(times) / len(times)
    plain_ms = None
    if split:  # the one-pass kernel on the same workload, for context (not the value)
        n_plain = max(5, min(a.steps, 200))
        ps = [torch.cuda.Event(enable_timing=True) for _ in range(n_plain)]
        pe = [torch.cuda.Event(enable_timing=True) for _ in range(n_plain)]
        with torch.cuda.stream(stream):
            for i in range(n_plain):
                flush.zero_()
                ps[i].record(stream)
                launch_plain()
                pe[i].record(stream)
        torch.cuda.synchronize(dev)
        plain_ms = sum(x.elapsed_time(y) for x, y in zip(ps, pe)) / n_plain
    mean_ms, value = replica_throughput(mean_ms, w.flops, world, dev)
    peaks, peak_kind = _peaks()
    peak = peaks["bf16_tflops"]
    achieved = w.flops / (mean_ms * 1e-3) / 1e12

    # ---- end to end through the host entry point (pinned host buffers)
    e2e = None
    if not a.no_e2e and split:
        # through the public Python API: pinned host -> device copies, the
        # split forward, device -> host copies, all on one stream
        qh, kh, vh = (t.pin_memory() for t in (q, k, v))
        oh = torch.empty(w.B, w.H, w.N, w.d, dtype=torch.bfloat16, pin_memory=True)
        lh = torch.empty(w.B, w.H, w.N, dtype=torch.float32, pin_memory=True)

        def e2e_step():
            qd.copy_(qh, non_blocking=True)
            kd.copy_(kh, non_blocking=True)
            vd.copy_(vh, non_blocking=True)
            oo, ll = fa.forward_splitkv(qd, kd, vd, scale=w.scale, causal=w.causal,
                                        num_splits=n_splits, workspace=ws, stream=stream)
            oh.copy_(oo, non_blocking=True)
            lh.copy_(ll, non_blocking=True)

        with torch.cuda.stream(stream):
            for _ in range(max(3, a.warmup)):
                e2e_step()
        stream.synchronize()
        n_e2e = max(5, min(a.steps, 20))
        es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            es.record(stream)
            for _ in range(n_e2e):
                e2e_step()
            ee.record(stream)
        stream.synchronize()
        st = lib.fa_check_errors(sh)
        if st != 0:
            raise fa.FAError(st, "e2e")
        e2e_ms = es.elapsed_time(ee) / n_e2e
        nb = w.B * w.H * w.N * w.d * 2
        e2e = {"value": w.flops * world / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOPS",
               "ms_per_step": e2e_ms, "h2d_bytes_per_step": 3 * nb,
               "d2h_bytes_per_step": nb + w.B * w.H * w.N * 4,
               "steps": n_e2e, "path": "forward_splitkv (pinned host -> device -> host)"}
    elif not a.no_e2e:
        qh, kh, vh = (t.pin_memory() for t in (q, k, v))
        oh = torch.empty(w.B, w.H, w.N, w.d, dtype=torch.bfloat16, pin_memory=True)
        lh = torch.empty(w.B, w.H, w.N, dtype=torch.float32, pin_memory=True)
        stage = (torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd),
                 torch.empty_like(qd), torch.empty_like(lse))

        def e2e_step():
            stt = lib.fa_fwd_host(qh.data_ptr(), kh.data_ptr(), vh.data_ptr(), oh.data_ptr(),
                                  lh.data_ptr(), *(t.data_ptr() for t in stage),
                                  w.B, w.H, w.N, w.d, w.scale, int(w.causal), sh)
            if stt != 0:
                raise fa.FAError(stt, "fa_fwd_host")

        with torch.cuda.stream(stream):
            for _ in range(max(3, a.warmup)):
                e2e_step()
        stream.synchronize()
        n_e2e = max(5, min(a.steps, 20))
        es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            es.record(stream)
            for _ in range(n_e2e):
                e2e_step()
            ee.record(stream)
        stream.synchronize()
        st = lib.fa_check_errors(sh)
        if st != 0:
            raise fa.FAError(st, "e2e")
        e2e_ms = es.elapsed_time(ee) / n_e2e
        nb = w.B * w.H * w.N * w.d * 2
        e2e = {"value": w.flops * world / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOPS",
               "ms_per_step": e2e_ms, "h2d_bytes_per_step": 3 * nb,
               "d2h_bytes_per_step": nb + w.B * w.H * w.N * 4,
               "steps": n_e2e, "path": "fa_fwd_host (pinned host -> device -> host)"}

    per_config = bwd_per_config = fp8_per_config = None
    if world == 1 and not split and not a.no_per_config:
        per_config = _per_config(a, lib, dev, stream, flush, peaks,
                                 main={"name": w.name, "times": times})
        bwd_per_config = _bwd_per_config(a, lib, dev, stream, flush, peaks)
        fp8_per_config = _fp8_per_config(a, lib, dev, stream, flush, peaks)

    cpu = None
    if rank == 0 and not a.no_cpu_baseline:
        # the oracle leg: a parity spot check on sampled rows, then the timing
        import oracle
        O_ref, L_ref = oracle.attention_rows(q, k, v, w.scale, w.causal, picks)
        spot = {"max_dO": (o_s - O_ref).abs().max().item(),
                "max_dL": (l_s - L_ref).abs().max().item()}
        f, s, heads = _oracle_sample(w, q, k, v, a.cpu_seconds)
        cpu = {"value": f / s / 1e12, "unit": "TFLOPS", "cores": os.cpu_count(),
               "kind": "oracle",
               "sample": f"{heads} of {w.B * w.H} heads of {w.describe()}, "
                         f"float64, {s:.1f} s"}

    if rank == 0:
        traffic = _traffic(("split:" if split and n_splits > 1 else "") + w.name)
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world,
            "steps": a.steps, "warmup": a.warmup, "ms_per_step": mean_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                       "causal": w.causal, "scale": w.scale,
                       "l2": "flushed between timed iterations (256 MiB write)",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "pct_of_peak": 100.0 * achieved / peak,
            "kernel_ms": {"mean": mean_ms, "median": statistics.median(times),
                          "min": min(times), "max": max(times)},
            "clocks": clocks,
            "e2e": e2e,
            "gpu_launches": a.steps * (2 if split and n_splits > 1 else 1),
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak,
                         "unit": "TFLOP/s", "frac": achieved / peak,
                         "peak_source": f"bf16_tflops ({peak_kind})",
                         "traffic": traffic,
                         # a timed region of seconds runs under the power cap: the
                         # measured sustained figure is the matching denominator
                         "timed_s": mean_ms * a.steps * 1e-3,
                         "frac_of_sustained": achieved / peaks.get("bf16_tflops_sustained", peak)},
            "mufu": _mufu(w, mean_ms, peaks),
            "cpu_baseline": cpu,
            "spot_check": spot,
        }
        if per_config is not None:
            line["per_config"] = per_config
        if bwd_per_config is not None:
            line["bwd_per_config"] = bwd_per_config
        if fp8_per_config is not None:
            line["fp8_per_config"] = fp8_per_config
        if split:
            line["config"]["path"] = "fa_fwd_splitkv"
            line["config"]["num_splits"] = n_splits
            line["roofline"]["note"] = ("per step: the split pair kernel and the merge kernel; "
                                        "achieved = metric FLOPs / step time")
            line["one_pass_kernel_ms"] = plain_ms
            line["speedup_vs_one_pass"] = plain_ms / mean_ms
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_bwd(a, w):
    """One step = one backward pass over the workload (the forward's O and L
    are computed once, untimed)."""
    import torch
    import exact_attention_forward_04_gb300 as fa
    from exact_attention_forward_04_gb300 import _build
    from exact_attention_forward_04_gb300.inputs import make_qkv, make_workload
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    _build.build()
    lib = fa.load_library()
    q, k, v = make_workload(w)
    g = make_qkv(w.B, w.H, w.N, w.d, seed=w.seed + 100)[0]
    qd, kd, vd, gd = (t.to(dev) for t in (q, k, v, g))
    o, lse = fa.forward(qd, kd, vd, scale=w.scale, causal=w.causal)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    ws_bytes = fa.bwd_workspace_size(w.B, w.H, w.N, w.d)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)
    sh = stream.cuda_stream
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    def launch():
        st = lib.fa_bwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), lse.data_ptr(),
                        gd.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), w.B, w.H, w.N,
                        w.d, w.scale, int(w.causal), ws.data_ptr(), ws_bytes, sh)
        if st != 0:
            raise fa.FAError(st, "fa_bwd")

    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        for _ in range(a.warmup):
            flush.zero_()
            launch()
    stream.synchronize()
    st = lib.fa_check_errors(sh)
    if st != 0:
        raise fa.FAError(st, "warmup")

    # outputs of the warm-up launches, for the oracle's spot check in the
    # CPU-baseline leg below
    sl = (slice(0, 1), slice(0, 1))
    oc, lc = o.cpu(), lse.cpu()
    grads_w = [t.cpu()[sl].double() for t in (dq, dk, dv)]
    spot = None

    sampler = ClockSampler(dev.index)
    sampler.start()
    time.sleep(0.3)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(a.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(a.steps)]
    torch.cuda.synchronize(dev)
    t0 = time.time()
    with torch.cuda.stream(stream):
        for i in range(a.steps):
            flush.zero_()
            starts[i].record(stream)
            launch()
            ends[i].record(stream)
    torch.cuda.synchronize(dev)
    t1 = time.time()
    clocks = sampler.stop(t0, t1)
    st = lib.fa_check_errors(sh)
    if st != 0:
        raise fa.FAError(st, "timed region")
    times = [x.elapsed_time(y) for x, y in zip(starts, ends)]
    mean_ms = sum(times) / len(times)
    flops = 2.5 * w.flops
    achieved = flops / (mean_ms * 1e-3) / 1e12
    peaks, peak_kind = _peaks()
    peak = peaks["bf16_tflops"]

    e2e = None
    if not a.no_e2e:
        host = [t.pin_memory() for t in (q, k, v, oc, lc, g)]
        dev_in = (qd, kd, vd, o, lse, gd)
        outs_h = [torch.empty(w.B, w.H, w.N, w.d, dtype=torch.bfloat16, pin_memory=True)
                  for _ in range(3)]

        def e2e_step():
            for d_, h_ in zip(dev_in, host):
                d_.copy_(h_, non_blocking=True)
            r = fa.backward(qd, kd, vd, o, lse, gd, scale=w.scale, causal=w.causal,
                            workspace=ws, stream=stream)
            for h_, d_ in zip(outs_h, r):
                h_.copy_(d_, non_blocking=True)

        with torch.cuda.stream(stream):
            for _ in range(3):
                e2e_step()
        stream.synchronize()
        n_e2e = max(5, min(a.steps, 20))
        es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            es.record(stream)
            for _ in range(n_e2e):
                e2e_step()
            ee.record(stream)
        stream.synchronize()
        e2e_ms = es.elapsed_time(ee) / n_e2e
        nb = w.B * w.H * w.N * w.d * 2
        e2e = {"value": flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOPS", "ms_per_step": e2e_ms,
               "h2d_bytes_per_step": 4 * nb + w.B * w.H * w.N * 4, "d2h_bytes_per_step": 3 * nb,
               "steps": n_e2e, "path": "backward (pinned host -> device -> host)"}

    cpu = None
    if not a.no_cpu_baseline:
        # the oracle leg: a parity spot check on one whole head, then the timing
        import oracle
        torch.set_num_threads(os.cpu_count())
        ref = oracle.attention_backward_from_lse(q[sl], k[sl], v[sl], oc[sl], lc[sl], g[sl],
                                                 w.scale, w.causal)
        spot = {}
        for nm, got, r in zip(("dQ", "dK", "dV"), grads_w, ref):
            spot[f"max_d{nm}_rel"] = (got - r).abs().max().item() / max(r.abs().max().item(), 1e-30)
        t_start = time.time()
        heads = 0
        while heads < w.B * w.H:
            b, h = divmod(heads, w.H)
            hs = (slice(b, b + 1), slice(h, h + 1))
            oracle.attention_backward_from_lse(q[hs], k[hs], v[hs], oc[hs], lc[hs], g[hs],
                                               w.scale, w.causal)
            heads += 1
            if time.time() - t_start > a.cpu_seconds:
                break
        secs = time.time() - t_start
        cpu = {"value": flops * heads / (w.B * w.H) / secs / 1e12, "unit": "TFLOPS",
               "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"{heads} of {w.B * w.H} heads of {w.describe()}, float64 backward, "
                         f"{secs:.1f} s"}

    line = {
        "metric": "attention bwd TFLOPS (bf16; 2.5x forward FLOPs) and % of GB300 dense BF16 peak, 1 GPU",
        "value": achieved, "unit": "TFLOPS", "n_gpus": 1, "steps": a.steps, "warmup": a.warmup,
        "ms_per_step": mean_ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "pass": "backward", "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                   "causal": w.causal, "scale": w.scale,
                   "l2": "flushed between timed iterations (256 MiB write)",
                   "parallelism": "single GPU"},
        "pct_of_peak": 100.0 * achieved / peak,
        "kernel_ms": {"mean": mean_ms, "median": statistics.median(times), "min": min(times),
                      "max": max(times)},
        "clocks": clocks, "e2e": e2e, "gpu_launches": 3 * a.steps,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "peak_source": f"bf16_tflops ({peak_kind})",
                     "traffic": _traffic("bwd:" + w.name),
                     "timed_s": mean_ms * a.steps * 1e-3,
                     "frac_of_sustained": achieved / peaks.get("bf16_tflops_sustained", peak),
                     "note": "per step: row statistics, then the dK/dV and dQ walks on two streams "
                             "(traffic: the three kernels summed); achieved = 2.5x forward FLOPs / step time"},
        "cpu_baseline": cpu, "spot_check": spot,
    }
    print(json.dumps(line))
    return 0


def run_fp8(a, w):
    """One step = one 8-bit forward pass over the workload's E4M3 codes."""
    import torch
    import exact_attention_forward_04_gb300 as fa
    from exact_attention_forward_04_gb300 import _build
    from exact_attention_forward_04_gb300.inputs import make_workload
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    _build.build()
    lib = fa.load_library()
    q, k, v = make_workload(w)
    qd, kd, vd = (t.to(dev) for t in (q, k, v))
    stream = torch.cuda.Stream(device=dev)
    sh = stream.cuda_stream
    with torch.cuda.stream(stream):
        q8, k8, vt8, dsq, dsk, dsv = fa.quantize_qkv_e4m3(qd, kd, vd, stream=stream)
        o = torch.empty(w.B, w.H, w.N, w.d, dtype=torch.bfloat16, device=dev)
        lse = torch.empty(w.B, w.H, w.N, dtype=torch.float32, device=dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    def launch():
        st = lib.fa_fwd_e4m3(q8.data_ptr(), k8.data_ptr(), vt8.data_ptr(), dsq.data_ptr(),
                             dsk.data_ptr(), dsv.data_ptr(), o.data_ptr(), lse.data_ptr(), w.B,
                             w.H, w.N, w.d, w.scale, int(w.causal), sh)
        if st != 0:
            raise fa.FAError(st, "fa_fwd_e4m3")

    def quantize_all():
        st = lib.fa_quantize_qkv_e4m3(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), q8.data_ptr(),
                                      k8.data_ptr(), vt8.data_ptr(), dsq.data_ptr(), dsk.data_ptr(),
                                      dsv.data_ptr(), w.B, w.H, w.N, w.d, sh)
        if st != 0:
            raise fa.FAError(st, "fa_quantize_qkv_e4m3")

    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        for _ in range(a.warmup):
            flush.zero_()
            launch()
    stream.synchronize()
    st = lib.fa_check_errors(sh)
    if st != 0:
        raise fa.FAError(st, "warmup")

    # outputs of the warm-up launches (one head), for the oracle's spot check
    # in the CPU-baseline leg below
    sl = (slice(0, 1), slice(0, 1))
    rows = torch.arange(0, w.N, max(1, w.N // 64))
    got_w = [t[sl].cpu() for t in (q8, k8, vt8)] + [o.cpu()[sl][:, :, rows].double(),
                                                    lse.cpu()[sl][:, :, rows].double()]
    spot = None

    sampler = ClockSampler(dev.index)
    sampler.start()
    time.sleep(0.3)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(a.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(a.steps)]
    torch.cuda.synchronize(dev)
    t0 = time.time()
    with torch.cuda.stream(stream):
        for i in range(a.steps):
            flush.zero_()
            starts[i].record(stream)
            launch()
            ends[i].record(stream)
    torch.cuda.synchronize(dev)
    t1 = time.time()
    clocks = sampler.stop(t0, t1)
    st = lib.fa_check_errors(sh)
    if st != 0:
        raise fa.FAError(st, "timed region")
    times = [x.elapsed_time(y) for x, y in zip(starts, ends)]
    mean_ms = sum(times) / len(times)
    achieved = w.flops / (mean_ms * 1e-3) / 1e12
    peaks, peak_kind = _peaks()
    peak = 2.0 * peaks["bf16_tflops"]

    # the quantisation of Q, K and V (fa_quantize_qkv_e4m3: four launches),
    # timed on its own
    qt = []
    with torch.cuda.stream(stream):
        for _ in range(3):
            quantize_all()
        for _ in range(10):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            quantize_all()
            e1.record(stream)
            qt.append((e0, e1))
    stream.synchronize()
    quant_ms = statistics.median(x.elapsed_time(y) for x, y in qt)

    e2e = None
    if not a.no_e2e:
        dev_in = (q8, k8, vt8, dsq, dsk, dsv)
        host = [t.cpu().pin_memory() for t in dev_in]
        o_h = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
        l_h = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)

        def e2e_step():
            for d_, h_ in zip(dev_in, host):
                d_.copy_(h_, non_blocking=True)
            oo, ll = fa.forward_e4m3(q8, k8, vt8, dsq, dsk, dsv, scale=w.scale, causal=w.causal,
                                     stream=stream)
            o_h.copy_(oo, non_blocking=True)
            l_h.copy_(ll, non_blocking=True)

        with torch.cuda.stream(stream):
            for _ in range(3):
                e2e_step()
        stream.synchronize()
        n_e2e = max(5, min(a.steps, 20))
        es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            es.record(stream)
            for _ in range(n_e2e):
                e2e_step()
            ee.record(stream)
        stream.synchronize()
        e2e_ms = es.elapsed_time(ee) / n_e2e
        e2e = {"value": w.flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOPS", "ms_per_step": e2e_ms,
               "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in host),
               "d2h_bytes_per_step": o_h.numel() * 2 + l_h.numel() * 4, "steps": n_e2e,
               "path": "forward_e4m3 (pinned host codes -> device -> host O, L)"}

    cpu = None
    if not a.no_cpu_baseline:
        # the oracle leg: a parity spot check on one head (codes bit-exact, O
        # within the 8-bit bound of the parity tests, L within 1e-3), then the
        # timing
        import oracle
        from tests.parity import fp8_o_bound as _bound
        torch.set_num_threads(os.cpu_count())
        refs = [oracle.quantize_e4m3(t[sl]) for t in (q, k, v)]
        codes_ok = bool(torch.equal(got_w[0], refs[0][0]) and torch.equal(got_w[1], refs[1][0])
                        and torch.equal(got_w[2], oracle.transpose_keys_last(refs[2][0],
                                                                             got_w[2].shape[-1])))
        deq = [oracle.dequantize_e4m3(c, s_) for c, s_ in refs]
        if w.causal:
            per_row = [oracle.attention_ref(deq[0][:, :, r:r + 1], deq[1][:, :, :r + 1],
                                            deq[2][:, :, :r + 1], w.scale) for r in rows.tolist()]
            O_ref = torch.cat([x[0] for x in per_row], 2)
            L_ref = torch.cat([x[1] for x in per_row], 2)
        else:
            O_ref, L_ref = oracle.attention_ref(deq[0][:, :, rows], deq[1], deq[2], w.scale)
        bound = _bound(deq[0], deq[1], deq[2], O_ref, w.scale, w.causal, rows)
        spot = {"codes_bit_exact": codes_ok, "rows": len(rows),
                "max_dO_over_bound": ((got_w[3] - O_ref).abs() / bound).max().item(),
                "max_dL": (got_w[4] - L_ref).abs().max().item()}
        # head by head: the quantisation (untimed, like the GPU's), then the
        # attention of the dequantised codes (timed)
        secs = 0.0
        heads = 0
        while heads < w.B * w.H:
            b, h = divmod(heads, w.H)
            hs = (slice(b, b + 1), slice(h, h + 1))
            (c_q, s_q), (c_k, s_k), (c_v, s_v) = (oracle.quantize_e4m3(t[hs]) for t in (q, k, v))
            t_start = time.time()
            oracle.attention_fp8(c_q, c_k, c_v, s_q, s_k, s_v, w.scale, w.causal)
            secs += time.time() - t_start
            heads += 1
            if secs > a.cpu_seconds:
                break
        cpu = {"value": w.flops * heads / (w.B * w.H) / secs / 1e12, "unit": "TFLOPS",
               "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"{heads} of {w.B * w.H} heads of {w.describe()}, float64 attention "
                         f"of the dequantised codes, {secs:.1f} s"}

    line = {
        "metric": "attention fwd TFLOPS (E4M3 inputs) and % of GB300 dense FP8 peak, 1 GPU",
        "value": achieved, "unit": "TFLOPS", "n_gpus": 1, "steps": a.steps, "warmup": a.warmup,
        "ms_per_step": mean_ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3", "data": "synthetic",
        "config": {"workload": w.name, "pass": "forward, 8-bit", "B": w.B, "H": w.H, "N": w.N,
                   "d": w.d, "causal": w.causal, "scale": w.scale,
                   "l2": "flushed between timed iterations (256 MiB write)",
                   "parallelism": "single GPU"},
        "pct_of_peak": 100.0 * achieved / peak,
        "kernel_ms": {"mean": mean_ms, "median": statistics.median(times), "min": min(times),
                      "max": max(times)},
        "quantize_ms": quant_ms,
        "clocks": clocks, "e2e": e2e, "gpu_launches": a.steps,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak,
                     "peak_source": f"2 x bf16_tflops ({peak_kind}; nominal FP8/BF16 ratio 4.5/2.25)",
                     "traffic": _traffic("e4m3:" + w.name),
                     "timed_s": mean_ms * a.steps * 1e-3,
                     "frac_of_sustained": achieved / (2 * peaks.get("bf16_tflops_sustained", peak / 2))},
        "cpu_baseline": cpu, "spot_check": spot,
    }
    print(json.dumps(line))
    return 0


def run_unfused(a, w):
    """One step = standard attention in three kernels (S = scale Q K^T to
    HBM, softmax to P and L, O = P V) over the workload; the fused forward is
    timed beside it on the same inputs.  HBM-bound: the roofline is the
    measured copy bandwidth over the algorithmic bytes of the three steps."""
    import torch
    import exact_attention_forward_04_gb300 as fa
    from exact_attention_forward_04_gb300 import _build
    from exact_attention_forward_04_gb300.inputs import make_workload
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    _build.build()
    lib = fa.load_library()
    q, k, v = make_workload(w)
    qd, kd, vd = (t.to(dev) for t in (q, k, v))
    o = torch.empty_like(qd)
    lse = torch.empty(w.B, w.H, w.N, dtype=torch.float32, device=dev)
    of, lf = torch.empty_like(qd), torch.empty_like(lse)
    ws_bytes = fa.unfused_workspace_size(w.B, w.H, w.N, w.d)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)
    sh = stream.cuda_stream
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    def launch():
        st = lib.fa_attn_unfused(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(),
                                 lse.data_ptr(), w.B, w.H, w.N, w.d, w.scale, int(w.causal),
                                 ws.data_ptr(), ws_bytes, sh)
        if st != 0:
            raise fa.FAError(st, "fa_attn_unfused")

    def launch_fused():
        st = lib.fa_fwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), of.data_ptr(),
                        lf.data_ptr(), w.B, w.H, w.N, w.d, w.scale, int(w.causal), sh)
        if st != 0:
            raise fa.FAError(st, "fa_fwd")

    _time_launches(launch, stream, flush, a.warmup)
    _time_launches(launch_fused, stream, flush, a.warmup)
    st = lib.fa_check_errors(sh)
    if st != 0:
        raise fa.FAError(st, "warmup")
    sampler = ClockSampler(dev.index)
    sampler.start()
    time.sleep(0.3)
    t0 = time.time()
    times = _time_launches(launch, stream, flush, a.steps)
    t1 = time.time()
    clocks = sampler.stop(t0, t1)
    fused_times = _time_launches(launch_fused, stream, flush, a.steps)
    st = lib.fa_check_errors(sh)
    if st != 0:
        raise fa.FAError(st, "timed region")
    mean_ms = sum(times) / len(times)
    fused_ms = sum(fused_times) / len(fused_times)
    peaks, peak_kind = _peaks()
    tf = w.flops / (mean_ms * 1e-3) / 1e12
    BH, N, d = w.B * w.H, w.N, w.d
    # algorithmic bytes of the three steps, per the kernels' dtypes: Q, K read
    # and S (fp32) written; S read and P (bf16) and L written; P and V read
    # and O written.  Causal: only the lower-triangular halves of S and P.
    nn = N * (N + 1) / 2 if w.causal else N * N
    alg = BH * (2 * N * d * 2 + nn * 4 + nn * 4 + nn * 2 + N * 4 + nn * 2 + N * d * 2 + N * d * 2)
    fused_alg = BH * (8 * N * d + 4 * N)
    gbs = alg / (mean_ms * 1e-3) / 1e9
    traffic = _traffic("unfused:" + w.name)
    fused_traffic = _traffic(w.name)
    spot = _parity_sample(w, q, k, v, o, lse)
    line = {
        "metric": "attention fwd TFLOPS (bf16), standard three-kernel attention with S and P "
                  "in HBM, beside the fused forward, 1 GPU",
        "value": tf, "unit": "TFLOPS", "n_gpus": 1, "steps": a.steps, "warmup": a.warmup,
        "ms_per_step": mean_ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "path": "fa_attn_unfused", "B": w.B, "H": w.H, "N": N,
                   "d": d, "causal": w.causal, "scale": w.scale,
                   "l2": "flushed between timed iterations (256 MiB write)",
                   "parallelism": "single GPU"},
        "kernel_ms": {"mean": mean_ms, "median": statistics.median(times), "min": min(times),
                      "max": max(times)},
        "fused": {"kernel_ms_mean": fused_ms, "tflops": w.flops / (fused_ms * 1e-3) / 1e12,
                  "speedup_over_unfused": mean_ms / fused_ms,
                  "algorithmic_bytes": fused_alg, "traffic_bytes": fused_traffic},
        "clocks": clocks, "gpu_launches": 3 * a.steps,
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / peaks["hbm_gbs"], "peak_source": f"hbm_gbs ({peak_kind})",
                     "traffic": traffic, "algorithmic_bytes": alg,
                     "note": "per step: S GEMM, softmax, P V GEMM; achieved = algorithmic "
                             "bytes of the three steps / step time"},
        "intensity": {
            "unfused_algorithmic_flop_per_byte": w.flops / alg,
            "unfused_measured_flop_per_byte": (w.flops / traffic) if traffic else None,
            "fused_measured_flop_per_byte": (w.flops / fused_traffic) if fused_traffic else None,
            "pages_formula_16bit": 4.0 * N * N * d / (4.0 * N * d * 2 + 2.0 * N * N * 2),
        },
        "spot_check": spot,
    }
    print(json.dumps(line))
    return 0


def main():
    a = _args()
    from exact_attention_forward_04_gb300.inputs import BY_NAME, WORKLOADS
    if a.workload is None:
        if a.splitkv >= 0:
            a.workload = "b1h1n8192d128"
        elif a.unfused or a.bwd or a.fp8:
            a.workload = "b4h16n2048d128"
        else:
            a.workload = DEFAULT_WORKLOAD
    w = BY_NAME.get(a.workload)
    if w is None:
        cands = [x for x in WORKLOADS if x.name.startswith(a.workload)]
        if not cands:
            raise SystemExit(f"unknown workload {a.workload}; have {[x.name for x in WORKLOADS]}")
        w = cands[0]
    if a.impl == "reference":
        return run_reference(a, w)
    if a.bwd:
        return run_bwd(a, w)
    if a.fp8:
        return run_fp8(a, w)
    if a.unfused:
        return run_unfused(a, w)
    return run_ours(a, w)


if __name__ == "__main__":
    sys.exit(main())
