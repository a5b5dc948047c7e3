#!/usr/bin/env python3
"""Benchmark: one training step of the FP8 block-scaled linear layers of a
decoder layer on B300, through the library's C ABI.

A step is one pass of the whole path over one batch: for each linear,
quantize X (1x128 row-wise and 128x1 transposed in one read), quantize W
(128x128 blocks plus the transposed copy), fprop, quantize dY (both
layouts), dgrad, wgrad.  The default workload is one decoder layer's four
linears at 32768 tokens (QKV 2048->3072, O 2048->2048, gate+up
2048->11264, down 5632->2048), synthetic inputs as in
fp8_block_scaled_16_b300/inputs.py.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  `value` is GEMM TFLOP/s of the whole step
(all GEMM FLOPs of all ranks / the slowest rank's step time, quantizers
included in the time).  `--impl reference` times the CPU oracle on a bounded
sample of the same workload instead.  With N > 1 (torchrun) the ranks are
independent replicas (weak scaling): the path has no exchange step.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from fp8_block_scaled_16_b300 import dist as D  # noqa: E402
from fp8_block_scaled_16_b300 import inputs  # noqa: E402

METRIC = "FP8 block-scaled GEMM TFLOPS fprop/dgrad/wgrad, % of B300 FP8 peak; quant GB/s"
UNIT = "TFLOP/s"
DEFAULT_WORKLOAD = "decoder_layer_32768"
SWEEP_WORKLOADS = ("attn_qkv_fprop_8192x3072x2048", "mlp_gate_up_16384x11264x2048", "mlp_down_16384x2048x5632")
FP8_PER_BF16 = 4.5 / 2.25        # nominal dense FP8 : BF16 tensor rate
FALLBACK = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK}, "measured"
    except Exception:
        return dict(FALLBACK), "fallback"


# ------------------------------------------------------------------ clocks

# Samplers run in their own process, so they keep their pace while the
# benchmark's launch loop holds the GIL.  With NVML's Python binding: a child
# interpreter samples every ~2 ms until a line (or EOF) arrives on stdin, then
# prints its samples.  Without it: `nvidia-smi -lms`.
_SAMPLER_SRC = r"""
import select, sys, time
try:
    import pynvml
    pynvml.nvmlInit()
    h = None
    for key in sys.argv[1:]:
        try:
            h = (pynvml.nvmlDeviceGetHandleByUUID(key) if key.startswith("GPU-")
                 else pynvml.nvmlDeviceGetHandleByIndex(int(key)))
            break
        except Exception:
            pass
    if h is None:
        raise RuntimeError("no NVML handle for " + " or ".join(sys.argv[1:]))
    print("ready", pynvml.nvmlDeviceGetMaxClockInfo(h, pynvml.NVML_CLOCK_SM), flush=True)
except Exception as e:
    print("error", repr(e).replace("\n", " "), flush=True)
    sys.exit(0)
out = []
while not select.select([sys.stdin], [], [], 0)[0]:
    out.append("%d %d %d" % (pynvml.nvmlDeviceGetClockInfo(h, pynvml.NVML_CLOCK_SM),
                             pynvml.nvmlDeviceGetMaxClockInfo(h, pynvml.NVML_CLOCK_SM),
                             pynvml.nvmlDeviceGetCurrentClocksEventReasons(h)))
    time.sleep(0.002)
print("\n".join(out), flush=True)
"""


class ClockSampler:
    """Samples the SM clock and the clock-event reasons of one GPU between
    start() and stop(), from a separate process (NVML, else nvidia-smi)."""

    REASONS = {
        "gpu_idle": 0x1, "applications_clocks_setting": 0x2, "sw_power_cap": 0x4, "hw_slowdown": 0x8,
        "sync_boost": 0x10, "sw_thermal_slowdown": 0x20, "hw_thermal_slowdown": 0x40,
        "hw_power_brake_slowdown": 0x80, "display_clock_setting": 0x100,
    }
    SMI_QUERY = "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active"

    def __init__(self, device: torch.device):
        # The device's UUID names the right GPU under CUDA_VISIBLE_DEVICES;
        # its index is the fallback.
        self.keys = []
        try:
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            self.keys.append(uuid if uuid.startswith("GPU-") else "GPU-" + uuid)
        except Exception:
            pass
        self.keys.append(str(device.index if device.index is not None else 0))
        self.samples = []          # (sm MHz, max sm MHz, reasons bitmask)
        self.source = None
        self.error = None
        self._proc = None

    def start(self):
        try:
            import importlib.util

            have_nvml = importlib.util.find_spec("pynvml") is not None
        except Exception:
            have_nvml = False
        try:
            if have_nvml:
                env = dict(os.environ)
                env["PYTHONPATH"] = os.pathsep.join(p for p in sys.path if p)
                self._proc = subprocess.Popen([sys.executable, "-c", _SAMPLER_SRC, *self.keys],
                                              stdin=subprocess.PIPE, stdout=subprocess.PIPE,
                                              stderr=subprocess.STDOUT, text=True, env=env)
                first = self._proc.stdout.readline()
                if first.startswith("ready"):
                    self.source = "nvml"
                    return
                self.error = first.strip()[:200] or "NVML sampler exited"
                self._proc.kill()
                self._proc.wait()
            key = None
            for k in self.keys:          # the first id nvidia-smi accepts
                r = subprocess.run(["nvidia-smi", "-i", k, "--query-gpu=clocks.max.sm", "--format=csv,noheader"],
                                   capture_output=True, text=True, timeout=60)
                if r.returncode == 0:
                    key = k
                    break
            if key is None:
                raise RuntimeError("nvidia-smi accepts none of " + ", ".join(self.keys))
            self._proc = subprocess.Popen(["nvidia-smi", "-i", key, self.SMI_QUERY,
                                           "--format=csv,noheader,nounits", "-lms", "10"],
                                          stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi"
        except Exception as e:
            self.error = ((self.error + "; ") if self.error else "") + repr(e)[:200]
            self._proc = None

    def stop(self):
        if self._proc is not None:
            try:
                if self.source == "nvml":
                    out, _ = self._proc.communicate("stop\n", timeout=30)
                    for line in out.splitlines():
                        f = line.split()
                        if len(f) == 3:
                            self.samples.append((int(f[0]), int(f[1]), int(f[2])))
                else:
                    self._proc.terminate()
                    out, _ = self._proc.communicate(timeout=30)
                    for line in out.splitlines():
                        f = [v.strip() for v in line.split(",")]
                        if len(f) == 3 and f[0].isdigit() and f[1].isdigit():
                            self.samples.append((int(f[0]), int(f[1]), int(f[2], 16)))
            except Exception as e:
                self.error = ((self.error + "; ") if self.error else "") + repr(e)[:200]
                self._proc.kill()
                self._proc.wait()
        seen = 0
        for _, _, r in self.samples:
            seen |= r
        names = sorted(n for n, bit in self.REASONS.items() if seen & bit)
        mhz = [m for m, _, _ in self.samples]
        out = {"sm_mhz": statistics.median(mhz) if mhz else None,
               "sm_max_mhz": max(x for _, x, _ in self.samples) if self.samples else None,
               "reasons": names, "samples": len(mhz), "source": self.source}
        if self.error:
            out["error"] = self.error
        return out


# ------------------------------------------------------------------ our arm

def time_step(launch_lists, steps, per_launch):
    """Runs `steps` steps on the current stream; returns total ms and, if
    per_launch, the ms of every launch (CUDA events between launches)."""
    flat = [l for ll in launch_lists for l in ll]
    st = torch.cuda.current_stream()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    marks = []
    t0.record(st)
    for _ in range(steps):
        if per_launch:
            prev = torch.cuda.Event(enable_timing=True)
            prev.record(st)
            for l in flat:
                l.run()
                ev = torch.cuda.Event(enable_timing=True)
                ev.record(st)
                marks.append((l, prev, ev))
                prev = ev
        else:
            for l in flat:
                l.run()
    t1.record(st)
    torch.cuda.synchronize()
    per = [(l, a.elapsed_time(b)) for l, a, b in marks]
    return t0.elapsed_time(t1), per


class L2Flush:
    """Leaves L2 holding none of the timed launch's data and no dirty lines:
    a 512 MiB read-modify-write (far more than the 126 MB L2), then a 256 MiB
    read whose clean lines replace the dirty ones, so that the timed launch
    does not pay for writing back the flush's own data (measured: 2-4 us on a
    10-30 us quantizer launch)."""

    def __init__(self):
        self.w = torch.zeros(128 << 20, dtype=torch.float32, device="cuda")
        self.r = torch.ones(64 << 20, dtype=torch.float32, device="cuda")
        self.acc = torch.zeros(1, dtype=torch.float32, device="cuda")

    def __call__(self):
        self.w.add_(1)
        torch.sum(self.r, dim=0, keepdim=True, out=self.acc)


def sweep(peaks, fp8_peak):
    """Per-kernel rates on the single-linear workloads (each launch timed
    alone with events, L2 flushed before it, median of 10)."""
    from fp8_block_scaled_16_b300.linear import Fp8LinearStep

    res = {}
    flush = L2Flush()
    for name in SWEEP_WORKLOADS:
        wl = inputs.WORKLOADS[name]
        lin = wl.linears[0]
        d = inputs.make_linear_inputs(wl, device="cuda")[0]
        st = Fp8LinearStep(lin.tokens, lin.out_features, lin.in_features, ops=lin.ops)
        ll = st.launch_list(d["x"], d["w"], d.get("dy"))
        for l in ll:
            l.run()
        torch.cuda.synchronize()
        out = {}
        from fp8_block_scaled_16_b300 import binding as B
        from fp8_block_scaled_16_b300.linear import Launch

        # The forward product with its FP8 1x128 output quantized in the epilogue
        # (no BF16 output): what a following linear would consume.
        yq = torch.empty(lin.tokens, lin.out_features, dtype=torch.uint8, device="cuda")
        sy = torch.empty(lin.out_features // 128, B.padded_tokens(lin.tokens), dtype=torch.float32, device="cuda")
        ll = ll + [Launch("fprop_fp8_out", 2 * lin.tokens * lin.out_features * lin.in_features, "flops",
                          lambda: B.fp8bs_gemm_fprop_quant(st.xq, st.sx, st.wq, st.sw, want_bf16=False, yq=yq,
                                                           sy=sy))]
        if name.startswith("mlp_gate_up"):
            # The gate+up forward with SiLU(gate) * up and the down projection's
            # FP8 input in the epilogue (the weight's rows taken as interleaved
            # gate/up blocks; the timing does not depend on the values).
            I = lin.out_features // 2
            hq = torch.empty(lin.tokens, I, dtype=torch.uint8, device="cuda")
            sh = torch.empty(I // 128, B.padded_tokens(lin.tokens), dtype=torch.float32, device="cuda")
            ll.append(Launch("fprop_swiglu_fp8_out", 2 * lin.tokens * lin.out_features * lin.in_features, "flops",
                             lambda: B.fp8bs_gemm_fprop_swiglu_quant(st.xq, st.sx, st.wq, st.sw, want_bf16=False,
                                                                     hq=hq, sh=sh)))
        for i, l in enumerate(ll):
            times = []
            for _ in range(10):
                flush()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                l.run()
                b.record()
                b.synchronize()
                times.append(a.elapsed_time(b))
            ms = statistics.median(times)
            key = l.op if l.op != "quant_act" else ("quant_x" if i == 0 else "quant_dy")
            if l.unit == "flops":
                tf = l.work / (ms * 1e-3) / 1e12
                out[key] = {"ms": round(ms, 4), "TFLOP/s": round(tf, 1), "frac_fp8_peak": round(tf / fp8_peak, 3)}
            else:
                gbs = l.work / (ms * 1e-3) / 1e9
                out[key] = {"ms": round(ms, 4), "GB/s": round(gbs, 1), "frac_hbm": round(gbs / peaks["hbm_gbs"], 3)}
        res[name] = out
        del st, d, ll, yq, sy
        torch.cuda.empty_cache()
    return res


def e2e_run(wl, steps_data, steps):
    """The step through the public API with host buffers: every step copies
    each linear's X, W, dY in from pinned host memory and its Y, dX, dW back
    out, and the host waits for each step's results.  Three streams pipeline
    the work: a linear's inputs are copied in while the previous linear
    computes and the one before is copied out (PCIe carries both directions
    at once), and the next step's first copies start while this step's last
    outputs are still coming back (the host output buffers alternate between
    steps, so a step's results stay intact until the host has read them).
    Events order every buffer's reuse: a linear's device inputs are
    overwritten only after its previous computation, its device outputs only
    after their previous copy-out."""
    host_in, host_out, dev, h2d, d2h = [], [[], []], [], 0, 0
    outs_dev = []
    for st, d in steps_data:
        hi = {k: v.cpu().pin_memory() for k, v in d.items()}
        host_in.append(hi)
        h2d += sum(v.numel() * v.element_size() for v in hi.values())
        outs = [t for t in (st.y, st.dx, st.dw) if t is not None]
        outs_dev.append(outs)
        for par in (0, 1):
            host_out[par].append([torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs])
        d2h += sum(t.numel() * t.element_size() for t in outs)
        dev.append({k: torch.empty_like(v) for k, v in d.items()})
    s_in, s_run, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    lls = [st.launch_list(dv["x"], dv["w"], dv.get("dy"), stream=s_run) for (st, _), dv in zip(steps_data, dev)]
    n = len(steps_data)
    ev_in = [torch.cuda.Event() for _ in range(n)]
    ev_run = [torch.cuda.Event() for _ in range(n)]
    ev_out = [torch.cuda.Event() for _ in range(n)]
    started = [False] * n

    def issue(k):
        par = k & 1
        for i in range(n):
            with torch.cuda.stream(s_in):
                if started[i]:
                    s_in.wait_event(ev_run[i])        # the previous computation has read the inputs
                for key, h in host_in[i].items():
                    dev[i][key].copy_(h, non_blocking=True)
                ev_in[i].record(s_in)
            s_run.wait_event(ev_in[i])
            if started[i]:
                s_run.wait_event(ev_out[i])           # the previous copy-out has read the outputs
            with torch.cuda.stream(s_run):
                for l in lls[i]:
                    l.run()
                ev_run[i].record(s_run)
            s_out.wait_event(ev_run[i])
            with torch.cuda.stream(s_out):
                for t, h in zip(outs_dev[i], host_out[par][i]):
                    h.copy_(t, non_blocking=True)
                ev_out[i].record(s_out)
            started[i] = True
        done = torch.cuda.Event()
        done.record(s_out)
        return done

    def read(done, k):
        done.synchronize()                            # the host reads step k's results
        return float(host_out[k & 1][-1][-1].view(-1)[0])

    read(issue(0), 0)
    t = time.perf_counter()
    prev = issue(1)
    for k in range(2, steps + 1):
        cur = issue(k)
        read(prev, k - 1)
        prev = cur
    read(prev, steps)
    dt = (time.perf_counter() - t) / steps
    return dt, h2d, d2h


def cpu_sample(lin_data, feats, rows, tokens=128):
    """The oracle (single-threaded C) on a bounded sample of the step: each
    linear restricted to its first `tokens` tokens and first `feats` output
    features (all input features), i.e. X[:tokens], W[:feats],
    dY[:tokens, :feats], run through every step of the path -- both
    quantizations of X and dY, the 128x128 weight quantization, then `rows`
    output rows of fprop, dgrad and wgrad of that sub-problem.  Returns
    (GEMM flops of the sampled rows, seconds), so that flops/seconds is in
    the same unit as the GPU figure (GEMM work over the whole path's time)."""
    import numpy as np

    import oracle

    flops, t = 0, time.perf_counter()
    for lin, d in lin_data:
        K = lin.in_features
        F = min(feats, lin.out_features)
        x = d["x"][:tokens].cpu().contiguous()
        w = d["w"][:F].cpu().contiguous()
        r = np.arange(min(rows, tokens))
        xq, sx = oracle.quant_rowwise_1x128(x)
        wq, _, sw = oracle.quant_weight_128x128(w, want_t=False)
        oracle.gemm_fprop(xq, sx, wq, sw, rows=r)
        flops += 2 * r.size * F * K
        if "dgrad" in lin.ops or "wgrad" in lin.ops:
            dy = d["dy"][:tokens, :F].cpu().contiguous()
        if "dgrad" in lin.ops:
            dyq, sdy = oracle.quant_rowwise_1x128(dy)
            oracle.gemm_dgrad(dyq, sdy, wq, sw, rows=r)
            flops += 2 * r.size * K * F
        if "wgrad" in lin.ops:
            xTq, sxT = oracle.quant_colwise_128x1_T(x)
            dyTq, sdyT = oracle.quant_colwise_128x1_T(dy)
            rw = np.arange(min(rows, F))
            oracle.gemm_wgrad(dyTq, sdyT, xTq, sxT, rows=rw)
            flops += 2 * rw.size * K * tokens
    return flops, time.perf_counter() - t


def cpu_per_config(rows_timed=32, rows_checked=256):
    """The oracle per configuration, single-threaded, inputs drawn by the CPU
    recipe (the parity tests' inputs):
      - quantizers on whole tensors: X both ways (1x128 and 128x1
        transposed) and W (128x128 with W^T), as GB/s of algorithmic bytes;
      - each GEMM on the first `rows_timed` of the `rows_checked` seeded
        output rows the parity tests check (weight gradient: the first
        `rows_timed` output features), then the time of all checked rows
        and of the full GEMM extrapolated from the per-row time (labelled).
    The tiny configuration's forward product is timed on its full output."""
    import numpy as np

    import oracle

    def timed(f):
        t = time.perf_counter()
        r = f()
        return r, time.perf_counter() - t

    res = {}
    t_all = time.perf_counter()
    for name in inputs.CONFIGS:
        wl = inputs.WORKLOADS[name]
        data = inputs.make_linear_inputs(wl, device="cpu")
        per_lin = {}
        for lin, d in zip(wl.linears, data):
            M, K, N = lin.tokens, lin.in_features, lin.out_features
            x, w = d["x"], d["w"]
            out = {}
            (xq, sx), t = timed(lambda: oracle.quant_rowwise_1x128(x))
            out["quant_x_rowwise"] = {"s": round(t, 3), "GB/s": round(M * K * (3 + 4 / 128) / t / 1e9, 3)}
            wq, _, sw = None, None, None
            (wq, _, sw), t = timed(lambda: oracle.quant_weight_128x128(w, want_t=True))
            out["quant_w"] = {"s": round(t, 3), "GB/s": round(N * K * 4.0 / t / 1e9, 3)}
            full = M <= rows_timed * 8 and name.startswith("tiny")
            rows = (np.arange(M) if full else
                    inputs.sample_rows(M, wl.seed + 1000, rows_checked).numpy()[:rows_timed])

            def gemm_entry(op, fn, n_rows_total, cols, kc, nrows):
                (_, sec) = timed(fn)
                per_row = sec / nrows
                e = {"rows_timed": int(nrows), "s_timed": round(sec, 3),
                     "GFLOP/s": round(2 * nrows * cols * kc / sec / 1e9, 3)}
                if nrows < n_rows_total:
                    e["s_256_rows_extrapolated"] = round(per_row * min(rows_checked, n_rows_total), 3)
                    e["s_full_extrapolated"] = round(per_row * n_rows_total, 2)
                out[op] = e

            gemm_entry("fprop", lambda: oracle.gemm_fprop(xq, sx, wq, sw, rows=rows), M, N, K, rows.size)
            if "dgrad" in lin.ops:
                dyq, sdy = oracle.quant_rowwise_1x128(d["dy"][torch.as_tensor(rows)])
                gemm_entry("dgrad", lambda: oracle.gemm_dgrad(dyq, sdy, wq, sw), M, K, N, rows.size)
            if "wgrad" in lin.ops:
                (xTq, sxT), t = timed(lambda: oracle.quant_colwise_128x1_T(x))
                out["quant_x_colwise_T"] = {"s": round(t, 3), "GB/s": round(M * K * (3 + 4 / 128) / t / 1e9, 3)}
                dyTq, sdyT = oracle.quant_colwise_128x1_T(d["dy"][:, :128].contiguous())
                nr = min(rows_timed, 128)
                gemm_entry("wgrad", lambda: oracle.gemm_wgrad(dyTq, sdyT, xTq, sxT, rows=np.arange(nr)),
                           N, K, padded(M), nr)
            per_lin[lin.name] = out
        res[name] = per_lin if len(per_lin) > 1 else next(iter(per_lin.values()))
        del data
    return res, time.perf_counter() - t_all


def padded(m):
    return (m + 127) // 128 * 128


def sample_note(feats, rows, tokens=128, max_features=11264):
    if feats >= max_features:
        which, wpart = "all output and input features", "W"
    else:
        which, wpart = f"its first {feats} output features (all input features)", f"W[:{feats}]"
    return (f"each linear restricted to its first {tokens} tokens and {which}: X and dY quantized both ways, "
            f"{wpart} quantized 128x128, {rows} output rows of fprop, dgrad and wgrad; single-threaded C oracle")


KERNEL_OF_OP = {
    "fprop": "gemm_kernel<SB_SCALAR>", "dgrad": "gemm_kernel<SB_SCALAR>", "wgrad": "gemm_kernel<SB_VECTOR>",
    "quant_act": "quant_tile_kernel<QM_ROW|QM_COLT>", "quant_weight": "quant_tile_kernel<QM_BLOCK>",
}


def summarize_kernels(per):
    """Per kernel function: launches, summed event time, algorithmic work."""
    agg = {}
    for l, ms in per:
        k = KERNEL_OF_OP[l.op]
        a = agg.setdefault(k, {"launches": 0, "ms": 0.0, "work": 0, "unit": l.unit, "ops": set()})
        a["launches"] += 1
        a["ms"] += ms
        a["work"] += l.work
        a["ops"].add(l.op)
    return agg


def kernel_source_hash():
    """Hash of the CUDA sources' code (comments and blank lines removed); a
    stored ncu traffic figure is only used while the kernels it was measured
    on are unchanged."""
    import hashlib
    import re

    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "fp8_block_scaled_16_b300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh")):
            with open(os.path.join(csrc, name), encoding="utf-8") as f:
                text = f.read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            text = re.sub(r"//[^\n]*", "", text)
            code = "\n".join(line.rstrip() for line in text.splitlines() if line.strip())
            h.update(name.encode() + b"\0" + code.encode())
    return h.hexdigest()[:16]


def stored_traffic(kernel, workload):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu
    summary (profiles/traffic.json), or None if absent or stale."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
        e = t["kernels"][kernel]
        if t.get("source_hash") != kernel_source_hash() or t.get("workload") != workload:
            return None
        return float(e["dram_bytes_per_launch"])
    except Exception:
        return None


def bf16_comparison(wl, steps_data, steps=10, warmup=3):
    """The same step's twelve GEMMs in plain BF16 through torch.matmul
    (cuBLAS), no quantization: a comparison for the FP8 path's speed-up, the
    B300 counterpart of the pages' FP8-vs-BF16 training-throughput ratio.
    Not part of the measured path."""
    mats = []
    for (st, d), lin in zip(steps_data, wl.linears):
        x, w, dy = d["x"], d["w"], d.get("dy")
        mats.append(lambda x=x, w=w: torch.matmul(x, w.t()))
        if "dgrad" in lin.ops:
            mats.append(lambda dy=dy, w=w: torch.matmul(dy, w))
        if "wgrad" in lin.ops:
            mats.append(lambda dy=dy, x=x: torch.matmul(dy.t(), x))
    for _ in range(warmup):
        for f in mats:
            f()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        for f in mats:
            f()
    b.record()
    b.synchronize()
    return a.elapsed_time(b) / steps


def run_ours(args):
    from fp8_block_scaled_16_b300 import binding as B
    from fp8_block_scaled_16_b300.linear import Fp8LinearStep

    ranks = D.init_from_env("nccl")
    torch.cuda.set_device(ranks.local_rank)
    device = torch.device("cuda", ranks.local_rank)
    B.load()
    peaks, peak_src = load_peaks()
    fp8_burst = peaks["bf16_tflops"] * FP8_PER_BF16
    fp8_sust = peaks["bf16_tflops_sustained"] * FP8_PER_BF16

    wl = inputs.WORKLOADS[args.workload]
    data = inputs.make_linear_inputs(wl, device="cuda")
    steps_data = []
    for lin, d in zip(wl.linears, data):
        steps_data.append((Fp8LinearStep(lin.tokens, lin.out_features, lin.in_features, ops=lin.ops), d))
    lls = [st.launch_list(d["x"], d["w"], d.get("dy")) for st, d in steps_data]
    flops_step = sum(l.work for ll in lls for l in ll if l.unit == "flops")
    launches_step = sum(len(ll) for ll in lls)
    in_bytes = sum(v.numel() * v.element_size() for _, d in steps_data for v in d.values())

    time_step(lls, args.warmup, per_launch=False)
    assert B.fp8bs_get_device_status() == 0, "device status after warm-up"
    count0 = B.fp8bs_launch_count()
    D.barrier(ranks, device)
    torch.cuda.synchronize()
    clocks = ClockSampler(device)
    clocks.start()
    total_ms, per = time_step(lls, args.steps, per_launch=True)
    clk = clocks.stop()
    torch.cuda.synchronize()
    D.barrier(ranks, device)
    launched = B.fp8bs_launch_count() - count0
    status = B.fp8bs_get_device_status()
    if status != 0:
        raise RuntimeError(f"device status {B.fp8bs_status_string(status)}")

    ms_step = total_ms / args.steps
    ms_max = D.max_over_ranks(ranks, ms_step, device)
    value = flops_step * ranks.world / (ms_max * 1e-3) / 1e12

    # Roofline of the kernel with the largest share of the step: algorithmic
    # work of its launches / their summed event time, over the timed region.
    agg = summarize_kernels(per)
    dom = max(agg, key=lambda k: agg[k]["ms"])
    a = agg[dom]
    per_launch_ms = a["ms"] / a["launches"]
    long_region = total_ms >= 2000.0
    traffic = stored_traffic(dom, wl.name)
    if a["unit"] == "flops":
        rate = a["work"] / (a["ms"] * 1e-3) / 1e12
        peak = fp8_sust if long_region else fp8_burst
        roof = {"bound": "tensor", "achieved": round(rate, 1), "peak": round(peak, 1), "unit": "TFLOP/s",
                "frac": round(rate / peak, 4), "traffic": traffic, "kernel": dom,
                "ops": sorted(a["ops"]), "launches_per_step": a["launches"] // args.steps,
                "avg_launch_ms": round(per_launch_ms, 4),
                "peak_note": (f"dense FP8 = {'sustained' if long_region else 'burst'} cuBLAS bf16 of measured "
                              f"x {FP8_PER_BF16:g} (nominal FP8:BF16 ratio); {peak_src}")}
    else:
        rate = a["work"] / (a["ms"] * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": round(rate, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(rate / peaks["hbm_gbs"], 4), "traffic": traffic, "kernel": dom,
                "ops": sorted(a["ops"]), "launches_per_step": a["launches"] // args.steps,
                "avg_launch_ms": round(per_launch_ms, 4), "peak_note": f"STREAM-style copy, {peak_src}"}
    breakdown = {}
    for k, s in sorted(agg.items(), key=lambda kv: -kv[1]["ms"]):
        if s["unit"] == "flops":
            r, u, pk = s["work"] / (s["ms"] * 1e-3) / 1e12, "TFLOP/s", fp8_sust if long_region else fp8_burst
        else:
            r, u, pk = s["work"] / (s["ms"] * 1e-3) / 1e9, "GB/s", peaks["hbm_gbs"]
        breakdown[k] = {"ops": sorted(s["ops"]), "launches_per_step": s["launches"] // args.steps,
                        "ms_per_step": round(s["ms"] / args.steps, 4),
                        "share": round(s["ms"] / sum(v["ms"] for v in agg.values()), 4),
                        u: round(r, 1), "frac_of_measured": round(r / pk, 3)}

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": ranks.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp8_e4m3",
        "data": "synthetic",
        "config": {"workload": wl.name, "tokens": wl.linears[0].tokens,
                   "linears": [f"{l.name} {l.in_features}->{l.out_features}" for l in wl.linears],
                   "step": "per linear: quantize X (1x128 + 128x1 transposed, one read), quantize W (128x128 "
                           "+ transposed copy), fprop, quantize dY (both layouts), dgrad, wgrad",
                   "gemm_tflop_per_step": round(flops_step / 1e12, 4),
                   "l2": f"no flush: inputs larger than L2 ({in_bytes / 1e9:.2f} GB of BF16 inputs per step; "
                         f"L2 126 MB)",
                   "inputs": "drawn on the GPU with torch's CUDA generator (distributions as in inputs.py)",
                   "parallelism": f"independent replicas x{ranks.world}" if ranks.world > 1 else "single GPU"},
        "regime": (f"sustained (timed region {total_ms / 1e3:.2f} s >= 2 s: compared with the sustained peak)"
                   if long_region else
                   f"burst (timed region {total_ms / 1e3:.2f} s < 2 s: compared with the burst peak)"),
        "roofline": roof, "breakdown": breakdown, "gpu_launches": launched,
        "gpu_launches_expected": launches_step * args.steps, "clocks": clk,
    }

    if not args.no_e2e:
        e2e_steps = max(1, min(args.steps, 3))
        dt, h2d, d2h = e2e_run(wl, steps_data, e2e_steps)
        dt_max = D.max_over_ranks(ranks, dt, device)
        result["e2e"] = {"value": round(flops_step * ranks.world / dt_max / 1e12, 2), "unit": UNIT,
                         "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                         "ms_per_step": round(dt_max * 1e3, 2), "steps": e2e_steps,
                         "note": "every step copies X, W, dY in from pinned host memory and Y, dX, dW back out "
                                 "around the same library calls; copy-in, compute and copy-out streams pipeline the "
                                 "four linears and the next step's first copies overlap this step's last; host "
                                 "clock, the host waits for and reads each step's results"}
    if ranks.rank == 0 and ranks.world == 1 and not args.no_cpu:
        fl, sec = cpu_sample(list(zip(wl.linears, data)), args.cpu_feats, args.cpu_rows)
        result["cpu_baseline"] = {
            "value": fl / sec / 1e12, "unit": UNIT, "cores": 1, "host_cores": os.cpu_count(), "kind": "oracle",
            "sample": sample_note(args.cpu_feats, args.cpu_rows,
                                  max_features=max(lin.out_features for lin in wl.linears)) + f", {sec:.1f} s"}
        if not args.no_cpu_configs:
            per_cfg, sec_cfg = cpu_per_config()
            result["cpu_baseline"]["per_config"] = per_cfg
            result["cpu_baseline"]["per_config_note"] = (
                f"every configuration, single-threaded oracle, CPU-recipe inputs ({sec_cfg:.0f} s in all): quantizers "
                "on whole tensors (GB/s of algorithmic bytes); GEMMs timed on the first 32 of the 256 seeded rows the "
                "parity tests check (weight gradient: the first 32 output features), with the time of all 256 rows "
                "and of the full GEMM extrapolated from the per-row time; the tiny configuration's forward product in "
                "full")
    if not args.no_grouped:
        from fp8_block_scaled_16_b300.linear import grouped_launch_list

        gl = grouped_launch_list([(st, d["x"], d["w"], d.get("dy")) for st, d in steps_data])
        time_step([gl], args.warmup, per_launch=False)
        g_ms, _ = time_step([gl], args.steps, per_launch=False)
        g_ms = D.max_over_ranks(ranks, g_ms / args.steps, device)
        assert B.fp8bs_get_device_status() == 0, "device status after the grouped step"
        result["grouped_step"] = {
            "ms_per_step": round(g_ms, 4), "value": round(flops_step * ranks.world / (g_ms * 1e-3) / 1e12, 2),
            "unit": UNIT, "launches_per_step": len(gl),
            "note": "the same step with each GEMM phase of the four linears in one grouped launch "
                    "(fp8bs_gemm_group: 4 forward, 4 data-gradient, 4 weight-gradient products; each member split "
                    "along K as it would be alone)"}
    if ranks.world == 1 and not args.no_bf16:
        bf_ms = bf16_comparison(wl, steps_data)
        result["bf16_comparison"] = {
            "ms_per_step": round(bf_ms, 4), "TFLOP/s": round(flops_step / (bf_ms * 1e-3) / 1e12, 1),
            "fp8_step_speedup": round(bf_ms / ms_max, 3),
            "note": "the step's twelve GEMMs in BF16 via torch.matmul (cuBLAS), no quantization; comparison only"}
    if ranks.world == 1 and not args.no_sweep:
        result["per_workload"] = sweep(peaks, fp8_burst)
        result["per_workload_note"] = ("each launch timed alone with CUDA events, median of 10; before each, L2 "
                                       "flushed by a 512 MiB write and a 256 MiB read (no data of the launch and "
                                       "no dirty lines left in L2)")
    if ranks.rank == 0:
        print(json.dumps(result), flush=True)
    D.shutdown(ranks)


# ------------------------------------------------------------------ reference arm

def run_reference(args):
    """The oracle as it stands, on the host cores, on bounded samples of the
    same workload (rank 0 only; other ranks exit without work)."""
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    wl = inputs.WORKLOADS[args.workload]
    tokens = 128
    data = []
    for lin in wl.linears:
        # The sample only touches the first 128 tokens: draw just those (same
        # distributions as the workload's recipe, CPU generator).
        sub = inputs.Workload(wl.name, wl.seed, (inputs.Linear(lin.name, tokens, lin.in_features,
                                                               lin.out_features, lin.ops),),
                              wl.x_dist, wl.outliers, wl.outlier_factor)
        data.append((lin, inputs.make_linear_inputs(sub, device="cpu")[0]))
    feats, rows = args.ref_feats, args.ref_rows
    for _ in range(args.warmup):
        cpu_sample(data, feats, rows)
    fl = sec = 0.0
    for _ in range(args.steps):
        f, s = cpu_sample(data, feats, rows)
        fl += f
        sec += s
    value = fl / sec / 1e12
    note = sample_note(feats, rows, max_features=max(lin.out_features for lin in wl.linears))
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 block sums, f32 promotion",
        "data": "synthetic", "config": {"workload": wl.name, "parallelism": "one host thread (rank 0)",
                                        "sample_per_step": note},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": note},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def free_port():
    import socket

    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def launch_ranks(n):
    """`--gpus N` without a rank environment: start N ranks of this same
    command line under torch.distributed.run (one process per GPU, rendezvous
    on 127.0.0.1) and return their exit status."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr=127.0.0.1", f"--master-port={free_port()}", os.path.abspath(__file__), *sys.argv[1:]]
    return subprocess.call(cmd)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--cpu-feats", type=int, default=1 << 20, help="output features per linear in the CPU sample")
    ap.add_argument("--cpu-rows", type=int, default=128)
    ap.add_argument("--ref-feats", type=int, default=1024)
    ap.add_argument("--ref-rows", type=int, default=32)
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-grouped", action="store_true", help="skip the grouped-launch step")
    ap.add_argument("--no-bf16", action="store_true")
    ap.add_argument("--no-cpu-configs", action="store_true", help="skip the per-configuration oracle timing")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.gpus < 1:
        ap.error("--gpus must be >= 1")
    world = os.environ.get("WORLD_SIZE")
    if world is None and args.gpus > 1:
        if args.impl == "ours" and torch.cuda.device_count() < args.gpus:
            sys.exit(f"bench.py: --gpus {args.gpus} needs {args.gpus} visible CUDA devices, "
                     f"found {torch.cuda.device_count()}")
        sys.exit(launch_ranks(args.gpus))
    if world is not None and int(world) != args.gpus:
        ap.error(f"--gpus {args.gpus} does not match WORLD_SIZE={world}")
    print(f"[bench] rank {os.environ.get('RANK', '0')}/{world or 1} ({args.impl} arm)", file=sys.stderr, flush=True)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
