#!/usr/bin/env python
"""FP8 delayed-scaling LayerNormMLP forward+backward throughput on GB300.

One step = ln_mlp_fwd + ln_mlp_bwd through the C ABI over one batch (up to 8
batches drawn once and cycled over the steps):
8192 tokens (32 x 256) of d_model 768, FFN 3072, HYBRID (E4M3 forward, E5M2
gradients), amax_history_len 16, X ~ N(0,1) with 0.1% x50 outliers, dY ~
N(0, 0.01), weights ~ N(0, 0.02), bias 0. FLOPs are the six FP8 GEMMs,
12 * M * D * F per step.

Prints one JSON line (rank 0). --impl reference times the CPU oracle on the
same metric instead (rank 0 only; other ranks exit at once).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "FP8 LayerNormMLP fwd+bwd TFLOP/s (D=768/2048) and % of GB300 FP8 dense peak"
M_TOK, D_MODEL, FFN = 8192, 768, 3072
HIST = 16
FMT = "hybrid"
L2_FLUSH_BYTES = 256 << 20
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_PER_BF16 = 2.0  # nominal dense ratio (4.5 / 2.25 PFLOP/s)


def flops_per_step(m=M_TOK, d=D_MODEL, f=FFN):
    return 12.0 * m * d * f


FORMAT_TEXT = {"hybrid": "HYBRID (E4M3 fwd / E5M2 grads)", "e4m3": "E4M3 everywhere", "e5m2": "E5M2 everywhere"}
DIST_TEXT = {"outliers": "N(0,1) + 0.1% entries x50", "normal": "N(0,1)", "t3": "Student-t(3)"}


def workload(m=M_TOK, d=D_MODEL, f=FFN, fmt=FMT, hist=HIST, dist="outliers", n_sets=8, inputs="host"):
    src = "seeded host generator" if inputs == "host" else "the device's generator"
    return {"workload": f"LayerNormMLP fwd+bwd, {m} tokens x {d} -> {f} -> {d}, {FORMAT_TEXT[fmt]}, "
                        f"amax_history_len {hist}, {n_sets} pre-drawn X / dY batches cycled over the steps",
            "tokens": m, "d_model": d, "ffn": f, "fp8_format": fmt, "amax_history_len": hist,
            "x_dist": DIST_TEXT[dist], "dy_dist": "N(0, 0.01)", "weights": "N(0, 0.02), bias 0",
            "inputs": f"{n_sets} batches drawn once by the {src}, device-resident, step i uses batch i mod {n_sets}",
            "l2": "flushed (256 MiB write) between timed steps", "parallelism": "replicas (one per GPU)"}


# ----------------------------------------------------------------- helpers
def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            return d, "measured"
        except Exception:
            pass
    return dict(FALLBACK), "fallback"


def _num(d, *keys):
    for k in keys:
        if k in d and isinstance(d[k], (int, float)):
            return float(d[k])
    return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons. The sampler starts
    before the timed region and keeps only the samples taken between mark_start()
    and mark_stop() (by nvidia-smi's own timestamps)."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, tag: str = ""):
        self.idx = gpu_index
        self.proc = None
        # raw samples; LNFP8_CLOCKS_DIR keeps them somewhere lasting (the JSON line has the summary)
        self.path = os.path.join(os.environ.get("LNFP8_CLOCKS_DIR", tempfile.gettempdir()),
                                 f"lnfp8_clocks_rank{gpu_index}{tag}.csv")
        self.t0 = self.t1 = None

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-lms", "50", "-i", str(self.idx)], stdout=self.fh,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            return
        deadline = time.time() + 10.0  # nvidia-smi needs a moment before its first sample
        while time.time() < deadline and self.proc.poll() is None:
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.02)

    def mark_start(self):
        self.t0 = time.time()

    def mark_stop(self):
        self.t1 = time.time()

    @staticmethod
    def _when(ts):
        base, _, frac = ts.partition(".")
        return time.mktime(time.strptime(base, "%Y/%m/%d %H:%M:%S")) + (float("0." + frac) if frac else 0.0)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.1)  # one more sample past the end of the region
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        with open(self.path) as f:
            return self.summarize(f, self.t0, self.t1)

    @classmethod
    def summarize(cls, lines, t0=None, t1=None):
        """Median SM clock, max clock and power, and the throttle reasons seen, over the
        samples taken between t0 and t1 (50 ms of slack on both sides; all when t0 is None)."""
        sm, smax, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            try:
                t = cls._when(f[0])
                if t0 is not None and not (t0 - 0.05 <= t <= (t1 or t) + 0.05):
                    continue
                sm.append(float(f[2]))
                smax.append(float(f[3]))
                pw.append(float(f[4]))
            except ValueError:
                continue
            for n, v in zip(names, f[6:10]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(pw) if pw else None, "reasons": sorted(reasons), "samples": len(sm)}


def gemm_sources_sha1():
    h = hashlib.sha1()
    for f in ("gemm.cu", "gemm_pair.cuh"):
        h.update(open(os.path.join(ROOT, "fp8_delayed_scaling_row_gb300", "csrc", f), "rb").read())
    return h.hexdigest()


def gemm_traffic_from_profile():
    """DRAM bytes of one step's GEMM launches from the committed ncu summary, if
    the GEMM sources are unchanged since it was captured (else None)."""
    p = os.path.join(ROOT, "profiles", "gemm_traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
        if d.get("gemm_sources_sha1") != gemm_sources_sha1():
            return None
        return d.get("dram_bytes_per_step")
    except Exception:
        return None


# ----------------------------------------------------------------- CPU oracle arm
def _oracle_setup(rows, ffn, seed=1234):
    from fp8_delayed_scaling_row_gb300 import synth
    from oracle.delayed_scaling import Recipe as ORecipe, ScalingState
    p = synth.mlp_params(D_MODEL, ffn, seed=seed)
    return p, ORecipe(FMT, HIST), ScalingState(4, HIST), ScalingState(2, HIST)


def _oracle_step(p, rec, fs, bs, rows, step, seed=1234):
    """One oracle step (LayerNormMLP fwd + bwd) on `rows` fresh tokens; returns its seconds."""
    from fp8_delayed_scaling_row_gb300 import synth
    from oracle import modules as om
    x = synth.activations(rows, D_MODEL, dist="outliers", seed=seed, step=step)
    dy = synth.grad(rows, D_MODEL, seed=seed, step=step)
    t0 = time.perf_counter()
    _, ctx, _ = om.ln_mlp_fwd(x, p["gamma"], p["beta"], p["w1"], p["b1"], p["w2"], p["b2"], fs, rec)
    om.ln_mlp_bwd(dy, ctx, bs, rec)
    return time.perf_counter() - t0


def oracle_rate(seconds: float, rows: int, ffn: int = FFN):
    """The oracle as it stands on `rows` tokens x `ffn` FFN columns per step, repeated for
    about `seconds`; returns (TFLOP/s, steps, elapsed)."""
    p, rec, fs, bs = _oracle_setup(rows, ffn)
    el, n = 0.0, 0
    while el < seconds:
        el += _oracle_step(p, rec, fs, bs, rows, n)
        n += 1
    return flops_per_step(rows, D_MODEL, ffn) * n / el / 1e12, n, el


def reference_sample(total_steps: int):
    """(tokens, FFN columns) of one oracle step so that the whole run stays within a few minutes."""
    budget = 150.0 / max(total_steps, 1)
    if budget >= 6.0:
        return 1024, FFN
    if budget >= 1.8:
        return 256, FFN
    if budget >= 0.5:
        return 128, 768
    return 32, 256


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    rows, ffn = reference_sample(args.steps + args.warmup)
    p, rec, fs, bs = _oracle_setup(rows, ffn)
    times = []
    for i in range(args.warmup + args.steps):
        t = _oracle_step(p, rec, fs, bs, rows, i)
        if i >= args.warmup:
            times.append(t)
    el = sum(times)
    val = flops_per_step(rows, D_MODEL, ffn) * len(times) / el / 1e12
    sample = (f"each step: {rows} of the {M_TOK} tokens and {ffn} of the {FFN} FFN columns (LayerNormMLP "
              f"{D_MODEL} -> {ffn} -> {D_MODEL}); numpy oracle, fp64 BLAS matmuls with the library's default "
              f"threads; {args.steps} timed steps after {args.warmup} warm-up")
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / len(times) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (fp8 codes decoded)",
            "data": "synthetic", "config": workload(),
            "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------- GPU arm
def device_draw(torch, g, shape, dist="normal", std=1.0):
    """bf16 tensor on the device: N(0,1) (x50 on 0.1% of entries for "outliers") or
    Student-t(3) = N / sqrt(chi2_3 / 3), times std."""
    z = torch.randn(*shape, generator=g, device=g.device, dtype=torch.float32)
    if dist == "outliers":
        z = torch.where(torch.rand(*shape, generator=g, device=g.device) < 1e-3, z * 50, z)
    elif dist == "t3":
        chi2 = sum(torch.randn(*shape, generator=g, device=g.device, dtype=torch.float32) ** 2 for _ in range(3))
        z = z / torch.sqrt(chi2 / 3.0)
    return (z * std).to(torch.bfloat16)


class MlpRun:
    """Device-resident workload: weights, state, saved tensors, gradient buffers,
    and n_sets input batches drawn once and cycled over the steps (inputs="host":
    the seeded host generator, also kept in pinned-able host arrays for the end-to-end
    leg; "device": the device's generator, for the large sweep points)."""

    def __init__(self, L, torch, dev, m, d, f, fmt, hist, dist, n_sets, seed, inputs="host", params=None):
        from fp8_delayed_scaling_row_gb300 import synth
        import numpy as np

        def bf(bits):
            return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)

        self.L, self.torch, self.m, self.d, self.f = L, torch, m, d, f
        self.p = params if params is not None else {k: bf(v) for k, v in synth.mlp_params(d, f, seed=seed).items()}
        self.rec = L.Recipe(fmt, hist)
        self.fm, self.bm = L.ScalingMeta(4, hist, device=dev), L.ScalingMeta(2, hist, device=dev)
        self.ctx = L.mlp_ctx(m, d, f, device=dev)
        self.grads = L.mlp_grads(m, d, f, device=dev)
        self.y = torch.empty(m, d, dtype=torch.bfloat16, device=dev)
        self.xs_host, self.dys_host = [], []
        if inputs == "host":
            for i in range(n_sets):
                self.xs_host.append(synth.activations(m, d, dist=dist, seed=seed, step=i))
                self.dys_host.append(synth.grad(m, d, seed=seed, step=i))
            self.xs = [bf(x) for x in self.xs_host]
            self.dys = [bf(x) for x in self.dys_host]
        else:
            g = torch.Generator(device=dev)
            g.manual_seed(seed)
            self.xs = [device_draw(torch, g, (m, d), dist) for _ in range(n_sets)]
            self.dys = [device_draw(torch, g, (m, d), "normal", 0.01) for _ in range(n_sets)]
        self.graphs = None

    def step(self, i, x=None, dy=None):
        """One fwd+bwd through the C ABI; replays the captured CUDA graph of this
        input batch when graphs are on (same kernels, no per-launch host cost)."""
        if x is None and self.graphs is not None:
            self.graphs[i % len(self.graphs)].replay()
            return
        self._call(self.xs[i % len(self.xs)] if x is None else x, self.dys[i % len(self.dys)] if dy is None else dy)

    def _call(self, x, dy):
        L, p = self.L, self.p
        L.ln_mlp_fwd(x, p["gamma"], p["beta"], p["w1"], p["b1"], p["w2"], p["b2"], self.fm, self.rec, y=self.y,
                     ctx=self.ctx)
        L.ln_mlp_bwd(dy, x, p["gamma"], self.ctx, self.bm, self.rec, grads=self.grads)

    def capture_one(self, i):
        """One CUDA graph of the step on input batch i, the state restored after capture."""
        torch = self.torch
        sd_f, sd_b = self.fm.state_dict(), self.bm.state_dict()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self._call(self.xs[i], self.dys[i])
        torch.cuda.synchronize()
        self.fm.load_state_dict(sd_f)
        self.bm.load_state_dict(sd_b)
        return g

    def capture(self):
        """Capture one CUDA graph per input batch (the state buffers are shared, so
        replays advance the delayed-scaling state exactly like direct calls)."""
        torch = self.torch
        self.graphs = None
        sd_f, sd_b = self.fm.state_dict(), self.bm.state_dict()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        graphs = []
        with torch.cuda.stream(s):
            for i in range(len(self.xs)):  # warm the stream once before capture
                c0 = self.L.launch_count()
                self._call(self.xs[i], self.dys[i])
                self.launches_per_step = self.L.launch_count() - c0
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        for i in range(len(self.xs)):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self._call(self.xs[i], self.dys[i])
            graphs.append(g)
        torch.cuda.synchronize()
        self.fm.load_state_dict(sd_f)
        self.bm.load_state_dict(sd_b)
        self.graphs = graphs


def stack_flops_per_step(layers, m, d, f):
    """Six GEMMs per module (forward, data and weight gradients): QKV d -> 3d, proj d -> d, MLP d -> f -> d."""
    return layers * 6.0 * m * d * (3 * d + d + 2 * f)


class StackRun:
    """A stack of transformer-block FP8 modules as one training step: per layer
    LayerNormLinear d -> 3d (QKV), Linear d -> d (attention-output projection, fed
    a synthetic attention output) and LayerNormMLP d -> f -> d, forward over the
    layers then backward in reverse, every module with its state update deferred
    and one state-update launch for all layers' sets at the end of the step.

    The forward is chained as a pre-LN block: the MLP's LayerNorm takes the
    residual stream plus the projection's output, the next layer's QKV LayerNorm
    the stream plus the MLP's output, both adds fused into those LayerNorm
    kernels. Device-resident inputs, generated once: the first layer's h ~ N(0,1)
    with 0.1% x50 outliers, each layer's attention output ~ N(0,1), dQKV and dY
    ~ N(0, 0.01) (the backward is not chained: attention is not on this path).
    The whole step is one captured CUDA graph."""

    PARAMS = ("wqkv", "bqkv", "g1", "be1", "wproj", "bproj", "g2", "be2", "w1", "b1", "w2", "b2")

    def __init__(self, L, torch, dev, layers, m, d, f, fmt, hist, seed, host_params=None, host_inputs=None,
                 keep_outputs=False):
        """host_params: None (weights drawn on the device), or per layer a dict of
        bf16 bit patterns (numpy uint16) under the names in PARAMS; host_inputs: None,
        or a dict of bf16 bit patterns h0 [m, d], attn [m, d], dqkv [m, 3d], dy [m, d]
        shared by every layer (the parity tests feed seeded host inputs this way);
        keep_outputs: every layer writes its QKV, projection and MLP outputs to buffers
        of its own (lay["yq"], lay["yp"], lay["ym"]) instead of sharing one set."""
        self.L, self.torch, self.layers, self.m, self.d, self.f = L, torch, layers, m, d, f
        g = torch.Generator(device=dev)
        g.manual_seed(seed)

        def randn(*shape, std=1.0, outliers=False):
            t = torch.randn(*shape, generator=g, device=dev, dtype=torch.float32) * std
            if outliers:
                t = torch.where(torch.rand(*shape, generator=g, device=dev) < 1e-3, t * 50, t)
            return t.to(torch.bfloat16)

        def ones_plus(n):
            return (1 + 0.1 * torch.randn(n, generator=g, device=dev)).to(torch.bfloat16)

        def from_bits(bits):
            import numpy as np
            return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)

        shared = None if host_inputs is None else {k: from_bits(v) for k, v in host_inputs.items()}
        self.rec = L.Recipe(fmt, hist)
        E4, E5 = L.E4M3, L.E5M2
        self.layer = []
        for li in range(layers):
            if host_params is None:
                lay = dict(
                    wqkv=randn(3 * d, d, std=0.02), bqkv=torch.zeros(3 * d, dtype=torch.bfloat16, device=dev),
                    g1=ones_plus(d), be1=randn(d, std=0.1),
                    wproj=randn(d, d, std=0.02), bproj=torch.zeros(d, dtype=torch.bfloat16, device=dev),
                    g2=ones_plus(d), be2=randn(d, std=0.1),
                    w1=randn(f, d, std=0.02), b1=torch.zeros(f, dtype=torch.bfloat16, device=dev),
                    w2=randn(d, f, std=0.02), b2=torch.zeros(d, dtype=torch.bfloat16, device=dev))
            else:
                lay = {k: from_bits(host_params[li][k]) for k in self.PARAMS}
            if shared is None:
                lay.update(attn=randn(m, d), dqkv=randn(m, 3 * d, std=0.01), dy=randn(m, d, std=0.01))
            else:
                lay.update(attn=shared["attn"], dqkv=shared["dqkv"], dy=shared["dy"])
            lay.update(
                fq=L.ScalingMeta(2, hist, device=dev), fp=L.ScalingMeta(2, hist, device=dev),
                fm=L.ScalingMeta(4, hist, device=dev), bq=L.ScalingMeta(1, hist, device=dev),
                bp=L.ScalingMeta(1, hist, device=dev), bm=L.ScalingMeta(2, hist, device=dev),
                cq=L.linear_ctx(m, d, 3 * d, device=dev), cp=L.linear_ctx(m, d, d, ln=False, device=dev),
                cm=L.mlp_ctx(m, d, f, device=dev),
                gq=L.linear_grads(m, d, 3 * d, device=dev), gp=L.linear_grads(m, d, d, ln=False, device=dev),
                gm=L.mlp_grads(m, d, f, device=dev))
            self.layer.append(lay)
        self.h0 = randn(m, d, outliers=True) if shared is None else shared["h0"]
        # the QKV output is not consumed (attention is synthetic); projection and MLP outputs
        # feed the next LayerNorm's fused residual add
        self.yq = torch.empty(m, 3 * d, dtype=torch.bfloat16, device=dev)
        self.yp = torch.empty(m, d, dtype=torch.bfloat16, device=dev)
        self.ym = torch.empty(m, d, dtype=torch.bfloat16, device=dev)
        for i, lay in enumerate(self.layer):
            own = keep_outputs and i < layers - 1  # the last layer writes the shared set
            lay["yq"] = torch.empty_like(self.yq) if own else self.yq
            lay["yp"] = torch.empty_like(self.yp) if own else self.yp
            lay["ym"] = torch.empty_like(self.ym) if own else self.ym
        self.order = ["fq", "fp", "fm", "bq", "bp", "bm"]
        dts = {"fq": [E4] * 2, "fp": [E4] * 2, "fm": [E4] * 4, "bq": [E5], "bp": [E5], "bm": [E5] * 2}
        self.metas = [lay[k] for lay in self.layer for k in self.order]
        self.dtypes = [dts[k] for _ in self.layer for k in self.order]
        self.graphs = None

    def _call(self):
        L, rec = self.L, self.rec
        x, r = self.h0, None  # the stream before the last add, and what is added to it
        for lay in self.layer:
            L.ln_linear_fwd(x, lay["g1"], lay["be1"], lay["wqkv"], lay["bqkv"], lay["fq"], rec, y=lay["yq"],
                            ctx=lay["cq"], defer_update=True, residual=r)
            lay["hq"] = lay["cq"].x_sum if r is not None else x  # this layer's stream (the QKV input)
            L.ln_linear_fwd(lay["attn"], None, None, lay["wproj"], lay["bproj"], lay["fp"], rec, y=lay["yp"],
                            ctx=lay["cp"], defer_update=True)
            L.ln_mlp_fwd(lay["hq"], lay["g2"], lay["be2"], lay["w1"], lay["b1"], lay["w2"], lay["b2"], lay["fm"], rec,
                         y=lay["ym"], ctx=lay["cm"], defer_update=True, residual=lay["yp"])
            x, r = lay["cm"].x_sum, lay["ym"]
        for lay in reversed(self.layer):
            L.ln_mlp_bwd(lay["dy"], lay["cm"].x_sum, lay["g2"], lay["cm"], lay["bm"], rec, grads=lay["gm"],
                         defer_update=True)
            L.ln_linear_bwd(lay["dy"], lay["attn"], None, lay["cp"], lay["bp"], rec, grads=lay["gp"],
                            defer_update=True)
            L.ln_linear_bwd(lay["dqkv"], lay["hq"], lay["g1"], lay["cq"], lay["bq"], rec, grads=lay["gq"],
                            defer_update=True)
        L.amax_history_update_many(self.metas, rec, self.dtypes)

    def step(self, i):
        if self.graphs is not None:
            self.graphs[0].replay()
        else:
            self._call()

    def capture(self, warm=True):
        torch = self.torch
        sds = [m.state_dict() for m in self.metas]
        if warm:  # one direct step on a side stream before the first capture
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                c0 = self.L.launch_count()
                self._call()
                self.launches_per_step = self.L.launch_count() - c0
            torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            self._call()
        torch.cuda.synchronize()
        for m, sd in zip(self.metas, sds):
            m.load_state_dict(sd)
        self.graphs = [gr]


def timed_steps(torch, run, steps, warmup, flush, barrier, clocks=None):
    """W untimed warm-up steps, then K steps each bracketed by CUDA events on the
    launching (current) stream, an L2 flush between them outside the events.
    Returns (device ms summed over the K steps, library kernel launches in them)."""
    for i in range(warmup):
        run.step(i)
    torch.cuda.synchronize()
    barrier()
    if clocks is not None:
        clocks.mark_start()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    n0 = run.L.launch_count()
    for i in range(steps):
        flush.zero_()
        ev[i][0].record()
        run.step(warmup + i)
        ev[i][1].record()
    n1 = run.L.launch_count()
    torch.cuda.synchronize()
    if clocks is not None:
        clocks.mark_stop()
    barrier()
    launches = n1 - n0
    if run.graphs is not None:
        launches = run.launches_per_step * steps  # replays launch the captured kernels
    return sum(a.elapsed_time(b) for a, b in ev), launches


def end_to_end(torch, run, steps, dev, barrier, max_over_ranks, world, graph=True):
    """Steps fed from and drained to pinned host memory through the public API.

    Every step copies its X and dY host->device and its Y and dX device->host inside
    the timed region. The copies run on their own streams and the device buffers
    alternate between two sets, so step i's input copies and step i-1's output
    copies overlap step i-1's and step i's compute (a training loop would stream
    batches the same way). Each set's step is one captured CUDA graph when graphs
    are on."""
    L = run.L
    xh = [torch.from_numpy(b.view("int16")).view(torch.bfloat16).pin_memory() for b in run.xs_host]
    dyh = [torch.from_numpy(b.view("int16")).view(torch.bfloat16).pin_memory() for b in run.dys_host]
    yh = [torch.empty(run.m, run.d, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    dxh = [torch.empty(run.m, run.d, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    xd = [torch.empty(run.m, run.d, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    dyd = [torch.empty_like(xd[0]) for _ in range(2)]
    yd = [run.y, torch.empty_like(run.y)]
    gd = [run.grads, L.mlp_grads(run.m, run.d, run.f, device=dev)]
    comp = torch.cuda.current_stream()
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()

    def call(b):
        L.ln_mlp_fwd(xd[b], run.p["gamma"], run.p["beta"], run.p["w1"], run.p["b1"], run.p["w2"], run.p["b2"], run.fm,
                     run.rec, y=yd[b], ctx=run.ctx)
        L.ln_mlp_bwd(dyd[b], xd[b], run.p["gamma"], run.ctx, run.bm, run.rec, grads=gd[b])

    graphs = None
    if graph:
        sd_f, sd_b = run.fm.state_dict(), run.bm.state_dict()
        s = torch.cuda.Stream()
        s.wait_stream(comp)
        with torch.cuda.stream(s):
            for b in range(2):
                call(b)
        comp.wait_stream(s)
        torch.cuda.synchronize()
        graphs = []
        for b in range(2):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                call(b)
            graphs.append(g)
        torch.cuda.synchronize()
        run.fm.load_state_dict(sd_f)
        run.bm.load_state_dict(sd_b)

    in_ready = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    out_read = [torch.cuda.Event() for _ in range(2)]

    copy_ev = []  # (h2d start, h2d end, d2h start, d2h end) per timed step

    def issue(i, timed=False):
        b = i % 2
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)] if timed else None
        with torch.cuda.stream(h2d):
            h2d.wait_event(done[b])       # step i-2 has finished reading this set's inputs
            if ev:
                ev[0].record(h2d)
            xd[b].copy_(xh[i % len(xh)], non_blocking=True)
            dyd[b].copy_(dyh[i % len(dyh)], non_blocking=True)
            if ev:
                ev[1].record(h2d)
            in_ready[b].record(h2d)
        comp.wait_event(in_ready[b])
        comp.wait_event(out_read[b])      # step i-2's outputs have left this set
        if graphs is not None:
            graphs[b].replay()
        else:
            call(b)
        done[b].record(comp)
        with torch.cuda.stream(d2h):
            d2h.wait_event(done[b])
            if ev:
                ev[2].record(d2h)
            yh[b].copy_(yd[b], non_blocking=True)
            dxh[b].copy_(gd[b].dx, non_blocking=True)
            if ev:
                ev[3].record(d2h)
            out_read[b].record(d2h)
        if ev:
            copy_ev.append(ev)

    for b in range(2):
        done[b].record(comp)
        out_read[b].record(comp)
    # warm-up: every pinned host batch and both device sets take part once before the
    # timed region, so first-use costs of the host buffers stay outside it
    for i in range(max(3, len(xh))):
        issue(i)
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    h2d.wait_stream(comp)
    d2h.wait_stream(comp)
    for i in range(steps):
        issue(i, timed=True)
    comp.wait_stream(d2h)
    e1.record(comp)
    torch.cuda.synchronize()
    barrier()
    ms = max_over_ranks(e0.elapsed_time(e1))
    h2d_ms = sum(a.elapsed_time(b) for a, b, _, _ in copy_ev) / len(copy_ev)
    d2h_ms = sum(c.elapsed_time(d) for _, _, c, d in copy_ev) / len(copy_ev)
    return {"value": flops_per_step(run.m, run.d, run.f) * steps * world / (ms / 1e3) / 1e12, "unit": "TFLOP/s",
            "h2d_bytes_per_step": 2 * run.m * run.d * 2, "d2h_bytes_per_step": 2 * run.m * run.d * 2,
            "steps": steps, "ms_per_step": ms / steps, "h2d_ms_per_step": h2d_ms, "d2h_ms_per_step": d2h_ms,
            "copies": "X, dY host->device (pinned) and Y, dX device->host every step, on their own streams, "
                      "overlapping the neighbouring steps' compute (two device buffer sets)"}


# A weight of this many elements or more is cast by its own (row-streaming) launch; a smaller
# one rides in its module's LayerNorm forward launch (the library's rule).
ROW_CAST_MIN_ELEMS = 1 << 24


def stack_hbm_bytes(layers, m, d, f):
    """Algorithmic bytes per stack step of the HBM-bound kernel kinds (each tensor read
    or written once): LayerNorm forward (x, and with the fused residual add r and the sum
    h, read/written as bf16; codes written; mu, rsigma; the launch also casts the module's
    weights below ROW_CAST_MIN_ELEMS: QKV, W1, W2), LayerNorm backward (dLN, x read, dX
    written), the gradient casts with column sums (dY of the MLP and the projection, dQKV)
    and the plain casts (the projection's weight and input, and the large weights)."""
    row = 8 * m
    weights = [3 * d * d, f * d, f * d]  # QKV, W1, W2 elements
    folded = sum(w for w in weights if w < ROW_CAST_MIN_ELEMS)
    own = sum(w for w in weights if w >= ROW_CAST_MIN_ELEMS)
    return {
        "ln_fwd_cast": (3 * m * d + row) + (2 * layers - 1) * (7 * m * d + row) + layers * 3 * folded,
        "ln_bwd": 2 * layers * (6 * m * d + row),
        "cast_colsum": layers * (3 * (m * d + m * d + 3 * m * d) + 4 * (d + d + 3 * d)),
        "cast": layers * (3 * d * d + 3 * m * d + 3 * own),
    }


def run_stack(L, torch, dev, args, flush, barrier, max_over_ranks, world, local, rank, fp8_peak, hbm,
              layers, m, d, f, hist, seed, k_max=40):
    """A transformer-block module stack step (StackRun), timed like the main workload,
    with its own clock record, per-kernel times and the HBM-bound kinds' fractions."""
    torch.cuda.empty_cache()
    srun = StackRun(L, torch, dev, layers, m, d, f, FMT, hist, seed=seed + rank)
    if args.graph:
        srun.capture()
    ks = max(3, min(args.steps, k_max))
    sclk = ClockSampler(local, f"_stack{d}x{layers}")
    sclk.start()
    sms, slaunch = timed_steps(torch, srun, ks, 3, flush, barrier, sclk)
    sclk = sclk.stop()
    sms = max_over_ranks(sms)
    L.sync_status()
    flops = stack_flops_per_step(layers, m, d, f)
    stack = {"value": flops * ks * world / (sms / 1e3) / 1e12,
             "unit": "TFLOP/s", "ms_per_step": sms / ks, "steps": ks, "gpu_launches": slaunch,
             "frac_of_fp8_peak": None, "cuda_graph": bool(args.graph), "clocks": sclk,
             "config": {"workload": f"transformer-block FP8 module stack fwd+bwd: {layers} layers x (LayerNormLinear "
                                    f"{d}->{3 * d}, Linear {d}->{d}, LayerNormMLP {d}->{f}->{d}), {m} "
                                    f"tokens, {FMT.upper()}, amax_history_len {hist}, one state-update launch for "
                                    f"all {6 * layers} state sets",
                        "layers": layers, "tokens": m, "d_model": d, "ffn": f, "amax_history_len": hist,
                        "inputs": "drawn once on the device and replayed every step: first layer's h N(0,1) + 0.1% "
                                  "x50; per layer attention output N(0,1), dQKV and dY N(0, 0.01); forward chained "
                                  "as a pre-LN block (residual adds fused into the next LayerNorm), backward per layer",
                        "flops": "six GEMMs per module"}}
    stack["frac_of_fp8_peak"] = stack["value"] / world / fp8_peak
    # per-kernel times of the same step (the library's event pairs as graph nodes)
    if args.graph:
        L.profile_enable(True)
        srun.capture(warm=False)
        for _ in range(3):
            flush.zero_()
            srun.step(0)
            L.profile_sample()
        sprof = L.profile_collect()
        L.profile_enable(False)
        tot = sum(v[0] for v in sprof.values()) or 1.0
        nbytes = stack_hbm_bytes(layers, m, d, f)
        pk = {}
        for k, v in sorted(sprof.items(), key=lambda kv: -kv[1][0]):
            pk[k] = {"ms_per_step": v[0] / 3, "launches_per_step": v[1] / 3, "share": v[0] / tot}
            if k in nbytes:
                gbs = nbytes[k] / (v[0] / 3 / 1e3) / 1e9
                pk[k].update({"algorithmic_bytes_per_step": nbytes[k], "gbs": gbs, "frac_hbm": gbs / hbm})
        stack["per_kernel"] = pk
        stack["per_kernel_timing"] = ("CUDA events around each launch inside replays of the captured step; each "
                                      "time includes the launch gap the event nodes add (a few us), so short "
                                      "kernels read low")
        gk = [v for k, v in sprof.items() if k.startswith("gemm")]
        if gk:
            stack["gemm_family_tflops"] = flops / (sum(v[0] for v in gk) / 3 / 1e3) / 1e12
    del srun
    torch.cuda.empty_cache()
    return stack


def run_config1(L, torch, dev, args, flush, fp8_peak, hbm):
    """LayerNormLinear forward 768 -> 2304 over 256 tokens (8 x 32), E4M3, history 16:
    one step, latency-bound; the median device time of replays of the captured call,
    for the library's automatic choice (the one-launch fused path here) and for the
    separate launches."""
    import numpy as np
    from fp8_delayed_scaling_row_gb300 import synth
    m, k, n, hist = 256, 768, 2304, 16

    def bf(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)

    p = synth.linear_params(n, k, seed=1234)
    x, g, b, w, bias = bf(synth.activations(m, k, seed=1234)), bf(p["gamma"]), bf(p["beta"]), bf(p["w"]), bf(p["b"])
    rec = L.Recipe("e4m3", hist)
    flops = 2.0 * m * k * n
    nbytes = m * k * (2 + 1) + 8 * m + n * k * (2 + 1) + m * n * 2  # x in, codes; W in, codes; y out

    def time_path(path):
        meta = L.ScalingMeta(2, hist, device=dev)
        ctx, y = L.linear_ctx(m, k, n, device=dev), torch.empty(m, n, dtype=torch.bfloat16, device=dev)

        def call():
            L.ln_linear_fwd(x, g, b, w, bias, meta, rec, y=y, ctx=ctx, path=path)

        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            c0 = L.launch_count()
            call()
            launches = L.launch_count() - c0
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        gr = None
        if args.graph:
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr):
                call()
        run = gr.replay if gr is not None else call
        steps = max(20, min(10 * args.steps, 500))
        for _ in range(5):
            run()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for a, e in ev:
            flush.zero_()
            a.record()
            run()
            e.record()
        torch.cuda.synchronize()
        L.sync_status()
        t = sorted(a.elapsed_time(e) for a, e in ev)
        med = t[len(t) // 2]
        return {"value": med * 1e3, "unit": "us/step", "min_us": t[0] * 1e3, "steps": steps,
                "tflops": flops / (med / 1e3) / 1e12, "frac_of_fp8_peak": flops / (med / 1e3) / 1e12 / fp8_peak,
                "gbs": nbytes / (med / 1e3) / 1e9, "frac_hbm": nbytes / (med / 1e3) / 1e9 / hbm,
                "gpu_launches_per_step": launches, "cuda_graph": gr is not None}

    auto = time_path(L.PATH_AUTO)
    fused, sep = time_path(L.PATH_FUSED), time_path(L.PATH_SEPARATE)
    out = dict(auto, higher_is_better=False, path="the library's automatic choice")
    out["fused_launch"] = fused
    out["separate_launches"] = sep
    out["config"] = {"workload": "LayerNormLinear forward 768 -> 2304 over 256 tokens (8 x 32), E4M3 activations and "
                                 "weights, amax_history_len 16, bias 0: LayerNorm + amax + cast, weight cast, FP8 GEMM, "
                                 "state update", "tokens": m, "in_features": k, "out_features": n,
                     "x_dist": "N(0,1)", "l2": "flushed between timed calls",
                     "timing": "median of per-call CUDA events"}
    return out


def run_sweep(L, torch, dev, args, flush, barrier, max_over_ranks, world, local, rank, fp8_peak):
    """Standalone LayerNormMLP 2048 -> 8192 -> 2048 fwd+bwd over tokens in {2048, 8192,
    32768, 65536}, E4M3 and HYBRID, N(0,1) and Student-t(3) activations, history 16
    and 1024: every point timed like the main workload (inputs drawn on the device)."""
    import numpy as np
    from fp8_delayed_scaling_row_gb300 import synth
    d, f = 2048, 8192
    params = {k: torch.from_numpy(np.ascontiguousarray(v).view(np.int16)).view(torch.bfloat16).to(dev)
              for k, v in synth.mlp_params(d, f, seed=2048).items()}
    clk = ClockSampler(local, "_sweep")
    clk.start()
    clk.mark_start()
    points = []
    for m in (2048, 8192, 32768, 65536):
        for fmt in ("e4m3", "hybrid"):
            for dist in ("normal", "t3"):
                for hist in (16, 1024):
                    run = MlpRun(L, torch, dev, m, d, f, fmt, hist, dist, 2, seed=m + 7 * hist + rank,
                                 inputs="device", params=params)
                    if args.graph:
                        run.capture()
                    k = max(3, min(args.steps, 20))
                    ms = max_over_ranks(timed_steps(torch, run, k, 3, flush, barrier)[0])
                    L.sync_status()
                    v = flops_per_step(m, d, f) * k * world / (ms / 1e3) / 1e12
                    points.append({"tokens": m, "fp8_format": fmt, "x_dist": DIST_TEXT[dist],
                                   "amax_history_len": hist, "value": v, "unit": "TFLOP/s",
                                   "ms_per_step": ms / k, "steps": k, "frac_of_fp8_peak": v / world / fp8_peak})
                    del run
                    torch.cuda.empty_cache()
    clk.mark_stop()
    return {"points": points, "clocks": clk.stop(),
            "config": {"workload": "LayerNormMLP 2048 -> 8192 -> 2048 fwd+bwd sweep: tokens x format x "
                                   "activation distribution x amax_history_len, each point timed alone",
                       "inputs": "2 X / dY batches per point drawn on the device, cycled; weights N(0, 0.02)",
                       "l2": "flushed (256 MiB write) between timed steps"}}


def run_gpu(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from fp8_delayed_scaling_row_gb300 import lnfp8 as L

    def barrier():
        if world > 1:
            dist.barrier()

    def max_over_ranks(v):
        if world == 1:
            return v
        t = torch.tensor([v], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    pk, how = peaks()
    bf16 = _num(pk, "bf16_tflops", "bf16_tflops_burst") or FALLBACK["bf16_tflops"]
    fp8_peak = bf16 * FP8_PER_BF16
    hbm = _num(pk, "hbm_gbs", "hbm_GBs", "hbm_copy_gbs") or FALLBACK["hbm_gbs"]
    if args.stack_only:  # diagnostic: the d 2048 stack step alone (e.g. a one-layer case to profile)
        stack = run_stack(L, torch, dev, args, flush, barrier, max_over_ranks, world, local, rank, fp8_peak, hbm,
                          args.stack_layers, 16384, 2048, 8192, 1024, seed=977)
        if rank == 0:
            print(json.dumps({"stack": stack}), flush=True)
        return 0
    n_sets = min(args.steps + args.warmup, 8)
    run = MlpRun(L, torch, dev, M_TOK, D_MODEL, FFN, FMT, HIST, "outliers", n_sets, seed=1234 + 7919 * rank)
    if args.graph:
        run.capture()

    # ---- main timed region (device time, CUDA events, L2 flushed between steps)
    clocks = ClockSampler(local)
    clocks.start()
    ms, gpu_launches = timed_steps(torch, run, args.steps, args.warmup, flush, barrier, clocks)
    clk = clocks.stop()
    L.sync_status()
    ms = max_over_ranks(ms)
    ms_step = ms / args.steps
    value = flops_per_step() * args.steps * world / (ms / 1e3) / 1e12

    # ---- per-kernel times inside the same workload (events on the launching stream)
    prof_steps = min(args.steps, 50)
    prof, prof_how = {}, "graph"
    if args.graph:
        # the step captured once more with the library's event pairs as graph nodes; every
        # replay re-records them (the event nodes sit between kernels, so no launch overlap)
        L.profile_enable(True)
        pg = run.capture_one(0)
        for i in range(prof_steps):
            flush.zero_()
            pg.replay()
            L.profile_sample()
        prof = L.profile_collect()
        L.profile_enable(False)
        del pg
    if not prof:
        prof_how = "direct calls"
        L.profile_enable(True)
        for i in range(prof_steps):  # direct calls: the library brackets each of its launches with events
            flush.zero_()
            run._call(run.xs[i % len(run.xs)], run.dys[i % len(run.dys)])
        prof = L.profile_collect()
        L.profile_enable(False)
    # the GEMM family: FC1 (+GELU), FC2, and the two backward launches that each run a data
    # gradient and its weight gradient together; one "launch" of the family = one step's set
    gemm_kinds = {k: v for k, v in prof.items() if k.startswith("gemm")}
    g_ms = sum(v[0] for v in gemm_kinds.values())
    g_n = sum(v[1] for v in gemm_kinds.values())
    g_flops = flops_per_step()  # the six GEMMs, 2 * M * D * F each
    achieved = g_flops / (g_ms / prof_steps / 1e3) / 1e12 if g_n else None
    roofline = {"kernel": "fp8 GEMM family (tcgen05 kind::f8f6f4): the step's six GEMMs in four launches",
                "bound": "tensor", "achieved": achieved, "peak": fp8_peak, "unit": "TFLOP/s",
                "frac": achieved / fp8_peak if achieved else None, "traffic": gemm_traffic_from_profile(),
                "peak_source": f"{how} bf16 dense x {FP8_PER_BF16:g} (nominal FP8/BF16 ratio)",
                "flops_per_launch": g_flops, "launch": "one step's GEMM launches (summed device time)",
                "gemm_launches_per_step": g_n / prof_steps, "launches_timed": g_n, "timed_from": prof_how,
                "share_of_step": g_ms / sum(v[0] for v in prof.values()) if prof else None}
    per_kernel = {}
    for k, (kms, cnt) in sorted(prof.items(), key=lambda kv: -kv[1][0]):
        per_kernel[k] = {"ms_per_launch": kms / cnt, "launches_per_step": cnt / prof_steps,
                         "share": kms / sum(v[0] for v in prof.values())}
    # LayerNorm / cast kernels against HBM (algorithmic bytes per launch)
    hbm_kernels = {
        # X read, codes written, mu/rsigma; the same launch casts W1 and W2 (read, codes written)
        "ln_fwd_cast": M_TOK * D_MODEL * (2 + 1) + M_TOK * 8 + 2 * FFN * D_MODEL * (2 + 1),
        "ln_bwd": M_TOK * D_MODEL * (2 + 2 + 2) + M_TOK * 8,         # dLN, X read, dX written, mu/rsigma
        "cast_colsum": M_TOK * D_MODEL * (2 + 1) + D_MODEL * 4,       # dY read, codes written, db2
    }
    for k, nbytes in hbm_kernels.items():
        if k in per_kernel:
            gbs = nbytes / (per_kernel[k]["ms_per_launch"] / 1e3) / 1e9
            per_kernel[k].update({"algorithmic_bytes": nbytes, "gbs": gbs, "frac_hbm": gbs / hbm})

    # ---- end to end through the C ABI with host buffers (pinned), copies timed
    e2e_steps = min(args.steps, 200)
    e2e = end_to_end(torch, run, e2e_steps, dev, barrier, max_over_ranks, world, graph=bool(args.graph))

    del run
    torch.cuda.empty_cache()

    # ---- the other workloads: the LN -> QKV forward alone (latency), the 4-layer d 768 and
    # 12-layer d 2048 module stacks, and the d 2048 LayerNormMLP format / size sweep
    config1 = None if args.no_config1 else run_config1(L, torch, dev, args, flush, fp8_peak, hbm)
    stack768 = None if args.no_stack else run_stack(L, torch, dev, args, flush, barrier, max_over_ranks, world, local,
                                                    rank, fp8_peak, hbm, 4, 8192, 768, 3072, 16, seed=768, k_max=50)
    stack = None if args.no_stack else run_stack(L, torch, dev, args, flush, barrier, max_over_ranks, world, local,
                                                 rank, fp8_peak, hbm, args.stack_layers, 16384, 2048, 8192, 1024,
                                                 seed=977)
    sweep = None if args.no_sweep else run_sweep(L, torch, dev, args, flush, barrier, max_over_ranks, world, local,
                                                 rank, fp8_peak)

    # ---- CPU baseline: the oracle as it stands, bounded sample, rank 0
    cpu = None
    if rank == 0 and not args.no_cpu:
        rows = args.cpu_rows
        val, n, el = oracle_rate(args.cpu_seconds, rows)
        cpu = {"value": val, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"{n} oracle steps of {rows} of the {M_TOK} tokens, full FFN ({el:.1f} s of CPU time; "
                         f"numpy, fp64 BLAS matmuls with the library's default threads)"}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "fp8 (e4m3/e5m2 operands, fp32 accumulate)", "data": "synthetic",
                "config": dict(workload(n_sets=n_sets), cuda_graph=bool(args.graph)), "frac_of_fp8_peak": value / world / fp8_peak,
                "clocks": clk, "e2e": e2e, "gpu_launches": gpu_launches, "roofline": roofline,
                "per_kernel": per_kernel, "hbm_peak_gbs": hbm, "cpu_baseline": cpu,
                "config1_ln_linear_fwd": config1, "stack768x4": stack768, "stack2048x12": stack,
                "sweep2048": sweep}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-rows", type=int, default=512, help="tokens per oracle step of the cpu_baseline leg")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-config1", action="store_true", help="skip the LN -> QKV forward latency leg")
    ap.add_argument("--no-sweep", action="store_true", help="skip the d 2048 LayerNormMLP format / size sweep")
    ap.add_argument("--no-stack", action="store_true", help="skip the d 768 and d 2048 module stack steps")
    ap.add_argument("--stack-only", action="store_true", help="run only the stack step (prints its own line)")
    ap.add_argument("--stack-layers", type=int, default=12)
    ap.add_argument("--graph", type=int, default=1, help="replay each step as a captured CUDA graph (1) or call (0)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
