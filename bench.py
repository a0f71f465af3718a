"""Benchmark of the blockwise-FP8 linear-layer step on GB300.

One step = the whole hot path over one batch, in the library's training form:
quantise x once into its 1x128 groups along K and its 128x1 groups along M,
and W once into its 128x128 tiles (as is and transposed), both in one launch;
forward GEMM
1x128 x 128x128; quantise dY once into its 1x128 groups along N and along M
(of dY^T); input-gradient GEMM 1x128 x 128x128 and weight-gradient GEMM
1x128 x 128x1.

Default workload: the MLP-up layer M=16384 tokens, N=14336, K=4096 (x ~N(0,1),
W ~N(0,0.02), dY ~N(0,1e-3)), the largest single-GPU problem; the pages' mid
shape 2048x4096x4096 is `--workload mid`.  L2 flushed between steps.

value = GEMM FLOPs of the step (3 * 2MNK) / device time of the whole step
(quantisation included), TFLOP/s.  Per-kernel times come from CUDA events on
the launching stream.  `--impl reference` times the CPU oracle instead.
`--only NAME` times one library call of the step by itself (for profilers).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synthetic as S  # noqa: E402

WORKLOADS = {
    "mid": S.FWD_MID,          # 2048 x 4096 x 4096
    "wgrad": S.WGRAD,          # 8192 tokens, 4096 x 4096 (dW = dY^T X over 8192 tokens)
    "square": S.FWD_SQUARE,    # 8192 x 8192 x 8192
    "mlp_up": S.MLP_UP,        # 16384 x 14336 x 4096
    "moe_up": S.MOE_UP,        # 16384 tokens over 8 experts of 14336 x 4096
    "moe_mid": S.MOE_MID,      # 4096 tokens over 8 experts of 4096 x 4096
}
METRIC = "blockwise FP8 GEMM TFLOPS & quant GB/s at 1 GB300, % of FP8/HBM roofline"
L2_FLUSH_BYTES = 256 << 20
PROFILE_DIR = os.path.join(ROOT, "profiles")
GEMM_SRC = os.path.join(ROOT, "blockwise_scaled_fp8_gb300", "csrc", "gemm.cu")
QUANT_SRC = os.path.join(ROOT, "blockwise_scaled_fp8_gb300", "csrc", "quant_tile.cu")


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def _sha(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def _profile_traffic(kernel_key: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if its source hash
    matches the current kernel source; else None."""
    fname = os.path.join(PROFILE_DIR, f"{kernel_key}_{workload}.md")
    if not os.path.exists(fname):
        return None
    vals = {}
    with open(fname) as f:
        for line in f:
            if ":" in line and line.startswith("- "):
                k, v = line[2:].split(":", 1)
                vals[k.strip()] = v.strip().strip("`")
    src = GEMM_SRC if kernel_key.startswith("gemm") else QUANT_SRC
    if vals.get("source_sha") != _sha(src):
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """Samples the GPU's SM clock, its maximum, the power draw and the active
    clock-event (throttle) reasons every `period_s` on a background thread,
    through NVML (read-only queries, loaded with ctypes), falling back to an
    `nvidia-smi -lms` subprocess when NVML cannot be loaded.  summary()
    reports the samples taken inside the marked region; a region shorter than
    the period has none, and then the last sample before it and the first
    after it are reported instead, labelled as bracketing it."""

    # NVML clock-event reason bits (nvml.h, nvmlClocksEventReason*)
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, index: int, uuid: str | None = None, period_s: float = 0.01):
        self.index, self.uuid, self.period_s = index, uuid, period_s
        self.samples = []  # (perf_counter, sm_mhz, max_mhz, power_w, reasons)
        self.t0 = self.t1 = None
        self.source = None
        self._stop = False
        self._thread = None
        self._proc = None

    def _nvml(self):
        import ctypes
        lib = None
        for name in ("libnvidia-ml.so.1", "libnvidia-ml.so"):
            try:
                lib = ctypes.CDLL(name)
                break
            except OSError:
                continue
        if lib is None or lib.nvmlInit_v2() != 0:
            return None
        h = ctypes.c_void_p()
        ok = False
        if self.uuid:
            ok = lib.nvmlDeviceGetHandleByUUID(self.uuid.encode(), ctypes.byref(h)) == 0
        if not ok:
            ok = lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.index), ctypes.byref(h)) == 0
        if not ok:
            return None
        mx = ctypes.c_uint(0)
        lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))  # NVML_CLOCK_SM = 1

        def read():
            clk, pw, rs = ctypes.c_uint(0), ctypes.c_uint(0), ctypes.c_ulonglong(0)
            if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) != 0:
                return None
            lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(pw))
            lib.nvmlDeviceGetCurrentClocksEventReasons(h, ctypes.byref(rs))
            return (float(clk.value), float(mx.value), pw.value / 1000.0,
                    sorted(n for bit, n in self.REASONS.items() if rs.value & bit))
        return read

    def _run(self, read):
        while not self._stop:
            s = read()
            if s is not None:
                self.samples.append((time.perf_counter(),) + s)
            time.sleep(self.period_s)

    def _run_smi(self):
        q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            self._proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits", "-i", str(self.index),
                 "-lms", str(max(20, int(self.period_s * 1000)))],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        for line in self._proc.stdout:
            p = [v.strip() for v in line.split(",")]
            try:
                self.samples.append((time.perf_counter(), float(p[0]), float(p[1]), float(p[2]),
                                     sorted(n for n, v in zip(names, p[3:7]) if v.lower() == "active")))
            except (ValueError, IndexError):
                continue

    def __enter__(self):
        import threading
        read = None
        try:
            read = self._nvml()
        except (OSError, AttributeError):
            read = None
        if read is not None:
            self.source = f"nvml every {self.period_s * 1000:.0f} ms"
            self._thread = threading.Thread(target=self._run, args=(read,), daemon=True)
        else:
            self.source = "nvidia-smi"
            self._thread = threading.Thread(target=self._run_smi, daemon=True)
        self._thread.start()
        return self

    def wait_first_sample(self, timeout_s=3.0):
        t0 = time.time()
        while not self.samples and time.time() - t0 < timeout_s:
            time.sleep(0.01)

    def mark_start(self):
        self.t0 = time.perf_counter()

    def mark_end(self):
        self.t1 = time.perf_counter()
        # let one more sample land after the region, for the bracketing fallback
        n = len(self.samples)
        t = time.time()
        while len(self.samples) == n and time.time() - t < 1.0:
            time.sleep(0.005)

    def __exit__(self, *a):
        self._stop = True
        if self._proc is not None:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self._proc.kill()
        if self._thread is not None:
            self._thread.join(timeout=5)

    def summary(self):
        if not self.samples or self.t0 is None or self.t1 is None:
            return None
        inside = [s for s in self.samples if self.t0 <= s[0] <= self.t1]
        window = "timed region"
        if not inside:
            before = [s for s in self.samples if s[0] < self.t0][-1:]
            after = [s for s in self.samples if s[0] > self.t1][:1]
            inside = before + after
            window = "bracketing the timed region (no sample fell inside it)"
        if not inside:
            return None
        reasons = sorted({r for s in inside for r in s[4]})
        return {"sm_mhz": statistics.median(s[1] for s in inside), "sm_max_mhz": max(s[2] for s in inside),
                "power_w_max": max(s[3] for s in inside), "samples": len(inside), "reasons": reasons,
                "window": window, "region_ms": round((self.t1 - self.t0) * 1e3, 2), "source": self.source}


# ---------------------------------------------------------------------------
# CPU oracle leg (the reported baseline; also the whole `--impl reference` arm)
# ---------------------------------------------------------------------------

def oracle_step_sample(x, w, dy, rows, nrows, nblocks, kblocks, parts=("fwd", "dgrad", "wgrad")):
    """One bounded sample of the step on the CPU oracle: forward outputs
    y[rows, n in nblocks], input-gradient outputs dx[rows, k in kblocks] and
    weight-gradient outputs dw[nrows, k in kblocks], each with every
    quantisation those outputs need (groups and tiles are local to rows,
    128-row blocks and columns, so the sub-problems quantise exactly as the
    full tensors would).  Returns the GEMM FLOPs the sample covers."""
    import oracle as O
    M, K = x.shape
    N = w.shape[0]
    ncols = np.concatenate([np.arange(b * 128, min(N, b * 128 + 128)) for b in nblocks])
    kcols = np.concatenate([np.arange(b * 128, min(K, b * 128 + 128)) for b in kblocks])
    flops = 0.0
    if "fwd" in parts:
        qa, sa = O.quant_lhs(np.ascontiguousarray(x[rows]))
        qw, _, sw = O.quant_weight(np.ascontiguousarray(w[ncols]))
        O.gemm(qa, sa, qw, sw, O.SB_TILE, K)
        flops += 2.0 * len(rows) * len(ncols) * K
    if "dgrad" in parts:
        qd, sd = O.quant_lhs(np.ascontiguousarray(dy[rows]))
        _, qwt, swt = O.quant_weight(np.ascontiguousarray(w[:, kcols]), with_t=True)
        O.gemm(qd, sd, qwt, swt, O.SB_TILE_T, N)
        flops += 2.0 * len(rows) * len(kcols) * N
    if "wgrad" in parts:
        qdt, sdt = O.quant_lhs(np.ascontiguousarray(dy[:, nrows]), transposed=True)
        qxt, sxt = O.quant_rhs(np.ascontiguousarray(x[:, kcols]))
        O.gemm(qdt, sdt, qxt, sxt, O.SB_COL, M)
        flops += 2.0 * len(nrows) * len(kcols) * M
    return flops


def _sample(wl, rows, blocks, seed):
    rng = np.random.default_rng(seed)
    r = np.sort(rng.choice(wl.M, size=min(wl.M, rows), replace=False))
    nr = np.sort(rng.choice(wl.N, size=min(wl.N, rows), replace=False))
    nb = np.sort(rng.choice((wl.N + 127) // 128, size=min((wl.N + 127) // 128, blocks), replace=False))
    kb = np.sort(rng.choice((wl.K + 127) // 128, size=min((wl.K + 127) // 128, blocks), replace=False))
    return r, nr, nb, kb


def _sample_text(wl, r, nr, nb, kb):
    return (f"fwd y[{len(r)} of {wl.M} rows, {len(nb)} of {(wl.N + 127) // 128} 128-col blocks], "
            f"dgrad dx[{len(r)} rows, {len(kb)} of {(wl.K + 127) // 128} blocks], "
            f"wgrad dw[{len(nr)} of {wl.N} rows, {len(kb)} blocks], each with the quantisations it needs")


def _oracle_problem(wl, x, w, dy):
    """The dense problem the oracle samples: the workload itself, or for a
    mixture-of-experts workload the first expert with tokens (each expert's
    layer is the dense method on its token slice)."""
    if not isinstance(wl, S.MoE):
        return wl, x, w, dy, ""
    offs = wl.offsets()
    e = next(i for i in range(wl.E) if offs[i + 1] > offs[i])
    r0, r1 = int(offs[e]), int(offs[e + 1])
    sub = S.Linear(f"{wl.name}_expert{e}", M=r1 - r0, N=wl.N, K=wl.K, seed=wl.seed)
    return (sub, x[r0:r1], w[e * wl.N:(e + 1) * wl.N], dy[r0:r1],
            f"expert {e} of {wl.E} (tokens {r0}..{r1}): ")


def cpu_unit_samples(args, wl, x, w, dy, reps, seed0):
    """`reps` bounded samples of the step on the oracle, each the same shape
    (--cpu-rows rows, --cpu-blocks 128-column blocks, all three GEMMs with
    their quantisations) at a different seeded position.  The cpu_baseline
    leg and the reference arm both time these units, so the two report the
    same oracle on the same sample shape.  Returns (flops, seconds, text)."""
    owl, ox, ow, ody, prefix = _oracle_problem(wl, x, w, dy)
    flops, dt, text = 0.0, 0.0, ""
    for i in range(reps):
        r, nr, nb, kb = _sample(owl, args.cpu_rows, args.cpu_blocks, seed0 + i)
        t0 = time.perf_counter()
        flops += oracle_step_sample(ox, ow, ody, r, nr, nb, kb)
        dt += time.perf_counter() - t0
        text = prefix + _sample_text(owl, r, nr, nb, kb)
    return flops, dt, text


def run_reference(args, wl):
    import oracle as O
    O.build()
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    x, w, dy = wl.x(), wl.w(), wl.dy()
    cpu_unit_samples(args, wl, x, w, dy, args.warmup, 1000)
    flops, dt, text = cpu_unit_samples(args, wl, x, w, dy, args.steps, 0)
    value = flops / dt / 1e12
    cores = O._threads()
    sample = "per step, one unit: " + text
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": wl.name, "M": wl.M, "N": wl.N, "K": wl.K},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# GPU leg
# ---------------------------------------------------------------------------

class Step:
    """Preallocated buffers and the kernel sequence of one linear step, each
    call recorded between CUDA events on the current stream.  For a
    mixture-of-experts workload the weights are the experts' stacked [E*N, K]
    and the three GEMMs are the grouped ones."""

    def __init__(self, wl, torch, B, dev):
        self.wl, self.torch, self.B = wl, torch, B
        M, N, K = wl.M, wl.N, wl.K
        E = getattr(wl, "E", 1)
        self.moe = isinstance(wl, S.MoE)
        rup = lambda a, b: (a + b - 1) // b * b
        cd = lambda a: (a + 127) // 128
        u8, f32, bf = torch.uint8, torch.float32, torch.bfloat16
        e = lambda *s, dt: torch.empty(s, dtype=dt, device=dev)
        self.qx, self.sx = e(M, rup(K, 16), dt=u8), e(cd(K), rup(M, 4), dt=f32)
        self.qxt, self.sxt = e(K, rup(M, 16), dt=u8), e(cd(M), rup(K, 4), dt=f32)
        self.qw, self.qwt = e(E * N, rup(K, 16), dt=u8), e(K, rup(E * N, 16), dt=u8)
        self.sw = e(E * cd(N), cd(K), dt=f32)
        self.qdy, self.sdy = e(M, rup(N, 16), dt=u8), e(cd(N), rup(M, 4), dt=f32)
        self.qdyt, self.sdyt = e(N, rup(M, 16), dt=u8), e(cd(M), rup(N, 4), dt=f32)
        self.y, self.dx = e(M, N, dt=bf), e(M, K, dt=bf)
        self.dw = e(E, N, K, dt=bf) if self.moe else e(N, K, dt=bf)
        self.offs = torch.from_numpy(wl.offsets()).to(dev) if self.moe else None
        self.names = ["quant_x_w", "gemm_fwd", "quant_dual_dy", "gemm_dgrad", "gemm_wgrad"]
        self.launches_per_step = len(self.names)

    def new_events(self):
        return [self.torch.cuda.Event(enable_timing=True) for _ in range(len(self.names) + 1)]

    def _calls(self, x, w, dy):
        B, wl = self.B, self.wl
        M, N, K = wl.M, wl.N, wl.K
        if self.moe:
            o = self.offs
            return [
                lambda: B.quant_dual_weight(x, w, q_row=self.qx, s_row=self.sx, q_col=self.qxt, s_col=self.sxt,
                                            qw=self.qw, qwt=self.qwt, sw=self.sw),
                lambda: B.gemm_grouped_1x128_128x128(self.qx, self.sx, self.qw, self.sw, o, N, K, out=self.y),
                lambda: B.quant_dual(dy, q_row=self.qdy, s_row=self.sdy, q_col=self.qdyt, s_col=self.sdyt),
                lambda: B.gemm_grouped_1x128_128x128(self.qdy, self.sdy, self.qwt, self.sw, o, K, N,
                                                     sb_transposed=True, out=self.dx),
                lambda: B.gemm_grouped_1x128_128x1(self.qdyt, self.sdyt, self.qxt, self.sxt, o, M, out=self.dw),
            ]
        return [
            lambda: B.quant_dual_weight(x, w, q_row=self.qx, s_row=self.sx, q_col=self.qxt, s_col=self.sxt,
                                        qw=self.qw, qwt=self.qwt, sw=self.sw),
            lambda: B.gemm_1x128_128x128(self.qx, self.sx, self.qw, self.sw, K, out=self.y, M=M, N=N),
            lambda: B.quant_dual(dy, q_row=self.qdy, s_row=self.sdy, q_col=self.qdyt, s_col=self.sdyt),
            lambda: B.gemm_1x128_128x128(self.qdy, self.sdy, self.qwt, self.sw, N, sb_transposed=True,
                                         out=self.dx, M=M, N=K),
            lambda: B.gemm_1x128_128x1(self.qdyt, self.sdyt, self.qxt, self.sxt, M, out=self.dw, M=N, N=K),
        ]

    def capture(self, x, w, dy):
        """The whole step as one CUDA graph (the timed step), and one graph per
        library call (per-kernel events between them); host-side launch work
        (argument checks, tensor-map encoding) stays off the device timeline."""
        torch = self.torch
        calls = self._calls(x, w, dy)
        for c in calls:  # warm: one-time attribute setup happens outside capture
            c()
        torch.cuda.synchronize()
        self.graphs = []
        for c in calls:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                c()
            self.graphs.append(g)
        self.step_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.step_graph):
            for c in calls:
                c()
        torch.cuda.synchronize()

    def run_step(self, ev=None):
        """One step as a single graph replay, bracketed by ev = (start, end)."""
        if ev is not None:
            ev[0].record()
        self.step_graph.replay()
        if ev is not None:
            ev[1].record()

    def run(self, x, w, dy, ev=None):
        timed = ev is not None
        if timed:
            ev[0].record()
        for i, g in enumerate(self.graphs):
            g.replay()
            if timed:
                ev[i + 1].record()

    def kernel_ms(self, ev):
        return [ev[i].elapsed_time(ev[i + 1]) for i in range(len(self.names))]


def algorithmic_units(wl):
    """Per-launch algorithmic work: FLOPs for the GEMMs, bytes for the quants
    (read 2 B/elem bf16 once, write 1 B/elem e4m3 per output form, plus 4 B
    per scale)."""
    M, N, K = wl.M, wl.N, wl.K
    E = getattr(wl, "E", 1)
    cd = lambda a: (a + 127) // 128
    gem = 2.0 * M * N * K
    return {
        "quant_x_w": ("GB/s", 4.0 * M * K + 4.0 * (M * cd(K) + K * cd(M)) + E * (4.0 * N * K + 4.0 * cd(N) * cd(K))),
        "gemm_fwd": ("TFLOP/s", gem),
        "quant_dual_dy": ("GB/s", 4.0 * M * N + 4.0 * (M * cd(N) + N * cd(M))),
        "gemm_dgrad": ("TFLOP/s", gem),
        "gemm_wgrad": ("TFLOP/s", gem),
    }


def aggregate_replicas(local_ms: float, units_per_rank: float, dist=None, device=None):
    """Whole-job throughput of N independent replicas: every rank processed
    `units_per_rank` units; the job took the slowest rank's time.
    Returns (max_ms over ranks, units_total / max_s)."""
    world = 1
    ms = float(local_ms)
    if dist is not None and dist.is_initialized():
        import torch
        world = dist.get_world_size()
        t = torch.tensor([ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, world * units_per_rank / (ms / 1e3)


# the buffers each library call of the step reads or writes (Step attributes)
ONLY_BUFFERS = {
    "quant_x_w": ("qx", "sx", "qxt", "sxt", "qw", "qwt", "sw"),
    "gemm_fwd": ("qx", "sx", "qw", "sw", "y"),
    "quant_dual_dy": ("qdy", "sdy", "qdyt", "sdyt"),
    "gemm_dgrad": ("qdy", "sdy", "qwt", "sw", "dx"),
    "gemm_wgrad": ("qdyt", "sdyt", "qxt", "sxt", "dw"),
}
ONLY_INPUTS = {"quant_x_w": ("x", "w"), "quant_dual_dy": ("dy",)}


def run_only(args, wl, torch, B, dev, todev, flush):
    """One library call of the step, by itself: every call of the step runs
    once (so the call's inputs exist), every buffer the named call does not
    touch is freed (a profiler that replays the call saves and restores less
    device memory), then the named call runs --warmup times untimed and
    --steps times between CUDA events, L2 flushed before each.  Launch order,
    for a profiler's skip count: the step's five calls (quant_x_w, gemm_fwd,
    quant_dual_dy, gemm_dgrad, gemm_wgrad), then the repeats of the named one."""
    step = Step(wl, torch, B, dev)
    inp = {"x": todev(wl.x()), "w": todev(wl.w()), "dy": todev(wl.dy())}
    for c in step._calls(inp["x"], inp["w"], inp["dy"]):
        c()
    torch.cuda.synchronize()
    for name in ("qx", "sx", "qxt", "sxt", "qw", "qwt", "sw", "qdy", "sdy", "qdyt", "sdyt", "y", "dx", "dw"):
        if name not in ONLY_BUFFERS[args.only]:
            setattr(step, name, None)
    for name in ("x", "w", "dy"):
        if name not in ONLY_INPUTS.get(args.only, ()):
            inp[name] = None
    torch.cuda.empty_cache()
    call = step._calls(inp["x"], inp["w"], inp["dy"])[step.names.index(args.only)]
    for _ in range(args.warmup):
        flush.fill_(0.0)
        call()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a, b in ev:
        flush.fill_(0.0)
        a.record()
        call()
        b.record()
    torch.cuda.synchronize()
    B.check_device_errors()
    ms = float(np.mean([a.elapsed_time(b) for a, b in ev]))
    unit, work = algorithmic_units(wl)[args.only]
    scale = 1e12 if unit == "TFLOP/s" else 1e9
    print(json.dumps({"only": args.only, "workload": wl.name, "ms": ms, unit: work / (ms / 1e3) / scale,
                      "steps": args.steps, "warmup": args.warmup,
                      "device_bytes_held": int(torch.cuda.memory_allocated(dev))}), flush=True)
    return 0


def run_ceiling(args, wl, torch, dev, flush):
    """A measured ceiling, not a result of this library: the vendor library's
    FP8 GEMM (`torch._scaled_mm`, cuBLASLt) at the workload's three GEMM
    shapes, tensorwise-scaled (one fp32 scale per operand, no per-block
    promotion), and block-scaled (1x128 x 128x128 fp32 scales) where this
    torch build accepts such scales.  Random e4m3 operands; L2 flushed before
    every call, CUDA events, median of --steps calls after --warmup."""
    M, N, K = wl.M, wl.N, wl.K
    shapes = {"gemm_fwd": (M, N, K), "gemm_dgrad": (M, K, N), "gemm_wgrad": (N, K, M)}
    gen = torch.Generator(device=dev)
    gen.manual_seed(0)
    steps = max(5, min(args.steps, 50))

    def timed(f):
        for _ in range(args.warmup):
            f()
        ts = []
        for _ in range(steps):
            flush.fill_(1.0)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            f()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        ts.sort()
        return ts[len(ts) // 2] * 1e3

    out = {}
    for name, (m, n, k) in shapes.items():
        a = (torch.randn(m, k, device=dev, generator=gen) * 0.5).to(torch.float8_e4m3fn)
        b = (torch.randn(n, k, device=dev, generator=gen) * 0.5).to(torch.float8_e4m3fn)
        one = torch.ones((), dtype=torch.float32, device=dev)
        flops = 2.0 * m * n * k
        rec = {"M": m, "N": n, "K": k}
        us = timed(lambda: torch._scaled_mm(a, b.t(), scale_a=one, scale_b=one, out_dtype=torch.bfloat16))
        rec["tensorwise_us"] = round(us, 1)
        rec["tensorwise_TFLOP/s"] = round(flops / (us / 1e6) / 1e12, 1)
        kb, nb = (k + 127) // 128, (n + 127) // 128
        # candidate layouts for 1x128 (A) and 128x128 (B) scales; the first one this build accepts is timed
        cands = [("a [M,Kb] outer-major, b [Nb,Kb]",
                  torch.rand(kb, m, device=dev).t(), torch.rand(nb, kb, device=dev)),
                 ("a [M,Kb] outer-major, b [Kb,Nb] outer-major",
                  torch.rand(kb, m, device=dev).t(), torch.rand(nb, kb, device=dev).t()),
                 ("a [M,Kb], b [Nb,Kb]", torch.rand(m, kb, device=dev), torch.rand(nb, kb, device=dev))]
        rec["blockwise"] = "not accepted by this build"
        errors = []
        for label, sa, sb in cands:
            try:
                torch._scaled_mm(a, b.t(), scale_a=sa, scale_b=sb, out_dtype=torch.bfloat16)
                torch.cuda.synchronize()
            except Exception as e:  # this build rejects the layout (a host-side check)
                errors.append(f"{label}: {str(e).splitlines()[0][:120]}")
                continue
            us = timed(lambda: torch._scaled_mm(a, b.t(), scale_a=sa, scale_b=sb, out_dtype=torch.bfloat16))
            rec["blockwise"] = {"scales": label, "us": round(us, 1),
                                "TFLOP/s": round(flops / (us / 1e6) / 1e12, 1)}
            break
        if errors and not isinstance(rec["blockwise"], dict):
            rec["blockwise_errors"] = errors
        out[name] = rec
    print(json.dumps({"ceiling": "torch._scaled_mm (cuBLASLt FP8), a measured reference point, not this library",
                      "workload": wl.name, "torch": torch.__version__, "steps": steps, "warmup": args.warmup,
                      "gemms": out}), flush=True)
    return 0


def run_gpu(args, wl):
    import torch

    import blockwise_scaled_fp8_gb300 as B
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    B.build()
    dev = torch.device("cuda", local)

    def todev(a):
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)

    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    if args.ceiling:
        return run_ceiling(args, wl, torch, dev, flush)
    if args.only:
        return run_only(args, wl, torch, B, dev, todev, flush)
    xh, wh, dyh = wl.x(), wl.w(), wl.dy()
    x, w, dy = todev(xh), todev(wh), todev(dyh)
    step = Step(wl, torch, B, dev)
    step.capture(x, w, dy)

    # Timed region: K steps, each the whole step as one graph replay between
    # two events, the L2 flushed before every step (outside the events).  Then
    # K more steps with one graph per call and events between the calls, for
    # the per-kernel times and the roofline of the dominant kernel.
    step_events = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(args.steps)]
    events = [step.new_events() for _ in range(args.steps)]
    props = torch.cuda.get_device_properties(dev)
    uuid = getattr(props, "uuid", None)
    with ClockSampler(local, uuid=f"GPU-{uuid}" if uuid is not None else None) as clk:
        for _ in range(args.warmup):
            step.run_step()
            flush.fill_(1.0)
            step.run(x, w, dy)
            flush.fill_(1.0)
        torch.cuda.synchronize()
        B.check_device_errors()
        clk.wait_first_sample()
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        clk.mark_start()
        for i in range(args.steps):
            flush.fill_(0.0)  # L2 flush between timed steps (outside the step's events)
            step.run_step(step_events[i])
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        clk.mark_end()
        for i in range(args.steps):
            flush.fill_(0.0)
            step.run(x, w, dy, events[i])
        torch.cuda.synchronize()
    B.check_device_errors()
    clocks = clk.summary()
    per_kernel = [step.kernel_ms(ev) for ev in events]
    step_ms = [a.elapsed_time(b) for a, b in step_events]

    flops_step = 3 * wl.gemm_flops
    total_ms, flops_per_s = aggregate_replicas(float(sum(step_ms)), flops_step * args.steps, dist, dev)
    value = flops_per_s / 1e12

    # per-kernel averages, rooflines
    units = algorithmic_units(wl)
    peaks = _peaks()
    fp8_peak = 2.0 * peaks["bf16_tflops"]  # fp8 dense = 2 x bf16 dense (nominal ratio)
    avg = np.mean(np.array(per_kernel), axis=0)
    parts = {}
    for name, ms in zip(step.names, avg):
        unit, work = units[name]
        if unit == "TFLOP/s":
            ach = work / (ms / 1e3) / 1e12
            parts[name] = {"ms": round(float(ms), 5), "TFLOP/s": round(ach, 2), "frac_fp8_peak": round(ach / fp8_peak, 4)}
        else:
            ach = work / (ms / 1e3) / 1e9
            parts[name] = {"ms": round(float(ms), 5), "GB/s": round(ach, 1), "frac_hbm": round(ach / peaks["hbm_gbs"], 4)}
    dom = max(range(len(step.names)), key=lambda i: avg[i])
    dname = step.names[dom]
    unit, work = units[dname]
    if unit == "TFLOP/s":
        ach = work / (avg[dom] / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": ach, "peak": fp8_peak, "unit": "TFLOP/s", "frac": ach / fp8_peak}
        peak_note = f"{peaks['source']} bf16 burst {peaks['bf16_tflops']} x 2 (fp8/bf16 nominal ratio)"
    else:
        ach = work / (avg[dom] / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": ach / peaks["hbm_gbs"]}
        peak_note = f"{peaks['source']} HBM copy bandwidth"
    kkey = "gemm_1x128_128x128" if dname in ("gemm_fwd", "gemm_dgrad") else (
        "gemm_1x128_128x1" if dname == "gemm_wgrad" else dname)
    if step.moe and dname.startswith("gemm"):
        kkey = "gemm_grouped" + kkey[4:]
    roof["traffic"] = _profile_traffic(kkey, wl.name)
    roof["kernel"] = dname
    roof["peak_source"] = peak_note

    # end to end through the public API: host (pinned) -> device, the step's
    # five library calls, device -> host
    e2e = None
    if not args.no_e2e:
        hx = torch.from_numpy(xh.view(np.int16)).view(torch.bfloat16).pin_memory()
        hw = torch.from_numpy(wh.view(np.int16)).view(torch.bfloat16).pin_memory()
        hdy = torch.from_numpy(dyh.view(np.int16)).view(torch.bfloat16).pin_memory()
        M, N, K = wl.M, wl.N, wl.K
        E = getattr(wl, "E", 1)
        oy = torch.empty(tuple(step.y.shape), dtype=torch.bfloat16).pin_memory()
        odx = torch.empty(tuple(step.dx.shape), dtype=torch.bfloat16).pin_memory()
        odw = torch.empty(tuple(step.dw.shape), dtype=torch.bfloat16).pin_memory()
        # the library's host-buffer steps: W and dY travel in column chunks,
        # each chunk's GEMMs run while the next arrives, outputs leave as they
        # are finished (mixture of experts: one such step per expert, two
        # experts' device buffers in turn, offsets read on the host)
        if step.moe:
            hoffs = torch.from_numpy(wl.offsets())
            hw3 = hw.view(E, N, K)
            hws = B.moe_step_host_workspace(int(np.max(np.diff(wl.offsets()))), N, K, device=dev)

            def e2e_step():
                B.moe_step_host(hx, hw3, hdy, hoffs, hws, y=oy, dx=odx, dw=odw, chunk_n=args.chunk_n)
        else:
            hws = B.linear_step_host_workspace(M, N, K, device=dev)

            def e2e_step():
                B.linear_step_host(hx, hw, hdy, hws, y=oy, dx=odx, dw=odw, chunk_n=args.chunk_n)

        for _ in range(args.warmup):
            e2e_step()
        torch.cuda.synchronize()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        tot = 0.0
        for _ in range(args.steps):
            flush.fill_(0.0)
            s0.record()
            e2e_step()
            s1.record()
            torch.cuda.synchronize()
            tot += s0.elapsed_time(s1)
        e2e = {"value": flops_step * args.steps / (tot / 1e3) / 1e12 * world, "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(2 * (M * K + E * N * K + M * N)),
               "d2h_bytes_per_step": int(2 * (M * N + M * K + E * N * K)),
               "ms_per_step": tot / args.steps,
               "path": ("bfp8_moe_step_host" if step.moe else "bfp8_linear_step_host") +
                       ": pinned host x, W, dY in, y, dX, dW out; copies on the library's two copy streams, "
                       "W and dY in column chunks overlapped with the GEMMs" +
                       ("; one dense step per expert, offsets on the host" if step.moe else "")}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        import oracle as O
        O.build()
        fl, dt, text = cpu_unit_samples(args, wl, xh, wh, dyh, args.cpu_reps, 0)
        cpu = {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": O._threads(), "kind": "oracle",
               "sample": f"{args.cpu_reps} units (the reference arm's per-step unit), each: " + text +
                         f"; {dt:.1f} s in all"}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "fp8_e4m3 (fp32 accumulate)",
                "data": "synthetic",
                "config": {"workload": wl.name, "M": wl.M, "N": wl.N, "K": wl.K,
                           **({"experts": wl.E, "expert_offsets": [int(v) for v in wl.offsets()],
                               "gemms": "grouped by expert"} if step.moe else {}),
                           "step": "quant x (1x128 + 128x1) and W (tiles + transposed) in one launch; fwd GEMM; "
                                   "quant dY (1x128 along N and M); dgrad GEMM; wgrad GEMM",
                           "l2": "flushed between steps (256 MiB write)", "parallelism": f"replicas x{world}",
                           "launch": "timed steps: the whole step replayed as one CUDA graph, events around "
                                     "each step; parts/roofline: as many steps again with one graph per "
                                     "library call and events between calls"},
                "gpu_launches": step.launches_per_step * args.steps,
                "parts_ms_per_step": round(float(np.sum(avg)), 5),
                "roofline": roof, "parts": parts, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks}
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="mlp_up", choices=sorted(WORKLOADS))
    ap.add_argument("--cpu-rows", type=int, default=512,
                    help="rows of one oracle sample unit (the reference arm's step; cpu_baseline repeats it)")
    ap.add_argument("--cpu-blocks", type=int, default=8, help="128-column blocks of one oracle sample unit")
    ap.add_argument("--cpu-reps", type=int, default=6, help="oracle sample units timed by the cpu_baseline leg")
    ap.add_argument("--only", default=None,
                    help="time one library call of the step by itself (quant_x_w, gemm_fwd, quant_dual_dy, "
                         "gemm_dgrad, gemm_wgrad), for profilers")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--chunk-n", type=int, default=0,
                    help="columns of W / dY per chunk of the host-buffer step (0 = automatic)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ceiling", action="store_true",
                    help="time the vendor library's FP8 GEMM (torch._scaled_mm) at the workload's GEMM shapes "
                         "as a measured ceiling, and nothing else")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    wl = WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, wl)
    return run_gpu(args, wl)


if __name__ == "__main__":
    sys.exit(main())
