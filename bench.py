"""Benchmark of the blockwise-FP8 linear-layer step on GB300.

One step = the whole hot path over one batch, in the library's training form:
quantise x once into its 1x128 groups along K and its 128x1 groups along M,
and W once into its 128x128 tiles (as is and transposed), both in one launch;
forward GEMM
1x128 x 128x128; quantise dY once into its 1x128 groups along N and along M
(of dY^T); input-gradient GEMM 1x128 x 128x128 and weight-gradient GEMM
1x128 x 128x1.

Default workload: the pages' mid shape M=2048, N=4096, K=4096 (x ~N(0,1) with
0.1% x100 outliers, W ~N(0,0.02), dY ~N(0,1e-3)), L2 flushed between steps.

value = GEMM FLOPs of the step (3 * 2MNK) / device time of the whole step
(quantisation included), TFLOP/s.  Per-kernel times come from CUDA events on
the launching stream.  `--impl reference` times the CPU oracle instead.
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
    """Samples nvidia-smi clocks and throttle reasons while running."""

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"bfp8_clocks_{os.getpid()}.csv")

    def __enter__(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits",
                                          "-i", str(self.index), "-lms", "200"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _lines(self):
        try:
            with open(self.path) as f:
                return sum(1 for _ in f)
        except OSError:
            return 0

    def wait_first_sample(self, timeout_s=3.0):
        t0 = time.time()
        while self.proc is not None and self._lines() == 0 and time.time() - t0 < timeout_s:
            time.sleep(0.05)

    def mark_start(self):
        self.n0 = self._lines()

    def mark_end(self):
        self.n1 = self._lines()

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            lines = f.readlines()
        n0, n1 = getattr(self, "n0", 0), getattr(self, "n1", len(lines))
        # samples taken during the timed region (plus the one in flight at its end)
        for line in lines[n0:min(len(lines), n1 + 1)]:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


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


def run_reference(args, wl):
    import oracle as O
    O.build()
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    full = wl
    wl, x, w, dy, prefix = _oracle_problem(wl, wl.x(), wl.w(), wl.dy())
    r, nr, nb, kb = _sample(wl, args.ref_rows, args.ref_blocks, 0)
    rot = [("fwd",), ("dgrad",), ("wgrad",)]  # one part of the step per iteration, in rotation
    for i in range(args.warmup):
        oracle_step_sample(x, w, dy, r, nr, nb, kb, rot[i % 3])
    t0 = time.perf_counter()
    flops = 0.0
    for i in range(args.steps):
        flops += oracle_step_sample(x, w, dy, r, nr, nb, kb, rot[i % 3])
    dt = time.perf_counter() - t0
    value = flops / dt / 1e12
    cores = O._threads()
    sample = "per step, one of (in rotation): " + prefix + _sample_text(wl, r, nr, nb, kb)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": full.name, "M": full.M, "N": full.N, "K": full.K},
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

    xh, wh, dyh = wl.x(), wl.w(), wl.dy()
    x, w, dy = todev(xh), todev(wh), todev(dyh)
    step = Step(wl, torch, B, dev)
    step.capture(x, w, dy)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    # Timed region: K steps, each the whole step as one graph replay between
    # two events, the L2 flushed before every step (outside the events).  Then
    # K more steps with one graph per call and events between the calls, for
    # the per-kernel times and the roofline of the dominant kernel.
    step_events = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(args.steps)]
    events = [step.new_events() for _ in range(args.steps)]
    with ClockSampler(local) as clk:
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
        owl, ox, ow, ody, prefix = _oracle_problem(wl, xh, wh, dyh)
        r, nr, nb, kb = _sample(owl, args.cpu_rows, args.cpu_blocks, 1)
        t0 = time.perf_counter()
        fl = oracle_step_sample(ox, ow, ody, r, nr, nb, kb)
        dt = time.perf_counter() - t0
        cpu = {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": O._threads(), "kind": "oracle",
               "sample": prefix + _sample_text(owl, r, nr, nb, kb) + f"; {dt:.1f} s"}

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
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="mid", choices=sorted(WORKLOADS))
    ap.add_argument("--ref-rows", type=int, default=4, help="oracle sample rows per reference step")
    ap.add_argument("--ref-blocks", type=int, default=1, help="oracle sample 128-col blocks per reference step")
    ap.add_argument("--cpu-rows", type=int, default=2048, help="oracle sample rows of the cpu_baseline leg (about 5 s on 16 Grace cores at the default workload)")
    ap.add_argument("--cpu-blocks", type=int, default=32, help="oracle sample 128-col blocks, cpu_baseline leg")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--chunk-n", type=int, default=0,
                    help="columns of W / dY per chunk of the host-buffer step (0 = automatic)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    wl = WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, wl)
    return run_gpu(args, wl)


if __name__ == "__main__":
    sys.exit(main())
