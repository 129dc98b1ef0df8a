"""Benchmark of the MoE decode step (weight-streaming GB/s over the unique expert bytes).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config NAME] [--rows M] [--no-sweep] [--no-cpu-baseline]

One step = router GEMV, top-k + route + FC1 input quantisation, gate_up + down (one
launch), finalize (moe_step: four chained launches) captured in a CUDA graph, on seeded
synthetic inputs of the workload's shapes. Between timed steps (untimed) a 512 MiB buffer is written and another
read, so every step streams its weights from HBM and finds no dirty line of the flush in L2.

The JSON line's value / config are the 8-row MXFP8 layer (H 7168, 256 experts, top-8);
its `sweep` object holds every other workload measured the same way (median, p10, p90 of
200 graph replays): the 1-row tiny layer, the 16-row NVFP4 layer, the 48-row skewed layer,
the 512-expert NVFP4 layer at 1, 2, 4, 8, 16, 32, 48 and 64 rows, and packed MXFP4 at 1, 8
and 64 rows. Under torchrun each rank runs an independent replica (the step has no
cross-GPU exchange); the JSON line reports the sum over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

HEADLINE = "mxfp8_h7168_e256_k8_8rows"
METRIC = "MoE decode step weight GB/s (unique expert + shared + router bytes per step / step time)"
L2_NOTE = "512 MiB buffer written, then another 512 MiB read, between timed steps (untimed)"
# every other workload: (name, rows or None for the workload's own)
SWEEP = ([("tiny_mxfp8", None), ("nvfp4_h6144_e256_k8_16rows", None), ("mxfp8_skew_48rows", None)] +
         [("nvfp4_h4096_e512_k10", m) for m in (1, 2, 4, 8, 16, 32, 48, 64)] +
         [("mxfp4_h7168_e256_k8", m) for m in (1, 8, 64)])
SWEEP_STEPS, SWEEP_WARMUP = 200, 20


def _args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default=HEADLINE)
    ap.add_argument("--rows", type=int, default=None)
    ap.add_argument("--experts", type=int, default=None, help="override E (smaller profiling cases)")
    ap.add_argument("--inter", type=int, default=None, help="override I and shared I (smaller profiling cases)")
    ap.add_argument("--swiglu-limit", type=float, default=None, help="clamped SwiGLU limit (default: plain SwiGLU)")
    ap.add_argument("--schedule", default="static", choices=["static", "hybrid", "dynamic"])
    ap.add_argument("--ffn-launches", type=int, default=1, choices=[1, 2])
    ap.add_argument("--front-launches", type=int, default=2, choices=[1, 2])
    ap.add_argument("--no-sweep", action="store_true", help="only the headline workload")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--seed", type=int, default=0)
    return ap.parse_args(argv)


class Clocks:
    """nvidia-smi sampling of SM clock and throttle reasons; only samples taken inside the
    timed windows (window() after each timed loop) are reported."""

    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []
        self.windows = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def window(self, t0, t1):
        self.windows.append((t0, t1))

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons, n_all = [], None, set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        # a sample describes the 50 ms before it was read
        inside = lambda t: any(a - 0.01 <= t <= b + 0.06 for a, b in self.windows)
        for t, ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 10:
                continue
            try:
                clk, mx = float(f[2]), float(f[3])
            except ValueError:
                continue
            n_all += 1
            if not inside(t):
                continue
            sm.append(clk)
            for n, v in zip(names, f[6:10]):
                if v.lower() == "active":
                    reasons.add(n)
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "samples_total": n_all, "interval_ms": 50,
                "timed_windows_s": round(sum(b - a for a, b in self.windows), 3)}


def _cfg(a, name=None, rows=None):
    from moe_decode_step_router_gb300 import synth
    over = {"schedule": a.schedule, "ffn_launches": a.ffn_launches, "front_launches": a.front_launches}
    rows = a.rows if name is None else rows
    if rows is not None:
        over["M"] = rows
    if a.experts is not None:
        over["E"] = a.experts
    if a.inter is not None:
        over["I"] = over["I_sh"] = a.inter
    if a.swiglu_limit is not None:
        over["swiglu_limit"] = a.swiglu_limit
    return synth.config(name or a.config, **over)


GEMM_SOURCES = ("gemm.cu", "ptx.cuh", "quant.cuh", "internal.h")


def _gemm_sources_sha():
    h = hashlib.sha256()
    for f in GEMM_SOURCES:
        with open(os.path.join(ROOT, "moe_decode_step_router_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _traffic_ratios():
    """DRAM traffic of k_expert_gemm per launch over its algorithmic bytes, from the ncu
    summary under profiles/; empty once the kernel sources differ from the captured ones."""
    path = os.path.join(ROOT, "profiles", "k_expert_gemm_traffic.txt")
    vals = {}
    if not os.path.exists(path):
        return vals
    for ln in open(path):
        ln = ln.split("#", 1)[0].strip()
        if "=" in ln:
            k, v = (x.strip() for x in ln.split("=", 1))
            vals[k] = v
    if vals.pop("kernel_sources_sha256", None) != _gemm_sources_sha():
        return {}
    out = {}
    for k, v in vals.items():
        try:
            out[k] = float(v)
        except ValueError:
            pass
    return out


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _max_over_ranks(v, world, device):
    """The job's figure from every rank's own: the largest (the slowest rank's step time)."""
    if world == 1:
        return float(v)
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _host_cpu():
    """Host cores and CPU model of the machine the oracle is timed on."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().lower().startswith("model name"):
                model = ln.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if not model:
        try:
            for ln in open("/proc/cpuinfo"):
                if ln.lower().startswith("model name"):
                    model = ln.split(":", 1)[1].strip()
                    break
        except OSError:
            pass
    return {"nproc": os.cpu_count(), "model": model or platform.processor() or platform.machine(),
            "machine": platform.machine()}


def _config_keys(cfg, n_active, ubytes):
    """The workload's identity: the same keys and values in both arms' lines."""
    return {"workload": cfg["name"], "rows": cfg["M"], "H": cfg["H"], "E": cfg["E"], "k": cfg["k"], "I": cfg["I"],
            "shared_I": cfg["I_sh"], "swiglu_limit": cfg.get("swiglu_limit", 0.0), "unique_experts": int(n_active),
            "unique_bytes": int(ubytes), "l2": L2_NOTE, "parallelism": "single GPU per rank (replicas)"}


# ------------------------------------------------------------------ the oracle on the host
def _host_experts(inp, experts, cache):
    import numpy as np
    n = lambda t: None if t is None else t.detach().cpu().numpy()
    E = inp["w13"][0].shape[0]
    w13, w2 = cache.setdefault("w13", [None] * E), cache.setdefault("w2", [None] * E)
    for e in sorted(set(int(v) for v in np.ravel(experts))):
        if w13[e] is None:
            w13[e] = (n(inp["w13"][0][e]), n(inp["w13"][1][e]) if inp["w13"][1] is not None else None,
                      float(inp["w13"][2][e]))
            w2[e] = (n(inp["w2"][0][e]), n(inp["w2"][1][e]) if inp["w2"][1] is not None else None,
                     float(inp["w2"][2][e]))
    if "sh13" in inp and "sh13" not in cache:
        sh = lambda k: (n(inp[k][0][0]), n(inp[k][1][0]) if inp[k][1] is not None else None, float(inp[k][2][0]))
        cache["sh13"], cache["sh2"] = sh("sh13"), sh("sh2")
    return w13, w2, cache.get("sh13"), cache.get("sh2")


class _Oracle:
    """The oracle, as it stands, on rows of one workload's inputs (host copies)."""

    def __init__(self, cfg, inp):
        import numpy as np
        import torch
        import oracle
        self.oracle = oracle
        u16 = lambda t: t.detach().cpu().contiguous().view(torch.int16).numpy().astype(np.uint16)
        self.cfg, self.inp = cfg, inp
        self.L = oracle.make_layer(cfg, inp["gs_a"])
        self.x16, self.wg16 = u16(inp["x"]), u16(inp["wg"])
        self.r16, self.g16 = u16(inp["residual"]), u16(inp["gamma"])
        self.bias = None if inp["bias"] is None else inp["bias"].detach().cpu().numpy()
        self.cache = {}
        _, _, self.idx, _, _ = oracle.router(self.L, self.x16, self.wg16, bias=self.bias)
        self.w13, self.w2, self.sh13, self.sh2 = _host_experts(inp, self.idx, self.cache)

    def n_active(self):
        import numpy as np
        return len(np.unique(self.idx))

    def rows(self, rows):
        return self.oracle.step_rows(self.L, rows, self.x16, self.r16, self.g16, self.wg16, self.bias, self.w13,
                                     self.w2, self.sh13, self.sh2, want_q=bool(self.cfg.get("emit_next")))


def _pinned_one_core(fn):
    """Runs fn() on one host core (this thread's affinity set to a single CPU, then restored)."""
    cpu = None
    old = None
    if hasattr(os, "sched_getaffinity"):
        old = os.sched_getaffinity(0)
        cpu = max(old)
        os.sched_setaffinity(0, {cpu})
    try:
        return fn(), cpu
    finally:
        if old is not None:
            os.sched_setaffinity(0, old)


def _oracle_row_seconds(orc, budget_s, max_rows=None):
    """Seconds per row of the oracle on one pinned core: whole rows until budget_s."""
    M = orc.cfg["M"] if max_rows is None else min(max_rows, orc.cfg["M"])

    def run():
        done, t = 0, 0.0
        for m in range(M):
            t0 = time.perf_counter()
            orc.rows([m])
            t += time.perf_counter() - t0
            done += 1
            if t > budget_s:
                break
        return t / done, done

    (per_row, done), cpu = _pinned_one_core(run)
    return per_row, done, cpu


# ------------------------------------------------------------------ reference arm
def _reference_arm(a):
    """The oracle as the reference implementation: whole steps of the same workload (all its
    rows, on parallel host threads, one row each), timed on the host, same metric and config."""
    import torch
    from concurrent.futures import ThreadPoolExecutor
    from moe_decode_step_router_gb300 import synth

    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    cfg = _cfg(a)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = synth.make_inputs(cfg, a.seed, device=dev)
    orc = _Oracle(cfg, inp)
    n_active = orc.n_active()
    ubytes = synth.unique_weight_bytes(cfg, n_active)
    M = cfg["M"]
    threads = max(1, min(M, os.cpu_count() or 1))
    times = []
    with ThreadPoolExecutor(max_workers=threads) as ex:
        t_region = time.perf_counter()
        for i in range(a.warmup + a.steps):
            if i == a.warmup:
                t_region = time.perf_counter()
            t0 = time.perf_counter()
            list(ex.map(lambda m: orc.rows([m]), range(M)))
            if i >= a.warmup:
                times.append(time.perf_counter() - t0)
        wall = time.perf_counter() - t_region
    t = sum(times) / len(times)
    val = ubytes / t / 1e9
    host = _host_cpu()
    sample = ("whole steps: all %d rows of the workload through the oracle, one row per host thread (%d threads); "
              "%d warm-up + %d timed steps" % (M, threads, a.warmup, a.steps))
    line = {"metric": METRIC, "value": val, "unit": "GB/s", "n_gpus": a.gpus, "steps": a.steps, "warmup": a.warmup,
            "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic (seeded): inputs of the workload's shapes, random weights",
            "impl": "reference", "config": _config_keys(cfg, n_active, ubytes),
            "timing": {"wall_s_timed_region": wall, "host": host},
            "cpu_baseline": {"value": val, "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": sample,
                             "nproc": host["nproc"], "cpu_model": host["model"]},
            "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU arm
def _stats(ms_list):
    import numpy as np
    a = np.asarray(ms_list, np.float64) * 1e3  # us
    return {"mean_us": float(a.mean()), "median_us": float(np.median(a)), "p10_us": float(np.percentile(a, 10)),
            "p90_us": float(np.percentile(a, 90)), "n": int(a.size)}


def _proj_bytes(fmt, rows, K):
    rb = 2 * K if fmt == 0 else (K if fmt == 1 else K // 2)
    rs = K // 32 if fmt in (1, 3) else (K // 16 if fmt == 2 else 0)
    return rows * (rb + rs) + (4 if fmt == 2 else 0)


def _gemm_bytes(cfg, n_active):
    """Algorithmic bytes of the gate_up and the down launch (weights, scales, global scales)."""
    H, I, Ish = cfg["H"], cfg["I"], cfg["I_sh"]
    gu = n_active * _proj_bytes(cfg["w_fmt"], 2 * I, H) + (_proj_bytes(cfg["sh_fmt"], 2 * Ish, H)
                                                           if cfg["has_shared"] else 0)
    dn = n_active * _proj_bytes(cfg["w_fmt"], H, I) + (_proj_bytes(cfg["sh_fmt"], H, Ish) if cfg["has_shared"] else 0)
    return gu, dn


class _Bench:
    def __init__(self, dev, stream, clocks):
        import torch
        self.torch = torch
        self.dev, self.stream, self.clocks = dev, stream, clocks
        # L2 flush between timed steps: write one 512 MiB buffer, then read another, so that no
        # step input stays in the 129 MB L2 and no dirty line of the flush is left for the step
        # to write back (between two MoE layers of a decode loop L2 holds mostly clean lines).
        self.flush_w = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
        self.flush_r = torch.zeros(128 << 20, dtype=torch.float32, device=dev)
        self.flush_acc = torch.zeros((), dtype=torch.float32, device=dev)

    def flush(self, v):
        self.flush_w.fill_(v)
        self.torch.sum(self.flush_r, dim=0, out=self.flush_acc)

    def timed(self, fn, steps, warmup, tag=1):
        """Per-call device time (ms) of fn on the stream, each call after an untimed L2 flush."""
        torch = self.torch
        for _ in range(warmup):
            with torch.cuda.stream(self.stream):
                self.flush(tag)
                fn()
        self.stream.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        torch.cuda.synchronize()
        t0 = time.time()
        for s, e in ev:
            with torch.cuda.stream(self.stream):
                self.flush(tag)
                s.record(self.stream)
                fn()
                e.record(self.stream)
        self.stream.synchronize()
        self.clocks.window(t0, time.time())
        return [s.elapsed_time(e) for s, e in ev], time.time() - t0

    def workload(self, layer, cfg, x, residual, steps, warmup, ffn_reps):
        """Graph-captured moe_step of `layer` on rows x: step statistics, unique bytes, and the
        one-launch FFN timed alone on the same routing."""
        import numpy as np
        from moe_decode_step_router_gb300 import moestep as ms
        from moe_decode_step_router_gb300 import synth
        torch = self.torch
        M, H = x.shape[0], cfg["H"]
        out = torch.zeros(M, H, dtype=torch.bfloat16, device=self.dev)
        res = residual.clone()
        M8 = -(-M // 8) * 8
        oq = torch.zeros(M8, H, dtype=torch.uint8, device=self.dev) if cfg["emit_next"] else None
        os_ = torch.zeros(M8, H // 32, dtype=torch.uint8, device=self.dev) if cfg["emit_next"] else None
        args = layer.args(x, res, out, oq, os_)
        with torch.cuda.stream(self.stream):
            layer.step(x, res, out, oq, os_, stream=self.stream, args=args)
        self.stream.synchronize()
        if layer.status(self.stream) != 0:
            raise RuntimeError("device status %d after the first step" % layer.status(self.stream))
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=self.stream):
            layer.step(x, res, out, oq, os_, stream=self.stream, args=args)
        step_ms, wall = self.timed(graph.replay, steps, max(3, warmup))
        st = layer.status(self.stream)
        if st != 0:
            raise RuntimeError("device status %d after the timed steps" % st)
        counts = layer.ws_tensor("expert_counts", torch.int32, (cfg["E"] + 1,)).cpu().numpy()
        n_active = int((counts[:cfg["E"]] > 0).sum())
        ubytes = synth.unique_weight_bytes(dict(cfg, M=M), n_active)
        gu_b, dn_b = _gemm_bytes(cfg, n_active)
        v, q = layer.view, layer.qw
        perm = layer.ws_tensor("perm", torch.int32, (M * cfg["k"] + M,))
        ffn = lambda: ms.moe_expert_ffn(layer.d, q["w13"], q["sh13"], q["w2"], q["sh2"], v.xq, v.xq_scales,
                                        v.xq_shared, v.xq_shared_scales, perm, M, v.hq, v.hq_scales, v.y_pairs,
                                        layer.ws, self.stream)
        ffn_ms, _ = self.timed(ffn, ffn_reps, 3, tag=2)
        return dict(graph=graph, step_ms=step_ms, wall=wall, n_active=n_active, ubytes=ubytes, gu_bytes=gu_b,
                    dn_bytes=dn_b, ffn_ms=float(np.mean(ffn_ms)), out=out, res=res, oq=oq, os_=os_, perm=perm)


def _e2e_pipelined(layer, cfg, inp, bench, dev, stream, warmup, steps):
    """End to end through the C ABI with host buffers, as a serving loop runs it: every step
    copies its x and residual in from pinned host memory and its out back, on a copy stream,
    while the compute stream runs the neighbouring step (two buffer sets, each with its own
    captured moe_step graph, ordered by events). Host wall seconds per step."""
    import torch
    M, H = cfg["M"], cfg["H"]
    cs = torch.cuda.Stream(device=dev)
    bufs = []
    for j in range(2):
        b = {"x_h": inp["x"].cpu().pin_memory(), "r_h": inp["residual"].cpu().pin_memory(),
             "o_h": torch.empty(M, H, dtype=torch.bfloat16).pin_memory(),
             "x": torch.empty_like(inp["x"]), "r": torch.empty_like(inp["residual"]),
             "o": torch.zeros(M, H, dtype=torch.bfloat16, device=dev)}
        M8 = -(-M // 8) * 8
        b["oq"] = torch.zeros(M8, H, dtype=torch.uint8, device=dev) if cfg["emit_next"] else None
        b["os"] = torch.zeros(M8, H // 32, dtype=torch.uint8, device=dev) if cfg["emit_next"] else None
        b["x"].copy_(inp["x"])
        b["r"].copy_(inp["residual"])
        args = layer.args(b["x"], b["r"], b["o"], b["oq"], b["os"])
        with torch.cuda.stream(stream):
            layer.step(b["x"], b["r"], b["o"], b["oq"], b["os"], stream=stream, args=args)
        stream.synchronize()
        b["g"] = torch.cuda.CUDAGraph()
        with torch.cuda.graph(b["g"], stream=stream):
            layer.step(b["x"], b["r"], b["o"], b["oq"], b["os"], stream=stream, args=args)
        b["ev_in"], b["ev_comp"], b["ev_out"] = (torch.cuda.Event(), torch.cuda.Event(), torch.cuda.Event())
        bufs.append(b)
    stream.synchronize()

    def h2d(b):
        b["x"].copy_(b["x_h"], non_blocking=True)
        b["r"].copy_(b["r_h"], non_blocking=True)
        b["ev_in"].record(cs)

    def run(n):
        with torch.cuda.stream(cs):
            h2d(bufs[0])
        for i in range(n):
            b, nb = bufs[i % 2], bufs[(i + 1) % 2]
            if i + 1 < n:  # the next step's inputs, while this one runs
                with torch.cuda.stream(cs):
                    if i >= 1:
                        cs.wait_event(nb["ev_comp"])  # step i - 1 is done with that buffer set
                    h2d(nb)
            with torch.cuda.stream(stream):
                stream.wait_event(b["ev_in"])
                if i >= 2:
                    stream.wait_event(b["ev_out"])  # step i - 2's output has been read back
                b["g"].replay()
                b["ev_comp"].record(stream)
            with torch.cuda.stream(cs):
                cs.wait_event(b["ev_comp"])
                b["o_h"].copy_(b["o"], non_blocking=True)
                b["ev_out"].record(cs)
        cs.synchronize()
        stream.synchronize()

    run(max(3, warmup))
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    run(steps)
    wall = time.perf_counter() - t0
    return wall / steps


def _sweep(a, bench, dev, peak, world, cpu_est):
    """Every other workload, measured as the headline is (graph replays, L2 flushed)."""
    import torch
    from moe_decode_step_router_gb300 import synth
    from moe_decode_step_router_gb300.runtime import MoELayer

    entries = []
    by_layer = {}
    for name, rows in SWEEP:
        by_layer.setdefault(name, []).append(rows)
    for name, rows_list in by_layer.items():
        base = _cfg(a, name, None)
        Mmax = max(r or base["M"] for r in rows_list)
        inp = synth.make_inputs(dict(base, M=Mmax), a.seed, device=dev, M=Mmax)
        layer = MoELayer(dict(base, M=Mmax), inp, dev)
        oracle_row_s = None
        if cpu_est:
            orc = _Oracle(dict(base, M=1), dict(inp, x=inp["x"][:1], residual=inp["residual"][:1]))
            oracle_row_s, _, _ = _oracle_row_seconds(orc, budget_s=3.0, max_rows=1)
            del orc
        for k in ("w13", "w2", "sh13", "sh2"):
            inp.pop(k, None)
        torch.cuda.empty_cache()
        for rows in rows_list:
            M = rows or base["M"]
            cfg = dict(base, M=M)
            x, r = inp["x"][:M].contiguous(), inp["residual"][:M].contiguous()
            w = bench.workload(layer, cfg, x, r, SWEEP_STEPS, SWEEP_WARMUP, ffn_reps=50)
            st = _stats(w["step_ms"])
            gbs_med = w["ubytes"] / (st["median_us"] * 1e-6) / 1e9
            ffn_gbs = (w["gu_bytes"] + w["dn_bytes"]) / (w["ffn_ms"] * 1e-3) / 1e9
            e = dict(_config_keys(cfg, w["n_active"], w["ubytes"]), **st)
            e.update({"rows_per_s": M / (st["median_us"] * 1e-6), "gbs_median": gbs_med,
                      "frac_of_measured_peak": gbs_med / peak, "frac_of_8000": gbs_med / 8000.0,
                      "ffn_launch_us": w["ffn_ms"] * 1e3, "ffn_roofline_frac": ffn_gbs / peak,
                      "w_fmt": synth.FMT_NAMES[cfg["w_fmt"]], "shared_fmt": synth.FMT_NAMES[cfg["sh_fmt"]]})
            if oracle_row_s is not None:
                e["oracle_ms_per_step_1core"] = oracle_row_s * M * 1e3
                e["oracle_note"] = "one row of the layer timed on one pinned host core, times the rows"
            entries.append(e)
            del w
        del layer, inp
        torch.cuda.empty_cache()
    return entries


def main(argv=None):
    a = _args(argv)
    if a.impl == "reference":
        return _reference_arm(a)

    import numpy as np
    import torch
    import torch.distributed as dist

    from moe_decode_step_router_gb300 import moestep as ms
    from moe_decode_step_router_gb300 import synth
    from moe_decode_step_router_gb300.runtime import MoELayer

    world, rank, local = _dist()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    cfg = _cfg(a)
    M, H = cfg["M"], cfg["H"]
    inp = synth.make_inputs(cfg, a.seed, device=dev)
    layer = MoELayer(cfg, inp, dev)
    keep_inputs = rank == 0 and not a.no_cpu_baseline
    canon = {k: inp[k] for k in ("w13", "w2", "sh13", "sh2") if k in inp}
    if not keep_inputs:
        for k in canon:
            inp.pop(k)
        del canon
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    stream = torch.cuda.Stream(device=dev)
    stream.wait_stream(torch.cuda.current_stream())
    clocks = Clocks(local)
    clocks.start()
    bench = _Bench(dev, stream, clocks)
    try:
        peak, peak_src = float(json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        peak, peak_src = 6800.0, "fallback"

    # ---- the headline: K timed graph replays
    if world > 1:
        dist.barrier()
    x_dev = inp["x"].clone()
    w = bench.workload(layer, cfg, x_dev, inp["residual"], a.steps, a.warmup, ffn_reps=max(10, a.steps // 2))
    if world > 1:
        dist.barrier()
    st = _stats(w["step_ms"])
    wall_timed = w["wall"]
    ms_step = _max_over_ranks(st["mean_us"] * 1e-3, world, dev)
    n_active, ubytes = w["n_active"], w["ubytes"]
    gbs = ubytes / (ms_step * 1e-3) / 1e9

    # ---- the separate gate_up and down launches, live, on the launching stream
    v, q, perm = layer.view, layer.qw, w["perm"]
    reps = max(10, a.steps // 2)
    gu_ms = float(np.mean(bench.timed(lambda: ms.moe_expert_gate_up(
        layer.d, q["w13"], q["sh13"], v.xq, v.xq_scales, v.xq_shared, v.xq_shared_scales, perm, M, v.hq,
        v.hq_scales, layer.ws, stream), reps, 3, tag=3)[0]))
    dn_ms = float(np.mean(bench.timed(lambda: ms.moe_expert_down(
        layer.d, q["w2"], q["sh2"], v.hq, v.hq_scales, M, v.y_pairs, layer.ws, stream), reps, 3, tag=4)[0]))
    full_size = a.rows is None and a.experts is None and a.inter is None
    tr = _traffic_ratios() if full_size else {}

    def kern(part, nbytes, t_ms):
        key = cfg["name"] + "." + part
        return {"achieved": nbytes / (t_ms * 1e-3) / 1e9, "ms": t_ms, "algorithmic_bytes": nbytes,
                "traffic": tr[key] * nbytes if key in tr else None}

    fused = cfg["ffn_launches"] != 2
    if fused:
        dom, name = kern("ffn", w["gu_bytes"] + w["dn_bytes"], w["ffn_ms"]), "k_expert_gemm(gate_up+down)"
    else:
        dom, name = kern("gate_up", w["gu_bytes"], gu_ms), "k_expert_gemm(gate_up)"
    roofline = {"bound": "hbm", "kernel": name, "achieved": dom["achieved"], "peak": peak, "peak_source": peak_src,
                "unit": "GB/s", "frac": dom["achieved"] / peak, "traffic": dom["traffic"],
                "algorithmic_bytes": dom["algorithmic_bytes"], "ms": dom["ms"],
                "note": ("the launch timed alone after an L2 flush, so every byte it reads (including its own "
                         "L2 prefetch of the shared expert's records) comes from HBM inside the timed launch; "
                         "the peak is a copy's (read + write), which a pure read stream can exceed slightly"),
                "gate_up": kern("gate_up", w["gu_bytes"], gu_ms), "down": kern("down", w["dn_bytes"], dn_ms),
                "step_frac": gbs / peak}

    # ---- end to end with host buffers: H2D of the step's inputs, the step, D2H of its output
    x_h = inp["x"].cpu().pin_memory()
    r_h = inp["residual"].cpu().pin_memory()
    o_h = torch.empty(M, H, dtype=torch.bfloat16).pin_memory()
    e2e, parts = [], []
    for i in range(a.warmup + max(10, a.steps // 2)):
        with torch.cuda.stream(stream):
            bench.flush(5)
        stream.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        t1 = time.perf_counter()
        with torch.cuda.stream(stream):
            ev[0].record(stream)
            x_dev.copy_(x_h, non_blocking=True)
            w["res"].copy_(r_h, non_blocking=True)
            ev[1].record(stream)
            w["graph"].replay()
            ev[2].record(stream)
            o_h.copy_(w["out"], non_blocking=True)
            ev[3].record(stream)
        stream.synchronize()
        if i >= a.warmup:
            e2e.append(time.perf_counter() - t1)
            parts.append([ev[0].elapsed_time(ev[1]), ev[1].elapsed_time(ev[2]), ev[2].elapsed_time(ev[3])])
    e2e_serial_s = float(np.median(e2e))
    pm = np.median(np.asarray(parts), axis=0)
    h2d = x_h.numel() * 2 + r_h.numel() * 2
    d2h = o_h.numel() * 2
    e2e_s = _e2e_pipelined(layer, cfg, inp, bench, dev, stream, a.warmup, max(20, a.steps))
    sweep = None
    if rank == 0 and not a.no_sweep and a.config == HEADLINE and full_size:
        del w
        cpu_est = not a.no_cpu_baseline
        sweep = _sweep(a, bench, dev, peak, world, cpu_est)
    clk = clocks.stop()

    cpu = None
    if keep_inputs:
        orc = _Oracle(cfg, dict(inp, **canon))
        per_row, rows_done, pinned = _oracle_row_seconds(orc, budget_s=20.0)
        t_cpu = per_row * M
        host = _host_cpu()
        cpu = {"value": ubytes / t_cpu / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": "%d of %d rows of the same workload through the oracle on one pinned core (cpu %s), "
                         "scaled to the full step" % (rows_done, M, pinned),
               "ms_per_step": t_cpu * 1e3, "nproc": host["nproc"], "cpu_model": host["model"]}

    if rank == 0:
        line = {"metric": METRIC, "value": gbs * world, "unit": "GB/s", "n_gpus": world, "steps": a.steps,
                "warmup": a.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": synth.FMT_NAMES[cfg["w_fmt"]],
                "data": "synthetic (seeded): inputs of the workload's shapes, random weights",
                "config": _config_keys(cfg, n_active, ubytes),
                "step": dict(st, us_per_step=ms_step * 1e3, rows_per_s=M / (ms_step * 1e-3),
                             frac_of_measured_peak=gbs / peak, frac_of_8000=gbs / 8000.0,
                             gbs_median=ubytes / (st["median_us"] * 1e-6) / 1e9, wall_s_timed_region=wall_timed),
                "e2e": {"value": ubytes / e2e_s / 1e9 * world, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                        "d2h_bytes_per_step": d2h, "ms_per_step": e2e_s * 1e3,
                        "path": "every step: pinned host x and residual copied in, the captured moe_step graph, out "
                                "copied back to pinned host memory; two buffer sets, the copies on a second stream "
                                "overlapping the neighbouring steps (a serving loop's order); no L2 flush (the "
                                "weights streamed per step are far larger than L2); host wall time over the run / "
                                "steps",
                        "serial": {"ms_per_step": e2e_serial_s * 1e3,
                                   "device_ms": {"h2d": float(pm[0]), "step_graph": float(pm[1]), "d2h": float(pm[2])},
                                   "path": "one step at a time, L2 flushed before each (untimed); host wall time "
                                           "per step (median)"}},
                "roofline": roofline, "cpu_baseline": cpu, "clocks": clk,
                "gpu_launches": ((4 if fused else 5) - (1 if cfg["front_launches"] == 1 else 0)) * a.steps,
                "sweep": sweep}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
